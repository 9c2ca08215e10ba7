// tc_common.cuh -- helpers shared by the tensor-core kernels (ssd_tc.cu, ssd_fused.cu):
// bf16 pair packing, the 128-byte swizzle, named barriers, the device error word, and the
// host-side tensor-map encoder.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "sm100_ptx.cuh"
#include "ssd_common.cuh"

namespace ssd {
namespace tc {

constexpr int kQ = 128;                       // tokens per tensor-core sub-chunk (MMA M)
constexpr uint32_t kAtom = kQ * 128;          // bytes of one 128-row x 128-byte swizzled region
// Bound on every wait of a kernel on another role's progress: 250 ms (legitimate waits take
// microseconds).  Kernels take it as an argument (ssd_desc flags can shorten it for tests);
// the waits that retire a kernel's own copies and MMAs before it exits always use this one.
constexpr uint64_t kWaitNs = 250000000ull;

// Device error word bits.
constexpr int kErrTimeout = 1;                // a bounded wait expired
constexpr int kErrSmemAlign = 4;              // the dynamic shared memory base was not 1024-byte aligned

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Two bf16 products (the low and high halves of u times w), rounded to bf16.
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t u, __nv_bfloat162 w)
{
    __nv_bfloat162 v = __hmul2(*reinterpret_cast<__nv_bfloat162 *>(&u), w);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t u)
{
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162 *>(&u);
    return __bfloat1622float2(v);
}

// Byte offset of 16-byte chunk c of row r inside a 1024-byte-aligned region of
// 128-byte rows with the 128-byte swizzle (the layout TMA writes and the MMA reads).
__device__ __forceinline__ uint32_t sw128(uint32_t r, uint32_t c) { return r * 128u + (((c ^ (r & 7u)) & 7u) << 4); }

// Hardware barrier among `nthreads` threads (named barrier `id`).  Callers keep their
// control flow uniform -- every participating thread reaches every call, errors or
// not -- so this never waits on a thread that left.
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier that also returns the OR of `pred` over the participating threads, so that
// a decision taken after it (stop, skip) is the same in every thread of the group.
__device__ __forceinline__ bool named_bar_or(uint32_t id, uint32_t nthreads, bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void set_error(int *err, int bit)
{
    if (err) atomicOr(err, bit);
}

// ---- host side ------------------------------------------------------------------

inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
    });
    return fn;
}

// 4-D bf16 tensor [d3][d2][d1][d0] (d0 contiguous), box {64, 1, rows, 1}, 128-byte swizzle.
inline bool make_map_4d(CUtensorMap *map, const void *ptr, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t d3,
                        uint32_t rows)
{
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[4] = {d0, d1, d2, d3};
    cuuint64_t strides[3] = {d0 * 2, d0 * d1 * 2, d0 * d1 * d2 * 2};
    cuuint32_t box[4] = {64, 1, rows, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline int current_sms()
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 1;
    return sms > 0 ? sms : 1;
}

}  // namespace tc
}  // namespace ssd
