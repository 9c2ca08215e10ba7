// CPU stand-in for the CUDA features the selective-scan kernel uses, so that its source can be
// compiled with g++ and run on the host (tests/test_s6_kernel_on_cpu.py).  A block's threads are
// host threads; __syncthreads and __syncwarp are barriers; shared memory is one static array,
// since blocks run one after another.  Only control flow and indexing are checked this way:
// the special-function exp2 is replaced by exp2f.
#pragma once
#include <barrier>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <functional>
#include <thread>
#include <vector>

#define __global__
#define __device__
#define __host__
#define __forceinline__ inline
#define __restrict__
#define __launch_bounds__(...)
#define __grid_constant__
#define __align__(n) __attribute__((aligned(n)))

struct dim3 { unsigned x = 1, y = 1, z = 1; dim3() {} dim3(unsigned a, unsigned b = 1, unsigned c = 1) : x(a), y(b), z(c) {} };
struct float2 { float x, y; };
struct float4 { float x, y, z, w; };
struct uint4 { unsigned x, y, z, w; };
inline float2 make_float2(float a, float b) { return {a, b}; }
inline float4 make_float4(float a, float b, float c, float d) { return {a, b, c, d}; }
inline uint4 make_uint4(unsigned a, unsigned b, unsigned c, unsigned d) { return {a, b, c, d}; }
inline float __uint_as_float(unsigned u) { float f; std::memcpy(&f, &u, 4); return f; }
inline unsigned __float_as_uint(float f) { unsigned u; std::memcpy(&u, &f, 4); return u; }
using std::exp2f;
using std::fmaf;
template <class T> inline T min(T a, T b) { return a < b ? a : b; }
template <class T> inline T max(T a, T b) { return a > b ? a : b; }

struct __nv_bfloat16 { uint16_t b; };
inline float __bfloat162float(__nv_bfloat16 v) { return __uint_as_float((unsigned)v.b << 16); }
inline __nv_bfloat16 __float2bfloat16_rn(float f)
{
    unsigned u = __float_as_uint(f);
    unsigned r = u + 0x7fffu + ((u >> 16) & 1u);   // round to nearest even (finite inputs)
    return __nv_bfloat16{(uint16_t)(r >> 16)};
}

// per-thread builtins
extern thread_local dim3 threadIdx, blockIdx;
extern dim3 blockDim, gridDim;

struct EmuBlock {
    std::barrier<> *bar;
    std::vector<std::barrier<> *> warp_bar;
    float shfl[64][32];
};
extern thread_local EmuBlock *emu_block;

inline void __syncthreads() { emu_block->bar->arrive_and_wait(); }
inline float __shfl_xor_sync(unsigned, float v, int off)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    emu_block->shfl[warp][lane] = v;
    emu_block->warp_bar[warp]->arrive_and_wait();
    const float r = emu_block->shfl[warp][lane ^ off];
    emu_block->warp_bar[warp]->arrive_and_wait();
    return r;
}
inline float __shfl_up_sync(unsigned, float v, int off)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    emu_block->shfl[warp][lane] = v;
    emu_block->warp_bar[warp]->arrive_and_wait();
    const float r = lane >= off ? emu_block->shfl[warp][lane - off] : v;
    emu_block->warp_bar[warp]->arrive_and_wait();
    return r;
}

// run fn() as a grid of blocks, one block at a time, each thread a host thread
inline void emu_launch(dim3 grid, dim3 block, const std::function<void()> &fn)
{
    gridDim = grid;
    blockDim = block;
    const unsigned nt = block.x;
    for (unsigned bz = 0; bz < grid.z; ++bz)
        for (unsigned by = 0; by < grid.y; ++by)
            for (unsigned bx = 0; bx < grid.x; ++bx) {
                EmuBlock eb;
                std::barrier<> bar((std::ptrdiff_t)nt);
                eb.bar = &bar;
                std::vector<std::barrier<> *> wb;
                for (unsigned w = 0; w < (nt + 31) / 32; ++w) eb.warp_bar.push_back(new std::barrier<>(32));
                std::vector<std::thread> th;
                for (unsigned t = 0; t < nt; ++t)
                    th.emplace_back([&, t] {
                        threadIdx = dim3(t, 0, 0);
                        blockIdx = dim3(bx, by, bz);
                        emu_block = &eb;
                        fn();
                    });
                for (auto &x : th) x.join();
                for (auto *p : eb.warp_bar) delete p;
            }
}
inline float2 __fmul2_rn(float2 a, float2 b) { return {a.x * b.x, a.y * b.y}; }
inline float2 __ffma2_rn(float2 a, float2 b, float2 c) { return {std::fmaf(a.x, b.x, c.x), std::fmaf(a.y, b.y, c.y)}; }
#include <type_traits>
inline void __syncwarp(unsigned = 0xffffffffu) { emu_block->warp_bar[threadIdx.x >> 5]->arrive_and_wait(); }
// the block's dynamic shared memory (blocks run one at a time)
inline float4 *emu_smem()
{
    static float4 buf[1 << 16];
    return buf;
}
