// CPU stand-in for the library's common header: the types and conversions the selective-scan
// kernel's source uses (tests/test_s6_kernel_on_cpu.py).
#pragma once
#include "cuda_shim.h"
namespace ssd {
constexpr float kLog2e = 1.4426950408889634f;
inline float to_f32(float v) { return v; }
inline float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T> inline T from_f32(float v);
template <> inline float from_f32<float>(float v) { return v; }
template <> inline __nv_bfloat16 from_f32<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }
struct S6Problem { int64_t B, L, dim, N, G; int in_dt, out_dt; };
}  // namespace ssd
