// Device helpers shared by the attention kernels (per-token and union
// tiles): warp reductions of the 8 heads of a KV group, half-CTA barriers and
// the q8_0 -> fp16 row conversion.
#pragma once

#include <cstdint>
#include <cstring>
#include <cuda_fp16.h>

namespace qsa {
namespace {

constexpr unsigned kWarpAll = 0xffffffffu;

// Reduces v[0..7] over the 32 lanes of a warp by a reduce-scatter (9
// shuffles for the 8 values): every lane returns the total of value
// (lane >> 2).
template <class Op>
__device__ __forceinline__ float warp_reduce8(const float (&v)[8], int lane, Op op) {
  const bool b4 = (lane & 16) != 0, b3 = (lane & 8) != 0, b2 = (lane & 4) != 0;
  float x4[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float keep = b4 ? v[i + 4] : v[i], send = b4 ? v[i] : v[i + 4];
    x4[i] = op(keep, __shfl_xor_sync(kWarpAll, send, 16));
  }
  float x2[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float keep = b3 ? x4[i + 2] : x4[i], send = b3 ? x4[i] : x4[i + 2];
    x2[i] = op(keep, __shfl_xor_sync(kWarpAll, send, 8));
  }
  float x = op(b2 ? x2[1] : x2[0], __shfl_xor_sync(kWarpAll, b2 ? x2[0] : x2[1], 4));
  x = op(x, __shfl_xor_sync(kWarpAll, x, 2));
  return op(x, __shfl_xor_sync(kWarpAll, x, 1));
}
struct OpMax {
  __device__ __forceinline__ float operator()(float a, float b) const { return fmaxf(a, b); }
};
struct OpAdd {
  __device__ __forceinline__ float operator()(float a, float b) const { return a + b; }
};

// Barrier among the 128 threads of warps 0-3 (id 1) or of warps 4-7 (id 2).
__device__ __forceinline__ void bar_half(int id) { asm volatile("bar.sync %0, 128;\n" ::"r"(id) : "memory"); }

// 8 int8 values * scale -> 8 fp16 packed in a uint4, with no int->float
// conversion (a quarter-rate pipe): byte b + 128 is placed in the low
// mantissa byte of 1024.0h (exactly 1024 + b + 128), 1152 is subtracted
// (exact), and the fp16 product with the scale is rounded once, which equals
// rounding the exact fp32 product d * q to fp16.
__device__ __forceinline__ uint4 dq8(uint2 raw, __half2 s2) {
  const uint32_t lo = raw.x ^ 0x80808080u, hi = raw.y ^ 0x80808080u;
  const __half2 bias = __float2half2_rn(1152.0f);
  uint32_t w[4] = {__byte_perm(lo, 0x64646464u, 0x5140), __byte_perm(lo, 0x64646464u, 0x5342),
                   __byte_perm(hi, 0x64646464u, 0x5140), __byte_perm(hi, 0x64646464u, 0x5342)};
  uint4 o;
  __half2* h = reinterpret_cast<__half2*>(&o);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __half2 v;
    memcpy(&v, &w[i], 4);
    h[i] = __hmul2(__hsub2(v, bias), s2);
  }
  return o;
}

}  // namespace
}  // namespace qsa
