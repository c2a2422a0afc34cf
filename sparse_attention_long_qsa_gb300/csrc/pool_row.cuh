// Pooled block key from its members' indexer-key rows, computed by one warp.
// Shared by the pool update kernel and the append kernel (which re-pools the
// blocks it dirties), so both produce bit-identical rows.
//
// llama.cpp issue #28734, fix summary, lever2: a block's key is its member
// cells' indexer keys gathered, mean-pooled, RMS-normed and re-RoPEd.
//
// Lane l owns dims {2l, 2l+1} and their NeoX partners {64+2l, 64+2l+1}, so
// every rotation pair lives in one lane.  Mean and RMSNorm are fp32.
// Rotation angles reach 2.5e5 rad at 250k context, where an fp32 angle would
// be off by ~1e-2 rad, so the angle is reduced exactly in integers: each
// frequency is a 64-bit fixed-point fraction of a turn (computed once on the
// host), the integer position times it wraps to the angle's fractional turn,
// and only that small remainder goes through fp32 sincospi.  No fp64 runs on
// the device (fp64 is a small fraction of fp32 throughput on this part).
#pragma once

#include <cmath>

#include "qsa_internal.cuh"

namespace qsa {

constexpr int kMaxR = 8;     // compress_ratio limit of the library

// Rotation frequencies as exact fixed-point fractions of a turn:
// turns[d] = round(theta^(-2d/128) / (2*pi) * 2^64).  For an integer position
// p, the low 64 bits of p * turns[d] are the angle's fractional turn (the
// integer multiply wraps modulo one turn exactly), accurate to p * 2^-64 turns.
struct Turns {
  unsigned long long f[kIdxDim / 2];
};

// f_d = theta^(-2d/128) in double (as the method's definition computes it),
// then its fraction of a turn in long double, scaled to 2^64.
inline Turns make_turns(float theta) {
  Turns turns{};
  const long double two_pi = 6.28318530717958647692528676655900577L;
  for (int d = 0; d < kIdxDim / 2; ++d) {
    const double f = std::pow((double)theta, (-2.0 * (double)d) / (double)kIdxDim);
    const long double x = ((long double)f / two_pi) * 18446744073709551616.0L;   // * 2^64
    turns.f[d] = x >= 18446744073709551615.0L ? ~0ull : (unsigned long long)(x + 0.5L);
  }
  return turns;
}

// cos and sin of 2*pi*(u / 2^64): the fraction of a turn is split into an
// fp32 hi part (top 24 bits, exact) and the rest, then
//   sin(pi*(x_hi + x_lo)) ~ sinpi(x_hi) + pi*x_lo*cospi(x_hi)
// with x = 2u/2^64 - 2 in [-2, 0) so the argument stays small.
__device__ __forceinline__ void sincos_turn(unsigned long long u, float* s, float* c) {
  const unsigned long long hi = u >> 40;                          // 24 bits
  const unsigned long long lo = u & ((1ull << 40) - 1ull);        // 40 bits
  const float xh = (float)hi * (2.0f / 16777216.0f) - 2.0f;       // 2*hi/2^24 - 2, exact
  const float xl = (float)lo * (2.0f / 1099511627776.0f / 16777216.0f);   // 2*lo/2^64
  float sh, ch;
  sincospif(xh, &sh, &ch);
  const float pxl = 3.14159265358979f * xl;
  *s = fmaf(pxl, ch, sh);
  *c = fmaf(-pxl, sh, ch);
}

// The pooled key of a block at block index `blk` from its members' rows: lane
// l holds lo[i] = dims {2l, 2l+1} and hi[i] = dims {64+2l, 64+2l+1} of member
// i, present[i] says whether member i exists.  Lane l returns the same dims
// of the key.  No present member gives zeros.
__device__ __forceinline__ void pool_rows_warp(const float2 (&lo)[kMaxR], const float2 (&hi)[kMaxR],
                                               const bool (&present)[kMaxR], int blk, int r,
                                               const float* __restrict__ norm_w, const Turns& turns,
                                               float eps, float2* lo_out, float2* hi_out) {
  const int lane = threadIdx.x & 31;
  float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
  int n = 0;
#pragma unroll
  for (int i = 0; i < kMaxR; ++i) {
    if (!present[i]) continue;
    a0 += lo[i].x; a1 += lo[i].y; b0 += hi[i].x; b1 += hi[i].y;
    ++n;
  }
  if (n == 0) {
    *lo_out = make_float2(0.f, 0.f);
    *hi_out = make_float2(0.f, 0.f);
    return;
  }
  const float inv_c = 1.0f / (float)n;
  a0 *= inv_c; a1 *= inv_c; b0 *= inv_c; b1 *= inv_c;

  // RMSNorm over the 128 dims.
  float ss = a0 * a0 + a1 * a1 + b0 * b0 + b1 * b1;
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
  const float inv = 1.0f / sqrtf(ss * (1.0f / (float)kIdxDim) + eps);
  const float2 wlo = reinterpret_cast<const float2*>(norm_w)[lane];
  const float2 whi = reinterpret_cast<const float2*>(norm_w)[32 + lane];
  const float x0 = a0 * inv * wlo.x, x1 = a1 * inv * wlo.y;
  const float y0 = b0 * inv * whi.x, y1 = b1 * inv * whi.y;

  // NeoX RoPE at the block's first position j*r: pair (d, d+64) turns by
  // pos * theta^(-2d/128).
  const unsigned long long pos = (unsigned long long)blk * (unsigned long long)r;
  float s0, c0, s1, c1;
  sincos_turn(pos * turns.f[2 * lane], &s0, &c0);
  sincos_turn(pos * turns.f[2 * lane + 1], &s1, &c1);
  *lo_out = make_float2(x0 * c0 - y0 * s0, x1 * c1 - y1 * s1);
  *hi_out = make_float2(y0 * c0 + x0 * s0, y1 * c1 + x1 * s1);
}

}  // namespace qsa
