// S1: persistent pooled block-key cache update.
//
// llama.cpp issue #28734 ("decode slows linearly with context"), fix summary,
// lever2: the indexer used to re-gather, mean-pool, RMS-norm and re-RoPE every
// cached block each token; a persistent buffer of pooled block keys is kept
// instead and only the blocks an ubatch dirtied are recomputed.  lever2b: the
// member cells of each block stay on the device (blk_cells).
//
// One warp per dirty slot.  Lane l owns dims {2l, 2l+1} and their NeoX partners
// {64+2l, 64+2l+1}, so every rotation pair lives in one lane and a row of 128
// fp16 keys is read as two coalesced 128-byte half2 sweeps.  All member cells
// are read first and all their key rows next (two dependent loads in all).
// Mean and RMSNorm are fp32.  Rotation angles reach 2.5e5 rad at 250k context,
// where an fp32 angle would be off by ~1e-2 rad, so the angle is reduced
// exactly in integers: each frequency is a 64-bit fixed-point fraction of a
// turn (computed once on the host), the integer position times it wraps to
// the angle's fractional turn, and only that small remainder goes through
// fp32 sincospi.  No fp64 runs on the device (fp64 is a small fraction of
// fp32 throughput on this part).
#include <cmath>

#include "qsa_internal.cuh"

QSA_TS_DECLARE(pool)

namespace qsa {
namespace {

constexpr int kPoolWarps = 4;
constexpr int kMaxR = 8;     // compress_ratio limit of the library

// Rotation frequencies as exact fixed-point fractions of a turn:
// turns[d] = round(theta^(-2d/128) / (2*pi) * 2^64).  For an integer position
// p, the low 64 bits of p * turns[d] are the angle's fractional turn (the
// integer multiply wraps modulo one turn exactly), accurate to p * 2^-64 turns.
struct Turns {
  unsigned long long f[kIdxDim / 2];
};

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

__global__ void __launch_bounds__(kPoolWarps * 32)
k_pool_update(const __half* __restrict__ idx_k, int64_t n_cells,
              const int32_t* __restrict__ blk_cells,
              const int32_t* __restrict__ slot_block_idx, int64_t n_slots,
              const int32_t* __restrict__ dirty, int n_dirty,
              const float* __restrict__ norm_w, float* __restrict__ pooled,
              int r, const Turns turns, float eps, unsigned* err) {
  const int lane = threadIdx.x & 31;
  const int64_t w = (int64_t)blockIdx.x * kPoolWarps + (threadIdx.x >> 5);
  QSA_TS(pool, 0);
  // The block table, keys and dirty list may come from the preceding kernel.
  grid_dep_wait();
  grid_dep_launch();
  QSA_TS(pool, 1);
  if (w >= n_dirty) return;
  const int slot = dirty[w];
  if (slot < 0) return;  // power-of-two padding
  if (slot >= n_slots) {
    if (lane == 0) atomicOr(err, kErrSlot);
    return;
  }

  // All member cells first, then all their key rows: two dependent loads in
  // all instead of two per member.
  int cell[kMaxR];
  const int32_t* mem = blk_cells + (int64_t)slot * r;
#pragma unroll
  for (int i = 0; i < kMaxR; ++i) cell[i] = i < r ? mem[i] : -1;
  const int blk = slot_block_idx[slot];
  float2 lo[kMaxR], hi[kMaxR];
#pragma unroll
  for (int i = 0; i < kMaxR; ++i) {
    const bool ok = cell[i] >= 0 && cell[i] < n_cells;
    if (cell[i] >= n_cells && lane == 0) atomicOr(err, kErrCell);
    const __half2* row = reinterpret_cast<const __half2*>(idx_k + (int64_t)(ok ? cell[i] : 0) * kIdxDim);
    lo[i] = ok ? __half22float2(row[lane]) : make_float2(0.f, 0.f);        // dims 2l, 2l+1
    hi[i] = ok ? __half22float2(row[32 + lane]) : make_float2(0.f, 0.f);   // dims 64+2l, 64+2l+1
    if (!ok) cell[i] = -1;
  }
  QSA_TS(pool, 2);
  float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
  int present = 0;
#pragma unroll
  for (int i = 0; i < kMaxR; ++i) {
    if (cell[i] < 0) continue;
    a0 += lo[i].x; a1 += lo[i].y; b0 += hi[i].x; b1 += hi[i].y;
    ++present;
  }
  float* out = pooled + (int64_t)slot * kIdxDim;
  if (present == 0) {
    reinterpret_cast<float2*>(out)[lane] = make_float2(0.f, 0.f);
    reinterpret_cast<float2*>(out)[32 + lane] = make_float2(0.f, 0.f);
    return;
  }
  const float inv_c = 1.0f / (float)present;
  a0 *= inv_c; a1 *= inv_c; b0 *= inv_c; b1 *= inv_c;
  QSA_TS(pool, 4);

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
  QSA_TS(pool, 3);
  reinterpret_cast<float2*>(out)[lane] = make_float2(x0 * c0 - y0 * s0, x1 * c1 - y1 * s1);
  reinterpret_cast<float2*>(out)[32 + lane] = make_float2(y0 * c0 + x0 * s0, y1 * c1 + x1 * s1);
}

}  // namespace

cudaError_t launch_pool_update(const qsa_config& cfg, const __half* idx_k, int64_t n_cells,
                               const int32_t* blk_cells, const int32_t* slot_block_idx,
                               int64_t n_slots, const int32_t* dirty, int n_dirty,
                               const float* norm_w, float* pooled, unsigned* err,
                               cudaStream_t stream) {
  if (n_dirty <= 0) return cudaSuccess;
  const unsigned blocks = (unsigned)ceil_div(n_dirty, kPoolWarps);
  // f_d = theta^(-2d/128) in double (as the reference definition computes it),
  // then its fraction of a turn in long double, scaled to 2^64.
  Turns turns{};
  const long double two_pi = 6.28318530717958647692528676655900577L;
  for (int d = 0; d < kIdxDim / 2; ++d) {
    const double f = std::pow((double)cfg.rope_theta, (-2.0 * (double)d) / (double)kIdxDim);
    const long double x = ((long double)f / two_pi) * 18446744073709551616.0L;   // * 2^64
    turns.f[d] = x >= 18446744073709551615.0L ? ~0ull : (unsigned long long)(x + 0.5L);
  }
  prof_before(kKPool, stream);
  cudaError_t e = launch_pdl(k_pool_update, dim3(blocks), dim3(kPoolWarps * 32), 0, stream, 1, idx_k, n_cells,
                             blk_cells, slot_block_idx, n_slots, dirty, n_dirty, norm_w, pooled,
                             cfg.compress_ratio, turns, cfg.rms_eps, err);
  prof_after(kKPool, stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace qsa
