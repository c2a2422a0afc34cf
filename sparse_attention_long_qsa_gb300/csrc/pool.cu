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
// fp16 keys is read as two coalesced 128-byte half2 sweeps.  Mean and RMS are
// accumulated in fp64 (means of at most r fp16 values are exact).  Rotation
// angles reach 2.5e5 rad at 250k context, where an fp32 angle would be off by
// ~1e-2 rad: the angle pos * theta^(-2d/128) is formed in fp64 from
// frequencies computed on the host in fp64, reduced to [-pi, pi] in fp64 with
// a two-part 2*pi, and only the reduced angle (as an fp32 hi + lo pair) goes
// through fp32 sincos, so no fp64 transcendental runs on the device (fp64
// throughput on this part is a small fraction of fp32).
#include <cmath>

#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kPoolWarps = 4;

struct InvFreq {
  double f[kIdxDim / 2];   // theta^(-2d/idx_dim), d < idx_dim/2
};

// cos and sin of an fp64 angle: reduction by 2*pi in fp64, then fp32 sincos of
// the reduced angle split into hi + lo.
__device__ __forceinline__ void sincos_reduced(double a, float* s, float* c) {
  const double two_pi_hi = 6.283185307179586;          // fp64 nearest to 2*pi
  const double two_pi_lo = 2.4492935982947064e-16;     // 2*pi - two_pi_hi
  const double k = rint(a * 0.15915494309189535);      // a / (2*pi)
  double r = fma(-k, two_pi_hi, a);
  r = fma(-k, two_pi_lo, r);
  const float rh = (float)r;
  const float rl = (float)(r - (double)rh);
  float sh, ch;
  sincosf(rh, &sh, &ch);
  *c = fmaf(-sh, rl, ch);
  *s = fmaf(ch, rl, sh);
}

__global__ void __launch_bounds__(kPoolWarps * 32)
k_pool_update(const __half* __restrict__ idx_k, int64_t n_cells,
              const int32_t* __restrict__ blk_cells,
              const int32_t* __restrict__ slot_block_idx, int64_t n_slots,
              const int32_t* __restrict__ dirty, int n_dirty,
              const float* __restrict__ norm_w, float* __restrict__ pooled,
              int r, const InvFreq inv_freq, double eps, unsigned* err) {
  const int lane = threadIdx.x & 31;
  const int64_t w = (int64_t)blockIdx.x * kPoolWarps + (threadIdx.x >> 5);
  if (w >= n_dirty) return;
  const int slot = dirty[w];
  if (slot < 0) return;  // power-of-two padding
  if (slot >= n_slots) {
    if (lane == 0) atomicOr(err, kErrSlot);
    return;
  }

  double a0 = 0.0, a1 = 0.0, b0 = 0.0, b1 = 0.0;
  int present = 0;
  for (int i = 0; i < r; ++i) {
    const int c = blk_cells[(int64_t)slot * r + i];
    if (c < 0) continue;
    if (c >= n_cells) {
      if (lane == 0) atomicOr(err, kErrCell);
      continue;
    }
    const __half2* row = reinterpret_cast<const __half2*>(idx_k + (int64_t)c * kIdxDim);
    const float2 lo = __half22float2(row[lane]);        // dims 2l, 2l+1
    const float2 hi = __half22float2(row[32 + lane]);   // dims 64+2l, 64+2l+1
    a0 += lo.x; a1 += lo.y; b0 += hi.x; b1 += hi.y;
    ++present;
  }
  float* out = pooled + (int64_t)slot * kIdxDim;
  if (present == 0) {
    reinterpret_cast<float2*>(out)[lane] = make_float2(0.f, 0.f);
    reinterpret_cast<float2*>(out)[32 + lane] = make_float2(0.f, 0.f);
    return;
  }
  const double inv_c = (double)present;
  a0 /= inv_c; a1 /= inv_c; b0 /= inv_c; b1 /= inv_c;

  // RMSNorm over the 128 dims.
  double ss = a0 * a0 + a1 * a1 + b0 * b0 + b1 * b1;
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
  const double den = sqrt(ss / (double)kIdxDim + eps);
  const float2 wlo = reinterpret_cast<const float2*>(norm_w)[lane];
  const float2 whi = reinterpret_cast<const float2*>(norm_w)[32 + lane];
  const double x0 = a0 / den * (double)wlo.x, x1 = a1 / den * (double)wlo.y;
  const double y0 = b0 / den * (double)whi.x, y1 = b1 / den * (double)whi.y;

  // NeoX RoPE at the block's first position j*r: pair (d, d+64) turns by
  // pos * theta^(-2d/128).
  const double pos = (double)slot_block_idx[slot] * (double)r;
  float s0, c0, s1, c1;
  sincos_reduced(pos * inv_freq.f[2 * lane], &s0, &c0);
  sincos_reduced(pos * inv_freq.f[2 * lane + 1], &s1, &c1);
  reinterpret_cast<float2*>(out)[lane] =
      make_float2((float)(x0 * c0 - y0 * s0), (float)(x1 * c1 - y1 * s1));
  reinterpret_cast<float2*>(out)[32 + lane] =
      make_float2((float)(y0 * c0 + x0 * s0), (float)(y1 * c1 + x1 * s1));
}

}  // namespace

cudaError_t launch_pool_update(const qsa_config& cfg, const __half* idx_k, int64_t n_cells,
                               const int32_t* blk_cells, const int32_t* slot_block_idx,
                               int64_t n_slots, const int32_t* dirty, int n_dirty,
                               const float* norm_w, float* pooled, unsigned* err,
                               cudaStream_t stream) {
  if (n_dirty <= 0) return cudaSuccess;
  const unsigned blocks = (unsigned)ceil_div(n_dirty, kPoolWarps);
  InvFreq inv{};
  for (int d = 0; d < kIdxDim / 2; ++d)
    inv.f[d] = std::pow((double)cfg.rope_theta, (-2.0 * (double)d) / (double)kIdxDim);
  prof_before(kKPool, stream);
  k_pool_update<<<blocks, kPoolWarps * 32, 0, stream>>>(
      idx_k, n_cells, blk_cells, slot_block_idx, n_slots, dirty, n_dirty, norm_w, pooled,
      cfg.compress_ratio, inv, (double)cfg.rms_eps, err);
  prof_after(kKPool, stream);
  return cudaGetLastError();
}

}  // namespace qsa
