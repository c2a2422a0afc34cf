// S1: persistent pooled block-key cache update.
//
// llama.cpp issue #28734 ("decode slows linearly with context"), fix summary,
// lever2: the indexer used to re-gather, mean-pool, RMS-norm and re-RoPE every
// cached block each token; a persistent buffer of pooled block keys is kept
// instead and only the blocks an ubatch dirtied are recomputed.  lever2b: the
// member cells of each block stay on the device (blk_cells).
//
// One warp per dirty slot; the row arithmetic is pool_rows_warp (pool_row.cuh).
// All member cells are read first and all their key rows next (two dependent
// loads in all).
#include "pool_row.cuh"

QSA_TS_DECLARE(pool)

namespace qsa {
namespace {

constexpr int kPoolWarps = 4;
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
  bool present[kMaxR];
#pragma unroll
  for (int i = 0; i < kMaxR; ++i) present[i] = cell[i] >= 0;
  float2 olo, ohi;
  pool_rows_warp(lo, hi, present, blk, r, norm_w, turns, eps, &olo, &ohi);
  QSA_TS(pool, 3);
  float* out = pooled + (int64_t)slot * kIdxDim;
  reinterpret_cast<float2*>(out)[lane] = olo;
  reinterpret_cast<float2*>(out)[32 + lane] = ohi;
}

}  // namespace

cudaError_t launch_pool_update(const qsa_config& cfg, const __half* idx_k, int64_t n_cells,
                               const int32_t* blk_cells, const int32_t* slot_block_idx,
                               int64_t n_slots, const int32_t* dirty, int n_dirty,
                               const float* norm_w, float* pooled, unsigned* err,
                               cudaStream_t stream) {
  if (n_dirty <= 0) return cudaSuccess;
  const unsigned blocks = (unsigned)ceil_div(n_dirty, kPoolWarps);
  const Turns turns = make_turns(cfg.rope_theta);
  prof_before(kKPool, stream);
  cudaError_t e = launch_pdl(k_pool_update, dim3(blocks), dim3(kPoolWarps * 32), 0, stream, 1, idx_k, n_cells,
                             blk_cells, slot_block_idx, n_slots, dirty, n_dirty, norm_w, pooled,
                             cfg.compress_ratio, turns, cfg.rms_eps, err);
  prof_after(kKPool, stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace qsa
