// Append of the step's new cells: K/V rows (fp16 copy or q8_0 encoding),
// indexer keys, block-table entries, and the list of blocks this dirties.
//
// llama.cpp issue #28734 ("decode slows linearly with context"), fix summary:
// lever2b keeps each block's member cells on the device; lever2 re-pools only
// the blocks an ubatch dirtied, their count bucketed to a power of two so a
// captured graph keeps its shape.  Here the dirtied blocks are found on the
// device from the appended positions, so a step needs no host round trip
// between writing its cells and re-pooling their blocks.  q8_0 (the author's
// q8-compact follow-up; README section 1 runs a q8_0 K/V cache): blocks of 32
// values, scale d = max|x| / 127 stored as fp16, codes x * (1/d) rounded half
// away from zero, all in fp32.
//
// One warp per (token, row): rows 0..G-1 are the K heads, G..2G-1 the V
// heads, 2G the indexer key together with the table entry; that warp of each
// block's first new token then re-pools the block.  An extra last CTA builds
// the dirty list: the distinct slots, ascending, padded with -1.
// Everything is read and encoded before the grid-dependency wait (the new
// rows are inputs, not outputs of the preceding kernel); only the stores wait.
#include <climits>

#include "pool_row.cuh"

QSA_TS_DECLARE(append)

namespace qsa {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kAppThreads = 256;
constexpr int kAppOffCache = 256;   // sequences whose block offsets a CTA preloads
constexpr int kAppWarps = kAppThreads / 32;

struct AppendArgs {
  int n_new;
  int G;
  int r;
  int kv_q8;
  const int32_t* tok_seq;
  const int32_t* tok_pos;
  const int32_t* cell;
  const __half* k_new;
  const __half* v_new;
  const __half* idx_new;
  unsigned char* k_cache;
  unsigned char* v_cache;
  __half* idx_k;
  int64_t n_cells;
  int32_t* blk_cells;
  int64_t n_slots;
  const int64_t* seq_blk_off;
  const int32_t* seq_blk_slots;
  int n_seq;
  int32_t* dirty;
  int n_dirty;
  // re-pooling of the dirtied blocks in the same launch (pooled == nullptr: off)
  const int32_t* slot_block_idx;
  const float* norm_w;
  float* pooled;
  float eps;
};

// A new token's sequence, position and cell.
struct NewTok {
  int s, p, c;
};
__device__ __forceinline__ NewTok load_tok(const AppendArgs& a, int t) { return {a.tok_seq[t], a.tok_pos[t], a.cell[t]}; }

// Slot of the block holding a token's position, or -1 when any index is out
// of range (flagged when `report`); s_off: the preloaded block offsets or null.
__device__ __forceinline__ int token_slot(const AppendArgs& a, NewTok k, const int64_t* s_off, int* in_block,
                                          unsigned* err, bool report) {
  const int s = k.s, p = k.p, c = k.c;
  if (s < 0 || s >= a.n_seq || p < 0) {
    if (report) atomicOr(err, kErrToken);
    return -1;
  }
  if (c < 0 || c >= a.n_cells) {
    if (report) atomicOr(err, kErrCell);
    return -1;
  }
  const int64_t off = s_off ? s_off[s] : a.seq_blk_off[s];
  const int64_t len = (s_off ? s_off[s + 1] : a.seq_blk_off[s + 1]) - off;
  const int64_t j = p / a.r;
  if (j >= len) {
    if (report) atomicOr(err, kErrBlockList);
    return -1;
  }
  const int slot = a.seq_blk_slots[off + j];
  if (slot < 0 || slot >= a.n_slots) {
    if (report) atomicOr(err, kErrSlot);
    return -1;
  }
  *in_block = p - (int)j * a.r;
  return slot;
}

__global__ void __launch_bounds__(kAppThreads)
k_append(const AppendArgs a, const Turns turns, unsigned* err) {
  QSA_TS_SCOPE_LAST(append, 1);
  QSA_TS(append, 0);
  // The successor may launch at once: the index kernels read nothing this
  // launch writes before their own dependency wait (see qsa_internal.cuh).
  grid_dep_launch();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kPer = kAppendMaxTokens / kAppThreads;   // tokens per thread in the dirty-list CTA
  const bool dirty_cta = blockIdx.x == gridDim.x - 1;
  // this thread's tokens' ids, loaded together with the sequences' block
  // offsets (one dependent load less on the way to the slots)
  const int rows = 2 * a.G + 1;
  const int64_t w = (int64_t)blockIdx.x * kAppWarps + warp;
  const bool active = !dirty_cta && w < (int64_t)a.n_new * rows;
  const int t = active ? (int)(w / rows) : 0;
  NewTok mine[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int u = dirty_cta ? tid + k * kAppThreads : t;
    mine[k] = ((dirty_cta && u < a.n_new) || (!dirty_cta && k == 0 && active)) ? load_tok(a, u) : NewTok{-1, -1, -1};
  }
  __shared__ int64_t s_off_buf[kAppOffCache + 1];
  const int64_t* s_off = nullptr;
  if (a.n_seq <= kAppOffCache) {
    for (int i = tid; i <= a.n_seq; i += kAppThreads) s_off_buf[i] = a.seq_blk_off[i];
    s_off = s_off_buf;
  }
  // every new token's sequence and position, for the re-pool's scan of the
  // tokens sharing a block (inputs: read before the dependency wait)
  __shared__ int s_tseq[kAppendMaxTokens], s_tpos[kAppendMaxTokens];
  for (int u = tid; u < a.n_new; u += kAppThreads) {
    s_tseq[u] = a.tok_seq[u];
    s_tpos[u] = a.tok_pos[u];
  }
  __syncthreads();
  if (dirty_cta) {
    // ---- the dirty list (n_new <= kAppendMaxTokens): every token's slot
    // (INT_MAX for an invalid token and past n_new), a bitonic sort of the
    // next power of two >= n_new, then the first of every run of equal slots
    // compacted in order: the distinct slots, ascending
    __shared__ int s_slot[kAppendMaxTokens];
    __shared__ unsigned s_warp[kAppWarps];
    int n2 = 2;
    while (n2 < a.n_new) n2 <<= 1;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int u = tid + k * kAppThreads;
      if (u >= n2) break;
      int sl = INT_MAX;
      if (u < a.n_new) {
        int ib = 0;
        const int x = token_slot(a, mine[k], s_off, &ib, err, false);
        sl = x < 0 ? INT_MAX : x;
      }
      s_slot[u] = sl;
    }
    __syncthreads();
    for (int k = 2; k <= n2; k <<= 1) {
      for (int j = k >> 1; j > 0; j >>= 1) {
        for (int i = tid; i < n2; i += kAppThreads) {
          const int l = i ^ j;
          if (l > i) {
            const int x = s_slot[i], y = s_slot[l];
            if ((x > y) == ((i & k) == 0)) {
              s_slot[i] = y;
              s_slot[l] = x;
            }
          }
        }
        __syncthreads();
      }
    }
    // thread tid takes the contiguous run [tid * per, tid * per + per)
    const int per = (n2 + kAppThreads - 1) / kAppThreads;   // <= 4
    const int i0 = min(n2, tid * per), i1 = min(n2, i0 + per);
    unsigned mine_n = 0;
    for (int i = i0; i < i1; ++i)
      mine_n += (s_slot[i] != INT_MAX && (i == 0 || s_slot[i] != s_slot[i - 1])) ? 1u : 0u;
    unsigned incl = mine_n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned y = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    unsigned at = incl - mine_n, n_lead = 0;
    for (int w2 = 0; w2 < kAppWarps; ++w2) {
      if (w2 < warp) at += s_warp[w2];
      n_lead += s_warp[w2];
    }
    grid_dep_wait();
    QSA_TS_IF(append, 2, tid == 0);
    for (int i = i0; i < i1; ++i) {
      const int sl = s_slot[i];
      if (sl != INT_MAX && (i == 0 || sl != s_slot[i - 1])) {
        if (at < (unsigned)a.n_dirty) a.dirty[at] = sl;
        ++at;
      }
    }
    for (int i = (int)n_lead + tid; i < a.n_dirty; i += kAppThreads) a.dirty[i] = -1;
    return;
  }

  // ---- one warp per (token, row)
  const int kind = active ? (int)(w - (int64_t)t * rows) : 0;
  int ib = 0;
  const int slot = active ? token_slot(a, mine[0], s_off, &ib, err, kind == 2 * a.G && lane == 0) : -1;
  const int64_t c = active ? mine[0].c : 0;
  const bool ok = active && slot >= 0;

  if (kind < 2 * a.G) {
    const int g = kind < a.G ? kind : kind - a.G;
    const __half* src = (kind < a.G ? a.k_new : a.v_new) + ((int64_t)t * a.G + g) * kHeadDim;
    unsigned char* cache = kind < a.G ? a.k_cache : a.v_cache;
    const uint4 raw = ok ? __ldg(reinterpret_cast<const uint4*>(src) + lane) : make_uint4(0, 0, 0, 0);
    if (!a.kv_q8) {
      grid_dep_wait();
      if (ok) reinterpret_cast<uint4*>(cache + (c * a.G + g) * kHeadDim * 2)[lane] = raw;
      return;
    }
    // q8_0: lanes 4b..4b+3 hold the 32 values of block b
    const __half2* h = reinterpret_cast<const __half2*>(&raw);
    float x[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __half22float2(h[i]);
      x[2 * i] = f.x;
      x[2 * i + 1] = f.y;
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
    amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
    const float d = amax / 127.0f;
    const float inv = d != 0.f ? 1.0f / d : 0.f;
    uint2 qs;
    signed char* qb = reinterpret_cast<signed char*>(&qs);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float v = x[i] * inv;
      // half away from zero, exactly: |v| - trunc(|v|) is exact in fp32,
      // while floor(|v| + 0.5) would round 0.5 - 2^-25 up to 1
      const float av = fabsf(v);
      float m = truncf(av);
      if (av - m >= 0.5f) m += 1.0f;
      m = fminf(m, 127.f);
      qb[i] = (signed char)(v < 0.f ? -(int)m : (int)m);
    }
    grid_dep_wait();
    if (ok) {
      reinterpret_cast<uint2*>(cache + (c * a.G + g) * kHeadDim)[lane] = qs;
      if ((lane & 3) == 0) {
        __half* sc = reinterpret_cast<__half*>(cache + a.n_cells * (int64_t)a.G * kHeadDim);
        sc[(c * a.G + g) * (kHeadDim / 32) + (lane >> 2)] = __float2half_rn(d);
      }
    }
    return;
  }
  // indexer key row (256 bytes: lanes 0..15) and the table entry
  uint4 raw = make_uint4(0, 0, 0, 0);
  if (ok && lane < 16) raw = __ldg(reinterpret_cast<const uint4*>(a.idx_new + (int64_t)t * kIdxDim) + lane);
  grid_dep_wait();
  if (!ok) return;
  if (lane < 16) reinterpret_cast<uint4*>(a.idx_k + c * kIdxDim)[lane] = raw;
  if (lane == 0) a.blk_cells[(int64_t)slot * a.r + ib] = (int32_t)c;
  if (a.pooled == nullptr) return;

  // ---- re-pool this token's block (as qsa_pool_update would after this
  // launch) if this is the block's first new token: the warps of all tokens
  // re-pool their blocks in parallel.  Members come from the table, except
  // the positions this launch appends, whose cells and keys come from the
  // inputs (other warps of this launch are writing them).  One pass over the
  // new tokens, 32 at a time, finds both.
  const int r = a.r;
  const int64_t jb = (int64_t)mine[0].p / r;
  int tn = -1;            // lane i < r: the new token at position jb * r + i
  bool earlier = false;   // a token before this one falls in the same block
  for (int u0 = 0; u0 < a.n_new; u0 += 32) {
    const int u = u0 + lane;
    bool hit = false;
    int pos_in = 0;
    if (u < a.n_new) {
      const int su = s_tseq[u], pu = s_tpos[u];
      hit = su == mine[0].s && pu >= 0 && (int64_t)pu / r == jb;
      pos_in = pu - (int)(jb * r);
    }
    earlier |= __any_sync(kFull, hit && u < t);
    unsigned m = __ballot_sync(kFull, hit);
    while (m) {
      const int src = __ffs(m) - 1;
      m &= m - 1u;
      const int at = __shfl_sync(kFull, pos_in, src);
      if (lane == at) tn = u0 + src;
    }
  }
  if (earlier) return;
  int mcell = -1;
  if (lane < r) mcell = tn >= 0 ? a.cell[tn] : a.blk_cells[(int64_t)slot * r + lane];
  int cell[kMaxR], tnew[kMaxR];
#pragma unroll
  for (int i = 0; i < kMaxR; ++i) {
    cell[i] = __shfl_sync(kFull, mcell, i);
    tnew[i] = __shfl_sync(kFull, tn, i);
    if (i >= r) cell[i] = -1;
  }
  const int blk = a.slot_block_idx[slot];
  float2 lo[kMaxR], hi[kMaxR];
  bool present[kMaxR];
#pragma unroll
  for (int i = 0; i < kMaxR; ++i) {
    const bool pok = cell[i] >= 0 && cell[i] < a.n_cells;
    if (cell[i] >= a.n_cells && lane == 0) atomicOr(err, kErrCell);
    const __half* src = (i < r && tnew[i] >= 0) ? a.idx_new + (int64_t)tnew[i] * kIdxDim
                                                : a.idx_k + (int64_t)(pok ? cell[i] : 0) * kIdxDim;
    const __half2* row = reinterpret_cast<const __half2*>(src);
    lo[i] = pok ? __half22float2(row[lane]) : make_float2(0.f, 0.f);
    hi[i] = pok ? __half22float2(row[32 + lane]) : make_float2(0.f, 0.f);
    present[i] = pok;
  }
  float2 olo, ohi;
  pool_rows_warp(lo, hi, present, blk, r, a.norm_w, turns, a.eps, &olo, &ohi);
  float* out = a.pooled + (int64_t)slot * kIdxDim;
  reinterpret_cast<float2*>(out)[lane] = olo;
  reinterpret_cast<float2*>(out)[32 + lane] = ohi;
}

}  // namespace

cudaError_t launch_append(const qsa_config& cfg, int n_new, const int32_t* tok_seq, const int32_t* tok_pos,
                          const int32_t* cell, const __half* k_new, const __half* v_new, const __half* idx_new,
                          void* k_cache, void* v_cache, __half* idx_k, int64_t n_cells, int32_t* blk_cells,
                          int64_t n_slots, const int64_t* seq_blk_off, const int32_t* seq_blk_slots, int n_seq,
                          int32_t* dirty, int n_dirty, const int32_t* slot_block_idx, const float* norm_w,
                          float* pooled, unsigned* err, cudaStream_t stream) {
  if (n_new <= 0) return cudaSuccess;
  AppendArgs a{};
  a.n_new = n_new;
  a.G = cfg.n_kv_heads;
  a.r = cfg.compress_ratio;
  a.kv_q8 = cfg.kv_type == QSA_KV_Q8_0;
  a.tok_seq = tok_seq;
  a.tok_pos = tok_pos;
  a.cell = cell;
  a.k_new = k_new;
  a.v_new = v_new;
  a.idx_new = idx_new;
  a.k_cache = static_cast<unsigned char*>(k_cache);
  a.v_cache = static_cast<unsigned char*>(v_cache);
  a.idx_k = idx_k;
  a.n_cells = n_cells;
  a.blk_cells = blk_cells;
  a.n_slots = n_slots;
  a.seq_blk_off = seq_blk_off;
  a.seq_blk_slots = seq_blk_slots;
  a.n_seq = n_seq;
  a.dirty = dirty;
  a.n_dirty = n_dirty;
  a.slot_block_idx = slot_block_idx;
  a.norm_w = norm_w;
  a.pooled = pooled;
  a.eps = cfg.rms_eps;
  const Turns turns = make_turns(cfg.rope_theta);
  const int64_t warps = (int64_t)n_new * (2 * cfg.n_kv_heads + 1);
  const unsigned blocks = (unsigned)ceil_div(warps, kAppWarps) + 1;   // + the dirty-list CTA
  prof_before(kKAppend, stream);
  cudaError_t e = launch_pdl(k_append, dim3(blocks), dim3(kAppThreads), 0, stream, 1, a, turns, err);
  prof_after(kKAppend, stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace qsa
