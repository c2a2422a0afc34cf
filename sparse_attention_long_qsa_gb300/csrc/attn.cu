// S5 + S6: sparse flash-decode over the selected cells, on 5th-generation
// tensor cores (tcgen05, accumulators in tensor memory), one thread-block
// cluster per (token, KV head).
//
// llama.cpp issue #28734 ("decode slows linearly with context"), fix summary,
// lever1: attention runs over only the top-k K/V set, so its cost is O(top_k)
// instead of O(n_kv); sparse256: the head shape is DKQ = DV = 256 with 8 query
// heads per KV head (ncols2 = 8).  The author's q8-compact follow-up keeps the
// sparse path for a q8_0 cache; here q8_0 rows are dequantised after the
// gather, so the whole cache is never converted (the O(n_kv) to_fp16 pass
// goodbadwolf's comment in the same issue points at).  The API is indices-in:
// no mask is built or re-scanned.
//
// Work split.  The token's cell list is cut into tiles of 128 cells; the
// cluster's CTA r takes tiles r, r + NC, ... (NC = cluster size <= 16).  Per
// tile a CTA
//   1. gathers the 128 K rows and V rows of its KV head into shared memory in
//      the 128-byte-swizzled canonical layout (16-byte cp.async for fp16; for
//      q8_0 int8 rows + scales through registers, dequantised to fp16),
//   2. S = K . Q^T with M = 128 cells, N = 16 (8 query heads + 8 zero rows),
//      K = 256: 16 tcgen05.mma into tensor memory,
//   3. reads S back (one cell per thread of warps 0-3), masks, takes the tile
//      softmax statistics per head and writes P (fp16) to shared memory,
//   4. O^T = V^T . P^T with M = 128 dims (two halves), N = 16, K = 128 cells:
//      16 tcgen05.mma (V is the MN-major operand of the same swizzled tile),
//   5. merges the tile into a running (max, sum, o) in registers.
// When a CTA takes several fp16 tiles, warps 4-7 gather them into three
// rotating K/V stages ahead of warps 0-3, which run steps 2-5 (full/empty
// mbarriers between the two groups); several q8_0 tiles load the next
// tile's rows into registers under this tile's steps 2-5.
// Then every CTA stores its (max, sum, o) slices straight into the shared
// memory of the CTA owning each range of dims (distributed shared memory), the
// cluster synchronises once, and CTA r reduces dims [r*256/NC, ...) over all
// NC partials from its own shared memory (log-sum-exp weights) and writes the
// fp32 output.  No partials go to global memory and no second kernel runs.
//
// Waits on the MMA completion and stage barriers are bounded: on timeout the CTA records
// an error bit and keeps going through every barrier (its output is then
// meaningless but nothing hangs).
#include <atomic>
#include <cstring>
#include <mutex>

#include "attn_pf.cuh"
#include "attn_util.cuh"
#include "index_util.cuh"
#include "qsa_internal.cuh"
#include "tc_util.cuh"

QSA_TS_DECLARE(attn)

namespace qsa {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kThreads = 256;
constexpr int kTile = 128;          // cells per MMA tile (M of the QK product)
constexpr int kMaxCluster = 16;
constexpr uint32_t kTmemCols = 64;  // S: cols [0,16); O half 0: [16,32); O half 1: [32,48)

// ---- shared-memory layout (offsets from a 1024-byte aligned base)
constexpr uint32_t kOffK = 0;                       // 128 rows x 512 B, 4 column atoms of 16 KB
constexpr uint32_t kOffV = kOffK + kTile * 512;     // same layout
constexpr uint32_t kOffQ = kOffV + kTile * 512;     // 16 rows x 512 B, 4 atoms of 2 KB
constexpr uint32_t kOffP = kOffQ + 16 * 512;        // 16 rows x 256 B, 2 atoms of 2 KB
constexpr uint32_t kOffO = kOffP + 16 * 256;        // fp32 [NC][8][256/NC] partials pushed by the cluster
constexpr uint32_t kOffM = kOffO + 8 * 256 * 4;     // fp32 [NC][16] their (max[8], sum[8])
constexpr uint32_t kOffRed = kOffM + 16 * 16 * 4;   // fp32 [2][4][8] cross-warp reductions
constexpr uint32_t kOffCell = kOffRed + 256;        // int [128]
constexpr uint32_t kOffBar = kOffCell + kTile * 4;  // u64 mbarrier
constexpr uint32_t kOffTmem = kOffBar + 8;          // u32 TMEM base address
// overflow cells (past NC full tiles, at most kOvf) on CUDA cores, warps 4-7
constexpr int kOvf = 32;
constexpr uint32_t kOffXK = kOffTmem + 8;           // fp16 [kOvf][256] K rows
constexpr uint32_t kOffXV = kOffXK + kOvf * 512;    // fp16 [kOvf][256] V rows
constexpr uint32_t kOffXS = kOffXV + kOvf * 512;    // fp32 [kOvf][8] scores / probabilities
constexpr uint32_t kOffXO = kOffXS + kOvf * 8 * 4;  // fp32 [8][256] partial output
constexpr uint32_t kOffXM = kOffXO + 8 * 256 * 4;   // fp32 [8] max, [8] sum
constexpr uint32_t kOffXC = kOffXM + 64;            // int [kOvf] cells
constexpr uint32_t kOffCellN = kOffXC + kOvf * 4;   // int [128] the next tile's cells (q8_0, several tiles)
constexpr uint32_t kSmemBytes = kOffCellN + kTile * 4 + 1024;   // + alignment slack

// ---- the selection run by the attention clusters (kSel variants)
constexpr int kFusedMaxList = 1024;                  // chosen blocks (top_k / r)
constexpr int kFusedMaxTiles = 8;                    // 128-cell tiles per CTA
constexpr int kFusedMaxWords = 2048;                 // bitmap words of CTA 0: 65,536 blocks
constexpr int kFusedMaxBlocks = kFusedMaxWords * 32;
constexpr int kFusedRankMax = 1024;                  // threshold-bin keys resolved in CTA 0
constexpr int kFusedSlots = 8192;                    // slot ids a CTA keeps for its range
constexpr int kFusedBatch = 16;                      // score words a warp loads before using any

struct SelArgs {
  IndexArgs ia;
  void* ws;          // the qsa_index_topk workspace (histograms, scores)
  int32_t* cells;    // outputs of the selection (written by the KV-head-0 clusters)
  int32_t* count;
};

// Selection state that lives through the whole kernel (after the attention
// layout).  `list`, `nsel`, `count` and `tail_cells` are CTA 0's, read by the
// peers through distributed shared memory.
struct SelFix {
  int list[kFusedMaxList];                   // slots of the chosen blocks, ascending block index
  int mycells[kFusedMaxTiles * kTile];       // this CTA's tiles' cells, tile-major
  int tail_cells[8];
  unsigned warp_tmp[8];
  unsigned ncand, ncent, ncut, sel, cbase;
  int thr, need, ncand_all, digit;
  unsigned above, eq;
  int nsel, count, last;
};
// Scratch of the selection, in the K and V tiles (free until the gather).
struct SelScratch {
  unsigned bitmap[kFusedMaxWords];           // CTA 0: every block; peers: their range
  unsigned long long cand[kFusedRankMax];    // this CTA's threshold-bin keys
  unsigned long long allc[kFusedRankMax];    // CTA 0: every CTA's threshold-bin keys
  unsigned hist[2][256];
  unsigned tot[256];
  int slots[kFusedSlots + 4];                // slot ids of this CTA's range
};
static_assert(sizeof(SelScratch) <= 2u * kTile * 512u, "selection scratch fits in the K and V tiles");
constexpr uint32_t kOffFix = (kOffCellN + kTile * 4 + 15u) & ~15u;
constexpr uint32_t kSmemBytesSel = kOffFix + (uint32_t)sizeof(SelFix) + 1024;
static_assert(kSmemBytesSel <= 227u * 1024u, "shared memory of the fused variant");

// fp16 with several tiles per CTA (the pipelined variant, no overflow
// cells): a third 64 KB row stage over the overflow buffers, two more cell
// lists and the stages' full and empty barriers.
constexpr uint32_t kOffX3 = (kOffTmem + 8 + 1023u) & ~1023u;
constexpr uint32_t kOffCell2 = kOffX3 + kTile * 512;
constexpr uint32_t kOffCell3 = kOffCell2 + kTile * 4;
constexpr uint32_t kOffPipeBar = kOffCell3 + kTile * 4;   // u64 full[3], empty[3]
constexpr uint32_t kSmemBytesPipe16 = kOffPipeBar + 6 * 8 + 1024;
static_assert(kSmemBytesPipe16 <= 227u * 1024u, "shared memory of the pipelined fp16 variant");

template <bool kSel>
constexpr uint32_t smem_bytes() { return kSel ? kSmemBytesSel : kSmemBytes; }
template <bool kQ8, bool kPipe, bool kSel>
constexpr uint32_t smem_bytes_of() { return (!kQ8 && kPipe && !kSel) ? kSmemBytesPipe16 : smem_bytes<kSel>(); }

__device__ __forceinline__ void arrive_cta(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}

// Instruction descriptor, kind::f16: fp32 accumulate, fp16 A and B,
// M = 128, N = 16; A K-major (QK) or MN-major (PV), B K-major.
constexpr uint32_t kIdescQK = (1u << 4) | ((16u >> 3) << 17) | ((128u >> 4) << 24);
constexpr uint32_t kIdescPV = kIdescQK | (1u << 15);

// Geometry of the fused selection for this CTA: the token's blocks are split
// into NC ranges of `per` blocks (a multiple of 32), one per CTA.
struct SelGeom {
  Tok tk;
  int nb;          // blocks that compete
  int64_t per, j0, j1;
  int nwords;      // bitmap words of this CTA's range
  int tail;        // tail cells (positions past the last whole block, <= p)
  bool tail_missing;
};

__device__ __forceinline__ SelGeom sel_geometry(const IndexArgs& ia, int t, uint32_t rank, uint32_t NC,
                                                unsigned* err) {
  SelGeom s;
  s.tk = token_geometry(ia, t, err, false);
  s.nb = s.tk.nb;
  s.per = round_up(ceil_div(s.nb > 0 ? s.nb : 1, (int64_t)NC), 32);
  s.j0 = (int64_t)rank * s.per;
  s.j1 = min((int64_t)s.nb, s.j0 + s.per);
  s.nwords = s.j1 > s.j0 ? (int)ceil_div(s.j1 - s.j0, 32) : 0;
  s.tail = 0;
  if (s.tk.ok && s.tk.nb == s.tk.nb_full) s.tail = s.tk.p + 1 - (int)(s.tk.nb_full * ia.r);
  s.tail_missing = s.tail > 0 && s.tk.nb_full >= s.tk.len;
  if (s.tail_missing) s.tail = 0;
  return s;
}

// Block selection and expansion of token t by the CTAs of one cluster (the
// method's lever3 steps, as k_select in index.cu runs them, here inside the
// attention clusters so that no kernel boundary and no global cell list sit
// between the selection and the gather).  Every cluster of the token (one per
// KV head) computes the same selection; the KV-head-0 cluster writes the
// cells and count outputs.  Steps:
//   1. the threshold bin of the B-th largest score from the token's
//      histogram (every CTA);
//   2. each CTA classifies its range: blocks above the bin into a bitmap,
//      blocks in the bin into unique 56-bit keys (ties to the lower index);
//   3a. (bin <= kFusedRankMax keys) the CTAs push bitmap words and keys into
//      CTA 0, which ranks the keys of the cut-off digit exactly and lists the
//      chosen blocks' slots in block order;
//   3b. (larger bins) a radix select over the bin's keys, one 8-bit digit per
//      round with cluster-summed digit histograms, after which each CTA
//      writes its chosen blocks' slots at its offset in CTA 0's list;
//   4. every CTA expands the list positions of its own attention tiles
//      (slot -> the block's member cells; then the tail cells).
// Returns the token's cell count; this CTA's cells are in fx->mycells.
__device__ __forceinline__ int select_in_cluster(const SelArgs& sa, const SelGeom& sg, int cells_pitch, int t,
                                                 int g, int G, uint32_t rank, uint32_t NC, SelFix* fx,
                                                 SelScratch* sx, unsigned* err) {
  const IndexArgs& ia = sa.ia;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kWarps = kThreads / 32;
  const int r = ia.r, B = ia.n_sel_blocks;
  const int nb = sg.nb, nwords = sg.nwords, tail = sg.tail;
  const int64_t j0 = sg.j0, j1 = sg.j1, per = sg.per;
  const int32_t* slots = ia.seq_blk_slots + sg.tk.off;
  unsigned* gh = hist_of(sa.ws, t);
  const float* srow = scores_of(sa.ws, ia.max_tokens) + (int64_t)t * ia.max_blocks;

  // ---- 1. first scores in flight; the threshold bin (16 bins per thread)
  float v0[kFusedBatch];
#pragma unroll
  for (int b = 0; b < kFusedBatch; ++b) {
    const int w = warp + kWarps * b;
    const int64_t j = j0 + (int64_t)w * 32 + lane;
    v0[b] = (w < nwords && j < j1) ? __ldcg(srow + j) : -INFINITY;
  }
  const int tslot = (rank == 0 && tid < tail) ? slots[sg.tk.nb_full] : -1;
  {
    constexpr int kPer = kHistBins / kThreads;
    static_assert(kPer == 16, "histogram split");
    unsigned h[kPer];
    unsigned sum = 0;
#pragma unroll
    for (int q = 0; q < kPer / 4; ++q) {
      const uint4 v = __ldcg(reinterpret_cast<const uint4*>(gh + tid * kPer) + q);
      h[4 * q] = v.x, h[4 * q + 1] = v.y, h[4 * q + 2] = v.z, h[4 * q + 3] = v.w;
    }
#pragma unroll
    for (int i = 0; i < kPer; ++i) sum += h[i];
    if (tid == 0) {
      fx->thr = -1;
      fx->need = 0;
      fx->ncand_all = 0;
    }
    unsigned cum = block_suffix_exclusive(sum, fx->warp_tmp);
    const unsigned Bu = (unsigned)B;
    if ((unsigned)nb > Bu) {
#pragma unroll
      for (int i = kPer - 1; i >= 0; --i) {
        const unsigned nxt = cum + h[i];
        if (cum < Bu && nxt >= Bu) {
          fx->thr = tid * kPer + i;
          fx->need = (int)(Bu - cum);
          fx->ncand_all = (int)h[i];
        }
        cum = nxt;
      }
    }
    __syncthreads();
  }
  // This CTA has read the histogram.  The last of the token's G x NC readers
  // clears it for the next call (before this kernel lets its successor start).
  if (tid == 0) fx->last = atomicAdd(readers_of(sa.ws, t), 1u) == (unsigned)(G * (int)NC) - 1u ? 1 : 0;
  const int thr = fx->thr, ncand_all = fx->ncand_all;
  const bool central = thr < 0 || ncand_all <= kFusedRankMax;
  if (rank == 0 && tid < tail) {
    if (tslot >= 0 && tslot < ia.n_slots) {
      cp_async4(&fx->tail_cells[tid], ia.blk_cells + (int64_t)tslot * r + tid);
    } else {
      atomicOr(err, kErrSlot);
      fx->tail_cells[tid] = -1;
    }
  }
  QSA_TS(attn, 18);

  // ---- 2. classify this CTA's blocks (words dealt round-robin to the warps)
  for (int wb = 0; wb * kWarps * kFusedBatch < nwords; ++wb) {
    const int wbase = wb * kWarps * kFusedBatch + warp;
    float v[kFusedBatch];
#pragma unroll
    for (int b = 0; b < kFusedBatch; ++b) {
      const int w = wbase + kWarps * b;
      const int64_t j = j0 + (int64_t)w * 32 + lane;
      v[b] = (wb == 0) ? v0[b] : ((w < nwords && j < j1) ? __ldcg(srow + j) : -INFINITY);
    }
#pragma unroll
    for (int b = 0; b < kFusedBatch; ++b) {
      const int w = wbase + kWarps * b;
      if (w >= nwords) break;
      const int64_t j = j0 + (int64_t)w * 32 + lane;
      const bool in = j < j1;
      const uint32_t key = score_key(v[b]);
      const int bin = (int)(key >> (32 - kHistBits));
      const unsigned am = __ballot_sync(kFull, in && bin > thr);
      if (lane == 0) sx->bitmap[w] = am;
      if (central && thr >= 0) {
        const bool isc = in && bin == thr;
        const unsigned cm = __ballot_sync(kFull, isc);
        if (cm) {
          const int leader = __ffs(cm) - 1;
          unsigned basei = 0;
          if (lane == leader) basei = atomicAdd(&fx->ncand, (unsigned)__popc(cm));
          basei = __shfl_sync(kFull, basei, leader);
          const unsigned idx = basei + __popc(cm & ((1u << lane) - 1u));
          if (isc && idx < (unsigned)kFusedRankMax) sx->cand[idx] = cand_key(key, j);
        }
      }
    }
  }
  // this range's slot ids (CTA 0 reads them through DSMEM to list the chosen
  // blocks): 16-byte copies where the list is aligned, single ids at the ends
  const bool slots_cached = per <= kFusedSlots;
  auto slot_shift = [&](int64_t lo) { return (int)((reinterpret_cast<uintptr_t>(slots + lo) >> 2) & 3); };
  int32_t* my_slots = sx->slots + slot_shift(j0);
  if (slots_cached && j1 > j0) {
    const int64_t n = j1 - j0;
    const int64_t head = min(n, (int64_t)((4 - slot_shift(j0)) & 3));
    const int64_t body = (n - head) / 4;
    if (tid < head) cp_async4(my_slots + tid, slots + j0 + tid);
    for (int64_t q = tid; q < body; q += kThreads) cp_async16_ptr(my_slots + head + 4 * q, slots + j0 + head + 4 * q);
    for (int64_t i = head + 4 * body + tid; i < n; i += kThreads) cp_async4(my_slots + i, slots + j0 + i);
  }
  asm volatile("cp.async.commit_group;\n" ::: "memory");
  __syncthreads();
  QSA_TS(attn, 19);
  // slot of block j (any range): from its owner's shared memory when cached
  auto slot_of = [&](int64_t j) -> int {
    if (!slots_cached) return slots[j];
    const int64_t p = j / per;
    return (int)ld_dsmem_u32(dsmem_addr(sx->slots + slot_shift(p * per) + (j - p * per), (uint32_t)p));
  };

  cluster_wait();   // pairs with the arrive before the dependency wait: every CTA's counters are set
  if (central) {
    // ---- 3a. bitmap words and threshold-bin keys into CTA 0
    if (rank != 0)
      for (int w = tid; w < nwords; w += kThreads)
        st_dsmem_u32(dsmem_addr(&sx->bitmap[(int)(j0 >> 5) + w], 0), sx->bitmap[w]);
    const unsigned ncl = min(fx->ncand, (unsigned)kFusedRankMax);
    if (tid == 0) fx->cbase = ncl ? atom_add_dsmem(dsmem_addr(&fx->ncent, 0), ncl) : 0u;
    __syncthreads();
    for (unsigned i = tid; i < ncl; i += kThreads) {
      const unsigned at = fx->cbase + i;
      if (at < (unsigned)kFusedRankMax) st_dsmem_u64(dsmem_addr(&sx->allc[at], 0), sx->cand[i]);
    }
    asm volatile("cp.async.wait_all;\n" ::: "memory");   // slot ids (and CTA 0's tail cells)
    cluster_sync();   // everything has landed in CTA 0; every range's slot ids are in place
    QSA_TS(attn, 20);
    if (rank == 0) {
      const unsigned nall = min(fx->ncent, (unsigned)kFusedRankMax);
      if (thr >= 0) {
        // one 8-bit digit below the bin (key bits 19..12) splits the keys;
        // keys above the cut-off digit are chosen, the digit's own keys are
        // ranked exactly by full key
        unsigned need = (unsigned)fx->need;
        unsigned* hh = sx->hist[0];
        hh[tid] = 0u;
        __syncthreads();
        for (unsigned i = tid; i < nall; i += kThreads) atomicAdd(&hh[(unsigned)(sx->allc[i] >> 48) & 255u], 1u);
        __syncthreads();
        if (warp == 0) {
          unsigned hv[8], hs = 0;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            hv[i] = hh[lane * 8 + i];
            hs += hv[i];
          }
          unsigned x = hs;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const unsigned y = __shfl_down_sync(kFull, x, o);
            if (lane + o < 32) x += y;
          }
          unsigned cum = x - hs;
#pragma unroll
          for (int i = 7; i >= 0; --i) {
            const unsigned nxt = cum + hv[i];
            if (cum < need && nxt >= need) {
              fx->digit = lane * 8 + i;
              fx->above = cum;
            }
            cum = nxt;
          }
        }
        if (tid == 0) fx->ncut = 0u;
        __syncthreads();
        const unsigned dstar = (unsigned)fx->digit;
        need -= fx->above;
        for (unsigned i = tid; i < nall; i += kThreads) {
          const unsigned long long c = sx->allc[i];
          const unsigned d = (unsigned)(c >> 48) & 255u;
          if (d > dstar) {
            const int64_t j = (int64_t)(~(uint32_t)(c >> 4));
            atomicOr(&sx->bitmap[j >> 5], 1u << (j & 31));
          } else if (d == dstar) {
            sx->cand[atomicAdd(&fx->ncut, 1u)] = c;   // ncut <= nall <= kFusedRankMax
          }
        }
        __syncthreads();
        const unsigned ncut = fx->ncut;
        for (unsigned i = tid; i < ncut; i += kThreads) {
          const unsigned long long c = sx->cand[i];
          unsigned above_c = 0;
          for (unsigned m = 0; m < ncut; ++m) above_c += sx->cand[m] > c ? 1u : 0u;
          if (above_c < need) {
            const int64_t j = (int64_t)(~(uint32_t)(c >> 4));
            atomicOr(&sx->bitmap[j >> 5], 1u << (j & 31));
          }
        }
      }
      __syncthreads();
      // the chosen blocks in order, as slots
      const int W = (int)ceil_div(nb, 32);
      const int wq = (int)ceil_div(W, kThreads);
      const int q0 = tid * wq, q1 = min(W, q0 + wq);
      unsigned mine = 0;
      for (int w = q0; w < q1; ++w) mine += __popc(sx->bitmap[w]);
      unsigned total = 0;
      unsigned k = block_prefix_exclusive(mine, fx->warp_tmp, &total);
      for (int w = q0; w < q1; ++w) {
        unsigned bits = sx->bitmap[w];
        while (bits) {
          if (k < (unsigned)B) fx->list[k] = w * 32 + (__ffs(bits) - 1);
          ++k;
          bits &= bits - 1u;
        }
      }
      const int nsel = (int)min(total, (unsigned)B);
      __syncthreads();
      // block -> slot, the loads of each thread's positions issued together
      constexpr int kPerT = kFusedMaxList / kThreads;
      int sv[kPerT];
#pragma unroll
      for (int q = 0; q < kPerT; ++q) {
        const int i = tid + q * kThreads;
        sv[q] = i < nsel ? slot_of(fx->list[i]) : 0;
      }
#pragma unroll
      for (int q = 0; q < kPerT; ++q) {
        const int i = tid + q * kThreads;
        if (i < nsel) fx->list[i] = sv[q];
      }
      if (tid == 0) {
        fx->nsel = nsel;
        fx->count = nsel * r + tail;
      }
    }
    QSA_TS(attn, 21);
    cluster_sync();   // CTA 0's list is complete
  } else {
    // ---- 3b. radix select over the threshold bin (thr >= 0 here)
    unsigned long long prefix = 0;
    int shift = 48;
    unsigned need = (unsigned)fx->need;
    int buf = 0;
    for (;;) {
      unsigned* hh = sx->hist[buf];
      hh[tid] = 0u;
      __syncthreads();
      for (int64_t j = j0 + tid; j < j1; j += kThreads) {
        const uint32_t key = score_key(__ldcg(srow + j));
        if ((int)(key >> (32 - kHistBits)) != thr) continue;
        const unsigned long long c = cand_key(key, j);
        if ((c >> (shift + 8)) == prefix) atomicAdd(&hh[(unsigned)(c >> shift) & 255u], 1u);
      }
      cluster_sync();
      {
        unsigned sum = 0;
        for (int p = 0; p < (int)NC; ++p) sum += ld_dsmem_u32(dsmem_addr(&hh[tid], (uint32_t)p));
        sx->tot[tid] = sum;
      }
      __syncthreads();
      if (warp == 0) {
        unsigned hv[8], hs = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          hv[i] = sx->tot[lane * 8 + i];
          hs += hv[i];
        }
        unsigned x = hs;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const unsigned y = __shfl_down_sync(kFull, x, o);
          if (lane + o < 32) x += y;
        }
        unsigned cum = x - hs;
#pragma unroll
        for (int i = 7; i >= 0; --i) {
          const unsigned nxt = cum + hv[i];
          if (cum < need && nxt >= need) {
            fx->digit = lane * 8 + i;
            fx->above = cum;
            fx->eq = hv[i];
          }
          cum = nxt;
        }
      }
      __syncthreads();
      need -= fx->above;
      const unsigned eq = fx->eq;
      prefix = (prefix << 8) | (unsigned long long)fx->digit;
      buf ^= 1;
      if (eq == need || shift == 0) break;
      shift -= 8;
    }
    // every key of the bin whose bits down to `shift` are >= prefix is chosen
    for (int64_t j = j0 + tid; j < j1; j += kThreads) {
      const uint32_t key = score_key(__ldcg(srow + j));
      if ((int)(key >> (32 - kHistBits)) != thr) continue;
      if ((cand_key(key, j) >> shift) >= prefix) atomicOr(&sx->bitmap[(j - j0) >> 5], 1u << ((j - j0) & 31));
    }
    __syncthreads();
    const int wpt = (int)ceil_div(nwords, kThreads);
    const int w0 = tid * wpt, w1 = min(nwords, w0 + wpt);
    unsigned mine = 0;
    for (int w = w0; w < w1; ++w) mine += __popc(sx->bitmap[w]);
    unsigned local_total = 0;
    unsigned k = block_prefix_exclusive(mine, fx->warp_tmp, &local_total);
    if (tid == 0) fx->sel = local_total;
    asm volatile("cp.async.wait_all;\n" ::: "memory");
    cluster_sync();   // every CTA's count is published
    QSA_TS(attn, 20);
    unsigned base = 0, total = 0;
    for (int p = 0; p < (int)NC; ++p) {
      const unsigned c = ld_dsmem_u32(dsmem_addr(&fx->sel, (uint32_t)p));
      if (p < (int)rank) base += c;
      total += c;
    }
    k += base;
    for (int w = w0; w < w1; ++w) {
      unsigned bits = sx->bitmap[w];
      while (bits) {
        const int64_t j = j0 + (int64_t)w * 32 + (__ffs(bits) - 1);
        bits &= bits - 1u;
        if (k < (unsigned)B)
          st_dsmem_u32(dsmem_addr(&fx->list[k], 0),
                       (unsigned)(slots_cached ? my_slots[j - j0] : slots[j]));
        ++k;
      }
    }
    if (rank == 0 && tid == 0) {
      const int nsel = (int)min(total, (unsigned)B);
      fx->nsel = nsel;
      fx->count = nsel * r + tail;
    }
    QSA_TS(attn, 21);
    cluster_sync();   // CTA 0's list is complete
  }
  QSA_TS(attn, 22);

  // ---- 4. the cells of this CTA's tiles (and, KV head 0, the outputs)
  const int nsel = (int)ld_dsmem_u32(dsmem_addr(&fx->nsel, 0));
  int count = (int)ld_dsmem_u32(dsmem_addr(&fx->count, 0));
  const int tiles_total = (int)ceil_div(cells_pitch, kTile);
  const int my_tiles = (int)rank < tiles_total ? (tiles_total - (int)rank + (int)NC - 1) / (int)NC : 0;
  int32_t* crow = sa.cells + (int64_t)t * cells_pitch;
  for (int idx = tid; idx < my_tiles * kTile; idx += kThreads) {
    const int i = ((int)rank + (idx >> 7) * (int)NC) * kTile + (idx & (kTile - 1));
    int cell = -1;
    if (i < nsel * r) {
      const int slot = (int)ld_dsmem_u32(dsmem_addr(&fx->list[i / r], 0));
      const bool sok = slot >= 0 && slot < ia.n_slots;
      if (!sok) atomicOr(err, kErrSlot);
      cell = flag_cell(sok ? ia.blk_cells[(int64_t)slot * r + i % r] : -1, ia.n_cells, err);
    } else if (i < count) {
      cell = flag_cell((int)ld_dsmem_u32(dsmem_addr(&fx->tail_cells[i - nsel * r], 0)), ia.n_cells, err);
    }
    fx->mycells[idx] = cell;
    if (g == 0 && i < cells_pitch) crow[i] = cell;
  }
  if (g == 0 && rank == 0 && tid == 0) {
    sa.count[t] = count;
    if (sg.tail_missing) atomicOr(err, kErrBlockList);
  }
  __syncthreads();
  if (fx->last) {
    uint4* h4 = reinterpret_cast<uint4*>(gh);
    for (int i = tid; i < kHistBins / 4; i += kThreads) h4[i] = make_uint4(0u, 0u, 0u, 0u);
    if (tid == 0) *readers_of(sa.ws, t) = 0u;
    __threadfence();
  }
  QSA_TS(attn, 23);
  count = count < 0 ? 0 : (count > cells_pitch ? cells_pitch : count);
  return count;
}

// kPipe: the launch gives CTAs several tiles each; the pipelined tile loops
// (fp16: cp.async groups into shared memory; q8_0: the next tile's rows in
// registers) are compiled only into this variant, so the one-tile decode
// variant keeps its code small (it runs from a cold instruction cache).
// kSel: the clusters first select and expand the token's blocks
// (select_in_cluster) and read the cells from shared memory; otherwise the
// cell list comes from global memory (written by qsa_index_topk).
template <bool kQ8, bool kPipe, bool kSel>
__global__ void __launch_bounds__(kThreads, 1)
k_attn_tc(const AttnArgs a, const SelArgs sa, unsigned* err) {
  QSA_TS_SCOPE_LAST(attn, 28);
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  const uint32_t base_s = (raw_s + 1023u) & ~1023u;
  unsigned char* base = smem_raw + (base_s - raw_s);
  const uint32_t sK = base_s + kOffK, sV = base_s + kOffV, sQ = base_s + kOffQ, sP = base_s + kOffP;
  float* so = reinterpret_cast<float*>(base + kOffO);
  float* sml = reinterpret_cast<float*>(base + kOffM);
  float* sred = reinterpret_cast<float*>(base + kOffRed);
  int* scell = reinterpret_cast<int*>(base + kOffCell);
  const uint32_t bar = base_s + kOffBar;
  uint32_t* stmem = reinterpret_cast<uint32_t*>(base + kOffTmem);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = blockIdx.y, t = blockIdx.z;
  const uint32_t rank = cluster_rank(), NC = cluster_size();
  const int G = a.n_kv_heads, Hq = G * kGqa;
  // scores live in the log2 domain: s * attn_scale * log2(e), exponentials by exp2f
  const float scale2 = a.attn_scale * 1.4426950408889634f;
  SelFix* fx = reinterpret_cast<SelFix*>(base + kOffFix);
  SelScratch* sx = reinterpret_cast<SelScratch*>(base + kOffK);

  QSA_TS(attn, 0);
  SelGeom sg{};
  if constexpr (kSel) {
    // the selection's geometry (inputs only); its counters are set before the
    // first half of a cluster barrier whose second half precedes any push
    sg = sel_geometry(sa.ia, t, rank, NC, err);
    if (tid == 0) {
      fx->ncand = 0u;
      fx->ncent = 0u;
    }
    cluster_arrive();
  }
  // ---- prologue (inputs not produced by the preceding index kernels)
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(base_s + kOffTmem),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
  }
  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(bar) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  {
    // Q rows 0..7 = the group's query heads, rows 8..15 zero; P rows 8..15 zero.
    const __half* qg = a.q + ((int64_t)t * Hq + g * kGqa) * kHeadDim;
    for (int i = tid; i < 16 * 32; i += kThreads) {
      const int row = i >> 5, c16 = i & 31;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (row < kGqa) v = __ldg(reinterpret_cast<const uint4*>(qg + row * kHeadDim + c16 * 8));
      *reinterpret_cast<uint4*>(base + kOffQ + sw128(16, row, c16)) = v;
    }
    for (int i = tid; i < 8 * 16; i += kThreads) {
      const int row = 8 + (i >> 4), c16 = i & 15;
      *reinterpret_cast<uint4*>(base + kOffP + sw128(16, row, c16)) = make_uint4(0, 0, 0, 0);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *stmem;

  // ---- the cell list is written by the index kernels (kSel: the scores
  // and histogram are)
  QSA_TS(attn, 1);
  grid_dep_wait();
  if constexpr (!kSel) grid_dep_launch();
  QSA_TS(attn, 2);
  const int32_t* crow = a.cells + (int64_t)t * a.cells_pitch;
  // cell id at position i of the token's list, for positions in this CTA's tiles
  auto list_cell = [&](int i) -> int {
    if constexpr (kSel) {
      return fx->mycells[(((i >> 7) - (int)rank) / (int)NC) * kTile + (i & (kTile - 1))];
    } else {
      return crow[i];
    }
  };
  int cfirst = -1;
  int cnt = 0;
  if constexpr (kSel) {
    cnt = select_in_cluster(sa, sg, a.cells_pitch, t, g, G, rank, NC, fx, sx, err);
    if (tid < kTile) cfirst = fx->mycells[tid];
    // the scores and the histogram are no longer read: the successor may start
    __syncthreads();
    grid_dep_launch();
  } else {
    // the first tile's cells and the count load together
    if (tid < kTile && (int)rank * kTile + tid < a.cells_pitch) cfirst = crow[(int)rank * kTile + tid];
    cnt = a.count[t];
    cnt = cnt < 0 ? 0 : (cnt > a.cells_pitch ? a.cells_pitch : cnt);
  }
  const int n_tiles = (cnt + kTile - 1) / kTile;

  float run_m[kGqa], run_l[kGqa], acc[2][kGqa];
#pragma unroll
  for (int h = 0; h < kGqa; ++h) {
    run_m[h] = -INFINITY;
    run_l[h] = 0.f;
    acc[0][h] = acc[1][h] = 0.f;
  }
  uint32_t phase = 0;
  bool timed_out = false;

  // A short last tile (at most kOvf cells past the full tiles) is attended on
  // CUDA cores by warps 4-7 of CTA (n_tiles - 1) mod NC, the CTA that would
  // otherwise run one MMA tile more than the others, while its warps 0-3 run
  // their MMA tiles: for q8_0 whenever the tiles outnumber the CTAs (several
  // tiles per CTA happen at 5 tokens and 250k), for fp16 when every CTA holds
  // one full tile (n_tiles = NC + 1; the pipelined fp16 variant covers the
  // rest).
  const int ovf_n = (kQ8 ? n_tiles > (int)NC : n_tiles == (int)NC + 1) ? cnt - (n_tiles - 1) * kTile : 0;
  const bool use_ovf = ovf_n > 0 && ovf_n <= kOvf;
  const int loop_tiles = use_ovf ? n_tiles - 1 : n_tiles;
  const int ovf_rank = (n_tiles - 1) % (int)NC;
  const bool my_ovf = use_ovf && (int)rank == ovf_rank;

  // the overflow cells' ids load with the first tile's (warps 4-7 of CTA 0)
  int* xc = reinterpret_cast<int*>(base + kOffXC);
  if (my_ovf && warp >= 4 && tid - 128 < kOvf) {
    const int tx = tid - 128;
    int c = -1;
    if (tx < ovf_n) {
      c = list_cell((n_tiles - 1) * kTile + tx);
      if (c < 0 || c >= a.n_cells) {
        atomicOr(err, kErrCell);
        c = -1;
      }
    }
    xc[tx] = c;
  }
  // fp16: with overflow cells, warps 0-3 gather the MMA tile alone while warps
  // 4-7 gather and attend the overflow cells from the start
  const bool split = !kQ8 && my_ovf && loop_tiles <= (int)NC;   // this CTA runs one MMA tile

  // Per-tile steps of warps 0-3 (tile: for the phase stamps only); uK and
  // uV are the shared-memory tiles the MMAs read (they rotate over three
  // stages in the pipelined fp16 variant)
  uint32_t uK = sK, uV = sV;
  float tmax[kGqa], pe[kGqa];
  auto qk_mma = [&](int tile) {
    // 2. S[cell][head] = K . Q^T
    if (tid == 0) {
#pragma unroll
      for (int kk = 0; kk < 16; ++kk) {
        const uint64_t ad = smem_desc(uK + (kk >> 2) * (kTile * 128) + (kk & 3) * 32, 16, 1024);
        const uint64_t bd = smem_desc(sQ + (kk >> 2) * (16 * 128) + (kk & 3) * 32, 16, 1024);
        mma_f16(tmem, ad, bd, kIdescQK, kk > 0);
      }
      mma_commit(bar);
    }
    if (!mbar_wait(bar, phase)) timed_out = true;
    phase ^= 1;
    tc_fence_after();
    QSA_TS(attn, 5 + 10 * (tile / (int)NC));
  };
  auto softmax_p = [&](int tile, const int* cells, int nv) {
    // 3. tile softmax statistics and P (one cell per thread); per-warp
    // statistics by reduce-scatter, lanes 4k hold head k's
    float sv[kGqa];
    tmem_ld8(tmem + ((uint32_t)(32 * warp) << 16) + 0, sv);
    if (tile < (int)NC) QSA_TS(attn, 8);
    const int cell = 32 * warp + lane;
    const bool valid = cell < nv && cells[cell] >= 0;
#pragma unroll
    for (int h = 0; h < kGqa; ++h) sv[h] = valid ? sv[h] * scale2 : -INFINITY;
    {
      const float m = warp_reduce8(sv, lane, OpMax());
      if ((lane & 3) == 0) sred[warp * 8 + (lane >> 2)] = m;
    }
    bar_half(1);
    if (tile < (int)NC) QSA_TS(attn, 9);
#pragma unroll
    for (int h = 0; h < kGqa; ++h) tmax[h] = fmaxf(fmaxf(sred[h], sred[8 + h]), fmaxf(sred[16 + h], sred[24 + h]));
#pragma unroll
    for (int h = 0; h < kGqa; ++h) {
      const float p = (tmax[h] == -INFINITY) ? 0.f : exp2f(sv[h] - tmax[h]);
      const __half ph = __float2half_rn(p);
      pe[h] = __half2float(ph);   // the sum uses the rounded p the MMA sees
      // P row h, column `cell`: atom cell/64, chunk (cell%64)/8, element cell%8
      const uint32_t off = (uint32_t)(cell >> 6) * (16 * 128) + h * 128 +
                           ((((uint32_t)(cell & 63) >> 3) ^ (uint32_t)(h & 7)) << 4) + (cell & 7) * 2;
      *reinterpret_cast<__half*>(base + kOffP + off) = ph;
    }
    if (tile < (int)NC) QSA_TS(attn, 10);
    fence_async_smem();
    tc_fence_before();
    bar_half(1);
    tc_fence_after();
    QSA_TS(attn, 6 + 10 * (tile / (int)NC));
  };
  auto pv_merge = [&](int tile) {
    // 4. O^T[dim][head] = V^T . P^T, two halves of 128 dims; the tile's
    // row sums are reduced while the MMAs run
    if (tid == 0) {
#pragma unroll
      for (int mh = 0; mh < 2; ++mh) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t ad = smem_desc(uV + mh * 2 * (kTile * 128) + kk * 2048, kTile * 128, 1024);
          const uint64_t bd = smem_desc(sP + (kk >> 2) * (16 * 128) + (kk & 3) * 32, 16, 1024);
          mma_f16(tmem + 16 + 16 * mh, ad, bd, kIdescPV, kk > 0);
        }
      }
      mma_commit(bar);
    }
    {
      const float e = warp_reduce8(pe, lane, OpAdd());
      if ((lane & 3) == 0) sred[32 + warp * 8 + (lane >> 2)] = e;
    }
    bar_half(1);
    float tsum[kGqa];
#pragma unroll
    for (int h = 0; h < kGqa; ++h)
      tsum[h] = (sred[32 + h] + sred[40 + h]) + (sred[48 + h] + sred[56 + h]);
    if (!mbar_wait(bar, phase)) timed_out = true;
    phase ^= 1;
    tc_fence_after();
    QSA_TS(attn, 7 + 10 * (tile / (int)NC));

    // 5. merge the tile into the running state (dims 32w+lane and +128)
    float o0[8], o1[8];
    tmem_ld8(tmem + ((uint32_t)(32 * warp) << 16) + 16, o0);
    tmem_ld8(tmem + ((uint32_t)(32 * warp) << 16) + 32, o1);
#pragma unroll
    for (int h = 0; h < kGqa; ++h) {
      const float mn = fmaxf(run_m[h], tmax[h]);
      const float fa = (run_m[h] == -INFINITY) ? 0.f : exp2f(run_m[h] - mn);
      const float fb = (tmax[h] == -INFINITY) ? 0.f : exp2f(tmax[h] - mn);
      acc[0][h] = acc[0][h] * fa + o0[h] * fb;
      acc[1][h] = acc[1][h] * fa + o1[h] * fb;
      run_l[h] = run_l[h] * fa + tsum[h] * fb;
      run_m[h] = mn;
    }
  };

  // fp16 with several tiles per CTA (no overflow cells; not with the fused
  // selection, whose state sits where the third stage would): warps 4-7
  // gather, warps 0-3 attend, meeting only at mbarriers.  Loads alternate
  // (load 2i: the K rows of this CTA's i-th tile, 2i + 1: its V rows) over
  // three 64 KB stages; a stage's full barrier completes once the gather
  // warps' copies into it have landed (each gather thread arrives for load
  // L - 1 after issuing load L, so two loads are in flight per thread), its
  // empty barrier once the MMA reading it has completed.  The gather warps
  // list a tile's cells with its K load into a ring of three lists; a list
  // is overwritten only by the K load three tiles later, which waits for
  // the V of the tile after it to be consumed.
  const bool pipe = kPipe && !kQ8 && !kSel && !use_ovf && (int)rank + (int)NC < loop_tiles;
  if constexpr (kPipe && !kQ8 && !kSel) {
    if (pipe) {
      const uint32_t sX3 = base_s + kOffX3;
      int* cl1 = reinterpret_cast<int*>(base + kOffCell2);
      int* cl2 = reinterpret_cast<int*>(base + kOffCell3);
      auto buf = [&](int x) { return x == 0 ? sK : (x == 1 ? sV : sX3); };
      auto cl = [&](int x) { return x == 0 ? scell : (x == 1 ? cl1 : cl2); };
      const uint32_t bfull = base_s + kOffPipeBar, bempty = bfull + 24;
      const int n_my = (loop_tiles - (int)rank + (int)NC - 1) / (int)NC;   // this CTA's tiles (>= 2)
      if (tid == 0) {
        for (int q = 0; q < 3; ++q) {
          mbar_init(bfull + 8 * q, kTile);
          mbar_init(bempty + 8 * q, 1);
        }
      }
      __syncthreads();
      if (warp >= 4) {
        const int tx = tid - kTile;
        const __half* kb = static_cast<const __half*>(a.k_cache);
        const __half* vb = static_cast<const __half*>(a.v_cache);
        for (int L = 0; L < 2 * n_my; ++L) {
          const int st = L % 3, use = L / 3, i = L >> 1;
          if (!mbar_wait(bempty + 8 * st, (uint32_t)((use & 1) ^ 1))) timed_out = true;
          int* cells = cl(i % 3);
          if ((L & 1) == 0) {
            const int c0 = ((int)rank + i * (int)NC) * kTile, nvt = min(kTile, cnt - c0);
            int c = -1;
            if (tx < nvt) {
              c = list_cell(c0 + tx);
              if (c < 0 || c >= a.n_cells) {
                atomicOr(err, kErrCell);
                c = -1;
              }
            }
            cells[tx] = c;
            bar_half(2);   // every row's cell is listed before any copy reads it
          }
          const __half* src = (L & 1) ? vb : kb;
          const uint32_t dst = buf(st);
          for (int k = tx; k < kTile * 32; k += kTile) {
            const int row = k >> 5, c16 = k & 31, c = cells[row];
            const int64_t off = ((int64_t)(c < 0 ? 0 : c) * G + g) * kHeadDim + c16 * 8;
            cp_async16(dst + sw128(kTile, row, c16), src + off, c >= 0);
          }
          asm volatile("cp.async.commit_group;\n" ::: "memory");
          if (L > 0) {
            asm volatile("cp.async.wait_group 1;\n" ::: "memory");   // load L - 1 has landed
            fence_async_smem();
            arrive_cta(bfull + 8 * ((L - 1) % 3));
          }
        }
        asm volatile("cp.async.wait_group 0;\n" ::: "memory");
        fence_async_smem();
        arrive_cta(bfull + 8 * ((2 * n_my - 1) % 3));
      } else {
        for (int i = 0; i < n_my; ++i) {
          const int tile = (int)rank + i * (int)NC;
          const int nv = min(kTile, cnt - tile * kTile);
          const int sk = (2 * i) % 3, sv = (2 * i + 1) % 3;
          uK = buf(sk);
          uV = buf(sv);
          if (!mbar_wait(bfull + 8 * sk, (uint32_t)(((2 * i) / 3) & 1))) timed_out = true;
          tc_fence_after();
          qk_mma(tile);
          if (tid == 0) arrive_cta(bempty + 8 * sk);   // Q.K^T has completed: the K stage is free
          softmax_p(tile, cl(i % 3), nv);
          if (!mbar_wait(bfull + 8 * sv, (uint32_t)(((2 * i + 1) / 3) & 1))) timed_out = true;
          tc_fence_after();
          pv_merge(tile);
          if (tid == 0) arrive_cta(bempty + 8 * sv);   // P.V has completed: the V stage is free
        }
      }
    }
  }

  // q8_0: each half warp takes one row at a time, lane l its 16 int8 at
  // dims 16 (l % 16) .. +15 (one 16-byte load of K and one of V, so a warp
  // load covers two whole 256-byte rows) plus the scale of their q8_0 block;
  // warp w takes rows 16 w + 2 j + l / 16, j = 0..7.  Fetched to registers,
  // then dequantised into the swizzled fp16 tiles: a warp's 16-byte stores
  // of one j cover the 8 chunk positions of a 128-byte line 4 times each.
  const int qc16 = lane & 15, qr0 = 16 * warp + (lane >> 4);
  uint4 qk[8], qv[8];
  __half qks[8], qvs[8];    // scales of rows j (not combined in the fetch, so
                            // nothing waits on a load before the MMAs)
  unsigned qvalid = 0u;     // bit j: row qr0 + 2j holds a cell
  auto q8_fetch = [&](const int* cl) {
    qvalid = 0u;
    if (a.n_cells <= 0) return;   // no row to read: every row is stored as zeros
    const int8_t* kq = static_cast<const int8_t*>(a.k_cache);
    const int8_t* vq = static_cast<const int8_t*>(a.v_cache);
    const int64_t nq = a.n_cells * (int64_t)G * kHeadDim;
    const __half* kd = reinterpret_cast<const __half*>(kq + nq);
    const __half* vd = reinterpret_cast<const __half*>(vq + nq);
    // every load is issued (an invalid row reads cell 0's, which exists,
    // and is zeroed when stored), so none waits behind a branch
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int c = cl[qr0 + 2 * j];
      const int64_t cg = (int64_t)(c < 0 ? 0 : c) * G + g;
      qk[j] = __ldg(reinterpret_cast<const uint4*>(kq + cg * kHeadDim) + qc16);
      qv[j] = __ldg(reinterpret_cast<const uint4*>(vq + cg * kHeadDim) + qc16);
      qks[j] = kd[cg * 8 + (qc16 >> 1)];
      qvs[j] = vd[cg * 8 + (qc16 >> 1)];
      qvalid |= (c >= 0 ? 1u : 0u) << j;
    }
  };
  auto q8_store = [&]() {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      // 16 int8 = dims 16 qc16 .. +15 of row qr0 + 2j -> two 16-byte fp16 chunks
      const __half2 skf = __half2half2(qks[j]), svf = __half2half2(qvs[j]);
      // lanes 4-7 of each quarter warp store their upper chunk first, so the
      // 8 lanes of a quarter cover the 8 chunk positions of the line
      const int row = qr0 + 2 * j, sw = (qc16 >> 2) & 1, ca = 2 * qc16 + sw, cb = 2 * qc16 + 1 - sw;
      const bool ok = (qvalid >> j) & 1u;
      const uint4 k0 = ok ? dq8(make_uint2(qk[j].x, qk[j].y), skf) : make_uint4(0, 0, 0, 0);
      const uint4 k1 = ok ? dq8(make_uint2(qk[j].z, qk[j].w), skf) : make_uint4(0, 0, 0, 0);
      const uint4 v0 = ok ? dq8(make_uint2(qv[j].x, qv[j].y), svf) : make_uint4(0, 0, 0, 0);
      const uint4 v1 = ok ? dq8(make_uint2(qv[j].z, qv[j].w), svf) : make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(base + kOffK + sw128(kTile, row, ca)) = sw ? k1 : k0;
      *reinterpret_cast<uint4*>(base + kOffK + sw128(kTile, row, cb)) = sw ? k0 : k1;
      *reinterpret_cast<uint4*>(base + kOffV + sw128(kTile, row, ca)) = sw ? v1 : v0;
      *reinterpret_cast<uint4*>(base + kOffV + sw128(kTile, row, cb)) = sw ? v0 : v1;
    }
  };
  // q8_0 with several tiles per CTA (kPipe): the registers hold the next
  // tile's rows while this tile's MMAs and softmax run.  The cell lists of
  // the current and the next tile alternate between two shared arrays
  // (`qcur`, `qnext`); thread p < 128 checks row p's id of the next tile
  // before the barrier that precedes this tile's MMAs, having read it one
  // tile earlier still, so no warp waits on a list read before its MMAs.
  int* qcur = scell;
  int* qnext = reinterpret_cast<int*>(base + kOffCellN);
  int qraw = 0;   // thread p < 128: row p's raw id two tiles ahead
  auto q8_cell = [&](int tile, int raw) {
    const int i = tile * kTile + tid;
    if (tile >= loop_tiles || i >= cnt) return -1;
    if (raw < 0 || raw >= a.n_cells) {
      atomicOr(err, kErrCell);
      return -1;
    }
    return raw;
  };
  auto q8_raw = [&](int tile) {
    const int i = tile * kTile + tid;
    return (tile < loop_tiles && i < cnt) ? list_cell(i) : 0;
  };
  if constexpr (kQ8 && kPipe) {
    if (tid < kTile) {
      qcur[tid] = q8_cell((int)rank, cfirst);
      qraw = q8_raw((int)rank + (int)NC);
    }
    __syncthreads();
    q8_fetch(qcur);
  }

  if (!pipe)
  for (int tile = (int)rank; tile < loop_tiles; tile += (int)NC) {
    const int c0 = tile * kTile;
    const int nv = min(kTile, cnt - c0);
    if constexpr (kQ8 && kPipe) {
      q8_store();
      if (tid < kTile && tile + (int)NC < loop_tiles) qnext[tid] = q8_cell(tile + (int)NC, qraw);
    } else {
    if (tid < kTile) {
      int c = -1;
      if (tid < nv) {
        c = (tile == (int)rank) ? cfirst : list_cell(c0 + tid);
        if (c < 0 || c >= a.n_cells) {
          atomicOr(err, kErrCell);
          c = -1;
        }
      }
      scell[tid] = c;
    }
    if (split) {
      if (warp < 4) bar_half(1);
    } else {
      __syncthreads();
    }
    QSA_TS(attn, 3 + 10 * (tile / (int)NC));

    // 1. gather K and V rows of KV head g into the swizzled tiles
    if constexpr (!kQ8) {
      const __half* kb = static_cast<const __half*>(a.k_cache);
      const __half* vb = static_cast<const __half*>(a.v_cache);
      if (!split || warp < 4) {
        const int nthr = split ? 128 : kThreads;
        for (int i = tid; i < kTile * 32; i += nthr) {
          const int row = i >> 5, c16 = i & 31, c = scell[row];
          const int64_t off = ((int64_t)(c < 0 ? 0 : c) * G + g) * kHeadDim + c16 * 8;
          cp_async16(sK + sw128(kTile, row, c16), kb + off, c >= 0);
          cp_async16(sV + sw128(kTile, row, c16), vb + off, c >= 0);
        }
        asm volatile("cp.async.wait_all;\n" ::: "memory");
      }
    } else {
      q8_fetch(scell);
      q8_store();
    }
    }
    fence_async_smem();
    tc_fence_before();
    if (split) {
      if (warp < 4) bar_half(1);
    } else {
      __syncthreads();
    }
    tc_fence_after();
    QSA_TS(attn, 4 + 10 * (tile / (int)NC));
    if constexpr (kQ8 && kPipe) {
      if (tile + (int)NC < loop_tiles) {
        q8_fetch(qnext);
        if (tid < kTile) qraw = q8_raw(tile + 2 * (int)NC);
      }
    }

    if (warp < 4) {
      qk_mma(tile);
      softmax_p(tile, (kQ8 && kPipe) ? qcur : scell, nv);
      pv_merge(tile);
    } else if (my_ovf && tile == (int)rank) {
      // Overflow cells on warps 4-7 (128 threads, tx = 0..127); their ids
      // were loaded before the tile loop
      const int tx = tid - 128;
      float* xs = reinterpret_cast<float*>(base + kOffXS);
      float* xo = reinterpret_cast<float*>(base + kOffXO);
      float* xm = reinterpret_cast<float*>(base + kOffXM);
      bar_half(2);
      // gather the rows as plain fp16 [cell][256]
      if constexpr (!kQ8) {
        const __half* kb = static_cast<const __half*>(a.k_cache);
        const __half* vb = static_cast<const __half*>(a.v_cache);
        for (int i = tx; i < kOvf * 32; i += 128) {
          const int row = i >> 5, c16 = i & 31, c = xc[row];
          const int64_t off = ((int64_t)(c < 0 ? 0 : c) * G + g) * kHeadDim + c16 * 8;
          cp_async16(base_s + kOffXK + row * 512 + c16 * 16, kb + off, c >= 0);
          cp_async16(base_s + kOffXV + row * 512 + c16 * 16, vb + off, c >= 0);
        }
        asm volatile("cp.async.wait_all;\n" ::: "memory");
      } else {
        const int8_t* kq = static_cast<const int8_t*>(a.k_cache);
        const int8_t* vq = static_cast<const int8_t*>(a.v_cache);
        const int64_t nq = a.n_cells * (int64_t)G * kHeadDim;
        const __half* kd = reinterpret_cast<const __half*>(kq + nq);
        const __half* vd = reinterpret_cast<const __half*>(vq + nq);
        for (int i = tx; i < kOvf * 16; i += 128) {   // (row, 16-value group)
          const int row = i >> 4, grp = i & 15, c = xc[row];
          uint4 kr = make_uint4(0, 0, 0, 0), vr = make_uint4(0, 0, 0, 0);
          __half2 sk = __float2half2_rn(0.f), svv = __float2half2_rn(0.f);
          if (c >= 0) {
            const int64_t cg = (int64_t)c * G + g;
            kr = __ldg(reinterpret_cast<const uint4*>(kq + cg * kHeadDim + grp * 16));
            vr = __ldg(reinterpret_cast<const uint4*>(vq + cg * kHeadDim + grp * 16));
            sk = __half2half2(kd[cg * 8 + (grp >> 1)]);
            svv = __half2half2(vd[cg * 8 + (grp >> 1)]);
          }
          uint4* kdst = reinterpret_cast<uint4*>(base + kOffXK + row * 512 + grp * 32);
          uint4* vdst = reinterpret_cast<uint4*>(base + kOffXV + row * 512 + grp * 32);
          kdst[0] = dq8(make_uint2(kr.x, kr.y), sk);
          kdst[1] = dq8(make_uint2(kr.z, kr.w), sk);
          vdst[0] = dq8(make_uint2(vr.x, vr.y), svv);
          vdst[1] = dq8(make_uint2(vr.z, vr.w), svv);
        }
      }
      bar_half(2);
      // scores: thread -> (cell tx/4, heads 2*(tx%4), +1)
      {
        const int c = tx >> 2, h0 = 2 * (tx & 3);
        const __half* kr = reinterpret_cast<const __half*>(base + kOffXK + c * 512);
        float d0 = 0.f, d1 = 0.f;
        for (int c16 = 0; c16 < 32; ++c16) {
          const uint4 kv = *reinterpret_cast<const uint4*>(kr + c16 * 8);
          const uint4 q0 = *reinterpret_cast<const uint4*>(base + kOffQ + sw128(16, h0, c16));
          const uint4 q1 = *reinterpret_cast<const uint4*>(base + kOffQ + sw128(16, h0 + 1, c16));
          const __half2* k2 = reinterpret_cast<const __half2*>(&kv);
          const __half2* a2 = reinterpret_cast<const __half2*>(&q0);
          const __half2* b2 = reinterpret_cast<const __half2*>(&q1);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 kf = __half22float2(k2[e]), af = __half22float2(a2[e]), bf = __half22float2(b2[e]);
            d0 = fmaf(af.x, kf.x, fmaf(af.y, kf.y, d0));
            d1 = fmaf(bf.x, kf.x, fmaf(bf.y, kf.y, d1));
          }
        }
        const bool ok = c < ovf_n && xc[c] >= 0;
        xs[c * 8 + h0] = ok ? d0 * scale2 : -INFINITY;
        xs[c * 8 + h0 + 1] = ok ? d1 * scale2 : -INFINITY;
      }
      bar_half(2);
      // softmax per head: 16 lanes per head, cells l and l+16
      {
        const int h = tx >> 4, l = tx & 15;
        const float s0v = xs[l * 8 + h], s1v = xs[(l + 16) * 8 + h];
        float m = fmaxf(s0v, s1v);
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
        const float p0 = (m == -INFINITY) ? 0.f : exp2f(s0v - m);
        const float p1 = (m == -INFINITY) ? 0.f : exp2f(s1v - m);
        float sum = p0 + p1;
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1) sum += __shfl_xor_sync(kFull, sum, o);
        xs[l * 8 + h] = p0;
        xs[(l + 16) * 8 + h] = p1;
        if (l == 0) {
          xm[h] = m;
          xm[8 + h] = sum;
        }
      }
      bar_half(2);
      // P.V: thread -> dims tx and tx + 128 for the 8 heads
      {
        float o[2][kGqa];
#pragma unroll
        for (int h = 0; h < kGqa; ++h) o[0][h] = o[1][h] = 0.f;
        const __half* vx = reinterpret_cast<const __half*>(base + kOffXV);
        for (int c = 0; c < ovf_n; ++c) {
          const float v0 = __half2float(vx[c * kHeadDim + tx]);
          const float v1 = __half2float(vx[c * kHeadDim + 128 + tx]);
#pragma unroll
          for (int h = 0; h < kGqa; ++h) {
            const float p = xs[c * 8 + h];
            o[0][h] = fmaf(p, v0, o[0][h]);
            o[1][h] = fmaf(p, v1, o[1][h]);
          }
        }
#pragma unroll
        for (int h = 0; h < kGqa; ++h) {
          xo[h * kHeadDim + tx] = o[0][h];
          xo[h * kHeadDim + 128 + tx] = o[1][h];
        }
      }
    }
    if (tile < (int)NC) QSA_TS(attn, 12);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if constexpr (kQ8 && kPipe) {
      int* const x = qcur;
      qcur = qnext;
      qnext = x;
    }
  }
  // fold the overflow partial into warps 0-3's running state
  if (my_ovf && warp < 4) {
    const float* xo = reinterpret_cast<const float*>(base + kOffXO);
    const float* xm = reinterpret_cast<const float*>(base + kOffXM);
#pragma unroll
    for (int h = 0; h < kGqa; ++h) {
      const float mx = xm[h];
      const float mn = fmaxf(run_m[h], mx);
      const float fa = (run_m[h] == -INFINITY) ? 0.f : exp2f(run_m[h] - mn);
      const float fb = (mx == -INFINITY) ? 0.f : exp2f(mx - mn);
      acc[0][h] = acc[0][h] * fa + xo[h * kHeadDim + 32 * warp + lane] * fb;
      acc[1][h] = acc[1][h] * fa + xo[h * kHeadDim + 128 + 32 * warp + lane] * fb;
      run_l[h] = run_l[h] * fa + xm[8 + h] * fb;
      run_m[h] = mn;
    }
  }
  if (timed_out) atomicOr(err, kErrTimeout);

  // ---- push this CTA's partial to the CTAs that own each dim range, then
  // every CTA reduces its range from its own shared memory
  QSA_TS(attn, 11);
  const int dpc = (kHeadDim + (int)NC - 1) / (int)NC;   // dims per owner (a multiple of 4)
  if (warp < 4) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int d = half * 128 + 32 * warp + lane;
      const uint32_t owner = (uint32_t)(d / dpc), e = (uint32_t)(d % dpc);
#pragma unroll
      for (int h = 0; h < kGqa; ++h)
        st_dsmem_f32(dsmem_addr(&so[((int)rank * kGqa + h) * dpc + e], owner), acc[half][h]);
    }
  }
  if (tid < (int)NC) {
    const uint32_t dst = dsmem_addr(&sml[(int)rank * 16], (uint32_t)tid);
    st_dsmem_f32x4(dst, make_float4(run_m[0], run_m[1], run_m[2], run_m[3]));
    st_dsmem_f32x4(dst + 16, make_float4(run_m[4], run_m[5], run_m[6], run_m[7]));
    st_dsmem_f32x4(dst + 32, make_float4(run_l[0], run_l[1], run_l[2], run_l[3]));
    st_dsmem_f32x4(dst + 48, make_float4(run_l[4], run_l[5], run_l[6], run_l[7]));
  }
  QSA_TS(attn, 25);
  cluster_sync();   // all pushes have landed; nobody touches a peer after this
  QSA_TS(attn, 26);
  {
    // output (head h, dim d0 + e) = sum_p w_p o_p / sum_p w_p l_p with
    // w_p = exp2(m_p - max_p m_p).  First the normalised weight of each
    // (partial p, head h), one per thread of warps 0-3 with a head's partials
    // in 16 consecutive lanes; then one output per thread.
    float* wgt = reinterpret_cast<float*>(base + kOffQ);   // the Q tile is no longer read
    if (tid < 16 * kGqa) {
      const int h = tid >> 4, p = tid & 15;
      const float mp = p < (int)NC ? sml[p * 16 + h] : -INFINITY;
      const float lp = p < (int)NC ? sml[p * 16 + 8 + h] : 0.f;
      float mx = mp;
#pragma unroll
      for (int o = 8; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
      const float w = (mp == -INFINITY) ? 0.f : exp2f(mp - mx);
      float den = w * lp;
#pragma unroll
      for (int o = 8; o >= 1; o >>= 1) den += __shfl_xor_sync(kFull, den, o);
      wgt[p * kGqa + h] = den > 0.f ? w / den : 0.f;
    }
    __syncthreads();
    const int d0 = (int)rank * dpc;
    for (int i = tid; i < kGqa * dpc; i += kThreads) {
      const int h = i / dpc, e = i % dpc, d = d0 + e;
      if (d >= kHeadDim) continue;
      float o = 0.f;
      for (int p = 0; p < (int)NC; ++p) o = fmaf(wgt[p * kGqa + h], so[(p * kGqa + h) * dpc + e], o);
      a.out[((int64_t)t * Hq + g * kGqa + h) * kHeadDim + d] = o;
    }
  }
  QSA_TS(attn, 27);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(kTmemCols) : "memory");
}

constexpr int kMaxDevices = 64;

// Cluster size for a launch of `clusters` clusters: 16 CTAs (one per 128-cell
// tile of the 2051-cell budget) when that many 16-CTA clusters are co-resident,
// else the largest smaller power of two that fits them.
template <bool kQ8, bool kSel>
cudaError_t pick_cluster(const AttnArgs& a, int* nc_out) {
  // per device: clusters of 16, 8, 4, 2, 1 that fit at once, measured once
  // under a lock and published by `configured`
  static int max_active[kMaxDevices][5];
  static std::atomic<bool> configured[kMaxDevices];
  static std::mutex mu;
  constexpr int kSmem = (int)smem_bytes<kSel>();
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!configured[dev].load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(mu);
    if (!configured[dev].load(std::memory_order_relaxed)) {
      e = cudaFuncSetAttribute(k_attn_tc<kQ8, false, kSel>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(k_attn_tc<kQ8, false, kSel>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(k_attn_tc<kQ8, true, kSel>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem_bytes_of<kQ8, true, kSel>());
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(k_attn_tc<kQ8, true, kSel>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
      for (int i = 0; i < 5; ++i) {
        const int nc = 16 >> i;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)nc, 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = (size_t)kSmem;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = (unsigned)nc;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, k_attn_tc<kQ8, false, kSel>, &cfg) != cudaSuccess) {
          (void)cudaGetLastError();
          n = 0;
        }
        max_active[dev][i] = n;
      }
      configured[dev].store(true, std::memory_order_release);
    }
  }
  const int tiles = (int)ceil_div(a.cells_pitch, kTile);
  const int want = tiles < kMaxCluster ? tiles : kMaxCluster;
  const int64_t clusters = (int64_t)a.n_tokens * a.n_kv_heads;
  int nc = 0;
  for (int i = 0; i < 5; ++i) {            // sizes 16, 8, 4, 2, 1
    const int c = 16 >> i;
    if (c > want || max_active[dev][i] <= 0) continue;
    if (clusters <= max_active[dev][i]) {  // the largest size that runs in one wave
      nc = c;
      break;
    }
  }
  if (nc == 0) {
    // Several waves at every size: a CTA costs about one tile's time of its
    // own (launch, prologue, cluster combine) plus one per tile it takes, so
    // pick the size with the fewest waves x (1 + tiles per CTA).
    int64_t best = -1;
    for (int i = 0; i < 5; ++i) {
      const int c = 16 >> i;
      if (c > want || max_active[dev][i] <= 0) continue;
      const int64_t waves = ceil_div(clusters, (int64_t)max_active[dev][i]);
      const int64_t cost = waves * (1 + ceil_div((int64_t)tiles, (int64_t)c));
      if (best < 0 || cost < best) {
        best = cost;
        nc = c;
      }
    }
    if (nc == 0) nc = 1;
  }
  *nc_out = nc;
  return cudaSuccess;
}

template <bool kQ8, bool kSel>
cudaError_t launch_tc(const AttnArgs& a, const SelArgs& sa, int nc, unsigned* err, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)nc, (unsigned)a.n_kv_heads, (unsigned)a.n_tokens);
  cfg.blockDim = dim3(kThreads, 1, 1);
  const int tiles = (int)ceil_div(a.cells_pitch, kTile);
  const bool piped = 2 * nc <= tiles;   // several tiles per CTA: the pipelined variant
  cfg.dynamicSmemBytes = piped ? smem_bytes_of<kQ8, true, kSel>() : smem_bytes_of<kQ8, false, kSel>();
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)nc;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (piped) return cudaLaunchKernelEx(&cfg, k_attn_tc<kQ8, true, kSel>, a, sa, err);
  return cudaLaunchKernelEx(&cfg, k_attn_tc<kQ8, false, kSel>, a, sa, err);
}

template <bool kQ8>
cudaError_t launch_plain(const AttnArgs& a, unsigned* err, cudaStream_t stream) {
  int nc = 1;
  cudaError_t e = pick_cluster<kQ8, false>(a, &nc);
  if (e != cudaSuccess) return e;
  // many tokens (one CTA per (token, KV head) and several tiles each), fp16:
  // the variant that puts two CTAs on an SM
  if (!kQ8 && nc == 1 && attn_pf_eligible(a)) return launch_attn_pf(a, err, stream);
  return launch_tc<kQ8, false>(a, SelArgs{}, nc, err, stream);
}

// The fused launch when its limits hold (*done = false otherwise, nothing
// launched): at most 65,536 blocks per token, 1,024 chosen blocks, 8 tiles
// per CTA.
template <bool kQ8>
cudaError_t launch_fused(const AttnArgs& a, const SelArgs& sa, unsigned* err, cudaStream_t stream, bool* done) {
  *done = false;
  if (sa.ia.max_blocks > kFusedMaxBlocks || sa.ia.n_sel_blocks > kFusedMaxList || sa.ia.r > 8) return cudaSuccess;
  int nc = 1;
  cudaError_t e = pick_cluster<kQ8, true>(a, &nc);
  if (e != cudaSuccess) return e;
  if (ceil_div(ceil_div(a.cells_pitch, kTile), nc) > kFusedMaxTiles) return cudaSuccess;
  *done = true;
  return launch_tc<kQ8, true>(a, sa, nc, err, stream);
}

}  // namespace

size_t attn_workspace_bytes(int, int, int) { return 0; }

cudaError_t launch_sparse_attn(const AttnArgs& a, void*, unsigned* err, cudaStream_t stream) {
  if (a.n_tokens <= 0) return cudaSuccess;
  prof_before(kKAttn, stream);
  cudaError_t e = a.kv_q8 ? launch_plain<true>(a, err, stream) : launch_plain<false>(a, err, stream);
  prof_after(kKAttn, stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t index_attn_plan(int n_tokens, int n_kv_heads, int kv_q8, int cells_pitch, int64_t max_blocks,
                            int n_sel_blocks, int r, bool* fused) {
  *fused = false;
  if (n_tokens <= 0 || max_blocks > kFusedMaxBlocks || n_sel_blocks > kFusedMaxList || r > 8) return cudaSuccess;
  AttnArgs a{};
  a.n_tokens = n_tokens;
  a.n_kv_heads = n_kv_heads;
  a.cells_pitch = cells_pitch;
  int nc = 1;
  cudaError_t e = kv_q8 ? pick_cluster<true, true>(a, &nc) : pick_cluster<false, true>(a, &nc);
  if (e != cudaSuccess) return e;
  *fused = ceil_div(ceil_div(cells_pitch, kTile), nc) <= kFusedMaxTiles;
  return cudaSuccess;
}

cudaError_t launch_index_attn(const IndexArgs& ia, const AttnArgs& a, int32_t* cells, int32_t* count, void* ws,
                              bool in_cluster, unsigned* err, cudaStream_t stream, bool* fused) {
  *fused = false;
  if (a.n_tokens <= 0) return cudaSuccess;
  SelArgs sa{};
  sa.ia = ia;
  sa.ia.max_blocks = ia.max_blocks > 0 ? ia.max_blocks : 1;
  sa.ws = ws;
  sa.cells = cells;
  sa.count = count;
  // the limits of the fused launch are known before anything is launched
  bool ok = false;
  if (in_cluster) {
    cudaError_t e0 = index_attn_plan(a.n_tokens, a.n_kv_heads, a.kv_q8, a.cells_pitch, sa.ia.max_blocks,
                                     ia.n_sel_blocks, ia.r, &ok);
    if (e0 != cudaSuccess) return e0;
  }
  if (!ok) {
    cudaError_t e = launch_index_topk(ia, cells, count, ws, err, stream);
    if (e != cudaSuccess) return e;
    return launch_sparse_attn(a, nullptr, err, stream);
  }
  cudaError_t e = launch_index_scores_topk(ia, ws, err, stream);
  if (e != cudaSuccess) return e;
  bool done = false;
  prof_before(kKFused, stream);
  e = a.kv_q8 ? launch_fused<true>(a, sa, err, stream, &done) : launch_fused<false>(a, sa, err, stream, &done);
  prof_after(kKFused, stream);
  if (e != cudaSuccess) return e;
  *fused = done;
  return cudaGetLastError();
}

}  // namespace qsa
