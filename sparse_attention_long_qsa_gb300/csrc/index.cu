// S2 + S3 + S4: indexer block scores, block-granular top-k, block -> cell
// expansion.
//
// llama.cpp issue #28734 ("decode slows linearly with context"), fix summary,
// lever3: scores are constant within a block and the budget is whole blocks,
// so blocks are selected first and only the chosen ones are expanded to cell
// indices through the block-member table (lever2b); blocks that are not yet
// complete for the token never compete (-inf), and the incomplete tail
// block's cells ride along as a side input.  The budget is top_k / r whole
// blocks plus at most r - 1 tail cells (goodbadwolf's comment in the same
// issue: n_kv_max = min(n_kv, indexer_top_k + r - 1)).
//
// The indexer score is not written out on the pages; the definition used is
//   S[t][j] = sum_h w[t][h] * max(0, q_idx[t][h] . pooled[slot(seq, j)])
// in fp32.
//
// Two kernels, chained by programmatic dependent launch, no host round trip:
//   k_score   streams the pooled rows of every visible block (the dominant
//             HBM traffic at long context: 512 B per block), writes fp32
//             scores and adds each block to a per-token 4096-bin histogram of
//             the top 12 bits of the order-preserving score key.
//   k_score_tc / k_hist  replace k_score when the call's tokens share
//             sequences (a verify batch, a prefill ubatch): each pooled row
//             is read once per tile of 32 tokens and scored on the
//             tensor cores (split-TF32, fp32-accurate), then k_hist builds the
//             histogram from the written scores.
//   k_select  one thread-block cluster per token (16 CTAs for one to four
//             tokens, 8 for a few more, down to 1 for many: select_cluster).  Every CTA reads the
//             histogram and finds the bin holding the B-th largest score.
//             Each CTA then takes a range of blocks: blocks above that bin go
//             straight into its shared selection bitmap (warp ballots), blocks
//             in the bin become unique 56-bit keys (low score bits,
//             complemented index).  The cluster runs a radix select over
//             those keys, one 8-bit digit per round, summing the CTAs' digit
//             histograms through distributed shared memory; unique keys make
//             ties resolve to the lower block index.  Finally every CTA writes
//             the member cells of its chosen blocks at its offset in the
//             token's list (blocks ascending), CTA 0 appends the tail cells
//             and clears the histogram for the next call.  A call with more
//             selection CTAs than SMs (a prefill ubatch) runs two CTAs per SM
//             (64 registers a thread, no slot-id cache), so one CTA's
//             classification loads overlap the other's serial phases.
#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>

#include "index_util.cuh"
#include "qsa_internal.cuh"
#include "tc_util.cuh"

QSA_TS_DECLARE(index)

namespace qsa {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kScoreThreads = 256;
constexpr int kScoreWarps = kScoreThreads / 32;
// Each warp streams its rows through a ring of kRingStages stages of 4 rows
// (one row per group of 8 lanes) by 16-byte cp.async copies: every lane copies
// its 16 bytes of each row, so a row is one warp instruction and up to
// kRingStages x 2 KiB per warp stay in flight without blocking the warp.
constexpr int kRingStages = 4;
constexpr int kRingFloats = kScoreWarps * kRingStages * 4 * kIdxDim;
constexpr int kScoreChunkMax = 2048;      // rows one CTA scores (their slot ids are kept in shared memory)
constexpr size_t kScoreSmem = sizeof(float) * kRingFloats + sizeof(int32_t) * kScoreChunkMax +
                              sizeof(unsigned) * kHistBins + sizeof(unsigned short) * kHistBins;
constexpr int kMaxHint = 32;              // recomputed-slot hints checked per CTA

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelCluster = 16;
constexpr int kSelMaxWords = 4096;        // bitmap words per CTA: 131072 blocks
constexpr int kSelLocalCand = 2048;       // candidate keys held per CTA
constexpr int kSelBatch = 16;             // score words a warp loads before using any
constexpr int kSelSlots = 16384;          // slot ids a CTA prefetches (rank 0: all, when they fit)
constexpr int kCentralBlocks = kSelMaxWords * 32 / 2;   // tokens up to 65536 blocks finish in CTA 0
constexpr int kRankMax = 1024;            // threshold-bin keys resolved by direct ranking
static_assert(kRankMax <= kSelLocalCand, "the cut-off digit's keys reuse the candidate list");
constexpr int kSelList = 2048;            // chosen blocks a CTA lists before expanding
// dynamic shared memory of k_select: the chosen-block list, then (one CTA
// per SM only) the slot-id cache, 0-3 ints of alignment shift included
constexpr size_t kSelDynBytes = sizeof(int32_t) * (kSelList + kSelSlots + 4);
constexpr size_t kSelDynBytes2 = sizeof(int32_t) * kSelList;

// ----------------------------------------------------------------- k_score
// Rows are read by groups of 8 lanes: lane `sub` of a group holds dims
// {32k + 4 sub .. 32k + 4 sub + 3 : k = 0..3} of the row and of the 4 query
// heads (64 fp32 registers), so each group reads the 512-byte row as four
// fully used 128-byte lines.  The 4 head dot products are reduced across the
// group with a reduce-scatter (6 shuffles per row in all).
__device__ __forceinline__ void ring_copy16(float* dst, const float* src, bool valid) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
  const int n = valid ? 16 : 0;   // 0: the 16 bytes are zero-filled
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(d), "l"(src), "r"(n) : "memory");
}

// Packed fp32 FMA on a pair of lanes of a register pair: d = a * b + c
// element-wise, each element rounded as fmaf.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  unsigned long long ra, rb, rc, rd;
  memcpy(&ra, &a, 8);
  memcpy(&rb, &b, 8);
  memcpy(&rc, &c, 8);
  asm("fma.rn.f32x2 %0, %1, %2, %3;\n" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
  float2 d;
  memcpy(&d, &rd, 8);
  return d;
}

template <bool kTopk>
__global__ void __launch_bounds__(kScoreThreads, 2)
k_score(const IndexArgs a, void* ws, float* __restrict__ scores, int chunk, unsigned* err) {
  QSA_TS_SCOPE_LAST(index, 4);
  // Shared memory: the warps' row rings, the slot ids of this CTA's range,
  // and a histogram of this CTA's scores plus the list of bins it touched (so
  // the flush to the token's global histogram costs one atomic per touched
  // bin instead of a sweep of all bins).
  extern __shared__ __align__(16) unsigned char score_smem[];
  float* ring = reinterpret_cast<float*>(score_smem);
  int32_t* s_slot = reinterpret_cast<int32_t*>(ring + kRingFloats);
  unsigned* s_hist = reinterpret_cast<unsigned*>(s_slot + kScoreChunkMax);
  unsigned short* s_touched = reinterpret_cast<unsigned short*>(s_hist + kHistBins);
  __shared__ unsigned s_ntouched;
  __shared__ int s_rec[kMaxHint];

  const int t = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (kTopk) QSA_TS(index, 0);
  // ---- before the wait: token geometry, query, slot ids (not written by
  // the pool update that precedes this kernel)
  __shared__ int64_t s_off[kOffCache + 1];
  const int seq_t = a.tok_seq[t], pos_t = a.tok_pos[t];
  const bool offc = preload_offsets(a.seq_blk_off, a.n_seq, s_off);
  __syncthreads();
  const Tok tk = token_geometry(a, seq_t, pos_t, offc ? s_off : nullptr, err, blockIdx.x == 0 && tid == 0);
  const int nb = tk.nb;
  float* srow = scores + (int64_t)t * a.max_blocks;
  const int64_t j0 = (int64_t)blockIdx.x * chunk;
  const int64_t j1 = min((int64_t)nb, j0 + chunk);
  const int nrows = j1 > j0 ? (int)(j1 - j0) : 0;
  if (kTopk) {
    for (int i = tid; i < kHistBins; i += kScoreThreads) s_hist[i] = 0u;
    if (tid == 0) s_ntouched = 0u;
  }
  unsigned* ghist = kTopk ? hist_of(ws, t) : nullptr;
  const int32_t* slots = a.seq_blk_slots + tk.off;
  for (int i = tid; i < nrows; i += kScoreThreads) s_slot[i] = __ldg(slots + j0 + i);
  const bool use_hint = kTopk && a.recomputed != nullptr && a.n_recomputed <= kMaxHint;
  // caller's assertion: the preceding call recomputed only blocks holding
  // the query tokens' own positions (an append of exactly these tokens)
  const bool query_hint = kTopk && a.recomputed == nullptr && a.n_recomputed == QSA_HINT_QUERY_BLOCKS;
  if (use_hint)
    for (int i = tid; i < a.n_recomputed; i += kScoreThreads) s_rec[i] = a.recomputed[i];

  const int sub = lane & 7, grp = lane >> 3;
  float4 qv[kIdxHeads][4];
  {
    const float* qt = a.q_idx + (int64_t)t * kIdxHeads * kIdxDim;
#pragma unroll
    for (int h = 0; h < kIdxHeads; ++h)
#pragma unroll
      for (int k = 0; k < 4; ++k)
        qv[h][k] = __ldg(reinterpret_cast<const float4*>(qt + h * kIdxDim + k * 32 + sub * 4));
  }
  const int bit2 = (lane >> 2) & 1, bit1 = (lane >> 1) & 1;
  const float wh = __ldg(a.w_idx + (int64_t)t * kIdxHeads + bit2 * 2 + bit1);
  __syncthreads();

  // ---- pooled rows are written by the pool update.  With the list of slots
  // that update recomputed, a CTA none of whose rows is in it reads nothing
  // the update writes and starts scoring without waiting; CTA x = 0 of each
  // token then waits at its end instead, so this kernel still completes after
  // the update and every later kernel that waits on it is ordered after both.
  bool must_wait = true;
  if (use_hint) {
    int hit = 0;
    for (int i = tid; i < nrows; i += kScoreThreads) {
      const int sl = s_slot[i];
      for (int e = 0; e < a.n_recomputed; ++e) hit |= (s_rec[e] == sl);
    }
    must_wait = __syncthreads_or(hit) != 0;
  } else if (query_hint) {
    // any token of this sequence whose own block lies in this CTA's range
    const int seq = a.tok_seq[t];
    int hit = 0;
    for (int u = tid; u < a.n_tokens; u += kScoreThreads) {
      const int64_t jb = (int64_t)a.tok_pos[u] / a.r;
      hit |= (a.tok_seq[u] == seq && jb >= j0 && jb < j1) ? 1 : 0;
    }
    must_wait = __syncthreads_or(hit) != 0;
  }
  if (kTopk) QSA_TS(index, 1);
  if (must_wait) grid_dep_wait();
  grid_dep_launch();
  if (kTopk) QSA_TS(index, 2);
  if (!kTopk) {
    const int64_t f1 = min(a.max_blocks, j0 + chunk);
    for (int64_t j = max((int64_t)nb, j0) + tid; j < f1; j += kScoreThreads) srow[j] = -INFINITY;
  } else {
    // the selection expands its chosen blocks through their table rows: ask
    // L2 for the rows of this CTA's blocks now (16 bytes each, ~3 % of the
    // pooled bytes), so the expansion does not wait on DRAM
    for (int i = tid; i < nrows; i += kScoreThreads) {
      const int sl = s_slot[i];
      if (sl >= 0 && sl < a.n_slots)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(a.blk_cells + (int64_t)sl * a.r));
    }
  }

  // ---- this warp's rows [r0, r1), 4 per stage
  const int per_w = (int)round_up(ceil_div(nrows, kScoreWarps), 4);
  const int r0 = min(nrows, warp * per_w), r1 = min(nrows, r0 + per_w);
  const int nst = (int)ceil_div(r1 - r0, 4);
  float* wring = ring + warp * (kRingStages * 4 * kIdxDim);
  // lane l copies row l / 8 of a stage: chunk k * 8 + l % 8 (16 bytes) for
  // k = 0..3, so each copy instruction moves one whole 128-byte line of each
  // of the 4 rows and every lane computes one row address per stage
  auto issue = [&](int st) {
    if (st < nst) {
      const int i = r0 + st * 4 + grp;
      const int slot = i < r1 ? s_slot[i] : -1;
      const bool ok = slot >= 0 && slot < a.n_slots;
      float* dst = wring + ((st % kRingStages) * 4 + grp) * kIdxDim + sub * 4;
      const float* src = a.pooled + (int64_t)(ok ? slot : 0) * kIdxDim + sub * 4;
#pragma unroll
      for (int k = 0; k < 4; ++k) ring_copy16(dst + k * 32, src + k * 32, ok);
    }
    asm volatile("cp.async.commit_group;\n" ::: "memory");
  };
#pragma unroll
  for (int st = 0; st < kRingStages - 1; ++st) issue(st);

  // Scores are collected 32 rows at a time (8 stages): lane L keeps the score
  // of group L % 4 of stage L / 4 of the batch, so the score stores and the
  // histogram updates run once per 32 rows with every lane busy.
  float hold = 0.f;
  for (int it = 0; it < nst; ++it) {
    issue(it + kRingStages - 1);
    asm volatile("cp.async.wait_group %0;\n" ::"n"(kRingStages - 1) : "memory");
    __syncwarp();
    const float4* row = reinterpret_cast<const float4*>(wring + ((it % kRingStages) * 4 + grp) * kIdxDim);
    float4 kv[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) kv[k] = row[k * 8 + sub];
    // per head: even and odd dims accumulate in the two halves of a packed
    // fp32 FMA, then add
    float acc[kIdxHeads];
#pragma unroll
    for (int h = 0; h < kIdxHeads; ++h) {
      float2 e = make_float2(0.f, 0.f);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        e = ffma2(make_float2(qv[h][k].x, qv[h][k].y), make_float2(kv[k].x, kv[k].y), e);
        e = ffma2(make_float2(qv[h][k].z, qv[h][k].w), make_float2(kv[k].z, kv[k].w), e);
      }
      acc[h] = e.x + e.y;
    }
    // reduce-scatter over the 8 lanes of the group
    float k0 = bit2 ? acc[2] : acc[0], k1 = bit2 ? acc[3] : acc[1];
    const float s0 = bit2 ? acc[0] : acc[2], s1 = bit2 ? acc[1] : acc[3];
    k0 += __shfl_xor_sync(kFull, s0, 4);
    k1 += __shfl_xor_sync(kFull, s1, 4);
    float d = bit1 ? k1 : k0;
    d += __shfl_xor_sync(kFull, bit1 ? k0 : k1, 2);
    d += __shfl_xor_sync(kFull, d, 1);               // head 2*bit2 + bit1, all 128 dims
    float v = wh * fmaxf(d, 0.f);
    v += __shfl_xor_sync(kFull, v, 2);
    v += __shfl_xor_sync(kFull, v, 4);               // sum over the 4 heads, on every lane of the group
    const float vg = __shfl_sync(kFull, v, (lane & 3) * 8);
    if ((it & 7) == (lane >> 2)) hold = vg;
    __syncwarp();   // every lane is done with this stage before it is refilled
    if ((it & 7) == 7 || it == nst - 1) {
      const int st = it - (it & 7) + (lane >> 2);
      const int i = r0 + st * 4 + (lane & 3);
      if (st <= it && i < r1) {
        const int slot = s_slot[i];
        const bool ok = slot >= 0 && slot < a.n_slots;
        if (!ok) atomicOr(err, kErrSlot);
        const float sc = ok ? hold : -INFINITY;
        srow[j0 + i] = sc;
        if (kTopk) {
          const unsigned bin = score_key(sc) >> (32 - kHistBits);
          if (atomicAdd(&s_hist[bin], 1u) == 0u) s_touched[atomicAdd(&s_ntouched, 1u)] = (unsigned short)bin;
        }
      }
    }
  }
  asm volatile("cp.async.wait_group 0;\n" ::: "memory");
  if (kTopk) {
    QSA_TS(index, 3);
    __syncthreads();
    const unsigned nt = s_ntouched;
    for (unsigned i = tid; i < nt; i += kScoreThreads) {
      const unsigned b = s_touched[i];
      atomicAdd(ghist + b, s_hist[b]);
    }
  }
  // the kernel completes only after its predecessor (see above)
  if (!must_wait && blockIdx.x == 0) grid_dep_wait();
}

// ------------------------------------------------------------- k_score_tc
// Token-tiled scores on the tensor cores: D[row][4u + h] = pooled[row] .
// q_idx[t0 + u][h] for M = 128 block rows x N = 128 (32 tokens x 4 heads) x
// K = 128 dims, tcgen05 kind::tf32 with each fp32 operand split in two,
// x = t(x) + l(x), t(x) = x with its low 13 mantissa bits cleared (a TF32
// value) and l(x) = x - t(x) rounded to TF32:
//   D = t(A) t(B) + t(A) l(B) + l(A) t(B),
// every product exact in fp32, accumulated in fp32 in tensor memory.  The
// omitted l(A) l(B) and the rounding of l(.) are below 2^-21 of each product,
// under the rounding of an fp32 FMA chain over 128 terms.
//
// The split query tile [t(B); l(B)] (256 rows) stays in shared memory; the
// split rows go to tensor memory, so per 8-dim K step three MMAs with
// N = 128 and A read from tensor memory accumulate t(A) t(B), t(A) l(B) and
// l(A) t(B) into the same columns, and the MMAs read only B from shared
// memory.  One CTA
// per SM, 288 threads in three roles that meet only at mbarriers (every wait
// bounded):
//   warps 0-3  gather: thread p takes row p of the tile, 32 dims (one
//              128-byte line) per chunk, loaded into registers three chunks
//              ahead, split into t(A) and l(A) and stored into its lane of
//              one of four tensor-memory stages;
//   warp 8     issues the MMAs of a chunk when its stage is full and frees
//              the stage (tcgen05.commit) when they complete; tensor memory
//              holds two accumulators so a row tile's MMAs run while the
//              previous tile is read out;
//   warps 4-7  epilogue: thread e reads row e of the accumulator and writes
//              the scores of the tile's tokens.
constexpr int kTcTok = 32;                       // tokens per tile
constexpr int kTcN = 4 * kTcTok;                 // B rows of t(B) (and of l(B))
constexpr int kTcKC = 32;                        // dims per chunk: one 128-byte swizzle atom of fp32
constexpr int kTcChunks = kIdxDim / kTcKC;       // 4
constexpr int kTcStages = 4;                     // tensor-memory stages of the split rows
constexpr int kTcAhead = 3;                      // chunks of a row in registers ahead of their store
constexpr int kTcGather = 128;                   // warps 0-3
constexpr int kTcEpi = 128;                      // warps 4-7
constexpr int kTcThreads = kTcGather + kTcEpi + 32;
constexpr int kTcMaxSeq = kTcTok;                // distinct sequences in a tile
constexpr uint32_t kTcOffB = 0;                                // [t(B); l(B)]: 256 rows x 128 fp32
constexpr uint32_t kTcBBytes = 2u * kTcN * 512u;               // 128 KB
constexpr uint32_t kTcOffBar = kTcOffB + kTcBBytes;
constexpr uint32_t kTcNumBars = 2 * kTcStages + 4;             // full, empty per stage; acc full, acc empty x 2
constexpr uint32_t kTcOffTmem = kTcOffBar + 8 * kTcNumBars;
constexpr size_t kTcSmem = kTcOffTmem + 16 + 1024;             // + alignment slack
// tensor memory: accumulators in columns [0, 128) and [128, 256); stage q's
// t(A) in [256 + 64 q, 256 + 64 q + 32), its l(A) in the next 32 columns
constexpr uint32_t kTcTmemCols = 512;
constexpr uint32_t kTcTmemA = 256;
// kind::tf32: fp32 accumulate, A and B TF32, both K-major, M = 128, N = 128
constexpr uint32_t kTcIdesc128 = (1u << 4) | (2u << 7) | (2u << 10) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
static_assert(kTcSmem + 1024 <= 227u * 1024u, "token-tiled scorer shared memory");
static_assert(kTcTmemA + 64u * kTcStages <= kTcTmemCols, "token-tiled scorer tensor memory");
static_assert(kTcStages == kTcChunks, "a row tile's chunks map onto the stages one to one");

__device__ __forceinline__ float tf32_trunc(float x) { return __uint_as_float(__float_as_uint(x) & 0xffffe000u); }
// x rounded to the nearest TF32 value (ties away from zero)
__device__ __forceinline__ float tf32_round(float x) {
  return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xffffe000u);
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}

template <bool kTopk>
__global__ void __launch_bounds__(kTcThreads, 1)
k_score_tc(const IndexArgs a, float* __restrict__ scores, unsigned* err) {
  extern __shared__ unsigned char tc_smem_raw[];
  const uint32_t raw_s = smem_u32(tc_smem_raw);
  const uint32_t base_s = (raw_s + 1023u) & ~1023u;
  unsigned char* base = tc_smem_raw + (base_s - raw_s);
  __shared__ int s_seq[kTcTok], s_nb[kTcTok];
  __shared__ int64_t s_off[kTcTok];
  __shared__ float s_w[kTcTok][kIdxHeads];
  // the tile's distinct sequences: token mask, blocks, list offset, and the
  // prefix of this CTA's row tiles over them
  __shared__ unsigned s_dmask[kTcMaxSeq];
  __shared__ int s_dnb[kTcMaxSeq], s_dpre[kTcMaxSeq + 1];
  __shared__ int64_t s_doff[kTcMaxSeq];
  __shared__ int s_nd;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t0 = blockIdx.y * kTcTok;
  const uint32_t bar_full = base_s + kTcOffBar, bar_empty = bar_full + 8 * kTcStages;
  const uint32_t bar_accf = bar_empty + 8 * kTcStages, bar_acce = bar_accf + 16;

  // ---- before the wait: tensor memory, barriers, tokens, the split query tile
  if (warp == 0) tmem_alloc(base_s + kTcOffTmem, kTcTmemCols);
  if (tid == 0) {
    for (int q = 0; q < kTcStages; ++q) {
      mbar_init(bar_full + 8 * q, kTcGather);
      mbar_init(bar_empty + 8 * q, 1);
    }
    for (int q = 0; q < 2; ++q) {
      mbar_init(bar_accf + 8 * q, 1);
      mbar_init(bar_acce + 8 * q, kTcEpi);
    }
  }
  if (tid < kTcTok) {
    const int t = t0 + tid;
    int seq = -1, nb = 0;
    int64_t off = 0;
    if (t < a.n_tokens) {
      const Tok tk = token_geometry(a, t, err, blockIdx.x == 0);
      if (tk.ok) {
        seq = a.tok_seq[t];
        nb = tk.nb;
        off = tk.off;
      }
    }
    s_seq[tid] = seq;
    s_nb[tid] = nb;
    s_off[tid] = off;
#pragma unroll
    for (int h = 0; h < kIdxHeads; ++h) s_w[tid][h] = t < a.n_tokens ? a.w_idx[(int64_t)t * kIdxHeads + h] : 0.f;
  }
  for (int i = tid; i < kTcN * (kIdxDim / 4); i += kTcThreads) {
    const int n = i / (kIdxDim / 4), c16 = i % (kIdxDim / 4);
    const int t = t0 + (n >> 2);
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (t < a.n_tokens)
      v = __ldg(reinterpret_cast<const float4*>(a.q_idx + ((int64_t)t * kIdxHeads + (n & 3)) * kIdxDim) + c16);
    const float4 vt = make_float4(tf32_trunc(v.x), tf32_trunc(v.y), tf32_trunc(v.z), tf32_trunc(v.w));
    const float4 vl = make_float4(tf32_round(v.x - vt.x), tf32_round(v.y - vt.y), tf32_round(v.z - vt.z),
                                  tf32_round(v.w - vt.w));
    *reinterpret_cast<float4*>(base + kTcOffB + sw128(2u * kTcN, (uint32_t)n, (uint32_t)c16)) = vt;
    *reinterpret_cast<float4*>(base + kTcOffB + sw128(2u * kTcN, (uint32_t)(kTcN + n), (uint32_t)c16)) = vl;
  }
  __syncthreads();
  if (tid == 0) {
    // distinct sequences in order of first token; this CTA's row tiles of
    // each are rt = blockIdx.x, blockIdx.x + gridDim.x, ...
    unsigned done = 0;
    for (int v = 0; v < kTcTok; ++v)
      if (s_seq[v] < 0) done |= 1u << v;
    int nd = 0, pre = 0;
    while (done != 0xffffffffu) {
      const int first = __ffs(~done) - 1;
      const int seq = s_seq[first];
      unsigned mask = 0;
      int nbmax = 0;
      for (int v = 0; v < kTcTok; ++v)
        if (s_seq[v] == seq) {
          mask |= 1u << v;
          nbmax = max(nbmax, s_nb[v]);
        }
      done |= mask;
      const int tiles = (nbmax + 127) / 128;
      s_dmask[nd] = mask;
      s_dnb[nd] = nbmax;
      s_doff[nd] = s_off[first];
      s_dpre[nd] = pre;
      pre += tiles > (int)blockIdx.x ? (tiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
      ++nd;
    }
    s_dpre[nd] = pre;
    s_nd = nd;
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<const uint32_t*>(base + kTcOffTmem);
  const int nd = s_nd;
  const int n_items = s_dpre[nd];
  // item k of this CTA: (distinct sequence, row tile)
  auto item_at = [&](int k, int* d, int* rt) {
    int x = 0;
    while (x + 1 < nd && s_dpre[x + 1] <= k) ++x;
    *d = x;
    *rt = (int)blockIdx.x + (k - s_dpre[x]) * (int)gridDim.x;
  };

  // ---- pooled rows are written by the preceding pool update / append
  grid_dep_wait();
  grid_dep_launch();

  bool timed_out = false;
  const int n_chunks = n_items * kTcChunks;
  if (warp < 4) {
    // ---- gather and split: thread p owns row p of every tile.  Chunk q's
    // line is loaded three chunks ahead into registers; once its stage is
    // free it is split and stored into the thread's lane of the stage, and
    // the load of chunk q + 3 takes its registers.  (Staging the lines
    // through a 5-deep cp.async ring in shared memory instead was measured
    // slower: 224 against 184 us for the 512-token ubatch.)
    const int p = tid;
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    const bool pooled32 = (reinterpret_cast<uintptr_t>(a.pooled) & 31u) == 0;   // else 16-byte loads
    auto row_slot = [&](int k) {
      int d, rt;
      item_at(k, &d, &rt);
      const int64_t j = (int64_t)rt * 128 + p;
      int sl = -1;
      if (j < s_dnb[d]) {
        sl = a.seq_blk_slots[s_doff[d] + j];
        if (sl < 0 || sl >= a.n_slots) {
          atomicOr(err, kErrSlot);
          sl = -1;
        }
      }
      return sl;
    };
    // the slot of row p in the item whose chunks are being loaded, and in
    // the next one (loaded one item ahead, so no load waits on it)
    int sl_cur = -1, sl_next = n_items > 0 ? row_slot(0) : -1;
    auto load = [&](int q, float4 (&r)[8]) {
      const int k = q / kTcChunks, c = q % kTcChunks;
      if (c == 0) {
        sl_cur = sl_next;
        sl_next = k + 1 < n_items ? row_slot(k + 1) : -1;
      }
      if (sl_cur >= 0 && pooled32) {
        // 32-byte loads: one L1 sector per load
        const float* src = a.pooled + (int64_t)sl_cur * kIdxDim + c * kTcKC;
#pragma unroll
        for (int m = 0; m < kTcKC / 8; ++m)
          asm volatile("ld.global.nc.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
                       : "=f"(r[2 * m].x), "=f"(r[2 * m].y), "=f"(r[2 * m].z), "=f"(r[2 * m].w),
                         "=f"(r[2 * m + 1].x), "=f"(r[2 * m + 1].y), "=f"(r[2 * m + 1].z), "=f"(r[2 * m + 1].w)
                       : "l"(src + 8 * m));
      } else if (sl_cur >= 0) {
        const float4* src = reinterpret_cast<const float4*>(a.pooled + (int64_t)sl_cur * kIdxDim + c * kTcKC);
#pragma unroll
        for (int m = 0; m < kTcKC / 4; ++m) r[m] = __ldg(src + m);
      } else {
#pragma unroll
        for (int m = 0; m < kTcKC / 4; ++m) r[m] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    };
    auto store = [&](int q, float4 (&r)[8]) {
      const int st = q % kTcStages, use = q / kTcStages;
      if (!mbar_wait(bar_empty + 8 * st, (uint32_t)((use & 1) ^ 1))) timed_out = true;
      tc_fence_after();
      const uint32_t col = tmem + lane_base + kTcTmemA + 64u * (uint32_t)st;
      {
        uint32_t v[kTcKC];   // t(A)
#pragma unroll
        for (int m = 0; m < kTcKC / 4; ++m) {
          v[4 * m] = __float_as_uint(tf32_trunc(r[m].x));
          v[4 * m + 1] = __float_as_uint(tf32_trunc(r[m].y));
          v[4 * m + 2] = __float_as_uint(tf32_trunc(r[m].z));
          v[4 * m + 3] = __float_as_uint(tf32_trunc(r[m].w));
        }
        tmem_st32(col, v);
      }
      {
        uint32_t v[kTcKC];   // l(A)
#pragma unroll
        for (int m = 0; m < kTcKC / 4; ++m) {
          v[4 * m] = __float_as_uint(tf32_round(r[m].x - tf32_trunc(r[m].x)));
          v[4 * m + 1] = __float_as_uint(tf32_round(r[m].y - tf32_trunc(r[m].y)));
          v[4 * m + 2] = __float_as_uint(tf32_round(r[m].z - tf32_trunc(r[m].z)));
          v[4 * m + 3] = __float_as_uint(tf32_round(r[m].w - tf32_trunc(r[m].w)));
        }
        tmem_st32(col + 32u, v);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar_full + 8 * st);
      if (q + kTcAhead < n_chunks) load(q + kTcAhead, r);
    };
    float4 r0[8], r1[8], r2[8];
    static_assert(kTcAhead == 3, "three register buffers");
    if (0 < n_chunks) load(0, r0);
    if (1 < n_chunks) load(1, r1);
    if (2 < n_chunks) load(2, r2);
    for (int q = 0; q < n_chunks; q += 3) {
      store(q, r0);
      if (q + 1 < n_chunks) store(q + 1, r1);
      if (q + 2 < n_chunks) store(q + 2, r2);
    }
  } else if (warp == 8) {
    // ---- the MMAs, issued by one thread
    if (lane == 0) {
      for (int q = 0; q < n_chunks; ++q) {
        const int k = q / kTcChunks, c = q % kTcChunks, st = q % kTcStages, use = q / kTcStages;
        const int b = k & 1;
        if (c == 0 && !mbar_wait(bar_acce + 8 * b, (uint32_t)(((k >> 1) & 1) ^ 1))) timed_out = true;
        if (!mbar_wait(bar_full + 8 * st, (uint32_t)(use & 1))) timed_out = true;
        tc_fence_after();
        const uint32_t a_t = tmem + kTcTmemA + 64u * (uint32_t)st;
        const uint32_t d = tmem + (uint32_t)b * 128u;
#pragma unroll
        for (int kk = 0; kk < kTcKC / 8; ++kk) {
          const int kg = c * (kTcKC / 8) + kk;            // K step of 8 dims over the whole row
          const uint32_t bo = base_s + kTcOffB + (uint32_t)(kg >> 2) * (2u * kTcN * 128u) + (uint32_t)(kg & 3) * 32u;
          const uint64_t bt = smem_desc(bo, 16, 1024);                     // t(B): rows 0-127
          const uint64_t bl = smem_desc(bo + (uint32_t)kTcN * 128u, 16, 1024);   // l(B): rows 128-255
          mma_tf32_ts(d, a_t + 8u * kk, bt, kTcIdesc128, (c | kk) ? 1u : 0u);   // t(A) t(B)
          mma_tf32_ts(d, a_t + 8u * kk, bl, kTcIdesc128, 1u);                   // + t(A) l(B)
          mma_tf32_ts(d, a_t + 32u + 8u * kk, bt, kTcIdesc128, 1u);             // + l(A) t(B)
        }
        mma_commit(bar_empty + 8 * st);
        if (c == kTcChunks - 1) mma_commit(bar_accf + 8 * b);
      }
    }
    __syncwarp();
  } else {
    // ---- epilogue: thread e reads row e of the accumulator
    const int e = tid - kTcGather;
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    for (int k = 0; k < n_items; ++k) {
      int d, rt;
      item_at(k, &d, &rt);
      const int64_t j = (int64_t)rt * 128 + e;
      const unsigned mask = s_dmask[d];
      // the row's slot (its validity), loaded before the accumulator is ready
      bool rok = false;
      if (j < s_dnb[d]) {
        const int sl = a.seq_blk_slots[s_doff[d] + j];
        rok = sl >= 0 && sl < a.n_slots;
      }
      const int b = k & 1;
      if (!mbar_wait(bar_accf + 8 * b, (uint32_t)((k >> 1) & 1))) timed_out = true;
      tc_fence_after();
#pragma unroll
      for (int gq = 0; gq < kTcN / 32; ++gq) {
        uint32_t r0[16], r1[16];
        tmem_ld16_nowait(tmem + lane_base + (uint32_t)b * 128u + (uint32_t)(32 * gq), r0);
        tmem_ld16_nowait(tmem + lane_base + (uint32_t)b * 128u + (uint32_t)(32 * gq + 16), r1);
        tmem_wait_ld();
#pragma unroll
        for (int uu = 0; uu < 8; ++uu) {
          const int u = gq * 8 + uu;
          if (((mask >> u) & 1u) && j < s_nb[u]) {
            const uint32_t* rr = uu < 4 ? r0 + 4 * uu : r1 + 4 * (uu - 4);
            float v[kIdxHeads];
#pragma unroll
            for (int h = 0; h < kIdxHeads; ++h) v[h] = s_w[u][h] * fmaxf(__uint_as_float(rr[h]), 0.f);
            scores[(int64_t)(t0 + u) * a.max_blocks + j] = rok ? (v[0] + v[1]) + (v[2] + v[3]) : -INFINITY;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(bar_acce + 8 * b);
    }
  }
  if (!kTopk) {
    // -inf for the blocks of this CTA's row tiles a token does not see
    __syncthreads();
    const int64_t all_tiles = ceil_div(a.max_blocks, 128);
    for (int64_t rt = blockIdx.x; rt < all_tiles; rt += gridDim.x)
      for (int i = tid; i < kTcTok * 128; i += kTcThreads) {
        const int v = i / 128;
        const int64_t j = rt * 128 + i % 128;
        const int t = t0 + v;
        if (t < a.n_tokens && j < a.max_blocks && j >= s_nb[v]) scores[(int64_t)t * a.max_blocks + j] = -INFINITY;
      }
  }
  if (timed_out) atomicOr(err, kErrTimeout);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTcTmemCols);
}

// ------------------------------------------------------------------ k_hist
// Threshold-bin histogram of the scores written by k_score_tc (k_score builds
// it while scoring): a CTA takes kHistChunk blocks of one token, counts
// them in shared memory (reductions whose result is not read) and adds its
// non-zero bins to the token's histogram.
constexpr int kHistChunk = 8192;
static_assert(kHistChunk % 1024 == 0, "whole 16-byte loads per thread");

__global__ void __launch_bounds__(256)
k_hist(const IndexArgs a, void* ws, const float* __restrict__ scores) {
  __shared__ unsigned s_hist[kHistBins];
  const int t = blockIdx.y, tid = threadIdx.x;
  const Tok tk = token_geometry(a, t, nullptr, false);
  const int64_t j0 = (int64_t)blockIdx.x * kHistChunk;
  const int64_t j1 = min((int64_t)tk.nb, j0 + kHistChunk);
  for (int i = tid; i < kHistBins; i += 256) s_hist[i] = 0u;
  __syncthreads();
  grid_dep_wait();
  grid_dep_launch();
  const float* srow = scores + (int64_t)t * a.max_blocks;
  auto add = [&](float x) { atomicAdd(&s_hist[score_key(x) >> (32 - kHistBits)], 1u); };
  const float* cs = srow + j0;
  const int n = j1 > j0 ? (int)(j1 - j0) : 0;
  if ((reinterpret_cast<uintptr_t>(cs) & 15u) == 0) {
    // every load of the chunk in flight before the first atomic: 16-byte
    // loads, kHistChunk / 1024 per thread
    constexpr int kV = kHistChunk / 4 / 256;
    const int n4 = n >> 2;
    float4 v[kV];
#pragma unroll
    for (int k = 0; k < kV; ++k) {
      const int q = tid + 256 * k;
      v[k] = q < n4 ? __ldcg(reinterpret_cast<const float4*>(cs) + q) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < kV; ++k) {
      if (tid + 256 * k < n4) {
        add(v[k].x);
        add(v[k].y);
        add(v[k].z);
        add(v[k].w);
      }
    }
    for (int j = 4 * n4 + tid; j < n; j += 256) add(__ldcg(cs + j));
  } else {
    for (int j = tid; j < n; j += 256) add(__ldcg(cs + j));
  }
  __syncthreads();
  unsigned* gh = hist_of(ws, t);
  for (int i = tid; i < kHistBins; i += 256) {
    const unsigned c = s_hist[i];
    if (c) atomicAdd(gh + i, c);
  }
}

// ---------------------------------------------------------------- k_select
struct SelSmem {
  unsigned bitmap[kSelMaxWords];
  unsigned long long cand[kSelLocalCand];
  unsigned long long allc[kRankMax];     // every CTA's threshold-bin keys (rank path)
  unsigned hist[2][256];
  unsigned tot[256];
  unsigned warp_tmp[32];
  unsigned selc[kSelCluster];            // chosen threshold-bin keys per CTA (rank path)
  unsigned ncand;
  unsigned ncent;                        // keys gathered in CTA 0 (central path)
  unsigned ncut;                         // keys in the cut-off digit (central path)
  unsigned cbase;
  unsigned sel;
  int digit;
  unsigned above, eq;
  int thr, need, ncand_all;
  int tail_cells[8];
};

// kCtasPerSm = 2 (calls with more CTAs than SMs): two CTAs share an SM (64
// registers a thread) and the launch gives only the chosen-block list as
// dynamic shared memory, so the slot ids are read from global memory.
template <int kCtasPerSm>
__global__ void __launch_bounds__(kSelThreads, kCtasPerSm)
k_select(const IndexArgs a, void* ws, const float* __restrict__ scores,
         int32_t* __restrict__ cells, int32_t* __restrict__ count, unsigned* err) {
  QSA_TS_SCOPE_LAST(index, 19);
  __shared__ SelSmem sm;
  extern __shared__ __align__(16) int32_t s_dyn[];
  int* s_list = s_dyn;                     // chosen blocks of this CTA, ascending (kSelList)
  const int t = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = cluster_rank(), NC = cluster_size();
  const int r = a.r;
  const int B = a.n_sel_blocks;

  // ---- before the wait: geometry only (the token ids and block lists are
  // inputs no kernel of the library writes); the slot ids and the tail cells
  // are fetched after the wait, under the threshold search and the
  // classification, since the block table is written by the append that may
  // still be running when this kernel starts
  QSA_TS(index, 10);
  __shared__ int64_t s_off[kOffCache + 1];
  const int seq_t = a.tok_seq[t], pos_t = a.tok_pos[t];
  const bool offc = preload_offsets(a.seq_blk_off, a.n_seq, s_off);
  __syncthreads();
  const Tok tk = token_geometry(a, seq_t, pos_t, offc ? s_off : nullptr, err, false);
  const int nb = tk.nb;
  const int64_t per = round_up(ceil_div(nb > 0 ? nb : 1, (int64_t)NC), 32);
  const int64_t j0 = (int64_t)rank * per;
  const int64_t j1 = min((int64_t)nb, j0 + per);
  const int nwords = j1 > j0 ? (int)ceil_div(j1 - j0, 32) : 0;
  const int32_t* slots = a.seq_blk_slots + tk.off;
  int tail = 0;
  if (tk.ok && tk.nb == tk.nb_full) tail = tk.p + 1 - (int)(tk.nb_full * r);
  const bool tail_missing = tail > 0 && tk.nb_full >= tk.len;
  if (tail_missing) tail = 0;
  if (tid == 0) {
    sm.ncand = 0u;
    sm.ncent = 0u;
  }
  // this CTA's slot ids (an input): copied into shared memory now, waited for
  // before they are read; 16-byte copies where the list is aligned
  const bool slots_cached = kCtasPerSm == 1 && per <= kSelSlots;
  // s_slots[j - j0] = slots[j]; the array starts 0-3 ints past the list so
  // that it shares the block list's alignment modulo 16 bytes
  int32_t* s_slots = s_dyn + kSelList + ((reinterpret_cast<uintptr_t>(slots + j0) >> 2) & 3);
  if (slots_cached && j1 > j0) {
    const int64_t n = j1 - j0;
    const int64_t head = min(n, (int64_t)((4 - ((reinterpret_cast<uintptr_t>(slots + j0) >> 2) & 3)) & 3));
    const int64_t body = (n - head) / 4;
    if (tid < head) cp_async4(s_slots + tid, slots + j0 + tid);
    for (int64_t q = tid; q < body; q += kSelThreads) cp_async16_ptr(s_slots + head + 4 * q, slots + j0 + head + 4 * q);
    for (int64_t i = head + 4 * body + tid; i < n; i += kSelThreads) cp_async4(s_slots + i, slots + j0 + i);
  }
  asm volatile("cp.async.commit_group;\n" ::: "memory");
  // first half of a cluster barrier: the counters above are set before any
  // peer writes into this CTA (the matching wait follows the classification)
  cluster_arrive();

  QSA_TS(index, 11);
  grid_dep_wait();
  grid_dep_launch();
  QSA_TS(index, 12);
  // First batch of this warp's scores in flight while the threshold bin is
  // found from the token's histogram (every CTA of the cluster).
  unsigned* gh = hist_of(ws, t);
  // Word w of this CTA's range holds blocks j0 + 32 w + lane.  Words are
  // dealt round-robin to the warps (word warp + kSelWarps * b of a batch), so
  // a lane's b-th load of a batch sits kStride * b blocks past its first one
  // and exists while that offset is below the blocks left (rem); a range
  // holds at most kSelMaxWords words, so the offsets fit 32 bits.
  constexpr int kStride = kSelWarps * 32;
  const int nloc = j1 > j0 ? (int)(j1 - j0) : 0;
  const float* srow = scores + (int64_t)t * a.max_blocks;
  const float* lp = srow + j0 + warp * 32 + lane;
  int rem = nloc - (warp * 32 + lane);
  float v0[kSelBatch];
#pragma unroll
  for (int b = 0; b < kSelBatch; ++b) v0[b] = b * kStride < rem ? __ldcg(lp + b * kStride) : -INFINITY;
  // the tail block's slot (its member cells are copied once it arrives)
  const int tslot = (rank == 0 && tid < tail) ? slots[tk.nb_full] : -1;
  {
    constexpr int kPer = kHistBins / kSelThreads;   // 8 consecutive bins per thread, 2 vector loads
    static_assert(kPer == 8, "histogram split");
    unsigned h[kPer];
    unsigned sum = 0;
    {
      const uint4 q0 = __ldcg(reinterpret_cast<const uint4*>(gh + tid * kPer));
      const uint4 q1 = __ldcg(reinterpret_cast<const uint4*>(gh + tid * kPer) + 1);
      h[0] = q0.x, h[1] = q0.y, h[2] = q0.z, h[3] = q0.w;
      h[4] = q1.x, h[5] = q1.y, h[6] = q1.z, h[7] = q1.w;
    }
#pragma unroll
    for (int i = 0; i < kPer; ++i) sum += h[i];
    if (tid == 0) {
      sm.thr = -1;
      sm.need = 0;
      sm.ncand_all = 0;
    }
    unsigned cum = block_suffix_exclusive(sum, sm.warp_tmp);
    const unsigned Bu = (unsigned)B;
    if ((unsigned)nb > Bu) {
#pragma unroll
      for (int i = kPer - 1; i >= 0; --i) {
        const unsigned nxt = cum + h[i];
        if (cum < Bu && nxt >= Bu) {
          sm.thr = tid * kPer + i;
          sm.need = (int)(Bu - cum);
          sm.ncand_all = (int)h[i];
        }
        cum = nxt;
      }
    }
    __syncthreads();
  }
  const int thr = sm.thr, ncand_all = sm.ncand_all;
  const bool fast = thr < 0 || ncand_all <= kSelLocalCand;
  // Which path resolves the cut (central: CTA 0 ranks every CTA's
  // threshold-bin keys, orders and expands the chosen blocks alone)
  const bool central = nb <= kCentralBlocks && (thr < 0 || ncand_all <= kRankMax);
  if (tid < tail && rank == 0) {
    if (tslot >= 0 && tslot < a.n_slots) {
      cp_async4(&sm.tail_cells[tid], a.blk_cells + (int64_t)tslot * r + tid);
    } else {
      atomicOr(err, kErrSlot);
      sm.tail_cells[tid] = -1;
    }
  }
  asm volatile("cp.async.commit_group;\n" ::: "memory");

  // ---- phase A: classify this CTA's blocks, a warp's next batch of words
  // in flight while it classifies the current one
  const int nbatch = (int)ceil_div(nwords, kSelWarps * kSelBatch);
  const bool collect = fast && thr >= 0;
  for (int wb = 0; wb < nbatch; ++wb) {
    const int wbase = wb * kSelWarps * kSelBatch + warp;
    const int wrem = nwords - wbase;   // the warp's b-th word of the batch exists while kSelWarps * b < wrem
    const float* ln = lp + kStride * kSelBatch;
    const int rn = rem - kStride * kSelBatch;
    float vn[kSelBatch];
#pragma unroll
    for (int b = 0; b < kSelBatch; ++b) vn[b] = b * kStride < rn ? __ldcg(ln + b * kStride) : -INFINITY;
#pragma unroll
    for (int b = 0; b < kSelBatch; ++b) {
      if (kSelWarps * b >= wrem) break;
      const bool in = b * kStride < rem;
      const uint32_t key = score_key(v0[b]);
      const int bin = (int)(key >> (32 - kHistBits));
      const unsigned am = __ballot_sync(kFull, in && bin > thr);
      if (lane == 0) sm.bitmap[wbase + kSelWarps * b] = am;
      if (collect) {
        const bool isc = in && bin == thr;
        const unsigned cm = __ballot_sync(kFull, isc);
        if (cm) {
          const int leader = __ffs(cm) - 1;
          unsigned basei = 0;
          if (lane == leader) basei = atomicAdd(&sm.ncand, (unsigned)__popc(cm));
          basei = __shfl_sync(kFull, basei, leader);
          const unsigned idx = basei + __popc(cm & ((1u << lane) - 1u));
          const int64_t j = j0 + (int64_t)(wbase + kSelWarps * b) * 32 + lane;
          if (isc && idx < (unsigned)kSelLocalCand) sm.cand[idx] = cand_key(key, j);
        }
      }
    }
#pragma unroll
    for (int b = 0; b < kSelBatch; ++b) v0[b] = vn[b];
    lp = ln;
    rem = rn;
  }
  __syncthreads();
  QSA_TS(index, 13);
  cluster_wait();

  if (central) {
    // ---- central path: every CTA sends its bitmap words and threshold-bin
    // keys into CTA 0's shared memory; CTA 0 ranks the keys, orders and
    // expands the chosen blocks alone.
    if (rank != 0)
      for (int w = tid; w < nwords; w += kSelThreads)
        st_dsmem_u32(dsmem_addr(&sm.bitmap[(int)(j0 >> 5) + w], 0), sm.bitmap[w]);
    const unsigned ncl = min(sm.ncand, (unsigned)kSelLocalCand);
    if (tid == 0) sm.cbase = ncl ? atom_add_dsmem(dsmem_addr(&sm.ncent, 0), ncl) : 0u;
    __syncthreads();
    for (unsigned i = tid; i < ncl; i += kSelThreads) {
      const unsigned at = sm.cbase + i;
      if (at < (unsigned)kRankMax) st_dsmem_u64(dsmem_addr(&sm.allc[at], 0), sm.cand[i]);
    }
    cluster_sync();   // everything has landed in CTA 0
    if (rank != 0) return;
    QSA_TS(index, 14);
    const unsigned nall = min(sm.ncent, (unsigned)kRankMax);
    if (thr >= 0) {
      // One 8-bit digit below the bin (key bits 19..12) splits the keys; keys
      // in higher sub-bins are chosen, the cut-off sub-bin (usually one or
      // two keys) is ranked exactly by full key.
      unsigned need = (unsigned)sm.need;
      unsigned* hh = sm.hist[0];
      if (tid < 256) hh[tid] = 0u;
      __syncthreads();
      for (unsigned i = tid; i < nall; i += kSelThreads) atomicAdd(&hh[(unsigned)(sm.allc[i] >> 48) & 255u], 1u);
      __syncthreads();
      QSA_TS(index, 24);
      if (warp == 0) {
        unsigned hv[8], sum = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          hv[i] = hh[lane * 8 + i];
          sum += hv[i];
        }
        unsigned x = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const unsigned y = __shfl_down_sync(kFull, x, o);
          if (lane + o < 32) x += y;
        }
        unsigned cum = x - sum;
#pragma unroll
        for (int i = 7; i >= 0; --i) {
          const unsigned nxt = cum + hv[i];
          if (cum < need && nxt >= need) {
            sm.digit = lane * 8 + i;
            sm.above = cum;
          }
          cum = nxt;
        }
      }
      if (tid == 0) sm.ncut = 0u;
      __syncthreads();
      QSA_TS(index, 25);
      const unsigned dstar = (unsigned)sm.digit;
      need -= sm.above;
      // keys above the cut-off digit are chosen; the digit's own keys (a few)
      // are gathered into this CTA's now unused candidate list and ranked
      // among themselves
      for (unsigned i = tid; i < nall; i += kSelThreads) {
        const unsigned long long c = sm.allc[i];
        const unsigned d = (unsigned)(c >> 48) & 255u;
        if (d > dstar) {
          const int64_t j = (int64_t)(~(uint32_t)(c >> 4));
          atomicOr(&sm.bitmap[j >> 5], 1u << (j & 31));
        } else if (d == dstar) {
          sm.cand[atomicAdd(&sm.ncut, 1u)] = c;     // ncut <= nall <= kRankMax < kSelLocalCand
        }
      }
      __syncthreads();
      QSA_TS(index, 26);
      const unsigned ncut = sm.ncut;
      for (unsigned i = tid; i < ncut; i += kSelThreads) {
        const unsigned long long c = sm.cand[i];
        unsigned above_c = 0;
        for (unsigned m = 0; m < ncut; ++m) above_c += sm.cand[m] > c ? 1u : 0u;
        if (above_c < need) {
          const int64_t j = (int64_t)(~(uint32_t)(c >> 4));
          atomicOr(&sm.bitmap[j >> 5], 1u << (j & 31));
        }
      }
    }
    __syncthreads();
    QSA_TS(index, 27);
    // ordered list of the chosen blocks (block prefix over the bitmap words)
    const int W = (int)ceil_div(nb, 32);
    const int wq = (int)ceil_div(W, kSelThreads);
    const int q0 = tid * wq, q1 = min(W, q0 + wq);
    unsigned mine = 0;
    for (int w = q0; w < q1; ++w) mine += __popc(sm.bitmap[w]);
    unsigned total_sel = 0;
    unsigned k = block_prefix_exclusive(mine, sm.warp_tmp, &total_sel);
    QSA_TS(index, 28);
    if (tid == 0) sm.sel = total_sel;
    for (int w = q0; w < q1; ++w) {
      unsigned bits = sm.bitmap[w];
      while (bits) {
        if (k < (unsigned)kSelList) s_list[k] = w * 32 + (__ffs(bits) - 1);
        ++k;
        bits &= bits - 1u;
      }
    }
    asm volatile("cp.async.wait_all;\n" ::: "memory");   // slot ids and tail cells
    __syncthreads();
    QSA_TS(index, 15);
    const unsigned total = sm.sel;
    const int nsel = (int)min(total, (unsigned)B);
    int32_t* crow = cells + (int64_t)t * a.cells_pitch;
    for (int i = tid; i < nsel; i += kSelThreads) {
      const int j = s_list[i];
      const int sl = (slots_cached && j < j1) ? s_slots[j] : slots[j];   // CTA 0's own range is cached
      const bool sok = sl >= 0 && sl < a.n_slots;
      if (!sok) atomicOr(err, kErrSlot);
      int cv[8];
#pragma unroll
      for (int m = 0; m < 8; ++m) cv[m] = (sok && m < r) ? a.blk_cells[(int64_t)sl * r + m] : -1;
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        if (m >= r) break;
        if (cv[m] < 0 || cv[m] >= a.n_cells) atomicOr(err, kErrCell);
        crow[(int64_t)i * r + m] = cv[m];
      }
    }
    if (tid < tail) crow[nsel * r + tid] = flag_cell(sm.tail_cells[tid], a.n_cells, err);
    if (tid == 0) {
      if (tail_missing) atomicOr(err, kErrBlockList);
      count[t] = nsel * r + tail;
    }
    for (int i = nsel * r + tail + tid; i < a.cells_pitch; i += kSelThreads) crow[i] = -1;
    for (int i = tid; i < kHistBins; i += kSelThreads) gh[i] = 0u;   // zero for the next call
    QSA_TS(index, 16);
    return;
  }

  const int wpt = (int)ceil_div(nwords, kSelThreads);
  const int w0 = tid * wpt, w1 = min(nwords, w0 + wpt);
  unsigned base = 0, total = 0;
  if (fast && ncand_all <= kRankMax) {
    // ---- phase B (rank path): every CTA pulls all threshold-bin keys and
    // ranks them directly; one cluster barrier gives the exact cut-off and
    // every CTA's output offset.
    unsigned mine = 0;
    for (int w = w0; w < w1; ++w) mine += __popc(sm.bitmap[w]);
    unsigned na = 0;
    block_prefix_exclusive(mine, sm.warp_tmp, &na);
    if (tid == 0) sm.sel = na;
    if (tid < kSelCluster) sm.selc[tid] = 0u;
    cluster_sync();   // keys and counts published; every CTA has read the histogram
    if (rank == 0)
      for (int i = tid; i < kHistBins; i += kSelThreads) gh[i] = 0u;   // zero for the next call
    unsigned nap[kSelCluster], ncp[kSelCluster];
#pragma unroll
    for (int p = 0; p < kSelCluster; ++p) {
      nap[p] = p < (int)NC ? ld_dsmem_u32(dsmem_addr(&sm.sel, p)) : 0u;
      ncp[p] = p < (int)NC ? min(ld_dsmem_u32(dsmem_addr(&sm.ncand, p)), (unsigned)kSelLocalCand) : 0u;
    }
    unsigned cpre[kSelCluster + 1];
    cpre[0] = 0;
#pragma unroll
    for (int p = 0; p < kSelCluster; ++p) cpre[p + 1] = cpre[p] + ncp[p];
    const unsigned nall = cpre[kSelCluster];
    for (unsigned i = tid; i < nall; i += kSelThreads) {
      int p = 0;
#pragma unroll
      for (int q = 1; q < kSelCluster; ++q) p += (i >= cpre[q]) ? 1 : 0;
      unsigned long long c;
      const uint32_t ad = dsmem_addr(&sm.cand[i - cpre[p]], p);
      asm("ld.shared::cluster.u64 %0, [%1];\n" : "=l"(c) : "r"(ad));
      sm.allc[i] = c;
    }
    __syncthreads();
    const unsigned need = (unsigned)sm.need;
    for (unsigned i = tid; i < nall; i += kSelThreads) {
      const unsigned long long c = sm.allc[i];
      unsigned above_c = 0;
      for (unsigned m = 0; m < nall; ++m) above_c += (sm.allc[m] > c) ? 1u : 0u;
      if (above_c < need) {
        int p = 0;
#pragma unroll
        for (int q = 1; q < kSelCluster; ++q) p += (i >= cpre[q]) ? 1 : 0;
        atomicAdd(&sm.selc[p], 1u);
        if (p == (int)rank) {
          const int64_t j = (int64_t)(~(uint32_t)(c >> 4));
          atomicOr(&sm.bitmap[(j - j0) >> 5], 1u << ((j - j0) & 31));
        }
      }
    }
    __syncthreads();
#pragma unroll
    for (int p = 0; p < kSelCluster; ++p) {
      const unsigned c = nap[p] + sm.selc[p];
      if (p < (int)rank) base += c;
      total += c;
    }
  } else {
    // ---- phase B (radix path): the `need` largest keys in the threshold bin,
    // one 8-bit digit per round, digit histograms summed over the cluster.
    if (thr >= 0) {
      const unsigned ncl = min(sm.ncand, (unsigned)kSelLocalCand);
      unsigned long long prefix = 0;
      int shift = 48;
      unsigned need = (unsigned)sm.need;
      int buf = 0;
      for (;;) {
        unsigned* hh = sm.hist[buf];
        if (tid < 256) hh[tid] = 0u;
        __syncthreads();
        if (fast) {
          for (unsigned i = tid; i < ncl; i += kSelThreads) {
            const unsigned long long c = sm.cand[i];
            if ((c >> (shift + 8)) == prefix) atomicAdd(&hh[(unsigned)(c >> shift) & 255u], 1u);
          }
        } else {
          for (int64_t j = j0 + tid; j < j1; j += kSelThreads) {
            const uint32_t key = score_key(__ldcg(srow + j));
            if ((int)(key >> (32 - kHistBits)) != thr) continue;
            const unsigned long long c = cand_key(key, j);
            if ((c >> (shift + 8)) == prefix) atomicAdd(&hh[(unsigned)(c >> shift) & 255u], 1u);
          }
        }
        cluster_sync();
        if (tid < 256) {
          unsigned v[kSelCluster];
#pragma unroll
          for (int p = 0; p < kSelCluster; ++p) v[p] = p < (int)NC ? ld_dsmem_u32(dsmem_addr(&hh[tid], p)) : 0u;
          unsigned sum = 0;
#pragma unroll
          for (int p = 0; p < kSelCluster; ++p) sum += v[p];
          sm.tot[tid] = sum;
        }
        __syncthreads();
        if (warp == 0) {
          unsigned hv[8], sum = 0;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            hv[i] = sm.tot[lane * 8 + i];
            sum += hv[i];
          }
          unsigned x = sum;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const unsigned y = __shfl_down_sync(kFull, x, o);
            if (lane + o < 32) x += y;
          }
          unsigned cum = x - sum;   // digits above this lane's 8
#pragma unroll
          for (int i = 7; i >= 0; --i) {
            const unsigned nxt = cum + hv[i];
            if (cum < need && nxt >= need) {
              sm.digit = lane * 8 + i;
              sm.above = cum;
              sm.eq = hv[i];
            }
            cum = nxt;
          }
        }
        __syncthreads();
        need -= sm.above;
        const unsigned eq = sm.eq;
        prefix = (prefix << 8) | (unsigned long long)sm.digit;
        buf ^= 1;
        QSA_TS(index, 20 + (shift == 48 ? 0 : (shift == 40 ? 1 : 2)));
        if (eq == need || shift == 0) break;
        shift -= 8;
      }
      // every key whose bits down to `shift` are >= prefix is chosen
      if (fast) {
        for (unsigned i = tid; i < ncl; i += kSelThreads) {
          const unsigned long long c = sm.cand[i];
          if ((c >> shift) >= prefix) {
            const int64_t j = (int64_t)(~(uint32_t)(c >> 4));
            atomicOr(&sm.bitmap[(j - j0) >> 5], 1u << ((j - j0) & 31));
          }
        }
      } else {
        for (int64_t j = j0 + tid; j < j1; j += kSelThreads) {
          const uint32_t key = score_key(__ldcg(srow + j));
          if ((int)(key >> (32 - kHistBits)) != thr) continue;
          if ((cand_key(key, j) >> shift) >= prefix) atomicOr(&sm.bitmap[(j - j0) >> 5], 1u << ((j - j0) & 31));
        }
      }
      __syncthreads();
    }
    unsigned mine = 0;
    for (int w = w0; w < w1; ++w) mine += __popc(sm.bitmap[w]);
    unsigned local_total = 0;
    block_prefix_exclusive(mine, sm.warp_tmp, &local_total);
    if (tid == 0) sm.sel = local_total;
    cluster_sync();   // every CTA has read the histogram and published its count
    if (rank == 0)
      for (int i = tid; i < kHistBins; i += kSelThreads) gh[i] = 0u;   // zero for the next call
    unsigned c[kSelCluster];
#pragma unroll
    for (int p = 0; p < kSelCluster; ++p) c[p] = p < (int)NC ? ld_dsmem_u32(dsmem_addr(&sm.sel, p)) : 0u;
#pragma unroll
    for (int p = 0; p < kSelCluster; ++p) {
      if (p < (int)rank) base += c[p];
      total += c[p];
    }
  }
  QSA_TS(index, 14);

  // ---- phase C: ordered expansion of this CTA's chosen blocks at `base`
  asm volatile("cp.async.wait_all;\n" ::: "memory");   // slot ids and tail cells
  __syncthreads();
  unsigned mine = 0;
  for (int w = w0; w < w1; ++w) mine += __popc(sm.bitmap[w]);
  unsigned local_total = 0;
  unsigned k = block_prefix_exclusive(mine, sm.warp_tmp, &local_total);
  QSA_TS(index, 15);
  int32_t* crow = cells + (int64_t)t * a.cells_pitch;
  if (local_total <= (unsigned)kSelList) {
    // list the chosen blocks in order, then expand one block per thread
    for (int w = w0; w < w1; ++w) {
      unsigned bits = sm.bitmap[w];
      while (bits) {
        s_list[k++] = (int)(w * 32 + (__ffs(bits) - 1));
        bits &= bits - 1u;
      }
    }
    __syncthreads();
    for (unsigned i = tid; i < local_total; i += kSelThreads) {
      const unsigned kk = base + i;
      if (kk >= (unsigned)B) continue;
      const int64_t j = j0 + s_list[i];
      const int sl = slots_cached ? s_slots[j - j0] : slots[j];
      const bool sok = sl >= 0 && sl < a.n_slots;
      if (!sok) atomicOr(err, kErrSlot);
      int cv[8];
#pragma unroll
      for (int m = 0; m < 8; ++m) cv[m] = (sok && m < r) ? a.blk_cells[(int64_t)sl * r + m] : -1;
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        if (m >= r) break;
        if (cv[m] < 0 || cv[m] >= a.n_cells) atomicOr(err, kErrCell);
        crow[(int64_t)kk * r + m] = cv[m];
      }
    }
  } else {
    k += base;
    for (int w = w0; w < w1; ++w) {
      unsigned bits = sm.bitmap[w];
      while (bits) {
        const int64_t j = j0 + (int64_t)w * 32 + (__ffs(bits) - 1);
        bits &= bits - 1u;
        if (k < (unsigned)B) {
          const int sl = slots_cached ? s_slots[j - j0] : slots[j];
          const bool sok = sl >= 0 && sl < a.n_slots;
          if (!sok) atomicOr(err, kErrSlot);
          for (int m = 0; m < r; ++m) {
            const int cidx = sok ? a.blk_cells[(int64_t)sl * r + m] : -1;
            if (cidx < 0 || cidx >= a.n_cells) atomicOr(err, kErrCell);
            crow[(int64_t)k * r + m] = cidx;
          }
        }
        ++k;
      }
    }
  }
  QSA_TS(index, 16);
  const int nsel = (int)min(total, (unsigned)B);
  if (rank == 0) {
    if (tid < tail) crow[nsel * r + tid] = flag_cell(sm.tail_cells[tid], a.n_cells, err);
    if (tid == 0) {
      if (tail_missing) atomicOr(err, kErrBlockList);
      count[t] = nsel * r + tail;
    }
  }
  for (int i = nsel * r + tail + (int)rank * kSelThreads + tid; i < a.cells_pitch; i += (int)NC * kSelThreads)
    crow[i] = -1;
  QSA_TS(index, 17);
  cluster_sync();   // peers read sm.sel and the digit histograms until here
  QSA_TS(index, 18);
}

// Rows per score CTA: every token's rows in one wave of 2 CTAs per SM, in
// whole warp stages (8 warps x 4 rows), at most kScoreChunkMax.
int score_chunk(int T, int64_t max_blocks, int sms) {
  const int64_t per = ceil_div(max_blocks * (int64_t)T, 2 * (int64_t)sms);
  int64_t chunk = round_up(per < 32 ? 32 : per, 32);
  if (chunk > kScoreChunkMax) chunk = kScoreChunkMax;
  return (int)chunk;
}

// CTAs per selection cluster.  One k_select<1> CTA fills an SM (512 threads,
// ~118 KB of shared memory).  A CTA costs about 5 us of its own (histogram,
// barriers, ordering, expansion) plus ~3 us per 62,500 blocks it classifies
// from L2, so few tokens take large clusters (one wave either way) and many
// tokens take small clusters (fewer waves); a CTA holds at most kSelMaxWords
// words.  The waves are counted at one CTA per SM also where the launch
// then takes k_select<2> (two per SM: a 512-token ubatch at 250,000 cells,
// one-CTA clusters, 68 us instead of 87 us with one per SM).
// 16-CTA clusters are taken only while the call's selection CTAs leave half
// of the SMs free: the attention CTAs launched behind the selection (one per
// SM) then become resident while it runs (measured: a 1-token step 0.3 us
// faster at 50k and 0.7 us at 250k than with 8-CTA clusters, a 5-token step
// 1 us slower).
int select_cluster(int T, int64_t max_blocks, int sms) {
  int best_nc = 8;
  double best = -1.0;
  for (int nc = kSelCluster; nc >= 1; nc >>= 1) {
    if (nc > 8 && (int64_t)T * nc > (int64_t)sms / 2) continue;
    if (ceil_div(max_blocks, (int64_t)nc) > (int64_t)kSelMaxWords * 32) break;
    const double waves = (double)ceil_div((int64_t)T * nc, (int64_t)(sms > 0 ? sms : 1));
    const double cost = waves * (5.0 + 3.0 * (double)max_blocks / 62500.0 / nc);
    if (best < 0.0 || cost < best) {
      best = cost;
      best_nc = nc;
    }
  }
  return best_nc;
}

// Per-device set-up of the index kernels (SM count, shared-memory limits):
// done once per device under a lock, then read from the published count.
cudaError_t index_setup(int* sms) {
  static std::atomic<int> sm_count[64];
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int n = sm_count[dev].load(std::memory_order_acquire);
  if (n > 0) {
    *sms = n;
    return cudaSuccess;
  }
  std::lock_guard<std::mutex> lock(mu);
  n = sm_count[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_score<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kScoreSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_score<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kScoreSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_select<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSelDynBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_select<1>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_select<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSelDynBytes2);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_select<2>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_score_tc<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTcSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_score_tc<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTcSmem);
    if (e != cudaSuccess) return e;
    if (n <= 0) return cudaErrorInvalidDevice;
    sm_count[dev].store(n, std::memory_order_release);
  }
  *sms = n;
  return cudaSuccess;
}

// Launches the token-tiled scores on the tensor cores: 32 tokens per CTA, one
// CTA per SM, the row tiles of each token tile dealt to sms / token tiles CTAs.
template <bool kTopk>
cudaError_t launch_tiled(const IndexArgs& a, float* scores, unsigned* err, cudaStream_t stream, int sms) {
  const int64_t row_tiles = ceil_div(a.max_blocks, 128);
  const int64_t tt = ceil_div(a.n_tokens, kTcTok);
  const int64_t x = std::min<int64_t>(row_tiles, std::max<int64_t>(1, (int64_t)sms / tt));
  return launch_pdl(k_score_tc<kTopk>, dim3((unsigned)std::max<int64_t>(x, 1), (unsigned)tt), dim3(kTcThreads),
                    kTcSmem, stream, 1, a, scores, err);
}

}  // namespace

// Up to 8 tokens, the per-token pass is faster even when they share a
// sequence: their CTAs read the same rows at about the same time and L2
// serves the repeats.
bool index_tiled(int n_tokens, int n_seq) { return n_tokens > 8 && n_tokens >= 2 * n_seq; }

// what an 8-CTA cluster holds (16-CTA clusters serve only calls of few tokens)
int64_t index_max_blocks_limit() { return (int64_t)8 * kSelMaxWords * 32; }

size_t index_workspace_bytes(int max_tokens, int64_t max_blocks) {
  static_assert(kCtrlBytes == (size_t)kIndexCtrlBytes, "workspace layout");
  return (size_t)index_workspace_bytes_max(max_tokens, max_blocks);
}

void index_workspace_zero_range(int n_tokens, int64_t, size_t* offset, size_t* bytes) {
  *offset = 0;
  *bytes = (size_t)n_tokens * kCtrlBytes;
}

cudaError_t launch_index_scores(const IndexArgs& a, float* scores, unsigned* err, cudaStream_t stream) {
  if (a.n_tokens <= 0 || a.max_blocks <= 0) return cudaSuccess;
  int sms = 0;
  cudaError_t e = index_setup(&sms);
  if (e != cudaSuccess) return e;
  if (index_tiled(a.n_tokens, a.n_seq)) return launch_tiled<false>(a, scores, err, stream, sms);
  const int chunk = score_chunk(a.n_tokens, a.max_blocks, sms);
  const dim3 grid((unsigned)ceil_div(a.max_blocks, chunk), (unsigned)a.n_tokens);
  return launch_pdl(k_score<false>, grid, dim3(kScoreThreads), kScoreSmem, stream, 1, a, (void*)nullptr, scores,
                    chunk, err);
}

cudaError_t launch_index_scores_topk(const IndexArgs& a, void* ws, unsigned* err, cudaStream_t stream) {
  if (a.n_tokens <= 0) return cudaSuccess;
  int sms = 0;
  cudaError_t e = index_setup(&sms);
  if (e != cudaSuccess) return e;
  IndexArgs b = a;
  b.max_blocks = a.max_blocks > 0 ? a.max_blocks : 1;
  float* sc = scores_of(ws, a.max_tokens);
  if (index_tiled(a.n_tokens, a.n_seq)) {
    // tokens sharing sequences: rows read once per token tile, then the
    // histogram from the written scores
    prof_before(kKScore, stream);
    e = launch_tiled<true>(b, sc, err, stream, sms);
    prof_after(kKScore, stream);
    if (e != cudaSuccess) return e;
    prof_before(kKHist, stream);
    const dim3 gh((unsigned)ceil_div(b.max_blocks, kHistChunk), (unsigned)a.n_tokens);
    e = launch_pdl(k_hist, gh, dim3(256), 0, stream, 1, b, ws, (const float*)sc);
    prof_after(kKHist, stream);
    return e;
  }
  const int chunk = score_chunk(a.n_tokens, b.max_blocks, sms);
  const dim3 g1((unsigned)ceil_div(b.max_blocks, chunk), (unsigned)a.n_tokens);
  prof_before(kKScore, stream);
  e = launch_pdl(k_score<true>, g1, dim3(kScoreThreads), kScoreSmem, stream, 1, b, ws, sc, chunk, err);
  prof_after(kKScore, stream);
  return e;
}

cudaError_t launch_index_topk(const IndexArgs& a, int32_t* cells, int32_t* count,
                              void* ws, unsigned* err, cudaStream_t stream) {
  if (a.n_tokens <= 0) return cudaSuccess;
  int sms = 0;
  cudaError_t e = launch_index_scores_topk(a, ws, err, stream);
  if (e != cudaSuccess) return e;
  e = index_setup(&sms);
  if (e != cudaSuccess) return e;
  IndexArgs b = a;
  b.max_blocks = a.max_blocks > 0 ? a.max_blocks : 1;
  float* sc = scores_of(ws, a.max_tokens);
  prof_before(kKFinal, stream);
  const int nc = select_cluster(a.n_tokens, b.max_blocks, sms);
  const dim3 grid((unsigned)nc, (unsigned)a.n_tokens);
  if ((int64_t)a.n_tokens * nc > (int64_t)sms)
    e = launch_pdl(k_select<2>, grid, dim3(kSelThreads), kSelDynBytes2, stream,
                   (unsigned)nc, b, ws, (const float*)sc, cells, count, err);
  else
    e = launch_pdl(k_select<1>, grid, dim3(kSelThreads), kSelDynBytes, stream,
                   (unsigned)nc, b, ws, (const float*)sc, cells, count, err);
  prof_after(kKFinal, stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace qsa
