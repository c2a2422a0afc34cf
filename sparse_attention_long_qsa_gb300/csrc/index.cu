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
// Kernels (one call = one memset + three launches, no host round trip):
//   k_score   streams the pooled rows of every visible block (the dominant
//             HBM traffic at long context: 512 B per block), writes fp32
//             scores and a 4096-bin histogram of the top 12 bits of the
//             order-preserving score key; the last CTA of a token (atomic
//             ticket, no waiting) locates the bin holding the B-th largest.
//   k_filter  re-reads the (L2-resident) scores: blocks above the threshold
//             bin go straight into a per-token selection bitmap (warp ballot,
//             one word per 32 blocks), blocks in the bin are appended to a
//             candidate list as unique 64-bit keys (score bits, ~index).
//   k_final   one CTA per token: radix select among the candidates (held in
//             registers) of exactly the number still needed - unique keys
//             make ties resolve to the lower block index - then an ordered
//             compaction of the bitmap (block ascending) that writes the
//             member cells of each chosen block and the tail cells.
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kScoreThreads = 256;
constexpr int kScoreWarps = kScoreThreads / 32;
constexpr int kScoreUnroll = 2;
// rows (blocks) one CTA covers per iteration: 8 warps x 4 rows x unroll
constexpr int kRowsPerIter = kScoreWarps * 4 * kScoreUnroll;
constexpr int kFilterThreads = 256;
constexpr int kFilterWordsPerCta = 32;
constexpr int kErrToken = 16;

struct Ws {
  float* scores;              // [T][max_blocks]
  unsigned* hist;             // [T][kHistBins]   } cleared
  unsigned* done;             // [T]              } by every
  unsigned* cand_cnt;         // [T]              } call
  int4* state;                // [T]              } {threshold bin, still needed, candidates, nb}
  unsigned* bitmap;           // [T][wpitch]
  unsigned long long* cand;   // [T][kCandCap]
  void* zero_base;
  size_t zero_bytes;
  int64_t wpitch;
  size_t total;
};

Ws carve(void* base, int T, int64_t max_blocks) {
  Ws w{};
  char* p = static_cast<char*>(base);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    char* q = p ? p + off : nullptr;
    off += (size_t)round_up((int64_t)bytes, 256);
    return q;
  };
  w.scores = reinterpret_cast<float*>(take(sizeof(float) * (size_t)T * (size_t)max_blocks));
  const size_t zoff = off;
  w.hist = reinterpret_cast<unsigned*>(take(sizeof(unsigned) * (size_t)T * kHistBins));
  w.done = reinterpret_cast<unsigned*>(take(sizeof(unsigned) * (size_t)T));
  w.cand_cnt = reinterpret_cast<unsigned*>(take(sizeof(unsigned) * (size_t)T));
  w.state = reinterpret_cast<int4*>(take(sizeof(int4) * (size_t)T));
  w.zero_base = p ? p + zoff : nullptr;
  w.zero_bytes = off - zoff;
  w.wpitch = round_up(ceil_div(max_blocks, 32), 4);
  w.bitmap = reinterpret_cast<unsigned*>(take(sizeof(unsigned) * (size_t)T * (size_t)w.wpitch));
  w.cand = reinterpret_cast<unsigned long long*>(take(sizeof(unsigned long long) * (size_t)T * kCandCap));
  w.total = off;
  return w;
}

// Per-token geometry, validated against the caller's bounds.
struct Tok {
  int64_t off;      // start of the sequence's block list
  int64_t len;      // its length
  int64_t nb_full;  // floor((p+1)/r)
  int nb;           // blocks scored: nb_full clamped to max_blocks and len
  int p;
  bool ok;
};

__device__ __forceinline__ Tok token_geometry(const IndexArgs& a, int t, unsigned* err, bool report) {
  Tok k{0, 0, 0, 0, -1, false};
  const int seq = a.tok_seq[t];
  const int p = a.tok_pos[t];
  if (seq < 0 || seq >= a.n_seq || p < 0) {
    if (report) atomicOr(err, (unsigned)kErrToken);
    return k;
  }
  k.off = a.seq_blk_off[seq];
  k.len = a.seq_blk_off[seq + 1] - k.off;
  k.p = p;
  k.nb_full = ((int64_t)p + 1) / a.r;
  int64_t nb = k.nb_full;
  if (nb > a.max_blocks) {
    if (report) atomicOr(err, kErrMaxBlocks);
    nb = a.max_blocks;
  }
  if (nb > k.len) {
    if (report) atomicOr(err, kErrBlockList);
    nb = k.len < 0 ? 0 : k.len;
  }
  k.nb = (int)nb;
  k.ok = true;
  return k;
}

// Exclusive sum over the threads with a HIGHER index (suffix sum) of a block.
__device__ __forceinline__ unsigned block_suffix_exclusive(unsigned v, unsigned* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  unsigned x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned y = __shfl_down_sync(kFull, x, o);
    if (lane + o < 32) x += y;
  }
  if (lane == 0) s_warp[warp] = x;
  __syncthreads();
  unsigned above = 0;
  for (int w = warp + 1; w < nw; ++w) above += s_warp[w];
  __syncthreads();
  return x - v + above;
}

// Exclusive prefix sum over the threads with a LOWER index; *total = block sum.
__device__ __forceinline__ unsigned block_prefix_exclusive(unsigned v, unsigned* s_warp, unsigned* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  unsigned x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  unsigned below = 0, all = 0;
  for (int w = 0; w < nw; ++w) {
    const unsigned s = s_warp[w];
    if (w < warp) below += s;
    all += s;
  }
  __syncthreads();
  *total = all;
  return x - v + below;
}

// Unique 56-bit selection key of a candidate inside the threshold bin: the 20
// low bits of the score key above the bitwise complement of the block index,
// so a larger key means a larger score, or an equal score at a lower index.
__device__ __forceinline__ unsigned long long cand_key(uint32_t key, int64_t j) {
  return ((unsigned long long)(key & 0xFFFFFu) << 36) |
         ((unsigned long long)(~(uint32_t)j) << 4);
}

// ----------------------------------------------------------------- k_score
// Rows are read by groups of 8 lanes: lane `sub` of a group holds dims
// {32k + 4 sub .. 32k + 4 sub + 3 : k = 0..3} of the row and of the 4 query
// heads (64 fp32 registers), so each group reads the 512-byte row as four
// fully used 128-byte lines.  The 4 head dot products are reduced across the
// group with a reduce-scatter (6 shuffles per row in all).
template <bool kTopk>
__global__ void __launch_bounds__(kScoreThreads, 2)
k_score(const IndexArgs a, float* __restrict__ scores, unsigned* __restrict__ hist,
        unsigned* __restrict__ done, int4* __restrict__ state, int chunk, unsigned* err) {
  __shared__ unsigned s_hist[kTopk ? kHistBins : 1];
  __shared__ unsigned s_warp[32];
  __shared__ int s_last;

  const int t = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const Tok tk = token_geometry(a, t, err, blockIdx.x == 0 && tid == 0);
  const int nb = tk.nb;
  float* srow = scores + (int64_t)t * a.max_blocks;
  const int64_t j0 = (int64_t)blockIdx.x * chunk;
  const int64_t j1 = min((int64_t)nb, j0 + chunk);

  if (kTopk) {
    for (int i = tid; i < kHistBins; i += kScoreThreads) s_hist[i] = 0u;
    __syncthreads();
  } else {
    const int64_t f1 = min(a.max_blocks, j0 + chunk);
    for (int64_t j = max((int64_t)nb, j0) + tid; j < f1; j += kScoreThreads) srow[j] = -INFINITY;
  }

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
  const int32_t* slots = a.seq_blk_slots + tk.off;

  for (int64_t base = j0 + warp * 4 * kScoreUnroll; base < j1; base += kRowsPerIter) {
    float4 kv[kScoreUnroll][4];
    bool ok[kScoreUnroll], live[kScoreUnroll];
#pragma unroll
    for (int u = 0; u < kScoreUnroll; ++u) {
      const int64_t j = base + u * 4 + grp;
      live[u] = j < j1;
      int slot = live[u] ? __ldg(slots + j) : 0;
      ok[u] = live[u] && slot >= 0 && slot < a.n_slots;
      if (live[u] && !ok[u] && sub == 0) atomicOr(err, kErrSlot);
      const float4* row = reinterpret_cast<const float4*>(a.pooled + (int64_t)(ok[u] ? slot : 0) * kIdxDim);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        kv[u][k] = ok[u] ? __ldg(row + k * 8 + sub) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kScoreUnroll; ++u) {
      float acc[kIdxHeads];
#pragma unroll
      for (int h = 0; h < kIdxHeads; ++h) {
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          s = fmaf(qv[h][k].x, kv[u][k].x, s);
          s = fmaf(qv[h][k].y, kv[u][k].y, s);
          s = fmaf(qv[h][k].z, kv[u][k].z, s);
          s = fmaf(qv[h][k].w, kv[u][k].w, s);
        }
        acc[h] = s;
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
      v += __shfl_xor_sync(kFull, v, 4);               // sum over the 4 heads
      if (live[u] && sub == 0) {
        const float sc = ok[u] ? v : -INFINITY;
        const int64_t j = base + u * 4 + grp;
        srow[j] = sc;
        if (kTopk) atomicAdd(&s_hist[score_key(sc) >> (32 - kHistBits)], 1u);
      }
    }
  }
  if (!kTopk) return;

  __syncthreads();
  unsigned* gh = hist + (int64_t)t * kHistBins;
  for (int i = tid; i < kHistBins; i += kScoreThreads) {
    const unsigned v = s_hist[i];
    if (v) atomicAdd(gh + i, v);
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(done + t, 1u) == gridDim.x - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // Last CTA of this token: find the bin holding the B-th largest score.
  const unsigned B = (unsigned)a.n_sel_blocks;
  if ((unsigned)nb <= B) {
    if (tid == 0) state[t] = make_int4(-1, 0, 0, nb);
    return;
  }
  constexpr int kPer = kHistBins / kScoreThreads;   // 16 bins per thread
  unsigned h[kPer];
  unsigned sum = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    h[i] = __ldcg(gh + tid * kPer + i);
    sum += h[i];
  }
  unsigned cum = block_suffix_exclusive(sum, s_warp);
#pragma unroll
  for (int i = kPer - 1; i >= 0; --i) {
    const unsigned nxt = cum + h[i];
    if (cum < B && nxt >= B) state[t] = make_int4(tid * kPer + i, (int)(B - cum), (int)h[i], nb);
    cum = nxt;
  }
}

// ---------------------------------------------------------------- k_filter
__global__ void __launch_bounds__(kFilterThreads)
k_filter(const float* __restrict__ scores, int64_t pitch, const int4* __restrict__ state,
         unsigned* __restrict__ bitmap, int64_t wpitch, unsigned* __restrict__ cand_cnt,
         unsigned long long* __restrict__ cand) {
  const int t = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int4 st = state[t];
  const int thr = st.x, ncand = st.z, nb = st.w;
  const bool keep_cand = thr >= 0 && ncand <= kCandCap;
  const int64_t W = ceil_div(nb, 32);
  const int64_t w0 = (int64_t)blockIdx.x * kFilterWordsPerCta;
  const int64_t w1 = min(W, w0 + kFilterWordsPerCta);
  const float* srow = scores + (int64_t)t * pitch;
  for (int64_t w = w0 + warp; w < w1; w += kFilterThreads / 32) {
    const int64_t j = w * 32 + lane;
    const bool in = j < nb;
    const uint32_t key = score_key(in ? __ldcg(srow + j) : 0.f);
    const int bin = (int)(key >> (32 - kHistBits));
    const bool above = in && bin > thr;
    const bool isc = in && bin == thr;
    const unsigned am = __ballot_sync(kFull, above);
    if (lane == 0) bitmap[(int64_t)t * wpitch + w] = am;
    if (keep_cand) {
      const unsigned cm = __ballot_sync(kFull, isc);
      if (cm) {
        const int leader = __ffs(cm) - 1;
        unsigned basei = 0;
        if (lane == leader) basei = atomicAdd(cand_cnt + t, (unsigned)__popc(cm));
        basei = __shfl_sync(kFull, basei, leader);
        if (isc)
          cand[(int64_t)t * kCandCap + basei + __popc(cm & ((1u << lane) - 1u))] = cand_key(key, j);
      }
    }
  }
}

// ----------------------------------------------------------------- k_final
__global__ void __launch_bounds__(kFinalThreads)
k_final(const IndexArgs a, const float* __restrict__ scores, const int4* __restrict__ state,
        unsigned* __restrict__ bitmap, int64_t wpitch,
        const unsigned long long* __restrict__ cand,
        int32_t* __restrict__ cells, int32_t* __restrict__ count, unsigned* err) {
  __shared__ unsigned s_hist[256];
  __shared__ unsigned s_warp[32];
  __shared__ int s_digit;
  __shared__ unsigned s_above, s_eq;

  const int t = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int4 st = state[t];
  const int thr = st.x, ncand = st.z, nb = st.w;
  unsigned* bm = bitmap + (int64_t)t * wpitch;
  const float* srow = scores + (int64_t)t * a.max_blocks;

  if (thr >= 0) {
    // Select the `need` largest unique keys among the threshold-bin blocks,
    // one radix digit (8 bits, most significant first) at a time.
    const bool fast = ncand <= kCandCap;
    constexpr int kPer = kCandCap / kFinalThreads;
    unsigned long long c[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int idx = tid + i * kFinalThreads;
      c[i] = (fast && idx < ncand) ? __ldcg(cand + (int64_t)t * kCandCap + idx) : 0ull;
    }
    unsigned long long prefix = 0;
    int shift = 48;
    unsigned need = (unsigned)st.y;
    for (;;) {
      for (int i = tid; i < 256; i += kFinalThreads) s_hist[i] = 0u;
      __syncthreads();
      if (fast) {
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          const int idx = tid + i * kFinalThreads;
          if (idx < ncand && (c[i] >> (shift + 8)) == prefix)
            atomicAdd(&s_hist[(unsigned)(c[i] >> shift) & 255u], 1u);
        }
      } else {
        for (int64_t j = tid; j < nb; j += kFinalThreads) {
          const uint32_t key = score_key(__ldcg(srow + j));
          if ((int)(key >> (32 - kHistBits)) != thr) continue;
          const unsigned long long ck = cand_key(key, j);
          if ((ck >> (shift + 8)) == prefix) atomicAdd(&s_hist[(unsigned)(ck >> shift) & 255u], 1u);
        }
      }
      __syncthreads();
      if (warp == 0) {
        unsigned hv[8], sum = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          hv[i] = s_hist[lane * 8 + i];
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
            s_digit = lane * 8 + i;
            s_above = cum;
            s_eq = hv[i];
          }
          cum = nxt;
        }
      }
      __syncthreads();
      const int d = s_digit;
      need -= s_above;
      const unsigned eq = s_eq;
      prefix = (prefix << 8) | (unsigned long long)d;
      __syncthreads();
      if (eq == need || shift == 0) break;
      shift -= 8;
    }
    // Every key whose top bits (down to `shift`) are >= prefix is chosen.
    if (fast) {
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int idx = tid + i * kFinalThreads;
        if (idx < ncand && (c[i] >> shift) >= prefix) {
          const uint32_t j = ~(uint32_t)(c[i] >> 4);
          atomicOr(bm + (j >> 5), 1u << (j & 31));
        }
      }
    } else {
      for (int64_t j = tid; j < nb; j += kFinalThreads) {
        const uint32_t key = score_key(__ldcg(srow + j));
        if ((int)(key >> (32 - kHistBits)) != thr) continue;
        if ((cand_key(key, j) >> shift) >= prefix) atomicOr(bm + (j >> 5), 1u << (j & 31));
      }
    }
    __syncthreads();
  }

  // Ordered compaction of the bitmap + expansion to member cells.
  const Tok tk = token_geometry(a, t, err, false);
  const int64_t W = ceil_div(nb, 32);
  const int64_t wpt = ceil_div(W, kFinalThreads);
  const int64_t w0 = (int64_t)tid * wpt, w1 = min(W, w0 + wpt);
  unsigned mine = 0;
  for (int64_t w = w0; w < w1; ++w) mine += __popc(__ldcg(bm + w));
  unsigned total = 0;
  unsigned k = block_prefix_exclusive(mine, s_warp, &total);
  const int r = a.r;
  const int B = a.n_sel_blocks;
  int32_t* crow = cells + (int64_t)t * a.cells_pitch;
  const int32_t* slots = a.seq_blk_slots + tk.off;
  for (int64_t w = w0; w < w1; ++w) {
    unsigned bits = __ldcg(bm + w);
    while (bits) {
      const int b = __ffs(bits) - 1;
      bits &= bits - 1u;
      const int64_t j = w * 32 + b;
      if (k < (unsigned)B) {
        const int slot = slots[j];
        const bool sok = slot >= 0 && slot < a.n_slots;
        if (!sok) atomicOr(err, kErrSlot);
        for (int i = 0; i < r; ++i) {
          const int cidx = sok ? a.blk_cells[(int64_t)slot * r + i] : -1;
          if (cidx < 0 || cidx >= a.n_cells) atomicOr(err, kErrCell);
          crow[(int64_t)k * r + i] = cidx;
        }
      }
      ++k;
    }
  }
  const int nsel = (int)min(total, (unsigned)B);
  int tail = 0;
  if (tk.ok && tk.nb == tk.nb_full) tail = tk.p + 1 - (int)(tk.nb_full * r);
  if (tid == 0) {
    if (tail > 0) {
      if (tk.nb_full < tk.len) {
        const int slot = slots[tk.nb_full];
        const bool sok = slot >= 0 && slot < a.n_slots;
        if (!sok) atomicOr(err, kErrSlot);
        for (int i = 0; i < tail; ++i) {
          const int cidx = sok ? a.blk_cells[(int64_t)slot * r + i] : -1;
          if (cidx < 0 || cidx >= a.n_cells) atomicOr(err, kErrCell);
          crow[nsel * r + i] = cidx;
        }
      } else {
        atomicOr(err, kErrBlockList);
        tail = 0;
      }
    }
    count[t] = nsel * r + tail;
  }
  for (int i = nsel * r + tail + tid; i < a.cells_pitch; i += kFinalThreads) crow[i] = -1;
}

int score_chunk(int T, int64_t max_blocks) {
  // Aim for ~4 CTAs per SM of a 152-SM part across all tokens.
  const int64_t target = 608;
  int64_t iters = ceil_div(max_blocks * (int64_t)T, target * kRowsPerIter);
  if (iters < 1) iters = 1;
  if (iters > 64) iters = 64;
  return (int)(iters * kRowsPerIter);
}

}  // namespace

size_t index_workspace_bytes(int n_tokens, int64_t max_blocks) {
  return carve(nullptr, n_tokens, max_blocks).total;
}

void index_workspace_zero_range(int n_tokens, int64_t max_blocks, size_t* offset, size_t* bytes) {
  const Ws w = carve(reinterpret_cast<void*>(static_cast<uintptr_t>(256)), n_tokens, max_blocks);
  *offset = static_cast<size_t>(static_cast<char*>(w.zero_base) - reinterpret_cast<char*>(static_cast<uintptr_t>(256)));
  *bytes = w.zero_bytes;
}

cudaError_t launch_index_scores(const IndexArgs& a, float* scores, unsigned* err, cudaStream_t stream) {
  if (a.n_tokens <= 0 || a.max_blocks <= 0) return cudaSuccess;
  const int chunk = score_chunk(a.n_tokens, a.max_blocks);
  const dim3 grid((unsigned)ceil_div(a.max_blocks, chunk), (unsigned)a.n_tokens);
  k_score<false><<<grid, kScoreThreads, 0, stream>>>(a, scores, nullptr, nullptr, nullptr, chunk, err);
  return cudaGetLastError();
}

cudaError_t launch_index_topk(const IndexArgs& a, int32_t* cells, int32_t* count,
                              void* wsp, unsigned* err, cudaStream_t stream) {
  if (a.n_tokens <= 0) return cudaSuccess;
  const int64_t mb = a.max_blocks > 0 ? a.max_blocks : 1;
  Ws w = carve(wsp, a.n_tokens, mb);
  cudaError_t e = cudaMemsetAsync(w.zero_base, 0, w.zero_bytes, stream);
  if (e != cudaSuccess) return e;
  IndexArgs b = a;
  b.max_blocks = mb;
  const int chunk = score_chunk(a.n_tokens, mb);
  const dim3 g1((unsigned)ceil_div(mb, chunk), (unsigned)a.n_tokens);
  prof_before(kKScore, stream);
  k_score<true><<<g1, kScoreThreads, 0, stream>>>(b, w.scores, w.hist, w.done, w.state, chunk, err);
  prof_after(kKScore, stream);
  const dim3 g2((unsigned)ceil_div(ceil_div(mb, 32), kFilterWordsPerCta), (unsigned)a.n_tokens);
  prof_before(kKFilter, stream);
  k_filter<<<g2, kFilterThreads, 0, stream>>>(w.scores, mb, w.state, w.bitmap, w.wpitch, w.cand_cnt, w.cand);
  prof_after(kKFilter, stream);
  prof_before(kKFinal, stream);
  k_final<<<(unsigned)a.n_tokens, kFinalThreads, 0, stream>>>(b, w.scores, w.state, w.bitmap, w.wpitch,
                                                               w.cand, cells, count, err);
  prof_after(kKFinal, stream);
  return cudaGetLastError();
}

}  // namespace qsa
