// Helpers shared by the index kernels (index.cu) and the selection that
// runs inside the attention clusters (attn.cu): workspace layout, token
// geometry, block-wide scans, selection keys, small asynchronous copies.
// Not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "qsa_internal.cuh"

namespace qsa {

constexpr unsigned kIdxFull = 0xffffffffu;

// Per-token control words at the front of the workspace: the threshold
// histogram, then a counter of the CTAs that have read it (the selection
// fused with the attention: the last reader clears the histogram).  Zero on
// first use; every call leaves them zero again.
constexpr size_t kCtrlBytes = (size_t)kIndexCtrlBytes;
static_assert(kCtrlBytes >= sizeof(unsigned) * kHistBins + 16 && kCtrlBytes % 16 == 0, "control words");

__host__ __device__ __forceinline__ unsigned* hist_of(void* ws, int t) {
  return reinterpret_cast<unsigned*>(static_cast<char*>(ws) + (size_t)t * kCtrlBytes);
}
__host__ __device__ __forceinline__ unsigned* readers_of(void* ws, int t) {
  return hist_of(ws, t) + kHistBins;
}

__host__ __device__ __forceinline__ float* scores_of(void* ws, int max_tokens) {
  return reinterpret_cast<float*>(static_cast<char*>(ws) + round_up((int64_t)max_tokens * kCtrlBytes, 256));
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

// Sequences whose block offsets a CTA preloads into shared memory (with the
// token ids, so finding a token's block list takes one dependent load less).
constexpr int kOffCache = 256;

// seq_blk_off[0..n_seq] into s_off when n_seq <= kOffCache (returns whether);
// the caller synchronises the CTA before reading s_off.
__device__ __forceinline__ bool preload_offsets(const int64_t* g, int n_seq, int64_t* s_off) {
  if (n_seq > kOffCache) return false;
  for (int i = threadIdx.x; i <= n_seq; i += blockDim.x) s_off[i] = g[i];
  return true;
}

// Geometry of a token at sequence `seq`, position `p`; s_off: the preloaded
// block offsets, or null to read them from global memory.
__device__ __forceinline__ Tok token_geometry(const IndexArgs& a, int seq, int p, const int64_t* s_off,
                                              unsigned* err, bool report) {
  Tok k{0, 0, 0, 0, -1, false};
  if (seq < 0 || seq >= a.n_seq || p < 0) {
    if (report) atomicOr(err, kErrToken);
    return k;
  }
  k.off = s_off ? s_off[seq] : a.seq_blk_off[seq];
  k.len = (s_off ? s_off[seq + 1] : a.seq_blk_off[seq + 1]) - k.off;
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

__device__ __forceinline__ Tok token_geometry(const IndexArgs& a, int t, unsigned* err, bool report) {
  return token_geometry(a, a.tok_seq[t], a.tok_pos[t], nullptr, err, report);
}

// Exclusive sum over the threads with a HIGHER index (suffix sum) of a block.
__device__ __forceinline__ unsigned block_suffix_exclusive(unsigned v, unsigned* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  unsigned x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned y = __shfl_down_sync(kIdxFull, x, o);
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
    const unsigned y = __shfl_up_sync(kIdxFull, x, o);
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

__device__ __forceinline__ void cp_async16_ptr(void* sdst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"((uint32_t)__cvta_generic_to_shared(sdst)),
               "l"(gsrc)
               : "memory");
}
__device__ __forceinline__ void cp_async4(void* sdst, const void* gsrc) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"((uint32_t)__cvta_generic_to_shared(sdst)),
               "l"(gsrc)
               : "memory");
}

// A cell id read from the block table, passed on as read (the attention masks
// it) with the error bit set when it is out of range.
__device__ __forceinline__ int flag_cell(int c, int64_t n_cells, unsigned* err) {
  if (c < 0 || c >= n_cells) atomicOr(err, kErrCell);
  return c;
}

// Unique 56-bit selection key of a block inside the threshold bin: the 20
// low bits of the score key above the bitwise complement of the block index,
// so a larger key means a larger score, or an equal score at a lower index.
__device__ __forceinline__ unsigned long long cand_key(uint32_t key, int64_t j) {
  return ((unsigned long long)(key & 0xFFFFFu) << 36) |
         ((unsigned long long)(~(uint32_t)j) << 4);
}

}  // namespace qsa
