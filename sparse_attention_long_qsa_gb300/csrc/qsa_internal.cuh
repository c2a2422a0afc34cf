// Internal helpers and launcher declarations shared by the libqsa sources.
// Not part of the public ABI (include/qsa.h is).
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/qsa.h"

namespace qsa {

// Device error-word bits (also documented at qsa_debug_check).
enum : unsigned {
  kErrSlot = 1u,       // a slot index outside [0, n_slots)
  kErrCell = 2u,       // a cell index outside [0, n_cells) where a cell is required
  kErrBlockList = 4u,  // a sequence's block list shorter than its tokens need
  kErrMaxBlocks = 8u,  // floor((p+1)/r) above the caller's max_blocks
};

constexpr int kHeadDim = 256;     // DKQ = DV
constexpr int kGqa = 8;           // query heads per KV head
constexpr int kIdxDim = 128;
constexpr int kIdxHeads = 4;

// First radix digit of the selection: the top 12 bits of the order-preserving
// key of an fp32 score.
constexpr int kHistBits = 12;
constexpr int kHistBins = 1 << kHistBits;
// Candidates (scores in the threshold bin) kept in a per-token list and held
// in registers by the final selection CTA: 1024 threads x 4.
constexpr int kFinalThreads = 1024;
constexpr int kCandCap = 4 * kFinalThreads;

// Order-preserving map of an fp32 bit pattern to uint32: a > b as floats
// (no NaN) iff key(a) > key(b).
__device__ __forceinline__ uint32_t score_key(float f) {
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__host__ __device__ __forceinline__ int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
__host__ __device__ __forceinline__ int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

// ------------------------------------------------------ measurement hook
// Kernel ids of qsa_profile_kernel (include/qsa.h).
enum KernelId : int { kKPool = 0, kKScore = 1, kKFilter = 2, kKFinal = 3, kKAttn = 4, kKCombine = 5,
                      kNumKernels = 6 };
struct ProfileHook {
  cudaEvent_t before[kNumKernels];
  cudaEvent_t after[kNumKernels];
};
extern ProfileHook g_profile;
// External records, so that inside a stream capture they become event-record
// nodes that timestamp each replay of the graph.
inline void prof_before(int k, cudaStream_t s) {
  if (g_profile.before[k]) cudaEventRecordWithFlags(g_profile.before[k], s, cudaEventRecordExternal);
}
inline void prof_after(int k, cudaStream_t s) {
  if (g_profile.after[k]) cudaEventRecordWithFlags(g_profile.after[k], s, cudaEventRecordExternal);
}

// ---------------------------------------------------------------- launchers
// All return cudaSuccess or the launch error.  Arguments are validated by the
// public entry points before these run.
cudaError_t launch_pool_update(const qsa_config& cfg, const __half* idx_k, int64_t n_cells,
                               const int32_t* blk_cells, const int32_t* slot_block_idx,
                               int64_t n_slots, const int32_t* dirty, int n_dirty,
                               const float* norm_w, float* pooled, unsigned* err,
                               cudaStream_t stream);

struct IndexArgs {
  int n_tokens;
  const float* q_idx;
  const float* w_idx;
  const int32_t* tok_seq;
  const int32_t* tok_pos;
  const float* pooled;
  const int32_t* blk_cells;
  int64_t n_slots;
  const int64_t* seq_blk_off;
  const int32_t* seq_blk_slots;
  int n_seq;
  int64_t max_blocks;
  int64_t n_cells;
  int r;
  int n_sel_blocks;   // top_k / r
  int cells_pitch;    // top_k + r - 1
};

size_t index_workspace_bytes(int n_tokens, int64_t max_blocks);
// Byte range of the workspace that must be zero when a call starts.
void index_workspace_zero_range(int n_tokens, int64_t max_blocks, size_t* offset, size_t* bytes);
cudaError_t launch_index_scores(const IndexArgs& a, float* scores, unsigned* err, cudaStream_t stream);
cudaError_t launch_index_topk(const IndexArgs& a, int32_t* cells, int32_t* count,
                              void* ws, unsigned* err, cudaStream_t stream);

struct AttnArgs {
  int n_tokens;
  int n_kv_heads;
  int kv_q8;
  const __half* q;
  const void* k_cache;
  const void* v_cache;
  int64_t n_cells;
  const int32_t* cells;
  int cells_pitch;
  const int32_t* count;
  float* out;
  float attn_scale;
};

size_t attn_workspace_bytes(int n_tokens, int n_q_heads, int cells_pitch);
cudaError_t launch_sparse_attn(const AttnArgs& a, void* ws, unsigned* err, cudaStream_t stream);

}  // namespace qsa
