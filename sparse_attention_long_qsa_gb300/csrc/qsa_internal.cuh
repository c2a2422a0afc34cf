// Internal helpers and launcher declarations shared by the libqsa sources.
// Not part of the public ABI (include/qsa.h is).
#pragma once

#include <cstdint>
#include <utility>
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
  kErrToken = 16u,     // a token with a sequence id outside [0, n_seq) or a negative position
  kErrTimeout = 32u,   // a bounded wait on a CTA's own tensor-core work gave up
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

// ------------------------------------------------ launch chaining, clusters
// Programmatic dependent launch: every kernel of the library is launched with
// programmatic stream serialisation, so it may start while its predecessor in
// the stream finishes.  Before grid_dep_wait() (which returns once the
// predecessor grid has completed and its memory is visible) a kernel writes
// nothing outside its own shared memory and reads only the call's inputs that
// no kernel of the library writes (token ids and positions, queries and
// weights, sequence block lists, the new rows of an append, a host-written
// hint).  Most kernels let their successor launch (grid_dep_launch) right
// after that wait; the append lets it launch at its start, and a score CTA
// that has no row to wait for lets it launch before its own wait, which it
// takes at its end.  Either way a kernel completes only after its
// predecessor, so every write of a kernel is visible to any kernel that
// waits on a later one in the stream.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;\n" : "=r"(r));
  return r;
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_addr(const void* local, uint32_t rank) {
  uint32_t remote;
  asm("mapa.shared::cluster.u32 %0, %1, %2;\n"
      : "=r"(remote)
      : "r"((uint32_t)__cvta_generic_to_shared(local)), "r"(rank));
  return remote;
}
// Reads of peers' shared memory after a cluster_sync (not volatile, so the
// compiler may issue several before using any).
__device__ __forceinline__ float ld_dsmem_f32(uint32_t addr) {
  float v;
  asm("ld.shared::cluster.f32 %0, [%1];\n" : "=f"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ unsigned ld_dsmem_u32(uint32_t addr) {
  unsigned v;
  asm("ld.shared::cluster.u32 %0, [%1];\n" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ void st_dsmem_u32(uint32_t addr, unsigned v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;\n" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_dsmem_u64(uint32_t addr, unsigned long long v) {
  asm volatile("st.shared::cluster.u64 [%0], %1;\n" ::"r"(addr), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned atom_or_dsmem(uint32_t addr, unsigned v) {
  unsigned old;
  asm volatile("atom.shared::cluster.or.b32 %0, [%1], %2;\n" : "=r"(old) : "r"(addr), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ unsigned atom_add_dsmem(uint32_t addr, unsigned v) {
  unsigned old;
  asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;\n" : "=r"(old) : "r"(addr), "r"(v) : "memory");
  return old;
}
// Split cluster barrier: arrive early, wait when the peers' earlier writes are needed.
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void st_dsmem_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;\n" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void st_dsmem_f32x4(uint32_t addr, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z),
               "f"(v.w)
               : "memory");
}

// cudaLaunchKernelEx with programmatic stream serialisation and an optional
// 1-D cluster.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, unsigned cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ------------------------------------------------------ phase timestamps
// Built only with -DQSA_PHASE_TIMING (a profiling build, never the product
// library): CTA 0 of a kernel records clock64() at numbered points into a
// per-file device array that an extern "C" reader copies out.
#ifdef QSA_PHASE_TIMING
#define QSA_TS_DECLARE(tu)                                                              \
  __device__ long long g_qsa_ts_##tu[64];                                               \
  extern "C" int qsa_probe_read_##tu(long long* host) {                                 \
    return (int)cudaMemcpyFromSymbol(host, g_qsa_ts_##tu, sizeof(long long) * 64);      \
  }                                                                                     \
  extern "C" int qsa_probe_reset_##tu() {                                               \
    static const long long z[64] = {};                                                  \
    return (int)cudaMemcpyToSymbol(g_qsa_ts_##tu, z, sizeof(z));                        \
  }
// Latest globaltimer over every CTA of a kernel (thread 0 of each), at scope
// exit of the enclosing block: the kernel's end as seen by its last CTA.
#define QSA_TS_SCOPE_LAST(tu, i)                                                        \
  struct QsaTsLast_ {                                                                   \
    __device__ ~QsaTsLast_() {                                                          \
      if (threadIdx.x == 0) {                                                           \
        unsigned long long g_;                                                          \
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(g_));                          \
        atomicMax(reinterpret_cast<unsigned long long*>(&g_qsa_ts_##tu[32 + (i)]), g_); \
      }                                                                                 \
    }                                                                                   \
  } qsa_ts_last_
#define QSA_TS_IF(tu, i, cond)                                                          \
  do {                                                                                  \
    if (cond) {                                                                         \
      long long g_;                                                                     \
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(g_));                            \
      g_qsa_ts_##tu[i] = clock64();                                                     \
      g_qsa_ts_##tu[32 + (i)] = g_;                                                     \
    }                                                                                   \
  } while (0)
#define QSA_TS(tu, i) \
  QSA_TS_IF(tu, i, blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && threadIdx.x == 0)
#else
#define QSA_TS_DECLARE(tu)
#define QSA_TS_IF(tu, i, cond) \
  do {                         \
  } while (0)
#define QSA_TS_SCOPE_LAST(tu, i) \
  do {                           \
  } while (0)
#define QSA_TS(tu, i) \
  do {                \
  } while (0)
#endif

// ------------------------------------------------------ measurement hook
// Kernel ids of qsa_profile_kernel (include/qsa.h).
enum KernelId : int { kKPool = 0, kKScore = 1, kKHist = 2, kKFinal = 3, kKAttn = 4, kKAppend = 5,
                      kKFused = 6, kNumKernels = 7 };
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
  int max_tokens;     // token capacity the workspace layout is sized for
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
  // slots the preceding pool update recomputed (scheduling hint, may be null)
  const int32_t* recomputed;
  int n_recomputed;
};

// Workspace of qsa_index_topk: per token a 4096-bin histogram and a reader
// counter (the control words, zero between calls), then the fp32 scores
// [max_tokens][max_blocks], each part 256-byte aligned.
constexpr int64_t kIndexCtrlBytes = (int64_t)sizeof(unsigned) * kHistBins + 256;
__host__ __device__ constexpr int64_t index_workspace_bytes_max(int64_t max_tokens, int64_t max_blocks) {
  return (max_tokens * kIndexCtrlBytes + 255) / 256 * 256 + (max_tokens * max_blocks * 4 + 255) / 256 * 256;
}
size_t index_workspace_bytes(int max_tokens, int64_t max_blocks);
// Whether qsa_index_topk / qsa_index_scores score with the token-tiled kernel
// (tokens share sequences: more than 8 tokens and 2 per sequence on average).
bool index_tiled(int n_tokens, int n_seq);
// Largest max_blocks the selection kernel supports (per-CTA bitmap capacity).
int64_t index_max_blocks_limit();
// Byte range of the workspace that must be zero when a call starts.
void index_workspace_zero_range(int n_tokens, int64_t max_blocks, size_t* offset, size_t* bytes);
cudaError_t launch_index_scores(const IndexArgs& a, float* scores, unsigned* err, cudaStream_t stream);
cudaError_t launch_index_topk(const IndexArgs& a, int32_t* cells, int32_t* count,
                              void* ws, unsigned* err, cudaStream_t stream);
// The score kernels of qsa_index_topk alone (scores and threshold histogram
// in the workspace), for a selection that runs elsewhere.
cudaError_t launch_index_scores_topk(const IndexArgs& a, void* ws, unsigned* err, cudaStream_t stream);

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
// Attention of token pairs (2i, 2i + 1) over the union of their lists
// (attn_union.cu); cells_pitch <= union_attn_max_pitch().
cudaError_t launch_sparse_attn_union(const AttnArgs& a, unsigned* err, cudaStream_t stream);
int union_attn_max_pitch();
// qsa_index_attn: the qsa_index_topk kernels and the attention kernel, or
// (in_cluster, when its limits hold: *fused = true) the score kernels and
// then the selection and the attention in one cluster kernel.
cudaError_t launch_index_attn(const IndexArgs& ia, const AttnArgs& a, int32_t* cells, int32_t* count, void* ws,
                              bool in_cluster, unsigned* err, cudaStream_t stream, bool* fused);
// Whether qsa_index_attn runs the selection inside the attention clusters
// for this shape (per-device occupancy decides the cluster size).
cudaError_t index_attn_plan(int n_tokens, int n_kv_heads, int kv_q8, int cells_pitch, int64_t max_blocks,
                            int n_sel_blocks, int r, bool* fused);

// Append of new cells (append.cu).  The dirty list is built by one CTA:
// at most kAppendMaxTokens tokens per call.
constexpr int kAppendMaxTokens = 1024;
cudaError_t launch_append(const qsa_config& cfg, int n_new, const int32_t* tok_seq, const int32_t* tok_pos,
                          const int32_t* cell, const __half* k_new, const __half* v_new, const __half* idx_new,
                          void* k_cache, void* v_cache, __half* idx_k, int64_t n_cells, int32_t* blk_cells,
                          int64_t n_slots, const int64_t* seq_blk_off, const int32_t* seq_blk_slots, int n_seq,
                          int32_t* dirty, int n_dirty, const int32_t* slot_block_idx, const float* norm_w,
                          float* pooled, unsigned* err, cudaStream_t stream);

}  // namespace qsa
