// Public C ABI of libqsa (declared in include/qsa.h): argument validation on
// the host, then the launches.  Nothing here allocates device memory.
#include <cmath>
#include <cstdint>
#include <cstring>

#include "qsa_internal.cuh"

// Device error word: bits of qsa::kErr*, set with atomicOr by kernels that
// meet an out-of-range index, read and cleared by qsa_debug_check.
__device__ unsigned int g_qsa_error_word;

namespace qsa {
ProfileHook g_profile = {};
}

namespace {

using namespace qsa;

qsa_status check_cfg(const qsa_config* c) {
  if (c == nullptr) return QSA_ERR_INVALID_ARG;
  if (c->n_q_heads <= 0 || c->n_kv_heads <= 0 || c->head_dim <= 0 || c->n_idx_heads <= 0 ||
      c->idx_dim <= 0 || c->compress_ratio <= 0 || c->top_k <= 0)
    return QSA_ERR_INVALID_ARG;
  if (c->kv_type != QSA_KV_F16 && c->kv_type != QSA_KV_Q8_0) return QSA_ERR_INVALID_ARG;
  if (!(c->rope_theta > 0.f) || !(c->rms_eps >= 0.f) || !std::isfinite(c->attn_scale) ||
      !std::isfinite(c->rope_theta))
    return QSA_ERR_INVALID_ARG;
  if (c->head_dim != kHeadDim || c->n_q_heads != kGqa * c->n_kv_heads || c->idx_dim != kIdxDim ||
      c->n_idx_heads != kIdxHeads || c->compress_ratio > 8 || c->top_k % c->compress_ratio != 0 ||
      c->top_k > (1 << 20) || c->n_kv_heads > 64)
    return QSA_ERR_UNSUPPORTED;
  return QSA_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

unsigned* error_word() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_qsa_error_word) != cudaSuccess) return nullptr;
  return static_cast<unsigned*>(p);
}

qsa_status from_cuda(cudaError_t e) { return e == cudaSuccess ? QSA_OK : QSA_ERR_CUDA; }

constexpr int64_t kMaxI32 = 2147483647;

qsa_status fill_index_args(const qsa_config* cfg, int32_t n_tokens, int32_t max_tokens, const float* q_idx,
                           const float* w_idx, const int32_t* tok_seq, const int32_t* tok_pos,
                           const float* pooled, int64_t n_slots, const int64_t* seq_blk_off,
                           const int32_t* seq_blk_slots, int32_t n_seq, int64_t max_blocks,
                           IndexArgs* a) {
  qsa_status st = check_cfg(cfg);
  if (st != QSA_OK) return st;
  if (n_tokens < 0 || n_slots < 0 || n_seq < 0 || max_blocks < 0) return QSA_ERR_INVALID_ARG;
  if (max_tokens < n_tokens) return QSA_ERR_SHAPE;
  if (max_tokens > 65535) return QSA_ERR_UNSUPPORTED;
  if (n_slots > kMaxI32 || max_blocks > index_max_blocks_limit()) return QSA_ERR_UNSUPPORTED;
  if (n_tokens > 0 && (!q_idx || !w_idx || !tok_seq || !tok_pos || !pooled || !seq_blk_off ||
                       !seq_blk_slots || n_seq <= 0))
    return QSA_ERR_INVALID_ARG;
  if (!aligned(q_idx, 16) || !aligned(pooled, 16) || !aligned(w_idx, 4) || !aligned(seq_blk_off, 8))
    return QSA_ERR_INVALID_ARG;
  a->n_tokens = n_tokens;
  a->max_tokens = max_tokens;
  a->q_idx = q_idx;
  a->w_idx = w_idx;
  a->tok_seq = tok_seq;
  a->tok_pos = tok_pos;
  a->pooled = pooled;
  a->blk_cells = nullptr;
  a->n_slots = n_slots;
  a->seq_blk_off = seq_blk_off;
  a->seq_blk_slots = seq_blk_slots;
  a->n_seq = n_seq;
  a->max_blocks = max_blocks;
  a->n_cells = 0;
  a->r = cfg->compress_ratio;
  a->n_sel_blocks = cfg->top_k / cfg->compress_ratio;
  a->cells_pitch = cfg->top_k + cfg->compress_ratio - 1;
  return QSA_OK;
}

}  // namespace

extern "C" {

qsa_status qsa_config_init(qsa_config* cfg) {
  if (cfg == nullptr) return QSA_ERR_INVALID_ARG;
  cfg->n_q_heads = 16;
  cfg->n_kv_heads = 2;
  cfg->head_dim = 256;
  cfg->n_idx_heads = 4;
  cfg->idx_dim = 128;
  cfg->compress_ratio = 4;
  cfg->top_k = 2048;
  cfg->rope_theta = 1.0e6f;
  cfg->rms_eps = 1.0e-6f;
  cfg->attn_scale = 1.0f / 16.0f;
  cfg->kv_type = QSA_KV_F16;
  return QSA_OK;
}

int32_t qsa_cells_per_token(const qsa_config* cfg) {
  if (check_cfg(cfg) != QSA_OK) return -1;
  return cfg->top_k + cfg->compress_ratio - 1;
}

qsa_status qsa_pool_update(const qsa_config* cfg, const void* idx_k, int64_t n_cells,
                           const int32_t* blk_cells, const int32_t* slot_block_idx,
                           int64_t n_slots, const int32_t* dirty, int32_t n_dirty,
                           const float* norm_w, float* pooled, qsa_stream_t stream) {
  qsa_status st = check_cfg(cfg);
  if (st != QSA_OK) return st;
  if (n_cells < 0 || n_slots < 0 || n_dirty < 0) return QSA_ERR_INVALID_ARG;
  if (n_cells > kMaxI32 || n_slots > kMaxI32) return QSA_ERR_UNSUPPORTED;
  if (n_dirty == 0) return QSA_OK;
  if (!idx_k || !blk_cells || !slot_block_idx || !dirty || !norm_w || !pooled) return QSA_ERR_INVALID_ARG;
  if (!aligned(idx_k, 4) || !aligned(norm_w, 8) || !aligned(pooled, 8)) return QSA_ERR_INVALID_ARG;
  unsigned* err = error_word();
  if (err == nullptr) return QSA_ERR_CUDA;
  return from_cuda(launch_pool_update(*cfg, static_cast<const __half*>(idx_k), n_cells, blk_cells,
                                      slot_block_idx, n_slots, dirty, n_dirty, norm_w, pooled, err,
                                      reinterpret_cast<cudaStream_t>(stream)));
}

qsa_status qsa_index_scores(const qsa_config* cfg, int32_t n_tokens, const float* q_idx,
                            const float* w_idx, const int32_t* tok_seq, const int32_t* tok_pos,
                            const float* pooled, int64_t n_slots, const int64_t* seq_blk_off,
                            const int32_t* seq_blk_slots, int32_t n_seq, int64_t max_blocks,
                            float* scores, qsa_stream_t stream) {
  IndexArgs a{};
  qsa_status st = fill_index_args(cfg, n_tokens, n_tokens, q_idx, w_idx, tok_seq, tok_pos, pooled, n_slots,
                                  seq_blk_off, seq_blk_slots, n_seq, max_blocks, &a);
  if (st != QSA_OK) return st;
  if (n_tokens == 0 || max_blocks == 0) return QSA_OK;
  if (scores == nullptr) return QSA_ERR_INVALID_ARG;
  unsigned* err = error_word();
  if (err == nullptr) return QSA_ERR_CUDA;
  return from_cuda(launch_index_scores(a, scores, err, reinterpret_cast<cudaStream_t>(stream)));
}

size_t qsa_index_topk_workspace_size(const qsa_config* cfg, int32_t max_tokens, int64_t max_blocks) {
  if (check_cfg(cfg) != QSA_OK || max_tokens < 0 || max_blocks < 0) return 0;
  return index_workspace_bytes(max_tokens, max_blocks > 0 ? max_blocks : 1);
}

qsa_status qsa_index_topk(const qsa_config* cfg, int32_t n_tokens, int32_t max_tokens, const float* q_idx,
                          const float* w_idx, const int32_t* tok_seq, const int32_t* tok_pos,
                          const float* pooled, const int32_t* blk_cells, int64_t n_slots,
                          const int64_t* seq_blk_off, const int32_t* seq_blk_slots,
                          int32_t n_seq, int64_t max_blocks, int64_t n_cells, int32_t* cells,
                          int32_t* count, const int32_t* recomputed, int32_t n_recomputed,
                          void* workspace, size_t ws_bytes, qsa_stream_t stream) {
  IndexArgs a{};
  qsa_status st = fill_index_args(cfg, n_tokens, max_tokens, q_idx, w_idx, tok_seq, tok_pos, pooled, n_slots,
                                  seq_blk_off, seq_blk_slots, n_seq, max_blocks, &a);
  if (st != QSA_OK) return st;
  if (n_cells < 0) return QSA_ERR_INVALID_ARG;
  if (n_cells > kMaxI32) return QSA_ERR_UNSUPPORTED;
  if (n_tokens == 0) return QSA_OK;
  if (!blk_cells || !cells || !count) return QSA_ERR_INVALID_ARG;
  if (workspace == nullptr || !aligned(workspace, 256) ||
      ws_bytes < qsa_index_topk_workspace_size(cfg, max_tokens, max_blocks))
    return QSA_ERR_WORKSPACE;
  const bool query_hint = n_recomputed == QSA_HINT_QUERY_BLOCKS && recomputed == nullptr;
  if ((n_recomputed < 0 && !query_hint) || (n_recomputed > 0 && recomputed == nullptr)) return QSA_ERR_INVALID_ARG;
  a.blk_cells = blk_cells;
  a.n_cells = n_cells;
  a.recomputed = recomputed;
  a.n_recomputed = n_recomputed;
  unsigned* err = error_word();
  if (err == nullptr) return QSA_ERR_CUDA;
  return from_cuda(launch_index_topk(a, cells, count, workspace, err, reinterpret_cast<cudaStream_t>(stream)));
}

size_t qsa_sparse_attn_workspace_size(const qsa_config* cfg, int32_t n_tokens) {
  if (check_cfg(cfg) != QSA_OK || n_tokens < 0) return 0;
  return attn_workspace_bytes(n_tokens, cfg->n_q_heads, cfg->top_k + cfg->compress_ratio - 1);
}

namespace {

// Checks of qsa_sparse_attn's arguments (shared by its union form); fills `a`.
qsa_status attn_args(const qsa_config* cfg, int32_t n_tokens, const void* q, const void* k_cache,
                     const void* v_cache, int64_t n_cells, const int32_t* cells, const int32_t* count, float* out,
                     void* workspace, size_t ws_bytes, AttnArgs* a) {
  qsa_status st = check_cfg(cfg);
  if (st != QSA_OK) return st;
  if (n_tokens < 0 || n_cells < 0) return QSA_ERR_INVALID_ARG;
  if (n_tokens > 65535) return QSA_ERR_UNSUPPORTED;
  if (n_cells > kMaxI32) return QSA_ERR_UNSUPPORTED;
  if (n_tokens == 0) return QSA_OK;
  if (!q || !k_cache || !v_cache || !cells || !count || !out) return QSA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 4))
    return QSA_ERR_INVALID_ARG;
  const size_t need = qsa_sparse_attn_workspace_size(cfg, n_tokens);
  if (need > 0 && (workspace == nullptr || !aligned(workspace, 256) || ws_bytes < need))
    return QSA_ERR_WORKSPACE;
  a->n_tokens = n_tokens;
  a->n_kv_heads = cfg->n_kv_heads;
  a->kv_q8 = cfg->kv_type == QSA_KV_Q8_0;
  a->q = static_cast<const __half*>(q);
  a->k_cache = k_cache;
  a->v_cache = v_cache;
  a->n_cells = n_cells;
  a->cells = cells;
  a->cells_pitch = cfg->top_k + cfg->compress_ratio - 1;
  a->count = count;
  a->out = out;
  a->attn_scale = cfg->attn_scale;
  return QSA_OK;
}

}  // namespace

qsa_status qsa_sparse_attn(const qsa_config* cfg, int32_t n_tokens, const void* q,
                           const void* k_cache, const void* v_cache, int64_t n_cells,
                           const int32_t* cells, const int32_t* count, float* out,
                           void* workspace, size_t ws_bytes, qsa_stream_t stream) {
  AttnArgs a{};
  const qsa_status st = attn_args(cfg, n_tokens, q, k_cache, v_cache, n_cells, cells, count, out, workspace,
                                  ws_bytes, &a);
  if (st != QSA_OK || n_tokens == 0) return st;
  unsigned* err = error_word();
  if (err == nullptr) return QSA_ERR_CUDA;
  return from_cuda(launch_sparse_attn(a, workspace, err, reinterpret_cast<cudaStream_t>(stream)));
}

qsa_status qsa_sparse_attn_union(const qsa_config* cfg, int32_t n_tokens, const void* q,
                                 const void* k_cache, const void* v_cache, int64_t n_cells,
                                 const int32_t* cells, const int32_t* count, float* out,
                                 void* workspace, size_t ws_bytes, qsa_stream_t stream) {
  AttnArgs a{};
  const qsa_status st = attn_args(cfg, n_tokens, q, k_cache, v_cache, n_cells, cells, count, out, workspace,
                                  ws_bytes, &a);
  if (st != QSA_OK) return st;
  if (cfg->top_k + cfg->compress_ratio - 1 > union_attn_max_pitch()) return QSA_ERR_UNSUPPORTED;
  if (n_tokens == 0) return QSA_OK;
  unsigned* err = error_word();
  if (err == nullptr) return QSA_ERR_CUDA;
  return from_cuda(launch_sparse_attn_union(a, err, reinterpret_cast<cudaStream_t>(stream)));
}

qsa_status qsa_index_attn(const qsa_config* cfg, int32_t n_tokens, int32_t max_tokens, const float* q_idx,
                          const float* w_idx, const int32_t* tok_seq, const int32_t* tok_pos,
                          const float* pooled, const int32_t* blk_cells, int64_t n_slots,
                          const int64_t* seq_blk_off, const int32_t* seq_blk_slots, int32_t n_seq,
                          int64_t max_blocks, const void* q, const void* k_cache, const void* v_cache,
                          int64_t n_cells, int32_t* cells, int32_t* count, float* out,
                          const int32_t* recomputed, int32_t n_recomputed, uint32_t flags, void* workspace,
                          size_t ws_bytes, qsa_stream_t stream) {
  IndexArgs ia{};
  qsa_status st = fill_index_args(cfg, n_tokens, max_tokens, q_idx, w_idx, tok_seq, tok_pos, pooled, n_slots,
                                  seq_blk_off, seq_blk_slots, n_seq, max_blocks, &ia);
  if (st != QSA_OK) return st;
  constexpr uint32_t kFlags = QSA_INDEX_ATTN_IN_CLUSTER | QSA_INDEX_ATTN_UNION;
  if (n_cells < 0 || (flags & ~kFlags) != 0u || flags == kFlags) return QSA_ERR_INVALID_ARG;
  const bool by_union = (flags & QSA_INDEX_ATTN_UNION) != 0u;
  if (by_union && cfg->top_k + cfg->compress_ratio - 1 > union_attn_max_pitch()) return QSA_ERR_UNSUPPORTED;
  if (n_cells > kMaxI32) return QSA_ERR_UNSUPPORTED;
  if (n_tokens == 0) return QSA_OK;
  if (!blk_cells || !cells || !count || !q || !k_cache || !v_cache || !out) return QSA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 4))
    return QSA_ERR_INVALID_ARG;
  if (workspace == nullptr || !aligned(workspace, 256) ||
      ws_bytes < qsa_index_topk_workspace_size(cfg, max_tokens, max_blocks))
    return QSA_ERR_WORKSPACE;
  const bool query_hint = n_recomputed == QSA_HINT_QUERY_BLOCKS && recomputed == nullptr;
  if ((n_recomputed < 0 && !query_hint) || (n_recomputed > 0 && recomputed == nullptr)) return QSA_ERR_INVALID_ARG;
  ia.blk_cells = blk_cells;
  ia.n_cells = n_cells;
  ia.recomputed = recomputed;
  ia.n_recomputed = n_recomputed;
  AttnArgs a{};
  a.n_tokens = n_tokens;
  a.n_kv_heads = cfg->n_kv_heads;
  a.kv_q8 = cfg->kv_type == QSA_KV_Q8_0;
  a.q = static_cast<const __half*>(q);
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.n_cells = n_cells;
  a.cells = cells;
  a.cells_pitch = cfg->top_k + cfg->compress_ratio - 1;
  a.count = count;
  a.out = out;
  a.attn_scale = cfg->attn_scale;
  unsigned* err = error_word();
  if (err == nullptr) return QSA_ERR_CUDA;
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (by_union) {
    cudaError_t e = launch_index_topk(ia, cells, count, workspace, err, cs);
    if (e == cudaSuccess) e = launch_sparse_attn_union(a, err, cs);
    return from_cuda(e);
  }
  bool fused = false;
  return from_cuda(launch_index_attn(ia, a, cells, count, workspace, (flags & QSA_INDEX_ATTN_IN_CLUSTER) != 0u,
                                     err, cs, &fused));
}

uint32_t qsa_index_attn_kernels(const qsa_config* cfg, int32_t n_tokens, int32_t n_seq, int64_t max_blocks,
                                uint32_t flags) {
  if (check_cfg(cfg) != QSA_OK || n_tokens <= 0) return 0u;
  constexpr uint32_t kFlags = QSA_INDEX_ATTN_IN_CLUSTER | QSA_INDEX_ATTN_UNION;
  if ((flags & ~kFlags) != 0u || flags == kFlags) return 0u;
  if ((flags & QSA_INDEX_ATTN_UNION) != 0u && cfg->top_k + cfg->compress_ratio - 1 > qsa::union_attn_max_pitch())
    return 0u;
  bool fused = false;
  if ((flags & QSA_INDEX_ATTN_IN_CLUSTER) != 0u && qsa::index_attn_plan(n_tokens, cfg->n_kv_heads, cfg->kv_type == QSA_KV_Q8_0,
                           cfg->top_k + cfg->compress_ratio - 1, max_blocks > 0 ? max_blocks : 1,
                           cfg->top_k / cfg->compress_ratio, cfg->compress_ratio, &fused) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0u;
  }
  const uint32_t scores = qsa_index_topk_kernels(n_tokens, n_seq) & ~(1u << qsa::kKFinal);
  if (fused) return scores | (1u << qsa::kKFused);
  return scores | (1u << qsa::kKFinal) | (1u << qsa::kKAttn);
}

qsa_status qsa_kv_append(const qsa_config* cfg, int32_t n_new, const int32_t* tok_seq, const int32_t* tok_pos,
                         const int32_t* cells, const void* k_new, const void* v_new, const void* idx_new,
                         void* k_cache, void* v_cache, void* idx_k, int64_t n_cells, int32_t* blk_cells,
                         int64_t n_slots, const int64_t* seq_blk_off, const int32_t* seq_blk_slots,
                         int32_t n_seq, int32_t* dirty, int32_t n_dirty, const int32_t* slot_block_idx,
                         const float* norm_w, float* pooled, qsa_stream_t stream) {
  qsa_status st = check_cfg(cfg);
  if (st != QSA_OK) return st;
  if (n_new < 0 || n_cells < 0 || n_slots < 0 || n_seq < 0 || n_dirty < 0) return QSA_ERR_INVALID_ARG;
  if (n_cells > kMaxI32 || n_slots > kMaxI32 || n_new > kAppendMaxTokens) return QSA_ERR_UNSUPPORTED;
  if (n_new == 0) return QSA_OK;
  if (n_dirty < n_new) return QSA_ERR_SHAPE;
  if (!tok_seq || !tok_pos || !cells || !k_new || !v_new || !idx_new || !k_cache || !v_cache || !idx_k ||
      !blk_cells || !seq_blk_off || !seq_blk_slots || !dirty || n_seq == 0)
    return QSA_ERR_INVALID_ARG;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(idx_new, 16) || !aligned(k_cache, 16) ||
      !aligned(v_cache, 16) || !aligned(idx_k, 16) || !aligned(seq_blk_off, 8))
    return QSA_ERR_INVALID_ARG;
  if (pooled != nullptr && (!slot_block_idx || !norm_w || !aligned(norm_w, 8) || !aligned(pooled, 8)))
    return QSA_ERR_INVALID_ARG;
  unsigned* err = error_word();
  if (err == nullptr) return QSA_ERR_CUDA;
  return from_cuda(launch_append(*cfg, n_new, tok_seq, tok_pos, cells, static_cast<const __half*>(k_new),
                                 static_cast<const __half*>(v_new), static_cast<const __half*>(idx_new), k_cache,
                                 v_cache, static_cast<__half*>(idx_k), n_cells, blk_cells, n_slots, seq_blk_off,
                                 seq_blk_slots, n_seq, dirty, n_dirty, slot_block_idx, norm_w, pooled, err,
                                 reinterpret_cast<cudaStream_t>(stream)));
}

qsa_status qsa_blocks_dirty(const int32_t* old_tbl, const int32_t* new_tbl, int64_t n_slots,
                            int32_t r, int32_t* out_dirty, int32_t cap, int32_t* n_dirty,
                            int32_t pad_pow2_min) {
  if (n_dirty == nullptr || n_slots < 0 || r <= 0 || cap < 0 || pad_pow2_min < 0) return QSA_ERR_INVALID_ARG;
  if (n_slots > 0 && (old_tbl == nullptr || new_tbl == nullptr)) return QSA_ERR_INVALID_ARG;
  int64_t n = 0;
  for (int64_t s = 0; s < n_slots; ++s)
    if (std::memcmp(old_tbl + s * r, new_tbl + s * r, sizeof(int32_t) * (size_t)r) != 0) ++n;
  int64_t padded = n;
  if (pad_pow2_min > 0) {
    int64_t p = 1;
    const int64_t want = n > pad_pow2_min ? n : pad_pow2_min;
    while (p < want) p *= 2;
    padded = p;
  }
  if (padded > kMaxI32) return QSA_ERR_UNSUPPORTED;
  *n_dirty = (int32_t)padded;
  if (padded > cap) return QSA_ERR_SHAPE;
  if (padded > 0 && out_dirty == nullptr) return QSA_ERR_INVALID_ARG;
  int64_t k = 0;
  for (int64_t s = 0; s < n_slots; ++s)
    if (std::memcmp(old_tbl + s * r, new_tbl + s * r, sizeof(int32_t) * (size_t)r) != 0)
      out_dirty[k++] = (int32_t)s;
  for (; k < padded; ++k) out_dirty[k] = -1;
  return QSA_OK;
}

qsa_status qsa_debug_check(qsa_stream_t stream, uint32_t* flags) {
  if (flags) *flags = 0;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return QSA_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, g_qsa_error_word, sizeof(v)) != cudaSuccess) return QSA_ERR_CUDA;
  if (v == 0) return QSA_OK;
  const unsigned zero = 0;
  if (cudaMemcpyToSymbol(g_qsa_error_word, &zero, sizeof(zero)) != cudaSuccess) return QSA_ERR_CUDA;
  if (flags) *flags = v;
  return QSA_ERR_DEVICE_BOUNDS;
}

uint32_t qsa_index_topk_kernels(int32_t n_tokens, int32_t n_seq) {
  if (n_tokens <= 0) return 0u;
  if (qsa::index_tiled(n_tokens, n_seq)) return (1u << qsa::kKScore) | (1u << qsa::kKHist) | (1u << qsa::kKFinal);
  return (1u << qsa::kKScore) | (1u << qsa::kKFinal);
}

qsa_status qsa_profile_kernel(int32_t kernel, void* before, void* after) {
  if (kernel < 0 || kernel >= kNumKernels) return QSA_ERR_INVALID_ARG;
  g_profile.before[kernel] = static_cast<cudaEvent_t>(before);
  g_profile.after[kernel] = static_cast<cudaEvent_t>(after);
  return QSA_OK;
}

const char* qsa_status_string(qsa_status s) {
  switch (s) {
    case QSA_OK: return "ok";
    case QSA_ERR_INVALID_ARG: return "invalid argument";
    case QSA_ERR_SHAPE: return "inconsistent shapes";
    case QSA_ERR_UNSUPPORTED: return "unsupported configuration";
    case QSA_ERR_WORKSPACE: return "workspace null, misaligned or too small";
    case QSA_ERR_CUDA: return "CUDA error";
    case QSA_ERR_DEVICE_BOUNDS: return "a kernel met an out-of-range index";
  }
  return "unknown status";
}

}  // extern "C"

// ---------------------------------------------------------------------------
// qsa_index_topk_noalloc: qsa_index_topk with its workspace in a static device
// array, for callers that cannot allocate device memory themselves: plugins
// hosted by an engine that owns every device allocation through its own pool
// and hands the plugin no allocator, and code on a latency-critical path where
// cudaMalloc (which may synchronise the device) is not allowed.
//
// The array lives in this library's device image: every GPU that loads the
// library holds kNoAllocScratchBytes of it until the process exits.  Host code
// cannot use the symbol as a device address; the address belongs to the
// current device's context, so every call looks it up with its device current
// (as the error word is looked up), and nothing is cached between calls.
namespace {

constexpr int kNoAllocMaxTokens = 8;
constexpr int64_t kNoAllocMaxBlocks = 262144;        // 1,048,576 cells per sequence at r = 4
constexpr size_t kNoAllocScratchBytes = 9u << 20;    // >= the workspace of 8 tokens x 262144 blocks
static_assert(qsa::index_workspace_bytes_max(kNoAllocMaxTokens, kNoAllocMaxBlocks) <= kNoAllocScratchBytes,
              "the scratch array holds the workspace of the largest call it accepts");

__device__ __align__(256) unsigned char g_qsa_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array in the current device's context.
qsa_status noalloc_scratch(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_qsa_noalloc_scratch) != cudaSuccess || p == nullptr) return QSA_ERR_CUDA;
  *out = p;
  return QSA_OK;
}

}  // namespace

extern "C" qsa_status qsa_index_topk_noalloc(
    const qsa_config* cfg, int32_t n_tokens, const float* q_idx, const float* w_idx,
    const int32_t* tok_seq, const int32_t* tok_pos, const float* pooled, const int32_t* blk_cells,
    int64_t n_slots, const int64_t* seq_blk_off, const int32_t* seq_blk_slots, int32_t n_seq,
    int64_t max_blocks, int64_t n_cells, int32_t* cells, int32_t* count, qsa_stream_t stream) {
  if (n_tokens > kNoAllocMaxTokens || max_blocks > kNoAllocMaxBlocks) return QSA_ERR_WORKSPACE;
  IndexArgs a{};
  qsa_status st = fill_index_args(cfg, n_tokens, kNoAllocMaxTokens, q_idx, w_idx, tok_seq, tok_pos, pooled,
                                  n_slots, seq_blk_off, seq_blk_slots, n_seq, max_blocks, &a);
  if (st != QSA_OK) return st;
  if (n_cells < 0) return QSA_ERR_INVALID_ARG;
  if (n_cells > kMaxI32) return QSA_ERR_UNSUPPORTED;
  if (n_tokens == 0) return QSA_OK;
  if (!blk_cells || !cells || !count) return QSA_ERR_INVALID_ARG;
  const int64_t mb = max_blocks > 0 ? max_blocks : 1;
  if (index_workspace_bytes(kNoAllocMaxTokens, mb) > kNoAllocScratchBytes) return QSA_ERR_WORKSPACE;
  void* scratch = nullptr;
  st = noalloc_scratch(&scratch);
  if (st != QSA_OK) return st;
  a.blk_cells = blk_cells;
  a.n_cells = n_cells;
  unsigned* err = error_word();
  if (err == nullptr) return QSA_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // The array keeps the previous call's contents: clear the counters and
  // histograms that must start at zero.
  size_t zoff = 0, zbytes = 0;
  index_workspace_zero_range(n_tokens, mb, &zoff, &zbytes);
  if (cudaMemsetAsync(static_cast<char*>(scratch) + zoff, 0, zbytes, s) != cudaSuccess) return QSA_ERR_CUDA;
  return from_cuda(launch_index_topk(a, cells, count, scratch, err, s));
}
