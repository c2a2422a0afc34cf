/*
 * qsa.h - C ABI of libqsa: the QSA sparse-attention step on one GB300 (sm_103a).
 *
 * The step has four parts, described in llama.cpp issue #28734 ("Eval bug:
 * qwen4exp (Qwen3.8-Flash-Next) CUDA: decode slows linearly with context"),
 * in the fix summary's sections lever1, lever2, lever2b, lever3 and sparse256:
 *
 *   qsa_kv_append     the step's new K/V cells, indexer keys and block-table
 *                     entries, and the list of blocks they dirty (lever2b)
 *   qsa_pool_update   persistent pooled block-key cache (lever2, lever2b)
 *   qsa_index_topk    indexer block scores, block-granular top-k, block -> cell
 *                     expansion with the tail cells carried along (lever3)
 *   qsa_sparse_attn   split-KV flash-decode over only the selected cells,
 *                     fp16 or q8_0 K/V dequantised after the gather (lever1,
 *                     sparse256, and the author's q8-compact follow-up)
 *
 * Conventions for every call:
 *  - Pointers named as device buffers are DEVICE pointers owned by the caller.
 *    The library never allocates, frees or keeps them.  Kernels launch on the
 *    calling thread's current device (cudaGetDevice), so every device buffer
 *    of a call must be that device's memory.
 *  - A step's own inputs and outputs (q_idx, w_idx, tok_seq, tok_pos, q and
 *    out; for qsa_kv_append tok_seq, tok_pos, cells, k_new, v_new and
 *    idx_new) may instead be page-locked host memory that the device
 *    addresses directly (cudaHostAlloc, or cudaHostRegister; with unified
 *    addressing the host pointer itself): the kernels read and write them in
 *    place over the host link (NVLink-C2C on a Grace system), so a step needs
 *    no copy to or from the device.  The host must not write them (or read
 *    `out`) before the stream has passed the calls.  Everything else is
 *    device memory.
 *  - Calls are asynchronous on `stream` and never synchronise it (only
 *    qsa_debug_check does).  Results are deterministic: identical inputs give
 *    bit-identical outputs.
 *  - Arguments are validated on the host before any launch; an invalid call
 *    returns a negative status and launches nothing.  A failed launch returns
 *    QSA_ERR_CUDA.  Indices read from device buffers (cells, slots) are
 *    range-checked by the kernels: an out-of-range index is skipped (treated
 *    as absent / masked) and recorded in a device error word that
 *    qsa_debug_check reads.  No kernel traps or spin-waits.
 *  - Host threads: calls may come from several host threads at once; each
 *    device's one-time kernel set-up (shared-memory limits, cluster
 *    occupancy) runs under a lock.  Calls that share output or workspace
 *    buffers must still be ordered by the caller, and qsa_index_topk_noalloc
 *    and qsa_profile_kernel carry the further limits stated with them.
 *  - Shapes: one instantiated geometry, the qwen4exp QSA layer: head_dim 256,
 *    8 query heads per KV head (n_q_heads = 8 * n_kv_heads), idx_dim 128,
 *    n_idx_heads 4, compress_ratio 4, top_k a multiple of compress_ratio.
 *    Anything else returns QSA_ERR_UNSUPPORTED.
 *
 * Data layout in device memory:
 *   idx_k          fp16  [n_cells][idx_dim]             indexer key of each cell
 *   k/v cache f16  fp16  [n_cells][n_kv_heads][head_dim]
 *   k/v cache q8_0 bytes: qs int8 [n_cells][n_kv_heads][head_dim], then at byte
 *                  offset n_cells*n_kv_heads*head_dim the scales d fp16
 *                  [n_cells][n_kv_heads][head_dim/32]; value = d[c][g][i/32]*qs[c][g][i]
 *   blk_cells      int32 [n_slots][compress_ratio]  cell of position j*r+i of the
 *                  slot's block, -1 = not (yet) present
 *   slot_block_idx int32 [n_slots]  block index j of the slot within its sequence
 *   pooled         fp32  [n_slots][idx_dim]
 *   seq_blk_off    int64 [n_seq+1], seq_blk_slots int32 [seq_blk_off[n_seq]]:
 *                  block j of sequence s lives in slot seq_blk_slots[seq_blk_off[s]+j]
 *   tok_seq/tok_pos int32 [T]: sequence and position p of each query token; the
 *                  token's own cell is present, positions 0..p are visible
 *   q_idx fp32 [T][n_idx_heads][idx_dim], w_idx fp32 [T][n_idx_heads]
 *   q     fp16 [T][n_q_heads][head_dim],  out fp32 [T][n_q_heads][head_dim]
 *   cells int32 [T][qsa_cells_per_token(cfg)], count int32 [T]
 */
#ifndef QSA_H
#define QSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* qsa_stream_t;

typedef enum {
  QSA_OK = 0,
  QSA_ERR_INVALID_ARG = -1,    /* null pointer, negative size, bad enum */
  QSA_ERR_SHAPE = -2,          /* sizes inconsistent with each other */
  QSA_ERR_UNSUPPORTED = -3,    /* configuration outside the instantiated geometry */
  QSA_ERR_WORKSPACE = -4,      /* workspace null, misaligned (256 B) or too small */
  QSA_ERR_CUDA = -5,           /* a CUDA call or launch failed */
  QSA_ERR_DEVICE_BOUNDS = -6   /* qsa_debug_check: a kernel met an out-of-range index */
} qsa_status;

typedef enum { QSA_KV_F16 = 0, QSA_KV_Q8_0 = 1 } qsa_kv_type;
/* n_recomputed value of qsa_index_topk's scheduling hint (see there). */
#define QSA_HINT_QUERY_BLOCKS (-1)

typedef struct {
  int32_t n_q_heads;       /* 16 */
  int32_t n_kv_heads;      /* 2: query head h reads KV head h / 8 */
  int32_t head_dim;        /* 256 (DKQ = DV) */
  int32_t n_idx_heads;     /* 4 */
  int32_t idx_dim;         /* 128 */
  int32_t compress_ratio;  /* r = 4 cells per block */
  int32_t top_k;           /* 2048 cells = top_k / r whole blocks */
  float rope_theta;        /* 1e6 */
  float rms_eps;           /* 1e-6 */
  float attn_scale;        /* 1 / sqrt(head_dim) */
  int32_t kv_type;         /* qsa_kv_type */
} qsa_config;

/* Fill *cfg with the qwen4exp QSA layer: 16/2 heads of 256, indexer 4 x 128,
 * r = 4, top_k = 2048, theta 1e6, eps 1e-6, scale 1/16, fp16 K/V. */
qsa_status qsa_config_init(qsa_config* cfg);

/* Cells a token may attend: top_k + r - 1 (512 whole blocks plus at most r-1
 * tail cells; llama.cpp issue #28734, goodbadwolf's comment: n_kv_max =
 * min(n_kv, indexer_top_k + r - 1) = 2051).  Row pitch of `cells`. */
int32_t qsa_cells_per_token(const qsa_config* cfg);

/* ---------------------------------------------------------------------------
 * S0  qsa_kv_append  (issue #28734, fix summary, lever2b: block members live in
 * a device table; lever2: only dirtied blocks are re-pooled, padded to a power
 * of two; q8_0 cache: the author's q8-compact follow-up)
 * Writes the step's new cells and lists the blocks they change, so that the
 * pool update that follows needs no host round trip.  Token t (sequence
 * tok_seq[t], position tok_pos[t]) occupies cell cells[t]:
 *   K/V rows of the cell <- k_new[t], v_new[t]  (fp16 [T][n_kv_heads][head_dim];
 *       kv_type f16: copied; q8_0: each 32-value block encoded with scale
 *       d = max|x| / 127 stored as fp16 and codes x * (1/d) rounded half away
 *       from zero, clamped to +-127, all in fp32)
 *   idx_k[cell] <- idx_new[t]  (fp16 [T][idx_dim])
 *   blk_cells[slot(seq, p / r)][p % r] <- cell
 *   dirty <- the distinct slots of the touched blocks, ascending, padded with
 *            -1 to n_dirty entries (a qsa_pool_update dirty list).
 * The block list of each sequence must already hold the slot of every block
 * a new position falls in.  Tokens must occupy distinct cells and positions.
 * pooled (optional, NULL to skip): when given, the dirtied blocks are also
 * re-pooled in the same launch, exactly as a qsa_pool_update(dirty) issued
 * after this call would (bit-identical rows); slot_block_idx and norm_w are
 * then required (as qsa_pool_update takes them).  (This list is written by
 * the launch, so it cannot serve as the scheduling hint of a qsa_index_topk
 * issued right after it.)
 * Limits: n_new <= 1024 (QSA_ERR_UNSUPPORTED beyond); n_dirty >= n_new
 * (QSA_ERR_SHAPE otherwise: room for every token in a block of its own).
 * All buffers 16-byte aligned except the int32 arrays.  A token with an
 * out-of-range sequence, position, block, slot or cell is skipped and flagged
 * in the device error word. */
qsa_status qsa_kv_append(const qsa_config* cfg, int32_t n_new,
                         const int32_t* tok_seq, const int32_t* tok_pos, const int32_t* cells,
                         const void* k_new, const void* v_new, const void* idx_new,
                         void* k_cache, void* v_cache, void* idx_k, int64_t n_cells,
                         int32_t* blk_cells, int64_t n_slots,
                         const int64_t* seq_blk_off, const int32_t* seq_blk_slots, int32_t n_seq,
                         int32_t* dirty, int32_t n_dirty,
                         const int32_t* slot_block_idx, const float* norm_w, float* pooled,
                         qsa_stream_t stream);
/* ---------------------------------------------------------------------------
 * S1  qsa_pool_update  (issue #28734, fix summary, lever2 and lever2b)
 * For each dirty slot s (entries < 0 are skipped; the caller pads the list to
 * a power of two >= 4 so a captured graph keeps its shape):
 *   m   = mean of idx_k[c] over the present cells c of blk_cells[s]
 *   x   = m / sqrt(mean(m^2) + rms_eps) * norm_w
 *   out = NeoX RoPE of x at position slot_block_idx[s] * r, theta = rope_theta
 *         (pair (d, d + idx_dim/2) turns by pos * theta^(-2d/idx_dim))
 *   pooled[s] = out (fp32).  A slot with no present cell gets zeros.
 * Only the dirty rows of `pooled` are written.  Mean and RMSNorm are fp32;
 * the rotation angle is reduced exactly in integers (each frequency a 64-bit
 * fixed-point fraction of a turn, computed on the host) and only the
 * remaining fraction of a turn goes through fp32 sincospi.  No fp64 runs on
 * the device.
 * Errors: QSA_ERR_INVALID_ARG (null pointer with n_dirty > 0, negative sizes),
 * QSA_ERR_UNSUPPORTED (geometry).  A dirty slot >= n_slots or a member cell
 * >= n_cells is skipped and flagged in the device error word. */
qsa_status qsa_pool_update(const qsa_config* cfg,
                           const void* idx_k, int64_t n_cells,
                           const int32_t* blk_cells, const int32_t* slot_block_idx,
                           int64_t n_slots,
                           const int32_t* dirty, int32_t n_dirty,
                           const float* norm_w, float* pooled,
                           qsa_stream_t stream);

/* ---------------------------------------------------------------------------
 * S2  qsa_index_scores  (indexer score as the build defines it; the pages name
 * build_qsa_top_k only - issue #28734, wussh's item 3)
 * For token t of sequence s = tok_seq[t] at position p = tok_pos[t], and each
 * block j < floor((p+1)/r) of s:
 *   scores[t][j] = sum_h w_idx[t][h] * max(0, q_idx[t][h] . pooled[slot(s,j)])
 * fp32, fixed summation order: the kernel qsa_index_topk runs for the same
 * n_tokens and n_seq (one pass per token, or token-tiled when tokens share
 * sequences: see qsa_index_topk_kernels), so the scores are the same bits.  Entries
 * j >= floor((p+1)/r) of the row (pitch max_blocks) are written as -inf.
 * max_blocks: host upper bound on floor((p+1)/r) over the tokens; a token
 * beyond it is clamped and flagged.  Exposed so the scores can be checked on
 * their own; the decode path calls qsa_index_topk. */
qsa_status qsa_index_scores(const qsa_config* cfg, int32_t n_tokens,
                            const float* q_idx, const float* w_idx,
                            const int32_t* tok_seq, const int32_t* tok_pos,
                            const float* pooled, int64_t n_slots,
                            const int64_t* seq_blk_off, const int32_t* seq_blk_slots,
                            int32_t n_seq, int64_t max_blocks,
                            float* scores, qsa_stream_t stream);

/* ---------------------------------------------------------------------------
 * S2+S3+S4  qsa_index_topk  (issue #28734, fix summary, lever3 and lever2b)
 * Per token: scores as in qsa_index_scores; the B = top_k / r blocks of
 * largest score among j < floor((p+1)/r) (ties to the lower j; all of them if
 * there are fewer); then
 *   cells[t] = r member cells of each chosen block, blocks ascending, then the
 *              tail cells of block floor((p+1)/r) at positions <= p
 *   count[t] = (#chosen blocks) * r + ((p + 1) mod r)
 * Entries of the row beyond count[t] are set to -1.  Blocks not yet complete
 * for the token are never scored (-inf in the reference description).
 * Selection is exact on the fp32 scores: a radix select on their bit patterns.
 * workspace: >= qsa_index_topk_workspace_size(cfg, max_tokens, max_blocks)
 * bytes, 256-byte aligned, ZERO-FILLED ONCE before its first use.  Its layout
 * depends on max_tokens only (per-token control words first, then scores), and
 * every call leaves the control words zero again, so one workspace serves any
 * number of calls with n_tokens <= max_tokens and any max_blocks it has room
 * for, as long as max_tokens stays the same.  max_blocks <= 1,048,576;
 * max_tokens <= 65535 (QSA_ERR_UNSUPPORTED beyond, QSA_ERR_SHAPE if
 * n_tokens > max_tokens).
 * recomputed / n_recomputed: optional scheduling hint, NULL / 0 for none;
 * NULL / QSA_HINT_QUERY_BLOCKS asserts instead that the preceding call on the
 * stream changed only the pooled keys of blocks holding the query tokens' own
 * positions (a qsa_kv_append of exactly these tokens, which re-pools them):
 * work on the other blocks then starts without waiting for that call.
 * When this call directly follows a qsa_pool_update on the same stream, pass
 * that update's dirty list (entries < 0 ignored): work on blocks whose slots
 * are not in the list then starts without waiting for the update to finish
 * (lists longer than 32 entries are not used).  The hint must name every slot
 * the preceding update writes, or stale pooled keys may be scored, and it is
 * read before the preceding call has finished: it must hold its values before
 * that call is issued (a host-written list, as qsa_pool_update takes; not the
 * list a qsa_kv_append just wrote).  Results do not depend on the hint
 * otherwise, and the token-tiled scorer (qsa_index_topk_kernels) always
 * waits.  QSA_ERR_INVALID_ARG if n_recomputed < 0 (other than
 * QSA_HINT_QUERY_BLOCKS with a NULL list), or > 0 with a NULL list. */
size_t qsa_index_topk_workspace_size(const qsa_config* cfg, int32_t max_tokens,
                                     int64_t max_blocks);
qsa_status qsa_index_topk(const qsa_config* cfg, int32_t n_tokens, int32_t max_tokens,
                          const float* q_idx, const float* w_idx,
                          const int32_t* tok_seq, const int32_t* tok_pos,
                          const float* pooled, const int32_t* blk_cells, int64_t n_slots,
                          const int64_t* seq_blk_off, const int32_t* seq_blk_slots,
                          int32_t n_seq, int64_t max_blocks, int64_t n_cells,
                          int32_t* cells, int32_t* count,
                          const int32_t* recomputed, int32_t n_recomputed,
                          void* workspace, size_t ws_bytes, qsa_stream_t stream);

/* qsa_index_topk_noalloc - the pages have no counterpart; this is a
 * convenience of this library.  Same computation and outputs as
 * qsa_index_topk, but the workspace is a static device array inside the
 * library, so the caller passes inputs and outputs only and nothing is
 * allocated.  It is for callers that cannot allocate device memory: plugins
 * hosted by an engine that owns every device allocation through its own pool
 * and gives the plugin no allocator, and code on a latency-critical path where
 * cudaMalloc (which may synchronise the device) is not allowed.
 * Limits: n_tokens <= 8 and max_blocks <= 262144 (1,048,576 cells per
 * sequence at r = 4); larger calls return QSA_ERR_WORKSPACE and launch
 * nothing.  The array takes 9 MiB on every GPU that loads the library, until
 * the process exits.  Every call looks up the array's address in the current
 * device's context (cudaGetSymbolAddress, as every call of the library looks
 * up its device error word); nothing is cached between calls, so the call
 * stays valid after cudaDeviceReset or under another context for the same
 * device.  All calls on a device share
 * the one array: calls whose work overlaps on the GPU (other streams, other
 * host threads) race and corrupt each other's results; serialise them.  Each
 * call clears the part of the array that must start at zero. */
qsa_status qsa_index_topk_noalloc(const qsa_config* cfg, int32_t n_tokens,
                                  const float* q_idx, const float* w_idx,
                                  const int32_t* tok_seq, const int32_t* tok_pos,
                                  const float* pooled, const int32_t* blk_cells, int64_t n_slots,
                                  const int64_t* seq_blk_off, const int32_t* seq_blk_slots,
                                  int32_t n_seq, int64_t max_blocks, int64_t n_cells,
                                  int32_t* cells, int32_t* count, qsa_stream_t stream);

/* ---------------------------------------------------------------------------
 * S5+S6  qsa_sparse_attn  (issue #28734, fix summary, lever1 and sparse256;
 * q8_0: the author's q8-compact follow-up in the same issue)
 * For token t, query head h, KV head g = h / (n_q_heads / n_kv_heads):
 *   out[t][h] = sum_{i < count[t]} softmax_i(attn_scale * q[t][h] . K[c_i][g]) V[c_i][g]
 * with c_i = cells[t][i] (row pitch qsa_cells_per_token).  One thread-block
 * cluster per (token, KV head): its CTAs take 128-cell tiles of the list,
 * compute Q.K^T and P.V on tcgen05 tensor cores (fp16 operands, K/V q8_0
 * rows dequantised to fp16 after the gather, fp32 accumulation), and merge
 * their partial (max, sum, o) through distributed shared memory with
 * log-sum-exp weights.  For fp16 K/V and calls with many tokens (where one
 * CTA per (token, KV head) is the cluster size the cost model gives) the
 * clusters are of two CTAs taking 64-cell tiles, small enough that two
 * share an SM; the result is the same within the stated tolerance.
 * count[t] == 0 gives zeros.  A cell outside [0, n_cells) is masked and
 * flagged.  The call needs no workspace (qsa_sparse_attn_workspace_size
 * returns 0; `workspace` may be NULL). */
size_t qsa_sparse_attn_workspace_size(const qsa_config* cfg, int32_t n_tokens);
qsa_status qsa_sparse_attn(const qsa_config* cfg, int32_t n_tokens,
                           const void* q, const void* k_cache, const void* v_cache,
                           int64_t n_cells, const int32_t* cells, const int32_t* count,
                           float* out, void* workspace, size_t ws_bytes,
                           qsa_stream_t stream);

/* ---------------------------------------------------------------------------
 * S5+S6 for token pairs  qsa_sparse_attn_union  (issue #28734, goodbadwolf's
 * comment on the merged sparse path: the union kernel that multi-token
 * batches run, tokens x heads over the union of their selected cells with a
 * mask per token)
 * Same arguments, layouts, outputs and errors as qsa_sparse_attn.  Tokens 2i
 * and 2i + 1 (any two tokens; they share work only when their lists share
 * cells, i.e. tokens of one sequence) are attended together: one cluster per
 * (pair, KV head) builds the union of the two cell lists in shared memory
 * (a cell on both lists is gathered once), the MMAs carry both tokens' 8 query
 * heads in their 16 columns, and each column's softmax sees only its token's
 * cells.  An odd last token is attended alone.  Each output is the same
 * attention as qsa_sparse_attn's, for lists in which no cell repeats; the
 * tiles hold other cells, so the fp16 rounding of the probabilities and the
 * order of the sums differ (both within 2e-3 max-relative of the exact
 * result for fp16 K/V, 5e-3 for q8_0).  cells_pitch (top_k + r - 1)
 * must be at most 4104, else QSA_ERR_UNSUPPORTED.  Needs no workspace. */
qsa_status qsa_sparse_attn_union(const qsa_config* cfg, int32_t n_tokens,
                                 const void* q, const void* k_cache, const void* v_cache,
                                 int64_t n_cells, const int32_t* cells, const int32_t* count,
                                 float* out, void* workspace, size_t ws_bytes,
                                 qsa_stream_t stream);

/* ---------------------------------------------------------------------------
 * S2+S3+S4+S5+S6  qsa_index_attn  (issue #28734, fix summary, lever3, lever1
 * and sparse256: block-granular top-k, then attention over only the chosen
 * K/V set)
 * qsa_index_topk followed by qsa_sparse_attn in one call: the arguments are
 * the union of theirs, with their meanings, layouts and limits, and the
 * workspace is qsa_index_topk's (same size, same zero-once contract, same
 * scheduling hint).  Outputs: cells and count exactly as qsa_index_topk
 * writes them, out as qsa_sparse_attn computes it.
 * flags = 0: the two calls' kernels in order (score, selection with
 * expansion, attention).
 * flags = QSA_INDEX_ATTN_IN_CLUSTER: when max_blocks <= 65,536,
 * top_k / r <= 1,024, r <= 8 and the attention's cluster size leaves each CTA
 * at most 8 tiles of 128 cells (decode and small verify batches), the
 * selection and the expansion of a token's blocks run inside the attention's
 * thread-block clusters, one cluster per (token, KV head), so no kernel
 * boundary and no global cell list separate them from the gather: the score
 * kernels, then one kernel (otherwise as flags = 0).  The cells and counts
 * are those of qsa_index_topk either way (the same exact selection), and the
 * output equals the two calls' up to the rounding of the split merge.  On a
 * GB300 this mode is slower than flags = 0 (its one large kernel waits longer
 * for its instructions and for free SMs), so it is not the default.
 * flags = QSA_INDEX_ATTN_UNION: the attention of qsa_sparse_attn_union (token
 * pairs over the union of their lists) after the index kernels.
 * qsa_index_attn_kernels says which kernels a call runs.
 * Errors: as qsa_index_topk and qsa_sparse_attn (all pointers required);
 * QSA_ERR_INVALID_ARG for an unknown flag or both flags;
 * QSA_ERR_UNSUPPORTED for QSA_INDEX_ATTN_UNION where qsa_sparse_attn_union
 * would return it. */
#define QSA_INDEX_ATTN_IN_CLUSTER 1u
#define QSA_INDEX_ATTN_UNION 2u
qsa_status qsa_index_attn(const qsa_config* cfg, int32_t n_tokens, int32_t max_tokens,
                          const float* q_idx, const float* w_idx,
                          const int32_t* tok_seq, const int32_t* tok_pos,
                          const float* pooled, const int32_t* blk_cells, int64_t n_slots,
                          const int64_t* seq_blk_off, const int32_t* seq_blk_slots,
                          int32_t n_seq, int64_t max_blocks,
                          const void* q, const void* k_cache, const void* v_cache, int64_t n_cells,
                          int32_t* cells, int32_t* count, float* out,
                          const int32_t* recomputed, int32_t n_recomputed, uint32_t flags,
                          void* workspace, size_t ws_bytes, qsa_stream_t stream);

/* Which kernels (bit k = kernel id k of qsa_profile_kernel) one
 * qsa_index_attn call with these flags launches on the current device: the
 * scores (1, plus 2 when token-tiled), then 3 and 4, or 6 (selection inside
 * the attention clusters; with QSA_INDEX_ATTN_UNION kernel 4 is the union
 * attention).  0 for an invalid configuration, flags or no tokens. */
uint32_t qsa_index_attn_kernels(const qsa_config* cfg, int32_t n_tokens, int32_t n_seq, int64_t max_blocks,
                                uint32_t flags);

/* ---------------------------------------------------------------------------
 * Host helpers (no GPU).
 *
 * qsa_blocks_dirty (issue #28734, fix summary, lever2: "host-side structural
 * compare of member cells", dirty count bucketed to a power of two >= 4):
 * compares two host block tables [n_slots][r]; writes the slots whose rows
 * differ, ascending, padded with -1 to the next power of two >= pad_pow2_min
 * (0 = no padding), into out_dirty (capacity `cap`), and the padded length to
 * *n_dirty.  QSA_ERR_SHAPE if cap is too small (nothing written but *n_dirty). */
qsa_status qsa_blocks_dirty(const int32_t* old_tbl, const int32_t* new_tbl,
                            int64_t n_slots, int32_t r, int32_t* out_dirty,
                            int32_t cap, int32_t* n_dirty, int32_t pad_pow2_min);

/* Synchronises `stream`, reads and clears the device error word of the
 * current device.  QSA_ERR_DEVICE_BOUNDS if a kernel met an out-of-range
 * index since the last check; *flags (if non-null) receives the bit set:
 * 1 slot, 2 cell, 4 block list too short, 8 token position beyond max_blocks,
 * 16 token with a sequence id outside [0, n_seq) or a negative position,
 * 32 a kernel's bounded wait on its own tensor-core work gave up. */
qsa_status qsa_debug_check(qsa_stream_t stream, uint32_t* flags);

/* Measurement hook (host state, process-wide, not for concurrent use from
 * several host threads).  While set, each launch of kernel `kernel` is
 * bracketed by records of `before` and `after` on the launch's stream
 * (cudaEventRecordExternal, so inside a stream capture they become event
 * nodes that timestamp every replay), and cudaEventElapsedTime gives that
 * launch's device time.
 * Kernel ids: 0 pool update (qsa_pool_update), 1 block scores (+ threshold
 * histogram when one token per sequence), 2 threshold histogram of
 * token-tiled scores, 3 cluster select + expansion (qsa_index_topk), 4
 * attention (qsa_sparse_attn), 5 append (qsa_kv_append), 6 selection,
 * expansion and attention in one cluster kernel (qsa_index_attn).  `before`/`after`
 * are cudaEvent_t handles; NULL clears.  QSA_ERR_INVALID_ARG for an unknown
 * id. */
qsa_status qsa_profile_kernel(int32_t kernel, void* before, void* after);

/* Which kernels (bit k = kernel id k above) one qsa_index_topk call of
 * n_tokens tokens over n_seq sequences launches.  Scoring is token-tiled
 * (each pooled row read once per tile of 32 tokens of one sequence and
 * scored on the tensor cores, kernel 1, then kernel 2 builds the threshold
 * histogram) when n_tokens > 8 and n_tokens >= 2 * n_seq; otherwise one pass
 * per token builds the histogram as it scores.  qsa_index_scores follows the same
 * rule, so both calls compute bit-identical scores. */
uint32_t qsa_index_topk_kernels(int32_t n_tokens, int32_t n_seq);

const char* qsa_status_string(qsa_status s);

#ifdef __cplusplus
}
#endif
#endif /* QSA_H */
