"""Plain CPU oracle of the QSA sparse-attention step (NumPy, float64).

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports, links or runs
this module; only the tests, the smoke check and the benchmark's CPU-baseline
leg call it.  It shares no code with the CUDA path: the only module both sides
read is the seeded input generator (qsa_workload), which holds no arithmetic
of the step.

Sources (three web pages on one subject):
  [README]  "llama.cpp-multigpu" README (lukolszewski), sections 1-14.
  [DISC]    llama.cpp discussion #30071, "Qwen3.8-Flash-Next on 6x3090 and
            6x4090 without NVLink ...", announcement and caveats.
  [ISSUE]   llama.cpp issue #28734, "Eval bug: qwen4exp (Qwen3.8-Flash-Next)
            CUDA: decode slows linearly with context": the LLM-written fix
            summary ("Changes", levers 1/2/2b/3, sparse256), wussh's A100
            reproduction (item 3), goodbadwolf's comment on the merged sparse
            path, and the author's q8-compact follow-up.

The pages describe the method in words only.  Where they leave a step open the
oracle takes the plainest reading; every such reading is listed with the
design notes of the repository and repeated at the function that takes it.

Pins (what ties each function to something other than itself) live in
tests/test_oracle_pins.py.  Every function below has at least one.
"""
from __future__ import annotations

from typing import List, Sequence

import numpy as np


# --------------------------------------------------------------------------
# K/V cache decoding
# --------------------------------------------------------------------------
def kv_rows(cfg: dict, cache: np.ndarray, n_cells: int, cells: Sequence[int], g: int) -> np.ndarray:
    """Rows of KV head g for the given cells, as float64 [len(cells)][D].

    f16: the stored half values.  q8_0 ([ISSUE] q8-compact follow-up; the
    README section 1 runs "q8_0 KV cache"): blocks of 32 int8 values along the
    head dimension with one fp16 scale d each; value = float(d) * q.  Byte
    layout: qs int8 [n_cells][G][D] followed by d fp16 [n_cells][G][D/32]."""
    G, D = cfg["n_kv_heads"], cfg["head_dim"]
    cells = np.asarray(cells, dtype=np.int64)
    if cfg["kv_type"] == "f16":
        arr = np.asarray(cache).reshape(n_cells, G, D)
        return arr[cells, g, :].astype(np.float64)
    if cfg["kv_type"] == "q8_0":
        raw = np.asarray(cache).view(np.uint8)
        nq = n_cells * G * D
        qs = raw[:nq].view(np.int8).reshape(n_cells, G, D)
        d = raw[nq:nq + n_cells * G * (D // 32) * 2].view(np.float16).reshape(n_cells, G, D // 32)
        q = qs[cells, g, :].astype(np.float64)
        scale = d[cells, g, :].astype(np.float64)
        return q * np.repeat(scale, 32, axis=1)
    raise ValueError(cfg["kv_type"])


# --------------------------------------------------------------------------
# S1: persistent pooled block-key cache
# --------------------------------------------------------------------------
def rms_norm(m: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """x = m / sqrt(mean(m^2) + eps) * w.  ([ISSUE] lever2 "RMS-normed";
    eps and weight are the workload's: 1e-6 and ones.)"""
    m = np.asarray(m, dtype=np.float64)
    return m / np.sqrt(np.mean(m * m) + eps) * np.asarray(w, dtype=np.float64)


def rope_neox(x: np.ndarray, pos: float, theta: float) -> np.ndarray:
    """NeoX ("half split") rotary embedding of a vector of even length n:
    dims d and d + n/2 form a pair rotated by pos * theta**(-2d/n).
    ([ISSUE] lever2 "re-RoPEd"; the half-split style over all dims and
    theta = 1e6 are the reading of the workload.)"""
    x = np.asarray(x, dtype=np.float64)
    n = x.shape[-1]
    h = n // 2
    d = np.arange(h, dtype=np.float64)
    ang = float(pos) * np.power(float(theta), -2.0 * d / n)
    c, s = np.cos(ang), np.sin(ang)
    a, b = x[..., :h], x[..., h:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def pool_block(cfg: dict, rows: np.ndarray, block_idx: int, norm_w: np.ndarray) -> np.ndarray:
    """Pooled key of one block ([ISSUE] lever2: block keys are "gathered,
    mean-pooled, RMS-normed and re-RoPEd").

    rows: the fp16 indexer keys of the block's present cells (c <= r rows).
    Mean over the present cells -> RMSNorm -> RoPE at the block's first
    position j*r (the pages do not give the position; this is the reading).
    A block with no present cell pools to zeros."""
    rows = np.asarray(rows)
    if rows.shape[0] == 0:
        return np.zeros(cfg["idx_dim"], dtype=np.float64)
    m = rows.astype(np.float64).sum(axis=0) / rows.shape[0]
    x = rms_norm(m, norm_w, cfg["rms_eps"])
    return rope_neox(x, block_idx * cfg["compress_ratio"], cfg["rope_theta"])


def pool_update(cfg: dict, idx_k: np.ndarray, blk_cells: np.ndarray,
                slot_block_idx: np.ndarray, dirty: Sequence[int],
                norm_w: np.ndarray, pooled: np.ndarray) -> np.ndarray:
    """Recompute the pooled rows of the dirty slots only ([ISSUE] lever2:
    "each ubatch recomputes only blocks it dirtied"); -1 entries of the dirty
    list are no-ops (the power-of-two padding of the same lever).  Rows are
    stored as float32.  Returns the updated copy of `pooled`."""
    out = np.array(pooled, dtype=np.float32, copy=True)
    for s in np.asarray(dirty).tolist():
        if s < 0:
            continue
        mem = blk_cells[s]
        present = [int(c) for c in mem if c >= 0]
        out[s] = pool_block(cfg, idx_k[present], int(slot_block_idx[s]), norm_w).astype(np.float32)
    return out


# --------------------------------------------------------------------------
# S2: indexer block scores
# --------------------------------------------------------------------------
def n_full_blocks(cfg: dict, pos: int) -> int:
    """Blocks wholly at or before position p: floor((p+1)/r).  Later blocks
    are fully or partly in the future and get -inf ([ISSUE] lever3)."""
    return (int(pos) + 1) // cfg["compress_ratio"]


def block_scores(cfg: dict, q_idx_t: np.ndarray, w_idx_t: np.ndarray,
                 keys: np.ndarray) -> np.ndarray:
    """S[j] = sum_h w_h * max(0, q_h . k_j) in float64 over the given pooled
    keys (float32 rows as stored).  The pages never write the indexer score
    out ([ISSUE] wussh item 3 names build_qsa_top_k only); this definition is
    the reading the build states, with no extra scale."""
    q = np.asarray(q_idx_t, dtype=np.float64)            # [HI][DI]
    w = np.asarray(w_idx_t, dtype=np.float64)            # [HI]
    k = np.asarray(keys, dtype=np.float64)               # [nb][DI]
    dots = k @ q.T                                       # [nb][HI]
    return np.maximum(dots, 0.0) @ w


def index_scores(cfg: dict, q_idx: np.ndarray, w_idx: np.ndarray,
                 tok_seq: np.ndarray, tok_pos: np.ndarray, pooled: np.ndarray,
                 seq_blk_off: np.ndarray, seq_blk_slots: np.ndarray) -> List[np.ndarray]:
    """Per token t: the scores of blocks j < floor((p_t+1)/r) of its sequence."""
    out = []
    for t in range(len(tok_pos)):
        s = int(tok_seq[t])
        nb = n_full_blocks(cfg, tok_pos[t])
        off = int(seq_blk_off[s])
        slots = np.asarray(seq_blk_slots[off:off + nb], dtype=np.int64)
        out.append(block_scores(cfg, q_idx[t], w_idx[t], pooled[slots]))
    return out


# --------------------------------------------------------------------------
# S3: block-granular top-k
# --------------------------------------------------------------------------
def select_blocks(scores: np.ndarray, n_select: int) -> np.ndarray:
    """The n_select highest-scoring blocks, ties to the lower block index,
    returned ascending ([ISSUE] lever3: blocks are chosen first because the
    budget is whole blocks).  A full stable sort by (-S, j): brute force by
    construction.  Fewer candidates than n_select selects all of them."""
    scores = np.asarray(scores)
    nb = scores.shape[0]
    k = min(int(n_select), nb)
    j = np.arange(nb)
    order = np.lexsort((j, -scores.astype(np.float64)))
    return np.sort(order[:k]).astype(np.int64)


def budget_blocks(cfg: dict) -> int:
    """Whole blocks in the budget: top_k / r = 512; the partial tail block
    rides on top, so at most top_k + r - 1 = 2051 cells ([ISSUE] goodbadwolf:
    n_kv_max = min(n_kv, indexer_top_k + r - 1))."""
    return cfg["top_k"] // cfg["compress_ratio"]


# --------------------------------------------------------------------------
# S4: block -> cell expansion
# --------------------------------------------------------------------------
def expand_cells(cfg: dict, sel: np.ndarray, seq: int, pos: int,
                 blk_cells: np.ndarray, seq_blk_off: np.ndarray,
                 seq_blk_slots: np.ndarray) -> np.ndarray:
    """Cell list of one token: the selected blocks ascending, each block's r
    cells in position order, then the tail cells (positions floor((p+1)/r)*r
    .. p), which are always attended and never scored ([ISSUE] lever3: "the
    incomplete tail block's cells ride a small per-token side input";
    lever2b: expansion through the block-member table)."""
    r = cfg["compress_ratio"]
    off = int(seq_blk_off[seq])
    parts = []
    for j in np.asarray(sel).tolist():
        parts.append(np.asarray(blk_cells[int(seq_blk_slots[off + j])], dtype=np.int64))
    nb = n_full_blocks(cfg, pos)
    tail = int(pos) + 1 - nb * r
    if tail > 0:
        trow = blk_cells[int(seq_blk_slots[off + nb])]
        parts.append(np.asarray(trow[:tail], dtype=np.int64))
    cells = np.concatenate(parts) if parts else np.zeros(0, dtype=np.int64)
    if np.any(cells < 0):
        raise ValueError("a selected or tail position has no cell")
    return cells.astype(np.int32)


def index_topk(cfg: dict, q_idx, w_idx, tok_seq, tok_pos, pooled, blk_cells,
               seq_blk_off, seq_blk_slots, scores: List[np.ndarray] = None):
    """S2 + S3 + S4 for every token.  With `scores` given, selection runs on
    those values (stage isolation: the GPU's own scores) instead of the
    oracle's float64 scores.  Returns (list of cell arrays, list of selected
    block arrays, list of score arrays)."""
    if scores is None:
        scores = index_scores(cfg, q_idx, w_idx, tok_seq, tok_pos, pooled,
                              seq_blk_off, seq_blk_slots)
    B = budget_blocks(cfg)
    cells, sels = [], []
    for t in range(len(tok_pos)):
        sel = select_blocks(scores[t], B)
        sels.append(sel)
        cells.append(expand_cells(cfg, sel, int(tok_seq[t]), int(tok_pos[t]),
                                  blk_cells, seq_blk_off, seq_blk_slots))
    return cells, sels, scores


# --------------------------------------------------------------------------
# S5 + S6: sparse attention over the selected cells
# --------------------------------------------------------------------------
def attend(cfg: dict, q_t: np.ndarray, k_cache, v_cache, n_cells: int,
           cells: np.ndarray) -> np.ndarray:
    """o[h] = sum_c softmax_c(scale * q_h . K_c[g]) V_c[g] over the given cells,
    g = h // (Hq/G), in float64 ([ISSUE] lever1: flash-attention over only the
    finite-mask K/V set; sparse256: DKQ = DV = 256 with 8 query heads per KV
    head).  Scale 1/sqrt(256); no softcap, sink or bias."""
    Hq, G, D = cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"]
    grp = Hq // G
    out = np.zeros((Hq, D), dtype=np.float64)
    if len(cells) == 0:
        return out
    for g in range(G):
        K = kv_rows(cfg, k_cache, n_cells, cells, g)
        V = kv_rows(cfg, v_cache, n_cells, cells, g)
        for h in range(g * grp, (g + 1) * grp):
            s = (K @ q_t[h].astype(np.float64)) * cfg["attn_scale"]
            e = np.exp(s - s.max())
            out[h] = (e / e.sum()) @ V
    return out


def sparse_attn(cfg: dict, q: np.ndarray, k_cache, v_cache, n_cells: int,
                cells: List[np.ndarray]) -> np.ndarray:
    return np.stack([attend(cfg, q[t], k_cache, v_cache, n_cells, cells[t])
                     for t in range(len(cells))])


# --------------------------------------------------------------------------
# Append of new cells (the cache write of the step's own K/V and indexer key)
# --------------------------------------------------------------------------
def q8_0_block(x32: np.ndarray):
    """q8_0 encoding of one block of 32 values ([ISSUE] q8-compact follow-up
    and [README] section 1 run "q8_0" K/V; the pages name the format, not its
    rounding).  Reading: scale d = max|x| / 127 and codes q = x * (1/d)
    rounded half away from zero, clamped to +-127, with every operation in
    float32 (the precision in which the kernel takes the same integer
    decision); d is stored as fp16.  A block of zeros gives d = 0, q = 0.
    Returns (q int8 [32], d float16)."""
    x = np.asarray(x32, dtype=np.float32).reshape(32)
    amax = np.float32(0.0)
    for v in x:
        a = np.float32(abs(v))
        if a > amax:
            amax = a
    d = np.float32(amax / np.float32(127.0))
    inv = np.float32(np.float32(1.0) / d) if d != 0 else np.float32(0.0)
    q = np.zeros(32, dtype=np.int8)
    for i, v in enumerate(x):
        t = np.float32(v * inv)
        a = np.float32(abs(t))
        m = int(np.trunc(a))
        if np.float32(a - np.float32(m)) >= np.float32(0.5):   # half away from zero (a - m is exact)
            m += 1
        m = min(m, 127)
        q[i] = -m if t < 0 else m
    return q, np.float16(d)


def kv_append(cfg: dict, tok_seq, tok_pos, cells, k_new, v_new, idx_new, k_cache, v_cache, idx_k,
              n_cells: int, blk_cells, seq_blk_off, seq_blk_slots, n_dirty: int, inplace: bool = False):
    """Write the step's new cells into the caches and the block table, and
    list the blocks that changed ([ISSUE] lever2b: block members live in a
    device table; lever2: only dirtied blocks are re-pooled, their count padded
    to a power of two by the caller).  For token t at position p of sequence
    s occupying cell c: K/V rows of c <- k_new[t], v_new[t] (fp16 copied, or
    q8_0-encoded per 32-value block by q8_0_block), idx_k[c] <- idx_new[t],
    blk_cells[slot(s, p // r)][p % r] <- c.  dirty = the distinct slots of the
    touched blocks, ascending, padded with -1 to n_dirty entries.
    Returns updated copies (k_cache, v_cache, idx_k, blk_cells) and dirty
    (with inplace=True the given arrays are updated and returned)."""
    r, G, D = cfg["compress_ratio"], cfg["n_kv_heads"], cfg["head_dim"]
    if inplace:
        kc, vc, ik, tbl = k_cache, v_cache, idx_k, blk_cells
    else:
        kc, vc = np.array(k_cache, copy=True), np.array(v_cache, copy=True)
        ik, tbl = np.array(idx_k, copy=True), np.array(blk_cells, copy=True)
    touched = set()
    for t in range(len(tok_pos)):
        s, p, c = int(tok_seq[t]), int(tok_pos[t]), int(cells[t])
        slot = int(seq_blk_slots[int(seq_blk_off[s]) + p // r])
        tbl[slot, p % r] = c
        ik[c] = idx_new[t]
        touched.add(slot)
        for cache, rows in ((kc, k_new[t]), (vc, v_new[t])):
            if cfg["kv_type"] == "f16":
                cache.reshape(n_cells, G, D)[c] = rows
                continue
            raw = cache.view(np.uint8)
            nq = n_cells * G * D
            qs = raw[:nq].view(np.int8).reshape(n_cells, G, D)
            dd = raw[nq:nq + n_cells * G * (D // 32) * 2].view(np.float16).reshape(n_cells, G, D // 32)
            for g in range(G):
                for b in range(D // 32):
                    q, d = q8_0_block(np.asarray(rows[g, 32 * b:32 * b + 32], dtype=np.float32))
                    qs[c, g, 32 * b:32 * b + 32] = q
                    dd[c, g, b] = d
    dirty = np.full(n_dirty, -1, dtype=np.int32)
    srt = sorted(touched)
    if len(srt) > n_dirty:
        raise ValueError("more dirty blocks than the list holds")
    dirty[:len(srt)] = srt
    return kc, vc, ik, tbl, dirty


# --------------------------------------------------------------------------
# One whole step
# --------------------------------------------------------------------------
def run_step(cfg: dict, idx_k, k_cache, v_cache, n_cells, blk_cells,
             slot_block_idx, seq_blk_off, seq_blk_slots, norm_w, pooled, step):
    """pool_update(dirty) -> index_topk -> sparse_attn for one step.
    `step` carries tok_seq, tok_pos, q, q_idx, w_idx, dirty.
    Returns (pooled_after, cells, out)."""
    pooled2 = pool_update(cfg, idx_k, blk_cells, slot_block_idx, step.dirty, norm_w, pooled)
    cells, _, _ = index_topk(cfg, step.q_idx, step.w_idx, step.tok_seq, step.tok_pos,
                             pooled2, blk_cells, seq_blk_off, seq_blk_slots)
    out = sparse_attn(cfg, step.q, k_cache, v_cache, n_cells, cells)
    return pooled2, cells, out
