"""Helpers shared by the GPU parity tests: run steps through the C ABI and
compare with the CPU oracle under the stated tolerances.

Tolerances (stated once, used everywhere):
  pooled keys   GPU: fp32 mean/RMS, the angle reduced exactly in 64-bit
                fixed-point turns (integer arithmetic), fp32 sincospi of the
                remaining fraction of a turn; oracle: float64 throughout:
                |gpu - oracle| <= 1e-6 * max|row|
  scores        fp32 GPU vs float64 oracle over the same pooled keys:
                |gpu - oracle| <= 1e-5 * |oracle| + 1e-6 * max|row|
  selection     exact on the GPU's own scores (integers, bit-exact); against
                the oracle's float64 scores, members may differ only for blocks
                whose oracle score lies within 1e-5 relative of the oracle's
                cutoff score, with equal counts
  attention     per (token, head) row: max|o - ref| / max|ref| <= 2e-3 for fp16
                K/V and 5e-3 for q8_0 K/V
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import qsa_oracle as O
from sparse_attention_long_qsa_gb300 import qsa
from sparse_attention_long_qsa_gb300.layer import QSALayer, append_rows, step_inputs

ATTN_TOL = {"f16": 2e-3, "q8_0": 5e-3}
SEL_REL = 1e-5


def max_rel(out, ref):
    out = np.asarray(out, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    num = np.abs(out - ref).max(axis=-1)
    den = np.abs(ref).max(axis=-1)
    return float((num / np.maximum(den, 1e-30)).max())


def check_pooled(gpu, ora):
    gpu = np.asarray(gpu, dtype=np.float64)
    ora = np.asarray(ora, dtype=np.float64)
    rowmax = np.abs(ora).max(axis=-1, keepdims=True)
    bound = 1e-6 * rowmax
    bad = np.abs(gpu - ora) > bound
    assert not bad.any(), f"pooled mismatch at {np.argwhere(bad)[:5]}: gpu {gpu[bad][:5]} oracle {ora[bad][:5]}"


def check_scores(gpu, ora):
    gpu = np.asarray(gpu, dtype=np.float64)
    ora = np.asarray(ora, dtype=np.float64)
    if len(ora) == 0:
        return
    bound = 1e-5 * np.abs(ora) + 1e-6 * np.abs(ora).max()
    bad = np.abs(gpu - ora) > bound
    assert not bad.any(), f"score mismatch at {np.where(bad)[0][:5]}"


def selected_blocks_from_cells(wl, blk_cells, seq, pos, cells, count):
    """Recover the chosen block indices of a token from its cell list."""
    r = wl.r
    nb = (pos + 1) // r
    tail = pos + 1 - nb * r
    nsel = (count - tail) // r
    assert nsel * r + tail == count
    off = int(wl.seq_blk_off[seq])
    slot_of = {int(wl.seq_blk_slots[off + j]): j for j in range(nb)}
    first_cells = cells[:nsel * r:r]
    # block -> first cell via the table
    cell_to_block = {int(blk_cells[s][0]): j for s, j in slot_of.items()}
    return np.array([cell_to_block[int(c)] for c in first_cells], dtype=np.int64)


def check_selection_q18(sel_gpu, scores_ora, B):
    ref = O.select_blocks(scores_ora, B)
    assert len(sel_gpu) == len(ref)
    a, b = set(sel_gpu.tolist()), set(ref.tolist())
    if a == b:
        return 0
    k = len(ref)
    cutoff = np.sort(np.asarray(scores_ora, dtype=np.float64))[::-1][k - 1]
    for j in a ^ b:
        assert abs(scores_ora[j] - cutoff) <= SEL_REL * abs(cutoff), \
            f"block {j} differs with score {scores_ora[j]} vs cutoff {cutoff}"
    return len(a ^ b)


def to_np(t):
    return t.detach().cpu().numpy()


class Runner:
    """A workload on the GPU, stepped through the C ABI, with the oracle
    state kept alongside for comparison."""

    def __init__(self, wl, warm_check_slots=None, mode="calls"):
        """mode "calls": pool update, index top-k, attention (three calls);
        "index_attn": pool update, then index top-k and attention in one
        qsa_index_attn call; "in_cluster": the same with the selection inside
        the attention clusters; "union": the same with token pairs attended
        over the union of their lists."""
        self.wl = wl
        self.mode = mode
        self.layer = QSALayer.from_workload(wl, 0)
        self.layer.warm(torch.from_numpy(wl.prompt_dirty()).cuda())
        self.step_idx = 0

    def pooled(self):
        return to_np(self.layer.pooled)

    def run_step(self, i):
        wl, L = self.wl, self.layer
        slots, rows = append_rows(wl, i)
        if len(slots):
            L.set_cells(slots, rows)
        st = wl.steps[i]
        inp = step_inputs(st)
        if self.mode in ("index_attn", "in_cluster", "union"):
            L.pool_update(inp["dirty"])
            L.index_attn(inp["tok_seq"], inp["tok_pos"], inp["q_idx"], inp["w_idx"], inp["q"],
                         recomputed=inp["dirty"], in_cluster=self.mode == "in_cluster",
                         union=self.mode == "union")
            out = L.out[:len(st.tok_pos)]
        else:
            out = L.step(**inp)
        torch.cuda.synchronize()
        T = len(st.tok_pos)
        return dict(out=to_np(out), cells=to_np(L.cells[:T]), count=to_np(L.count[:T]),
                    pooled=self.pooled(), table=wl.blk_cells_state(i + 1))

    def gpu_scores(self, st):
        L = self.layer
        T = len(st.tok_pos)
        sc = torch.empty((T, L.max_blocks), dtype=torch.float32, device="cuda")
        inp = step_inputs(st)
        qsa.index_scores(L.cfg, inp["q_idx"], inp["w_idx"], inp["tok_seq"], inp["tok_pos"], L.pooled,
                         L.seq_blk_off, L.seq_blk_slots, L.max_blocks, sc)
        torch.cuda.synchronize()
        return to_np(sc)


def assert_no_device_errors():
    st, flags = qsa.debug_check()
    assert st == 0, f"device error word set: flags={flags:#x}"


def check_step(run: Runner, i: int, *, pool_sample=None, oracle_e2e=True, token_sample=None):
    """Run step i and check every stage against the oracle (stage isolation:
    each stage's oracle is fed the GPU's own upstream result), then the
    end-to-end output when the selections agree."""
    wl = run.wl
    cfg = wl.cfg
    st = wl.steps[i]
    res = run.run_step(i)
    table = res["table"]
    # S1: every dirty slot (or a sample) vs the oracle's pooled key
    dirty = [int(s) for s in st.dirty if s >= 0]
    slots = dirty + list(pool_sample if pool_sample is not None else [])
    for s in slots:
        mem = [int(c) for c in table[s] if c >= 0]
        want = O.pool_block(cfg, wl.idx_k[mem], int(wl.slot_block_idx[s]), wl.norm_w).astype(np.float32)
        check_pooled(res["pooled"][s], want)
    # S2 on the GPU's pooled keys
    gsc = run.gpu_scores(st)
    toks = range(len(st.tok_pos)) if token_sample is None else token_sample
    B = O.budget_blocks(cfg)
    n_swaps = 0
    for t in toks:
        seq, pos = int(st.tok_seq[t]), int(st.tok_pos[t])
        nb = (pos + 1) // wl.r
        off = int(wl.seq_blk_off[seq])
        keys = res["pooled"][wl.seq_blk_slots[off:off + nb]]
        osc = O.block_scores(cfg, st.q_idx[t], st.w_idx[t], keys)
        check_scores(gsc[t, :nb], osc)
        assert np.all(np.isneginf(gsc[t, nb:]))
        # S3+S4 exact on the GPU's own scores
        sel_g = O.select_blocks(gsc[t, :nb], B)
        want_cells = O.expand_cells(cfg, sel_g, seq, pos, table, wl.seq_blk_off, wl.seq_blk_slots)
        cnt = int(res["count"][t])
        assert cnt == len(want_cells)
        np.testing.assert_array_equal(res["cells"][t, :cnt], want_cells)
        assert np.all(res["cells"][t, cnt:] == -1)
        # Q18 against the float64 scores
        n_swaps += check_selection_q18(sel_g, osc, B)
        # S5+S6 on the GPU's cells
        ref = O.attend(cfg, st.q[t], wl.k_cache, wl.v_cache, wl.n_cells, want_cells)
        err = max_rel(res["out"][t], ref)
        assert err <= ATTN_TOL[cfg["kv_type"]], f"token {t}: attention max-rel {err}"
    assert_no_device_errors()
    return res, n_swaps


def run_lists(wl, L, lists, q, union):
    """Attention of len(lists) tokens over explicit cell lists (list t of
    token t) through qsa_sparse_attn or qsa_sparse_attn_union; returns the
    fp32 output [T][n_q_heads][head_dim]."""
    T = len(lists)
    cells = np.full((T, L.pitch), -1, dtype=np.int32)
    count = np.zeros(T, dtype=np.int32)
    for t, c in enumerate(lists):
        cells[t, :len(c)] = c
        count[t] = len(c)
    out = torch.full((T, wl.cfg["n_q_heads"], wl.cfg["head_dim"]), float("nan"), device="cuda")
    qsa.sparse_attn(L.cfg, torch.from_numpy(q).cuda(), L.k_cache, L.v_cache, L.n_cells,
                    torch.from_numpy(cells).cuda(), torch.from_numpy(count).cuda(), out, None, union=union)
    torch.cuda.synchronize()
    return to_np(out)
