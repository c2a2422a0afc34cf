"""Pins of the CPU oracle against what the pages and mathematics fix.

Each test ties an oracle function to something other than itself: a
hand-derived closed form (tests/golden/closed_forms.json), an invariant, a
special case that reduces to a library routine (torch's scaled-dot-product
attention, heapq), or an independent formulation (complex multiplication for
the rotary embedding).  A plausible slip in the oracle (a dropped term, a
wrong sign or index, a transposed operand) fails at least one of them.
"""
import heapq
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import qsa_oracle as O
from qsa_workload import default_cfg, make_workload, quantize_q8_0

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")))
CFG = default_cfg()


# ------------------------------------------------------------------ pooling
@pytest.mark.parametrize("case", ["rope_e0_pos1", "rope_e32_pos1000", "rope_e64_pos1"])
def test_rope_closed_forms(case):
    c = GOLDEN[case]
    x = np.zeros(c["dim"])
    x[c["hot"]] = 1.0
    y = O.rope_neox(x, c["pos"], c["theta"])
    for k, v in c["expect"].items():
        assert y[int(k)] == pytest.approx(v, abs=1e-12)
    rest = [i for i in range(c["dim"]) if str(i) not in c["expect"]]
    assert np.abs(y[rest]).max() == 0.0


def test_rope_matches_complex_rotation():
    """Independent formulation: the pair (d, d+64) is the complex number
    x_d + i x_{d+64}, multiplied by exp(i p theta^(-2d/128))."""
    rng = np.random.default_rng(1)
    x = rng.standard_normal(128)
    for p in (0, 1, 17, 4 * 62_531, 250_511):
        z = x[:64] + 1j * x[64:]
        ang = p * 1e6 ** (-np.arange(64) / 64.0)
        w = z * np.exp(1j * ang)
        y = O.rope_neox(x, p, 1e6)
        np.testing.assert_allclose(y[:64], w.real, rtol=0, atol=1e-12)
        np.testing.assert_allclose(y[64:], w.imag, rtol=0, atol=1e-12)


def test_rope_relative_position():
    """<R(p1)x, R(p2)y> depends only on p1 - p2, and R(-p) undoes R(p)."""
    rng = np.random.default_rng(2)
    x, y = rng.standard_normal(128), rng.standard_normal(128)
    a = O.rope_neox(x, 40, 1e6) @ O.rope_neox(y, 12, 1e6)
    b = O.rope_neox(x, 1040, 1e6) @ O.rope_neox(y, 1012, 1e6)
    assert a == pytest.approx(b, rel=1e-10)
    np.testing.assert_allclose(O.rope_neox(O.rope_neox(x, 777, 1e6), -777, 1e6), x, atol=1e-12)


def test_pool_ones_block0_closed_form():
    c = GOLDEN["pool_ones_block0"]
    rows = np.full((c["rows"], 128), c["value"], dtype=np.float16)
    y = O.pool_block(CFG, rows, c["block"], np.ones(128))
    np.testing.assert_allclose(y, c["expect_each"], rtol=1e-15)


def test_pool_block0_is_unit_rms_mean():
    """At position 0 RoPE is the identity: the pooled key is the mean row
    scaled to mean square ms/(ms+eps)."""
    rng = np.random.default_rng(3)
    rows = rng.standard_normal((4, 128)).astype(np.float16)
    m = rows.astype(np.float64).mean(axis=0)
    y = O.pool_block(CFG, rows, 0, np.ones(128))
    ms = np.mean(m ** 2)
    np.testing.assert_allclose(y, m * math.sqrt(1.0 / (ms + 1e-6)), rtol=1e-13)


def test_pool_norm_invariant_and_scale_invariance():
    rng = np.random.default_rng(4)
    rows = rng.standard_normal((4, 128)).astype(np.float16)
    m = rows.astype(np.float64).mean(axis=0)
    ms = np.mean(m ** 2)
    for j in (0, 1, 999, 62_627):
        y = O.pool_block(CFG, rows, j, np.ones(128))
        assert float(y @ y) == pytest.approx(128 * ms / (ms + 1e-6), rel=1e-12)
    y1 = O.pool_block(CFG, rows, 5, np.ones(128))
    y2 = O.pool_block(CFG, (rows.astype(np.float32) * 4).astype(np.float16), 5, np.ones(128))
    np.testing.assert_allclose(y1, y2, atol=1e-5)


def test_pool_partial_block_means_present_cells():
    """A block with cells [a, b] pools like one holding [a, b, a, b]; the
    order of member cells does not matter."""
    rng = np.random.default_rng(5)
    a, b = rng.standard_normal((2, 128)).astype(np.float16)
    y2 = O.pool_block(CFG, np.stack([a, b]), 7, np.ones(128))
    y4 = O.pool_block(CFG, np.stack([a, b, a, b]), 7, np.ones(128))
    y4r = O.pool_block(CFG, np.stack([b, a, b, a]), 7, np.ones(128))
    np.testing.assert_allclose(y2, y4, rtol=1e-13)
    np.testing.assert_allclose(y4, y4r, rtol=1e-13)


def test_pool_norm_weight_applies_before_rope():
    """The weight scales dims before rotation: with weight 2 everywhere the
    key doubles; with weight on the first half only, the rotated key equals
    the rotation of the half-masked normalised mean."""
    rng = np.random.default_rng(6)
    rows = rng.standard_normal((4, 128)).astype(np.float16)
    y1 = O.pool_block(CFG, rows, 9, np.ones(128))
    y2 = O.pool_block(CFG, rows, 9, np.full(128, 2.0))
    np.testing.assert_allclose(y2, 2 * y1, rtol=1e-13)
    w = np.concatenate([np.ones(64), np.zeros(64)])
    y3 = O.pool_block(CFG, rows, 9, w)
    base = O.pool_block(CFG, rows, 0, w)   # position 0: no rotation
    assert np.all(base[64:] == 0)
    z = (base[:64] + 0j) * np.exp(1j * 36 * 1e6 ** (-np.arange(64) / 64.0))
    np.testing.assert_allclose(y3[:64], z.real, atol=1e-12)
    np.testing.assert_allclose(y3[64:], z.imag, atol=1e-12)


def test_pool_update_touches_only_dirty_slots():
    wl = make_workload(n_seq=1, prompt_len=64, n_steps=1, seed=11)
    tbl = wl.blk_cells_state(1)
    pooled = np.full((wl.n_slots, 128), 7.0, dtype=np.float32)
    out = O.pool_update(wl.cfg, wl.idx_k, tbl, wl.slot_block_idx, np.array([3, -1, 9, -1]), wl.norm_w, pooled)
    changed = np.where(np.any(out != pooled, axis=1))[0].tolist()
    assert changed == [3, 9]
    want = O.pool_block(wl.cfg, wl.idx_k[tbl[3]], int(wl.slot_block_idx[3]), wl.norm_w)
    np.testing.assert_array_equal(out[3], want.astype(np.float32))
    # recomputing an unchanged block is idempotent
    again = O.pool_update(wl.cfg, wl.idx_k, tbl, wl.slot_block_idx, np.array([3]), wl.norm_w, out)
    np.testing.assert_array_equal(again, out)


# ------------------------------------------------------------------ scores
def test_score_closed_form():
    c = GOLDEN["score_basis"]
    s = O.block_scores(CFG, np.array(c["q"]), np.array(c["w"]), np.array([c["key"]]))
    assert s[0] == pytest.approx(c["expect"], abs=1e-15)


def test_score_basis_vectors_pick_coordinates():
    rng = np.random.default_rng(7)
    keys = rng.standard_normal((50, 128)).astype(np.float32)
    w = rng.random(4)
    dims = [3, 70, 127, 0]
    q = np.zeros((4, 128))
    for h, d in enumerate(dims):
        q[h, d] = 1.0
    s = O.block_scores(CFG, q, w, keys)
    want = sum(w[h] * np.maximum(keys[:, d].astype(np.float64), 0) for h, d in enumerate(dims))
    np.testing.assert_allclose(s, want, rtol=1e-14)


def test_score_relu_identity():
    """S(q) + S(-q) = sum_h w_h |q_h . k|  (ReLU(x) + ReLU(-x) = |x|)."""
    rng = np.random.default_rng(8)
    keys = rng.standard_normal((64, 128)).astype(np.float32)
    q = rng.standard_normal((4, 128))
    w = rng.random(4)
    lhs = O.block_scores(CFG, q, w, keys) + O.block_scores(CFG, -q, w, keys)
    rhs = np.abs(keys.astype(np.float64) @ q.T) @ w
    np.testing.assert_allclose(lhs, rhs, rtol=1e-13)
    # one-hot weight isolates a head
    e = np.zeros(4)
    e[2] = 1.0
    np.testing.assert_allclose(O.block_scores(CFG, q, e, keys),
                               np.maximum(keys.astype(np.float64) @ q[2], 0), rtol=1e-14)


def test_index_scores_causal_range():
    wl = make_workload(n_seq=2, prompt_len=[41, 90], n_steps=3, seed=12)
    pooled = np.random.default_rng(0).standard_normal((wl.n_slots, 128)).astype(np.float32)
    for st in wl.steps:
        sc = O.index_scores(wl.cfg, st.q_idx, st.w_idx, st.tok_seq, st.tok_pos, pooled,
                            wl.seq_blk_off, wl.seq_blk_slots)
        for t in range(len(st.tok_pos)):
            assert len(sc[t]) == (int(st.tok_pos[t]) + 1) // 4


# ------------------------------------------------------------------ select
def _nlargest_ref(scores, k):
    """heapq.nlargest on (score, -j): an independent top-k."""
    top = heapq.nlargest(k, ((float(s), -j) for j, s in enumerate(scores)))
    return np.sort(np.array([-j for _, j in top], dtype=np.int64))


@pytest.mark.parametrize("seed", range(6))
def test_select_matches_heap_topk_with_ties(seed):
    rng = np.random.default_rng(100 + seed)
    nb = int(rng.integers(1, 4096))
    k = int(rng.integers(1, 700))
    s = rng.standard_normal(nb)
    if seed % 2:
        s = np.round(s * 3) / 3          # heavy ties
    got = O.select_blocks(s.astype(np.float32), k)
    np.testing.assert_array_equal(got, _nlargest_ref(s.astype(np.float32), min(k, nb)))


def test_select_degenerate_cases():
    np.testing.assert_array_equal(O.select_blocks(np.ones(3000), 512), np.arange(512))
    np.testing.assert_array_equal(O.select_blocks(np.random.rand(300), 512), np.arange(300))
    np.testing.assert_array_equal(O.select_blocks(np.zeros(0), 512), np.zeros(0))
    s = np.zeros(2000)
    s[[5, 1999, 700]] = 1.0
    got = O.select_blocks(s, 4)
    np.testing.assert_array_equal(got, [0, 5, 700, 1999])


# ------------------------------------------------------------------ expand
def test_expand_contiguous_positions():
    wl = make_workload(n_seq=1, prompt_len=9001, n_steps=3, seed=13)
    pooled = np.random.default_rng(1).standard_normal((wl.n_slots, 128)).astype(np.float32)
    for i, st in enumerate(wl.steps):
        tbl = wl.blk_cells_state(i + 1)
        cells, sels, _ = O.index_topk(wl.cfg, st.q_idx, st.w_idx, st.tok_seq, st.tok_pos,
                                      pooled, tbl, wl.seq_blk_off, wl.seq_blk_slots)
        p = int(st.tok_pos[0])
        nb = (p + 1) // 4
        c = cells[0]
        assert len(sels[0]) == min(nb, 512)
        assert len(c) == min(nb, 512) * 4 + (p + 1 - nb * 4)
        assert len(np.unique(c)) == len(c)
        assert c.max() <= p                      # cell == position here
        tail = p + 1 - nb * 4
        np.testing.assert_array_equal(c[len(c) - tail:], np.arange(nb * 4, p + 1))
        body = c[:len(c) - tail].reshape(-1, 4)
        np.testing.assert_array_equal(body // 4, np.repeat(sels[0][:, None], 4, 1))


def test_expand_shuffled_allocation_maps_positions():
    wl = make_workload(n_seq=3, prompt_len=[300, 2100, 5000], n_steps=2, seed=14, shuffled=True)
    pooled = np.random.default_rng(2).standard_normal((wl.n_slots, 128)).astype(np.float32)
    st = wl.steps[1]
    tbl = wl.blk_cells_state(2)
    cells, sels, _ = O.index_topk(wl.cfg, st.q_idx, st.w_idx, st.tok_seq, st.tok_pos,
                                  pooled, tbl, wl.seq_blk_off, wl.seq_blk_slots)
    for t in range(len(st.tok_pos)):
        s, p = int(st.tok_seq[t]), int(st.tok_pos[t])
        inv = {int(c): q for q, c in enumerate(wl.seq_cells[s][:p + 1])}
        pos = np.array([inv[int(c)] for c in cells[t]])
        assert pos.max() <= p and len(np.unique(pos)) == len(pos)
        nb = (p + 1) // 4
        want = np.concatenate([np.arange(j * 4, j * 4 + 4) for j in sels[t]] + [np.arange(nb * 4, p + 1)])
        np.testing.assert_array_equal(pos, want)


# ------------------------------------------------------------------ attention
def _sdpa(q, K, V, scale, mask=None):
    """torch CPU float64 scaled-dot-product attention; q [H][D], K/V [N][D]."""
    qt = torch.from_numpy(np.asarray(q, dtype=np.float64))[None, :, None, :]
    kt = torch.from_numpy(np.asarray(K, dtype=np.float64))[None, None].expand(1, qt.shape[1], -1, -1)
    vt = torch.from_numpy(np.asarray(V, dtype=np.float64))[None, None].expand(1, qt.shape[1], -1, -1)
    m = None if mask is None else torch.from_numpy(mask)[None, None, None, :]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=m, scale=scale)
    return o[0, :, 0, :].numpy()


def test_attend_closed_form():
    c = GOLDEN["attend_two_cells"]
    cfg = default_cfg(n_q_heads=1, n_kv_heads=1, head_dim=2, attn_scale=1.0)
    K = np.array([[0.0, 0.0], [c["logits_after_scale"][1], 0.0]], dtype=np.float16)
    # fp16 cannot hold ln 3 exactly: feed the stored value back into the expectation
    l1 = float(K[1, 0])
    V = np.array(c["v"], dtype=np.float16)
    o = O.attend(cfg, np.array([[1.0, 0.0]], dtype=np.float16), K.reshape(2, 1, 2), V.reshape(2, 1, 2), 2, np.array([0, 1]))
    p1 = math.exp(l1) / (1 + math.exp(l1))
    want = (1 - p1) * np.array(c["v"][0]) + p1 * np.array(c["v"][1])
    np.testing.assert_allclose(o[0], want, rtol=1e-14)
    np.testing.assert_allclose(o[0], c["expect"], atol=2e-3)


def test_attend_gqa_matches_sdpa_and_mask():
    """Sparse attention over a subset == dense attention with -inf outside it
    (torch SDPA, float64, boolean mask), for every query head and its KV head
    h // 8."""
    rng = np.random.default_rng(9)
    n = 300
    k = rng.standard_normal((n, 2, 256)).astype(np.float16)
    v = rng.standard_normal((n, 2, 256)).astype(np.float16)
    q = rng.standard_normal((16, 256)).astype(np.float16)
    sub = np.sort(rng.choice(n, 77, replace=False))
    o = O.attend(CFG, q, k, v, n, sub)
    mask = np.zeros(n, dtype=bool)
    mask[sub] = True
    for g in range(2):
        ref = _sdpa(q[8 * g:8 * g + 8], k[:, g], v[:, g], 1 / 16, mask)
        np.testing.assert_allclose(o[8 * g:8 * g + 8], ref, rtol=1e-10, atol=1e-12)
    # cell order does not matter
    o2 = O.attend(CFG, q, k, v, n, sub[::-1].copy())
    np.testing.assert_allclose(o, o2, rtol=1e-12, atol=1e-13)


def test_attend_special_cases():
    rng = np.random.default_rng(10)
    n = 40
    k = rng.standard_normal((n, 2, 256)).astype(np.float16)
    v = rng.standard_normal((n, 2, 256)).astype(np.float16)
    q = rng.standard_normal((16, 256)).astype(np.float16)
    o = O.attend(CFG, q, k, v, n, np.array([13]))
    for h in range(16):
        np.testing.assert_array_equal(o[h], v[13, h // 8].astype(np.float64))
    k2 = np.repeat(k[:1], n, axis=0)
    sel = np.array([2, 9, 33])
    o = O.attend(CFG, q, k2, v, n, sel)
    for h in range(16):
        np.testing.assert_allclose(o[h], v[sel, h // 8].astype(np.float64).mean(0), rtol=1e-12, atol=1e-14)


def test_q8_0_layout_and_exact_dequant():
    """Values d * k with d a power of two and |k| <= 127 integral round-trip
    exactly, chunk by chunk, through the generator's encoding and the oracle's
    decoding; a wrong chunk index (i % 8 instead of i // 32) or a swapped
    byte region fails."""
    rng = np.random.default_rng(11)
    n, G, D = 5, 2, 256
    x = np.zeros((n, G, D), dtype=np.float32)
    for c in range(n):
        for g in range(G):
            for b in range(8):
                d = 2.0 ** (b - 4 + c - g)
                ks = rng.integers(-126, 127, 32).astype(np.float32)
                ks[rng.integers(0, 32)] = 127.0
                x[c, g, 32 * b:32 * b + 32] = d * ks
    qs, d = quantize_q8_0(x)
    raw = np.concatenate([qs.reshape(-1).view(np.uint8), d.reshape(-1).view(np.uint8)])
    cfg = default_cfg(kv_type="q8_0")
    for g in range(G):
        np.testing.assert_array_equal(O.kv_rows(cfg, raw, n, np.arange(n), g), x[:, g].astype(np.float64))
    # general values: error at most half a step plus 127 times the fp16
    # rounding of the scale (2^-11 relative)
    y = rng.standard_normal((n, G, D)).astype(np.float32)
    qs, d = quantize_q8_0(y)
    raw = np.concatenate([qs.reshape(-1).view(np.uint8), d.reshape(-1).view(np.uint8)])
    for g in range(G):
        got = O.kv_rows(cfg, raw, n, np.arange(n), g)
        step = np.repeat(np.abs(y[:, g]).reshape(n, 8, 32).max(-1) / 127, 32, axis=1)
        assert np.all(np.abs(got - y[:, g]) <= step * (0.5 + 127 * 2.0 ** -11) * 1.0001)


# ------------------------------------------------------------------ whole step
@pytest.mark.parametrize("n", [1, 2, 5, 2048, 2051])
def test_step_degenerates_to_dense_causal(n):
    """With n <= top_k + r - 1 cells every visible block is selected and the
    tail rides along: the step equals dense causal GQA attention of the last
    token over all n cells."""
    wl = make_workload(n_seq=1, prompt_len=n - 1, n_steps=1, seed=20 + n)
    st = wl.steps[0]
    tbl = wl.blk_cells_state(1)
    pooled = np.zeros((wl.n_slots, 128), dtype=np.float32)
    pooled = O.pool_update(wl.cfg, wl.idx_k, tbl, wl.slot_block_idx, wl.prompt_dirty(), wl.norm_w, pooled)
    _, cells, out = O.run_step(wl.cfg, wl.idx_k, wl.k_cache, wl.v_cache, wl.n_cells, tbl,
                               wl.slot_block_idx, wl.seq_blk_off, wl.seq_blk_slots, wl.norm_w, pooled, st)
    assert sorted(cells[0].tolist()) == list(range(n))
    for g in range(2):
        ref = _sdpa(st.q[0, 8 * g:8 * g + 8], wl.k_cache[:n, g], wl.v_cache[:n, g], 1 / 16)
        np.testing.assert_allclose(out[0, 8 * g:8 * g + 8], ref, rtol=1e-10, atol=1e-12)


def test_step_past_budget_is_sparse():
    """At n = 2052 the budget binds: 512 blocks + 0 tail = 2048 cells, and the
    result equals dense attention masked to those cells."""
    n = 2052
    wl = make_workload(n_seq=1, prompt_len=n - 1, n_steps=1, seed=31)
    st = wl.steps[0]
    tbl = wl.blk_cells_state(1)
    pooled = O.pool_update(wl.cfg, wl.idx_k, tbl, wl.slot_block_idx, wl.prompt_dirty(), wl.norm_w,
                           np.zeros((wl.n_slots, 128), dtype=np.float32))
    _, cells, out = O.run_step(wl.cfg, wl.idx_k, wl.k_cache, wl.v_cache, wl.n_cells, tbl,
                               wl.slot_block_idx, wl.seq_blk_off, wl.seq_blk_slots, wl.norm_w, pooled, st)
    assert len(cells[0]) == 2048
    mask = np.zeros(n, dtype=bool)
    mask[cells[0]] = True
    ref = _sdpa(st.q[0, :8], wl.k_cache[:n, 0], wl.v_cache[:n, 0], 1 / 16, mask)
    np.testing.assert_allclose(out[0, :8], ref, rtol=1e-10, atol=1e-12)


# ------------------------------------------------------------------ append
def _q8_cases():
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "q8_0_blocks.json")))
    return [(k, v) for k, v in g.items() if not k.startswith("_")]


@pytest.mark.parametrize("name,case", _q8_cases())
def test_q8_0_block_closed_forms(name, case):
    x = np.zeros(32, np.float32)
    x[:len(case["x"])] = case["x"]
    q, d = O.q8_0_block(x)
    want = np.zeros(32, np.int8)
    want[:len(case["q"])] = case["q"]
    np.testing.assert_array_equal(q, want)
    assert float(d) == case["d"]


@pytest.mark.parametrize("name,case", _q8_cases())
def test_input_encoder_closed_forms(name, case):
    """The workload generator's own q8_0 encoder on the same hand-derived
    blocks (its codes are the bytes the GPU append must reproduce)."""
    x = np.zeros((1, 32), np.float32)
    x[0, :len(case["x"])] = case["x"]
    qs, d = quantize_q8_0(x)
    want = np.zeros(32, np.int8)
    want[:len(case["q"])] = case["q"]
    np.testing.assert_array_equal(qs[0], want)
    assert float(d[0, 0]) == case["d"]


def test_q8_0_block_error_bound_and_extremes():
    rng = np.random.default_rng(5)
    for _ in range(200):
        x = (rng.standard_normal(32) * rng.uniform(1e-3, 1e3)).astype(np.float32)
        q, d = O.q8_0_block(x)
        d32 = np.abs(x).max() / 127.0
        # codes are within half a step of x/d; the largest magnitude maps to +-127
        assert np.all(np.abs(x - d32 * q.astype(np.float64)) <= 0.5 * d32 * (1 + 1e-5))
        k = int(np.argmax(np.abs(x)))
        assert abs(int(q[k])) == 127 and np.sign(q[k]) == np.sign(x[k])
        assert abs(float(d) - d32) <= d32 * 2.0 ** -11


def test_q8_0_block_agrees_with_the_input_encoder():
    """The workload generator encodes its q8_0 caches with its own code; the
    two independent implementations of the same reading agree bit for bit."""
    rng = np.random.default_rng(6)
    x = rng.standard_normal((64, 256)).astype(np.float16).astype(np.float32)
    qs, d = quantize_q8_0(x)
    for i in range(64):
        for b in range(8):
            q1, d1 = O.q8_0_block(x[i, 32 * b:32 * b + 32])
            np.testing.assert_array_equal(q1, qs[i, 32 * b:32 * b + 32])
            assert d1 == d[i, b]


@pytest.mark.parametrize("kv_type,shuffled,tps", [("f16", False, 1), ("q8_0", True, 1), ("q8_0", False, 5)])
def test_kv_append_reproduces_the_workload_state(kv_type, shuffled, tps):
    """Appending a step's new cells to the state before it gives the state
    after it: the generator wrote every cell's encoded row up front, so the
    caches must come out byte-identical, the table equal to the next state,
    and the dirty list equal to the step's."""
    n_seq = 1 if tps > 1 else 3
    wl = make_workload(n_seq=n_seq, prompt_len=[103, 58, 9][:n_seq], n_steps=3, tokens_per_step=tps,
                       seed=31, shuffled=shuffled, kv_type=kv_type)
    for i in range(3):
        st = wl.steps[i]
        kc, vc, ik, tbl, dirty = O.kv_append(wl.cfg, st.tok_seq, st.tok_pos, st.cells, st.k_new, st.v_new,
                                             st.idx_new, wl.k_cache, wl.v_cache, wl.idx_k, wl.n_cells,
                                             wl.blk_cells_state(i), wl.seq_blk_off, wl.seq_blk_slots,
                                             len(st.dirty))
        np.testing.assert_array_equal(kc.view(np.uint8), np.asarray(wl.k_cache).view(np.uint8))
        np.testing.assert_array_equal(vc.view(np.uint8), np.asarray(wl.v_cache).view(np.uint8))
        np.testing.assert_array_equal(ik, wl.idx_k)
        np.testing.assert_array_equal(tbl, wl.blk_cells_state(i + 1))
        np.testing.assert_array_equal(dirty, st.dirty)


def test_kv_append_writes_only_the_new_cells():
    wl = make_workload(n_seq=2, prompt_len=[40, 21], n_steps=1, seed=32, kv_type="q8_0")
    st = wl.steps[0]
    zk = np.zeros_like(wl.k_cache)
    kc, vc, ik, tbl, dirty = O.kv_append(wl.cfg, st.tok_seq, st.tok_pos, st.cells, st.k_new, st.v_new,
                                         st.idx_new, zk, zk, np.zeros_like(wl.idx_k), wl.n_cells,
                                         wl.blk_cells_state(0), wl.seq_blk_off, wl.seq_blk_slots, 8)
    others = np.setdiff1d(np.arange(wl.n_cells), st.cells)
    assert not O.kv_rows(wl.cfg, kc, wl.n_cells, others, 0).any()
    assert not ik[others].any()
    # the new rows dequantise to within half a step of their fp16 source
    for t, c in enumerate(st.cells):
        for g in range(2):
            got = O.kv_rows(wl.cfg, kc, wl.n_cells, [c], g)[0]
            src = st.k_new[t, g].astype(np.float64)
            step = np.repeat(np.abs(src.reshape(8, 32)).max(1) / 127.0, 32)
            assert np.all(np.abs(got - src) <= 0.5 * step + 127 * step * 2.0 ** -11 + 1e-12)
    assert list(dirty[:2]) == sorted(dirty[:2]) and np.all(dirty[2:] == -1)
