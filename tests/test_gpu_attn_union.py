"""qsa_sparse_attn_union (and qsa_index_attn with QSA_INDEX_ATTN_UNION): token
pairs (2i, 2i + 1) attended over the union of their cell lists with a mask
per token.  Every token's output is checked against the oracle over its own
list (the same tolerance as qsa_sparse_attn), on lists with full, partial and
no overlap, empty and odd cases, invalid cells, every budget, and through the
whole index step."""
import numpy as np
import pytest
import torch

from oracle import qsa_oracle as O
from qsa_workload import make_workload
from sparse_attention_long_qsa_gb300 import qsa
from sparse_attention_long_qsa_gb300.layer import QSALayer, append_rows, step_inputs

from gpu_util import ATTN_TOL, Runner, assert_no_device_errors, check_step, max_rel, run_lists, to_np

pytestmark = pytest.mark.gpu


def _cache(kv_type, n, seed, top_k=2048):
    wl = make_workload(n_seq=1, prompt_len=n, n_steps=1, seed=seed, kv_type=kv_type, cfg={"top_k": top_k})
    L = QSALayer.from_workload(wl, 0, max_tokens=16)
    return wl, L


@pytest.mark.parametrize("kv_type", ["f16", "q8_0"])
def test_overlap_patterns(kv_type):
    """Pairs with identical lists, disjoint lists, half-shared lists in
    different orders and lengths, an empty first list, and an odd last token."""
    wl, L = _cache(kv_type, 40_000, 900 + (kv_type == "q8_0"))
    rng = np.random.default_rng(901)
    perm = rng.permutation(wl.n_cells).astype(np.int32)
    a = perm[:2051]
    b = perm[2051:4102]
    shared = perm[5000:6000]
    c0 = np.concatenate([shared, perm[7000:8051]])            # 2051 cells
    c1 = rng.permutation(np.concatenate([shared[::-1], perm[9000:9500]]))   # 1500, half of c0's shared
    lists = [a, a, a, b, c0, c1, np.zeros(0, np.int32), perm[12000:12300], perm[13000:13777]]
    T = len(lists)
    q = rng.standard_normal((T, 16, 256)).astype(np.float16)
    out = run_lists(wl, L, lists, q, union=True)
    ref_tok = run_lists(wl, L, lists, q, union=False)
    tol = ATTN_TOL[kv_type]
    for t in range(T):
        if len(lists[t]) == 0:
            assert np.all(out[t] == 0)
            continue
        ref = O.attend(wl.cfg, q[t], wl.k_cache, wl.v_cache, wl.n_cells, lists[t])
        assert max_rel(out[t], ref) <= tol, f"token {t}"
        assert max_rel(out[t], ref_tok[t]) <= tol, f"token {t} vs the per-token kernel"
    assert_no_device_errors()


def test_identical_tokens_give_identical_bits():
    """Two tokens with the same query and the same list fill the two halves
    of every MMA with the same rows: their outputs are equal bit for bit."""
    wl, L = _cache("f16", 30_000, 910)
    rng = np.random.default_rng(911)
    lst = rng.permutation(wl.n_cells)[:2051].astype(np.int32)
    q1 = rng.standard_normal((1, 16, 256)).astype(np.float16)
    q = np.concatenate([q1, q1])
    out = run_lists(wl, L, [lst, lst], q, union=True)
    assert np.array_equal(out[0], out[1])


@pytest.mark.parametrize("kv_type,top_k,n", [("f16", 16, 403), ("f16", 256, 9_001), ("f16", 4096, 30_003),
                                              ("q8_0", 4096, 30_003), ("q8_0", 512, 5_001)])
def test_budgets(kv_type, top_k, n):
    """One tile per pair, several tiles per CTA (top_k 4096: up to 65 union
    tiles), a 5-token verify step through the index kernels."""
    wl = make_workload(n_seq=1, prompt_len=n - 5, n_steps=2, tokens_per_step=5, seed=920 + top_k,
                       kv_type=kv_type, cfg={"top_k": top_k})
    run = Runner(wl, mode="union")
    for i in range(2):
        check_step(run, i)


@pytest.mark.parametrize("kv_type", ["f16", "q8_0"])
def test_multi_seq_shuffled_batches(kv_type):
    """Pairs that straddle two sequences (no shared cells) and pairs within
    one, over shuffled cells and slots."""
    wl = make_workload(n_seq=3, prompt_len=[3_001, 9_001, 20_002], n_steps=2, tokens_per_step=3, seed=930,
                       shuffled=True, kv_type=kv_type)
    run = Runner(wl, mode="union")
    for i in range(2):
        check_step(run, i, pool_sample=range(0, wl.n_slots, 211))


def test_equals_the_separate_calls_on_a_prefill_slice():
    """40 consecutive tokens of one sequence: qsa_index_attn with the union
    flag writes the same cells and counts as the two calls, and outputs within
    the attention tolerance of the per-token kernel's."""
    wl = make_workload(n_seq=1, prompt_len=30_000, n_steps=1, tokens_per_step=40, seed=940)
    L = QSALayer.from_workload(wl, 0)
    L.warm(torch.from_numpy(wl.prompt_dirty()).cuda())
    L.set_cells(*append_rows(wl, 0))
    st = wl.steps[0]
    inp = step_inputs(st)
    T = len(st.tok_pos)
    L.pool_update(inp["dirty"])
    L.index_topk(inp["tok_seq"], inp["tok_pos"], inp["q_idx"], inp["w_idx"])
    L.sparse_attn(inp["q"], T)
    torch.cuda.synchronize()
    c0, n0, o0 = L.cells[:T].clone(), L.count[:T].clone(), to_np(L.out[:T])
    L.out.fill_(float("nan"))
    L.index_attn(inp["tok_seq"], inp["tok_pos"], inp["q_idx"], inp["w_idx"], inp["q"], union=True)
    torch.cuda.synchronize()
    assert torch.equal(L.cells[:T], c0) and torch.equal(L.count[:T], n0)
    out = to_np(L.out[:T])
    cells, count = to_np(c0), to_np(n0)
    for t in range(T):
        ref = O.attend(wl.cfg, st.q[t], wl.k_cache, wl.v_cache, wl.n_cells, cells[t, :count[t]])
        assert max_rel(out[t], ref) <= ATTN_TOL["f16"]
        assert max_rel(out[t], o0[t]) <= ATTN_TOL["f16"]
    assert_no_device_errors()


def test_invalid_cells_are_flagged_and_masked():
    """An out-of-range cell in either list of a pair is reported and left
    out of that token's attention."""
    wl, L = _cache("f16", 20_000, 950)
    rng = np.random.default_rng(951)
    perm = rng.permutation(wl.n_cells).astype(np.int32)
    a = perm[:700].copy()
    b = np.concatenate([perm[300:900], perm[5000:5100]]).astype(np.int32)
    a_bad, b_bad = a.copy(), b.copy()
    a_bad[10] = wl.n_cells + 3
    b_bad[650] = -7
    q = rng.standard_normal((2, 16, 256)).astype(np.float16)
    qsa.debug_check()
    out = run_lists(wl, L, [a_bad, b_bad], q, union=True)
    st_, flags = qsa.debug_check()
    assert st_ == -6 and (flags & 2)
    for t, lst in enumerate((np.delete(a, 10), np.delete(b, 650))):
        ref = O.attend(wl.cfg, q[t], wl.k_cache, wl.v_cache, wl.n_cells, lst)
        assert max_rel(out[t], ref) <= ATTN_TOL["f16"]


def test_limits_and_flags():
    wl, L = _cache("f16", 2_000, 960, top_k=8192)
    cells = torch.full((2, L.pitch), -1, dtype=torch.int32, device="cuda")
    count = torch.zeros(2, dtype=torch.int32, device="cuda")
    q = torch.zeros((2, 16, 256), dtype=torch.float16, device="cuda")
    out = torch.zeros((2, 16, 256), dtype=torch.float32, device="cuda")
    with pytest.raises(qsa.QSAError, match="UNSUPPORTED"):
        qsa.sparse_attn(L.cfg, q, L.k_cache, L.v_cache, L.n_cells, cells, count, out, None, union=True)
    assert qsa.index_attn_kernels(L.cfg, 2, 1, L.max_blocks, union=True) == []
    wl2, L2 = _cache("f16", 5_000, 961)
    assert qsa.index_attn_kernels(L2.cfg, 5, 1, L2.max_blocks, in_cluster=True, union=True) == []
    assert "attn" in qsa.index_attn_kernels(L2.cfg, 5, 1, L2.max_blocks, union=True)
