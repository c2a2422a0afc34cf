"""qsa_index_attn: index top-k and sparse attention in one call; with
QSA_INDEX_ATTN_IN_CLUSTER the selection and expansion run inside the
attention's thread-block clusters where the call's limits allow.  Every stage is checked against the oracle as for the
separate calls (tests/gpu_util.check_step), and the outputs against the
separate calls on the same inputs."""
import numpy as np
import pytest
import torch

from oracle import qsa_oracle as O
from qsa_workload import make_workload
from sparse_attention_long_qsa_gb300 import qsa
from sparse_attention_long_qsa_gb300.layer import QSALayer, append_rows, step_inputs

from gpu_util import ATTN_TOL, Runner, assert_no_device_errors, check_step, max_rel, to_np

pytestmark = pytest.mark.gpu


def _fused(L, T, n_seq):
    return "select_attn" in qsa.index_attn_kernels(L.cfg, T, n_seq, L.max_blocks, in_cluster=True)


def test_tiny_and_budget_edges():
    for n in (1, 4, 7, 2050, 2051, 2052, 4096):
        wl = make_workload(n_seq=1, prompt_len=n - 1, n_steps=1, seed=500 + n)
        run = Runner(wl, mode="in_cluster")
        assert _fused(run.layer, 1, 1)
        res, _ = check_step(run, 0)
        nb = n // 4
        assert int(res["count"][0]) == min(nb, 512) * 4 + n % 4


@pytest.mark.parametrize("kv_type", ["f16", "q8_0"])
def test_multi_seq_shuffled_decode(kv_type):
    wl = make_workload(n_seq=3, prompt_len=[3001, 9001, 20_002], n_steps=4, seed=505, shuffled=True,
                       kv_type=kv_type)
    run = Runner(wl, mode="in_cluster")
    assert _fused(run.layer, 3, 3)
    for i in range(4):
        check_step(run, i, pool_sample=range(0, wl.n_slots, 211))


@pytest.mark.parametrize("top_k,n,kv_type", [(16, 403, "f16"), (256, 9_001, "f16"), (512, 600, "f16"),
                                              (4096, 30_003, "f16"), (256, 9_001, "q8_0"),
                                              (4096, 30_003, "q8_0")])
def test_other_budgets(top_k, n, kv_type):
    """One tile, 2-CTA clusters with overflow cells, exactly NC tiles, and
    several tiles per CTA (top_k 4096: 33 tiles over 16 CTAs)."""
    wl = make_workload(n_seq=1, prompt_len=n - 1, n_steps=2, seed=600 + top_k, cfg={"top_k": top_k},
                       kv_type=kv_type)
    run = Runner(wl, mode="in_cluster")
    assert _fused(run.layer, 1, 1)
    for i in range(2):
        res, _ = check_step(run, i)
        assert int(res["count"][0]) == min((n + i) // 4, top_k // 4) * 4 + (n + i) % 4


@pytest.mark.parametrize("tps,kv_type", [(5, "q8_0"), (8, "f16")])
def test_verify_batches(tps, kv_type):
    """Several consecutive tokens of one sequence (clusters of 8 or 4 CTAs,
    several tiles per CTA)."""
    wl = make_workload(n_seq=1, prompt_len=40_001, n_steps=2, tokens_per_step=tps, seed=610 + tps,
                       kv_type=kv_type)
    run = Runner(wl, mode="in_cluster")
    assert _fused(run.layer, tps, 1)
    for i in range(2):
        check_step(run, i)


def test_many_tokens_fall_back_to_the_separate_kernels():
    """Past the fused limits (here: a cluster size that would leave a CTA more
    than 8 tiles) the call runs the index and attention kernels in order."""
    wl = make_workload(n_seq=1, prompt_len=10_001, n_steps=1, tokens_per_step=40, seed=620)
    run = Runner(wl, mode="in_cluster")
    assert not _fused(run.layer, 40, 1)
    check_step(run, 0)


@pytest.mark.parametrize("kv_type,seed", [("f16", 701), ("q8_0", 702)])
def test_equals_the_separate_calls(kv_type, seed):
    """Same inputs through qsa_index_topk + qsa_sparse_attn and through
    qsa_index_attn: identical cells and counts, the same attention output."""
    wl = make_workload(n_seq=2, prompt_len=[25_001, 7_003], n_steps=3, seed=seed, shuffled=True, kv_type=kv_type)
    L = QSALayer.from_workload(wl, 0)
    L.warm(torch.from_numpy(wl.prompt_dirty()).cuda())
    T = len(wl.steps[0].tok_pos)
    for i in range(3):
        L.set_cells(*append_rows(wl, i))
        inp = step_inputs(wl.steps[i])
        L.pool_update(inp["dirty"])
        L.index_topk(inp["tok_seq"], inp["tok_pos"], inp["q_idx"], inp["w_idx"])
        L.sparse_attn(inp["q"], T)
        torch.cuda.synchronize()
        c0, n0, o0 = L.cells[:T].clone(), L.count[:T].clone(), L.out[:T].clone()
        L.cells.fill_(7)
        L.count.fill_(-5)
        L.out.fill_(float("nan"))
        L.index_attn(inp["tok_seq"], inp["tok_pos"], inp["q_idx"], inp["w_idx"], inp["q"], in_cluster=True)
        torch.cuda.synchronize()
        assert torch.equal(L.count[:T], n0)
        assert torch.equal(L.cells[:T], c0)
        assert max_rel(to_np(L.out[:T]), to_np(o0)) <= 1e-6
        # the default mode runs the two calls' kernels: the same bits
        L.out.fill_(float("nan"))
        L.index_attn(inp["tok_seq"], inp["tok_pos"], inp["q_idx"], inp["w_idx"], inp["q"])
        torch.cuda.synchronize()
        assert torch.equal(L.out[:T], o0) and torch.equal(L.cells[:T], c0)
    assert_no_device_errors()


@pytest.mark.parametrize("T", [1, 5])
def test_threshold_bins_of_every_size(T):
    """Pooled rows c_s * v make every score c_s times one factor per token;
    400 slots get c in [2^12, 2^16), K slots c within 1e-4 of 2^8 (one
    histogram bin), the rest c in [1, 16), so the 512-block cut falls in a
    bin of exactly K keys: K = 600 is ranked in CTA 0, K = 1,500 and 5,000
    take the radix rounds across the cluster.  Each choice equals a stable
    sort of the GPU's own scores; the attention matches the oracle on it."""
    wl = make_workload(n_seq=1, prompt_len=200_000, n_steps=1, tokens_per_step=T, seed=330 + T)
    L = QSALayer.from_workload(wl, 0)
    assert _fused(L, T, 1)
    L.set_cells(*append_rows(wl, 0))
    st = wl.steps[0]
    inp = step_inputs(st)
    table = wl.blk_cells_state(1)
    g = torch.Generator(device="cpu").manual_seed(T)
    v = torch.from_numpy(st.q_idx[0, 0].astype(np.float32))
    sc = torch.empty((T, L.max_blocks), dtype=torch.float32, device="cuda")
    for k_bin in (600, 1_500, 5_000):
        perm = torch.randperm(L.n_slots, generator=g)
        u = torch.rand(L.n_slots, generator=g, dtype=torch.float64)
        c = torch.exp2(u * 4.0)
        c[perm[:400]] = torch.exp2(12.0 + u[perm[:400]] * 4.0)
        mid = perm[400:400 + k_bin]
        c[mid] = 256.0 * (1.0 + 1e-4 * u[mid])
        L.pooled.copy_((c.float()[:, None] * v[None, :]).cuda())
        L.index_attn(inp["tok_seq"], inp["tok_pos"], inp["q_idx"], inp["w_idx"], inp["q"], in_cluster=True)
        qsa.index_scores(L.cfg, inp["q_idx"], inp["w_idx"], inp["tok_seq"], inp["tok_pos"], L.pooled,
                         L.seq_blk_off, L.seq_blk_slots, L.max_blocks, sc)
        torch.cuda.synchronize()
        scores = to_np(sc)
        out = to_np(L.out[:T])
        for t in range(T):
            seq, pos = int(st.tok_seq[t]), int(st.tok_pos[t])
            nb = (pos + 1) // 4
            sel = O.select_blocks(scores[t, :nb], 512)
            want = O.expand_cells(wl.cfg, sel, seq, pos, table, wl.seq_blk_off, wl.seq_blk_slots)
            np.testing.assert_array_equal(to_np(L.cells[t, :len(want)]), want)
            assert int(L.count[t]) == len(want)
            assert np.all(to_np(L.cells[t, len(want):]) == -1)
            ref = O.attend(wl.cfg, st.q[t], wl.k_cache, wl.v_cache, wl.n_cells, want)
            assert max_rel(out[t], ref) <= ATTN_TOL["f16"]
    assert_no_device_errors()


def test_out_of_range_table_entries_are_flagged():
    """A bad member cell in a chosen block and a bad tail cell are reported and
    masked, as qsa_index_topk does."""
    wl = make_workload(n_seq=1, prompt_len=4_002, n_steps=1, seed=640)
    L = QSALayer.from_workload(wl, 0)
    L.warm(torch.from_numpy(wl.prompt_dirty()).cuda())
    L.set_cells(*append_rows(wl, 0))
    st = wl.steps[0]
    inp = step_inputs(st)
    qsa.debug_check()
    # every block is chosen at this size (1,000 blocks > 512: not all) - make block 0
    # and the tail hold an out-of-range cell
    L.blk_cells[int(wl.seq_blk_slots[0]), 2] = wl.n_cells + 5
    nb = (int(st.tok_pos[0]) + 1) // 4
    L.blk_cells[int(wl.seq_blk_slots[nb]), 0] = wl.n_cells + 9
    L.index_attn(inp["tok_seq"], inp["tok_pos"], inp["q_idx"], inp["w_idx"], inp["q"], in_cluster=True)
    st_, flags = qsa.debug_check()
    assert st_ == -6 and (flags & 2)
    assert torch.isfinite(L.out[0]).all()
