"""GPU parity: every stage of the step through the C ABI against the oracle,
at sizes the oracle finishes in seconds (several tiles, ragged tails), plus
the degenerate cases of the method.  Tolerances: tests/gpu_util.py."""
import numpy as np
import pytest
import torch

from oracle import qsa_oracle as O
from qsa_workload import make_workload
from sparse_attention_long_qsa_gb300 import qsa
from sparse_attention_long_qsa_gb300.layer import QSALayer, append_rows, step_inputs

from gpu_util import (ATTN_TOL, Runner, assert_no_device_errors, check_pooled, check_step, max_rel,
                      to_np)

pytestmark = pytest.mark.gpu


def _all_slots_vs_oracle(run: Runner, table):
    wl = run.wl
    pooled = run.pooled()
    want = O.pool_update(wl.cfg, wl.idx_k, table, wl.slot_block_idx, np.arange(wl.n_slots),
                         wl.norm_w, np.zeros_like(pooled))
    check_pooled(pooled, want)


def test_pool_warm_all_slots_and_idempotent():
    wl = make_workload(n_seq=3, prompt_len=[2999, 9001, 4094], n_steps=2, seed=3, shuffled=True)
    run = Runner(wl)
    _all_slots_vs_oracle(run, wl.blk_cells_state(0))
    before = run.layer.pooled.clone()
    # recomputing unchanged blocks is bit-identical (padding entries are no-ops)
    run.layer.pool_update(np.array([5, -1, 17, -1, 0, -1, -1, -1], dtype=np.int32))
    torch.cuda.synchronize()
    assert torch.equal(before, run.layer.pooled)
    # rebuilding everything from the key cache reproduces the cache bit for bit
    run.layer.pooled.zero_()
    run.layer.warm(torch.from_numpy(wl.prompt_dirty()).cuda())
    torch.cuda.synchronize()
    assert torch.equal(before, run.layer.pooled)
    assert_no_device_errors()


def test_pool_partial_and_empty_blocks():
    wl = make_workload(n_seq=1, prompt_len=4097, n_steps=5, seed=4)
    run = Runner(wl)
    tbl = wl.blk_cells_state(0).copy()
    # slot 1025 holds no cell yet: pools to zeros
    L = run.layer
    L.set_cells([1025], tbl[[1025]])
    L.pool_update(np.array([1024, 1025, -1, -1], dtype=np.int32))
    torch.cuda.synchronize()
    p = run.pooled()
    assert np.all(p[1025] == 0)
    want = O.pool_block(wl.cfg, wl.idx_k[[c for c in tbl[1024] if c >= 0]], 1024, wl.norm_w)
    check_pooled(p[1024], want.astype(np.float32))


def test_tiny_decode_step():
    wl = make_workload("tiny")
    run = Runner(wl)
    res, swaps = check_step(run, 0, pool_sample=range(0, wl.n_slots, 37))
    assert int(res["count"][0]) == 2048
    assert swaps == 0


@pytest.mark.parametrize("kv_type", ["f16", "q8_0"])
def test_multi_seq_shuffled_decode(kv_type):
    wl = make_workload(n_seq=3, prompt_len=[3001, 9001, 20_002], n_steps=5, seed=5, shuffled=True,
                       kv_type=kv_type)
    run = Runner(wl)
    for i in range(5):
        check_step(run, i, pool_sample=range(0, wl.n_slots, 101))
    _all_slots_vs_oracle(run, wl.blk_cells_state(5))


def test_prefill_chunk_causal():
    wl = make_workload(n_seq=1, prompt_len=10_001, n_steps=1, tokens_per_step=96, seed=6)
    run = Runner(wl)
    res, _ = check_step(run, 0)
    st = wl.steps[0]
    # causality: no token sees a cell past its own position
    for t in range(len(st.tok_pos)):
        cnt = int(res["count"][t])
        assert np.all(res["cells"][t, :cnt] <= st.tok_pos[t])


@pytest.mark.parametrize("T", [20, 40])
def test_multi_token_select_cluster_sizes(T):
    """Selection clusters shrink as tokens grow (8 CTAs for a few tokens, 4 at
    20 tokens, 2 at 40, 1 at 96 on a 152-SM GPU): each size is exact."""
    wl = make_workload(n_seq=1, prompt_len=10_001, n_steps=1, tokens_per_step=T, seed=7 + T)
    run = Runner(wl)
    res, _ = check_step(run, 0)
    st = wl.steps[0]
    for t in range(T):
        cnt = int(res["count"][t])
        assert np.all(res["cells"][t, :cnt] <= st.tok_pos[t])


@pytest.mark.parametrize("n_seq,tps,kv_type", [(3, 3, "f16"), (2, 6, "q8_0"), (2, 12, "f16"),
                                              (3, 170, "f16"), (2, 256, "q8_0")])
def test_batched_verify_several_sequences(n_seq, tps, kv_type):
    """Several tokens per sequence for several sequences (token-tiled scoring
    with more than one sequence in a token tile, shuffled slots and cells);
    510-512 tokens: one selection CTA and one attention CTA per (token, KV
    head) in the cost models, i.e. the two-CTAs-per-SM fp16 attention and the
    pipelined q8_0 one over several sequences."""
    wl = make_workload(n_seq=n_seq, prompt_len=[4001 + 997 * s for s in range(n_seq)], n_steps=2,
                       tokens_per_step=tps, seed=40 + tps, shuffled=True, kv_type=kv_type)
    assert "hist" in qsa.index_topk_kernels(n_seq * tps, n_seq)
    run = Runner(wl)
    for i in range(2):
        check_step(run, i)


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 7, 2048, 2050, 2051, 2052, 2055])
def test_degenerate_and_budget_edges(n):
    """n <= top_k + r - 1: dense causal attention over all n cells; past it
    the budget binds at 512 blocks plus the tail."""
    wl = make_workload(n_seq=1, prompt_len=n - 1, n_steps=1, seed=100 + n)
    run = Runner(wl)
    res, _ = check_step(run, 0)
    cnt = int(res["count"][0])
    nb = n // 4
    assert cnt == min(nb, 512) * 4 + n % 4
    if n <= 2051:
        assert sorted(res["cells"][0, :cnt].tolist()) == list(range(n))


@pytest.mark.parametrize("nb_target", [3000, 40_000])
def test_all_equal_scores_pick_lowest_blocks(nb_target):
    """Every block scores the same: the lowest 512 indices win (candidate list
    in registers at 3000 blocks, the global re-scan path at 40000)."""
    n = nb_target * 4 + 1
    wl = make_workload(n_seq=1, prompt_len=n - 1, n_steps=1, seed=7)
    L = QSALayer.from_workload(wl, 0)
    st = wl.steps[0]
    inp = step_inputs(st)
    L.set_cells(*append_rows(wl, 0))
    L.pooled[:] = torch.linspace(-1, 1, 128, device="cuda")[None, :]
    L.index_topk(inp["tok_seq"], inp["tok_pos"], inp["q_idx"], inp["w_idx"])
    torch.cuda.synchronize()
    cells = to_np(L.cells[0])
    cnt = int(L.count[0])
    assert cnt == 512 * 4 + 1
    np.testing.assert_array_equal(cells[:2048], np.arange(2048))
    assert cells[2048] == n - 1
    assert_no_device_errors()


def test_heavy_ties_exact_on_gpu_scores():
    """Pooled rows drawn from 5 distinct rows: scores tie in large groups; the
    GPU choice equals a stable sort of its own scores."""
    wl = make_workload(n_seq=2, prompt_len=[30_000, 7_001], n_steps=1, seed=8, shuffled=True)
    L = QSALayer.from_workload(wl, 0)
    L.set_cells(*append_rows(wl, 0))
    g = torch.Generator(device="cpu").manual_seed(0)
    base = torch.randn(5, 128, generator=g)
    pick = torch.randint(0, 5, (L.n_slots,), generator=g)
    L.pooled.copy_(base[pick].cuda())
    st = wl.steps[0]
    inp = step_inputs(st)
    L.index_topk(inp["tok_seq"], inp["tok_pos"], inp["q_idx"], inp["w_idx"])
    sc = torch.empty((2, L.max_blocks), dtype=torch.float32, device="cuda")
    qsa.index_scores(L.cfg, inp["q_idx"], inp["w_idx"], inp["tok_seq"], inp["tok_pos"], L.pooled,
                     L.seq_blk_off, L.seq_blk_slots, L.max_blocks, sc)
    torch.cuda.synchronize()
    table = wl.blk_cells_state(1)
    for t in range(2):
        seq, pos = int(st.tok_seq[t]), int(st.tok_pos[t])
        nb = (pos + 1) // 4
        sel = O.select_blocks(to_np(sc[t, :nb]), 512)
        want = O.expand_cells(wl.cfg, sel, seq, pos, table, wl.seq_blk_off, wl.seq_blk_slots)
        np.testing.assert_array_equal(to_np(L.cells[t, :len(want)]), want)
        assert int(L.count[t]) == len(want)
    assert_no_device_errors()


def test_attention_special_cases():
    """count 0 -> zeros; one cell -> its V row; identical K rows -> mean of V."""
    wl = make_workload(n_seq=1, prompt_len=300, n_steps=1, seed=9)
    L = QSALayer.from_workload(wl, 0, max_tokens=3)
    q = torch.from_numpy(wl.steps[0].q).cuda().repeat(3, 1, 1)
    L.cells[:3] = -1
    L.cells[1, 0] = 17
    L.cells[2, :5] = torch.tensor([3, 9, 40, 41, 299], dtype=torch.int32)
    L.count[:3] = torch.tensor([0, 1, 5], dtype=torch.int32)
    k = L.k_cache.view(torch.float16).view(wl.n_cells, 2, 256)
    k[[3, 9, 40, 41, 299]] = k[3].clone()
    L.sparse_attn(q, 3)
    torch.cuda.synchronize()
    out = to_np(L.out[:3])
    v = wl.v_cache.astype(np.float64)
    assert np.all(out[0] == 0)
    for h in range(16):
        np.testing.assert_allclose(out[1, h], v[17, h // 8], rtol=1e-6, atol=1e-6)
        np.testing.assert_allclose(out[2, h], v[[3, 9, 40, 41, 299], h // 8].mean(0), rtol=2e-3, atol=2e-3)
    assert_no_device_errors()


def test_deterministic_repeat():
    wl = make_workload(n_seq=2, prompt_len=[12_345, 6_789], n_steps=1, seed=10, kv_type="q8_0")
    outs = []
    for _ in range(2):
        run = Runner(wl)
        res = run.run_step(0)
        outs.append(res)
    for k in ("out", "cells", "count", "pooled"):
        np.testing.assert_array_equal(outs[0][k], outs[1][k])


def test_out_of_range_indices_are_masked_and_flagged():
    """Bad cell indices in the inputs never fault: they are skipped, masked and
    reported by qsa_debug_check."""
    wl = make_workload(n_seq=1, prompt_len=600, n_steps=1, seed=11)
    L = QSALayer.from_workload(wl, 0)
    qsa.debug_check()
    q = torch.from_numpy(wl.steps[0].q).cuda()
    L.cells[0] = -1
    L.cells[0, :4] = torch.tensor([5, wl.n_cells + 7, -3, 6], dtype=torch.int32)
    L.count[0] = 4
    L.sparse_attn(q, 1)
    st, flags = qsa.debug_check()
    assert st == -6 and (flags & 2)
    out = to_np(L.out[0])
    ref = O.attend(wl.cfg, wl.steps[0].q[0], wl.k_cache, wl.v_cache, wl.n_cells, np.array([5, 6]))
    assert max_rel(out, ref) <= ATTN_TOL["f16"]
    # a dirty slot beyond the table and a bad member cell
    tbl = L.blk_cells.clone()
    L.blk_cells[3, 1] = wl.n_cells + 100
    L.pool_update(np.array([3, L.n_slots + 5, -1, -1], dtype=np.int32))
    st, flags = qsa.debug_check()
    assert st == -6 and (flags & 1) and (flags & 2)
    L.blk_cells.copy_(tbl)
    assert qsa.debug_check()[0] == 0


@pytest.mark.parametrize("top_k,n,kv_type", [(16, 403, "f16"), (256, 9_001, "f16"), (512, 600, "f16"),
                                              (4096, 30_003, "f16"), (256, 9_001, "q8_0"),
                                              (4096, 30_003, "q8_0")])
def test_other_budgets_cover_every_tile_layout(top_k, n, kv_type):
    """Budgets other than 2048 exercise the other attention layouts: one tile
    (top_k 16), a 2-CTA cluster plus overflow cells (256), exactly NC tiles
    (512 with a full budget), and several tiles per CTA (4096: the pipelined
    loops, cp.async for fp16 and register prefetch for q8_0)."""
    wl = make_workload(n_seq=1, prompt_len=n - 1, n_steps=3, seed=200 + top_k, cfg={"top_k": top_k},
                       kv_type=kv_type)
    run = Runner(wl)
    for i in range(3):
        res, _ = check_step(run, i)
        nb = (n + i) // 4
        assert int(res["count"][0]) == min(nb, top_k // 4) * 4 + (n + i) % 4


def test_q8_bad_indices_in_later_tiles_are_masked_and_flagged():
    """q8_0 with two 128-cell tiles per CTA (the register-prefetch loop) and
    overflow cells: bad ids in a CTA's second tile and among the overflow
    cells are skipped and reported, the rest attended exactly."""
    wl = make_workload(n_seq=1, prompt_len=30_002, n_steps=1, seed=13, kv_type="q8_0", cfg={"top_k": 4096})
    L = QSALayer.from_workload(wl, 0)
    qsa.debug_check()
    q = torch.from_numpy(wl.steps[0].q).cuda()
    rng = np.random.default_rng(14)
    cnt = 4096 + 3
    assert L.cells.shape[1] >= cnt
    cells = rng.choice(30_002, cnt, replace=False).astype(np.int32)
    bad = {16 * 128 + 5: wl.n_cells + 9, 31 * 128 + 127: -2, 4097: wl.n_cells}
    for i, c in bad.items():
        cells[i] = c
    L.cells[0] = -1
    L.cells[0, :cnt] = torch.from_numpy(cells)
    L.count[0] = cnt
    L.sparse_attn(q, 1)
    st, flags = qsa.debug_check()
    assert st == -6 and (flags & 2)
    keep = np.array([c for i, c in enumerate(cells) if i not in bad])
    ref = O.attend(wl.cfg, wl.steps[0].q[0], wl.k_cache, wl.v_cache, wl.n_cells, keep)
    assert max_rel(to_np(L.out[0]), ref) <= ATTN_TOL["q8_0"]
    assert qsa.debug_check()[0] == 0


@pytest.mark.parametrize("T", [1, 40, 160])
def test_selection_paths_past_65536_blocks(T):
    """Past 65,536 blocks per token the selection cannot finish in CTA 0 of
    the cluster.  Pooled rows c_s * v make every score c_s times one factor
    per token; 400 slots get c in [2^12, 2^16), K slots c within 1e-4 of 2^8
    (one histogram bin), the rest c in [1, 16), so the 512-block cut falls in
    a bin of exactly K keys: K = 600 ranks them directly across the cluster,
    1,500 runs radix rounds over the kept candidates, 5,000 radix rounds that
    re-scan the scores.  One token takes an 8-CTA cluster; 40 tokens take
    2-CTA clusters whose ranges exceed the cached slot ids; 160 tokens take
    one CTA each, more CTAs than SMs (two CTAs per SM, the slot ids read
    from global memory).  Each choice equals a stable sort of the GPU's own
    scores."""
    wl = make_workload(n_seq=1, prompt_len=280_000, n_steps=1, tokens_per_step=T, seed=300 + T)
    L = QSALayer.from_workload(wl, 0)
    L.set_cells(*append_rows(wl, 0))
    st = wl.steps[0]
    inp = step_inputs(st)
    table = wl.blk_cells_state(1)
    g = torch.Generator(device="cpu").manual_seed(T)
    v = torch.from_numpy(st.q_idx[0, 0].astype(np.float32))   # token 0, head 0: a positive factor
    sc = torch.empty((T, L.max_blocks), dtype=torch.float32, device="cuda")
    for k_bin in (600, 1_500, 5_000):
        perm = torch.randperm(L.n_slots, generator=g)
        u = torch.rand(L.n_slots, generator=g, dtype=torch.float64)
        c = torch.exp2(u * 4.0)                                   # below the cut
        c[perm[:400]] = torch.exp2(12.0 + u[perm[:400]] * 4.0)    # above it
        mid = perm[400:400 + k_bin]
        c[mid] = 256.0 * (1.0 + 1e-4 * u[mid])                    # the cut's bin
        L.pooled.copy_((c.float()[:, None] * v[None, :]).cuda())
        L.index_topk(inp["tok_seq"], inp["tok_pos"], inp["q_idx"], inp["w_idx"])
        qsa.index_scores(L.cfg, inp["q_idx"], inp["w_idx"], inp["tok_seq"], inp["tok_pos"], L.pooled,
                         L.seq_blk_off, L.seq_blk_slots, L.max_blocks, sc)
        torch.cuda.synchronize()
        scores = to_np(sc)
        for t in range(T):
            seq, pos = int(st.tok_seq[t]), int(st.tok_pos[t])
            nb = (pos + 1) // 4
            assert nb > 65_536
            sel = O.select_blocks(scores[t, :nb], 512)
            want = O.expand_cells(wl.cfg, sel, seq, pos, table, wl.seq_blk_off, wl.seq_blk_slots)
            np.testing.assert_array_equal(to_np(L.cells[t, :len(want)]), want)
            assert int(L.count[t]) == len(want)
    assert_no_device_errors()


@pytest.mark.parametrize("kv_type", ["f16", "q8_0"])
@pytest.mark.parametrize("T", [1, 2, 5, 512])
def test_empty_cache_every_cell_invalid(kv_type, T):
    """n_cells = 0 with full cell lists (every id out of range): the ids are
    reported, no row is read and the outputs are zero — one tile per CTA (1
    token), the union of a pair (2), several tiles per CTA (5 tokens: the
    pipelined variants) and one CTA per (token, KV head) (512 tokens: the
    two-CTAs-per-SM fp16 variant, the pipelined q8_0 one)."""
    wl = make_workload(n_seq=1, prompt_len=600, n_steps=1, seed=12, kv_type=kv_type)
    L = QSALayer.from_workload(wl, 0, max_tokens=T)
    pitch = L.pitch
    cells = torch.arange(pitch, dtype=torch.int32, device="cuda").repeat(T, 1).contiguous()
    count = torch.full((T,), pitch, dtype=torch.int32, device="cuda")
    q = torch.randn((T, 16, 256), device="cuda").to(torch.float16)
    for union in ([False, True] if T == 2 else [False]):
        out = torch.full((T, 16, 256), float("nan"), dtype=torch.float32, device="cuda")
        qsa.debug_check()
        qsa.sparse_attn(L.cfg, q, L.k_cache, L.v_cache, 0, cells, count, out, None, union=union)
        st, flags = qsa.debug_check()
        assert st == -6 and (flags & 2)
        assert torch.count_nonzero(out).item() == 0
