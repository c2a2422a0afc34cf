"""GPU parity of qsa_kv_append (the in-library write of the step's new
cells) against the oracle, bit for bit: caches (fp16 copies or q8_0 codes and
scales), indexer keys, block table and the device-built dirty list; then the
whole step fed by it against the step fed by the host-side table append."""
import numpy as np
import pytest
import torch

from oracle import qsa_oracle as O
from qsa_workload import make_workload
from sparse_attention_long_qsa_gb300 import qsa
from sparse_attention_long_qsa_gb300.layer import QSALayer, append_rows, step_inputs

from gpu_util import assert_no_device_errors, to_np

pytestmark = pytest.mark.gpu


def _poison_new_cells(wl, L):
    """Overwrite the rows of every cell the steps append with garbage on both
    sides, so the comparison shows what the append itself wrote."""
    new = np.unique(np.concatenate([st.cells for st in wl.steps]))
    kc, vc, ik = (np.array(x, copy=True) for x in (wl.k_cache, wl.v_cache, wl.idx_k))
    G, D = wl.cfg["n_kv_heads"], wl.cfg["head_dim"]
    rng = np.random.default_rng(99)
    if wl.cfg["kv_type"] == "f16":
        for arr in (kc, vc):
            arr.reshape(wl.n_cells, G, D)[new] = rng.standard_normal((len(new), G, D)).astype(np.float16)
    else:
        nq = wl.n_cells * G * D
        for arr in (kc, vc):
            raw = arr.view(np.uint8)
            raw[:nq].reshape(wl.n_cells, G * D)[new] = rng.integers(0, 256, (len(new), G * D), dtype=np.uint8)
            raw[nq:].reshape(wl.n_cells, G * D // 16)[new] = rng.integers(0, 256, (len(new), G * D // 16),
                                                                           dtype=np.uint8)
    ik[new] = 7.0
    for dst, src in ((L.k_cache, kc), (L.v_cache, vc), (L.idx_k, ik)):
        dst.copy_(torch.from_numpy(np.ascontiguousarray(src).view(np.uint8)).cuda().view(dst.dtype).view(dst.shape))
    return kc, vc, ik


@pytest.mark.parametrize("kw", [
    dict(n_seq=1, prompt_len=5001, n_steps=4, kv_type="f16"),
    dict(n_seq=3, prompt_len=[3001, 9002, 1203], n_steps=5, kv_type="q8_0", shuffled=True),
    dict(n_seq=1, prompt_len=7003, n_steps=3, tokens_per_step=5, kv_type="q8_0"),
    dict(n_seq=1, prompt_len=2001, n_steps=1, tokens_per_step=96, kv_type="f16", shuffled=True),
    # the per-call maximum: 1,024 new tokens (512 per sequence), ~260 blocks re-pooled in the launch
    dict(n_seq=2, prompt_len=[3001, 5002], n_steps=1, tokens_per_step=512, kv_type="q8_0", shuffled=True),
])
def test_append_matches_oracle_bit_for_bit(kw):
    wl = make_workload(seed=41, **kw)
    L = QSALayer.from_workload(wl, 0)
    L2 = QSALayer.from_workload(wl, 0)
    kc, vc, ik = _poison_new_cells(wl, L)
    _poison_new_cells(wl, L2)
    for X in (L, L2):
        X.warm(torch.from_numpy(wl.prompt_dirty()).cuda())
    tbl = wl.blk_cells_state(0)
    for i, st in enumerate(wl.steps):
        inp = step_inputs(st, new_cells=True)
        args = (inp["tok_seq"], inp["tok_pos"], inp["cells"], inp["k_new"], inp["v_new"], inp["idx_new"])
        # L re-pools the dirtied blocks inside the append; L2 runs the pool update after it
        d = L.kv_append(*args, pool=True)
        d2 = L2.kv_append(*args)
        L2.pool_update(d2)
        torch.cuda.synchronize()
        assert torch.equal(L.pooled, L2.pooled)
        kc, vc, ik, tbl, dirty = O.kv_append(wl.cfg, st.tok_seq, st.tok_pos, st.cells, st.k_new, st.v_new,
                                             st.idx_new, kc, vc, ik, wl.n_cells, tbl, wl.seq_blk_off,
                                             wl.seq_blk_slots, int(d.numel()))
        np.testing.assert_array_equal(to_np(L.k_cache).view(np.uint8).reshape(-1), kc.view(np.uint8).reshape(-1))
        np.testing.assert_array_equal(to_np(L.v_cache).view(np.uint8).reshape(-1), vc.view(np.uint8).reshape(-1))
        np.testing.assert_array_equal(to_np(L.idx_k), ik)
        np.testing.assert_array_equal(to_np(L.blk_cells), tbl)
        np.testing.assert_array_equal(to_np(d), dirty)
    # the generator wrote each new cell's encoded row up front: the appends reproduce it
    np.testing.assert_array_equal(kc.view(np.uint8), np.asarray(wl.k_cache).view(np.uint8))
    assert_no_device_errors()


@pytest.mark.parametrize("kv_type", ["f16", "q8_0"])
def test_full_step_equals_host_appended_step(kv_type):
    """append -> pool -> index -> attention on poisoned new cells gives the
    same pooled keys, cells, counts and outputs as the three calls on the
    workload's caches with the table appended on the host."""
    wl = make_workload(n_seq=2, prompt_len=[12_001, 4_003], n_steps=6, seed=42, kv_type=kv_type, shuffled=True)
    A = QSALayer.from_workload(wl, 0)
    B = QSALayer.from_workload(wl, 0)
    for L in (A, B):
        L.warm(torch.from_numpy(wl.prompt_dirty()).cuda())
    _poison_new_cells(wl, B)
    for i, st in enumerate(wl.steps):
        A.set_cells(*append_rows(wl, i))
        oa = A.step(**step_inputs(st)).clone()
        ob = B.full_step(**step_inputs(st, new_cells=True)).clone()
        torch.cuda.synchronize()
        T = len(st.tok_pos)
        assert torch.equal(A.pooled, B.pooled)
        assert torch.equal(A.count[:T], B.count[:T]) and torch.equal(A.cells[:T], B.cells[:T])
        assert torch.equal(oa, ob)
    assert_no_device_errors()


def test_append_bad_inputs_are_skipped_and_flagged():
    wl = make_workload(n_seq=1, prompt_len=301, n_steps=1, tokens_per_step=3, seed=43)
    L = QSALayer.from_workload(wl, 0)
    qsa.debug_check()
    inp = step_inputs(wl.steps[0], new_cells=True)
    before = L.blk_cells.clone()
    inp["cells"][1] = wl.n_cells + 3                    # a cell beyond the cache
    inp["tok_seq"][2] = 4                               # an unknown sequence
    d = L.kv_append(inp["tok_seq"], inp["tok_pos"], inp["cells"], inp["k_new"], inp["v_new"], inp["idx_new"])
    st, flags = qsa.debug_check()
    assert st == -6 and (flags & 2) and (flags & 16)
    # only token 0 was written: one table entry and one dirty block
    diff = (L.blk_cells != before).nonzero()
    assert diff.shape[0] == 1
    dd = to_np(d)
    assert (dd >= 0).sum() == 1 and np.all(dd[1:] == -1)
