"""A step's inputs and output in pinned host memory: the kernels read the
token ids, queries, weights and new rows in place over the host link and the
attention stores its output into host memory.  The results equal those of the
same step with every buffer in device memory, bit for bit."""
import numpy as np
import pytest
import torch

from qsa_workload import make_workload
from sparse_attention_long_qsa_gb300.layer import PackedInputs, QSALayer, step_inputs

from gpu_util import assert_no_device_errors

pytestmark = pytest.mark.gpu

KEYS = ("tok_seq", "tok_pos", "q", "q_idx", "w_idx", "cells", "k_new", "v_new", "idx_new")


@pytest.mark.parametrize("kv_type,n_seq", [("f16", 1), ("q8_0", 3)])
def test_full_step_with_host_inputs_and_output(kv_type, n_seq):
    wl = make_workload(n_seq=n_seq, prompt_len=[20_001 + 3_001 * s for s in range(n_seq)], n_steps=3,
                       seed=900 + n_seq, kv_type=kv_type, shuffled=n_seq > 1)
    dev = QSALayer.from_workload(wl, 0)
    hst = QSALayer.from_workload(wl, 0)
    for L in (dev, hst):
        L.warm(torch.from_numpy(wl.prompt_dirty()).cuda())
    inputs0 = step_inputs(wl.steps[0], new_cells=True)
    pk = PackedInputs({k: (tuple(inputs0[k].shape), inputs0[k].dtype) for k in KEYS})
    for i, st in enumerate(wl.steps):
        T = len(st.tok_pos)
        a = dev.full_step(**step_inputs(st, new_cells=True))
        host = pk.pack({k: getattr(st, k) for k in KEYS})
        out = torch.empty((T, wl.cfg["n_q_heads"], wl.cfg["head_dim"]), dtype=torch.float32).pin_memory()
        b = hst.full_step(**pk.host_views(host), out=out)
        torch.cuda.synchronize()
        assert b is out
        assert torch.equal(out, a.cpu())
        assert torch.equal(hst.cells[:T], dev.cells[:T]) and torch.equal(hst.count[:T], dev.count[:T])
        assert torch.equal(hst.k_cache, dev.k_cache) and torch.equal(hst.blk_cells, dev.blk_cells)
        assert torch.equal(hst.pooled, dev.pooled)
    assert_no_device_errors()


def test_separate_calls_with_host_query_and_output():
    wl = make_workload(n_seq=1, prompt_len=30_001, n_steps=1, seed=910)
    L = QSALayer.from_workload(wl, 0)
    L.warm(torch.from_numpy(wl.prompt_dirty()).cuda())
    st = wl.steps[0]
    inp = step_inputs(st)
    from sparse_attention_long_qsa_gb300.layer import append_rows
    L.set_cells(*append_rows(wl, 0))
    L.pool_update(inp["dirty"])
    L.index_topk(inp["tok_seq"], inp["tok_pos"], inp["q_idx"], inp["w_idx"])
    L.sparse_attn(inp["q"], 1)
    torch.cuda.synchronize()
    ref = L.out[:1].cpu()
    from sparse_attention_long_qsa_gb300 import qsa
    qh = torch.from_numpy(np.ascontiguousarray(st.q)).pin_memory()
    out = torch.full((1, wl.cfg["n_q_heads"], wl.cfg["head_dim"]), float("nan")).pin_memory()
    qsa.sparse_attn(L.cfg, qh, L.k_cache, L.v_cache, L.n_cells, L.cells[:1], L.count[:1], out, L.ws_attn)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    # a pageable host tensor is refused
    with pytest.raises(ValueError):
        qsa.sparse_attn(L.cfg, torch.from_numpy(np.ascontiguousarray(st.q)), L.k_cache, L.v_cache, L.n_cells,
                        L.cells[:1], L.count[:1], out, L.ws_attn)
    assert_no_device_errors()
