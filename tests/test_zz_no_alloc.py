"""qsa_index_topk_noalloc against qsa_index_topk, through the C ABI.

The no-allocation entry point serves callers that cannot allocate device
memory for a workspace (plugins inside an engine that owns every device
allocation, latency-critical paths where cudaMalloc is not allowed).  It must
give exactly the cells and counts of the workspace entry point, on
consecutive calls that share its static scratch array.  This file is
collected last so that a run stopping at the first failure has already run
every other test; it also passes alone in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

from qsa_workload import make_workload
from sparse_attention_long_qsa_gb300 import qsa
from sparse_attention_long_qsa_gb300.layer import QSALayer, append_rows, step_inputs

pytestmark = pytest.mark.gpu


def _noalloc(L, inp, cells, count):
    T = int(inp["tok_pos"].numel())
    st = qsa.lib().qsa_index_topk_noalloc(
        ctypes.byref(L.cfg), T, inp["q_idx"].data_ptr(), inp["w_idx"].data_ptr(),
        inp["tok_seq"].data_ptr(), inp["tok_pos"].data_ptr(), L.pooled.data_ptr(),
        L.blk_cells.data_ptr(), L.n_slots, L.seq_blk_off.data_ptr(), L.seq_blk_slots.data_ptr(),
        int(L.seq_blk_off.numel()) - 1, L.max_blocks, L.n_cells, cells.data_ptr(), count.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    return st


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    from sparse_attention_long_qsa_gb300 import build
    build.build()
    wl = make_workload(n_seq=3, prompt_len=[30_001, 9_002, 1_500], n_steps=2, seed=21, shuffled=True)
    L = QSALayer.from_workload(wl, 0)
    L.warm(torch.from_numpy(wl.prompt_dirty()).cuda())
    T = len(wl.steps[0].tok_pos)
    for i in range(2):
        L.set_cells(*append_rows(wl, i))
        inp = step_inputs(wl.steps[i])
        L.pool_update(inp["dirty"])
        L.index_topk(inp["tok_seq"], inp["tok_pos"], inp["q_idx"], inp["w_idx"])
        cells = torch.full((T, L.pitch), 7, dtype=torch.int32, device="cuda")
        count = torch.full((T,), -5, dtype=torch.int32, device="cuda")
        assert _noalloc(L, inp, cells, count) == 0
        torch.cuda.synchronize()
        assert torch.equal(count, L.count[:T]), (count, L.count[:T])
        assert torch.equal(cells, L.cells[:T])
    st, flags = qsa.debug_check()
    assert st == 0, hex(flags)


def test_noalloc_at_its_limits():
    """8 tokens (one per sequence) with max_blocks = 262,144: the largest call
    the scratch array takes, so the token scores use its last rows.  Two calls
    in a row match qsa_index_topk run with a workspace of the same layout."""
    wl = make_workload(n_seq=8, prompt_len=[2_001 + 997 * s for s in range(8)], n_steps=2, seed=23,
                       shuffled=True)
    L = QSALayer.from_workload(wl, 0, max_tokens=8)
    L.max_blocks = 262_144
    L.ws_index = torch.zeros(qsa.index_topk_workspace_size(L.cfg, 8, L.max_blocks), dtype=torch.uint8,
                             device="cuda")
    L.warm(torch.from_numpy(wl.prompt_dirty()).cuda())
    T = len(wl.steps[0].tok_pos)
    assert T == 8
    for i in range(2):
        L.set_cells(*append_rows(wl, i))
        inp = step_inputs(wl.steps[i])
        L.pool_update(inp["dirty"])
        L.index_topk(inp["tok_seq"], inp["tok_pos"], inp["q_idx"], inp["w_idx"])
        cells = torch.full((T, L.pitch), 7, dtype=torch.int32, device="cuda")
        count = torch.full((T,), -5, dtype=torch.int32, device="cuda")
        assert _noalloc(L, inp, cells, count) == 0
        torch.cuda.synchronize()
        assert torch.equal(count, L.count[:T]), (count, L.count[:T])
        assert torch.equal(cells, L.cells[:T])
    st, flags = qsa.debug_check()
    assert st == 0, hex(flags)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    wl = make_workload(n_seq=1, prompt_len=100, n_steps=1, seed=22)
    L = QSALayer.from_workload(wl, 0, max_tokens=9)
    inp = step_inputs(wl.steps[0])
    q = {k: v.repeat(9, *([1] * (v.dim() - 1))).contiguous() for k, v in inp.items()}
    cells = torch.zeros((9, L.pitch), dtype=torch.int32, device="cuda")
    count = torch.zeros(9, dtype=torch.int32, device="cuda")
    assert _noalloc(L, q, cells, count) == -4          # 9 tokens > 8
    L.max_blocks = 262145
    assert _noalloc(L, inp, cells[:1], count[:1]) == -4
    torch.cuda.synchronize()
    assert int(count.abs().sum()) == 0                 # nothing launched
