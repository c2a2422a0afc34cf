"""The method's O(top_k) claim (llama.cpp issue #28734, fix summary, lever1:
attention over only the selected K/V set): the sparse attention's time does
not grow with the context.  qsa_sparse_attn over the selected cells of one
decode token at 50,000 and at 250,000 fp16 cells (the same ~2,051 cells
each) is timed on the device, each launch between two event nodes after an
L2 flush, and the medians must agree within 10 %."""
import numpy as np
import pytest
import torch

import bench
from qsa_workload import make_workload
from sparse_attention_long_qsa_gb300.layer import QSALayer, append_rows, step_inputs

from gpu_util import assert_no_device_errors

pytestmark = pytest.mark.gpu


def _attn_us(name, reps=32):
    wl = make_workload(name, seed=0, n_steps=2)
    L = QSALayer.from_workload(wl, 0)
    L.warm(torch.from_numpy(wl.prompt_dirty()).cuda())
    L.set_cells(*append_rows(wl, 0))
    inp = step_inputs(wl.steps[0])
    L.pool_update(inp["dirty"])
    L.index_topk(inp["tok_seq"], inp["tok_pos"], inp["q_idx"], inp["w_idx"])
    torch.cuda.synchronize()
    count = int(L.count[0])
    flush = torch.empty(1 << 28, dtype=torch.float32, device="cuda")   # 1 GiB, past the L2
    xev = bench._ExternalEvents()
    ev = [(xev.new(), xev.new()) for _ in range(reps)]
    for _ in range(3):
        L.sparse_attn(inp["q"], 1)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for a, b in ev:
            flush.fill_(1.0)
            xev.record(a)
            L.sparse_attn(inp["q"], 1)
            xev.record(b)
    g.replay()
    torch.cuda.synchronize()
    us = float(np.median([a.elapsed_time(b) * 1e3 for a, b in ev]))
    del g, L, flush
    torch.cuda.empty_cache()
    return us, count


def test_attention_time_flat_in_context():
    t50, n50 = _attn_us("50k")
    t250, n250 = _attn_us("250k_f16")
    assert n50 == n250 == 2049          # 512 blocks of 4 + the tail cell of position 50,000 / 250,000
    assert abs(t250 - t50) <= 0.10 * t50, f"attention {t50:.2f} us at 50k vs {t250:.2f} us at 250k"
    assert_no_device_errors()
