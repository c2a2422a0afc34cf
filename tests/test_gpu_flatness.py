"""The method's O(top_k) claim (llama.cpp issue #28734, fix summary, lever1:
attention over only the selected K/V set): the sparse attention's time does
not grow with the context.  qsa_sparse_attn over the selected cells of one
decode token at 50,000 and at 250,000 fp16 cells (the same ~2,051 cells
each) is timed on the device, each launch between two event nodes after an
L2 flush; the two graphs are replayed alternately, and the medians (the
lowest of the rounds' medians, which drops rounds disturbed by clock ramps
or other work) must agree within 10 %."""
import numpy as np
import pytest
import torch

import bench
from qsa_workload import make_workload
from sparse_attention_long_qsa_gb300.layer import QSALayer, append_rows, step_inputs

from gpu_util import assert_no_device_errors

pytestmark = pytest.mark.gpu


class _Timed:
    """One token's selected cells at a given depth and a captured graph of
    `reps` flushed, event-bracketed attention launches over them."""

    def __init__(self, name, flush, xev, reps=32):
        wl = make_workload(name, seed=0, n_steps=2)
        L = QSALayer.from_workload(wl, 0)
        L.warm(torch.from_numpy(wl.prompt_dirty()).cuda())
        L.set_cells(*append_rows(wl, 0))
        inp = step_inputs(wl.steps[0])
        L.pool_update(inp["dirty"])
        L.index_topk(inp["tok_seq"], inp["tok_pos"], inp["q_idx"], inp["w_idx"])
        torch.cuda.synchronize()
        self.count = int(L.count[0])
        self.ev = [(xev.new(), xev.new()) for _ in range(reps)]
        for _ in range(3):
            L.sparse_attn(inp["q"], 1)
        torch.cuda.synchronize()
        self.g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.g):
            for a, b in self.ev:
                flush.fill_(1.0)
                xev.record(a)
                L.sparse_attn(inp["q"], 1)
                xev.record(b)
        self.L, self.inp = L, inp

    def median_us(self):
        self.g.replay()
        torch.cuda.synchronize()
        return float(np.median([a.elapsed_time(b) * 1e3 for a, b in self.ev]))


def test_attention_time_flat_in_context():
    flush = torch.empty(1 << 28, dtype=torch.float32, device="cuda")   # 1 GiB, past the L2
    xev = bench._ExternalEvents()
    d50, d250 = _Timed("50k", flush, xev), _Timed("250k_f16", flush, xev)
    # 512 blocks of 4 cells + the tail cell of position 50,000 / 250,000
    assert d50.count == d250.count == 2049
    r50, r250 = [], []
    for _ in range(5):
        r50.append(d50.median_us())
        r250.append(d250.median_us())
    t50, t250 = min(r50), min(r250)
    assert abs(t250 - t50) <= 0.10 * t50, f"attention {t50:.2f} us at 50k vs {t250:.2f} us at 250k ({r50}, {r250})"
    assert_no_device_errors()
