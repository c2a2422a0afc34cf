"""q8_0 dequantisation pinned bit for bit (the author's q8-compact follow-up
in llama.cpp issue #28734 runs the sparse path on a q8_0 cache): attention
over a single cell is that cell's V row (the softmax of one score is 1, and
P = 1 times the row is exact), so the output must equal the fp16 rounding of
d * q for every value of the row: what both attention kernels dequantise
after the gather.  The oracle's rows (float(d) * q, exact) are rounded to
fp16 once for the comparison."""
import numpy as np
import pytest

from oracle import qsa_oracle as O
from qsa_workload import make_workload
from sparse_attention_long_qsa_gb300.layer import QSALayer

from gpu_util import assert_no_device_errors, run_lists

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("union", [False, True])
def test_single_cell_attention_is_the_dequantised_row(union):
    wl = make_workload(n_seq=1, prompt_len=5_000, n_steps=1, seed=970, kv_type="q8_0")
    L = QSALayer.from_workload(wl, 0, max_tokens=8)
    rng = np.random.default_rng(971)
    cells = rng.choice(wl.n_cells, 7, replace=False).astype(np.int32)
    q = rng.standard_normal((7, 16, 256)).astype(np.float16)
    out = run_lists(wl, L, [[int(c)] for c in cells], q, union)
    G = wl.cfg["n_kv_heads"]
    for t, c in enumerate(cells):
        for g in range(G):
            v = O.kv_rows(wl.cfg, wl.v_cache, wl.n_cells, [int(c)], g)[0]
            want = v.astype(np.float16).astype(np.float32)
            for h in range(8):
                np.testing.assert_array_equal(out[t, 8 * g + h], want)
    assert_no_device_errors()
