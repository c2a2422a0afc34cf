"""The fp16 attention of calls with many tokens (attn_pf.cu: tiles of 64
cells, a cluster of two CTAs per (token, KV head), two CTAs per SM), taken
when the cluster-size model gives one CTA per (token, KV head).  Every
token's output is checked against the oracle over its own list: counts 0,
1, 63-65, 127-129 and the full budget (either CTA of a pair without a tile,
a partial last tile), out-of-range ids, budgets 256-2048."""
import re

import numpy as np
import pytest
import torch

from oracle import qsa_oracle as O
from qsa_workload import make_workload
from sparse_attention_long_qsa_gb300 import qsa
from sparse_attention_long_qsa_gb300.layer import QSALayer

from gpu_util import ATTN_TOL, assert_no_device_errors, max_rel, run_lists

pytestmark = pytest.mark.gpu


def _kernel_names(fn):
    """Names of the CUDA kernels fn() launches (empty when the profiler
    records no device activity on this machine)."""
    from torch.profiler import ProfilerActivity, profile
    try:
        with profile(activities=[ProfilerActivity.CUDA]) as prof:
            fn()
            torch.cuda.synchronize()
        return {e.name for e in prof.events() if e.device_type == torch.autograd.DeviceType.CUDA}
    except RuntimeError:
        return set()


@pytest.mark.parametrize("top_k", [2048, 256])
def test_many_tokens_every_count(top_k):
    T = 512
    wl = make_workload(n_seq=1, prompt_len=30_000, n_steps=1, seed=970 + top_k // 256, cfg={"top_k": top_k})
    L = QSALayer.from_workload(wl, 0, max_tokens=T)
    pitch = L.pitch
    rng = np.random.default_rng(971)
    counts = [0, 1, 63, 64, 65, 127, 128, 129, pitch - 1, pitch]
    counts += [int(c) for c in rng.integers(0, pitch + 1, T - len(counts))]
    lists = [rng.choice(wl.n_cells, size=c, replace=False).astype(np.int32) for c in counts]
    q = rng.standard_normal((T, 16, 256)).astype(np.float16)
    qsa.debug_check()
    out = run_lists(wl, L, lists, q, union=False)
    _kernel_names(lambda: run_lists(wl, L, lists[:1], q[:1], union=False))   # the profiler's first use
    names = _kernel_names(lambda: run_lists(wl, L, lists, q, union=False))
    print("attention kernels:", sorted({m.group(0) for n in names for m in [re.search(r"k_attn\w*", n)] if m}))
    if names:
        assert any("k_attn_pf" in n for n in names), sorted(names)
    assert_no_device_errors()
    for t in range(T):
        if len(lists[t]) == 0:
            assert np.all(out[t] == 0), t
            continue
        ref = O.attend(wl.cfg, q[t], wl.k_cache, wl.v_cache, wl.n_cells, lists[t])
        assert max_rel(out[t], ref) <= ATTN_TOL["f16"], f"token {t}, {len(lists[t])} cells"


def test_out_of_range_ids_are_flagged_and_masked():
    T = 512
    wl = make_workload(n_seq=1, prompt_len=20_000, n_steps=1, seed=975)
    L = QSALayer.from_workload(wl, 0, max_tokens=T)
    rng = np.random.default_rng(976)
    lists, clean = [], []
    for t in range(T):
        c = rng.choice(wl.n_cells, size=int(rng.integers(100, L.pitch + 1)), replace=False).astype(np.int32)
        bad = c.copy()
        if t % 3 == 0:
            k = int(rng.integers(0, len(c)))
            bad[k] = wl.n_cells + 5 if t % 2 else -4
            c = np.delete(c, k)
        lists.append(bad)
        clean.append(c)
    q = rng.standard_normal((T, 16, 256)).astype(np.float16)
    qsa.debug_check()
    out = run_lists(wl, L, lists, q, union=False)
    st, flags = qsa.debug_check()
    assert st == -6 and (flags & 2)
    for t in range(0, T, 7):
        ref = O.attend(wl.cfg, q[t], wl.k_cache, wl.v_cache, wl.n_cells, clean[t])
        assert max_rel(out[t], ref) <= ATTN_TOL["f16"], t
