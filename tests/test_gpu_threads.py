"""Several host threads calling the library at once, each on its own stream
and buffers, in a fresh process so that their calls are the first ones on
the device: the per-device kernel set-up (shared-memory limits, cluster
occupancy) runs once under a lock, and every thread's results equal those of
the same steps run one after another, bit for bit."""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent("""
    import sys, threading
    import numpy as np
    import torch
    sys.path.insert(0, {root!r})
    from qsa_workload import make_workload
    from sparse_attention_long_qsa_gb300.layer import QSALayer, append_rows, step_inputs

    cases = [dict(n_seq=1, prompt_len=9001, seed=60, kv_type="f16"),
             dict(n_seq=1, prompt_len=9001, seed=61, kv_type="q8_0"),
             dict(n_seq=2, prompt_len=[4001, 5003], tokens_per_step=12, seed=62, kv_type="f16"),
             dict(n_seq=2, prompt_len=[4001, 5003], tokens_per_step=12, seed=63, kv_type="q8_0")]
    wls = [make_workload(n_steps=1, **c) for c in cases]

    def prepare(wl):
        # torch-only uploads plus the pool warm-up (the pool kernel has no
        # per-device set-up); no index or attention call yet
        L = QSALayer.from_workload(wl, 0)
        L.warm(torch.from_numpy(wl.prompt_dirty()).cuda())
        slots, rows = append_rows(wl, 0)
        if len(slots):
            L.set_cells(slots, rows)
        return L, step_inputs(wl.steps[0])

    def result(L, wl):
        T = len(wl.steps[0].tok_pos)
        return [L.out[:T].cpu().numpy(), L.cells[:T].cpu().numpy(), L.count[:T].cpu().numpy()]

    prepared = [prepare(wl) for wl in wls]
    torch.cuda.synchronize()
    start = threading.Barrier(len(wls))
    got, errors = [None] * len(wls), []

    def work(i):
        try:
            L, inp = prepared[i]
            s = torch.cuda.Stream()
            start.wait()
            with torch.cuda.stream(s):
                for _ in range(3):   # the same step again: pooled rows are recomputed identically
                    L.step(**inp, stream=s)
            s.synchronize()
            got[i] = result(L, wls[i])
        except Exception as e:   # reported by the parent
            errors.append(repr(e))

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(wls))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i, wl in enumerate(wls):
        L, inp = prepare(wl)
        for _ in range(3):
            L.step(**inp)
        torch.cuda.synchronize()
        want = result(L, wl)
        for a, b in zip(got[i], want):
            np.testing.assert_array_equal(a, b)
    print("ok", flush=True)
""")


def test_concurrent_first_calls_from_host_threads():
    r = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT)], cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout[-2000:] + r.stderr[-4000:]
