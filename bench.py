#!/usr/bin/env python
"""Benchmark of the QSA sparse-attention step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config 50k] [--impl native|reference]

A step is one decode step of one QSA layer over all sequences of the
workload, through the C ABI on one stream: qsa_kv_append (the step's new
cells, the device dirty list and the re-pooling of the dirtied blocks) ->
qsa_index_attn (score, select with expansion, attention with the split
merge).  --path calls times qsa_pool_update -> qsa_index_topk ->
qsa_sparse_attn with the table appended outside the timed region instead.
Inputs are resident in HBM when the timed region starts; L2 is flushed
before every step, outside the per-step events: a 1 GiB write, then a
256 MiB read of its head, so the step starts with no line of its own data in
L2 and no dirty line whose write-back it would pay for.
Prints one JSON line (rank 0).

Workloads (seeded, synthetic; shapes of the qwen4exp QSA layer):
  50k        1 seq, 50,000-cell fp16 prompt, 128 decode steps (default)
  250k_q8    1 seq, 250,000-cell q8_0 prompt, 128 decode steps
  5x250k_q8  5 seqs x 250,000 cells in one q8_0 cache, 5 tokens per step
  tiny       1 seq, 4,096 cells
  prefill    512-token ubatch on a 250,000-cell fp16 prompt
  verify5_250k_q8  1 seq, 250,000-cell q8_0 prompt, 5 consecutive query tokens per step

--impl reference times the CPU oracle (NumPy float64) on the host cores on
the same workload, as the slow baseline arm.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "QSA-layer decode tokens/s at 50k/250k ctx (1 and 5 seqs); HBM GB/s vs peak"
# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of
# a workload's roofline kernel, taken by ncu from the kernel built from the
# sources whose hash is stored beside it.  The line reports the number only
# while the kernel's sources still hash to that value (null otherwise, and for
# a workload or kernel without an entry).
NCU_CMD = ("ncu --set full --clock-control none -k regex:<kernel> -s 6 -c 1 python bench.py --config {cfg} "
           "--path calls --steps 8 --warmup 3 --secondary none --target none --no-cpu --no-compare --flush-mb 256")
NCU_TRAFFIC = {
    ("250k_q8", "score"): {"bytes": 33_290_496, "source": "9307ab22e5a2fb45", "capture": NCU_CMD.format(cfg="250k_q8")},
    ("250k_q8", "select"): {"bytes": 647_680, "source": "148ee2a21a8bb81c", "capture": NCU_CMD.format(cfg="250k_q8")},
    ("250k_q8", "attn"): {"bytes": 2_318_336, "source": "77a789af3a3d43c7", "capture": NCU_CMD.format(cfg="250k_q8")},
    ("50k", "score"): {"bytes": 6_690_048, "source": "9307ab22e5a2fb45", "capture": NCU_CMD.format(cfg="50k")},
    ("50k", "select"): {"bytes": 239_360, "source": "148ee2a21a8bb81c", "capture": NCU_CMD.format(cfg="50k")},
    ("50k", "attn"): {"bytes": 4_279_296, "source": "77a789af3a3d43c7", "capture": NCU_CMD.format(cfg="50k")},
}
KERNEL_SOURCES = {
    "append": ("append.cu", "pool_row.cuh", "qsa_internal.cuh"),
    "pool": ("pool.cu", "pool_row.cuh", "qsa_internal.cuh"),
    "score": ("index.cu", "index_util.cuh", "tc_util.cuh", "qsa_internal.cuh"),
    "hist": ("index.cu", "index_util.cuh", "qsa_internal.cuh"),
    "select": ("index.cu", "index_util.cuh", "qsa_internal.cuh"),
    "attn": ("attn.cu", "attn_pf.cu", "attn_pf.cuh", "attn_util.cuh", "index_util.cuh", "tc_util.cuh",
             "qsa_internal.cuh"),
    "select_attn": ("attn.cu", "attn_util.cuh", "index_util.cuh", "tc_util.cuh", "qsa_internal.cuh"),
}
FLUSH_BYTES = [1 << 30]   # L2 flush buffer (--flush-mb)
FLUSH_READ_BYTES = 256 << 20   # read after the flush write (> the 129 MB L2)

DESCR = {
    "50k": "decode, 1 seq, 50,000-cell fp16 K/V prompt + 1 cell/step (tails cycle 1,2,3,0), "
           "16q/2kv heads x 256, indexer 4x128, r=4, top_k=2048",
    "250k_q8": "decode, 1 seq, 250,000-cell q8_0 K/V prompt + 1 cell/step, same heads, top_k=2048",
    "250k_f16": "decode, 1 seq, 250,000-cell fp16 K/V prompt + 1 cell/step, same heads, top_k=2048",
    "5x250k_q8": "decode, 5 seqs x 250,000 cells in one 1.25M-cell q8_0 cache, 5 tokens/step, top_k=2048 per seq",
    "tiny": "decode, 1 seq, 4,096 cells fp16, top_k=2048",
    "prefill": "prefill ubatch, 512 tokens appended to a 250,000-cell fp16 prompt, 128 dirty blocks",
    "verify5_250k_q8": "verify batch, 1 seq, 250,000-cell q8_0 K/V prompt + 5 consecutive query tokens/step, "
                       "same heads, top_k=2048",
    "prefill_corr": "prefill ubatch as `prefill`, the tokens' indexer queries correlated (rho 0.98 with a shared "
                    "component, shared indexer weights), so consecutive tokens choose overlapping blocks",
    "verify5_250k_q8_corr": "verify batch as `verify5_250k_q8`, the tokens' indexer queries correlated (rho 0.98 "
                            "with a shared component, shared indexer weights)",
}


def kernel_source_hash(kernel: str) -> str:
    """sha256 (first 16 hex digits) of the CUDA sources a kernel is built from."""
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "sparse_attention_long_qsa_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str, kernel: str):
    """(bytes, source note) of the stored ncu traffic of this kernel build, or
    (None, reason)."""
    e = NCU_TRAFFIC.get((workload, kernel))
    if e is None:
        return None, "no ncu capture of this kernel on this workload"
    if e["source"] != kernel_source_hash(kernel):
        return None, "the kernel's sources changed since its ncu capture"
    return e["bytes"], ("ncu dram__bytes_read.sum + dram__bytes_write.sum of one launch "
                        f"({e['capture']}; sources {e['source']})")


L2_NOTE = ("GPU arm, headline and e2e: the timed layer-steps run back to back over copies of the layer's "
           "state (each one more layer of the model: its own caches, keys, block table and pooled keys), "
           "enough that the other copies' steps move more than 3x the 129 MB L2 between two steps of one "
           "copy (inputs larger than L2, no flush); per-kernel times: L2 flushed before every step (a 1 GiB "
           "write, then a 256 MiB read of its head), outside the step's events")
L2_BYTES = 129 * 10 ** 6
CHAIN_MEM_BYTES = 48 << 30   # device memory the layer copies may take


def bench_config(name: str, tokens_per_step: int) -> dict:
    """The `config` object of both arms' lines (identical for the same workload)."""
    return {"workload": DESCR[name], "name": name, "tokens_per_step": int(tokens_per_step), "l2": L2_NOTE}


def _env_rank():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), \
        int(os.environ.get("LOCAL_RANK", 0))


def _peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        return None


def algorithmic_bytes(wl, step_idx: int):
    """Algorithmic bytes of each kernel for one step (what the method must
    move at least once), by stage:
      append: per new cell its fp16 K/V rows read and written in the cache's
              encoding, its indexer key read and written, table entry, dirty list
      pool:   per dirty slot r fp16 idx-key rows (256 B) + table row + 512 B write
      score:  per visible block of a sequence a 512 B pooled row + 4 B slot id
              (once per step however many of its tokens score it), per token
              and visible block a 4 B score write, plus the token's 2 KiB
              query and 16 B weights
      hist:   (token-tiled scoring only) the scores read back, 4 B each
      select: 4 B score read per visible block, per chosen block 4 B slot +
              r*4 B members, + the cell list written
      attn:   per selected cell and KV head one K and one V row (512 B each fp16,
              272 B each q8_0), + 4 B index, + the token's 8 KiB query and its
              16 KiB fp32 output"""
    cfg = wl.cfg
    r = cfg["compress_ratio"]
    B = cfg["top_k"] // r
    G = cfg["n_kv_heads"]
    st = wl.steps[step_idx]
    row_b = 2 * 256 if cfg["kv_type"] == "f16" else 256 + 16
    out = dict(append=0.0, pool=0.0, score=0.0, hist=0.0, select=0.0, attn=0.0)
    nd = int((st.dirty >= 0).sum())
    T = len(st.tok_pos)
    # per new cell: its K and V rows read (fp16) and written (cache encoding),
    # its indexer key read and written, token ids, the table entry, the dirty list
    out["append"] = T * (2 * G * 512 + 2 * G * row_b + 2 * 256 + 3 * 4 + 4) + 4 * max(4, T)
    out["pool"] = nd * (r * 256 + 4 * r + 4 + 512)
    rows = {}
    for s_, p in zip(st.tok_seq.tolist(), st.tok_pos.tolist()):
        rows[s_] = max(rows.get(s_, 0), (p + 1) // r)
    out["score"] = float(sum(rows.values()) * (512 + 4))
    for p in st.tok_pos.tolist():
        nb = (p + 1) // r
        tail = p + 1 - nb * r
        nsel = min(nb, B) * r + tail
        out["score"] += nb * 4 + 2048 + 16
        out["hist"] += nb * 4
        out["select"] += nb * 4 + min(nb, B) * (4 + 4 * r) + (cfg["top_k"] + r - 1) * 4
        out["attn"] += (nsel * G * 2 * row_b + nsel * 4 + cfg["n_q_heads"] * cfg["head_dim"] * 2
                        + cfg["n_q_heads"] * cfg["head_dim"] * 4)
    return out


class Clocks:
    """nvidia-smi clock/throttle sampling around a timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.p = None
        self.path = os.path.join("/tmp", f"qsa_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.p = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None
        time.sleep(0.3)

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except Exception:
            self.p.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit())
                if any(r[3].replace(".", "").isdigit() for r in rows) else None}


# ---------------------------------------------------------------------------
class OracleRunner:
    """The CPU oracle as it stands, stepping through a workload: each step
    appends the step's cells (caches, keys, table), then runs the full oracle
    step (pool the dirty blocks, score every visible block, select, expand,
    attend).  For steps
    with many tokens (prefill) a bounded sample of the tokens is attended."""

    def __init__(self, wl, max_tokens_per_step: int = 8):
        from oracle import qsa_oracle as O
        self.O, self.wl = O, wl
        self.cap = max_tokens_per_step
        cfg = wl.cfg
        self.table0 = wl.blk_cells_state(0)
        self.pooled = O.pool_update(cfg, wl.idx_k, self.table0, wl.slot_block_idx, wl.prompt_dirty(),
                                    wl.norm_w, np.zeros((wl.n_slots, cfg["idx_dim"]), np.float32))
        self.table = self.table0.copy()
        self.next = 0

    def step(self, i: int) -> int:
        """Run workload step i (steps must come in order, wrapping to 0).
        Returns the tokens attended; only the oracle call is meant to be timed
        by the caller via the returned duration."""
        wl, O = self.wl, self.O
        i %= len(wl.steps)
        if i == 0:
            self.table = self.table0.copy()
        st = wl.steps[i]
        a = time.perf_counter()
        # the step's own cells: K/V rows (encoded as the cache stores them),
        # indexer keys and table entries, written in place
        self.O.kv_append(wl.cfg, st.tok_seq, st.tok_pos, st.cells, st.k_new, st.v_new, st.idx_new,
                         wl.k_cache, wl.v_cache, wl.idx_k, wl.n_cells, self.table, wl.seq_blk_off,
                         wl.seq_blk_slots, len(st.dirty), inplace=True)
        t_append = time.perf_counter() - a
        if len(st.tok_pos) > self.cap:
            import dataclasses
            sel = np.linspace(0, len(st.tok_pos) - 1, self.cap).astype(int)
            st = dataclasses.replace(st, tok_seq=st.tok_seq[sel], tok_pos=st.tok_pos[sel], q=st.q[sel],
                                     q_idx=st.q_idx[sel], w_idx=st.w_idx[sel])
        a = time.perf_counter()
        self.pooled, _, _ = O.run_step(wl.cfg, wl.idx_k, wl.k_cache, wl.v_cache, wl.n_cells, self.table,
                                       wl.slot_block_idx, wl.seq_blk_off, wl.seq_blk_slots, wl.norm_w,
                                       self.pooled, st)
        self.last_s = time.perf_counter() - a + t_append
        return len(st.tok_pos)


def cpu_oracle_rate(wl, max_seconds: float, min_steps: int = 2):
    """Oracle tokens/s over consecutive steps until max_seconds of oracle
    time.  Returns (tokens/s, steps run, seconds, threads)."""
    run = OracleRunner(wl)
    tokens = steps = 0
    elapsed = 0.0
    while steps < min_steps or elapsed < max_seconds:
        tokens += run.step(steps)
        elapsed += run.last_s
        steps += 1
    return tokens / elapsed, steps, elapsed, _blas_threads()


def _blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [d.get("num_threads", 1) for d in threadpool_info() if d.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return len(os.sched_getaffinity(0))


# ---------------------------------------------------------------------------
def run_reference(args, rank, world):
    """--impl reference: the CPU oracle on the host cores (rank 0 only):
    W untimed then exactly K timed workload steps."""
    if rank != 0:
        return
    from qsa_workload import make_workload
    wl = make_workload(args.config, seed=0)
    run = OracleRunner(wl)
    for n in range(args.warmup):
        run.step(n)
    tokens, secs = 0, 0.0
    for n in range(args.steps):
        tokens += run.step(args.warmup + n)
        secs += run.last_s
    rate = tokens / secs
    threads = _blas_threads()
    per = min(len(wl.steps[0].tok_pos), run.cap)
    sample = (f"{args.steps} consecutive steps of the {args.config} workload, full oracle step each "
              f"({per} token(s) attended per step)")
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": bench_config(args.config, len(wl.steps[0].tok_pos)),
        "cpu_baseline": {"value": rate, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": rate, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
class _ExternalEvents:
    """CUDA events recorded as graph event nodes (cudaEventRecordExternal), so
    a captured graph timestamps every step on the device."""

    def __init__(self):
        import ctypes
        self.rt = ctypes.CDLL("libcudart.so.13")
        self.rt.cudaEventRecordWithFlags.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint]
        self.rt.cudaEventRecordWithFlags.restype = ctypes.c_int

    def new(self):
        import torch
        e = torch.cuda.Event(enable_timing=True)
        e.record()                      # creates the CUDA event
        return e

    def record(self, ev):
        import torch
        st = self.rt.cudaEventRecordWithFlags(ev.cuda_event, torch.cuda.current_stream().cuda_stream, 1)
        if st != 0:
            raise RuntimeError(f"cudaEventRecordWithFlags failed: {st}")


def measure_config(name, K, W, dev, *, path="full", e2e=True, clocks=None, in_cluster=False, union=False):
    """Time K decode steps of workload `name` on the device.  The K timed
    steps are captured as ONE CUDA graph: per step an L2 flush (write, then
    read; outside the step's events), a start event node, the step, an end event node.  Path
    "full" (the layer's whole step): qsa_kv_append (the step's new cells, the
    device dirty list and, in the same launch, the re-pooling of the dirtied
    blocks), qsa_index_topk, qsa_sparse_attn.  Path "calls": qsa_pool_update,
    qsa_index_topk, qsa_sparse_attn, the block table appended by a torch index
    write outside the step's events and the dirty list from the host.
    The graph is replayed once; the step time is end - start of each step.
    union (path "full"): token pairs attend over the union of their lists
    (QSA_INDEX_ATTN_UNION)."""
    import torch
    from qsa_workload import make_workload
    from sparse_attention_long_qsa_gb300 import qsa
    from sparse_attention_long_qsa_gb300.layer import PackedInputs, QSALayer, append_rows, step_inputs

    t_gen = time.perf_counter()
    wl = make_workload(name, seed=0)
    t_gen = time.perf_counter() - t_gen
    n_steps = len(wl.steps)
    L = QSALayer.from_workload(wl, 0, device=dev)
    tbl0 = L.blk_cells.clone()
    L.warm(torch.from_numpy(wl.prompt_dirty()).to(dev))
    full = path == "full"
    inputs = [step_inputs(st, device=dev, new_cells=full) for st in wl.steps]
    appends = []
    for i in range(n_steps):
        s_, rows = append_rows(wl, i)
        appends.append((torch.from_numpy(s_).to(dev), torch.from_numpy(rows).to(dev)))
    flush = torch.empty(FLUSH_BYTES[0] // 4, dtype=torch.float32, device=dev)
    rsum = torch.zeros((), dtype=torch.float32, device=dev)
    toks = [len(st.tok_pos) for st in wl.steps]
    alg = [algorithmic_bytes(wl, i) for i in range(n_steps)]
    # path "full": the append kernel also re-pools the blocks it dirties, and
    # one qsa_index_attn call scores, selects and attends (the selection inside
    # the attention clusters where its limits hold)
    if full:
        kernels = ["append"] + qsa.index_attn_kernels(L.cfg, toks[0], wl.n_seq, L.max_blocks,
                                                      in_cluster=in_cluster, union=union)
    else:
        kernels = ["pool"] + qsa.index_topk_kernels(toks[0], wl.n_seq) + ["attn"]
    for a in alg:
        if full:
            a["append"] += a.pop("pool")
        else:
            a.pop("append")
        if "hist" not in kernels:
            a.pop("hist")
        if "select_attn" in kernels:
            a["select_attn"] = a.pop("select") + a.pop("attn")
    step_fn = (lambda **kw: L.full_step(**kw, in_cluster=in_cluster, union=union)) if full else L.step
    xev = _ExternalEvents()

    def do_append(i):
        # outside the step's events: the table back to the prompt state when
        # the workload wraps around, and (path "calls") the step's own entries
        if i == 0:
            L.blk_cells.copy_(tbl0)
        if not full:
            s_, rows = appends[i]
            L.blk_cells[s_] = rows

    def order(start, n):
        return [(start + k) % n_steps for k in range(n)]

    def set_state(start):
        # the table as it stands before step `start` (every earlier step's
        # entries present), set up outside any timed region
        L.blk_cells.copy_(tbl0)
        for i in range(start % n_steps):
            s_, rows = appends[i]
            L.blk_cells[s_] = rows

    # eager warm-up: W steps (also loads the module, sets kernel attributes)
    set_state(0)
    for i in order(0, max(W, 1)):
        do_append(i)
        step_fn(**inputs[i])
    torch.cuda.synchronize()

    io_keys = ("tok_seq", "tok_pos", "q", "q_idx", "w_idx") + (
        ("cells", "k_new", "v_new", "idx_new") if full else ("dirty",))
    host = None
    if e2e:
        # each step's inputs packed in one pinned host buffer.  Path "full":
        # the kernels read them in place over the host link and the attention
        # writes its output straight into a pinned host buffer (no copy
        # node); path "calls": one host-to-device copy of the packed inputs
        # and one device-to-host copy of the output per step.
        staging = PackedInputs({k: (tuple(inputs[0][k].shape), inputs[0][k].dtype) for k in io_keys}, device=dev)
        host = []
        for i, st in enumerate(wl.steps):
            h = {"in": staging.pack({k: getattr(st, k) for k in io_keys})}
            h["views"] = staging.host_views(h["in"])
            h["out"] = torch.empty((toks[i], wl.cfg["n_q_heads"], wl.cfg["head_dim"]),
                                   dtype=torch.float32).pin_memory()
            host.append(h)

    def run_graph(idx, hook=(), with_io=False):
        """Capture len(idx) steps as one graph, replay it once; returns the
        per-step device ms and the hooked kernels' per-launch ms."""
        ev = [(xev.new(), xev.new()) for _ in idx]
        hk = [{k: (xev.new(), xev.new()) for k in hook} for _ in idx]
        set_state(idx[0])
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for n, i in enumerate(idx):
                do_append(i)
                flush.fill_(float(n))
                # read back the buffer's head (> L2): the flush's dirty lines
                # are written back here, not by the step's first reads
                rsum.copy_(flush[:FLUSH_READ_BYTES // 4].sum())
                for k, (a, b) in hk[n].items():
                    qsa.profile_kernel(k, a, b)
                xev.record(ev[n][0])
                d = inputs[i]
                if with_io and full:
                    step_fn(**{**d, **host[i]["views"]}, out=host[i]["out"])
                else:
                    if with_io:
                        staging.upload(host[i]["in"])
                        d = {**d, **staging.views}
                    step_fn(**d)
                    if with_io:
                        host[i]["out"].copy_(L.out[:toks[i]], non_blocking=True)
                xev.record(ev[n][1])
        for k in hook:
            qsa.profile_kernel(k, None, None)
        set_state(idx[0])
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        ms = [a.elapsed_time(b) for a, b in ev]
        kms = {k: [h[k][0].elapsed_time(h[k][1]) for h in hk] for k in hook}
        del g
        return ms, kms

    # per-kernel breakdown (every kernel hooked; hooks cut the launch overlap)
    br = order(W, min(max(K, 8), 64))
    _, kms = run_graph(br, hook=kernels)
    kern_us = {k: 1e3 * float(np.mean(v)) for k, v in kms.items()}
    kbytes = {k: float(np.mean([alg[i][k] for i in br])) for k in kernels}
    # roofline kernel: the one moving the most algorithmic bytes per step (the
    # HBM-bound stage; the longest kernel is reported beside it)
    dominant = max(kbytes, key=kbytes.get)
    longest = max(kern_us, key=kern_us.get)

    # headline: K steps, no hooks
    idx = order(W, K)
    if clocks:
        clocks.start()
    wall0 = time.perf_counter()
    ms, _ = run_graph(idx)
    wall = time.perf_counter() - wall0
    # the roofline kernel, timed live over the same K steps
    _, dk = run_graph(idx, hook=[dominant])
    dom_ms = float(np.mean(dk[dominant]))
    dom_bytes = float(np.mean([alg[i][dominant] for i in idx]))
    dev_ms = float(np.sum(ms))
    tokens = sum(toks[i] for i in idx)
    res = dict(value=tokens / (dev_ms / 1e3), ms_per_step=dev_ms / K, tokens=tokens, wall_s=wall, path=path,
               launches_per_step=len(kernels), kernels=kernels,
               dominant=dominant, longest=longest, dom_ms=dom_ms, dom_bytes=dom_bytes, kern_us=kern_us,
               kern_gbs={k: kbytes[k] / (kern_us[k] * 1e-6) / 1e9 for k in kernels if kern_us[k] > 0},
               gen_s=t_gen, wl=wl, step_bytes=float(np.mean([sum(alg[i].values()) for i in idx])),
               step_us_p50=1e3 * float(np.median(ms)), step_us_p90=1e3 * float(np.percentile(ms, 90)))

    if e2e:
        # the same steps with the inputs in pinned host memory and the output
        # going back to it, inside each step's events
        ms2, _ = run_graph(idx, with_io=True)
        h2d = float(sum(n for (_, _, _, n) in staging.fields.values()))
        d2h = float(np.mean([host[i]["out"].numel() * 4 for i in idx]))
        res["e2e"] = {"value": tokens / (float(np.sum(ms2)) / 1e3), "unit": "tokens/s",
                      "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                      "how": ("the step's inputs in pinned host memory, read in place by the kernels over NVLink-C2C; "
                              "the output stored by the attention kernel into pinned host memory"
                              if full else "one copy of the packed inputs to the device and one copy of the "
                              "output back per step, inside the step's events")}
        # the host sees the last step's output as the device-input run wrote it
        last = idx[-1]
        if full and not torch.equal(host[last]["out"], L.out[:toks[last]].cpu()):
            raise RuntimeError("the in-place host-memory step differs from the device-memory step")
    res["clocks"] = clocks.stop() if clocks else None
    st, flags = qsa.debug_check()
    if st != 0:
        raise RuntimeError(f"device error word set during the bench: {flags:#x}")
    del L, flush
    torch.cuda.empty_cache()
    return res


def clone_layer(L):
    """Another layer of the same model: a copy of the layer's state (caches,
    indexer keys, block table, pooled keys, outputs, workspaces); the
    sequences' block lists and the norm weight are shared."""
    import copy
    C = copy.copy(L)
    for k in ("idx_k", "k_cache", "v_cache", "blk_cells", "pooled", "cells", "count", "out", "ws_index",
              "ws_attn"):
        setattr(C, k, getattr(L, k).clone())
    C._dirty = None
    return C


def chain_layers(step_bytes: float, state_bytes: float) -> int:
    """Layer copies for back-to-back timing: enough that the other copies'
    steps move more than 3x the L2 between two steps of one copy, at least
    2, at most 64 and at most what CHAIN_MEM_BYTES holds."""
    n = max(2, int(np.ceil(3 * L2_BYTES / max(step_bytes, 1.0))) + 1)
    return max(2, min(n, 64, int(CHAIN_MEM_BYTES // max(state_bytes, 1))))


def measure_chain(name, K, W, dev, *, e2e=True, clocks=None, union=False, in_cluster=False):
    """Headline timing of the whole layer step (qsa_kv_append re-pooling the
    blocks it dirties, then qsa_index_attn): K layer-steps back to back in
    one CUDA graph, events only at its two ends, replayed once.  Layer-step n
    is token (n // n_layers) of the workload on layer copy n % n_layers, the
    copies being enough that the other copies' steps move more than 3x the L2
    between two steps of one copy (so no flush is needed and none is timed).
    A 4-byte fill between layer-steps ends the launch overlap: each step's
    first kernel starts after the previous step's last one has completed, as
    after the other ops of a model.  With e2e, each step's inputs are read in
    place from pinned host memory and its output is stored there."""
    import torch
    from qsa_workload import make_workload
    from sparse_attention_long_qsa_gb300.layer import PackedInputs, QSALayer, step_inputs

    wl = make_workload(name, seed=0)
    n_tok = len(wl.steps)
    L0 = QSALayer.from_workload(wl, 0, device=dev)
    L0.warm(torch.from_numpy(wl.prompt_dirty()).to(dev))
    step_bytes = float(np.mean([sum(algorithmic_bytes(wl, i).values()) for i in range(n_tok)]))
    state_bytes = sum(getattr(L0, k).numel() * getattr(L0, k).element_size()
                      for k in ("idx_k", "k_cache", "v_cache", "blk_cells", "pooled", "cells", "count", "out",
                                "ws_index", "ws_attn"))
    n_layers = chain_layers(step_bytes, state_bytes)
    layers = [L0] + [clone_layer(L0) for _ in range(n_layers - 1)]
    inputs = [step_inputs(st, device=dev, new_cells=True) for st in wl.steps]
    toks = [len(st.tok_pos) for st in wl.steps]
    sep = torch.zeros(1, dtype=torch.int32, device=dev)
    xev = _ExternalEvents()
    io_keys = ("tok_seq", "tok_pos", "q", "q_idx", "w_idx", "cells", "k_new", "v_new", "idx_new")
    host = None
    if e2e:
        staging = PackedInputs({k: (tuple(inputs[0][k].shape), inputs[0][k].dtype) for k in io_keys}, device=dev)
        host = []
        for i, st in enumerate(wl.steps):
            h = {"in": staging.pack({k: getattr(st, k) for k in io_keys})}
            h["views"] = staging.host_views(h["in"])
            h["out"] = torch.empty((toks[i], wl.cfg["n_q_heads"], wl.cfg["head_dim"]),
                                   dtype=torch.float32).pin_memory()
            host.append(h)

    def step(n, with_io=False):
        i, l = (n // n_layers) % n_tok, n % n_layers
        if with_io:
            layers[l].full_step(**{**inputs[i], **host[i]["views"]}, out=host[i]["out"], union=union,
                                in_cluster=in_cluster)
        else:
            layers[l].full_step(**inputs[i], union=union, in_cluster=in_cluster)
        sep.zero_()
        return toks[i]

    for n in range(W):
        step(n)
    torch.cuda.synchronize()

    def timed(with_io):
        """Median over replays of the K-step graph (one replay, then ~1 s of
        replays with the clocks sampled, or 3 with host I/O)."""
        e0, e1 = xev.new(), xev.new()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        tokens = 0
        with torch.cuda.graph(g):
            xev.record(e0)
            for n in range(W, W + K):
                tokens += step(n, with_io)
            xev.record(e1)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        reps = [e0.elapsed_time(e1)]
        n_rep = 2 if with_io else min(200, max(3, int(np.ceil(1000.0 / max(reps[0], 1e-3)))))
        if clocks and not with_io:
            clocks.start()
        for _ in range(n_rep):
            g.replay()
            torch.cuda.synchronize()
            reps.append(e0.elapsed_time(e1))
        ck = clocks.stop() if clocks and not with_io else None
        del g
        return float(np.median(reps)), tokens, ck, len(reps)

    ms, tokens, ck, n_rep = timed(False)
    res = dict(value=tokens / (ms / 1e3), ms_per_step=ms / K, tokens=tokens, n_layers=n_layers,
               state_bytes=state_bytes, step_bytes=step_bytes, clocks=ck, replays=n_rep)
    if e2e:
        ms2, tokens2, _, _ = timed(True)
        h2d = float(sum(n for (_, _, _, n) in staging.fields.values()))
        d2h = float(np.mean([host[i]["out"].numel() * 4 for i in range(n_tok)]))
        res["e2e"] = {"value": tokens2 / (ms2 / 1e3), "unit": "tokens/s",
                      "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                      "how": "the same back-to-back layer-steps with each step's inputs in pinned host memory, "
                             "read in place by the kernels over NVLink-C2C, and its output stored by the "
                             "attention kernel into pinned host memory"}
    st, flags = __import__("sparse_attention_long_qsa_gb300.qsa", fromlist=["qsa"]).debug_check()
    if st != 0:
        raise RuntimeError(f"device error word set during the bench: {flags:#x}")
    del layers, L0, inputs
    torch.cuda.empty_cache()
    return res


def replica_value(local_ms: float, tokens: int, world: int, dist=None, device="cpu"):
    """Whole-job tokens/s of `world` replicas that each processed `tokens` in
    their own `local_ms`: all replicas' tokens over the slowest replica's
    time (max over ranks).  Returns (tokens/s, max ms)."""
    import torch
    if dist is not None and world > 1:
        t = torch.tensor([float(local_ms)], device=device, dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        local_ms = float(t.item())
    return world * tokens / (local_ms / 1e3), local_ms


def launch_note(res, path, ch=None):
    kern = f"{res['launches_per_step']} kernels ({', '.join(res['kernels'])}) chained by programmatic dependent launch"
    if ch is not None:
        return ("the K timed layer-steps captured back to back as one CUDA graph with an event node at each "
                "end: per layer-step qsa_kv_append (re-pooling the blocks it dirties) + "
                f"qsa_index_attn = {kern}, then a 4-byte fill that ends the launch overlap; {chain_note(ch)} "
                "(gpu_launches counts one replay)")
    return ("the K timed steps captured as one CUDA graph (per step: L2 flush, start event, "
            + ("qsa_kv_append (re-pooling the blocks it dirties) + qsa_index_attn"
               if path == "full" else
               "table append outside the events, qsa_pool_update + qsa_index_topk + qsa_sparse_attn")
            + f" = {kern}, end event), replayed once")


def roofline_of(res, name, hbm, peak_src):
    """The roofline object of a measured workload: its dominant kernel's
    algorithmic bytes over that kernel's live event time."""
    achieved = res["dom_bytes"] / (res["dom_ms"] * 1e-3) / 1e9
    traffic, tsrc = ncu_traffic(name, res["dominant"])
    return {"kernel": res["dominant"], "choice": "kernel moving the most algorithmic bytes per step",
            "longest_kernel": res["longest"], "bound": "hbm", "achieved": achieved,
            "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
            "peak_source": f"hbm_gbs {peak_src}",
            "bytes_per_launch": res["dom_bytes"], "us_per_launch": res["dom_ms"] * 1e3,
            "traffic": traffic, "traffic_source": tsrc}


def event_line(res):
    """The event-bracketed timing of measure_config (each step between its own
    event nodes after an L2 flush)."""
    return {"value": res["value"], "ms_per_step": res["ms_per_step"], "step_us_p50": res["step_us_p50"],
            "step_us_p90": res["step_us_p90"],
            "how": "each step between two event nodes of the graph, the L2 flushed before it (the event nodes "
                   "and the first launch after them add ~6 us per step)"}


def chain_note(ch):
    return (f"{ch['n_layers']} layer copies of {ch['state_bytes'] / 1e6:.0f} MB, "
            f"{ch['step_bytes'] / 1e6:.1f} MB of algorithmic bytes per layer-step; median of "
            f"{ch['replays']} replays of the K-step graph")


def workload_line(res, name, hbm, peak_src, cpu=None, chain=None):
    """Per-workload results: throughput (back-to-back layer-steps when `chain`
    is given, else event-bracketed), end to end, roofline, kernel times."""
    top = chain if chain is not None else res
    line = {
        "workload": DESCR[name], "value": top["value"], "unit": "tokens/s",
        "ms_per_step": top["ms_per_step"],
        "e2e": top.get("e2e"), "cpu_baseline": cpu,
        "roofline": roofline_of(res, name, hbm, peak_src),
        "kernels_us": {k: round(v, 3) for k, v in res["kern_us"].items()},
        "kernels_gbs": {k: round(v, 1) for k, v in res["kern_gbs"].items()},
        "step_bytes": res["step_bytes"],
        "step_gbs": res["step_bytes"] / (top["ms_per_step"] * 1e-3) / 1e9,
    }
    if chain is not None:
        line["chain"] = chain_note(chain)
        line["event_bracketed"] = event_line(res)
    else:
        line["step_us_p50"], line["step_us_p90"] = res["step_us_p50"], res["step_us_p90"]
    return line


def cpu_line(wl, name, seconds):
    rate, steps, secs, threads = cpu_oracle_rate(wl, seconds)
    per = min(len(wl.steps[0].tok_pos), 8)
    return {"value": rate, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{steps} consecutive steps of the {name} workload, full oracle step each (append, "
                      f"pool the dirty blocks, score every block, select, expand, attend {per} token(s)), "
                      f"{secs:.1f} s"}


def run_native(args, rank, world, local):
    import torch
    import __graft_entry__
    __graft_entry__.build()
    dev = f"cuda:{local}"
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl", device_id=torch.device(dev))
    peaks = _peaks()
    hbm = peaks["hbm_gbs"] if peaks else 6800.0
    peak_src = "of measured" if peaks else "of fallback"

    clocks = Clocks(local)
    chained = args.path == "full"
    # per-kernel breakdown, roofline kernel and event-bracketed steps (rank 0
    # only when chained: the headline comes from the chain)
    res = None
    if rank == 0 or not chained:
        res = measure_config(args.config, args.steps, args.warmup, dev, path=args.path,
                             clocks=None if chained else clocks, e2e=not chained, union=args.union,
                             in_cluster=args.in_cluster)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    ch = (measure_chain(args.config, args.steps, args.warmup, dev, clocks=clocks, union=args.union,
                        in_cluster=args.in_cluster) if chained else None)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    top = ch if chained else res
    value, max_ms = replica_value(top["ms_per_step"] * args.steps, top["tokens"], world, dist, dev)

    paths = None
    if rank == 0:
        paths = {args.path: {"value": top["value"], "ms_per_step": top["ms_per_step"],
                             "launches_per_step": res["launches_per_step"],
                             "timing": "back-to-back layer-steps" if chained else "event-bracketed"}}
        if chained:
            paths[args.path]["event_bracketed"] = {"value": res["value"], "ms_per_step": res["ms_per_step"]}
    if rank == 0 and args.compare:
        other = "calls" if args.path == "full" else "full"
        ro = measure_config(args.config, args.steps, args.warmup, dev, path=other, e2e=False)
        paths[other] = {"value": ro["value"], "ms_per_step": ro["ms_per_step"],
                        "launches_per_step": ro["launches_per_step"],
                        "timing": "event-bracketed",
                        "kernels_us": {k: round(v, 3) for k, v in ro["kern_us"].items()}}

    # the 250k q8_0 decode (the long-context target) on a complete line of its
    # own: end to end, CPU baseline, roofline
    target = None
    if args.target not in ("", "none", args.config) and rank == 0:
        rt = measure_config(args.target, min(args.steps, 256), args.warmup, dev, path=args.path,
                            e2e=not chained)
        ct = measure_chain(args.target, min(args.steps, 256), args.warmup, dev) if chained else None
        cpu_t = None if args.no_cpu else cpu_line(rt["wl"], args.target, args.cpu_seconds)
        target = workload_line(rt, args.target, hbm, peak_src, cpu_t, chain=ct)
        target["config"] = bench_config(args.target, len(rt["wl"].steps[0].tok_pos))
        del rt

    secondary = {}
    if args.secondary and rank == 0:
        for item in args.secondary.split(","):
            # "name" or "name:union" (the pairs' union attention)
            name, _, mode = item.partition(":")
            if item in (args.config, args.target, "", "none"):
                continue
            r2 = measure_config(name, min(args.steps, 128), args.warmup, dev, path=args.path, e2e=False,
                                union=mode == "union")
            c2 = (measure_chain(name, min(args.steps, 128), args.warmup, dev, e2e=False, union=mode == "union")
                  if chained else None)
            secondary[item] = workload_line(r2, name, hbm, peak_src, chain=c2)
            if mode == "union":
                secondary[item]["roofline"].update(traffic=None,
                                                   traffic_source="no ncu capture of the union attention")
            del r2

    cpu = None
    if rank == 0 and not args.no_cpu:
        cpu = cpu_line(res["wl"], args.config, args.cpu_seconds)
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return
    wl = res["wl"]
    main_line = workload_line(res, args.config, hbm, peak_src, cpu, chain=ch)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": max_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16" if wl.cfg["kv_type"] == "f16" else "q8_0",
        "data": "synthetic (seeded N(0,1) K/V/keys, U(0,1) weights)",
        "config": bench_config(args.config, len(wl.steps[0].tok_pos)),
        "launch": {"path": args.path, "steps": launch_note(res, args.path, ch),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": main_line["roofline"],
        "kernels_us": main_line["kernels_us"],
        "kernels_gbs": main_line["kernels_gbs"],
        "step_bytes": res["step_bytes"],
        "step_gbs": main_line["step_gbs"],
        "cpu_baseline": cpu,
        "e2e": top.get("e2e"),
        "gpu_launches": res["launches_per_step"] * args.steps,
        "paths": paths,
        "clocks": top["clocks"],
        "target": target,
        "secondary": secondary or None,
    }
    if chained:
        line["chain"] = main_line["chain"]
        line["event_bracketed"] = main_line["event_bracketed"]
    else:
        line["step_us_p50"], line["step_us_p90"] = res["step_us_p50"], res["step_us_p90"]
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1024)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--config", default="50k", choices=list(DESCR))
    ap.add_argument("--target", default="250k_q8",
                    help="workload given a complete line of its own under `target` (rank 0; '' for none)")
    ap.add_argument("--secondary", default="250k_f16,5x250k_q8",
                    help="comma list of further workloads timed on rank 0 ('none': no others); "
                         "'name:union' times a workload with the token pairs' union attention")
    ap.add_argument("--path", default="full", choices=["full", "calls"],
                    help="full: append (with the pool update) + index + attention (the layer's whole step); "
                         "calls: the last three, the table appended outside the timed region")
    ap.add_argument("--in-cluster", action="store_true",
                    help="path full: the selection inside the attention clusters (QSA_INDEX_ATTN_IN_CLUSTER)")
    ap.add_argument("--union", action="store_true",
                    help="path full: token pairs attend over the union of their lists (QSA_INDEX_ATTN_UNION)")
    ap.add_argument("--no-compare", dest="compare", action="store_false",
                    help="do not also time the other path")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--flush-mb", type=int, default=1024,
                    help="L2 flush write per step, MiB (must exceed the 129 MB L2)")
    args = ap.parse_args()
    FLUSH_BYTES[0] = max(args.flush_mb, 256) << 20
    rank, world, local = _env_rank()
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_native(args, rank, world, local)


if __name__ == "__main__":
    main()
