"""The C-ABI library without a GPU: it builds, loads, exports every symbol
include/qsa.h declares, and rejects invalid calls on the host before any CUDA
work.  No compute call is made here."""
import ctypes
import os
import re

import numpy as np
import pytest

from sparse_attention_long_qsa_gb300 import build as qbuild
from sparse_attention_long_qsa_gb300 import qsa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qsa.h")


@pytest.fixture(scope="module")
def L():
    qbuild.build()
    return qsa.lib()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qsa_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    names = _declared()
    assert names == sorted(qsa.EXPORTS)
    out = os.popen(f"nm -D --defined-only {qsa.LIB_PATH}").read()
    exported = set(re.findall(r" T (qsa_[a-z0-9_]+)", out))
    for n in names:
        assert n in exported, n
        assert hasattr(L, n)


def test_config_defaults_and_pitch(L):
    c = qsa.config()
    assert (c.n_q_heads, c.n_kv_heads, c.head_dim, c.n_idx_heads, c.idx_dim) == (16, 2, 256, 4, 128)
    assert (c.compress_ratio, c.top_k, c.kv_type) == (4, 2048, 0)
    assert c.rope_theta == 1e6 and abs(c.rms_eps - 1e-6) < 1e-12 and c.attn_scale == 1 / 16
    assert qsa.cells_per_token(c) == 2051
    assert qsa.cells_per_token(qsa.config(top_k=16)) == 19


@pytest.mark.parametrize("over,status", [
    (dict(head_dim=128), -3), (dict(idx_dim=64), -3), (dict(n_q_heads=12), -3),
    (dict(top_k=2050), -3), (dict(compress_ratio=0), -1), (dict(kv_type=7), -1),
    (dict(n_idx_heads=2), -3), (dict(rope_theta=-1.0), -1),
])
def test_config_rejected_before_launch(L, over, status):
    c = qsa.config(**over)
    fake = ctypes.c_void_p(0x10000)
    st = L.qsa_pool_update(ctypes.byref(c), fake, 10, fake, fake, 10, fake, 4, fake, fake, None)
    assert st == status
    assert L.qsa_cells_per_token(ctypes.byref(c)) == -1


def test_null_and_workspace_checks(L):
    c = qsa.config()
    fake = ctypes.c_void_p(0x10000)
    # null pointer with work to do
    assert L.qsa_pool_update(ctypes.byref(c), None, 10, fake, fake, 10, fake, 4, fake, fake, None) == -1
    # nothing to do: no pointer is read
    assert L.qsa_pool_update(ctypes.byref(c), None, 10, None, None, 10, None, 0, None, None, None) == 0
    # negative sizes
    assert L.qsa_pool_update(ctypes.byref(c), fake, -1, fake, fake, 10, fake, 4, fake, fake, None) == -1
    need = L.qsa_index_topk_workspace_size(ctypes.byref(c), 5, 62_532)
    assert need > 5 * 62_532 * 4
    args = [ctypes.byref(c), 5, 5] + [fake] * 6 + [100, fake, fake, 1, 62_532, 1000, fake, fake, None, 0]
    assert L.qsa_index_topk(*args, fake, need - 1, None) == -4
    assert L.qsa_index_topk(*args, ctypes.c_void_p(0x10010), need, None) == -4   # misaligned
    assert L.qsa_index_topk(*args, None, need, None) == -4
    # sparse attention merges its splits in distributed shared memory: no workspace
    assert L.qsa_sparse_attn_workspace_size(ctypes.byref(c), 5) == 0
    # misaligned K cache
    bad = [ctypes.byref(c), 5, fake, ctypes.c_void_p(0x10002), fake, 1000, fake, fake, fake]
    assert L.qsa_sparse_attn(*bad, None, 0, None) == -1
    assert L.qsa_sparse_attn(ctypes.byref(c), 5, None, fake, fake, 1000, fake, fake, fake, None, 0, None) == -1
    assert L.qsa_index_topk(ctypes.byref(c), 70_000, 70_000, *([fake] * 6), 100, fake, fake, 1, 10, 10,
                            fake, fake, None, 0, fake, need, None) == -3
    # a hint length without a list; a negative length other than the query-blocks hint
    assert L.qsa_index_topk(*args[:-2], None, 3, fake, need, None) == -1
    assert L.qsa_index_topk(*args[:-2], None, -2, fake, need, None) == -1
    assert L.qsa_index_topk(*args[:-2], fake, -1, fake, need, None) == -1
    # more tokens than the workspace was sized for
    assert L.qsa_index_topk(ctypes.byref(c), 6, 5, *([fake] * 6), 100, fake, fake, 1, 10, 10,
                            fake, fake, None, 0, fake, need, None) == -2
    # beyond the selection kernel's per-token block limit
    assert L.qsa_index_topk(ctypes.byref(c), 1, 1, *([fake] * 6), 100, fake, fake, 1, (1 << 20) + 1, 10,
                            fake, fake, None, 0, fake, need, None) == -3
    assert L.qsa_status_string(-4) == b"workspace null, misaligned or too small"


def test_union_attention_host_checks(L):
    """qsa_sparse_attn_union takes qsa_sparse_attn's checks, and refuses lists
    longer than its shared-memory union holds (top_k 8192) before any launch;
    qsa_index_attn refuses both attention flags at once."""
    fake = ctypes.c_void_p(0x10000)
    c = qsa.config()
    bad = [ctypes.byref(c), 5, fake, ctypes.c_void_p(0x10002), fake, 1000, fake, fake, fake]
    assert L.qsa_sparse_attn_union(*bad, None, 0, None) == -1
    big = qsa.config(top_k=8192)
    assert L.qsa_sparse_attn_union(ctypes.byref(big), 5, fake, fake, fake, 1000, fake, fake, fake,
                                   None, 0, None) == -3
    assert L.qsa_sparse_attn_union(ctypes.byref(big), 0, None, None, None, 0, None, None, None,
                                   None, 0, None) == -3
    need = L.qsa_index_topk_workspace_size(ctypes.byref(c), 5, 1000)
    args = [ctypes.byref(c), 5, 5] + [fake] * 6 + [100, fake, fake, 1, 1000, fake, fake, fake, 1000,
                                                   fake, fake, fake, None, 0]
    assert L.qsa_index_attn(*args, 3, fake, need, None) == -1
    assert L.qsa_index_attn(*args, 4, fake, need, None) == -1
    assert L.qsa_index_attn_kernels(ctypes.byref(c), 5, 1, 1000, 3) == 0


def test_blocks_dirty_host_helper(L):
    rng = np.random.default_rng(0)
    old = rng.integers(-1, 1000, (300, 4)).astype(np.int32)
    new = old.copy()
    for s in (3, 77, 78, 299):
        new[s, rng.integers(0, 4)] += 1
    got = qsa.blocks_dirty(old, new, 4)
    np.testing.assert_array_equal(got, [3, 77, 78, 299])
    new[5, 0] = -7
    got = qsa.blocks_dirty(old, new, 4)
    np.testing.assert_array_equal(got, [3, 5, 77, 78, 299, -1, -1, -1])
    np.testing.assert_array_equal(qsa.blocks_dirty(old, old, 4), [-1, -1, -1, -1])
    np.testing.assert_array_equal(qsa.blocks_dirty(old, old, 0), np.zeros(0, dtype=np.int32))
    # capacity too small: status -2 and the needed length
    n = ctypes.c_int32(0)
    buf = np.zeros(2, dtype=np.int32)
    st = L.qsa_blocks_dirty(old.ctypes.data, new.ctypes.data, 300, 4, buf.ctypes.data, 2, ctypes.byref(n), 4)
    assert st == -2 and n.value == 8


def test_binding_refuses_cpu_tensors(L):
    import torch
    c = qsa.config()
    t = torch.zeros(4, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        qsa.pool_update(c, torch.zeros((4, 128), dtype=torch.float16), torch.zeros((1, 4), dtype=torch.int32),
                        torch.zeros(1, dtype=torch.int32), t, torch.ones(128), torch.zeros((1, 128)))


def test_kv_append_host_checks(L):
    c = qsa.config()
    f = 0x10000
    base = [ctypes.byref(c), 4, f, f, f, f, f, f, f, f, f, 1000, f, 100, f, f, 1, f, 4, None, None, None, None]
    def call(**kw):
        args = list(base)
        for i, v in kw.items():
            args[int(i[1:])] = v
        return L.qsa_kv_append(*args)
    assert call(a1=0) == 0                      # nothing to append: no pointer is read
    assert call(a1=1025) == -3                  # beyond the dirty-list kernel's token limit
    assert call(a18=3) == -2                    # fewer dirty entries than tokens
    assert call(a2=None) == -1
    assert call(a5=f + 8) == -1                 # new K rows must be 16-byte aligned
    assert call(a10=f + 2) == -1                # indexer keys must be 16-byte aligned
    assert call(a16=0) == -1                    # no sequence
    assert call(a21=f) == -1                    # re-pooling needs slot_block_idx and norm_w
    assert L.qsa_kv_append(ctypes.byref(qsa.config(kv_type=7)), *base[1:]) == -1


def test_index_topk_kernel_plan(L):
    """Token-tiled scoring (score + hist + select) exactly when tokens share
    sequences: n_tokens > 8 and n_tokens >= 2 * n_seq."""
    plain, tiled = ["score", "select"], ["score", "hist", "select"]
    assert qsa.index_topk_kernels(1, 1) == plain
    assert qsa.index_topk_kernels(5, 5) == plain
    assert qsa.index_topk_kernels(5, 1) == plain
    assert qsa.index_topk_kernels(8, 1) == plain
    assert qsa.index_topk_kernels(9, 5) == plain
    assert qsa.index_topk_kernels(9, 1) == tiled
    assert qsa.index_topk_kernels(10, 5) == tiled
    assert qsa.index_topk_kernels(512, 1) == tiled
    assert L.qsa_index_topk_kernels(0, 1) == 0


def test_packed_inputs_layout_round_trip():
    """One-copy staging of a step's inputs: 256-byte aligned fields, the
    views read back exactly the packed arrays (host-only check)."""
    import numpy as np
    import torch
    from sparse_attention_long_qsa_gb300.layer import PackedInputs
    rng = np.random.default_rng(0)
    arrs = {"tok_seq": np.array([3], dtype=np.int32), "q": rng.standard_normal((1, 16, 256)).astype(np.float16),
            "q_idx": rng.standard_normal((1, 4, 128)).astype(np.float32), "w": np.arange(5, dtype=np.int64)}
    fields = {k: (a.shape, {np.int32: torch.int32, np.float16: torch.float16, np.float32: torch.float32,
                            np.int64: torch.int64}[a.dtype.type]) for k, a in arrs.items()}
    p = PackedInputs(fields, device="cpu", pin=False)
    offs = [o for o, *_ in p.fields.values()]
    assert all(o % 256 == 0 for o in offs) and offs == sorted(offs)
    host = p.pack(arrs)
    p.dev[:host.numel()].copy_(host)
    for k, a in arrs.items():
        np.testing.assert_array_equal(p.views[k].numpy(), a)


def test_index_topk_noalloc_host_limits(L):
    """The no-allocation entry point refuses, before any CUDA call, what its
    static scratch array cannot hold (more than 8 tokens or 262,144 blocks per
    sequence), and validates like qsa_index_topk otherwise."""
    c = qsa.config()
    f = ctypes.c_void_p(0x10000)
    def call(n_tokens, max_blocks, cells=f, cfg=c):
        return L.qsa_index_topk_noalloc(ctypes.byref(cfg), n_tokens, f, f, f, f, f, f, 100, f, f, 1,
                                        max_blocks, 1000, cells, f, None)
    assert call(9, 1000) == -4
    assert call(1, 262_145) == -4
    assert call(0, 262_144) == 0                 # nothing to do
    assert call(1, 1000, cells=None) == -1
    assert call(1, -1) == -1
    assert call(1, 1000, cfg=qsa.config(head_dim=128)) == -3
