"""ctypes binding of libqsa (include/qsa.h): argument marshalling only.

Every function takes CUDA torch tensors (device memory and the current
stream come from PyTorch), checks dtype / device / contiguity, and calls the
C entry point of the same name.  No step of the computation runs here, and
there is no CPU fallback: a missing libqsa.so or a CPU tensor raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqsa.so")

QSA_OK = 0
QSA_KV_F16 = 0
QSA_KV_Q8_0 = 1
QSA_HINT_QUERY_BLOCKS = -1
QSA_INDEX_ATTN_IN_CLUSTER = 1
QSA_INDEX_ATTN_UNION = 2
STATUS = {0: "QSA_OK", -1: "QSA_ERR_INVALID_ARG", -2: "QSA_ERR_SHAPE", -3: "QSA_ERR_UNSUPPORTED",
          -4: "QSA_ERR_WORKSPACE", -5: "QSA_ERR_CUDA", -6: "QSA_ERR_DEVICE_BOUNDS"}

# Every symbol include/qsa.h declares.
EXPORTS = ("qsa_config_init", "qsa_cells_per_token", "qsa_pool_update", "qsa_index_scores",
           "qsa_index_topk_workspace_size", "qsa_index_topk", "qsa_index_topk_noalloc",
           "qsa_sparse_attn_workspace_size",
           "qsa_sparse_attn", "qsa_sparse_attn_union", "qsa_index_attn", "qsa_index_attn_kernels", "qsa_kv_append", "qsa_blocks_dirty",
           "qsa_debug_check", "qsa_profile_kernel", "qsa_index_topk_kernels", "qsa_status_string")

# Kernel ids of qsa_profile_kernel.
KERNELS = {"pool": 0, "score": 1, "hist": 2, "select": 3, "attn": 4, "append": 5, "select_attn": 6}


class QSAError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS.get(status, status)}")
        self.status = status


class Config(ctypes.Structure):
    _fields_ = [("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("n_idx_heads", ctypes.c_int32),
                ("idx_dim", ctypes.c_int32), ("compress_ratio", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("rope_theta", ctypes.c_float),
                ("rms_eps", ctypes.c_float), ("attn_scale", ctypes.c_float),
                ("kv_type", ctypes.c_int32)]


_lib = None
_lib_lock = threading.Lock()
_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t


def lib():
    """Load libqsa.so (built in-tree by sparse_attention_long_qsa_gb300.build);
    safe to call from several threads."""
    if _lib is not None:
        return _lib
    with _lib_lock:
        return _load()


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "`python -m sparse_attention_long_qsa_gb300.build`")
    L = ctypes.CDLL(LIB_PATH)
    CP = ctypes.POINTER(Config)
    L.qsa_config_init.argtypes = [CP]
    L.qsa_config_init.restype = _I32
    L.qsa_cells_per_token.argtypes = [CP]
    L.qsa_cells_per_token.restype = _I32
    L.qsa_pool_update.argtypes = [CP, _P, _I64, _P, _P, _I64, _P, _I32, _P, _P, _P]
    L.qsa_pool_update.restype = _I32
    L.qsa_index_scores.argtypes = [CP, _I32, _P, _P, _P, _P, _P, _I64, _P, _P, _I32, _I64, _P, _P]
    L.qsa_index_scores.restype = _I32
    L.qsa_index_topk_workspace_size.argtypes = [CP, _I32, _I64]
    L.qsa_index_topk_workspace_size.restype = _SZ
    L.qsa_index_topk.argtypes = [CP, _I32, _I32, _P, _P, _P, _P, _P, _P, _I64, _P, _P, _I32, _I64, _I64,
                                 _P, _P, _P, _I32, _P, _SZ, _P]
    L.qsa_index_topk.restype = _I32
    L.qsa_index_topk_noalloc.argtypes = [CP, _I32, _P, _P, _P, _P, _P, _P, _I64, _P, _P, _I32, _I64,
                                         _I64, _P, _P, _P]
    L.qsa_index_topk_noalloc.restype = _I32
    L.qsa_sparse_attn_workspace_size.argtypes = [CP, _I32]
    L.qsa_sparse_attn_workspace_size.restype = _SZ
    L.qsa_sparse_attn.argtypes = [CP, _I32, _P, _P, _P, _I64, _P, _P, _P, _P, _SZ, _P]
    L.qsa_sparse_attn.restype = _I32
    L.qsa_sparse_attn_union.argtypes = [CP, _I32, _P, _P, _P, _I64, _P, _P, _P, _P, _SZ, _P]
    L.qsa_sparse_attn_union.restype = _I32
    L.qsa_index_attn.argtypes = [CP, _I32, _I32, _P, _P, _P, _P, _P, _P, _I64, _P, _P, _I32, _I64,
                                 _P, _P, _P, _I64, _P, _P, _P, _P, _I32, ctypes.c_uint32, _P, _SZ, _P]
    L.qsa_index_attn.restype = _I32
    L.qsa_index_attn_kernels.argtypes = [CP, _I32, _I32, _I64, ctypes.c_uint32]
    L.qsa_index_attn_kernels.restype = ctypes.c_uint32
    L.qsa_kv_append.argtypes = [CP, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _P, _I64, _P, _P, _I32,
                                _P, _I32, _P, _P, _P, _P]
    L.qsa_kv_append.restype = _I32
    L.qsa_blocks_dirty.argtypes = [_P, _P, _I64, _I32, _P, _I32, ctypes.POINTER(_I32), _I32]
    L.qsa_blocks_dirty.restype = _I32
    L.qsa_debug_check.argtypes = [_P, ctypes.POINTER(ctypes.c_uint32)]
    L.qsa_debug_check.restype = _I32
    L.qsa_profile_kernel.argtypes = [_I32, _P, _P]
    L.qsa_profile_kernel.restype = _I32
    L.qsa_index_topk_kernels.argtypes = [_I32, _I32]
    L.qsa_index_topk_kernels.restype = ctypes.c_uint32
    L.qsa_status_string.argtypes = [_I32]
    L.qsa_status_string.restype = ctypes.c_char_p
    _lib = L
    return L


def config(**over) -> Config:
    """The qwen4exp QSA layer's configuration, with fields overridden by name
    (kv_type may be given as "f16" / "q8_0")."""
    c = Config()
    _check(lib().qsa_config_init(ctypes.byref(c)), "qsa_config_init")
    for k, v in over.items():
        if k == "kv_type" and isinstance(v, str):
            v = {"f16": QSA_KV_F16, "q8_0": QSA_KV_Q8_0}[v]
        if not hasattr(c, k):
            raise KeyError(k)
        setattr(c, k, v)
    return c


def config_from_dict(d: dict) -> Config:
    keys = [f for f, _ in Config._fields_]
    return config(**{k: d[k] for k in keys if k in d})


def _check(st: int, what: str):
    if st != QSA_OK:
        raise QSAError(st, what)


def _stream(stream):
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ptr(t, dtype, name, allow_none=False, host_ok=False):
    """Device address of a CUDA tensor on the current device.  host_ok: a
    step's own inputs and outputs may instead be page-locked (pinned) host
    tensors, which the kernels read and write in place over the host link."""
    import torch
    if t is None:
        if allow_none:
            return None
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if not t.is_cuda:
        if not (host_ok and t.is_pinned()):
            raise ValueError(f"{name} must be a CUDA tensor" + (" or a pinned host tensor" if host_ok else "")
                             + " (libqsa has no CPU path)")
    elif t.get_device() != torch.cuda.current_device():
        # the library launches on the current device: another device's
        # memory would be read through an address that is not mapped there
        raise ValueError(f"{name} is on {t.device}, the current device is cuda:{torch.cuda.current_device()}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _io(t, dtype, name):
    """A step input or output: device memory or pinned host memory."""
    return _ptr(t, dtype, name, host_ok=True)


def cells_per_token(cfg: Config) -> int:
    return int(lib().qsa_cells_per_token(ctypes.byref(cfg)))


def pool_update(cfg, idx_k, blk_cells, slot_block_idx, dirty, norm_w, pooled, stream=None):
    import torch
    L = lib()
    n_cells = idx_k.shape[0]
    n_slots = pooled.shape[0]
    st = L.qsa_pool_update(ctypes.byref(cfg), _ptr(idx_k, torch.float16, "idx_k"), n_cells,
                           _ptr(blk_cells, torch.int32, "blk_cells"),
                           _ptr(slot_block_idx, torch.int32, "slot_block_idx"), n_slots,
                           _ptr(dirty, torch.int32, "dirty"), int(dirty.numel()),
                           _ptr(norm_w, torch.float32, "norm_w"),
                           _ptr(pooled, torch.float32, "pooled"), _stream(stream))
    _check(st, "qsa_pool_update")


def index_scores(cfg, q_idx, w_idx, tok_seq, tok_pos, pooled, seq_blk_off, seq_blk_slots,
                 max_blocks: int, scores, stream=None):
    import torch
    T = int(tok_pos.numel())
    st = lib().qsa_index_scores(
        ctypes.byref(cfg), T, _io(q_idx, torch.float32, "q_idx"), _io(w_idx, torch.float32, "w_idx"),
        _io(tok_seq, torch.int32, "tok_seq"), _io(tok_pos, torch.int32, "tok_pos"),
        _ptr(pooled, torch.float32, "pooled"), int(pooled.shape[0]),
        _ptr(seq_blk_off, torch.int64, "seq_blk_off"), _ptr(seq_blk_slots, torch.int32, "seq_blk_slots"),
        int(seq_blk_off.numel()) - 1, int(max_blocks), _ptr(scores, torch.float32, "scores"),
        _stream(stream))
    _check(st, "qsa_index_scores")


def index_topk_workspace_size(cfg, max_tokens: int, max_blocks: int) -> int:
    return int(lib().qsa_index_topk_workspace_size(ctypes.byref(cfg), int(max_tokens), int(max_blocks)))


def index_topk(cfg, q_idx, w_idx, tok_seq, tok_pos, pooled, blk_cells, seq_blk_off, seq_blk_slots,
               max_blocks: int, n_cells: int, cells, count, workspace, max_tokens: int,
               recomputed=None, stream=None):
    """workspace: a uint8 CUDA tensor of index_topk_workspace_size(cfg,
    max_tokens, max_blocks) bytes, zero-filled once when allocated.
    recomputed: optional scheduling hint: an int32 CUDA tensor, the
    (host-written) dirty list of the pool update issued just before on the
    same stream, or "query_blocks" after an append of exactly these tokens."""
    import torch
    T = int(tok_pos.numel())
    if isinstance(recomputed, str) and recomputed == "query_blocks":
        rec_ptr, rec_n = None, QSA_HINT_QUERY_BLOCKS
    else:
        rec_ptr = _ptr(recomputed, torch.int32, "recomputed") if recomputed is not None else None
        rec_n = int(recomputed.numel()) if recomputed is not None else 0
    st = lib().qsa_index_topk(
        ctypes.byref(cfg), T, int(max_tokens), _io(q_idx, torch.float32, "q_idx"),
        _io(w_idx, torch.float32, "w_idx"),
        _io(tok_seq, torch.int32, "tok_seq"), _io(tok_pos, torch.int32, "tok_pos"),
        _ptr(pooled, torch.float32, "pooled"), _ptr(blk_cells, torch.int32, "blk_cells"),
        int(pooled.shape[0]), _ptr(seq_blk_off, torch.int64, "seq_blk_off"),
        _ptr(seq_blk_slots, torch.int32, "seq_blk_slots"), int(seq_blk_off.numel()) - 1,
        int(max_blocks), int(n_cells), _ptr(cells, torch.int32, "cells"),
        _ptr(count, torch.int32, "count"), rec_ptr, rec_n, _ptr(workspace, torch.uint8, "workspace"),
        int(workspace.numel()), _stream(stream))
    _check(st, "qsa_index_topk")


def index_attn(cfg, q_idx, w_idx, tok_seq, tok_pos, pooled, blk_cells, seq_blk_offs, seq_blk_slots,
               max_blocks: int, q, k_cache, v_cache, n_cells: int, cells, count, out, workspace,
               max_tokens: int, recomputed=None, stream=None, in_cluster: bool = False,
               union: bool = False):
    """qsa_index_topk then qsa_sparse_attn in one call (same workspace and
    hint as index_topk); fills cells, count and out.  in_cluster: the
    selection runs inside the attention clusters where the call's limits
    allow (QSA_INDEX_ATTN_IN_CLUSTER); union: token pairs attend over the
    union of their lists (QSA_INDEX_ATTN_UNION)."""
    import torch
    T = int(tok_pos.numel())
    if isinstance(recomputed, str) and recomputed == "query_blocks":
        rec_ptr, rec_n = None, QSA_HINT_QUERY_BLOCKS
    else:
        rec_ptr = _ptr(recomputed, torch.int32, "recomputed") if recomputed is not None else None
        rec_n = int(recomputed.numel()) if recomputed is not None else 0
    st = lib().qsa_index_attn(
        ctypes.byref(cfg), T, int(max_tokens), _io(q_idx, torch.float32, "q_idx"),
        _io(w_idx, torch.float32, "w_idx"),
        _io(tok_seq, torch.int32, "tok_seq"), _io(tok_pos, torch.int32, "tok_pos"),
        _ptr(pooled, torch.float32, "pooled"), _ptr(blk_cells, torch.int32, "blk_cells"),
        int(pooled.shape[0]), _ptr(seq_blk_offs, torch.int64, "seq_blk_off"),
        _ptr(seq_blk_slots, torch.int32, "seq_blk_slots"), int(seq_blk_offs.numel()) - 1,
        int(max_blocks), _io(q, torch.float16, "q"), _ptr(k_cache, None, "k_cache"),
        _ptr(v_cache, None, "v_cache"), int(n_cells), _ptr(cells, torch.int32, "cells"),
        _ptr(count, torch.int32, "count"), _io(out, torch.float32, "out"), rec_ptr, rec_n,
        _attn_flags(in_cluster, union),
        _ptr(workspace, torch.uint8, "workspace"), int(workspace.numel()), _stream(stream))
    _check(st, "qsa_index_attn")


def _attn_flags(in_cluster: bool, union: bool) -> int:
    return (QSA_INDEX_ATTN_IN_CLUSTER if in_cluster else 0) | (QSA_INDEX_ATTN_UNION if union else 0)


def index_attn_kernels(cfg, n_tokens: int, n_seq: int, max_blocks: int, in_cluster: bool = False,
                       union: bool = False) -> list:
    """Names of the kernels one index_attn call launches on the current device."""
    m = int(lib().qsa_index_attn_kernels(ctypes.byref(cfg), int(n_tokens), int(n_seq), int(max_blocks),
                                         _attn_flags(in_cluster, union)))
    return [k for k, v in KERNELS.items() if (m >> v) & 1]


def sparse_attn_workspace_size(cfg, n_tokens: int) -> int:
    return int(lib().qsa_sparse_attn_workspace_size(ctypes.byref(cfg), int(n_tokens)))


def sparse_attn(cfg, q, k_cache, v_cache, n_cells: int, cells, count, out, workspace=None, stream=None,
                union: bool = False):
    """qsa_sparse_attn (union: qsa_sparse_attn_union, token pairs over the
    union of their lists)."""
    import torch
    T = int(count.numel())
    ws_ptr = _ptr(workspace, torch.uint8, "workspace") if workspace is not None and workspace.numel() else None
    ws_len = int(workspace.numel()) if workspace is not None else 0
    name = "qsa_sparse_attn_union" if union else "qsa_sparse_attn"
    st = getattr(lib(), name)(
        ctypes.byref(cfg), T, _io(q, torch.float16, "q"), _ptr(k_cache, None, "k_cache"),
        _ptr(v_cache, None, "v_cache"), int(n_cells), _ptr(cells, torch.int32, "cells"),
        _ptr(count, torch.int32, "count"), _io(out, torch.float32, "out"),
        ws_ptr, ws_len, _stream(stream))
    _check(st, name)


def kv_append(cfg, tok_seq, tok_pos, cells, k_new, v_new, idx_new, k_cache, v_cache, idx_k, blk_cells,
              seq_blk_off, seq_blk_slots, dirty, slot_block_idx=None, norm_w=None, pooled=None, stream=None):
    """Write the step's new cells (K/V rows, indexer keys, block-table
    entries) and fill `dirty` with the slots of the blocks they change; with
    `pooled` (and slot_block_idx, norm_w) also re-pool those blocks."""
    import torch
    pool_args = (None, None, None)
    if pooled is not None:
        pool_args = (_ptr(slot_block_idx, torch.int32, "slot_block_idx"), _ptr(norm_w, torch.float32, "norm_w"),
                     _ptr(pooled, torch.float32, "pooled"))
    n_cells = int(idx_k.shape[0])
    st = lib().qsa_kv_append(
        ctypes.byref(cfg), int(tok_pos.numel()), _io(tok_seq, torch.int32, "tok_seq"),
        _io(tok_pos, torch.int32, "tok_pos"), _io(cells, torch.int32, "cells"),
        _io(k_new, torch.float16, "k_new"), _io(v_new, torch.float16, "v_new"),
        _io(idx_new, torch.float16, "idx_new"), _ptr(k_cache, None, "k_cache"), _ptr(v_cache, None, "v_cache"),
        _ptr(idx_k, torch.float16, "idx_k"), n_cells, _ptr(blk_cells, torch.int32, "blk_cells"),
        int(blk_cells.shape[0]), _ptr(seq_blk_off, torch.int64, "seq_blk_off"),
        _ptr(seq_blk_slots, torch.int32, "seq_blk_slots"), int(seq_blk_off.numel()) - 1,
        _ptr(dirty, torch.int32, "dirty"), int(dirty.numel()), *pool_args, _stream(stream))
    _check(st, "qsa_kv_append")


def blocks_dirty(old_tbl: np.ndarray, new_tbl: np.ndarray, pad_pow2_min: int = 4) -> np.ndarray:
    """Host helper: slots whose member cells differ, padded with -1 to a power
    of two >= pad_pow2_min."""
    old = np.ascontiguousarray(old_tbl, dtype=np.int32)
    new = np.ascontiguousarray(new_tbl, dtype=np.int32)
    if old.shape != new.shape or old.ndim != 2:
        raise ValueError("tables must have the same [n_slots][r] shape")
    n = _I32(0)
    L = lib()
    st = L.qsa_blocks_dirty(old.ctypes.data, new.ctypes.data, old.shape[0], old.shape[1], None, 0,
                            ctypes.byref(n), int(pad_pow2_min))
    if st not in (QSA_OK, -2):
        _check(st, "qsa_blocks_dirty")
    out = np.empty(max(n.value, 1), dtype=np.int32)
    _check(L.qsa_blocks_dirty(old.ctypes.data, new.ctypes.data, old.shape[0], old.shape[1],
                              out.ctypes.data, out.shape[0], ctypes.byref(n), int(pad_pow2_min)),
           "qsa_blocks_dirty")
    return out[:n.value]


def index_topk_kernels(n_tokens: int, n_seq: int) -> list:
    """Names of the kernels one index_topk call of n_tokens tokens over n_seq
    sequences launches (token-tiled scoring adds "hist")."""
    m = int(lib().qsa_index_topk_kernels(int(n_tokens), int(n_seq)))
    return [k for k, v in KERNELS.items() if (m >> v) & 1]


def profile_kernel(kernel: str, before=None, after=None):
    """Record torch.cuda.Event `before`/`after` around each launch of the
    named kernel (see KERNELS); None clears."""
    for ev in (before, after):
        if ev is not None and not ev.cuda_event:
            ev.record()   # torch creates the CUDA event on first record
    eb = before.cuda_event if before is not None else None
    ea = after.cuda_event if after is not None else None
    _check(lib().qsa_profile_kernel(KERNELS[kernel], eb, ea), "qsa_profile_kernel")


def debug_check(stream=None):
    """(status, flags): synchronises the stream and reads/clears the device
    error word of the current device."""
    f = ctypes.c_uint32(0)
    st = lib().qsa_debug_check(_stream(stream), ctypes.byref(f))
    return st, f.value
