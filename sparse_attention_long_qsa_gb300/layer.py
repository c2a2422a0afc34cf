"""Device-resident state of one QSA layer and its step.

QSALayer owns the caller-side buffers of include/qsa.h (caches, block tables,
the pooled block-key cache, workspaces, outputs) as torch CUDA tensors and
runs a step as the C-ABI calls on one stream:

    step:       pool_update(dirty) -> index_topk(tokens) -> sparse_attn(tokens)
    full_step:  kv_append(new cells, re-pooling the blocks they dirty) ->
                index_attn(tokens)  (index top-k and sparse attention in one call)

It holds no arithmetic of its own.
"""
from __future__ import annotations

import contextlib
from typing import Optional

import numpy as np
import torch

from . import qsa


def _dev(x, dtype=None, device="cuda"):
    t = torch.from_numpy(np.ascontiguousarray(x))
    if dtype is not None:
        t = t.to(dtype)
    return t.to(device)


class QSALayer:
    def __init__(self, cfg: dict, idx_k, k_cache, v_cache, n_cells: int, blk_cells, slot_block_idx,
                 seq_blk_off, seq_blk_slots, norm_w, max_blocks: int, max_tokens: int,
                 device: str = "cuda"):
        self.cfgd = dict(cfg)
        self.cfg = qsa.config_from_dict(cfg)
        self.device = device
        self.n_cells = int(n_cells)
        self.max_blocks = max(int(max_blocks), 1)
        self.max_tokens = int(max_tokens)
        self.idx_k = _dev(idx_k, device=device)
        kv_dtype = torch.float16 if cfg["kv_type"] == "f16" else torch.uint8
        self.k_cache = _dev(k_cache, device=device).view(kv_dtype)
        self.v_cache = _dev(v_cache, device=device).view(kv_dtype)
        self.blk_cells = _dev(blk_cells, device=device)
        self.slot_block_idx = _dev(slot_block_idx, device=device)
        self.seq_blk_off = _dev(seq_blk_off, device=device)
        self.seq_blk_slots = _dev(seq_blk_slots, device=device)
        self.norm_w = _dev(norm_w, device=device)
        self.n_slots = int(self.blk_cells.shape[0])
        self.pooled = torch.zeros((self.n_slots, cfg["idx_dim"]), dtype=torch.float32, device=device)
        self.pitch = qsa.cells_per_token(self.cfg)
        T = self.max_tokens
        self.cells = torch.full((T, self.pitch), -1, dtype=torch.int32, device=device)
        self.count = torch.zeros(T, dtype=torch.int32, device=device)
        self.out = torch.zeros((T, cfg["n_q_heads"], cfg["head_dim"]), dtype=torch.float32, device=device)
        # zero-filled once; the library leaves its control words zero after every call
        self.ws_index = torch.zeros(qsa.index_topk_workspace_size(self.cfg, T, self.max_blocks),
                                    dtype=torch.uint8, device=device)
        self.ws_attn = torch.empty(qsa.sparse_attn_workspace_size(self.cfg, T),
                                   dtype=torch.uint8, device=device)
        self._dirty = None

    @classmethod
    def from_workload(cls, wl, step: int = 0, max_tokens: Optional[int] = None, device="cuda"):
        """Upload a qsa_workload.Workload with the block table as it stands
        before steps[step] (that step's cells not yet appended)."""
        T = max_tokens or max(len(s.tok_pos) for s in wl.steps)
        return cls(wl.cfg, wl.idx_k, wl.k_cache, wl.v_cache, wl.n_cells, wl.blk_cells_state(step),
                   wl.slot_block_idx, wl.seq_blk_off, wl.seq_blk_slots, wl.norm_w,
                   wl.max_blocks(), T, device=device)

    # ---- the three calls
    def pool_update(self, dirty, stream=None):
        d = dirty if isinstance(dirty, torch.Tensor) else _dev(np.asarray(dirty, dtype=np.int32), device=self.device)
        qsa.pool_update(self.cfg, self.idx_k, self.blk_cells, self.slot_block_idx, d, self.norm_w,
                        self.pooled, stream)

    def index_topk(self, tok_seq, tok_pos, q_idx, w_idx, recomputed=None, stream=None):
        T = int(tok_pos.numel())
        qsa.index_topk(self.cfg, q_idx, w_idx, tok_seq, tok_pos, self.pooled, self.blk_cells,
                       self.seq_blk_off, self.seq_blk_slots, self.max_blocks, self.n_cells,
                       self.cells[:T], self.count[:T], self.ws_index, self.max_tokens,
                       recomputed, stream)

    def index_attn(self, tok_seq, tok_pos, q_idx, w_idx, q, recomputed=None, stream=None, in_cluster=False,
                   out=None, union=False):
        """index_topk then sparse_attn in one call (qsa_index_attn); out:
        where the attention output goes (default the layer's buffer; may be a
        pinned host tensor); union: token pairs attend over the union of
        their lists."""
        T = int(tok_pos.numel())
        qsa.index_attn(self.cfg, q_idx, w_idx, tok_seq, tok_pos, self.pooled, self.blk_cells,
                       self.seq_blk_off, self.seq_blk_slots, self.max_blocks, q, self.k_cache, self.v_cache,
                       self.n_cells, self.cells[:T], self.count[:T], self.out[:T] if out is None else out,
                       self.ws_index, self.max_tokens, recomputed, stream, in_cluster=in_cluster, union=union)

    def sparse_attn(self, q, n_tokens: int, stream=None, union=False):
        T = int(n_tokens)
        qsa.sparse_attn(self.cfg, q, self.k_cache, self.v_cache, self.n_cells, self.cells[:T],
                        self.count[:T], self.out[:T], self.ws_attn, stream, union=union)

    def step(self, tok_seq, tok_pos, q, q_idx, w_idx, dirty, stream=None):
        """One QSA step for T tokens; returns the out[:T] view (fp32)."""
        d = dirty if isinstance(dirty, torch.Tensor) else _dev(np.asarray(dirty, dtype=np.int32), device=self.device)
        self.pool_update(d, stream)
        self.index_topk(tok_seq, tok_pos, q_idx, w_idx, recomputed=d, stream=stream)
        self.sparse_attn(q, int(tok_pos.numel()), stream)
        return self.out[:int(tok_pos.numel())]

    def kv_append(self, tok_seq, tok_pos, cells, k_new, v_new, idx_new, stream=None, pool=False):
        """Write the step's new cells and build the dirty list on the device
        (with pool=True also re-pool the dirtied blocks in the same launch);
        returns the dirty-list view (padded to a power of two >= max(4, T))."""
        T = int(tok_pos.numel())
        nd = 4
        while nd < T:
            nd *= 2
        if self._dirty is None or self._dirty.numel() < nd:
            self._dirty = torch.full((max(nd, 4),), -1, dtype=torch.int32, device=self.device)
        d = self._dirty[:nd]
        extra = dict(slot_block_idx=self.slot_block_idx, norm_w=self.norm_w, pooled=self.pooled) if pool else {}
        qsa.kv_append(self.cfg, tok_seq, tok_pos, cells, k_new, v_new, idx_new, self.k_cache, self.v_cache,
                      self.idx_k, self.blk_cells, self.seq_blk_off, self.seq_blk_slots, d, stream=stream, **extra)
        return d

    def full_step(self, tok_seq, tok_pos, q, q_idx, w_idx, cells, k_new, v_new, idx_new, stream=None,
                  in_cluster=False, out=None, union=False, **_):
        """The whole layer step from the new tokens on: append of their cells
        (K/V, indexer keys, table, device dirty list) with the pool update of
        the blocks they dirty in the same launch, then index top-k and sparse
        attention in one qsa_index_attn call (in_cluster: the selection inside
        the attention clusters; union: token pairs over the union of their
        lists).  The step's inputs and `out` may be pinned
        host tensors.  Returns the output (fp32 [T][n_q_heads][head_dim])."""
        # the append re-pooled only the query tokens' own blocks: score work on
        # the other blocks may start before it finishes
        self.kv_append(tok_seq, tok_pos, cells, k_new, v_new, idx_new, stream, pool=True)
        self.index_attn(tok_seq, tok_pos, q_idx, w_idx, q, recomputed="query_blocks", stream=stream,
                        in_cluster=in_cluster, out=out, union=union)
        return self.out[:int(tok_pos.numel())] if out is None else out

    def set_cells(self, slots, rows):
        """Write block-table rows (the append of new cells), device side."""
        s = _dev(np.asarray(slots, dtype=np.int64), device=self.device)
        self.blk_cells[s] = _dev(np.asarray(rows, dtype=np.int32), device=self.device)

    def warm(self, dirty_all):
        """Pool every listed slot (cold start / rebuild from the key cache)."""
        self.pool_update(dirty_all)


def step_inputs(st, device="cuda", new_cells=False):
    """Device tensors of a qsa_workload.Step (with new_cells: also the
    step's own cells and their rows, the inputs of full_step)."""
    d = dict(tok_seq=_dev(st.tok_seq, device=device), tok_pos=_dev(st.tok_pos, device=device),
             q=_dev(st.q, device=device), q_idx=_dev(st.q_idx, device=device),
             w_idx=_dev(st.w_idx, device=device), dirty=_dev(st.dirty, device=device))
    if new_cells:
        d.update(cells=_dev(st.cells, device=device), k_new=_dev(st.k_new, device=device),
                 v_new=_dev(st.v_new, device=device), idx_new=_dev(st.idx_new, device=device))
    return d


class PackedInputs:
    """A step's input tensors laid out back to back (256-byte aligned) in one
    pinned host buffer and one device buffer, so that moving a step's inputs
    to the device is a single copy.  `views` are the device tensors to pass to
    the layer's calls; `pack` fills a pinned host buffer from host arrays and
    `host_views` gives the tensors of such a buffer, which the calls can also
    take directly (read in place over the host link)."""

    def __init__(self, fields: dict, device="cuda", pin=True):
        self.fields = {}
        off = 0
        for k, (shape, dtype) in fields.items():
            n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
            self.fields[k] = (off, tuple(shape), dtype, n)
            off += -(-n // 256) * 256
        self.nbytes = off
        self.pin = pin
        self.dev = torch.empty(max(off, 256), dtype=torch.uint8, device=device)
        self.views = {k: self.dev[o:o + n].view(dtype).view(shape) for k, (o, shape, dtype, n) in self.fields.items()}

    def pack(self, arrays: dict):
        """A (pinned) host buffer holding `arrays` (numpy, same shapes and
        dtypes as the fields) in this layout."""
        host = torch.zeros(max(self.nbytes, 256), dtype=torch.uint8)
        if self.pin:
            host = host.pin_memory()
        hv = host.numpy()
        for k, (o, shape, dtype, n) in self.fields.items():
            a = np.ascontiguousarray(arrays[k])
            if a.nbytes != n or tuple(a.shape) != shape:
                raise ValueError(f"{k}: expected {shape} ({n} bytes), got {a.shape} ({a.nbytes} bytes)")
            hv[o:o + n] = a.view(np.uint8).reshape(-1)
        return host

    def host_views(self, host):
        """Tensors of the fields of a pinned host buffer made by `pack`."""
        return {k: host[o:o + n].view(dtype).view(shape) for k, (o, shape, dtype, n) in self.fields.items()}

    def upload(self, host, stream=None):
        """One host-to-device copy of a packed step (asynchronous on `stream`,
        default the current stream)."""
        with torch.cuda.stream(stream) if stream is not None else contextlib.nullcontext():
            self.dev[:host.numel()].copy_(host, non_blocking=True)


def append_rows(wl, step: int):
    """Block-table rows changed by steps[step]: (slots, rows) of the state
    after the step's cells are appended (only the blocks the step touches)."""
    r = wl.r
    lens = wl.seq_len_after(step + 1)
    slots, rows = [], []
    for s, ps in enumerate(wl.steps[step].new_pos):
        if len(ps) == 0:
            continue
        off = int(wl.seq_blk_off[s])
        for j in sorted({int(p) // r for p in ps}):
            row = np.full(r, -1, dtype=np.int32)
            hi = min(lens[s], (j + 1) * r)
            row[:hi - j * r] = wl.seq_cells[s][j * r:hi]
            slots.append(int(wl.seq_blk_slots[off + j]))
            rows.append(row)
    return np.array(slots, dtype=np.int64), np.array(rows, dtype=np.int32).reshape(-1, r)
