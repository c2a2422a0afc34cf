"""bench.py's back-to-back timing runs each layer-step on one of several
copies of the layer's state: the copies must own their caches, keys, table,
pooled keys, outputs and workspaces (so no step finds another copy's rows in
L2 and no step overwrites another copy's state), and the copy count must put
more than 3x the L2 between two steps of one copy.  Checked on CPU tensors
(no kernel runs)."""
import numpy as np
import pytest

import bench
from qsa_workload import make_workload
from sparse_attention_long_qsa_gb300 import build as qbuild
from sparse_attention_long_qsa_gb300.layer import QSALayer

OWN = ("idx_k", "k_cache", "v_cache", "blk_cells", "pooled", "cells", "count", "out", "ws_index", "ws_attn")
SHARED = ("slot_block_idx", "seq_blk_off", "seq_blk_slots", "norm_w")


@pytest.fixture(scope="module")
def layer():
    qbuild.build()
    wl = make_workload(n_seq=2, prompt_len=[1_001, 2_003], n_steps=2, seed=5)
    return wl, QSALayer.from_workload(wl, 0, device="cpu")


def test_clone_owns_its_state(layer):
    _, L = layer
    C = bench.clone_layer(L)
    for k in OWN:
        a, b = getattr(L, k), getattr(C, k)
        assert a.numel() == 0 or a.data_ptr() != b.data_ptr(), k   # (the attention needs no workspace)
        assert a.shape == b.shape and a.dtype == b.dtype and bool((a == b).all()), k
    for k in SHARED:
        assert getattr(L, k).data_ptr() == getattr(C, k).data_ptr(), k
    C.pooled.add_(1.0)
    C.blk_cells[0, 0] = -7
    assert not bool((L.pooled == C.pooled).all()) and int(L.blk_cells[0, 0]) != -7


def test_copy_count():
    """50k, 250k q8_0 and 5x250k q8_0 step and state sizes: > 3x L2 between
    two steps of one copy; the memory cap and the floor of 2 apply."""
    for step, state in ((10.9e6, 122e6), (35.3e6, 369e6), (176.5e6, 1847e6), (2.6e9, 610e6)):
        n = bench.chain_layers(step, state)
        assert 2 <= n <= 64 and n * state <= bench.CHAIN_MEM_BYTES
        assert n == 2 or (n - 1) * step > 3 * bench.L2_BYTES
    assert bench.chain_layers(10.9e6, 122e6) == 37
    assert bench.chain_layers(1e3, 1e6) == 64                       # tiny steps: capped
    assert bench.chain_layers(1e6, 40e9) == 2                       # huge state: floor
