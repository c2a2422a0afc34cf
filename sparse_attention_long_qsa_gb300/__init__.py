"""QSA sparse-attention step for GB300 (sm_103a): Python binding of libqsa.

    from sparse_attention_long_qsa_gb300 import qsa
    cfg = qsa.config(kv_type="q8_0")
    qsa.pool_update(cfg, ...); qsa.index_topk(cfg, ...); qsa.sparse_attn(cfg, ...)

The computation lives in the CUDA library (csrc/, C ABI in include/qsa.h);
this package only marshals torch tensors into its calls.
"""
from . import qsa  # noqa: F401
from .qsa import QSAError, config  # noqa: F401
