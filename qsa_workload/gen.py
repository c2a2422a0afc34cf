"""Seeded synthetic workloads (inputs only, no arithmetic of the step).

Shapes follow the qwen4exp QSA layer described in llama.cpp issue #28734
("decode slows linearly with context"), fix summary: 16 query heads over 2 KV
heads, head dim 256, indexer 4 heads x 128 dims, compress_ratio r = 4,
indexer top_k = 2048 cells.  Depths, slot counts and the 512-token ubatch are
the ones the llama.cpp-multigpu README (section 1) measures at.

Layouts (shared by every consumer):
  idx_k      fp16  [n_cells][idx_dim]                  per-cell indexer key
  k/v cache  fp16  [n_cells][n_kv_heads][head_dim]     (kv_type "f16")
             q8_0  bytes: qs int8 [n_cells][G][D] then d fp16 [n_cells][G][D/32]
  blk_cells  int32 [n_slots][r]   cell of position j*r+i of the slot's block, -1 = absent
  slot_block_idx int32 [n_slots]  block index j of the slot within its sequence
  seq_blk_off int64 [n_seq+1], seq_blk_slots int32: block j of seq s -> slot
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np

CONFIG_NAMES = ("tiny", "50k", "250k_q8", "250k_f16", "5x250k_q8", "prefill", "verify5_250k_q8",
                "prefill_corr", "verify5_250k_q8_corr")


def default_cfg(**over) -> dict:
    """Head shapes and hyper-parameters of the qwen4exp QSA layer."""
    cfg = dict(
        n_q_heads=16, n_kv_heads=2, head_dim=256,
        n_idx_heads=4, idx_dim=128,
        compress_ratio=4, top_k=2048,
        rope_theta=1.0e6, rms_eps=1.0e-6,
        attn_scale=1.0 / 16.0,
        kv_type="f16",
    )
    cfg.update(over)
    return cfg


def quantize_q8_0(x: np.ndarray):
    """q8_0 encoding of the last axis in blocks of 32: d = amax/127,
    q = round-half-away(x/d) clamped to +-127, d stored as fp16.

    Returns (qs int8 same shape as x, d fp16 with last axis D/32)."""
    x = np.asarray(x, dtype=np.float32)
    lead = x.shape[:-1]
    D = x.shape[-1]
    xb = x.reshape(*lead, D // 32, 32)
    amax = np.abs(xb).max(axis=-1)
    d = amax / np.float32(127.0)
    inv = np.zeros_like(d)
    nz = d > 0
    inv[nz] = np.float32(1.0) / d[nz]
    v = xb * inv[..., None]
    a = np.abs(v)
    m = np.trunc(a)
    m = m + (a - m >= np.float32(0.5))          # half away from zero; a - m is exact in float32
    q = np.clip(np.sign(v) * m, -127, 127).astype(np.int8)
    return q.reshape(x.shape), d.astype(np.float16)


@dataclasses.dataclass
class Step:
    """Inputs of one step: T query tokens."""
    tok_seq: np.ndarray      # int32 [T]
    tok_pos: np.ndarray      # int32 [T] position p_t of the token (its own cell is present)
    q: np.ndarray            # fp16 [T][Hq][D]
    q_idx: np.ndarray        # fp32 [T][HI][DI]
    w_idx: np.ndarray        # fp32 [T][HI]
    dirty: np.ndarray        # int32 [pow2 >= 4] slots whose blocks gained cells, -1 = no-op
    new_pos: List[np.ndarray]  # per seq: positions appended by this step
    cells: np.ndarray = None   # int32 [T] the cell each token's own (new) position occupies
    k_new: np.ndarray = None   # fp16 [T][G][D] K row of that cell before any cache encoding
    v_new: np.ndarray = None   # fp16 [T][G][D]
    idx_new: np.ndarray = None  # fp16 [T][DI] its indexer key


@dataclasses.dataclass
class Workload:
    name: str
    cfg: dict
    n_seq: int
    n_cells: int
    idx_k: np.ndarray                # fp16 [n_cells][DI]
    k_cache: np.ndarray              # fp16 [n][G][D] or uint8 q8_0 bytes
    v_cache: np.ndarray
    seq_cells: List[np.ndarray]      # per seq: int32 cell of each position (all steps)
    prompt_len: List[int]
    n_slots: int
    slot_block_idx: np.ndarray       # int32 [n_slots]
    slot_seq: np.ndarray             # int32 [n_slots]
    seq_blk_off: np.ndarray          # int64 [n_seq+1]
    seq_blk_slots: np.ndarray        # int32
    norm_w: np.ndarray               # fp32 [DI]
    steps: List[Step]
    seed: int

    @property
    def r(self) -> int:
        return self.cfg["compress_ratio"]

    def max_blocks(self) -> int:
        """Upper bound on the full blocks any token of any step scores."""
        m = 0
        for st in self.steps:
            m = max(m, int(((st.tok_pos.astype(np.int64) + 1) // self.r).max()))
        return m

    def seq_len_after(self, step: int) -> List[int]:
        """Positions present per sequence after steps[0..step) were appended."""
        out = list(self.prompt_len)
        for st in self.steps[:step]:
            for s, ps in enumerate(st.new_pos):
                if len(ps):
                    out[s] = max(out[s], int(ps.max()) + 1)
        return out

    def blk_cells_state(self, step: int) -> np.ndarray:
        """Block table with every position of the prompt and of steps[0..step)
        present (step = 0: prompt only; step = i: state in which step i-1's
        tokens attend)."""
        r = self.r
        tbl = np.full((self.n_slots, r), -1, dtype=np.int32)
        lens = self.seq_len_after(step)
        for s in range(self.n_seq):
            L = lens[s]
            if L == 0:
                continue
            off = int(self.seq_blk_off[s])
            nb = -(-L // r)
            slots = self.seq_blk_slots[off:off + nb]
            cells = np.full(nb * r, -1, dtype=np.int32)
            cells[:L] = self.seq_cells[s][:L]
            tbl[slots] = cells.reshape(nb, r)
        return tbl

    def prompt_dirty(self) -> np.ndarray:
        """Every slot holding at least one prompt position (pooled-cache warm-up)."""
        r = self.r
        out = []
        for s in range(self.n_seq):
            nb = -(-self.prompt_len[s] // r)
            off = int(self.seq_blk_off[s])
            out.append(self.seq_blk_slots[off:off + nb])
        return np.sort(np.concatenate(out)).astype(np.int32)


def _pad_pow2(x: np.ndarray, minimum: int = 4) -> np.ndarray:
    n = max(minimum, 1)
    while n < len(x):
        n *= 2
    out = np.full(n, -1, dtype=np.int32)
    out[:len(x)] = x
    return out


def _normal_f16(rng, shape, chunk_rows=65536):
    out = np.empty(shape, dtype=np.float16)
    n = shape[0]
    for a in range(0, n, chunk_rows):
        b = min(n, a + chunk_rows)
        out[a:b] = rng.standard_normal((b - a,) + tuple(shape[1:]), dtype=np.float32)
    return out


def _normal_q8_0(rng, n_cells, G, D, keep=None, chunk_rows=65536):
    """q8_0 cache bytes of N(0,1) rows rounded to fp16 (the K/V precision a
    model writes), and the fp16 rows of the sorted cells `keep` (the cells
    appended by the steps, so that an append can be fed the same rows)."""
    qs = np.empty((n_cells, G, D), dtype=np.int8)
    d = np.empty((n_cells, G, D // 32), dtype=np.float16)
    kept = np.empty((0 if keep is None else len(keep), G, D), dtype=np.float16)
    for a in range(0, n_cells, chunk_rows):
        b = min(n_cells, a + chunk_rows)
        x = rng.standard_normal((b - a, G, D), dtype=np.float32).astype(np.float16)
        qs[a:b], d[a:b] = quantize_q8_0(x.astype(np.float32))
        if keep is not None:
            lo, hi = np.searchsorted(keep, [a, b])
            kept[lo:hi] = x[keep[lo:hi] - a]
    return np.concatenate([qs.reshape(-1).view(np.uint8), d.reshape(-1).view(np.uint8)]), kept


PRESETS = {
    # name: (n_seq, prompt_len, n_steps, tokens_per_step, kv_type)
    "tiny": (1, 4095, 1, 1, "f16"),
    "50k": (1, 50_000, 128, 1, "f16"),
    "250k_q8": (1, 250_000, 128, 1, "q8_0"),
    # the same depth with fp16 K/V (attention time flat in n_kv: compare with 50k)
    "250k_f16": (1, 250_000, 128, 1, "f16"),
    "5x250k_q8": (5, 250_000, 128, 1, "q8_0"),
    "prefill": (1, 250_000, 1, 512, "f16"),
    # speculative verify batch: 5 consecutive query tokens of one sequence per step
    "verify5_250k_q8": (1, 250_000, 128, 5, "q8_0"),
    # the same two batches with the indexer queries of a sequence's tokens
    # correlated (idx_corr below), so consecutive tokens choose overlapping blocks
    "prefill_corr": (1, 250_000, 1, 512, "f16", 0.98),
    "verify5_250k_q8_corr": (1, 250_000, 128, 5, "q8_0", 0.98),
}


def make_workload(name: str = "custom", *, n_seq: Optional[int] = None,
                  prompt_len=None, n_steps: Optional[int] = None,
                  tokens_per_step: Optional[int] = None,
                  kv_type: Optional[str] = None, seed: int = 0,
                  shuffled: bool = False, cfg: Optional[dict] = None,
                  idx_corr: Optional[float] = None) -> Workload:
    """Build a workload.  Named presets: tiny, 50k, 250k_q8, 5x250k_q8, prefill, verify5_250k_q8.

    Decode (tokens_per_step == 1): every step appends one position to each
    sequence and queries it; n_seq tokens per step.  Prefill or verify
    (tokens_per_step > 1): every step appends tokens_per_step consecutive
    positions to each sequence and queries all of them (tokens ordered by
    sequence, then position).

    Cells: prompts occupy contiguous cell ranges (sequence-major), decode cells
    are appended interleaved across sequences; shuffled=True permutes all cells
    and all slots.  Slots: prompt blocks sequence-major, later blocks in order
    of first appearance.

    idx_corr = rho > 0: within a step, the tokens of one sequence share their
    indexer weights w_idx (the sequence's first token's draw) and their
    indexer queries are sqrt(1 - rho^2) z_t + rho z_seq with z_t, z_seq
    N(0,1), drawn after the independent draws (rho = 0 leaves every array
    as it was)."""
    if name in PRESETS:
        p = PRESETS[name]
        n_seq = p[0] if n_seq is None else n_seq
        prompt_len = p[1] if prompt_len is None else prompt_len
        n_steps = p[2] if n_steps is None else n_steps
        tokens_per_step = p[3] if tokens_per_step is None else tokens_per_step
        kv_type = p[4] if kv_type is None else kv_type
        if idx_corr is None and len(p) > 5:
            idx_corr = p[5]
    idx_corr = 0.0 if idx_corr is None else float(idx_corr)
    assert 0.0 <= idx_corr < 1.0
    n_seq = 1 if n_seq is None else n_seq
    n_steps = 1 if n_steps is None else n_steps
    tokens_per_step = 1 if tokens_per_step is None else tokens_per_step
    kv_type = "f16" if kv_type is None else kv_type
    if prompt_len is None:
        prompt_len = 4096
    if np.isscalar(prompt_len):
        prompt_len = [int(prompt_len)] * n_seq
    prompt_len = [int(x) for x in prompt_len]
    assert len(prompt_len) == n_seq

    c = default_cfg(kv_type=kv_type, **(cfg or {}))
    r = c["compress_ratio"]
    G, D, DI = c["n_kv_heads"], c["head_dim"], c["idx_dim"]
    Hq, HI = c["n_q_heads"], c["n_idx_heads"]

    ss = np.random.SeedSequence(seed)
    s_cells, s_idx, s_k, s_v, s_perm = ss.spawn(5)

    # ---- positions appended per step
    step_pos = []   # per step: list over seqs of appended positions
    lens = list(prompt_len)
    for i in range(n_steps):
        per = []
        for s in range(n_seq):
            per.append(np.arange(lens[s], lens[s] + tokens_per_step, dtype=np.int64))
            lens[s] += tokens_per_step
        step_pos.append(per)
    final_len = lens

    # ---- cells
    n_prompt = sum(prompt_len)
    n_cells = sum(final_len)
    seq_cells = []
    base = 0
    for s in range(n_seq):
        seq_cells.append(np.empty(final_len[s], dtype=np.int64))
        seq_cells[s][:prompt_len[s]] = base + np.arange(prompt_len[s])
        base += prompt_len[s]
    nxt = n_prompt
    for i in range(n_steps):
        for k in range(tokens_per_step):
            for s in range(n_seq):
                seq_cells[s][prompt_len[s] + i * tokens_per_step + k] = nxt
                nxt += 1
    assert nxt == n_cells
    if shuffled:
        perm = np.random.default_rng(s_perm).permutation(n_cells)
        seq_cells = [perm[x] for x in seq_cells]
    seq_cells = [x.astype(np.int32) for x in seq_cells]

    # ---- slots
    nb_prompt = [-(-L // r) for L in prompt_len]
    nb_final = [-(-L // r) for L in final_len]
    seq_slots = [np.full(nb_final[s], -1, dtype=np.int64) for s in range(n_seq)]
    nxt = 0
    for s in range(n_seq):
        seq_slots[s][:nb_prompt[s]] = nxt + np.arange(nb_prompt[s])
        nxt += nb_prompt[s]
    for i in range(n_steps):
        for s in range(n_seq):
            for pos in step_pos[i][s]:
                j = int(pos) // r
                if seq_slots[s][j] < 0:
                    seq_slots[s][j] = nxt
                    nxt += 1
    n_slots = nxt
    if shuffled:
        sperm = np.random.default_rng(s_perm.spawn(1)[0]).permutation(n_slots)
        seq_slots = [sperm[x] for x in seq_slots]
    slot_block_idx = np.zeros(n_slots, dtype=np.int32)
    slot_seq = np.zeros(n_slots, dtype=np.int32)
    for s in range(n_seq):
        slot_block_idx[seq_slots[s]] = np.arange(nb_final[s])
        slot_seq[seq_slots[s]] = s
    seq_blk_off = np.zeros(n_seq + 1, dtype=np.int64)
    seq_blk_off[1:] = np.cumsum(nb_final)
    seq_blk_slots = np.concatenate(seq_slots).astype(np.int32)

    # ---- per-cell data
    step_cells = [np.concatenate([seq_cells[s][step_pos[i][s]] for s in range(n_seq)]).astype(np.int64)
                  for i in range(n_steps)]
    new_cells = np.unique(np.concatenate(step_cells)) if n_steps else np.zeros(0, np.int64)
    idx_k = _normal_f16(np.random.default_rng(s_idx), (n_cells, DI))
    if kv_type == "f16":
        k_cache = _normal_f16(np.random.default_rng(s_k), (n_cells, G, D))
        v_cache = _normal_f16(np.random.default_rng(s_v), (n_cells, G, D))
        k_src, v_src = k_cache[new_cells], v_cache[new_cells]
    elif kv_type == "q8_0":
        k_cache, k_src = _normal_q8_0(np.random.default_rng(s_k), n_cells, G, D, keep=new_cells)
        v_cache, v_src = _normal_q8_0(np.random.default_rng(s_v), n_cells, G, D, keep=new_cells)
    else:
        raise ValueError(kv_type)

    # ---- steps
    steps = []
    for i in range(n_steps):
        rng = np.random.default_rng([seed, 7919, i])
        tok_seq = np.concatenate([np.full(len(step_pos[i][s]), s) for s in range(n_seq)]).astype(np.int32)
        tok_pos = np.concatenate(step_pos[i]).astype(np.int32)
        T = len(tok_pos)
        q = rng.standard_normal((T, Hq, D), dtype=np.float32).astype(np.float16)
        q_idx = rng.standard_normal((T, HI, DI), dtype=np.float32)
        w_idx = rng.random((T, HI), dtype=np.float32)
        if idx_corr > 0.0:
            z_seq = rng.standard_normal((n_seq, HI, DI), dtype=np.float32)
            q_idx = (np.float32(np.sqrt(1.0 - idx_corr ** 2)) * q_idx +
                     np.float32(idx_corr) * z_seq[tok_seq]).astype(np.float32)
            first = np.searchsorted(tok_seq, tok_seq)   # tokens are ordered by sequence
            w_idx = w_idx[first]
        dslots = sorted({int(seq_slots[s][int(p) // r]) for s in range(n_seq) for p in step_pos[i][s]})
        dirty = _pad_pow2(np.array(dslots, dtype=np.int32), 4)
        at = np.searchsorted(new_cells, step_cells[i])
        steps.append(Step(tok_seq, tok_pos, q, q_idx, w_idx, dirty,
                          [x.astype(np.int32) for x in step_pos[i]],
                          cells=step_cells[i].astype(np.int32), k_new=k_src[at], v_new=v_src[at],
                          idx_new=idx_k[step_cells[i]]))

    return Workload(
        name=name, cfg=c, n_seq=n_seq, n_cells=n_cells, idx_k=idx_k,
        k_cache=k_cache, v_cache=v_cache, seq_cells=seq_cells,
        prompt_len=prompt_len, n_slots=n_slots, slot_block_idx=slot_block_idx,
        slot_seq=slot_seq, seq_blk_off=seq_blk_off, seq_blk_slots=seq_blk_slots,
        norm_w=np.ones(DI, dtype=np.float32), steps=steps, seed=seed)
