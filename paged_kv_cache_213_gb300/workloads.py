"""Seeded synthetic inputs for paged decode attention.

This module builds inputs only: random fp16 values, sequence lengths, a
physical block pool in random order, per-sequence block tables (with shared
prefix blocks where a workload has them) and slot mappings for the one-token
append.  It holds none of the attention arithmetic.  The CUDA path and the
CPU oracle both take their inputs from here and from nowhere else.

The five standard workloads are shaped like the decode batches the serving
pages talk about (LLaMA-3-8B, Mistral-7B and LLaMA-3-70B attention layers,
block size 16, fp16 K/V, values drawn from N(0, 1)):

  1  tiny        B=4,   4/2 heads,  d=64,  L~U{1..64}, 64-block pool, append
  2  llama3-8b   B=32,  32/8 heads, d=128, L~U{128..2048}, pool +10 %, append
  3  mix         B=128, 32/8 heads, d=128, L log-uniform [16, 4096],
                 one 512-token prefix (32 blocks) in every block table
  4  long        B=8,   32/8 heads, d=128, L=32768, pool +10 %
  5  llama3-70b  B=64 = 16 prompts x 4 completions, 64/8 heads, d=128,
                 L=4000: 248 prefix blocks shared by the 4 completions of a
                 prompt, then 2 private blocks per completion

Seeds are 20260 + workload number.  "poison" fills every cache row that no
sequence may read (rows past a sequence's length inside its last block, free
blocks, the slot about to be appended) with an fp16 NaN, and every unused
block-table entry with an id outside the pool, so that a kernel that touches
them shows it.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

F16_NAN_BITS = 0x7E00
SEED_BASE = 20260


@dataclass
class PagedBatch:
    name: str
    q: np.ndarray              # fp16 [B, H, d]
    k_cache: np.ndarray        # fp16 [NB, Hk, bs, d]  (before the append, if any)
    v_cache: np.ndarray        # fp16 [NB, Hk, bs, d]
    block_tables: np.ndarray   # int32 [B, MB]
    context_lens: np.ndarray   # int32 [B]  (includes the appended token)
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    block_size: int
    scale: float
    k_new: np.ndarray | None = None        # fp16 [B, Hk, d]
    v_new: np.ndarray | None = None
    slot_mapping: np.ndarray | None = None  # int64 [B]
    unique_blocks: int = 0                  # physical blocks referenced by some table
    meta: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_blocks(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.context_lens.size else 0

    @property
    def has_append(self) -> bool:
        return self.slot_mapping is not None


def _randn16(rng, shape):
    return rng.standard_normal(shape, dtype=np.float32).astype(np.float16)


def make_batch(name, lens, n_q_heads, n_kv_heads, head_dim, block_size, rng, *,
               scale=None, pool_blocks=None, pool_extra=0.10, shared=None, append=True,
               poison=True, max_blocks_per_seq=None, append_padding=0,
               physical_order="random"):
    """Build one batch.

    lens: attention length per sequence (the appended token included).
    shared: list of (member sequence ids, number of leading logical blocks the
      members share).  Each group gets its own physical blocks; a member whose
      own block count is smaller uses only the first ones.
    pool_blocks: pool size; default = blocks referenced + ceil(pool_extra * that).
    append: also build k_new / v_new / slot_mapping for one new token per
      sequence, written at position L-1 (that cache row holds poison or noise).
    append_padding: number of extra padding tokens (slot -1) in the append.
    physical_order: "random" (a random permutation of the pool) or "identity"
      (blocks laid out in logical order, for comparisons of access patterns).
    """
    lens = np.asarray(lens, dtype=np.int64)
    B = len(lens)
    bs = block_size
    nblk = [(int(L) + bs - 1) // bs for L in lens]
    MB = max_blocks_per_seq or max(1, max(nblk) if nblk else 1)
    if any(n > MB for n in nblk):
        raise ValueError("max_blocks_per_seq too small")

    # logical -> unique-block key; shared groups first
    owner = {}
    keys = []                       # one entry per unique physical block
    table_keys = [[None] * n for n in nblk]
    for g, (members, n_shared) in enumerate(shared or []):
        for lb in range(n_shared):
            users = [b for b in members if lb < nblk[b]]
            if not users:
                continue
            key = ("shared", g, lb)
            owner[key] = len(keys)
            keys.append(key)
            for b in users:
                table_keys[b][lb] = key
    for b in range(B):
        for lb in range(nblk[b]):
            if table_keys[b][lb] is None:
                key = ("private", b, lb)
                owner[key] = len(keys)
                keys.append(key)
                table_keys[b][lb] = key
    used = len(keys)
    NB = pool_blocks if pool_blocks is not None else used + int(math.ceil(pool_extra * used))
    if NB < used:
        raise ValueError("pool too small")
    if physical_order == "identity":
        perm = np.arange(NB, dtype=np.int32)
    else:
        perm = rng.permutation(NB).astype(np.int32)
    phys_of = perm[:used]           # k-th unique block -> physical id

    bt = np.empty((B, MB), dtype=np.int32)
    if poison:
        bt[:] = rng.integers(NB, NB + 1_000_000, size=(B, MB), dtype=np.int32)
        bt[:, ::2] = -1 - bt[:, ::2] % 1000
    else:
        bt[:] = -1
    for b in range(B):
        for lb in range(nblk[b]):
            bt[b, lb] = phys_of[owner[table_keys[b][lb]]]

    Hk, d = n_kv_heads, head_dim
    k_cache = _randn16(rng, (NB, Hk, bs, d))
    v_cache = _randn16(rng, (NB, Hk, bs, d))
    # a shared block is one physical block: every member sees the same rows
    if poison:
        valid = np.zeros((NB, bs), dtype=bool)
        for b in range(B):
            L = int(lens[b])
            readable = L - 1 if append else L   # the append target is not yet written
            t = np.arange(readable)
            valid[bt[b, t // bs], t % bs] = True
        kb = k_cache.view(np.uint16)
        vb = v_cache.view(np.uint16)
        inv = ~valid
        kb.transpose(0, 2, 1, 3)[inv] = F16_NAN_BITS
        vb.transpose(0, 2, 1, 3)[inv] = F16_NAN_BITS

    H = n_q_heads
    q = _randn16(rng, (B, H, d))
    batch = PagedBatch(name=name, q=q, k_cache=k_cache, v_cache=v_cache, block_tables=bt,
                       context_lens=lens.astype(np.int32), n_q_heads=H, n_kv_heads=Hk,
                       head_dim=d, block_size=bs,
                       scale=float(scale if scale is not None else 1.0 / math.sqrt(d)),
                       unique_blocks=used)
    if append:
        if np.any(lens < 1):
            raise ValueError("append needs L >= 1")
        T = B + append_padding
        batch.k_new = _randn16(rng, (T, Hk, d))
        batch.v_new = _randn16(rng, (T, Hk, d))
        slots = np.full(T, -1, dtype=np.int64)
        for b in range(B):
            pos = int(lens[b]) - 1
            slots[b] = int(bt[b, pos // bs]) * bs + pos % bs
        if append_padding:
            order = rng.permutation(T)
            batch.k_new = batch.k_new[order].copy()
            batch.v_new = batch.v_new[order].copy()
            slots = slots[order].copy()
            batch.meta["append_order"] = order
        batch.slot_mapping = slots
    batch.meta["shared"] = shared or []
    return batch


WORKLOADS = {
    1: "tiny paged decode: B=4, 4/2 heads, d=64, bs=16, L~U{1..64}, 64-block pool, append+attend",
    2: "LLaMA-3-8B-shaped layer: B=32, 32/8 heads, d=128, bs=16, L~U{128..2048}, pool +10%, "
       "append+attend",
    3: "continuous-batching mix (Mistral-7B shape): B=128, 32/8 heads, d=128, bs=16, "
       "L log-uniform [16,4096], shared 512-token prefix in every table",
    4: "long-context split-K: B=8, 32/8 heads, d=128, bs=16, L=32768",
    5: "LLaMA-3-70B-shaped parallel sampling: 16 prompts x 4 completions (B=64), 64/8 heads, "
       "d=128, bs=16, L=4000, 248 prefix blocks shared per prompt + 2 private",
}


def workload(i: int, poison: bool = False, seed: int | None = None) -> PagedBatch:
    """One of the five standard workloads (see the module docstring)."""
    rng = np.random.default_rng(SEED_BASE + i if seed is None else seed)
    if i == 1:
        lens = rng.integers(1, 65, size=4)
        return make_batch("tiny", lens, 4, 2, 64, 16, rng, scale=1.0 / 8.0, pool_blocks=64,
                          append=True, poison=poison, max_blocks_per_seq=4)
    if i == 2:
        lens = rng.integers(128, 2049, size=32)
        return make_batch("llama3-8b", lens, 32, 8, 128, 16, rng, append=True, poison=poison)
    if i == 3:
        u = rng.uniform(math.log(16), math.log(4096), size=128)
        lens = np.clip(np.floor(np.exp(u)), 16, 4096).astype(np.int64)
        return make_batch("mix", lens, 32, 8, 128, 16, rng, append=False, poison=poison,
                          shared=[(list(range(128)), 32)])
    if i == 4:
        lens = np.full(8, 32768)
        return make_batch("long", lens, 32, 8, 128, 16, rng, append=False, poison=poison)
    if i == 5:
        lens = np.full(64, 4000)
        groups = [(list(range(4 * p, 4 * p + 4)), 248) for p in range(16)]
        return make_batch("llama3-70b", lens, 64, 8, 128, 16, rng, append=False, poison=poison,
                          shared=groups)
    raise ValueError(f"unknown workload {i}")


def stats(batch: PagedBatch, kv_bytes: int = 2) -> dict:
    """Byte counts of one decode step (element counts times element sizes).

    unique_kv: K+V bytes of every (physical block, KV head) row some sequence
      reads, each counted once -- what the step must move from HBM.
    logical_kv: K+V bytes gathered per sequence, sum over sequences.
    kv_bytes: bytes per cached value (2 for fp16, 1 for E4M3 codes); the
      append reads fp16 k_new / v_new and writes kv_bytes per value.
    """
    bs, d, Hk = batch.block_size, batch.head_dim, batch.n_kv_heads
    rows = set()
    for b in range(batch.num_seqs):
        L = int(batch.context_lens[b])
        for lb in range((L + bs - 1) // bs):
            n = min(bs, L - lb * bs)
            rows.add((int(batch.block_tables[b, lb]), n))
    # a block read by several sequences is counted once, with its longest reach
    reach = {}
    for blk, n in rows:
        reach[blk] = max(reach.get(blk, 0), n)
    unique_tokens = sum(reach.values())
    logical_tokens = int(batch.context_lens.astype(np.int64).sum())
    per_token = 2 * Hk * d * kv_bytes
    B, H = batch.num_seqs, batch.n_q_heads
    qo = 2 * B * H * d * 2
    meta = batch.block_tables.nbytes + batch.context_lens.nbytes
    app = 0
    if batch.has_append:
        new_bytes = batch.k_new.nbytes + batch.v_new.nbytes
        app = new_bytes + new_bytes * kv_bytes // 2 + batch.slot_mapping.nbytes
    return {
        "unique_kv": unique_tokens * per_token,
        "logical_kv": logical_tokens * per_token,
        "qo": qo,
        "meta": meta,
        "append": app,
        "step_unique": unique_tokens * per_token + qo + meta + app,
        "step_logical": logical_tokens * per_token + qo + meta + app,
    }


def prefix_groups(batch: PagedBatch):
    """Consecutive-range groups of the batch's shared prefixes, for the
    prefix-shared entry point: (offsets int32 [G+1], prefix tokens int32 [G],
    largest group, longest prefix).  Sequences outside any shared group form
    one-sequence groups with prefix 0."""
    B = batch.num_seqs
    member_of = {}
    for members, n_shared in batch.meta.get("shared", []):
        ms = sorted(members)
        if ms != list(range(ms[0], ms[0] + len(ms))):
            raise ValueError("shared groups must be consecutive sequences")
        for b in ms:
            member_of[b] = (ms[0], len(ms), n_shared * batch.block_size)
    offsets, prefix = [0], []
    b = 0
    while b < B:
        if b in member_of:
            first, n, tokens = member_of[b]
            offsets.append(first + n)
            prefix.append(tokens)
            b = first + n
        else:
            offsets.append(b + 1)
            prefix.append(0)
            b += 1
    sizes = np.diff(offsets)
    return (np.asarray(offsets, dtype=np.int32), np.asarray(prefix, dtype=np.int32),
            int(sizes.max()) if sizes.size else 0, int(max(prefix) if prefix else 0))
