"""Seeded synthetic inputs for the paged decode path.

This module only draws inputs: context lengths, a shuffled assignment of physical
blocks, N(0,1) bf16 values, the new token's slot, and copy-on-write block pairs.  It
holds none of the attention arithmetic and imports neither the CUDA binding nor the
oracle, so both sides of a parity test read the same bytes from it.

Recipe (every draw is seeded; structure comes from numpy's PCG64, values from a torch
generator on the requested device):

* A decode step appends one token per sequence.  Before the step a sequence holds
  ``ctx - 1`` tokens; the step writes the new token's K/V at position ``ctx - 1``
  through ``slot_mapping`` and then attends over all ``ctx`` tokens.
* Physical block ids are a seeded permutation of the pool; logical blocks take them in
  order.  Every block no table reaches, the new token's slot, and every copy-on-write
  destination is filled with NaN, so a kernel that reads outside the table, skips the
  write or skips the copy produces NaN.
* Shared prefix (parallel sampling): the prefix blocks appear in every table.  A
  sequence whose last block is partly filled shares it with a sampling sibling, so the
  step copies it to a fresh block (copy-on-write) before writing into it.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

BLOCK_SIZE = 16
NAN_BF16 = 0x7FC0


@dataclass
class Workload:
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    num_blocks: int
    context_lens: np.ndarray        # int32 [S], tokens attended (new token included)
    block_tables: np.ndarray        # int32 [S][MB], as attention reads them (after COW)
    slot_mapping: np.ndarray        # int64 [T]
    cow_pairs: np.ndarray           # int32 [P][2] (src, dst)
    q: torch.Tensor                 # bf16 [S][Hq][D]
    k_new: torch.Tensor             # bf16 [T][Hkv][D]
    v_new: torch.Tensor
    k_cache: torch.Tensor           # bf16 [NB][Hkv][16][D], state before the step
    v_cache: torch.Tensor
    scale: float
    partition_size: int = 512
    block_size: int = BLOCK_SIZE
    shared_prefix_blocks: int = 0
    meta: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.num_seqs else 0


def _values(shape, gen: torch.Generator, device) -> torch.Tensor:
    return torch.randn(*shape, generator=gen, device=device, dtype=torch.float32).to(
        torch.bfloat16)


def build(name: str, context_lens, num_q_heads: int, num_kv_heads: int, head_dim: int,
          seed: int, device="cpu", num_blocks: int | None = None, free_fraction: float = 0.10,
          shared_prefix_tokens: int = 0, cow_last_block: bool = False,
          write_new_token: bool = True, poison: bool = True, partition_size: int = 512,
          max_blocks: int | None = None) -> Workload:
    """Draw one decode step.

    ``context_lens`` are the lengths attention sees.  With ``shared_prefix_tokens`` > 0
    (a multiple of 16) every sequence starts with the same prefix blocks.  With
    ``cow_last_block`` each sequence whose pre-step length is not a multiple of 16
    gets a copy-on-write pair for its last block.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    ctx = np.asarray(context_lens, dtype=np.int64)
    S = ctx.shape[0]
    bs = BLOCK_SIZE
    assert shared_prefix_tokens % bs == 0
    npre = shared_prefix_tokens // bs
    assert (ctx >= 1).all() and (ctx > shared_prefix_tokens).all()
    prev = ctx - 1 if write_new_token else ctx
    nblk = (ctx + bs - 1) // bs
    own = nblk - npre                                   # blocks not in the shared prefix
    cow = np.zeros(S, dtype=bool)
    if cow_last_block:
        cow = (prev % bs != 0) & (prev > shared_prefix_tokens)
    needed = npre + int(own.sum()) + int(cow.sum())     # + sibling-held source blocks
    if num_blocks is None:
        num_blocks = int(np.ceil(needed * (1.0 + free_fraction)))
    assert num_blocks >= needed, (num_blocks, needed)
    perm = rng.permutation(num_blocks).astype(np.int32)
    MB = int(nblk.max()) if max_blocks is None else max_blocks
    tables = np.full((S, MB), -1, dtype=np.int32)
    cursor = 0
    prefix = perm[cursor:cursor + npre]
    cursor += npre
    cow_pairs = []
    for s in range(S):
        tables[s, :npre] = prefix
        tables[s, npre:nblk[s]] = perm[cursor:cursor + own[s]]
        cursor += own[s]
    for s in range(S):
        if cow[s]:
            src = int(perm[cursor])
            cursor += 1
            dst = int(tables[s, (prev[s]) // bs])
            cow_pairs.append((src, dst))
    cow_pairs = np.asarray(cow_pairs, dtype=np.int32).reshape(-1, 2)
    pos = ctx - 1
    slots = (tables[np.arange(S), pos // bs].astype(np.int64) * bs + pos % bs)

    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    D, Hkv, Hq = head_dim, num_kv_heads, num_q_heads
    q = _values((S, Hq, D), gen, device)
    k_cache = _values((num_blocks, Hkv, bs, D), gen, device)
    v_cache = _values((num_blocks, Hkv, bs, D), gen, device)
    T = S if write_new_token else 0
    k_new = _values((T, Hkv, D), gen, device)
    v_new = _values((T, Hkv, D), gen, device)
    if cow.any():
        # The source of a copy holds the sibling's (pre-step) content of the block.
        src_t = torch.as_tensor(cow_pairs[:, 0].astype(np.int64), device=device)
        dst_t = torch.as_tensor(cow_pairs[:, 1].astype(np.int64), device=device)
        k_cache[src_t] = k_cache[dst_t]
        v_cache[src_t] = v_cache[dst_t]
    if poison:
        used = np.zeros(num_blocks, dtype=bool)
        for s in range(S):
            used[tables[s, :nblk[s]]] = True
        if cow_pairs.size:
            used[cow_pairs[:, 0]] = True
        nan = torch.tensor(NAN_BF16, dtype=torch.int16).view(torch.bfloat16).item()
        unused = torch.as_tensor(np.nonzero(~used)[0].astype(np.int64), device=device)
        if unused.numel():
            k_cache[unused] = nan
            v_cache[unused] = nan
        if cow_pairs.size:
            dst_t = torch.as_tensor(cow_pairs[:, 1].astype(np.int64), device=device)
            k_cache[dst_t] = nan
            v_cache[dst_t] = nan
        if write_new_token:
            b = torch.as_tensor((slots // bs).astype(np.int64), device=device)
            o = torch.as_tensor((slots % bs).astype(np.int64), device=device)
            k_cache[b, :, o] = nan
            v_cache[b, :, o] = nan
    return Workload(name=name, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                    num_blocks=num_blocks, context_lens=ctx.astype(np.int32),
                    block_tables=tables, slot_mapping=slots if write_new_token else
                    np.zeros(0, dtype=np.int64), cow_pairs=cow_pairs, q=q, k_new=k_new,
                    v_new=v_new, k_cache=k_cache, v_cache=v_cache, scale=D ** -0.5,
                    partition_size=partition_size, shared_prefix_blocks=npre)


# The five workloads (shapes of the pages' Llama-2-7B / Llama-3-70B serving cases).
CONFIG_NAMES = {
    1: "tiny-gqa2-d64",
    2: "llama2-7b-mha-b64",
    3: "llama3-70b-gqa8-b256",
    4: "shared-prefix-gqa8-50seq",
    5: "long-context-mixed-gqa8",
}


def config_context_lens(n: int, seed: int) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed + 7919))
    if n == 1:
        return np.array([1, 15, 16, 37], dtype=np.int32)
    if n == 2:
        return rng.integers(128, 4096, size=64, endpoint=True).astype(np.int32)
    if n == 3:
        z = rng.standard_normal(256)
        return np.clip(np.rint(np.exp(np.log(1024.0) + 0.8 * z)), 16, 8192).astype(np.int32)
    if n == 4:
        # pre-step length = 2000-token prefix + suffix in [0, 512]; +1 for the new token
        return (2000 + rng.integers(0, 512, size=50, endpoint=True) + 1).astype(np.int32)
    if n == 5:
        short = rng.integers(256, 4096, size=120, endpoint=True)
        return np.concatenate([np.full(8, 131072), short]).astype(np.int32)
    raise ValueError(f"unknown config {n}")


def make_config(n: int, device="cpu", seed: int | None = None, **kw) -> Workload:
    """Workload ``n`` (1..5) drawn with seed 1000 + n unless given."""
    seed = 1000 + n if seed is None else seed
    ctx = config_context_lens(n, seed)
    name = CONFIG_NAMES[n]
    if n == 1:
        return build(name, ctx, 2, 1, 64, seed, device, num_blocks=16, **kw)
    if n == 2:
        return build(name, ctx, 32, 32, 128, seed, device, **kw)
    if n == 3:
        return build(name, ctx, 64, 8, 128, seed, device, **kw)
    if n == 4:
        return build(name, ctx, 64, 8, 128, seed, device, shared_prefix_tokens=2000,
                     cow_last_block=True, **kw)
    if n == 5:
        return build(name, ctx, 64, 8, 128, seed, device, **kw)
    raise ValueError(n)


def unique_kv_read_bytes(w: Workload) -> int:
    """KV bytes of the distinct (physical block, token offset) slots a step reads: a
    shared prefix block counts once however many tables point at it."""
    depth = {}  # physical block -> tokens read from it (the deepest use if shared)
    for s in range(w.num_seqs):
        n = int(w.context_lens[s])
        for b in range((n + w.block_size - 1) // w.block_size):
            blk = int(w.block_tables[s, b])
            depth[blk] = max(depth.get(blk, 0), min(w.block_size, n - b * w.block_size))
    return sum(depth.values()) * 2 * w.num_kv_heads * w.head_dim * 2


def kv_read_bytes(w: Workload) -> int:
    """Algorithmic KV bytes one decode step reads: every context token's K and V row
    for every KV head, once."""
    return int(w.context_lens.astype(np.int64).sum()) * 2 * w.num_kv_heads * w.head_dim * 2


# -------------------------------------------------------------------------------------
# Chunked prefill: several new tokens per sequence
# -------------------------------------------------------------------------------------
@dataclass
class PrefillWorkload:
    """One chunked-prefill step.  Sequence s ends the step with context_lens[s] tokens,
    the last L_s = query_start[s+1] - query_start[s] of them new: their K/V are written
    at slots slot_mapping[query_start[s]:query_start[s+1]] (positions ctx - L .. ctx - 1)
    and their queries are rows query_start[s] .. query_start[s+1] - 1 of q."""
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    num_blocks: int
    context_lens: np.ndarray        # int32 [S]
    query_start: np.ndarray         # int32 [S+1]
    block_tables: np.ndarray        # int32 [S][MB]
    slot_mapping: np.ndarray        # int64 [T]
    q: torch.Tensor                 # bf16 [T][Hq][D]
    k_new: torch.Tensor             # bf16 [T][Hkv][D]
    v_new: torch.Tensor
    k_cache: torch.Tensor           # bf16 [NB][Hkv][16][D], state before the step
    v_cache: torch.Tensor
    scale: float
    block_size: int = BLOCK_SIZE

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def num_tokens(self) -> int:
        return int(self.query_start[-1])

    @property
    def query_lens(self) -> np.ndarray:
        return np.diff(self.query_start)

    @property
    def max_query_len(self) -> int:
        return int(self.query_lens.max()) if self.num_seqs else 0

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.num_seqs else 0

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])


def build_prefill(name: str, context_lens, query_lens, num_q_heads: int, num_kv_heads: int,
                  head_dim: int, seed: int, device="cpu", num_blocks: int | None = None,
                  free_fraction: float = 0.10, poison: bool = True,
                  max_blocks: int | None = None) -> PrefillWorkload:
    """Draw one chunked-prefill step: tables from a seeded permutation of the pool,
    N(0,1) bf16 values; blocks no table reaches and the slots of the step's new tokens
    hold NaN before the step."""
    rng = np.random.Generator(np.random.PCG64(seed))
    ctx = np.asarray(context_lens, dtype=np.int64)
    L = np.asarray(query_lens, dtype=np.int64)
    S = ctx.shape[0]
    assert L.shape == (S,) and (L >= 0).all() and (L <= ctx).all()
    bs = BLOCK_SIZE
    nblk = (ctx + bs - 1) // bs
    needed = int(nblk.sum())
    if num_blocks is None:
        num_blocks = max(1, int(np.ceil(needed * (1.0 + free_fraction))))
    assert num_blocks >= needed
    perm = rng.permutation(num_blocks).astype(np.int32)
    MB = max(1, int(nblk.max()) if S else 1) if max_blocks is None else max_blocks
    tables = np.full((S, MB), -1, dtype=np.int32)
    cursor = 0
    for s in range(S):
        tables[s, :nblk[s]] = perm[cursor:cursor + nblk[s]]
        cursor += nblk[s]
    qs = np.zeros(S + 1, dtype=np.int32)
    qs[1:] = np.cumsum(L)
    T = int(qs[-1])
    slots = np.zeros(T, dtype=np.int64)
    for s in range(S):
        pos = np.arange(ctx[s] - L[s], ctx[s])
        slots[qs[s]:qs[s + 1]] = tables[s, pos // bs].astype(np.int64) * bs + pos % bs

    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    D, Hkv, Hq = head_dim, num_kv_heads, num_q_heads
    q = _values((T, Hq, D), gen, device)
    k_cache = _values((num_blocks, Hkv, bs, D), gen, device)
    v_cache = _values((num_blocks, Hkv, bs, D), gen, device)
    k_new = _values((T, Hkv, D), gen, device)
    v_new = _values((T, Hkv, D), gen, device)
    if poison:
        used = np.zeros(num_blocks, dtype=bool)
        for s in range(S):
            used[tables[s, :nblk[s]]] = True
        nan = torch.tensor(NAN_BF16, dtype=torch.int16).view(torch.bfloat16).item()
        unused = torch.as_tensor(np.nonzero(~used)[0].astype(np.int64), device=device)
        if unused.numel():
            k_cache[unused] = nan
            v_cache[unused] = nan
        if T:
            b = torch.as_tensor((slots // bs).astype(np.int64), device=device)
            o = torch.as_tensor((slots % bs).astype(np.int64), device=device)
            k_cache[b, :, o] = nan
            v_cache[b, :, o] = nan
    return PrefillWorkload(name=name, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                           num_blocks=num_blocks, context_lens=ctx.astype(np.int32),
                           query_start=qs, block_tables=tables, slot_mapping=slots, q=q,
                           k_new=k_new, v_new=v_new, k_cache=k_cache, v_cache=v_cache,
                           scale=D ** -0.5)


PREFILL_CONFIG_NAMES = {
    1: "prefill-tiny-gqa2-d64",
    2: "chunked-prefill-llama3-70b-gqa8",
    3: "chunked-prefill-llama2-7b-mha",
    4: "chunked-prefill-gqa4-d64",
}


def make_prefill_config(n: int, device="cpu", seed: int | None = None, **kw) -> PrefillWorkload:
    """Chunked-prefill workloads, seed 2000 + n unless given.

    1: five sequences of mixed shape (decode row, whole prompt, chunk after a cached
       prefix, ragged lengths), GQA-2, head_dim 64 -- small enough for the oracle.
    2: Llama-3-70B attention shapes (64 query heads, 8 KV heads, head_dim 128): 16
       sequences, each prefilling a 512-token chunk after a cached prefix of
       U{0..3584} tokens (a scheduler's per-step token budget of 8192).
    3: Llama-2-7B shapes (32 heads, MHA, head_dim 128): 8 sequences, 512-token chunks
       after U{0..3584} cached tokens.
    4: head_dim 64 at scale (32 query heads, 8 KV heads): 16 sequences, 512-token
       chunks after U{0..3584} cached tokens.
    """
    seed = 2000 + n if seed is None else seed
    rng = np.random.Generator(np.random.PCG64(seed + 7919))
    name = PREFILL_CONFIG_NAMES[n]
    if n == 1:
        ctx, L = [1, 5, 40, 70, 100], [1, 5, 17, 2, 64]
        return build_prefill(name, ctx, L, 4, 2, 64, seed, device, **kw)
    if n in (2, 3, 4):
        S = 8 if n == 3 else 16
        prior = rng.integers(0, 3584, size=S, endpoint=True)
        L = np.full(S, 512)
        Hq, Hkv, D = {2: (64, 8, 128), 3: (32, 32, 128), 4: (32, 8, 64)}[n]
        return build_prefill(name, prior + L, L, Hq, Hkv, D, seed, device, **kw)
    raise ValueError(n)


def prefill_flops(w: PrefillWorkload) -> int:
    """Algorithmic flops of the step's attention: each (query token, head) row at
    position p multiplies its q with p + 1 keys and sums p + 1 value rows, 2 D flops
    each (4 D per visible key)."""
    total = 0
    for s in range(w.num_seqs):
        L = int(w.query_start[s + 1] - w.query_start[s])
        c = int(w.context_lens[s])
        # sum over i < L of (c - L + i + 1)
        total += L * (c - L) + L * (L + 1) // 2
    return total * 4 * w.head_dim * w.num_q_heads


# -------------------------------------------------------------------------------------
# Request streams for the continuous-batching scheduler and the prefix cache
# -------------------------------------------------------------------------------------
@dataclass
class Request:
    rid: int
    prompt: np.ndarray      # int32 token ids
    output_len: int


def pareto_output_lens(rng, n, xm=16, alpha=1.5, cap=2048) -> np.ndarray:
    """Output lengths floor(xm * U^(-1/alpha)) clipped to cap (a Pareto law: most
    requests short, a few hundreds of times longer)."""
    u = 1.0 - rng.random(n)
    return np.minimum(cap, np.floor(xm * u ** (-1.0 / alpha))).astype(np.int64)


def make_requests(kind: str, seed: int = 0, n: int | None = None) -> list[Request]:
    """Seeded request streams.

    ``pareto``: n (default 50) requests, prompts U{16..256} random tokens, Pareto output
    lengths (xm 16, shape 1.5, at most 2048).
    ``shared-prefix``: n (default 1000) requests; 60% start with one of 5 common prefixes
    (U{64..256} tokens each) followed by a private U{8..64}-token suffix, the rest are
    private prompts of U{32..256} tokens; Pareto output lengths capped at 256.
    """
    rng = np.random.Generator(np.random.PCG64(seed + 4242))
    reqs = []
    if kind == "pareto":
        n = 50 if n is None else n
        outs = pareto_output_lens(rng, n)
        for i in range(n):
            P = int(rng.integers(16, 256, endpoint=True))
            reqs.append(Request(i, rng.integers(0, 32000, P).astype(np.int32), int(outs[i])))
        return reqs
    if kind == "shared-prefix":
        n = 1000 if n is None else n
        prefixes = [rng.integers(0, 32000, int(rng.integers(64, 256, endpoint=True)))
                    .astype(np.int32) for _ in range(5)]
        outs = pareto_output_lens(rng, n, cap=256)
        for i in range(n):
            if rng.random() < 0.6:
                pre = prefixes[int(rng.integers(5))]
                suf = rng.integers(0, 32000, int(rng.integers(8, 64, endpoint=True)))
                prompt = np.concatenate([pre, suf.astype(np.int32)])
            else:
                prompt = rng.integers(0, 32000, int(rng.integers(32, 256, endpoint=True)))
            reqs.append(Request(i, prompt.astype(np.int32), int(outs[i])))
        return reqs
    raise ValueError(kind)
