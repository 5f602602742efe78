"""Helpers shared by the GPU parity tests: run one decode step through the C ABI and
compare it with the oracle."""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
from paged_kv_cache_272_gb300 import workloads

ATOL, RTOL, MEAN_TOL = 1e-2, 1e-2, 2e-3
K_SCALE, V_SCALE = 0.02, 0.015  # E4M3 cache scales of the FP8 tests
NTHREADS = max(1, min(32, os.cpu_count() or 1))


def ops():
    from paged_kv_cache_272_gb300 import ops as _ops
    return _ops


def to_cuda(w: workloads.Workload):
    """Device copies of everything one step reads."""
    dev = "cuda"
    return dict(
        k=w.k_cache.to(dev).contiguous().clone(), v=w.v_cache.to(dev).contiguous().clone(),
        q=w.q.to(dev).contiguous(), k_new=w.k_new.to(dev).contiguous(),
        v_new=w.v_new.to(dev).contiguous(),
        slots=torch.as_tensor(w.slot_mapping, dtype=torch.int64, device=dev),
        pairs=torch.as_tensor(w.cow_pairs.reshape(-1, 2), dtype=torch.int32, device=dev),
        bt=torch.as_tensor(w.block_tables, dtype=torch.int32, device=dev),
        ctx=torch.as_tensor(w.context_lens, dtype=torch.int32, device=dev))


def gpu_step(w: workloads.Workload, variant=None, partition_size=None, max_context_len=None,
             d=None, block_tables=None, context_lens=None):
    """copy-on-write -> write -> attention through the C ABI.  Returns (out, k, v, err)."""
    o = ops()
    d = d or to_cuda(w)
    if variant is not None:
        o.set_attention_variant(variant)
    P = w.partition_size if partition_size is None else partition_size  # 0: automatic
    mcl = w.max_context_len if max_context_len is None else max_context_len
    bt = d["bt"] if block_tables is None else block_tables
    ctx = d["ctx"] if context_lens is None else context_lens
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    if d["pairs"].numel():
        o.paged_block_copy(d["k"], d["v"], d["pairs"], err_flag=err)
    if d["slots"].numel():
        o.paged_kv_write(d["k_new"], d["v_new"], d["slots"], d["k"], d["v"], err_flag=err)
    S, Hq, D = d["q"].shape
    out = torch.full((S, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = o.alloc_workspace(S, Hq, D, mcl, P)
    ws.fill_(0xFF)  # stale workspace content must not matter
    o.paged_attention_decode(out, d["q"], d["k"], d["v"], bt, ctx, w.scale, mcl, ws, P,
                             err_flag=err)
    torch.cuda.synchronize()
    if variant is not None:
        o.set_attention_variant(o.PKV_ATTN_AUTO)
    return out, d["k"], d["v"], int(err.item())


def u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def oracle_caches(w: workloads.Workload):
    k, v = u16(w.k_cache).copy(), u16(w.v_cache).copy()
    if w.cow_pairs.size:
        oracle.block_copy(k, v, w.cow_pairs)
    if w.slot_mapping.size:
        oracle.kv_write(k, v, u16(w.k_new), u16(w.v_new), w.slot_mapping)
    return k, v


def oracle_out(w, k, v, sel=None, context_lens=None, block_tables=None):
    ctx = w.context_lens if context_lens is None else context_lens
    bt = w.block_tables if block_tables is None else block_tables
    return oracle.attention(u16(w.q), k, v, bt, ctx, w.scale, sel=sel, nthreads=NTHREADS)


def assert_attention_close(gpu_out: torch.Tensor, ref: np.ndarray, what=""):
    g = gpu_out.detach().float().cpu().double().numpy().reshape(ref.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = np.abs(g - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} elements out of tolerance, max err "
                           f"{err.max():.3g} at {np.unravel_index(err.argmax(), err.shape)}")
    assert err.mean() <= MEAN_TOL, f"{what}: mean |err| {err.mean():.3g} > {MEAN_TOL}"
    return float(err.max()), float(err.mean())


def sample_pairs(w, n_short=64, seed=0):
    """(sequence, head) pairs: every sequence of the longest context with one head per
    KV head, plus random others."""
    rng = np.random.default_rng(seed)
    G = w.num_q_heads // w.num_kv_heads
    longest = np.flatnonzero(w.context_lens == w.context_lens.max())
    pairs = [(int(s), int(g * G + rng.integers(G))) for s in longest
             for g in range(w.num_kv_heads)]
    for _ in range(n_short):
        pairs.append((int(rng.integers(w.num_seqs)), int(rng.integers(w.num_q_heads))))
    return np.array(pairs, dtype=np.int32)


def wide_pairs(w, n_short=256, seed=0):
    """(sequence, head) pairs: every query head of every sequence of the longest context
    (each of their split-K merges in full), plus n_short distinct random rows of the
    other sequences."""
    rng = np.random.default_rng(seed)
    longest = np.flatnonzero(w.context_lens == w.context_lens.max())
    pairs = [(int(s), h) for s in longest for h in range(w.num_q_heads)]
    others = np.setdiff1d(np.arange(w.num_seqs), longest)
    cand = np.stack(np.meshgrid(others, np.arange(w.num_q_heads), indexing="ij"), -1)
    cand = cand.reshape(-1, 2)
    pick = rng.choice(len(cand), size=min(n_short, len(cand)), replace=False)
    pairs += [tuple(int(x) for x in cand[i]) for i in pick]
    return np.array(pairs, dtype=np.int32)


def rows_of(cache: torch.Tensor) -> torch.Tensor:
    """[NB][Hkv][16][D] -> [NB*16][Hkv][D] in slot order (to quantise a whole cache)."""
    NB, Hkv, bs, D = cache.shape
    return cache.permute(0, 2, 1, 3).reshape(NB * bs, Hkv, D).contiguous()


def fp8_step(w, ks=K_SCALE, vs=V_SCALE, partition_size=None, block_tables=None):
    """Quantise the pre-step cache, then COW copy + new-token write + attention, on the
    GPU and in the oracle.  Returns (gpu_out, gpu k/v codes, oracle k/v codes, err).
    ks/vs: one scale each, or one per KV head (sequences of num_kv_heads)."""
    o = ops()
    dev = "cuda"
    NB, Hkv, bs, D = w.k_cache.shape
    kq = torch.zeros(NB, Hkv, bs, D, dtype=torch.uint8, device=dev)
    vq = torch.zeros_like(kq)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    if np.ndim(ks) or np.ndim(vs):  # one scale per KV head: the _per_head entry points
        kst = torch.as_tensor(np.broadcast_to(np.asarray(ks, np.float32), (Hkv,)).copy(),
                              device=dev)
        vst = torch.as_tensor(np.broadcast_to(np.asarray(vs, np.float32), (Hkv,)).copy(),
                              device=dev)
        write = lambda kn, vn, sl: o.paged_kv_write_fp8_per_head(kn, vn, sl, kq, vq, kst, vst,
                                                                 err_flag=err)
        attend = lambda out, q, bt, ctx, ws, P: o.paged_attention_decode_fp8_per_head(
            out, q, kq, vq, bt, ctx, w.scale, kst, vst, w.max_context_len, ws, P, err_flag=err)
    else:
        write = lambda kn, vn, sl: o.paged_kv_write_fp8(kn, vn, sl, kq, vq, ks, vs, err_flag=err)
        attend = lambda out, q, bt, ctx, ws, P: o.paged_attention_decode_fp8(
            out, q, kq, vq, bt, ctx, w.scale, ks, vs, w.max_context_len, ws, P, err_flag=err)
    slots_all = torch.arange(NB * bs, dtype=torch.int64, device=dev)
    write(rows_of(w.k_cache.to(dev)), rows_of(w.v_cache.to(dev)), slots_all)
    d = to_cuda(w)
    if d["pairs"].numel():
        o.paged_block_copy_fp8(kq, vq, d["pairs"], err_flag=err)
    if d["slots"].numel():
        write(d["k_new"], d["v_new"], d["slots"])
    S, Hq, _ = d["q"].shape
    P = w.partition_size if partition_size is None else partition_size  # 0: automatic
    out = torch.full((S, Hq, D), float("nan"), dtype=torch.bfloat16, device=dev)
    ws = o.alloc_workspace(S, Hq, D, w.max_context_len, P)
    bt = d["bt"] if block_tables is None else block_tables
    attend(out, d["q"], bt, d["ctx"], ws, P)
    torch.cuda.synchronize()
    # oracle
    ko = np.zeros((NB, Hkv, bs, D), np.uint8)
    vo = np.zeros_like(ko)
    oracle.kv_write_fp8(ko, vo, u16(rows_of(w.k_cache.cpu())), u16(rows_of(w.v_cache.cpu())),
                        np.arange(NB * bs), ks, vs)
    if w.cow_pairs.size:
        oracle.block_copy_fp8(ko, vo, w.cow_pairs)
    if w.slot_mapping.size:
        oracle.kv_write_fp8(ko, vo, u16(w.k_new), u16(w.v_new), w.slot_mapping, ks, vs)
    return out, kq.cpu().numpy(), vq.cpu().numpy(), ko, vo, int(err.item())


def fp8_ref(w, ko, vo, ks=K_SCALE, vs=V_SCALE, sel=None):
    return oracle.attention_fp8(u16(w.q), ko, vo, w.block_tables, w.context_lens, w.scale, ks,
                                vs, sel=sel, nthreads=NTHREADS)


def spread_heads(w, factors):
    """Scale KV head h of the workload's caches and new rows by factors[h] (powers of two,
    exact in bf16), so that the heads span different ranges."""
    for h, f in enumerate(factors):
        for t in (w.k_cache, w.v_cache):
            t[:, h].mul_(f)
        for t in (w.k_new, w.v_new):
            if t.numel():
                t[:, h].mul_(f)


def per_head_scales(w, margin=1.0):
    """Per-KV-head calibration: the largest |value| of head h over the cache and the new
    rows (finite values only), divided by 448 (the largest E4M3 value), times margin."""
    def fin_amax(x):  # poisoned free blocks hold NaN; they take no part in the range
        x = x.float().abs()
        return float(torch.where(torch.isfinite(x), x, torch.zeros_like(x)).max())

    def amax(c, n):  # one KV head at a time (bounded temporaries on large caches)
        a = np.array([max(fin_amax(c[:, h]), fin_amax(n[:, h]) if n.numel() else 0.0)
                      for h in range(c.shape[1])])
        return (a / 448.0 * margin).astype(np.float32)
    return amax(w.k_cache, w.k_new), amax(w.v_cache, w.v_new)
