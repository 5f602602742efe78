"""Pins of the fp64 oracle to facts outside itself.

Each ``pin_*`` takes a loaded oracle library and raises AssertionError when the oracle
disagrees with a value the pages print, a closed form, a library routine, an
invariant of the method, or brute force on a tiny input.  ``test_oracle_pins.py`` runs
them on the real oracle; ``test_oracle_mutants.py`` plants plausible mistakes in the
oracle's C source and checks that every mistake trips at least one pin.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

import oracle
from oracle.block_manager import BlockManager
from paged_kv_cache_272_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
BS = 16


def _rows(path):
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            data, cite = line.split("|", 1)
            yield data.split(), cite.strip()


def bf16(a) -> torch.Tensor:
    return torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)


def host_caches(w):
    """uint16 copies of the workload's caches (the oracle's working state)."""
    k = w.k_cache.cpu().contiguous().view(torch.int16).numpy().view(np.uint16).copy()
    v = w.v_cache.cpu().contiguous().view(torch.int16).numpy().view(np.uint16).copy()
    return k, v


def run_step(w, lib):
    """Oracle decode step: copy-on-write, write the new token, attend.  fp64 out."""
    k, v = host_caches(w)
    if w.cow_pairs.size:
        oracle.block_copy(k, v, w.cow_pairs, lib=lib)
    if w.slot_mapping.size:
        oracle.kv_write(k, v, w.k_new, w.v_new, w.slot_mapping, lib=lib)
    return oracle.attention(w.q, k, v, w.block_tables, w.context_lens, w.scale, lib=lib), k, v


def gather(k, table, ctx, kv_head):
    """Contiguous [ctx][D] rows of one KV head (fp64), read through the block table."""
    rows = []
    for t in range(ctx):
        rows.append(k[table[t // BS], kv_head, t % BS])
    u = np.stack(rows).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().double().numpy()


# -------------------------------------------------------------------------------------
# Values printed on the pages
# -------------------------------------------------------------------------------------
def pin_kv_bytes_golden(lib):
    n = 0
    for (L, H, D, B, T, expect), cite in _rows(os.path.join(GOLDEN, "kv_bytes.txt")):
        got = oracle.kv_bytes_per_token(int(L), int(H), int(D), int(B), lib=lib) * int(T)
        assert got == int(expect), (got, expect, cite)
        n += 1
    for (L, H, D, B, T, div, printed, tol), cite in _rows(
            os.path.join(GOLDEN, "kv_bytes_rounded.txt")):
        got = oracle.kv_bytes_per_token(int(L), int(H), int(D), int(B), lib=lib) * int(T)
        assert abs(got / float(div) - float(printed)) <= float(tol), (got, printed, cite)
        n += 1
    assert n >= 6


def pin_gqa_reduction(lib):
    # Inference optimization, exercise 3: 64 query heads over 8 KV heads -> 8x less KV.
    mha = oracle.kv_bytes_per_token(80, 64, 128, 2, lib=lib)
    gqa = oracle.kv_bytes_per_token(80, 8, 128, 2, lib=lib)
    assert mha == 8 * gqa


def pin_block_counts():
    for (tokens, blocks), cite in _rows(os.path.join(GOLDEN, "block_counts.txt")):
        bm = BlockManager(64, BS)
        bm.add_seq(0)
        bm.append_tokens(0, int(tokens))
        assert len(bm.block_table(0)) == int(blocks), cite
        assert 0 <= bm.internal_waste(0) < BS


# -------------------------------------------------------------------------------------
# Closed forms and special cases
# -------------------------------------------------------------------------------------
def pin_ctx1_returns_v(lib):
    """One token: its softmax weight is exp(0)/exp(0) = 1, so the output is V exactly."""
    w = workloads.build("ctx1", [1, 1, 1], 4, 2, 64, seed=11)
    out, k, v = run_step(w, lib)
    for s in range(3):
        for h in range(4):
            want = to_f64(w.v_new[s, h // 2])
            assert np.array_equal(out[s, h], want), (s, h)


def pin_uniform_scores_mean(lib):
    """q = 0 makes every score equal, so the output is the plain mean of V."""
    w = workloads.build("uniform", [5, 16, 33, 70], 4, 2, 64, seed=12)
    w.q.zero_()
    out, k, v = run_step(w, lib)
    for s in range(w.num_seqs):
        for h in range(4):
            vc = gather(v, w.block_tables[s], int(w.context_lens[s]), h // 2)
            np.testing.assert_allclose(out[s, h], vc.mean(axis=0), rtol=1e-13, atol=1e-15)


def pin_equal_keys_mean(lib):
    """All keys of a sequence equal: scores equal again, output = mean of V."""
    w = workloads.build("eqk", [9, 40], 2, 1, 64, seed=13)
    k, v = host_caches(w)
    oracle.kv_write(k, v, w.k_new, w.v_new, w.slot_mapping, lib=lib)
    for s in range(2):
        n = int(w.context_lens[s])
        row = k[w.block_tables[s][0], 0, 0].copy()
        for t in range(n):
            k[w.block_tables[s][t // BS], 0, t % BS] = row
        out = oracle.attention(w.q, k, v, w.block_tables, w.context_lens, w.scale, lib=lib)
        vc = gather(v, w.block_tables[s], n, 0)
        for h in range(2):
            np.testing.assert_allclose(out[s, h], vc.mean(axis=0), rtol=1e-13, atol=1e-15)


def pin_two_token_closed_form(lib):
    """Two tokens with scores a*scale and 0: weights are the logistic function of a*scale.

    Two KV heads with different keys and four query heads pin the consecutive
    query-head grouping (head h reads KV head h // 2)."""
    D, Hq, Hkv = 64, 4, 2
    w = workloads.build("closed", [2], Hq, Hkv, D, seed=14, poison=False)
    k, v = host_caches(w)
    oracle.kv_write(k, v, w.k_new, w.v_new, w.slot_mapping, lib=lib)
    b = w.block_tables[0][0]
    e = np.zeros(D, np.float32)
    one = bf16(e).view(torch.int16).numpy().view(np.uint16)  # zeros
    k[b, :, 0:2] = one
    # KV head 0: k_0 = e_3, KV head 1: k_0 = e_7; k_1 = 0 for both
    for g, axis in ((0, 3), (1, 7)):
        e = np.zeros(D, np.float32)
        e[axis] = 1.0
        k[b, g, 0] = bf16(e).view(torch.int16).numpy().view(np.uint16)
    a = np.array([2.0, -3.0, 5.0, 0.5], np.float32)
    qv = np.zeros((1, Hq, D), np.float32)
    for h in range(Hq):
        qv[0, h, 3] = a[h]          # only KV head 0's key sees this
        qv[0, h, 7] = -a[h] / 2     # only KV head 1's key sees this
    q = bf16(qv)
    out = oracle.attention(q, k, v, w.block_tables, w.context_lens, w.scale, lib=lib)
    for h in range(Hq):
        g = h // 2
        x0 = (a[h] if g == 0 else -a[h] / 2) * w.scale
        w0 = 1.0 / (1.0 + math.exp(-x0))
        v0 = gather(v, w.block_tables[0], 2, g)
        want = w0 * v0[0] + (1.0 - w0) * v0[1]
        np.testing.assert_allclose(out[0, h], want, rtol=1e-13, atol=1e-15)


def pin_ctx_zero(lib):
    w = workloads.build("zero", [3, 3], 2, 1, 64, seed=15)
    k, v = host_caches(w)
    oracle.kv_write(k, v, w.k_new, w.v_new, w.slot_mapping, lib=lib)
    ctx = w.context_lens.copy()
    ctx[1] = 0
    out = oracle.attention(w.q, k, v, w.block_tables, ctx, w.scale, lib=lib)
    assert np.all(out[1] == 0.0)
    assert np.all(np.isfinite(out[0]))


# -------------------------------------------------------------------------------------
# Library routine and brute force
# -------------------------------------------------------------------------------------
class AppendOnlyKV:
    """A sequence's KV held contiguously, as "Inference optimization" ("KV cache") describes
    it: each step computes only its new tokens' K/V and appends them along the sequence
    axis.  Kept here as a list of the appended pieces, each [heads][new tokens][D];
    `rows()` joins them into the [heads][tokens so far][D] view attention reads."""

    def __init__(self):
        self._k, self._v = [], []

    def append(self, new_k, new_v):
        self._k.append(np.asarray(new_k, np.float64))
        self._v.append(np.asarray(new_v, np.float64))

    def rows(self):
        return np.concatenate(self._k, axis=1), np.concatenate(self._v, axis=1)


def contiguous_from_paged(k, v, table, ctx, Hkv, D, chunk=7):
    """Feed a sequence's tokens, in logical order and in chunks, through the
    contiguous cache."""
    cache = AppendOnlyKV()
    for t0 in range(0, ctx, chunk):
        t1 = min(ctx, t0 + chunk)
        cache.append(np.stack([gather(k, table, t1, g)[t0:t1] for g in range(Hkv)]),
                     np.stack([gather(v, table, t1, g)[t0:t1] for g in range(Hkv)]))
    return cache.rows()


def pin_sdpa_contiguous(lib, cfg=1, ctx_override=None, Hq=None, Hkv=None, seed=16):
    """Paged oracle == torch's fp64 scaled_dot_product_attention over the contiguous
    cache (the library routine of "System-level optimization", section 3.3)."""
    if ctx_override is None:
        w = workloads.make_config(cfg)
    else:
        w = workloads.build("sdpa", ctx_override, Hq, Hkv, 64, seed=seed)
    out, k, v = run_step(w, lib)
    G = w.num_q_heads // w.num_kv_heads
    for s in range(w.num_seqs):
        n = int(w.context_lens[s])
        kk, vv = contiguous_from_paged(k, v, w.block_tables[s], n, w.num_kv_heads,
                                       w.head_dim)
        qt = torch.from_numpy(to_f64(w.q[s])).view(1, w.num_q_heads, 1, w.head_dim)
        kt = torch.from_numpy(kk).repeat_interleave(G, dim=0).unsqueeze(0)
        vt = torch.from_numpy(vv).repeat_interleave(G, dim=0).unsqueeze(0)
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=w.scale)
        np.testing.assert_allclose(out[s], ref[0, :, 0].numpy(), rtol=1e-11, atol=1e-12)


def pin_brute_force_tiny(lib):
    """Configuration 1 recomputed with explicit Python loops and math.exp."""
    w = workloads.make_config(1)
    out, k, v = run_step(w, lib)
    q = to_f64(w.q)
    G = w.num_q_heads // w.num_kv_heads
    for s in range(w.num_seqs):
        n = int(w.context_lens[s])
        for h in range(w.num_q_heads):
            kc = gather(k, w.block_tables[s], n, h // G)
            vc = gather(v, w.block_tables[s], n, h // G)
            xs = [w.scale * sum(q[s, h, d] * kc[t, d] for d in range(w.head_dim))
                  for t in range(n)]
            mx = max(xs)
            ws = [math.exp(x - mx) for x in xs]
            tot = sum(ws)
            for d in range(w.head_dim):
                want = sum(ws[t] * vc[t, d] for t in range(n)) / tot
                assert abs(out[s, h, d] - want) <= 1e-12 * (1 + abs(want)), (s, h, d)


def pin_large_magnitude(lib):
    """q scaled by 30: scores reach hundreds; the result stays finite and equals the
    library routine."""
    w = workloads.build("big", [17, 64, 200], 4, 2, 64, seed=17)
    w.q.mul_(30)
    out, k, v = run_step(w, lib)
    assert np.all(np.isfinite(out))
    for s in range(w.num_seqs):
        n = int(w.context_lens[s])
        for h in range(4):
            kc = gather(k, w.block_tables[s], n, h // 2)
            vc = gather(v, w.block_tables[s], n, h // 2)
            x = torch.from_numpy(to_f64(w.q[s, h]) @ kc.T * w.scale)
            want = torch.softmax(x, 0).numpy() @ vc
            np.testing.assert_allclose(out[s, h], want, rtol=1e-10, atol=1e-12)


# -------------------------------------------------------------------------------------
# Invariants of the paged layout
# -------------------------------------------------------------------------------------
def pin_permutation_invariance(lib):
    """Relabelling the physical blocks (and the tables with them) changes nothing:
    the table alone decides which bytes a sequence sees."""
    w = workloads.build("perm", [3, 16, 17, 50, 90], 4, 2, 64, seed=18)
    out, k, v = run_step(w, lib)
    rng = np.random.default_rng(5)
    perm = rng.permutation(w.num_blocks)
    k2 = np.empty_like(k)
    v2 = np.empty_like(v)
    k2[perm] = k
    v2[perm] = v
    bt = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    out2 = oracle.attention(w.q, k2, v2, bt, w.context_lens, w.scale, lib=lib)
    assert np.array_equal(out, out2)


def pin_gqa_equals_mha(lib):
    """GQA equals MHA whose KV heads are the GQA heads repeated G times (consecutive
    grouping)."""
    G = 4
    w = workloads.build("gqa", [5, 31, 47], 8, 2, 64, seed=19)
    out, k, v = run_step(w, lib)
    km = np.ascontiguousarray(np.repeat(k, G, axis=1))
    vm = np.ascontiguousarray(np.repeat(v, G, axis=1))
    out2 = oracle.attention(w.q, km, vm, w.block_tables, w.context_lens, w.scale, lib=lib)
    assert np.array_equal(out, out2)


def pin_shared_prefix_equals_private(lib):
    """Sequences that share prefix blocks give the same result as if each had a
    private copy of those blocks."""
    w = workloads.build("prefix", [40, 33, 50, 65], 4, 2, 64, seed=20,
                        shared_prefix_tokens=32, cow_last_block=True, free_fraction=3.0)
    out, k, v = run_step(w, lib)
    free = sorted(set(range(w.num_blocks)) - set(w.block_tables[w.block_tables >= 0].tolist())
                  - set(w.cow_pairs[:, 0].tolist()))
    bt = w.block_tables.copy()
    it = iter(free)
    for s in range(1, w.num_seqs):
        for j in range(2):
            nb = next(it)
            k[nb] = k[bt[s, j]]
            v[nb] = v[bt[s, j]]
            bt[s, j] = nb
    assert len(set(bt[:, 0].tolist())) == w.num_seqs
    out2 = oracle.attention(w.q, k, v, bt, w.context_lens, w.scale, lib=lib)
    assert np.array_equal(out, out2)


def pin_write_matches_kvcache_update(lib):
    """Appending tokens one by one through slots, read back through the block table,
    gives the same rows as appending them to a contiguous per-sequence KV."""
    Hkv, D, n = 2, 64, 37
    bm = BlockManager(12, BS, free_order=np.random.default_rng(3).permutation(12))
    bm.add_seq(0)
    k = np.full((12, Hkv, BS, D), workloads.NAN_BF16, np.uint16)
    v = k.copy()
    gen = torch.Generator().manual_seed(4)
    newk = torch.randn(n, Hkv, D, generator=gen).to(torch.bfloat16)
    newv = torch.randn(n, Hkv, D, generator=gen).to(torch.bfloat16)
    cache = AppendOnlyKV()
    for t in range(n):
        slot, cow = bm.append_slot(0)
        assert cow is None
        oracle.kv_write(k, v, newk[t:t + 1], newv[t:t + 1], [slot], lib=lib)
        cache.append(to_f64(newk[t:t + 1]).transpose(1, 0, 2),
                     to_f64(newv[t:t + 1]).transpose(1, 0, 2))
    kk, vv = cache.rows()
    table = bm.block_table(0)
    for g in range(Hkv):
        assert np.array_equal(gather(k, table, n, g), kk[g])
        assert np.array_equal(gather(v, table, n, g), vv[g])


def pin_write_bytes(lib):
    """Only the addressed rows change; a negative slot is skipped."""
    NB, Hkv, D = 6, 2, 64
    rng = np.random.default_rng(21)
    k = rng.integers(0, 2 ** 16, size=(NB, Hkv, BS, D), dtype=np.uint16)
    v = rng.integers(0, 2 ** 16, size=(NB, Hkv, BS, D), dtype=np.uint16)
    k0, v0 = k.copy(), v.copy()
    newk = rng.integers(0, 2 ** 16, size=(3, Hkv, D), dtype=np.uint16)
    newv = rng.integers(0, 2 ** 16, size=(3, Hkv, D), dtype=np.uint16)
    slots = [5 * BS + 15, -1, 0 * BS + 3]
    oracle.kv_write(k, v, newk, newv, slots, lib=lib)
    k0[5, :, 15] = newk[0]
    v0[5, :, 15] = newv[0]
    k0[0, :, 3] = newk[2]
    v0[0, :, 3] = newv[2]
    assert np.array_equal(k, k0) and np.array_equal(v, v0)


def pin_copy_bytes(lib):
    """Copy-on-write: the destination block equals the source in every KV head, for K
    and V; nothing else changes."""
    NB, Hkv, D = 8, 3, 64
    rng = np.random.default_rng(22)
    k = rng.integers(0, 2 ** 16, size=(NB, Hkv, BS, D), dtype=np.uint16)
    v = rng.integers(0, 2 ** 16, size=(NB, Hkv, BS, D), dtype=np.uint16)
    k0, v0 = k.copy(), v.copy()
    pairs = [(1, 6), (4, 2), (7, 0)]
    oracle.block_copy(k, v, pairs, lib=lib)
    for s, d in pairs:
        k0[d] = k0[s]
        v0[d] = v0[s]
    assert np.array_equal(k, k0) and np.array_equal(v, v0)


ALL_PINS = [
    pin_kv_bytes_golden, pin_gqa_reduction, pin_ctx1_returns_v, pin_uniform_scores_mean,
    pin_equal_keys_mean, pin_two_token_closed_form, pin_ctx_zero, pin_sdpa_contiguous,
    pin_brute_force_tiny, pin_large_magnitude, pin_permutation_invariance, pin_gqa_equals_mha,
    pin_shared_prefix_equals_private, pin_write_matches_kvcache_update, pin_write_bytes,
    pin_copy_bytes,
]


# -------------------------------------------------------------------------------------
# FP8 (E4M3) cache
# -------------------------------------------------------------------------------------
def pin_quant_capacity(lib):
    """The byte formula is linear in the element width: at the same memory an fp8 cache
    holds 2x the tokens of a 16-bit one and an int4 cache about 4x (the pages' figures).
    The width argument is given in bits here, so the ratio is width-independent."""
    for (fmt, bits, gain), cite in _rows(os.path.join(GOLDEN, "kv_quant_capacity.txt")):
        b16 = oracle.kv_bytes_per_token(80, 8, 128, 16, lib=lib)
        bq = oracle.kv_bytes_per_token(80, 8, 128, int(bits), lib=lib)
        assert b16 / bq == float(gain), (fmt, cite)


def pin_e4m3_table(lib):
    for (code, value), what in _rows(os.path.join(GOLDEN, "e4m3_codes.txt")):
        got = oracle.e4m3_decode(int(code, 16), lib=lib)
        if value == "nan":
            assert math.isnan(got), what
        else:
            assert got == float(value) and math.copysign(1, got) == math.copysign(1, float(value)), \
                (code, got, what)


def _grid():
    vals = []
    for c in range(256):
        if (c & 0x7F) == 0x7F:
            continue
        s = -1.0 if c & 0x80 else 1.0
        e, m = (c >> 3) & 15, c & 7
        v = m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
        vals.append((s * v, c))
    return vals


def pin_e4m3_nearest(lib):
    """Every code decodes to its grid value and encodes back; random floats encode to
    the nearest grid value (ties to the even mantissa); beyond 448 saturates.  The grid
    here is enumerated independently of the oracle's codec."""
    grid = _grid()
    for v, c in grid:
        assert oracle.e4m3_decode(c, lib=lib) == v
        if v != 0 or c in (0x00, 0x80):
            assert oracle.e4m3_encode(v, lib=lib) == c, (v, c)
    finite = sorted({v for v, c in grid})
    rng = np.random.default_rng(23)
    xs = np.concatenate([rng.uniform(-500, 500, 4000), rng.uniform(-0.05, 0.05, 4000),
                         rng.standard_normal(4000) * 3]).astype(np.float32)
    # exact midpoints between neighbours, to exercise ties
    mids = [(a + b) / 2 for a, b in zip(finite[:-1], finite[1:])]
    xs = np.concatenate([xs, np.asarray(mids, np.float32)])
    for x in xs:
        x = float(x)
        code = oracle.e4m3_encode(x, lib=lib)
        got = oracle.e4m3_decode(code, lib=lib)
        if abs(x) > 448:
            assert got == math.copysign(448.0, x), x
            continue
        best = min(abs(x - v) for v in finite)
        cands = [c for v, c in grid if abs(x - v) == best]
        if len(cands) > 1:  # a tie: the even mantissa wins (signed zeros aside)
            cands = [c for c in cands if (c & 1) == 0 and (c & 0x7F) != 0 or
                     (c & 0x7F) == 0 and math.copysign(1, x) == (-1 if c & 0x80 else 1)]
        assert abs(got - x) == best and code in cands, (x, code, got, cands)


def _fp8_workload(seed, ctx, Hq=8, Hkv=2, D=128, **kw):
    w = workloads.build("fp8", ctx, Hq, Hkv, D, seed=seed, **kw)
    return w


def pin_fp8_write(lib):
    """The written byte is E4M3(bf16 / scale) (division in fp32), slots skipped when
    negative, everything else untouched; the stored value is within half a grid step.
    K codes sit at [block][head][offset][d], V codes at [block][head][d][offset].  Run
    with one scale for the cache and with a different scale for each KV head (head h
    divides by its own entry)."""
    for ks, vs in ((0.37, 0.0021), ([0.37, 1.5, 0.011], [0.0021, 0.25, 3.0])):
        _fp8_write_case(lib, ks, vs)


def _fp8_write_case(lib, ks, vs):
    NB, Hkv, D = 6, 3, 128
    ksh = np.broadcast_to(np.asarray(ks, np.float32), (Hkv,))
    vsh = np.broadcast_to(np.asarray(vs, np.float32), (Hkv,))
    rng = np.random.default_rng(29)
    k = rng.integers(0, 256, size=(NB, Hkv, BS, D), dtype=np.uint8)
    v = rng.integers(0, 256, size=(NB, Hkv, BS, D), dtype=np.uint8)
    k0, v0 = k.copy(), v.copy()
    gen = torch.Generator().manual_seed(31)
    newk = (torch.randn(3, Hkv, D, generator=gen) * 40).to(torch.bfloat16)
    newv = (torch.randn(3, Hkv, D, generator=gen) * 0.01).to(torch.bfloat16)
    slots = [4 * BS + 9, -1, 1 * BS + 0]
    oracle.kv_write_fp8(k, v, newk, newv, slots, ks, vs, lib=lib)
    for t, slot in enumerate(slots):
        if slot < 0:
            continue
        b, o = slot // BS, slot % BS
        for h in range(Hkv):
            for d in range(D):
                xk = float(np.float32(float(newk[t, h, d])) / ksh[h])
                xv = float(np.float32(float(newv[t, h, d])) / vsh[h])
                k0[b, h, o, d] = oracle.e4m3_encode(xk, lib=lib)
                v0.reshape(NB, Hkv, D, BS)[b, h, d, o] = oracle.e4m3_encode(xv, lib=lib)
                dk = oracle.e4m3_decode(int(k0[b, h, o, d]), lib=lib)
                if abs(xk) <= 448:
                    assert abs(dk - xk) <= max(abs(xk) / 16, 2.0 ** -10)
    assert np.array_equal(k, k0) and np.array_equal(v, v0)


def pin_fp8_attention_equals_bf16(lib):
    """With power-of-two scales every decoded element is a bf16 value, so attention over
    the E4M3 cache equals the pinned bf16 oracle over those values, bit for bit.  Run
    with one scale pair for the cache and with a different pair for each KV head (a
    query head takes the scales of the KV head it reads)."""
    w = _fp8_workload(37, [1, 5, 16, 33, 70], Hq=12, Hkv=3, poison=False)
    out16, k16, v16 = run_step(w, lib)
    NB, Hkv, bs, D = k16.shape
    dec = np.vectorize(lambda c: oracle.e4m3_decode(int(c), lib=lib))
    for ks, vs in ((0.25, 2.0), ([0.25, 4.0, 0.0625], [2.0, 0.5, 8.0])):
        kq = np.zeros(k16.shape, np.uint8)
        vq = np.zeros(v16.shape, np.uint8)
        oracle.kv_write_fp8(kq, vq, _all_rows(k16), _all_rows(v16), np.arange(NB * BS),
                            ks, vs, lib=lib)
        ksh = np.broadcast_to(np.asarray(ks, np.float64), (Hkv,))[None, :, None, None]
        vsh = np.broadcast_to(np.asarray(vs, np.float64), (Hkv,))[None, :, None, None]
        kd = torch.from_numpy(dec(kq) * ksh).to(torch.bfloat16)
        # V codes are stored [block][head][d][offset]
        vt = np.ascontiguousarray(vq.reshape(NB, Hkv, D, bs).transpose(0, 1, 3, 2))
        vd = torch.from_numpy(dec(vt) * vsh).to(torch.bfloat16)
        assert torch.equal(kd.double(), torch.from_numpy(dec(kq) * ksh))  # exact in bf16
        ref = oracle.attention(w.q, kd, vd, w.block_tables, w.context_lens, w.scale, lib=lib)
        got = oracle.attention_fp8(w.q, kq, vq, w.block_tables, w.context_lens, w.scale, ks,
                                   vs, lib=lib)
        assert np.array_equal(ref, got), (ks, vs)


def _all_rows(cache_u16):
    """[NB][Hkv][16][D] uint16 -> [NB*16][Hkv][D] rows in slot order (for a full write)."""
    NB, Hkv, bs, D = cache_u16.shape
    return np.ascontiguousarray(cache_u16.transpose(0, 2, 1, 3).reshape(NB * bs, Hkv, D))


def pin_fp8_copy(lib):
    NB, Hkv, D = 8, 2, 128
    rng = np.random.default_rng(41)
    k = rng.integers(0, 256, size=(NB, Hkv, BS, D), dtype=np.uint8)
    v = rng.integers(0, 256, size=(NB, Hkv, BS, D), dtype=np.uint8)
    k0, v0 = k.copy(), v.copy()
    pairs = [(1, 6), (4, 2)]
    oracle.block_copy_fp8(k, v, pairs, lib=lib)
    for s, d in pairs:
        k0[d] = k0[s]
        v0[d] = v0[s]
    assert np.array_equal(k, k0) and np.array_equal(v, v0)


FP8_PINS = [pin_quant_capacity, pin_e4m3_table, pin_e4m3_nearest, pin_fp8_write,
            pin_fp8_attention_equals_bf16, pin_fp8_copy]
ALL_PINS = ALL_PINS + FP8_PINS


# -------------------------------------------------------------------------------------
# Chunked prefill (causal attention of several new tokens per sequence)
# -------------------------------------------------------------------------------------
def run_prefill(w, lib, sel=None):
    """Oracle chunked-prefill step: write the step's new tokens, attend.  fp64 out."""
    k, v = host_caches(w)
    if w.slot_mapping.size:
        oracle.kv_write(k, v, w.k_new, w.v_new, w.slot_mapping, lib=lib)
    out = oracle.attention_prefill(w.q, k, v, w.block_tables, w.context_lens, w.query_start,
                                   w.scale, sel=sel, lib=lib)
    return out, k, v


def pin_prefill_sdpa_causal(lib):
    """Whole prompts (L == context) equal torch's fp64 scaled_dot_product_attention
    with is_causal=True over the contiguous cache ("System-level optimization",
    section 3.3 calls the routine that way); GQA by repeating each KV head."""
    ctx = [1, 2, 15, 16, 17, 40]
    w = workloads.build_prefill("sdpa-causal", ctx, ctx, 6, 2, 64, seed=81)
    out, k, v = run_prefill(w, lib)
    G = 3
    for s in range(w.num_seqs):
        n, t0 = int(w.context_lens[s]), int(w.query_start[s])
        kk, vv = contiguous_from_paged(k, v, w.block_tables[s], n, 2, 64)
        qt = torch.from_numpy(to_f64(w.q[t0:t0 + n])).permute(1, 0, 2).unsqueeze(0)
        kt = torch.from_numpy(kk).repeat_interleave(G, dim=0).unsqueeze(0)
        vt = torch.from_numpy(vv).repeat_interleave(G, dim=0).unsqueeze(0)
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True,
                                                                scale=w.scale)
        np.testing.assert_allclose(out[t0:t0 + n], ref[0].permute(1, 0, 2).numpy(),
                                   rtol=1e-11, atol=1e-12)


def pin_prefill_chunks_equal_whole(lib):
    """Cutting a prompt into chunks changes nothing: causality makes a token's output
    depend only on the tokens up to it, so the chunk that ends at position c, attended
    with context c, reproduces those rows of the whole-prompt prefill exactly."""
    N, cuts = 90, [0, 23, 24, 57, 90]
    w = workloads.build_prefill("whole", [N], [N], 4, 2, 64, seed=82)
    whole, k, v = run_prefill(w, lib)
    for a, b in zip(cuts[:-1], cuts[1:]):
        part = oracle.attention_prefill(w.q[a:b], k, v, w.block_tables, [b], [0, b - a],
                                        w.scale, lib=lib)
        assert np.array_equal(part, whole[a:b]), (a, b)


def pin_prefill_last_row_is_decode(lib):
    """The last new token of each sequence attends over the whole context, as a decode
    step's query does."""
    ctx, L = [3, 40, 70, 33], [3, 17, 5, 1]
    w = workloads.build_prefill("lastrow", ctx, L, 4, 1, 64, seed=83)
    out, k, v = run_prefill(w, lib)
    last = w.query_start[1:] - 1
    dec = oracle.attention(w.q[torch.as_tensor(last.astype(np.int64))], k, v, w.block_tables,
                           w.context_lens, w.scale, lib=lib)
    assert np.array_equal(out[last], dec)


def pin_prefill_brute_force(lib):
    """A chunk after a cached prefix recomputed with explicit Python loops: row i of
    the chunk sees tokens 0 .. ctx - L + i."""
    ctx, L = [21, 9], [6, 9]
    w = workloads.build_prefill("brute", ctx, L, 2, 1, 64, seed=84)
    out, k, v = run_prefill(w, lib)
    q = to_f64(w.q)
    for s in range(w.num_seqs):
        n = int(w.context_lens[s])
        kc = gather(k, w.block_tables[s], n, 0)
        vc = gather(v, w.block_tables[s], n, 0)
        for i in range(L[s]):
            tok = int(w.query_start[s]) + i
            vis = n - L[s] + i + 1
            for h in range(2):
                xs = [w.scale * sum(q[tok, h, d] * kc[t, d] for d in range(64))
                      for t in range(vis)]
                mx = max(xs)
                ws = [math.exp(x - mx) for x in xs]
                tot = sum(ws)
                for d in range(0, 64, 7):
                    want = sum(ws[t] * vc[t, d] for t in range(vis)) / tot
                    assert abs(out[tok, h, d] - want) <= 1e-12 * (1 + abs(want)), (s, i, h, d)


PREFILL_PINS = [pin_prefill_sdpa_causal, pin_prefill_chunks_equal_whole,
                pin_prefill_last_row_is_decode, pin_prefill_brute_force]
ALL_PINS = ALL_PINS + PREFILL_PINS
