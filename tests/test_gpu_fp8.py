"""E4M3 (FP8) KV cache through the C ABI: the quantising write and the block copy match
the oracle byte for byte; decode attention over the E4M3 cache matches the fp64 oracle
(every element decode(code) * scale) within |err| <= 1e-2 + 1e-2 |ref|, mean <= 2e-3."""
import numpy as np
import pytest
import torch

import gpu_helpers as H
import oracle
from paged_kv_cache_272_gb300 import workloads

pytestmark = pytest.mark.gpu
BS = 16
K_SCALE, V_SCALE = H.K_SCALE, H.V_SCALE


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def same_codes(a: np.ndarray, b: np.ndarray) -> bool:
    """Equal bytes; a NaN code may differ only in its sign bit."""
    a, b = np.asarray(a, np.uint8), np.asarray(b, np.uint8)
    nan = ((a & 0x7F) == 0x7F) & ((b & 0x7F) == 0x7F)
    return bool(np.all((a == b) | nan))


rows_of, fp8_step, fp8_ref = H.rows_of, H.fp8_step, H.fp8_ref


def test_write_fp8_all_bf16_patterns():
    """Every bf16 bit pattern (NaNs, infinities, subnormals, values far beyond 448 x
    scale) quantises to the oracle's code."""
    o = H.ops()
    NB, Hkv, D = 64, 4, 128
    T = 65536 // (Hkv * D)
    kn = torch.arange(65536, dtype=torch.int32).sub(32768).to(torch.int16).view(T, Hkv, D)
    vn = kn.flip(0).contiguous()
    g = torch.Generator().manual_seed(3)
    slots = torch.randperm(NB * BS, generator=g)[:T].to(torch.int64)
    kq = torch.zeros(NB, Hkv, BS, D, dtype=torch.uint8, device="cuda")
    vq = torch.zeros_like(kq)
    for ks, vs in ((K_SCALE, V_SCALE), (1.0, 3.0e-3), (0.5, 448.0)):
        o.paged_kv_write_fp8(kn.view(torch.bfloat16).cuda(), vn.view(torch.bfloat16).cuda(),
                             slots.cuda(), kq, vq, ks, vs)
        torch.cuda.synchronize()
        ko = np.zeros((NB, Hkv, BS, D), np.uint8)
        vo = np.zeros_like(ko)
        oracle.kv_write_fp8(ko, vo, kn.numpy().view(np.uint16), vn.numpy().view(np.uint16),
                            slots.numpy(), ks, vs)
        assert same_codes(kq.cpu().numpy(), ko) and same_codes(vq.cpu().numpy(), vo), (ks, vs)
        kq.zero_()
        vq.zero_()



@pytest.mark.parametrize("D,Hkv", [(48, 1), (64, 3), (96, 2), (128, 5), (256, 3), (512, 1)])
def test_write_fp8_head_dims(D, Hkv):
    """The quantising write at head dims whose row of 16-byte vectors is a power of two up
    to 32 (64, 128, 256: the lanes of a row trade V codes so each store round covers
    consecutive head-dim rows) and at the others (48, 96, 512: each lane stores its own
    codes), with one scale per cache and one per KV head: codes equal the oracle's byte
    for byte, slots out of order, some skipped (-1)."""
    o = H.ops()
    g = torch.Generator().manual_seed(D * 7 + Hkv)
    NB, T = 9, 40
    kn = (torch.randn(T, Hkv, D, generator=g) * 3).to(torch.bfloat16)
    vn = (torch.randn(T, Hkv, D, generator=g) * 2).to(torch.bfloat16)
    slots = torch.randperm(NB * BS, generator=g)[:T].to(torch.int64)
    slots[::7] = -1
    ks_h = (torch.rand(Hkv, generator=g) * 0.05 + 0.005).to(torch.float32)
    vs_h = (torch.rand(Hkv, generator=g) * 0.05 + 0.005).to(torch.float32)
    kn16, vn16 = kn.view(torch.int16).numpy().view(np.uint16), vn.view(torch.int16).numpy().view(np.uint16)
    for per_head in (False, True):
        kq = torch.zeros(NB, Hkv, BS, D, dtype=torch.uint8, device="cuda")
        vq = torch.zeros_like(kq)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        if per_head:
            o.paged_kv_write_fp8_per_head(kn.cuda(), vn.cuda(), slots.cuda(), kq, vq, ks_h.cuda(),
                                          vs_h.cuda(), err_flag=err)
            ks, vs = ks_h.numpy(), vs_h.numpy()
        else:
            o.paged_kv_write_fp8(kn.cuda(), vn.cuda(), slots.cuda(), kq, vq, K_SCALE, V_SCALE,
                                 err_flag=err)
            ks, vs = K_SCALE, V_SCALE
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        ko = np.zeros((NB, Hkv, BS, D), np.uint8)
        vo = np.zeros_like(ko)
        oracle.kv_write_fp8(ko, vo, kn16, vn16, slots.numpy(), ks, vs)
        assert same_codes(kq.cpu().numpy(), ko), (D, Hkv, per_head, "K")
        assert same_codes(vq.cpu().numpy(), vo), (D, Hkv, per_head, "V")

@pytest.mark.parametrize("cfg", [1, 2, 3, 4])
def test_fp8_config_parity(cfg):
    w = workloads.make_config(cfg, device="cpu" if cfg == 1 else "cuda")
    out, kq, vq, ko, vo, err = fp8_step(w)
    assert err == 0
    assert same_codes(kq, ko) and same_codes(vq, vo), "E4M3 write/copy not bit-exact"
    H.assert_attention_close(out, fp8_ref(w, ko, vo), f"fp8 config {cfg}")


def test_fp8_long_context_sampled():
    w = workloads.make_config(5, device="cuda")
    out, kq, vq, ko, vo, err = fp8_step(w)
    assert err == 0
    assert same_codes(kq, ko) and same_codes(vq, vo)
    sel = H.wide_pairs(w, n_short=256)  # all 512 long rows + 256 short ones
    assert len(sel) >= 768
    ref = fp8_ref(w, ko, vo, sel=sel)
    got = out[torch.as_tensor(sel[:, 0].astype(np.int64), device="cuda"),
              torch.as_tensor(sel[:, 1].astype(np.int64), device="cuda")]
    H.assert_attention_close(got, ref, "fp8 config 5 sample")


@pytest.mark.parametrize("cfg", [3, 5])
def test_fp8_auto_partition(cfg):
    """partition_size 0 (the plan picks 1536 / 4096-token partitions for these batches):
    config 3 in full, config 5 on every long row plus 256 short ones."""
    w = workloads.make_config(cfg, device="cuda")
    out, kq, vq, ko, vo, err = fp8_step(w, partition_size=0)
    assert err == 0
    sel = H.wide_pairs(w, n_short=256) if cfg == 5 else None
    ref = fp8_ref(w, ko, vo, sel=sel)
    got = out if sel is None else out[torch.as_tensor(sel[:, 0].astype(np.int64), device="cuda"),
                                      torch.as_tensor(sel[:, 1].astype(np.int64), device="cuda")]
    H.assert_attention_close(got, ref, f"fp8 config {cfg}, automatic split")


@pytest.mark.parametrize("G", [1, 2, 3, 8, 16])
@pytest.mark.parametrize("P", [48, 64, 512, 768, 8192])
def test_fp8_groups_and_partitions(G, P):
    ctx = [1, 2, 15, 16, 17, 33, 511, 512, 513, 1500, 2999]
    w = workloads.build("fp8-edges", ctx, 2 * G, 2, 128, seed=60 + G, device="cuda")
    out, kq, vq, ko, vo, err = fp8_step(w, partition_size=P)
    assert err == 0
    H.assert_attention_close(out, fp8_ref(w, ko, vo), f"fp8 G={G} P={P}")


def test_fp8_scales_and_magnitude():
    """Power-of-two and odd scales, large-magnitude queries."""
    w = workloads.build("fp8-big", [40, 600, 1500], 16, 2, 128, seed=71, device="cuda")
    w.q.mul_(30)
    for ks, vs in ((0.0625, 0.25), (0.0173, 0.0091)):
        out, kq, vq, ko, vo, err = fp8_step(w, ks, vs)
        assert err == 0
        H.assert_attention_close(out, fp8_ref(w, ko, vo, ks, vs), f"fp8 scales {ks} {vs}")


def test_fp8_bad_block_id_is_flagged_not_read():
    """A block id outside the pool (in the first or the second block of a two-block
    stage) is flagged and skipped; the other sequences are unaffected."""
    w = workloads.build("fp8-badblk", [40, 70, 100, 333], 8, 2, 128, seed=98, device="cuda")
    for pos in (2, 3):
        bt = torch.as_tensor(w.block_tables, dtype=torch.int32, device="cuda").clone()
        bt[1, pos] = w.num_blocks + 1000
        out, kq, vq, ko, vo, err = fp8_step(w, block_tables=bt)
        assert err & H.ops().DEV_BAD_BLOCK
        ref = fp8_ref(w, ko, vo)
        keep = [0, 2, 3]
        H.assert_attention_close(out[keep], ref[keep], f"untouched sequences (block {pos})")


@pytest.mark.parametrize("G", [1, 2, 8])
@pytest.mark.parametrize("P", [64, 512])
def test_fp8_head_dim_64(G, P):
    """head_dim 64 (64-byte E4M3 rows, the 64-byte swizzle): boundary contexts, groups and
    partitions, one scale per cache and one per KV head."""
    ctx = [1, 2, 15, 16, 17, 33, 511, 512, 513, 1500, 2999]
    w = workloads.build("fp8-d64", ctx, 2 * G, 2, 64, seed=90 + G, device="cuda")
    out, kq, vq, ko, vo, err = fp8_step(w, partition_size=P)
    assert err == 0
    assert same_codes(kq, ko) and same_codes(vq, vo)
    H.assert_attention_close(out, fp8_ref(w, ko, vo), f"fp8 d64 G={G} P={P}")
    ks, vs = np.array([0.02, 0.05], np.float32), np.array([0.015, 0.03], np.float32)
    out, kq, vq, ko, vo, err = fp8_step(w, ks, vs, partition_size=P)
    assert err == 0
    assert same_codes(kq, ko) and same_codes(vq, vo)
    H.assert_attention_close(out, fp8_ref(w, ko, vo, ks, vs), f"fp8 d64 per head G={G} P={P}")


def test_fp8_rejects_other_head_dims():
    o = H.ops()
    q = torch.zeros(1, 2, 96, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(4, 1, 16, 96, dtype=torch.uint8, device="cuda")
    ws = o.alloc_workspace(1, 2, 96, 16)
    with pytest.raises(o.PagedKVError):
        o.paged_attention_decode_fp8(q.clone(), q, kc, kc.clone(),
                                     torch.zeros(1, 1, dtype=torch.int32, device="cuda"),
                                     torch.ones(1, dtype=torch.int32, device="cuda"), 0.125, 1.0,
                                     1.0, 16, ws)


# ---- one scale per KV head ------------------------------------------------------------
@pytest.mark.parametrize("cfg", [2, 3, 4, 5])
def test_fp8_per_head_config_parity(cfg):
    """KV heads spread over 2^-3 .. 2^3 in range, each quantised with its own calibrated
    scale: the write/copy bytes match the oracle and the output is within tolerance."""
    w = workloads.make_config(cfg, device="cuda")
    Hkv = w.num_kv_heads
    H.spread_heads(w, [2.0 ** ((h % 7) - 3) for h in range(Hkv)])
    ks, vs = H.per_head_scales(w)
    assert len(set(ks.tolist())) > 1
    out, kq, vq, ko, vo, err = fp8_step(w, ks, vs)
    assert err == 0
    assert same_codes(kq, ko) and same_codes(vq, vo), "per-head E4M3 write/copy not bit-exact"
    if cfg in (2, 4):
        H.assert_attention_close(out, fp8_ref(w, ko, vo, ks, vs), f"fp8 per-head config {cfg}")
    else:
        sel = H.sample_pairs(w, n_short=256)
        got = out[torch.as_tensor(sel[:, 0].astype(np.int64), device="cuda"),
                  torch.as_tensor(sel[:, 1].astype(np.int64), device="cuda")]
        H.assert_attention_close(got, fp8_ref(w, ko, vo, ks, vs, sel=sel),
                                 f"fp8 per-head config {cfg} sample")


@pytest.mark.parametrize("G", [1, 3, 8, 16])
def test_fp8_per_head_groups(G):
    """Every query head of a group takes its KV head's scales (three KV heads with
    different scales; groups below, at and above the kernel's 8-row tile)."""
    ctx = [1, 16, 17, 513, 1500]
    w = workloads.build("fp8-ph", ctx, 3 * G, 3, 128, seed=120 + G, device="cuda")
    H.spread_heads(w, [0.25, 1.0, 8.0])
    ks = np.array([0.0005, 0.004, 0.03], np.float32)
    vs = np.array([0.03, 0.0007, 0.005], np.float32)
    for P in (64, 512):
        out, kq, vq, ko, vo, err = fp8_step(w, ks, vs, partition_size=P)
        assert err == 0
        assert same_codes(kq, ko) and same_codes(vq, vo)
        H.assert_attention_close(out, fp8_ref(w, ko, vo, ks, vs), f"fp8 per-head G={G} P={P}")


def test_fp8_per_head_equal_entries_match_per_cache():
    """Equal per-head entries write the same bytes as the one-scale write."""
    w = workloads.build("fp8-eq", [30, 300], 8, 2, 128, seed=131, device="cuda")
    _, kq1, vq1, _, _, err1 = fp8_step(w)
    _, kq2, vq2, _, _, err2 = fp8_step(w, [K_SCALE] * 2, [V_SCALE] * 2)
    assert err1 == err2 == 0
    assert np.array_equal(kq1, kq2) and np.array_equal(vq1, vq2)


def test_fp8_per_head_bad_scale_is_flagged():
    """A scale that is not > 0 is reported: the write skips that head's rows, attention
    flags it; the other KV head's rows are written and attended as usual."""
    o = H.ops()
    w = workloads.build("fp8-badscale", [20, 70], 8, 2, 128, seed=133, device="cuda",
                        poison=False)
    d = H.to_cuda(w)
    NB, Hkv, bs, D = w.k_cache.shape
    for bad in (0.0, -0.5, float("nan")):
        kq = torch.zeros(NB, Hkv, bs, D, dtype=torch.uint8, device="cuda")
        vq = torch.zeros_like(kq)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        kst = torch.tensor([K_SCALE, K_SCALE], dtype=torch.float32, device="cuda")
        vst = torch.tensor([V_SCALE, bad], dtype=torch.float32, device="cuda")
        o.paged_kv_write_fp8_per_head(H.rows_of(w.k_cache.cuda()), H.rows_of(w.v_cache.cuda()),
                                      torch.arange(NB * bs, device="cuda"), kq, vq, kst, vst,
                                      err_flag=err)
        torch.cuda.synchronize()
        assert int(err.item()) == o.DEV_BAD_SCALE, bad
        assert not kq[:, 1].any() and not vq[:, 1].any()  # head 1 untouched
        ko = np.zeros((NB, Hkv, bs, D), np.uint8)
        vo = np.zeros_like(ko)
        oracle.kv_write_fp8(ko, vo, H.u16(H.rows_of(w.k_cache.cpu())),
                            H.u16(H.rows_of(w.v_cache.cpu())), np.arange(NB * bs), K_SCALE,
                            V_SCALE)
        assert same_codes(kq.cpu().numpy()[:, 0], ko[:, 0])
        assert same_codes(vq.cpu().numpy()[:, 0], vo[:, 0])
        if bad != bad:  # NaN: the write check only
            continue
        err.zero_()
        out = torch.zeros(w.num_seqs, 8, D, dtype=torch.bfloat16, device="cuda")
        ws = o.alloc_workspace(w.num_seqs, 8, D, w.max_context_len, 64)
        o.paged_attention_decode_fp8_per_head(out, d["q"], kq, vq, d["bt"], d["ctx"], w.scale,
                                              kst, vst, w.max_context_len, ws, 64, err_flag=err)
        torch.cuda.synchronize()
        assert int(err.item()) == o.DEV_BAD_SCALE, bad
        ref = fp8_ref(w, ko, vo)
        H.assert_attention_close(out[:, :4], ref[:, :4], "heads of the good KV head")
