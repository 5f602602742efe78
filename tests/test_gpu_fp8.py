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
K_SCALE, V_SCALE = 0.02, 0.015


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def same_codes(a: np.ndarray, b: np.ndarray) -> bool:
    """Equal bytes; a NaN code may differ only in its sign bit."""
    a, b = np.asarray(a, np.uint8), np.asarray(b, np.uint8)
    nan = ((a & 0x7F) == 0x7F) & ((b & 0x7F) == 0x7F)
    return bool(np.all((a == b) | nan))


def rows_of(cache: torch.Tensor) -> torch.Tensor:
    """[NB][Hkv][16][D] -> [NB*16][Hkv][D] in slot order (to quantise a whole cache)."""
    NB, Hkv, bs, D = cache.shape
    return cache.permute(0, 2, 1, 3).reshape(NB * bs, Hkv, D).contiguous()


def fp8_step(w, ks=K_SCALE, vs=V_SCALE, partition_size=None):
    """Quantise the pre-step cache, then COW copy + new-token write + attention, on the
    GPU and in the oracle.  Returns (gpu_out, gpu k/v codes, oracle k/v codes, err)."""
    o = H.ops()
    dev = "cuda"
    NB, Hkv, bs, D = w.k_cache.shape
    kq = torch.zeros(NB, Hkv, bs, D, dtype=torch.uint8, device=dev)
    vq = torch.zeros_like(kq)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    slots_all = torch.arange(NB * bs, dtype=torch.int64, device=dev)
    o.paged_kv_write_fp8(rows_of(w.k_cache.to(dev)), rows_of(w.v_cache.to(dev)), slots_all, kq, vq,
                         ks, vs, err_flag=err)
    d = H.to_cuda(w)
    if d["pairs"].numel():
        o.paged_block_copy_fp8(kq, vq, d["pairs"], err_flag=err)
    if d["slots"].numel():
        o.paged_kv_write_fp8(d["k_new"], d["v_new"], d["slots"], kq, vq, ks, vs, err_flag=err)
    S, Hq, _ = d["q"].shape
    P = partition_size or w.partition_size
    out = torch.full((S, Hq, D), float("nan"), dtype=torch.bfloat16, device=dev)
    ws = o.alloc_workspace(S, Hq, D, w.max_context_len, P)
    o.paged_attention_decode_fp8(out, d["q"], kq, vq, d["bt"], d["ctx"], w.scale, ks, vs,
                                 w.max_context_len, ws, P, err_flag=err)
    torch.cuda.synchronize()
    # oracle
    ko = np.zeros((NB, Hkv, bs, D), np.uint8)
    vo = np.zeros_like(ko)
    oracle.kv_write_fp8(ko, vo, H.u16(rows_of(w.k_cache.cpu())), H.u16(rows_of(w.v_cache.cpu())),
                        np.arange(NB * bs), ks, vs)
    if w.cow_pairs.size:
        oracle.block_copy_fp8(ko, vo, w.cow_pairs)
    if w.slot_mapping.size:
        oracle.kv_write_fp8(ko, vo, H.u16(w.k_new), H.u16(w.v_new), w.slot_mapping, ks, vs)
    return out, kq.cpu().numpy(), vq.cpu().numpy(), ko, vo, int(err.item())


def fp8_ref(w, ko, vo, ks=K_SCALE, vs=V_SCALE, sel=None):
    return oracle.attention_fp8(H.u16(w.q), ko, vo, w.block_tables, w.context_lens, w.scale, ks,
                                vs, sel=sel, nthreads=H.NTHREADS)


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


@pytest.mark.parametrize("cfg", [1, 2, 3, 4])
def test_fp8_config_parity(cfg):
    w = workloads.make_config(cfg, device="cpu" if cfg == 1 else "cuda")
    if w.head_dim != 128:  # the E4M3 attention kernel takes head_dim 128
        w = workloads.build("tiny-d128", w.context_lens, w.num_q_heads, w.num_kv_heads, 128,
                            seed=1001, device="cpu", num_blocks=16)
    out, kq, vq, ko, vo, err = fp8_step(w)
    assert err == 0
    assert same_codes(kq, ko) and same_codes(vq, vo), "E4M3 write/copy not bit-exact"
    H.assert_attention_close(out, fp8_ref(w, ko, vo), f"fp8 config {cfg}")


def test_fp8_long_context_sampled():
    w = workloads.make_config(5, device="cuda")
    out, kq, vq, ko, vo, err = fp8_step(w)
    assert err == 0
    assert same_codes(kq, ko) and same_codes(vq, vo)
    sel = H.sample_pairs(w, n_short=32)
    ref = fp8_ref(w, ko, vo, sel=sel)
    got = out[torch.as_tensor(sel[:, 0].astype(np.int64), device="cuda"),
              torch.as_tensor(sel[:, 1].astype(np.int64), device="cuda")]
    H.assert_attention_close(got, ref, "fp8 config 5 sample")


@pytest.mark.parametrize("G", [1, 2, 3, 8, 16])
@pytest.mark.parametrize("P", [64, 512, 8192])
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


def test_fp8_rejects_other_head_dims():
    o = H.ops()
    q = torch.zeros(1, 2, 64, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(4, 1, 16, 64, dtype=torch.uint8, device="cuda")
    ws = o.alloc_workspace(1, 2, 64, 16)
    with pytest.raises(o.PagedKVError):
        o.paged_attention_decode_fp8(q.clone(), q, kc, kc.clone(),
                                     torch.zeros(1, 1, dtype=torch.int32, device="cuda"),
                                     torch.ones(1, dtype=torch.int32, device="cuda"), 0.125, 1.0,
                                     1.0, 16, ws)
