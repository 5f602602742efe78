"""GPU parity of the fused decode step (paged_decode_step, paged_decode_step_fp8) through
the C ABI.  After the step the caches are bit-exact against the oracle's copies followed
by its writes; attention matches the fp64 oracle within |err| <= 1e-2 + 1e-2 |ref| (mean
<= 2e-3); and the output equals the three separate calls' output bit for bit (the same
partition and merge kernels run on the same plan)."""
import numpy as np
import pytest
import torch

import gpu_helpers as H
import oracle
from paged_kv_cache_272_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def fused_step(w, d=None, pairs=None, slots=None, k_new=None, v_new=None, partition_size=None):
    """paged_decode_step on device copies of the workload; returns (out, k, v, err)."""
    P = w.partition_size if partition_size is None else partition_size  # 0: automatic
    o = H.ops()
    d = d or H.to_cuda(w)
    pairs = d["pairs"] if pairs is None else pairs
    slots = d["slots"] if slots is None else slots
    k_new = d["k_new"] if k_new is None else k_new
    v_new = d["v_new"] if v_new is None else v_new
    S, Hq, D = d["q"].shape
    out = torch.full((S, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = o.alloc_workspace(S, Hq, D, w.max_context_len, P)
    ws.fill_(0xFF)  # stale workspace content must not matter
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o.paged_decode_step(out, d["q"], d["k"], d["v"], d["bt"], d["ctx"], w.scale,
                        w.max_context_len, ws, k_new=k_new, v_new=v_new, slot_mapping=slots,
                        block_pairs=pairs, partition_size=P, err_flag=err)
    torch.cuda.synchronize()
    return out, d["k"], d["v"], int(err.item())


def _check(w, out, k, v, err, sel=None):
    assert err == 0
    ko, vo = H.oracle_caches(w)
    assert np.array_equal(H.u16(k), ko), "fused copy + write not bit-exact (K)"
    assert np.array_equal(H.u16(v), vo), "fused copy + write not bit-exact (V)"
    ref = H.oracle_out(w, ko, vo, sel=sel)
    got = out if sel is None else out[torch.as_tensor(sel[:, 0].astype(np.int64), device="cuda"),
                                      torch.as_tensor(sel[:, 1].astype(np.int64), device="cuda")]
    H.assert_attention_close(got, ref, w.name)


@pytest.mark.parametrize("P", [None, 0])
@pytest.mark.parametrize("cfg", [1, 2, 3, 4])
def test_step_configs(cfg, P):
    """The workload's 512-token split, and the automatic one (P = 0)."""
    w = workloads.make_config(cfg, device="cpu" if cfg == 1 else "cuda")
    out, k, v, err = fused_step(w, partition_size=P)
    _check(w, out, k, v, err)
    # the three separate calls give the same bits
    out3, k3, v3, err3 = H.gpu_step(w, partition_size=P)
    assert err3 == 0
    assert torch.equal(out.view(torch.int16), out3.view(torch.int16))
    assert torch.equal(k.view(torch.int16), k3.view(torch.int16))


def test_step_config5_sampled():
    w = workloads.make_config(5, device="cuda")
    out, k, v, err = fused_step(w)
    _check(w, out, k, v, err, sel=H.sample_pairs(w, n_short=64))
    assert torch.isfinite(out.float()).all()


def _free_blocks(w):
    used = np.zeros(w.num_blocks, dtype=bool)
    for s in range(w.num_seqs):
        n = (int(w.context_lens[s]) + 15) // 16
        used[w.block_tables[s, :n]] = True
    if w.cow_pairs.size:
        used[w.cow_pairs.reshape(-1)] = True
    return np.flatnonzero(~used)


def test_step_writes_into_copied_blocks():
    """New tokens that land in a copy's source block, in a destination block's other rows,
    several destinations of one source, and plain tokens, all in one step: every copy
    happens before every write."""
    w = workloads.build("step-conflicts", [40, 53, 70, 100, 131, 77], 16, 2, 128, seed=31,
                        shared_prefix_tokens=32, cow_last_block=True, free_fraction=0.6)
    assert w.cow_pairs.shape[0] >= 3
    free = _free_blocks(w)
    src0, dst0 = (int(x) for x in w.cow_pairs[0])
    src1 = int(w.cow_pairs[1, 0])
    extra_pairs = [(src0, int(free[0])), (src0, int(free[1])), (src1, int(free[2]))]
    pairs = np.concatenate([w.cow_pairs, np.asarray(extra_pairs, np.int32)])
    used_slots = set(int(x) for x in w.slot_mapping)
    extra_slots = []
    for b in (src0, src1, dst0, int(free[1]), int(free[3])):
        for r in (15, 3):  # rows not written by the sequences' own tokens
            sl = b * 16 + r
            if sl not in used_slots:
                extra_slots.append(sl)
                used_slots.add(sl)
    g = torch.Generator().manual_seed(5)
    T0 = w.slot_mapping.shape[0]
    kx = torch.randn(len(extra_slots), 2, 128, generator=g).to(torch.bfloat16)
    vx = torch.randn(len(extra_slots), 2, 128, generator=g).to(torch.bfloat16)
    w.k_new = torch.cat([w.k_new, kx])
    w.v_new = torch.cat([w.v_new, vx])
    w.slot_mapping = np.concatenate([w.slot_mapping, np.asarray(extra_slots, np.int64)])
    w.cow_pairs = pairs
    assert w.slot_mapping.shape[0] == T0 + len(extra_slots)
    out, k, v, err = fused_step(w)
    _check(w, out, k, v, err)


def test_step_more_pairs_than_the_prologue_takes():
    """1100 copy pairs (beyond the prologue's table): the copies take a launch of their own
    first; the result is unchanged."""
    ctx = [34 + (i % 7) for i in range(1100)]
    w = workloads.build("step-many-pairs", ctx, 2, 1, 64, seed=32, cow_last_block=True,
                        shared_prefix_tokens=0)
    assert w.cow_pairs.shape[0] == 1100
    out, k, v, err = fused_step(w)
    _check(w, out, k, v, err)


def test_step_without_tokens_pairs_or_sequences():
    o = H.ops()
    w = workloads.build("step-bare", [5, 17, 600], 8, 2, 128, seed=33, write_new_token=False)
    d = H.to_cuda(w)
    out, k, v, err = fused_step(w, d=d, pairs=torch.zeros(0, 2, dtype=torch.int32,
                                                              device="cuda"),
                                slots=torch.zeros(0, dtype=torch.int64, device="cuda"))
    _check(w, out, k, v, err)
    # no sequences: the copies and the write still run
    w = workloads.build("step-noseq", [40, 53], 8, 2, 128, seed=34, shared_prefix_tokens=32,
                        cow_last_block=True)
    d = H.to_cuda(w)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    empty_q = torch.zeros(0, 8, 128, dtype=torch.bfloat16, device="cuda")
    o.paged_decode_step(torch.zeros_like(empty_q), empty_q, d["k"], d["v"],
                        torch.zeros(0, d["bt"].shape[1], dtype=torch.int32, device="cuda"),
                        torch.zeros(0, dtype=torch.int32, device="cuda"), w.scale, 0,
                        torch.zeros(256, dtype=torch.uint8, device="cuda"), k_new=d["k_new"],
                        v_new=d["v_new"], slot_mapping=d["slots"], block_pairs=d["pairs"],
                        err_flag=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    ko, vo = H.oracle_caches(w)
    assert np.array_equal(H.u16(d["k"]), ko) and np.array_equal(H.u16(d["v"]), vo)


def test_step_flags_bad_slot_and_pair():
    o = H.ops()
    w = workloads.build("step-bad", [40, 53, 70], 8, 2, 128, seed=35, shared_prefix_tokens=32,
                        cow_last_block=True, free_fraction=0.5)
    d = H.to_cuda(w)
    free = _free_blocks(w)
    k0, v0 = d["k"].clone(), d["v"].clone()
    bad_pairs = torch.cat([d["pairs"], torch.tensor([[w.num_blocks + 5, int(free[0])]],
                                                     dtype=torch.int32, device="cuda")])
    bad_slots = d["slots"].clone()
    bad_slots[0] = w.num_blocks * 16 + 3
    out, k, v, err = fused_step(w, d=d, pairs=bad_pairs, slots=bad_slots)
    assert err & o.DEV_BAD_SLOT and err & o.DEV_BAD_BLOCK
    # everything else happened: the valid pairs copied, the other tokens written
    kh, vh = H.u16(k0).copy(), H.u16(v0).copy()
    oracle.block_copy(kh, vh, w.cow_pairs)
    oracle.kv_write(kh, vh, H.u16(w.k_new[1:]), H.u16(w.v_new[1:]), w.slot_mapping[1:])
    assert np.array_equal(H.u16(k), kh) and np.array_equal(H.u16(v), vh)


@pytest.mark.parametrize("per_head", [False, True])
@pytest.mark.parametrize("cfg", [3, 4])
def test_step_fp8(cfg, per_head):
    o = H.ops()
    w = workloads.make_config(cfg, device="cuda")
    NB, Hkv, bs, D = w.k_cache.shape
    if per_head:
        ks = np.array([0.02 * (1 + h / 8) for h in range(Hkv)], np.float32)
        vs = np.array([0.015 * (1 + h / 5) for h in range(Hkv)], np.float32)
        ksa, vsa = torch.as_tensor(ks, device="cuda"), torch.as_tensor(vs, device="cuda")
    else:
        ks, vs = H.K_SCALE, H.V_SCALE
        ksa, vsa = ks, vs
    # the pre-step cache quantised by the library's own write, as in the E4M3 tests
    kq = torch.zeros(NB, Hkv, bs, D, dtype=torch.uint8, device="cuda")
    vq = torch.zeros_like(kq)
    slots_all = torch.arange(NB * bs, dtype=torch.int64, device="cuda")
    if per_head:
        o.paged_kv_write_fp8_per_head(H.rows_of(w.k_cache), H.rows_of(w.v_cache), slots_all, kq,
                                      vq, ksa, vsa)
    else:
        o.paged_kv_write_fp8(H.rows_of(w.k_cache), H.rows_of(w.v_cache), slots_all, kq, vq, ks,
                             vs)
    d = H.to_cuda(w)
    S, Hq, _ = d["q"].shape
    out = torch.full((S, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = o.alloc_workspace(S, Hq, D, w.max_context_len, w.partition_size)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o.paged_decode_step_fp8(out, d["q"], kq, vq, d["bt"], d["ctx"], w.scale, ksa, vsa,
                            w.max_context_len, ws, k_new=d["k_new"], v_new=d["v_new"],
                            slot_mapping=d["slots"], block_pairs=d["pairs"],
                            partition_size=w.partition_size, err_flag=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    ko = np.zeros((NB, Hkv, bs, D), np.uint8)
    vo = np.zeros_like(ko)
    oracle.kv_write_fp8(ko, vo, H.u16(H.rows_of(w.k_cache.cpu())), H.u16(H.rows_of(w.v_cache.cpu())),
                        np.arange(NB * bs), ks, vs)
    if w.cow_pairs.size:
        oracle.block_copy_fp8(ko, vo, w.cow_pairs)
    oracle.kv_write_fp8(ko, vo, H.u16(w.k_new), H.u16(w.v_new), w.slot_mapping, ks, vs)
    assert np.array_equal(kq.cpu().numpy(), ko) and np.array_equal(vq.cpu().numpy(), vo)
    H.assert_attention_close(out, H.fp8_ref(w, ko, vo, ks, vs), f"fp8 step config {cfg}")
