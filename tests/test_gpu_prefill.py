"""Chunked prefill through the C ABI: the chunk's K/V written with paged_kv_write, then
paged_attention_prefill, against the fp64 oracle on the same seeded inputs
(|err| <= 1e-2 + 1e-2 |ref| per element, mean <= 2e-3)."""
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


@pytest.fixture(params=["tc", "tc_sep", "tc_pair", "tc_2sm", "mma"])
def variant(request):
    """Run a test with each prefill kernel: tcgen05 with one 128-row tile per CTA, tcgen05
    with two tiles per CTA sharing the K/V tiles, tcgen05 on SM pairs (head_dim 128; 64
    runs the one-tile kernel), and mma.sync (all take head_dim 64 and 128)."""
    o = H.ops()
    prev = o.set_prefill_variant({"tc": o.PKV_PREFILL_TC, "tc_pair": o.PKV_PREFILL_TC_PAIR,
                                  "tc_2sm": o.PKV_PREFILL_TC_2SM, "tc_sep": o.PKV_PREFILL_TC_SEP,
                                  "mma": o.PKV_PREFILL_MMA}[request.param])
    yield request.param
    o.set_prefill_variant(prev)


def dev(w):
    d = "cuda"
    return dict(k=w.k_cache.to(d).contiguous().clone(), v=w.v_cache.to(d).contiguous().clone(),
                q=w.q.to(d).contiguous(), k_new=w.k_new.to(d).contiguous(),
                v_new=w.v_new.to(d).contiguous(),
                slots=torch.as_tensor(w.slot_mapping, dtype=torch.int64, device=d),
                bt=torch.as_tensor(w.block_tables, dtype=torch.int32, device=d),
                ctx=torch.as_tensor(w.context_lens, dtype=torch.int32, device=d),
                qs=torch.as_tensor(w.query_start, dtype=torch.int32, device=d))


def gpu_prefill(w, d=None, max_query_len=None, context_lens=None, query_start=None,
                block_tables=None):
    """write -> prefill through the C ABI.  Returns (out, err)."""
    o = H.ops()
    d = d or dev(w)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    if d["slots"].numel():
        o.paged_kv_write(d["k_new"], d["v_new"], d["slots"], d["k"], d["v"], err_flag=err)
    T, Hq, D = d["q"].shape
    out = torch.full((T, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    o.paged_attention_prefill(out, d["q"], d["k"], d["v"],
                              d["bt"] if block_tables is None else block_tables,
                              d["ctx"] if context_lens is None else context_lens,
                              d["qs"] if query_start is None else query_start, w.scale,
                              w.max_query_len if max_query_len is None else max_query_len,
                              err_flag=err)
    torch.cuda.synchronize()
    return out, int(err.item())


def oracle_prefill(w, sel=None):
    k, v = H.u16(w.k_cache).copy(), H.u16(w.v_cache).copy()
    if w.slot_mapping.size:
        oracle.kv_write(k, v, H.u16(w.k_new), H.u16(w.v_new), w.slot_mapping)
    return oracle.attention_prefill(H.u16(w.q), k, v, w.block_tables, w.context_lens,
                                    w.query_start, w.scale, sel=sel, nthreads=H.NTHREADS)


def sample_rows(w, n=384, seed=0):
    """(token, head) pairs: the first and last token of every chunk (one head per KV
    head) plus random rows."""
    rng = np.random.default_rng(seed)
    G = w.num_q_heads // w.num_kv_heads
    pairs = []
    for s in range(w.num_seqs):
        for t in (int(w.query_start[s]), int(w.query_start[s + 1]) - 1):
            if w.query_start[s + 1] > w.query_start[s]:
                pairs += [(t, g * G + int(rng.integers(G))) for g in range(w.num_kv_heads)]
    for _ in range(n):
        pairs.append((int(rng.integers(w.num_tokens)), int(rng.integers(w.num_q_heads))))
    return np.array(pairs, dtype=np.int32)


def test_prefill_tiny_config():
    w = workloads.make_prefill_config(1)
    out, err = gpu_prefill(w)
    assert err == 0
    H.assert_attention_close(out, oracle_prefill(w), "prefill config 1")


@pytest.mark.parametrize("cfg", [2, 3, 4])
def test_prefill_full_size_sampled(cfg, variant):
    w = workloads.make_prefill_config(cfg, device="cuda")
    out, err = gpu_prefill(w)
    assert err == 0
    assert torch.isfinite(out.float()).all(), "non-finite rows"
    sel = sample_rows(w)
    got = out[torch.as_tensor(sel[:, 0].astype(np.int64), device="cuda"),
              torch.as_tensor(sel[:, 1].astype(np.int64), device="cuda")]
    H.assert_attention_close(got, oracle_prefill(w, sel=sel), f"prefill config {cfg}")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 3, 8, 16])
def test_prefill_shapes(G, D, variant):
    """Ragged chunk and context lengths around the 64-row and 64-key tile edges, a
    decode row (L = 1), a whole prompt (L = ctx), contexts not a multiple of 16."""
    ctx = [1, 16, 17, 64, 65, 130, 200, 300, 77]
    L = [1, 16, 9, 64, 33, 65, 1, 129, 77]
    w = workloads.build_prefill("prefill-shapes", ctx, L, 2 * G, 2, D, seed=90 + G + D,
                                device="cuda")
    out, err = gpu_prefill(w)
    assert err == 0
    H.assert_attention_close(out, oracle_prefill(w), f"prefill G={G} D={D}")


def test_prefill_empty_chunks_and_bound(variant):
    """Sequences with no new token produce nothing; max_query_len above every chunk only
    adds CTAs that exit; rows outside every chunk stay untouched."""
    ctx, L = [40, 10, 90, 5], [0, 10, 0, 3]
    w = workloads.build_prefill("prefill-empty", ctx, L, 4, 2, 128, seed=95, device="cuda")
    out, err = gpu_prefill(w, max_query_len=200)
    assert err == 0
    H.assert_attention_close(out, oracle_prefill(w), "prefill with empty chunks")


def test_prefill_chunks_match_whole_prompt(variant):
    """A prompt prefilled in three chunks (three calls, growing context) gives the rows
    of the single whole-prompt call."""
    N, cuts = 300, [0, 100, 228, 300]
    w = workloads.build_prefill("prefill-whole", [N], [N], 16, 2, 128, seed=96, device="cuda")
    d = dev(w)
    whole, err = gpu_prefill(w, d)
    assert err == 0
    o = H.ops()
    for a, b in zip(cuts[:-1], cuts[1:]):
        part = torch.full((b - a, 16, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        o.paged_attention_prefill(part, d["q"][a:b].contiguous(), d["k"], d["v"], d["bt"],
                                  torch.tensor([b], dtype=torch.int32, device="cuda"),
                                  torch.tensor([0, b - a], dtype=torch.int32, device="cuda"),
                                  w.scale, b - a)
        torch.cuda.synchronize()
        assert torch.equal(part, whole[a:b]), (a, b)


def test_prefill_decode_rows_match_decode_kernel(variant):
    """L = 1 everywhere is a decode step: the prefill kernel and the decode path agree
    with the oracle (and so within twice the tolerance with each other)."""
    ctx = [5, 100, 700, 1500]
    w = workloads.build_prefill("prefill-decode", ctx, [1] * 4, 8, 1, 128, seed=97,
                                device="cuda")
    d = dev(w)
    out, err = gpu_prefill(w, d)
    assert err == 0
    ref = oracle_prefill(w)
    H.assert_attention_close(out, ref, "prefill L=1")
    o = H.ops()
    dec = torch.empty_like(out)
    ws = o.alloc_workspace(4, 8, 128, max(ctx))
    o.paged_attention_decode(dec, d["q"], d["k"], d["v"], d["bt"], d["ctx"], w.scale, max(ctx),
                             ws)
    torch.cuda.synchronize()
    H.assert_attention_close(dec, ref, "decode of the same rows")


def test_prefill_flags_bad_inputs(variant):
    """A chunk longer than its context and a block id outside the pool are reported in
    the error flag (the kernel skips them; nothing faults)."""
    ctx, L = [40, 30], [8, 8]
    w = workloads.build_prefill("prefill-bad", ctx, L, 4, 2, 128, seed=98, device="cuda")
    d = dev(w)
    bad_ctx = torch.tensor([5, 30], dtype=torch.int32, device="cuda")
    _, err = gpu_prefill(w, d, context_lens=bad_ctx)
    assert err & H.ops().DEV_BAD_CONTEXT
    bt = d["bt"].clone()
    bt[1, 0] = w.num_blocks + 3
    _, err = gpu_prefill(w, dev(w), block_tables=bt)
    assert err & H.ops().DEV_BAD_BLOCK
    _, err = gpu_prefill(w, dev(w), max_query_len=4)  # chunks longer than the bound
    assert err & H.ops().DEV_BAD_CONTEXT


def test_prefill_long_context_rows():
    """A short chunk after a long cached context (many key tiles, lazy rescaling of the
    output as the running maximum grows) and a chunk spanning several 128-row tiles."""
    o = H.ops()
    ctx, L = [9000, 3000, 700], [40, 300, 129]
    w = workloads.build_prefill("prefill-long", ctx, L, 16, 2, 128, seed=99, device="cuda")
    w.q.mul_(4)  # sharper softmax: the running maximum moves more
    for v in (o.PKV_PREFILL_TC, o.PKV_PREFILL_TC_SEP, o.PKV_PREFILL_TC_PAIR, o.PKV_PREFILL_TC_2SM,
              o.PKV_PREFILL_MMA):
        prev = o.set_prefill_variant(v)
        try:
            out, err = gpu_prefill(w)
        finally:
            o.set_prefill_variant(prev)
        assert err == 0
        sel = sample_rows(w, n=256, seed=5)
        got = out[torch.as_tensor(sel[:, 0].astype(np.int64), device="cuda"),
                  torch.as_tensor(sel[:, 1].astype(np.int64), device="cuda")]
        H.assert_attention_close(got, oracle_prefill(w, sel=sel), f"prefill long variant {v}")
