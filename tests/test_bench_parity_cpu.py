"""The benchmark's parity report (its own output against the oracle on sampled rows)
passes the oracle's own rounded output and flags a planted error, for the decode
(bf16 and E4M3 caches, with copy-on-write) and chunked-prefill lines.  CPU only."""
import os
import sys

import numpy as np
import torch

import oracle
from paged_kv_cache_272_gb300 import workloads

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def u16(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def step_caches(w, fp8):
    """Post-step caches built here independently: copy-on-write, then the write."""
    k, v = u16(w.k_cache).copy(), u16(w.v_cache).copy()
    if fp8:
        NB, Hkv, bs, D = k.shape
        rows = lambda c: np.ascontiguousarray(c.transpose(0, 2, 1, 3).reshape(NB * bs, Hkv, D))
        kq, vq = np.zeros(k.shape, np.uint8), np.zeros(k.shape, np.uint8)
        oracle.kv_write_fp8(kq, vq, rows(k), rows(v), np.arange(NB * bs), bench.FP8_K_SCALE,
                            bench.FP8_V_SCALE)
        k, v = kq, vq
    if w.cow_pairs.size:
        (oracle.block_copy_fp8 if fp8 else oracle.block_copy)(k, v, w.cow_pairs)
    if w.slot_mapping.size:
        if fp8:
            oracle.kv_write_fp8(k, v, u16(w.k_new), u16(w.v_new), w.slot_mapping,
                                bench.FP8_K_SCALE, bench.FP8_V_SCALE)
        else:
            oracle.kv_write(k, v, u16(w.k_new), u16(w.v_new), w.slot_mapping)
    return k, v


def test_decode_parity_report():
    w = workloads.build("parity", [40, 70, 100, 17], 8, 2, 128, seed=5, cow_last_block=True)
    for fp8 in (False, True):
        k, v = step_caches(w, fp8)
        if fp8:
            ref = oracle.attention_fp8(u16(w.q), k, v, w.block_tables, w.context_lens, w.scale,
                                       bench.FP8_K_SCALE, bench.FP8_V_SCALE)
        else:
            ref = oracle.attention(u16(w.q), k, v, w.block_tables, w.context_lens, w.scale)
        out = torch.from_numpy(ref).to(torch.bfloat16)
        r = bench.sample_parity(w, out, fp8, n_pairs=24)
        assert r["within_tolerance"] and r["elements_out_of_tolerance"] == 0, r
        bad = out.clone()
        bad[int(np.argmax(w.context_lens))] += 0.5  # the longest sequence is always sampled
        r = bench.sample_parity(w, bad, fp8, n_pairs=24)
        assert not r["within_tolerance"] and r["elements_out_of_tolerance"] > 0, r


def test_prefill_parity_report():
    w = workloads.make_prefill_config(1)
    k, v = u16(w.k_cache).copy(), u16(w.v_cache).copy()
    oracle.kv_write(k, v, u16(w.k_new), u16(w.v_new), w.slot_mapping)
    ref = oracle.attention_prefill(u16(w.q), k, v, w.block_tables, w.context_lens,
                                   w.query_start, w.scale)
    out = torch.from_numpy(ref).to(torch.bfloat16)
    assert bench.prefill_sample_parity(w, out, n_rows=32)["within_tolerance"]
    bad = out.clone()
    bad[int(w.query_start[1]) - 1] -= 0.5  # a chunk's last token is always sampled
    assert not bench.prefill_sample_parity(w, bad, n_rows=32)["within_tolerance"]
