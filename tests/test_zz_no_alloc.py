"""The allocation-free attention entry point against the fp64 oracle and the regular one.

paged_attention_decode_noalloc serves callers that cannot allocate device memory (no
cudaMalloc on their thread, memory owned by another runtime, a stream someone else is
capturing): its split-K scratch is a fixed array inside the library.  This file is
collected last so a run that stops at the first failure has run everything else; it
also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_272_gb300 import workloads

pytestmark = pytest.mark.gpu

ATOL, RTOL, MEAN_TOL = 1e-2, 1e-2, 2e-3
ERR_WORKSPACE = -5


def _dev(w, ops):
    """Device inputs of one decode step, with the step's new token already written
    (the workloads leave that slot as NaN until the write)."""
    d = "cuda"
    t = dict(q=w.q.to(d).contiguous(), k=w.k_cache.to(d).contiguous(),
             v=w.v_cache.to(d).contiguous(),
             bt=torch.as_tensor(w.block_tables, dtype=torch.int32, device=d),
             ctx=torch.as_tensor(w.context_lens, dtype=torch.int32, device=d))
    ops.paged_kv_write(w.k_new.to(d).contiguous(), w.v_new.to(d).contiguous(),
                       torch.as_tensor(w.slot_mapping, device=d), t["k"], t["v"])
    return t


def _noalloc(lib, out, d, w, err):
    S, Hq, D = d["q"].shape
    NB, Hkv, bs, _ = d["k"].shape
    return lib.paged_attention_decode_noalloc(
        out.data_ptr(), d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(),
        d["bt"].data_ptr(), d["ctx"].data_ptr(), S, d["bt"].shape[1], Hq, Hkv, D, bs, NB,
        ctypes.c_float(w.scale), w.partition_size, w.max_context_len, err.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


def _regular(ops, d, w, err):
    S, Hq, D = d["q"].shape
    out = torch.empty(S, Hq, D, dtype=torch.bfloat16, device="cuda")
    ws = ops.alloc_workspace(S, Hq, D, w.max_context_len, w.partition_size)
    ops.paged_attention_decode(out, d["q"], d["k"], d["v"], d["bt"], d["ctx"], w.scale,
                               w.max_context_len, ws, w.partition_size, err_flag=err)
    return out


def _close(a, b, what):
    a = a.float().cpu().double().numpy()
    b = b.float().cpu().double().numpy()
    assert np.all(np.isfinite(a)) and np.all(np.isfinite(b)), what
    e = np.abs(a - b)
    assert np.all(e <= ATOL + RTOL * np.abs(b)), f"{what}: max err {e.max()}"
    assert e.mean() <= MEAN_TOL, f"{what}: mean err {e.mean()}"


def _u16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _oracle(w):
    """fp64 oracle output of the step: the new token written into host copies of the
    caches, then attention over every sequence and head."""
    k, v = _u16(w.k_cache).copy(), _u16(w.v_cache).copy()
    oracle.kv_write(k, v, _u16(w.k_new), _u16(w.v_new), w.slot_mapping)
    return oracle.attention(_u16(w.q), k, v, w.block_tables, w.context_lens, w.scale,
                            nthreads=8)


def _close_ref(a, ref, what):
    a = a.float().cpu().double().numpy().reshape(ref.shape)
    e = np.abs(a - ref)
    assert np.all(e <= ATOL + RTOL * np.abs(ref)), f"{what}: max err {e.max()}"
    assert e.mean() <= MEAN_TOL, f"{what}: mean err {e.mean()}"


def test_noalloc_matches_regular_entry_point_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_272_gb300 import ops
    lib = ops.lib
    # Two different decode steps in a row through the same fixed scratch: the second
    # must not see anything the first left behind.
    steps = [workloads.make_config(2, device="cuda"),
             workloads.build("noalloc-gqa", [1, 17, 511, 513, 2000, 3001], 64, 8, 128, seed=5,
                             device="cuda")]
    for i, w in enumerate(steps):
        d = _dev(w, ops)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        ref = _regular(ops, d, w, err)
        out = torch.full_like(ref, float("nan"))
        rc = _noalloc(lib, out, d, w, err)
        assert rc == 0, ops.lib.paged_kv_strerror(rc)
        torch.cuda.synchronize()
        assert err.item() == 0
        _close(out, ref, f"call {i + 1}")
        _close_ref(out, _oracle(w), f"call {i + 1} against the oracle")


def test_noalloc_rejects_sizes_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_272_gb300 import ops
    w = workloads.make_config(3, device="cuda")  # needs far more than the fixed scratch
    need = ops.paged_attention_workspace_size(w.num_seqs, w.num_q_heads, w.head_dim,
                                              w.max_context_len, w.partition_size)
    assert need > 16 * 2 ** 20
    d = _dev(w, ops)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.zeros(w.num_seqs, w.num_q_heads, w.head_dim, dtype=torch.bfloat16,
                      device="cuda")
    assert _noalloc(ops.lib, out, d, w, err) == ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(out == 0) and err.item() == 0
