"""fp64 CPU oracle for the paged KV-cache decode path.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this package; the product path never does.  It shares
no code with the CUDA library under ``paged_kv_cache_272_gb300/``.

The arithmetic lives in ``oracle.c`` (plain loops, fp64); this module only compiles
it with gcc and marshals numpy arrays through ctypes.  ``block_manager.py`` holds the
plain-Python reference of the host block manager.

Every bf16 tensor crosses this boundary as its raw uint16 bit pattern, so the oracle
reads exactly the bytes the GPU reads.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()
ABI_VERSION = 2


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile ``oracle.c`` into a shared library with gcc (OpenMP for the
    multi-threaded CPU baseline).  Returns the library path."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", *extra_flags, src,
           "-o", out + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


def load(path: str | None = None):
    """Load (building first if needed) and return the ctypes handle."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
    return _lib


def _declare(lib):
    P = ctypes.c_void_p
    I = ctypes.c_int
    lib.oracle_abi_version.restype = I
    if lib.oracle_abi_version() != ABI_VERSION:
        raise OracleError(f"stale oracle library (ABI {lib.oracle_abi_version()}, "
                          f"expected {ABI_VERSION}): rebuild it with build(force=True)")
    lib.oracle_kv_write.argtypes = [P, P, P, P, P, I, I, I, I, I]
    lib.oracle_kv_write.restype = I
    lib.oracle_block_copy.argtypes = [P, P, P, I, I, I, I, I]
    lib.oracle_block_copy.restype = I
    lib.oracle_attention.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, ctypes.c_double,
                                     P, I, I]
    lib.oracle_attention.restype = I
    lib.oracle_kv_bytes_per_token.argtypes = [I, I, I, I]
    lib.oracle_kv_bytes_per_token.restype = ctypes.c_int64
    lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_decode.restype = ctypes.c_double
    lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
    lib.oracle_e4m3_encode.restype = ctypes.c_uint8
    lib.oracle_kv_write_fp8.argtypes = [P, P, P, P, P, I, I, I, I, I, P, P]
    lib.oracle_kv_write_fp8.restype = I
    lib.oracle_block_copy_fp8.argtypes = [P, P, P, I, I, I, I, I]
    lib.oracle_block_copy_fp8.restype = I
    lib.oracle_attention_fp8.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, ctypes.c_double,
                                         P, P, P, I, I]
    lib.oracle_attention_fp8.restype = I
    lib.oracle_attention_prefill.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, I,
                                             ctypes.c_double, P, I, I]
    lib.oracle_attention_prefill.restype = I
    return lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def _u16(a) -> np.ndarray:
    """Raw bf16 bit patterns as a contiguous uint16 array (numpy or torch input)."""
    if hasattr(a, "detach"):  # torch tensor
        import torch
        a = a.detach().cpu().contiguous()
        assert a.dtype == torch.bfloat16, a.dtype
        return a.view(torch.int16).numpy().view(np.uint16)
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, a.dtype
    return a


class OracleError(RuntimeError):
    pass


def _check(rc: int, what: str):
    if rc != 0:
        raise OracleError(f"{what} failed with code {rc}")


def kv_write(k_cache: np.ndarray, v_cache: np.ndarray, k_new, v_new, slot_mapping,
             lib=None) -> None:
    """In place: K/V cache[slot // bs][h][slot % bs][:] = new[t][h][:] (uint16 arrays)."""
    lib = lib or load()
    NB, Hkv, bs, D = k_cache.shape
    k_new, v_new = _u16(k_new), _u16(v_new)
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    T = slots.shape[0]
    assert k_new.shape == (T, Hkv, D) and v_new.shape == (T, Hkv, D)
    _check(lib.oracle_kv_write(_ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new),
                               _ptr(slots), T, NB, Hkv, D, bs), "oracle_kv_write")


def block_copy(k_cache: np.ndarray, v_cache: np.ndarray, pairs, lib=None) -> None:
    """In place: K/V cache[dst] = K/V cache[src] for each (src, dst) row of ``pairs``."""
    lib = lib or load()
    NB, Hkv, bs, D = k_cache.shape
    pairs = np.ascontiguousarray(pairs, dtype=np.int32).reshape(-1, 2)
    _check(lib.oracle_block_copy(_ptr(k_cache), _ptr(v_cache), _ptr(pairs), pairs.shape[0],
                                 NB, Hkv, D, bs), "oracle_block_copy")


def attention(q, k_cache, v_cache, block_tables, context_lens, scale: float, sel=None,
              nthreads: int = 1, lib=None) -> np.ndarray:
    """fp64 decode attention.  Returns out[S][Hq][D], or out[len(sel)][D] when ``sel``
    lists (sequence, query head) pairs."""
    lib = lib or load()
    q, k_cache, v_cache = _u16(q), _u16(k_cache), _u16(v_cache)
    S, Hq, D = q.shape
    NB, Hkv, bs, D2 = k_cache.shape
    assert D2 == D and v_cache.shape == k_cache.shape
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    ctx = np.ascontiguousarray(context_lens, dtype=np.int32)
    assert bt.ndim == 2 and bt.shape[0] == S and ctx.shape == (S,)
    MB = bt.shape[1]
    if sel is None:
        out = np.empty((S, Hq, D), dtype=np.float64)
        sel_p, nsel = None, 0
    else:
        sel_a = np.ascontiguousarray(sel, dtype=np.int32).reshape(-1, 2)
        out = np.empty((sel_a.shape[0], D), dtype=np.float64)
        sel_p, nsel = _ptr(sel_a), sel_a.shape[0]
    _check(lib.oracle_attention(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt),
                                _ptr(ctx), S, MB, Hq, Hkv, D, bs, NB, float(scale), sel_p, nsel,
                                int(nthreads)), "oracle_attention")
    return out


def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, bytes_per_elem: int,
                       lib=None) -> int:
    """2 x layers x kv_heads x head_dim x bytes ("Inference optimization", KV cache)."""
    lib = lib or load()
    return int(lib.oracle_kv_bytes_per_token(layers, kv_heads, head_dim, bytes_per_elem))


# ---- FP8 (E4M3) cache -------------------------------------------------------------
def e4m3_decode(code: int, lib=None) -> float:
    return float((lib or load()).oracle_e4m3_decode(int(code)))


def e4m3_encode(x: float, lib=None) -> int:
    return int((lib or load()).oracle_e4m3_encode(float(x)))


def _per_head(scale, num_kv_heads: int, dtype) -> np.ndarray:
    """A scale per KV head: a scalar (one scale for the whole cache) or num_kv_heads
    values."""
    a = np.asarray(scale, dtype=dtype)
    assert a.ndim == 0 or a.shape == (num_kv_heads,), a.shape
    return np.ascontiguousarray(np.broadcast_to(a, (num_kv_heads,)))


def kv_write_fp8(k_cache: np.ndarray, v_cache: np.ndarray, k_new, v_new, slot_mapping,
                 k_scale, v_scale, lib=None) -> None:
    """In place on uint8 caches: code = E4M3(bf16 / scale) at each slot (scale in fp32,
    one value for the cache or one per KV head)."""
    lib = lib or load()
    assert k_cache.dtype == np.uint8 and v_cache.dtype == np.uint8
    NB, Hkv, bs, D = k_cache.shape
    k_new, v_new = _u16(k_new), _u16(v_new)
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    T = slots.shape[0]
    ks, vs = _per_head(k_scale, Hkv, np.float32), _per_head(v_scale, Hkv, np.float32)
    _check(lib.oracle_kv_write_fp8(_ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new),
                                   _ptr(slots), T, NB, Hkv, D, bs, _ptr(ks), _ptr(vs)),
           "oracle_kv_write_fp8")


def block_copy_fp8(k_cache: np.ndarray, v_cache: np.ndarray, pairs, lib=None) -> None:
    lib = lib or load()
    NB, Hkv, bs, D = k_cache.shape
    pairs = np.ascontiguousarray(pairs, dtype=np.int32).reshape(-1, 2)
    _check(lib.oracle_block_copy_fp8(_ptr(k_cache), _ptr(v_cache), _ptr(pairs), pairs.shape[0],
                                     NB, Hkv, D, bs), "oracle_block_copy_fp8")


def attention_fp8(q, k_cache, v_cache, block_tables, context_lens, scale: float,
                  k_scale, v_scale, sel=None, nthreads: int = 1,
                  lib=None) -> np.ndarray:
    """fp64 decode attention over an E4M3 cache (element = decode(code) * scale; the
    scales are one value for the cache or one per KV head)."""
    lib = lib or load()
    q = _u16(q)
    k_cache = np.ascontiguousarray(k_cache, dtype=np.uint8)
    v_cache = np.ascontiguousarray(v_cache, dtype=np.uint8)
    S, Hq, D = q.shape
    NB, Hkv, bs, D2 = k_cache.shape
    assert D2 == D and v_cache.shape == k_cache.shape
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    ctx = np.ascontiguousarray(context_lens, dtype=np.int32)
    MB = bt.shape[1]
    if sel is None:
        out = np.empty((S, Hq, D), dtype=np.float64)
        sel_p, nsel = None, 0
    else:
        sel_a = np.ascontiguousarray(sel, dtype=np.int32).reshape(-1, 2)
        out = np.empty((sel_a.shape[0], D), dtype=np.float64)
        sel_p, nsel = _ptr(sel_a), sel_a.shape[0]
    ks, vs = _per_head(k_scale, Hkv, np.float64), _per_head(v_scale, Hkv, np.float64)
    _check(lib.oracle_attention_fp8(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt),
                                    _ptr(ctx), S, MB, Hq, Hkv, D, bs, NB, float(scale),
                                    _ptr(ks), _ptr(vs), sel_p, nsel, int(nthreads)),
           "oracle_attention_fp8")
    return out


# ---- chunked prefill ----------------------------------------------------------------
def attention_prefill(q, k_cache, v_cache, block_tables, context_lens, query_start,
                      scale: float, sel=None, nthreads: int = 1, lib=None) -> np.ndarray:
    """fp64 causal attention of each sequence's last L = query_start[s+1] - query_start[s]
    tokens over its paged cache.  q is [T][Hq][D]; returns out[T][Hq][D], or
    out[len(sel)][D] for the (token, head) pairs in ``sel``."""
    lib = lib or load()
    q, k_cache, v_cache = _u16(q), _u16(k_cache), _u16(v_cache)
    T, Hq, D = q.shape
    NB, Hkv, bs, D2 = k_cache.shape
    assert D2 == D and v_cache.shape == k_cache.shape
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    ctx = np.ascontiguousarray(context_lens, dtype=np.int32)
    qs = np.ascontiguousarray(query_start, dtype=np.int32)
    S = ctx.shape[0]
    assert bt.ndim == 2 and bt.shape[0] == S and qs.shape == (S + 1,)
    if sel is None:
        out = np.empty((T, Hq, D), dtype=np.float64)
        sel_p, nsel = None, 0
    else:
        sel_a = np.ascontiguousarray(sel, dtype=np.int32).reshape(-1, 2)
        out = np.empty((sel_a.shape[0], D), dtype=np.float64)
        sel_p, nsel = _ptr(sel_a), sel_a.shape[0]
    _check(lib.oracle_attention_prefill(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                        _ptr(bt), _ptr(ctx), _ptr(qs), S, T, bt.shape[1], Hq,
                                        Hkv, D, bs, NB, float(scale), sel_p, nsel,
                                        int(nthreads)), "oracle_attention_prefill")
    return out
