"""Thin Python binding of libpagedkv.so (argument marshalling only).

Every function here takes torch tensors on the GPU, checks dtypes and shapes, and
passes raw pointers, sizes and the current CUDA stream to the C entry point of the
same name declared in ``include/pagedkv.h``.  All work runs in the library's CUDA
kernels.  If the library is missing the import raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpagedkv.so")

PKV_ATTN_AUTO, PKV_ATTN_FMA, PKV_ATTN_MMA = 0, 1, 2
PKV_PREFILL_AUTO, PKV_PREFILL_MMA, PKV_PREFILL_TC, PKV_PREFILL_TC_PAIR = 0, 1, 2, 3
PKV_PREFILL_TC_2SM, PKV_PREFILL_TC_SEP = 4, 5
DEV_BAD_BLOCK, DEV_BAD_SLOT, DEV_BAD_CONTEXT, DEV_TIMEOUT = 1, 2, 4, 8
DEV_BAD_SCALE, DEV_BAD_ROW = 32, 64
DEFAULT_PARTITION = 512

# Every entry point the header declares: name -> (restype, argtypes).
_P, _I, _F, _SZ, _I64 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t,
                         ctypes.c_int64)
ABI_VERSION = 4  # PKV_ABI_VERSION of include/pagedkv.h
SIGNATURES = {
    "paged_kv_version": (_I, []),
    "paged_kv_strerror": (ctypes.c_char_p, [_I]),
    "paged_kv_write": (_I, [_P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _P, _P]),
    "paged_block_copy": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P]),
    "paged_kv_check_slots": (_I, [_P, _I, _I, _I]),
    "paged_attention_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "paged_attention_decode": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I,
                                    _I, _P, _SZ, _P, _P]),
    "paged_decode_step": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _I,
                               _P, _P, _P, _I, _P, _I, _P, _SZ, _P, _P]),
    "paged_decode_step_fp8": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _F,
                                   _F, _P, _P, _I, _I, _P, _P, _P, _I, _P, _I, _P, _SZ, _P,
                                   _P]),
    "paged_attention_set_variant": (_I, [_I]),
    "paged_attention_prefill_set_variant": (_I, [_I]),
    "paged_attention_decode_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I,
                                            _F, _I, _I, _P, _P]),
    "paged_kv_write_fp8": (_I, [_P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _F, _F, _P, _P]),
    "paged_kv_write_fp8_per_head": (_I, [_P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _P, _P, _P,
                                         _P]),
    "paged_block_copy_fp8": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P]),
    "paged_attention_decode_fp8": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F,
                                        _F, _F, _I, _I, _P, _SZ, _P, _P]),
    "paged_attention_decode_fp8_per_head": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                                                 _I, _F, _P, _P, _I, _I, _P, _SZ, _P, _P]),
    "paged_attention_prefill": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I,
                                     _F, _I, _P, _P]),
    "pkv_pool_create": (_I, [_I, _I, _P, ctypes.POINTER(_P)]),
    "pkv_pool_destroy": (None, [_P]),
    "pkv_pool_num_free": (_I, [_P]),
    "pkv_block_refcount": (_I, [_P, _I]),
    "pkv_seq_add": (_I, [_P, _I64]),
    "pkv_seq_fork": (_I, [_P, _I64, _I64]),
    "pkv_seq_free": (_I, [_P, _I64]),
    "pkv_seq_num_tokens": (_I, [_P, _I64, _P]),
    "pkv_seq_num_blocks": (_I, [_P, _I64, _P]),
    "pkv_seq_append_slot": (_I, [_P, _I64, _P, _P, _P]),
    "pkv_seq_append_tokens": (_I, [_P, _I64, _I, _P, _P, _P]),
    "pkv_pool_step": (_I, [_P, _P, _I, _P, _P, _P]),
    "pkv_pool_export": (_I, [_P, _P, _I, _I, ctypes.c_int32, _P, _P]),
    "pkv_pool_save": (_I64, [_P, _P, _I64]),
    "pkv_pool_load": (_I, [_P, _I64, ctypes.POINTER(_P)]),
    "pkv_seq_add_shared": (_I, [_P, _I64, _P, _I]),
    "pkv_block_retain": (_I, [_P, _I]),
    "pkv_block_release": (_I, [_P, _I]),
    "pkv_pcache_create": (_I, [_P, _I, ctypes.POINTER(_P)]),
    "pkv_pcache_destroy": (None, [_P]),
    "pkv_pcache_lookup": (_I, [_P, _P, _I, _P, _I]),
    "pkv_pcache_use": (_I, [_P, _P, _I, _I]),
    "pkv_pcache_insert": (_I, [_P, _P, _I, _P, _I]),
    "pkv_pcache_evict_free_one": (_I, [_P]),
    "pkv_pcache_stats": (_I, [_P, _P]),
    "pkv_sched_create": (_I, [_P, _P, _I, _I, _I, ctypes.POINTER(_P)]),
    "pkv_sched_destroy": (None, [_P]),
    "pkv_sched_add_request": (_I, [_P, _I64, _I, _P, _I]),
    "pkv_sched_step": (_I, [_P, _P]),
    "pkv_sched_done": (_I, [_P]),
    "pkv_sched_pack": (_I, [_P, _P, _I64, _I, _I, _I, _P]),
    "pkv_step_synthetic_rows": (_I, [_P, _P, _I64]),
    "paged_gather_rows": (_I, [_P, _P, _P, _I, _I64, _I, _P, _P]),
    "pkv_step_launch": (_I, [_P, _P, _I, _P, _P]),
    "pkv_engine_step": (_I, [_P, _P, _P, _I, _P, _P]),
    "pkv_sched_get_stats": (_I, [_P, _P]),
    "pkv_selftest_bounded_wait": (_I, [_P, _P, ctypes.c_longlong, _I, _P]),
}


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with __graft_entry__.build() or "
            "python -m paged_kv_cache_272_gb300.build (there is no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if lib.paged_kv_version() != ABI_VERSION:
        raise ImportError(f"{LIB_PATH} has ABI version {lib.paged_kv_version()}, this binding "
                          f"expects {ABI_VERSION}: rebuild the library")
    return lib


lib = _load()


class PagedKVError(RuntimeError):
    def __init__(self, code: int, what: str):
        msg = lib.paged_kv_strerror(code).decode()
        super().__init__(f"{what}: {msg} (code {code})")
        self.code = code


def check(code: int, what: str) -> None:
    if code != 0:
        raise PagedKVError(code, what)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _bf16_cuda(name, t):
    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous bf16 CUDA tensor")


def _i32(name, t):
    if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous int32 CUDA tensor")


def paged_kv_write(k_new, v_new, slot_mapping, k_cache, v_cache, err_flag=None, stream=None):
    """Scatter k_new/v_new [T][Hkv][D] into the caches [NB][Hkv][16][D] at slot_mapping."""
    for n, t in (("k_new", k_new), ("v_new", v_new), ("k_cache", k_cache), ("v_cache", v_cache)):
        _bf16_cuda(n, t)
    if slot_mapping.dtype != torch.int64 or not slot_mapping.is_cuda:
        raise TypeError("slot_mapping must be an int64 CUDA tensor")
    NB, Hkv, bs, D = k_cache.shape
    T = slot_mapping.shape[0]
    if tuple(k_new.shape) != (T, Hkv, D) or k_new.shape != v_new.shape:
        raise ValueError("k_new/v_new must be [num_tokens][num_kv_heads][head_dim]")
    check(lib.paged_kv_write(_ptr(k_new), _ptr(v_new), _ptr(slot_mapping.contiguous()), T,
                             _ptr(k_cache), _ptr(v_cache), NB, Hkv, D, bs, _ptr(err_flag),
                             _stream(stream)), "paged_kv_write")


def paged_kv_check_slots(slot_mapping, num_blocks, block_size=16) -> None:
    """Raise if a host slot mapping has an out-of-range or repeated slot."""
    import numpy as np
    a = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    check(lib.paged_kv_check_slots(a.ctypes.data if a.size else None, a.shape[0], num_blocks,
                                   block_size), "paged_kv_check_slots")


def paged_block_copy(k_cache, v_cache, block_pairs, err_flag=None, stream=None):
    """Copy whole blocks src -> dst for each row of block_pairs [P][2] (int32)."""
    _bf16_cuda("k_cache", k_cache)
    _bf16_cuda("v_cache", v_cache)
    _i32("block_pairs", block_pairs)
    NB, Hkv, bs, D = k_cache.shape
    P = block_pairs.numel() // 2
    check(lib.paged_block_copy(_ptr(k_cache), _ptr(v_cache), _ptr(block_pairs), P, NB, Hkv, D,
                               bs, _ptr(err_flag), _stream(stream)), "paged_block_copy")


def paged_gather_rows(dst, src, idx, err_flag=None, stream=None):
    """dst[i] = src[idx[i]] for i < len(idx): whole rows (the leading dimension) of
    contiguous CUDA tensors of one dtype; idx int64."""
    if not (dst.is_cuda and src.is_cuda and idx.is_cuda) or dst.dtype != src.dtype:
        raise ValueError("dst, src and idx must be CUDA tensors; dst and src of one dtype")
    if idx.dtype != torch.int64 or not (dst.is_contiguous() and src.is_contiguous()):
        raise ValueError("idx must be int64; dst and src contiguous")
    row = src[0].numel() * src.element_size() if src.shape[0] else 0
    if dst.shape[1:] != src.shape[1:] or dst.shape[0] < idx.numel():
        raise ValueError("dst rows must match src rows and hold len(idx) rows")
    check(lib.paged_gather_rows(_ptr(dst), _ptr(src), _ptr(idx), idx.numel(), src.shape[0], row,
                                _ptr(err_flag), _stream(stream)), "paged_gather_rows")


def paged_attention_workspace_size(num_seqs, num_q_heads, head_dim, max_context_len,
                                   partition_size=DEFAULT_PARTITION) -> int:
    return int(lib.paged_attention_workspace_size(num_seqs, num_q_heads, head_dim,
                                                  max_context_len, partition_size))


def alloc_workspace(num_seqs, num_q_heads, head_dim, max_context_len,
                    partition_size=DEFAULT_PARTITION, device="cuda"):
    n = paged_attention_workspace_size(num_seqs, num_q_heads, head_dim, max_context_len,
                                       partition_size)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def paged_attention_decode(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                           max_context_len, workspace, partition_size=DEFAULT_PARTITION,
                           err_flag=None, stream=None):
    """out[S][Hq][D] = softmax(scale q K^T) V over each sequence's paged context."""
    for n, t in (("out", out), ("q", q), ("k_cache", k_cache), ("v_cache", v_cache)):
        _bf16_cuda(n, t)
    _i32("block_tables", block_tables)
    _i32("context_lens", context_lens)
    S, Hq, D = q.shape
    NB, Hkv, bs, D2 = k_cache.shape
    if D2 != D or tuple(out.shape) != (S, Hq, D) or v_cache.shape != k_cache.shape:
        raise ValueError("shape mismatch between q, out and the caches")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or context_lens.shape != (S,):
        raise ValueError("block_tables must be [S][max_blocks] and context_lens [S]")
    check(lib.paged_attention_decode(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        _ptr(context_lens), S, block_tables.shape[1], Hq, Hkv, D, bs, NB, float(scale),
        int(partition_size), int(max_context_len), _ptr(workspace), workspace.numel(),
        _ptr(err_flag), _stream(stream)), "paged_attention_decode")


def _step_io(k_new, v_new, slot_mapping, pairs, Hkv, D):
    """Checks of the write and copy arguments of a decode step; returns (T, P)."""
    T = 0 if slot_mapping is None else slot_mapping.shape[0]
    if T:
        _bf16_cuda("k_new", k_new)
        _bf16_cuda("v_new", v_new)
        if slot_mapping.dtype != torch.int64 or not slot_mapping.is_cuda \
                or not slot_mapping.is_contiguous():
            raise TypeError("slot_mapping must be a contiguous int64 CUDA tensor")
        if tuple(k_new.shape) != (T, Hkv, D) or k_new.shape != v_new.shape:
            raise ValueError("k_new/v_new must be [num_tokens][num_kv_heads][head_dim]")
    P = 0 if pairs is None else pairs.numel() // 2
    if P:
        _i32("block_pairs", pairs)
    return T, P


def paged_decode_step(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                      max_context_len, workspace, k_new=None, v_new=None, slot_mapping=None,
                      block_pairs=None, partition_size=DEFAULT_PARTITION, err_flag=None,
                      stream=None):
    """One decode step: copy-on-write of block_pairs [P][2], the write of k_new/v_new
    [T][Hkv][D] at slot_mapping, then paged decode attention into out [S][Hq][D]."""
    for n, t in (("out", out), ("q", q), ("k_cache", k_cache), ("v_cache", v_cache)):
        _bf16_cuda(n, t)
    _i32("block_tables", block_tables)
    _i32("context_lens", context_lens)
    S, Hq, D = q.shape
    NB, Hkv, bs, D2 = k_cache.shape
    if D2 != D or tuple(out.shape) != (S, Hq, D) or v_cache.shape != k_cache.shape:
        raise ValueError("shape mismatch between q, out and the caches")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or context_lens.shape != (S,):
        raise ValueError("block_tables must be [S][max_blocks] and context_lens [S]")
    T, P = _step_io(k_new, v_new, slot_mapping, block_pairs, Hkv, D)
    check(lib.paged_decode_step(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        _ptr(context_lens), S, block_tables.shape[1], Hq, Hkv, D, bs, NB, float(scale),
        int(partition_size), int(max_context_len), _ptr(k_new) if T else None,
        _ptr(v_new) if T else None, _ptr(slot_mapping) if T else None, T,
        _ptr(block_pairs) if P else None, P, _ptr(workspace), workspace.numel(),
        _ptr(err_flag), _stream(stream)), "paged_decode_step")


def paged_attention_prefill(out, q, k_cache, v_cache, block_tables, context_lens, query_start,
                            scale, max_query_len, err_flag=None, stream=None):
    """Chunked prefill: rows query_start[s] .. query_start[s+1]-1 of q [T][Hq][D] are the
    last tokens of sequence s and attend causally over its paged context; out [T][Hq][D]."""
    for n, t in (("out", out), ("q", q), ("k_cache", k_cache), ("v_cache", v_cache)):
        _bf16_cuda(n, t)
    _i32("block_tables", block_tables)
    _i32("context_lens", context_lens)
    _i32("query_start", query_start)
    T, Hq, D = q.shape
    NB, Hkv, bs, D2 = k_cache.shape
    S = context_lens.shape[0]
    if D2 != D or tuple(out.shape) != (T, Hq, D) or v_cache.shape != k_cache.shape:
        raise ValueError("shape mismatch between q, out and the caches")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or query_start.shape != (S + 1,):
        raise ValueError("block_tables must be [S][max_blocks] and query_start [S+1]")
    check(lib.paged_attention_prefill(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        _ptr(context_lens), _ptr(query_start), S, T, block_tables.shape[1], Hq, Hkv, D, bs, NB,
        float(scale), int(max_query_len), _ptr(err_flag), _stream(stream)),
        "paged_attention_prefill")


def set_prefill_variant(variant: int) -> int:
    """Select the chunked-prefill kernel (PKV_PREFILL_AUTO / _MMA / _TC); returns the
    previous selection."""
    prev = lib.paged_attention_prefill_set_variant(int(variant))
    if prev < 0:
        raise PagedKVError(prev, "paged_attention_prefill_set_variant")
    return prev


def set_attention_variant(variant: int) -> int:
    prev = lib.paged_attention_set_variant(int(variant))
    if prev < 0:
        raise PagedKVError(prev, "paged_attention_set_variant")
    return prev


# ---- E4M3 (FP8) cache ----------------------------------------------------------------
def _u8_cuda(name, t):
    if t.dtype != torch.uint8 or not t.is_cuda or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous uint8 CUDA tensor (E4M3 codes)")


def paged_kv_write_fp8(k_new, v_new, slot_mapping, k_cache, v_cache, k_scale, v_scale,
                       err_flag=None, stream=None):
    """Quantise bf16 k_new/v_new [T][Hkv][D] to E4M3 and scatter into uint8 caches."""
    _bf16_cuda("k_new", k_new)
    _bf16_cuda("v_new", v_new)
    _u8_cuda("k_cache", k_cache)
    _u8_cuda("v_cache", v_cache)
    NB, Hkv, bs, D = k_cache.shape
    T = slot_mapping.shape[0]
    if tuple(k_new.shape) != (T, Hkv, D) or k_new.shape != v_new.shape:
        raise ValueError("k_new/v_new must be [num_tokens][num_kv_heads][head_dim]")
    check(lib.paged_kv_write_fp8(_ptr(k_new), _ptr(v_new), _ptr(slot_mapping.contiguous()), T,
                                 _ptr(k_cache), _ptr(v_cache), NB, Hkv, D, bs, float(k_scale),
                                 float(v_scale), _ptr(err_flag), _stream(stream)),
          "paged_kv_write_fp8")


def _scales_cuda(name, t, num_kv_heads):
    if (t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous()
            or tuple(t.shape) != (num_kv_heads,)):
        raise TypeError(f"{name} must be a contiguous float32 CUDA tensor of num_kv_heads")


def paged_kv_write_fp8_per_head(k_new, v_new, slot_mapping, k_cache, v_cache, k_scales,
                                v_scales, err_flag=None, stream=None):
    """paged_kv_write_fp8 with one scale per KV head (k_scales, v_scales: float32 CUDA
    tensors [num_kv_heads])."""
    _bf16_cuda("k_new", k_new)
    _bf16_cuda("v_new", v_new)
    _u8_cuda("k_cache", k_cache)
    _u8_cuda("v_cache", v_cache)
    NB, Hkv, bs, D = k_cache.shape
    _scales_cuda("k_scales", k_scales, Hkv)
    _scales_cuda("v_scales", v_scales, Hkv)
    T = slot_mapping.shape[0]
    if tuple(k_new.shape) != (T, Hkv, D) or k_new.shape != v_new.shape:
        raise ValueError("k_new/v_new must be [num_tokens][num_kv_heads][head_dim]")
    check(lib.paged_kv_write_fp8_per_head(
        _ptr(k_new), _ptr(v_new), _ptr(slot_mapping.contiguous()), T, _ptr(k_cache),
        _ptr(v_cache), NB, Hkv, D, bs, _ptr(k_scales), _ptr(v_scales), _ptr(err_flag),
        _stream(stream)), "paged_kv_write_fp8_per_head")


def paged_block_copy_fp8(k_cache, v_cache, block_pairs, err_flag=None, stream=None):
    _u8_cuda("k_cache", k_cache)
    _u8_cuda("v_cache", v_cache)
    _i32("block_pairs", block_pairs)
    NB, Hkv, bs, D = k_cache.shape
    check(lib.paged_block_copy_fp8(_ptr(k_cache), _ptr(v_cache), _ptr(block_pairs),
                                   block_pairs.numel() // 2, NB, Hkv, D, bs, _ptr(err_flag),
                                   _stream(stream)), "paged_block_copy_fp8")


def paged_attention_decode_fp8(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                               k_scale, v_scale, max_context_len, workspace,
                               partition_size=DEFAULT_PARTITION, err_flag=None, stream=None):
    _bf16_cuda("out", out)
    _bf16_cuda("q", q)
    _u8_cuda("k_cache", k_cache)
    _u8_cuda("v_cache", v_cache)
    _i32("block_tables", block_tables)
    _i32("context_lens", context_lens)
    S, Hq, D = q.shape
    NB, Hkv, bs, D2 = k_cache.shape
    if D2 != D or tuple(out.shape) != (S, Hq, D) or v_cache.shape != k_cache.shape:
        raise ValueError("shape mismatch between q, out and the caches")
    check(lib.paged_attention_decode_fp8(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        _ptr(context_lens), S, block_tables.shape[1], Hq, Hkv, D, bs, NB, float(scale),
        float(k_scale), float(v_scale), int(partition_size), int(max_context_len),
        _ptr(workspace), workspace.numel(), _ptr(err_flag), _stream(stream)),
        "paged_attention_decode_fp8")


def paged_attention_decode_fp8_per_head(out, q, k_cache, v_cache, block_tables, context_lens,
                                        scale, k_scales, v_scales, max_context_len, workspace,
                                        partition_size=DEFAULT_PARTITION, err_flag=None,
                                        stream=None):
    """paged_attention_decode_fp8 with one scale per KV head (k_scales, v_scales: float32
    CUDA tensors [num_kv_heads])."""
    _bf16_cuda("out", out)
    _bf16_cuda("q", q)
    _u8_cuda("k_cache", k_cache)
    _u8_cuda("v_cache", v_cache)
    _i32("block_tables", block_tables)
    _i32("context_lens", context_lens)
    S, Hq, D = q.shape
    NB, Hkv, bs, D2 = k_cache.shape
    _scales_cuda("k_scales", k_scales, Hkv)
    _scales_cuda("v_scales", v_scales, Hkv)
    if D2 != D or tuple(out.shape) != (S, Hq, D) or v_cache.shape != k_cache.shape:
        raise ValueError("shape mismatch between q, out and the caches")
    check(lib.paged_attention_decode_fp8_per_head(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        _ptr(context_lens), S, block_tables.shape[1], Hq, Hkv, D, bs, NB, float(scale),
        _ptr(k_scales), _ptr(v_scales), int(partition_size), int(max_context_len),
        _ptr(workspace), workspace.numel(), _ptr(err_flag), _stream(stream)),
        "paged_attention_decode_fp8_per_head")


def selftest_bounded_wait(err_flag, result, limit_cycles, use_spin=False, stream=None):
    """Launch the bounded-wait self-test: one thread waits `limit_cycles` clock cycles on
    an mbarrier phase that nothing completes, then gives up as the library's kernels do
    (PKV_DEV_TIMEOUT ORed into err_flag).  result: int64 CUDA tensor of 3 (wait
    succeeded, cycles spent, abort flag)."""
    _i32("err_flag", err_flag)
    if result.dtype != torch.int64 or not result.is_cuda or result.numel() < 3:
        raise TypeError("result must be an int64 CUDA tensor of at least 3 elements")
    check(lib.pkv_selftest_bounded_wait(_ptr(err_flag), _ptr(result), int(limit_cycles),
                                        1 if use_spin else 0, _stream(stream)),
          "pkv_selftest_bounded_wait")


def paged_decode_step_fp8(out, q, k_cache, v_cache, block_tables, context_lens, scale, k_scale,
                          v_scale, max_context_len, workspace, k_new=None, v_new=None,
                          slot_mapping=None, block_pairs=None, partition_size=DEFAULT_PARTITION,
                          err_flag=None, stream=None):
    """paged_decode_step over E4M3 caches.  k_scale/v_scale: floats (one scale per cache)
    or float32 CUDA tensors [num_kv_heads] (one scale per KV head)."""
    _bf16_cuda("out", out)
    _bf16_cuda("q", q)
    _u8_cuda("k_cache", k_cache)
    _u8_cuda("v_cache", v_cache)
    _i32("block_tables", block_tables)
    _i32("context_lens", context_lens)
    S, Hq, D = q.shape
    NB, Hkv, bs, D2 = k_cache.shape
    if D2 != D or tuple(out.shape) != (S, Hq, D) or v_cache.shape != k_cache.shape:
        raise ValueError("shape mismatch between q, out and the caches")
    T, P = _step_io(k_new, v_new, slot_mapping, block_pairs, Hkv, D)
    per_head = torch.is_tensor(k_scale)
    if per_head:
        for n, t in (("k_scales", k_scale), ("v_scales", v_scale)):
            if t.dtype != torch.float32 or not t.is_cuda or tuple(t.shape) != (Hkv,):
                raise TypeError(f"{n} must be a float32 CUDA tensor [num_kv_heads]")
    check(lib.paged_decode_step_fp8(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        _ptr(context_lens), S, block_tables.shape[1], Hq, Hkv, D, bs, NB, float(scale),
        1.0 if per_head else float(k_scale), 1.0 if per_head else float(v_scale),
        _ptr(k_scale) if per_head else None, _ptr(v_scale) if per_head else None,
        int(partition_size), int(max_context_len), _ptr(k_new) if T else None,
        _ptr(v_new) if T else None, _ptr(slot_mapping) if T else None, T,
        _ptr(block_pairs) if P else None, P, _ptr(workspace), workspace.numel(),
        _ptr(err_flag), _stream(stream)), "paged_decode_step_fp8")
