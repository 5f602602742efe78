"""The oracle against values the pages print, closed forms, a library routine,
layout invariants and brute force (CPU only)."""
import pytest

import oracle
import oracle_pins as P


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, lib):
    pin(lib)


def test_block_counts_figure():
    P.pin_block_counts()


def test_sdpa_gqa4(lib):
    P.pin_sdpa_contiguous(lib, ctx_override=[1, 2, 15, 16, 17, 100], Hq=8, Hkv=2, seed=31)


def test_sdpa_mha(lib):
    P.pin_sdpa_contiguous(lib, ctx_override=[33, 48, 64], Hq=3, Hkv=3, seed=32)


def test_index_errors(lib):
    import numpy as np
    from paged_kv_cache_272_gb300 import workloads
    w = workloads.build("err", [20], 2, 1, 64, seed=40)
    k, v = P.host_caches(w)
    bt = w.block_tables.copy()
    bt[0, 1] = w.num_blocks  # out of range
    with pytest.raises(oracle.OracleError):
        oracle.attention(w.q, k, v, bt, w.context_lens, w.scale, lib=lib)
    with pytest.raises(oracle.OracleError):
        oracle.kv_write(k, v, w.k_new, w.v_new, np.array([w.num_blocks * 16]), lib=lib)
    with pytest.raises(oracle.OracleError):
        oracle.block_copy(k, v, [(0, w.num_blocks)], lib=lib)
    ctx = w.context_lens.copy()
    ctx[0] = bt.shape[1] * 16 + 1  # beyond the table
    with pytest.raises(oracle.OracleError):
        oracle.attention(w.q, k, v, w.block_tables, ctx, w.scale, lib=lib)


def test_prefill_rejects_bad_query_start(lib):
    import numpy as np
    from paged_kv_cache_272_gb300 import workloads
    w = workloads.build_prefill("err", [20, 8], [4, 8], 2, 1, 64, seed=41)
    k, v = P.host_caches(w)
    for ctx, qs in (([3, 8], [0, 4, 12]),      # chunk longer than its context
                    ([20, 8], [0, 4, 11]),     # last entry is not the token count
                    ([20, 8], [1, 4, 12])):    # does not start at 0
        with pytest.raises(oracle.OracleError):
            oracle.attention_prefill(w.q, k, v, w.block_tables, np.array(ctx, np.int32),
                                     np.array(qs, np.int32), w.scale, lib=lib)
