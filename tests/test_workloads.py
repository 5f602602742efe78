"""The seeded input generators: KV byte counts (logical and unique) and the structure of
the prefill workloads (CPU only)."""
import numpy as np

from paged_kv_cache_272_gb300 import workloads


def test_unique_bytes_count_a_shared_prefix_once():
    w = workloads.make_config(4)
    per_token = 2 * w.num_kv_heads * w.head_dim * 2
    prefix = w.shared_prefix_blocks * w.block_size
    assert workloads.kv_read_bytes(w) == int(w.context_lens.sum()) * per_token
    unique_tokens = prefix + int((w.context_lens - prefix).sum())
    assert workloads.unique_kv_read_bytes(w) == unique_tokens * per_token


def test_unique_bytes_equal_logical_without_sharing():
    for n in (1, 3):
        w = workloads.make_config(n)
        assert workloads.unique_kv_read_bytes(w) == workloads.kv_read_bytes(w)


def test_prefill_workload_structure():
    w = workloads.make_prefill_config(1)
    L = np.diff(w.query_start)
    assert (L <= w.context_lens).all() and w.num_tokens == L.sum()
    # the chunk's slots are the last L positions of each sequence, in its own blocks
    for s in range(w.num_seqs):
        pos = np.arange(w.context_lens[s] - L[s], w.context_lens[s])
        want = w.block_tables[s, pos // 16].astype(np.int64) * 16 + pos % 16
        assert (w.slot_mapping[w.query_start[s]:w.query_start[s + 1]] == want).all()
    assert len(set(w.slot_mapping.tolist())) == w.num_tokens
