"""Plant plausible mistakes in the oracle's C source and check that each one trips at
least one pin.  The mistakes live only in temporary copies built on the CPU."""
import os
import tempfile

import pytest

import oracle
import oracle_pins as P

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, original text, mistaken text)
MUTANTS = [
    ("gqa-modulo", "const int kv_head = head / group;",
     "const int kv_head = head % num_kv_heads;"),
    ("scale-dropped", "x[t] = scale * acc;", "x[t] = acc;"),
    ("offset-shifted", "int offset = t % block_size;", "int offset = (t + 1) % block_size;"),
    ("block-index-mod", "int32_t block = block_table[t / block_size];",
     "int32_t block = block_table[t % block_size];"),
    ("layout-transposed",
     "size_t row = (((size_t)block * num_kv_heads + kv_head) * block_size + offset) * head_dim;",
     "size_t row = (((size_t)block * block_size + offset) * num_kv_heads + kv_head) * head_dim;"),
    ("v-from-k", "vc[(size_t)t * head_dim + d] = bf16_to_f64(v_cache[row + d]);",
     "vc[(size_t)t * head_dim + d] = bf16_to_f64(k_cache[row + d]);"),
    ("not-normalised", "out[d] = acc / denom;", "out[d] = acc;"),
    ("sign-flipped", "x[t] = exp(x[t] - m);", "x[t] = exp(m - x[t]);"),
    ("base-two", "x[t] = exp(x[t] - m);", "x[t] = exp2(x[t] - m);"),
    ("last-token-dropped", "for (int t = 0; t < ctx; ++t) acc += x[t]",
     "for (int t = 0; t + 1 < ctx; ++t) acc += x[t]"),
    ("q-transposed", "q + ((size_t)s * num_q_heads + h) * head_dim",
     "q + ((size_t)h * num_seqs + s) * head_dim"),
    ("write-layout",
     "size_t dst = (((size_t)block * num_kv_heads + h) * block_size + offset) * head_dim;",
     "size_t dst = (((size_t)block * block_size + offset) * num_kv_heads + h) * head_dim;"),
    ("write-v-from-k", "v_cache[dst + d] = v_new[src + d];", "v_cache[dst + d] = k_new[src + d];"),
    ("copy-k-only",
     "v_cache[(size_t)dst * block_elems + e] = v_cache[(size_t)src * block_elems + e];", ""),
    ("copy-reversed",
     "k_cache[(size_t)dst * block_elems + e] = k_cache[(size_t)src * block_elems + e];",
     "k_cache[(size_t)src * block_elems + e] = k_cache[(size_t)dst * block_elems + e];"),
    ("bytes-no-kv-factor", "return (int64_t)2 * layers", "return (int64_t)layers"),
]


def _pins_fail(lib):
    failed = []
    for pin in P.ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, oracle.OracleError):
            failed.append(pin.__name__)
    return failed


@pytest.mark.parametrize("name,orig,bad", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, orig, bad, tmp_path):
    src = open(SRC).read()
    assert src.count(orig) == 1, f"mutation anchor for {name} not unique"
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src.replace(orig, bad))
    so = str(tmp_path / "libmutant.so")
    oracle.build(force=True, src=str(mpath), out=so)
    lib = oracle.load(so)
    failed = _pins_fail(lib)
    assert failed, f"mutant {name} passed every pin"
