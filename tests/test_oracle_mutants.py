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
    ("not-normalised", "for (int d = 0; d < head_dim; ++d) out[d] /= denom;", ""),
    ("sign-flipped", "x[t] = exp(x[t] - m);", "x[t] = exp(m - x[t]);"),
    ("base-two", "x[t] = exp(x[t] - m);", "x[t] = exp2(x[t] - m);"),
    ("last-token-dropped", "const double *vt = vc + (size_t)t * head_dim;",
     "if (t + 1 == ctx) break;\n const double *vt = vc + (size_t)t * head_dim;"),
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
    ("e4m3-bias-8", "ldexp(1.0 + m / 8.0, e - 7)", "ldexp(1.0 + m / 8.0, e - 8)"),
    ("e4m3-truncate", "const double r = rint(a / spacing);",
     "const double r = floor(a / spacing);"),
    ("e4m3-no-saturate", "if (a >= 448.0) return sign | 0x7E;", "if (a >= 480.0) return sign | 0x7F;"),
    ("fp8-write-no-scale", "k_cache[dst + d] = oracle_e4m3_encode(kx / k_scales[h]);",
     "k_cache[dst + d] = oracle_e4m3_encode(kx);"),
    ("fp8-write-first-head-scale", "oracle_e4m3_encode(vx / v_scales[h]);",
     "oracle_e4m3_encode(vx / v_scales[0]);"),
    ("fp8-attn-v-scale", "oracle_e4m3_decode(v_cache[vcol + (size_t)d * block_size]) * v_scale;",
     "oracle_e4m3_decode(v_cache[vcol + (size_t)d * block_size]) * k_scale;"),
    ("fp8-attn-scale-by-query-head",
     "const double k_scale = k_scales[kv_head], v_scale = v_scales[kv_head];",
     "const double k_scale = k_scales[h % num_kv_heads], v_scale = v_scales[h % num_kv_heads];"),
    ("fp8-v-untransposed", "oracle_e4m3_decode(v_cache[vcol + (size_t)d * block_size])",
     "oracle_e4m3_decode(v_cache[row + d])"),
    ("fp8-write-v-untransposed", "v_cache[vbase + (size_t)d * block_size] =",
     "v_cache[dst + d] ="),
    ("fp8-copy-k-only",
     "memcpy(v_cache + (size_t)dst * block_elems, v_cache + (size_t)src * block_elems, block_elems);",
     ""),
    ("prefill-position-from-chunk",
     "const int pos = context_lens[s] - L + (tok - query_start[s]);",
     "const int pos = tok - query_start[s];"),
    ("prefill-excludes-self", "pos + 1, max_blocks, h,", "pos, max_blocks, h,"),
    ("prefill-not-causal", "pos + 1, max_blocks, h,", "context_lens[s], max_blocks, h,"),
    ("prefill-q-row-of-sequence", "q + ((size_t)tok * num_q_heads + h) * head_dim",
     "q + ((size_t)s * num_q_heads + h) * head_dim"),
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
    # a mistake in text that several routines share is planted in all of them
    assert src.count(orig) >= 1, f"mutation anchor for {name} not found"
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src.replace(orig, bad))
    so = str(tmp_path / "libmutant.so")
    oracle.build(force=True, src=str(mpath), out=so)
    lib = oracle.load(so)
    failed = _pins_fail(lib)
    assert failed, f"mutant {name} passed every pin"
