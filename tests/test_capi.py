"""The C-ABI library loads on a machine without a GPU, exports every entry point the
header declares, and rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedkv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_lists_the_path():
    names = declared_functions()
    for want in ("paged_kv_write", "paged_attention_decode", "paged_block_copy",
                 "paged_attention_workspace_size", "paged_kv_strerror", "pkv_pool_create",
                 "pkv_pool_step", "pkv_seq_append_slot"):
        assert want in names


def test_library_exports_every_declared_symbol():
    from paged_kv_cache_272_gb300 import ops
    lib = ctypes.CDLL(ops.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert set(declared_functions()) <= set(ops.SIGNATURES)


def _declarations():
    """(return type, name, [parameter declarations]) of every function the header
    declares."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    text = re.sub(r"#.*", "", text)
    out = []
    for ret, name, params in re.findall(r"([A-Za-z_][\w\s\*]*?)\b([a-z_0-9]+)\s*\(([^;{]*?)\)\s*;",
                                        text, flags=re.S):
        ps = " ".join(params.split())
        out.append((" ".join(ret.split()), name,
                    [] if ps in ("", "void") else [p.strip() for p in ps.split(",")]))
    return out


def _ctype_of(decl: str):
    """The ctypes type a C parameter (or return) declaration needs."""
    if "*" in decl:
        return "pointer"
    words = decl.replace("const ", "").split()
    base = " ".join(words[:-1]) if len(words) > 1 else words[0]
    return {"int": ctypes.c_int, "int32_t": ctypes.c_int32, "int64_t": ctypes.c_int64,
            "long long": ctypes.c_longlong, "size_t": ctypes.c_size_t,
            "float": ctypes.c_float, "double": ctypes.c_double, "void": None}[base]


def _same(want, got):
    if want == "pointer":
        return got is ctypes.c_void_p or got is ctypes.c_char_p or (
            isinstance(got, type) and issubclass(got, ctypes._Pointer))
    if want is None:
        return got is None
    return ctypes.sizeof(want) == ctypes.sizeof(got) and (
        issubclass(want, (ctypes.c_float, ctypes.c_double)) ==
        issubclass(got, (ctypes.c_float, ctypes.c_double)))


def test_binding_matches_header_parameter_by_parameter():
    """Every declared function's ctypes signature has the header's parameter count and,
    position by position, a pointer where the header has a pointer and an integer or
    float of the header's width elsewhere (a mismatch would hand the library a wrong
    value or pointer)."""
    from paged_kv_cache_272_gb300 import ops
    decls = _declarations()
    assert len(decls) >= len(declared_functions())
    for ret, name, params in decls:
        restype, argtypes = ops.SIGNATURES[name]
        assert len(argtypes) == len(params), (name, params, argtypes)
        for i, (p, a) in enumerate(zip(params, argtypes)):
            assert _same(_ctype_of(p), a), (name, i, p, a)
        assert _same(_ctype_of(ret + " r"), restype), (name, ret, restype)


def test_host_side_validation():
    from paged_kv_cache_272_gb300.ops import lib
    fake = 1 << 20  # never dereferenced: every call below fails validation first
    # block size other than 16
    assert lib.paged_kv_write(fake, fake, fake, 4, fake, fake, 8, 1, 64, 8, None, None) == -3
    # head_dim not a multiple of 8
    assert lib.paged_kv_write(fake, fake, fake, 4, fake, fake, 8, 1, 60, 16, None, None) == -2
    # NULL pointer
    assert lib.paged_kv_write(None, fake, fake, 4, fake, fake, 8, 1, 64, 16, None, None) == -1
    # misaligned
    assert lib.paged_kv_write(fake + 2, fake, fake, 4, fake, fake, 8, 1, 64, 16, None, None) == -4
    # nothing to do is fine and touches nothing
    assert lib.paged_kv_write(None, None, None, 0, None, None, 8, 1, 64, 16, None, None) == 0
    assert lib.paged_block_copy(fake, fake, fake, 2, 8, 1, 64, 12, None, None) == -3
    assert lib.paged_block_copy(None, None, None, 0, 8, 1, 64, 16, None, None) == 0
    ws = lib.paged_attention_workspace_size(4, 8, 128, 1000, 512)
    assert ws > 0 and ws % 256 == 0
    args = lambda **kw: [kw.get("out", fake), fake, fake, fake, fake, fake, kw.get("S", 4), 8,
                         kw.get("Hq", 8), kw.get("Hkv", 2), kw.get("D", 128), kw.get("bs", 16),
                         16, ctypes.c_float(0.1), kw.get("part", 512), 1000, fake,
                         kw.get("ws", ws), None, None]
    assert lib.paged_attention_decode(*args(bs=32)) == -3
    assert lib.paged_attention_decode(*args(D=96)) == -2
    assert lib.paged_attention_decode(*args(Hq=6, Hkv=4)) == -2
    assert lib.paged_attention_decode(*args(part=100)) == -2
    assert lib.paged_attention_decode(*args(out=None)) == -1
    assert lib.paged_attention_decode(*args(ws=ws - 1)) == -5
    assert lib.paged_attention_decode(*args(S=0)) == 0
    assert lib.paged_attention_set_variant(7) == -14
    pre = lambda **kw: [kw.get("out", fake), kw.get("q", fake), fake, fake, fake, fake, fake,
                        kw.get("S", 4), kw.get("T", 64), 8, kw.get("Hq", 8), kw.get("Hkv", 2),
                        kw.get("D", 128), kw.get("bs", 16), 16, ctypes.c_float(0.1),
                        kw.get("maxq", 16), None, None]
    assert lib.paged_attention_prefill(*pre(bs=8)) == -3
    assert lib.paged_attention_prefill(*pre(D=80)) == -2
    assert lib.paged_attention_prefill(*pre(Hq=6, Hkv=4)) == -2
    assert lib.paged_attention_prefill(*pre(maxq=-1)) == -2
    assert lib.paged_attention_prefill(*pre(S=70000)) == -2
    assert lib.paged_attention_prefill(*pre(q=None)) == -1
    assert lib.paged_attention_prefill(*pre(out=fake + 4)) == -4
    assert lib.paged_attention_prefill(*pre(S=0)) == 0
    assert lib.paged_attention_prefill(*pre(T=0)) == 0


def test_fp8_per_head_host_validation():
    """The per-KV-head E4M3 entry points reject missing scale arrays and bad shapes on the
    host; with nothing to do they touch nothing."""
    from paged_kv_cache_272_gb300.ops import lib
    fake = 1 << 20
    w = lambda **kw: [fake, fake, fake, kw.get("T", 4), fake, fake, 8, 2, kw.get("D", 128),
                      kw.get("bs", 16), kw.get("ks", fake), kw.get("vs", fake), None, None]
    assert lib.paged_kv_write_fp8_per_head(*w(ks=None)) == -1
    assert lib.paged_kv_write_fp8_per_head(*w(vs=None)) == -1
    assert lib.paged_kv_write_fp8_per_head(*w(bs=8)) == -3
    assert lib.paged_kv_write_fp8_per_head(*w(D=72)) == -2
    assert lib.paged_kv_write_fp8_per_head(*w(T=0, ks=None, vs=None)) == 0
    ws = lib.paged_attention_workspace_size(4, 8, 128, 1000, 512)
    a = lambda **kw: [fake, fake, fake, fake, fake, fake, kw.get("S", 4), 8, 8, 2,
                      kw.get("D", 128), kw.get("bs", 16), 16, ctypes.c_float(0.1),
                      kw.get("ks", fake), kw.get("vs", fake), 512, 1000, fake,
                      kw.get("ws", ws), None, None]
    assert lib.paged_attention_decode_fp8_per_head(*a(ks=None)) == -1
    assert lib.paged_attention_decode_fp8_per_head(*a(vs=None)) == -1
    assert lib.paged_attention_decode_fp8_per_head(*a(D=96)) == -2
    assert lib.paged_attention_decode_fp8_per_head(*a(bs=32)) == -3
    assert lib.paged_attention_decode_fp8_per_head(*a(ws=ws - 1)) == -5
    assert lib.paged_attention_decode_fp8_per_head(*a(S=0, ks=None, vs=None)) == 0


def test_abi_version_matches_header():
    from paged_kv_cache_272_gb300 import ops
    m = re.search(r"#define PKV_ABI_VERSION (\d+)", open(HEADER).read())
    assert m and int(m.group(1)) == ops.ABI_VERSION == ops.lib.paged_kv_version()


def test_strerror():
    from paged_kv_cache_272_gb300.ops import lib
    for code in (0, -1, -2, -3, -4, -5, -6, -10, -11, -12, -13, -14, -99):
        assert lib.paged_kv_strerror(code)


def test_workspace_size_formula():
    from paged_kv_cache_272_gb300.ops import paged_attention_workspace_size as wsz
    # Partials dominate: S * max_parts * Hq * (D + 1) floats, plus one chunk result
    # (same shape) per 32 partitions, the work records, merge units and counters.
    S, Hq, D, P = 128, 64, 128, 256
    C, G8 = P // 32, Hq // 8
    n = wsz(S, Hq, D, 131072, 512)
    part = S * P * Hq * (D + 1) * 4
    chunk = S * C * Hq * (D + 1) * 4
    assert n >= part + chunk
    assert n < part + chunk + S * P * 16 + S * G8 * C * 16 + S * Hq * 4 + S * 4 + 16 * 256


def test_slot_mapping_check():
    import numpy as np
    from paged_kv_cache_272_gb300 import ops
    ops.paged_kv_check_slots(np.array([0, 5, 17, -1, -1, 63]), 4)
    ops.paged_kv_check_slots(np.zeros(0, np.int64), 4)
    with pytest.raises(ops.PagedKVError):
        ops.paged_kv_check_slots(np.array([3, 9, 3]), 4)       # two tokens, one slot
    with pytest.raises(ops.PagedKVError):
        ops.paged_kv_check_slots(np.array([64]), 4)             # past the pool


def test_selftest_bounded_wait_validates_on_host():
    """The bounded-wait self-test rejects null pointers (PKV_ERR_NULL) and out-of-range
    limits (PKV_ERR_SHAPE) before launching anything, so this runs without a GPU."""
    from paged_kv_cache_272_gb300 import ops
    ERR_NULL, ERR_SHAPE = -1, -2
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: validation fails first
    assert ops.lib.pkv_selftest_bounded_wait(None, fake, 1000, 0, None) == ERR_NULL
    assert ops.lib.pkv_selftest_bounded_wait(fake, None, 1000, 0, None) == ERR_NULL
    assert ops.lib.pkv_selftest_bounded_wait(fake, fake, 0, 0, None) == ERR_SHAPE
    assert ops.lib.pkv_selftest_bounded_wait(fake, fake, 1 << 40, 1, None) == ERR_SHAPE


def test_decode_step_host_validation():
    """The fused decode-step entry points check the write and copy arguments on the host
    before anything is enqueued."""
    from paged_kv_cache_272_gb300.ops import lib
    fake = 1 << 20
    ws = lib.paged_attention_workspace_size(4, 8, 128, 1000, 512)

    def st(**kw):
        return [fake, fake, fake, fake, fake, fake, kw.get("S", 4), 8, 8, 2, kw.get("D", 128),
                16, 16, ctypes.c_float(0.1), 512, 1000, kw.get("kn", fake), kw.get("vn", fake),
                kw.get("sl", fake), kw.get("T", 4), kw.get("pr", fake), kw.get("P", 2), fake,
                kw.get("ws", ws), None, None]
    assert lib.paged_decode_step(*st(kn=None)) == -1          # k_new missing
    assert lib.paged_decode_step(*st(sl=None)) == -1          # slot_mapping missing
    assert lib.paged_decode_step(*st(pr=None)) == -1          # pairs missing
    assert lib.paged_decode_step(*st(kn=fake + 8)) == -4      # k_new misaligned
    assert lib.paged_decode_step(*st(T=-1)) == -2
    assert lib.paged_decode_step(*st(P=-1)) == -2
    assert lib.paged_decode_step(*st(D=96)) == -2
    assert lib.paged_decode_step(*st(ws=ws - 1)) == -5

    def st8(**kw):
        return [fake, fake, fake, fake, fake, fake, 4, 8, 8, 2, kw.get("D", 128), 16, 16,
                ctypes.c_float(0.1), ctypes.c_float(kw.get("k", 0.02)), ctypes.c_float(0.015),
                kw.get("ks", None), kw.get("vs", None), 512, 1000, fake, fake, fake, 4, None, 0,
                fake, ws, None, None]
    assert lib.paged_decode_step_fp8(*st8(k=0.0)) == -2       # per-cache scale not > 0
    assert lib.paged_decode_step_fp8(*st8(ks=fake)) == -1     # one per-head array only
    assert lib.paged_decode_step_fp8(*st8(D=96)) == -2


def _c_layout(struct: str, fields):
    """(sizeof, {field: offsetof}) of a header struct, from a C program compiled with gcc."""
    import subprocess
    import tempfile
    body = "".join(f'  printf(" %zu", offsetof({struct}, {f}));\n' for f in fields)
    src = ("#include <stddef.h>\n#include <stdio.h>\n#include \"pagedkv.h\"\n"
           f"int main(void) {{\n  printf(\"%zu\", sizeof({struct}));\n{body}"
           "  printf(\"\\n\");\n  return 0;\n}\n")
    with tempfile.TemporaryDirectory() as d:
        c, exe = os.path.join(d, "layout.c"), os.path.join(d, "layout")
        with open(c, "w") as f:
            f.write(src)
        subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), c, "-o", exe],
                       check=True)
        vals = [int(x) for x in subprocess.run([exe], check=True, capture_output=True,
                                               text=True).stdout.split()]
    return vals[0], dict(zip(fields, vals[1:]))


@pytest.mark.parametrize("struct,pyname", [("pkv_step_io", "StepIO"),
                                           ("pkv_step_pack", "StepPack"),
                                           ("pkv_sched_stats", "SchedStats")])
def test_struct_layouts_match_the_header(struct, pyname):
    """The ctypes mirrors of the header's structs have the C compiler's size and field
    offsets (a mismatch would hand the library shifted pointers)."""
    from paged_kv_cache_272_gb300 import serving
    py = getattr(serving, pyname)
    names = [f[0] for f in py._fields_]
    size, offs = _c_layout(struct, names)
    assert ctypes.sizeof(py) == size
    for n in names:
        assert getattr(py, n).offset == offs[n], (struct, n)


def test_step_launch_and_gather_host_validation():
    """pkv_step_launch and paged_gather_rows reject bad arguments on the host, before
    anything is queued (so this runs without a GPU)."""
    from paged_kv_cache_272_gb300 import ops
    from paged_kv_cache_272_gb300.serving import StepIO, StepPack
    lib = ops.lib
    fake = 1 << 20
    # gather: row size not a multiple of 16, null, misaligned, too many vectors, n == 0
    assert lib.paged_gather_rows(fake, fake, fake, 4, 10, 24, None, None) == -2
    assert lib.paged_gather_rows(None, fake, fake, 4, 10, 32, None, None) == -1
    assert lib.paged_gather_rows(fake + 8, fake, fake, 4, 10, 32, None, None) == -4
    assert lib.paged_gather_rows(fake, fake, fake, 1 << 21, 10, 1 << 14, None, None) == -2
    assert lib.paged_gather_rows(fake, fake, fake, 4, 0, 32, None, None) == -2
    assert lib.paged_gather_rows(None, None, None, 0, 10, 32, None, None) == 0
    io, pk = StepIO(), StepPack()
    io.max_tokens, io.max_seqs, io.stage_bytes = 64, 8, 4096
    pk.total, pk.num_tokens, pk.num_seqs, pk.num_decode = 1024, 16, 4, 2
    assert lib.pkv_step_launch(None, ctypes.byref(pk), 0, None, None) == -1
    assert lib.pkv_step_launch(ctypes.byref(io), ctypes.byref(pk), 2, None, None) == -14
    pk.num_tokens = 65  # above the capacity
    assert lib.pkv_step_launch(ctypes.byref(io), ctypes.byref(pk), 0, None, None) == -2
    pk.num_tokens, pk.num_decode = 16, 5  # more decode entries than sequences
    assert lib.pkv_step_launch(ctypes.byref(io), ctypes.byref(pk), 0, None, None) == -2
    pk.num_decode, pk.total = 2, 8192  # pack larger than the staging buffer
    assert lib.pkv_step_launch(ctypes.byref(io), ctypes.byref(pk), 0, None, None) == -2
    pk.total = 1024  # buffers missing
    assert lib.pkv_step_launch(ctypes.byref(io), ctypes.byref(pk), 0, None, None) == -1
    pk.num_tokens = 0  # nothing to do
    assert lib.pkv_step_launch(ctypes.byref(io), ctypes.byref(pk), 0, None, None) == 0


def test_engine_step_host_validation():
    """pkv_engine_step checks its arguments first, and a step with nothing to schedule
    packs an empty plan and launches nothing (so this runs without a GPU)."""
    from paged_kv_cache_272_gb300 import ops
    from paged_kv_cache_272_gb300.block_pool import BlockPool
    from paged_kv_cache_272_gb300.serving import Scheduler, StepIO, StepPack
    lib = ops.lib
    pool = BlockPool(64)
    sched = Scheduler(pool, 4, 64)
    io, pk = StepIO(), StepPack()
    buf = (ctypes.c_uint8 * 65536)()
    io.host_stage[0] = io.host_stage[1] = ctypes.addressof(buf)
    io.stage_bytes, io.max_tokens, io.max_seqs, io.table_stride = 65536, 68, 4, 8
    assert lib.pkv_engine_step(None, ctypes.byref(io), ctypes.byref(pk), 0, None, None) == -1
    assert lib.pkv_engine_step(sched._h, None, ctypes.byref(pk), 0, None, None) == -1
    assert lib.pkv_engine_step(sched._h, ctypes.byref(io), ctypes.byref(pk), 3, None, None) == -14
    assert lib.pkv_engine_step(sched._h, ctypes.byref(io), ctypes.byref(pk), 1, None, None) == 0
    assert pk.num_tokens == 0 and pk.num_seqs == 0 and pk.total > 0
