"""Both placements of the tcgen05 chunked-prefill kernel's P tile (chosen once per
process through PKV_PREFILL_P: "tmem", the default, or "smem"): the prefill parity
tests of the tcgen05 variant, then repeated calls on the full-size workload with the
device error flag checked (the P-ready barriers must never run a phase ahead)."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

REPEAT = r"""
import sys
sys.path.insert(0, {root!r})
import torch
from paged_kv_cache_272_gb300 import ops as o, workloads as W
o.set_prefill_variant(o.PKV_PREFILL_TC)
for cfg in (2, 3):
    w = W.make_prefill_config(cfg, device="cuda")
    k, v = w.k_cache.clone(), w.v_cache.clone()
    o.paged_kv_write(w.k_new, w.v_new, torch.as_tensor(w.slot_mapping, device="cuda"), k, v)
    out = torch.empty_like(w.q)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    args = (torch.as_tensor(w.block_tables, device="cuda"), torch.as_tensor(w.context_lens, device="cuda"),
            torch.as_tensor(w.query_start, device="cuda"), w.scale, w.max_query_len)
    for _ in range(40):
        o.paged_attention_prefill(out, w.q, k, v, *args, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, (cfg, int(err.item()))
print("ok")
"""


def _run(args, placement, script=None):
    env = dict(os.environ, PKV_PREFILL_P=placement)
    cmd = [sys.executable] + (["-c", script] if script else args)
    return subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=900, cwd=ROOT)


@pytest.mark.parametrize("placement", ["smem", "tmem"])
def test_prefill_parity_per_p_placement(placement):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    r = _run(["-m", "pytest", os.path.join(HERE, "test_gpu_prefill.py"), "-q", "-x", "-m", "gpu",
              "-k", "tc or long or tiny", "-p", "no:cacheprovider"], placement)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]


@pytest.mark.parametrize("placement", ["smem", "tmem"])
def test_repeated_calls_per_p_placement(placement):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    r = _run(None, placement, REPEAT.format(root=ROOT))
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]
