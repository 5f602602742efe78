"""Every ring shape of the tensor-core kernel (consumer warps x stages, chosen once per
process through PKV_MMA_RING) on partitions shorter and longer than 32 blocks, with the
bf16 and the E4M3 cache, checked against the oracle in a fresh process each."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

SCRIPT = r"""
import sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {here!r})
import gpu_helpers as H
from paged_kv_cache_272_gb300 import workloads
w = workloads.build("rings", [1, 17, 40, 600, 1111, 2999], 16, 2, 128, seed=7, device="cuda")
ko, vo = H.oracle_caches(w)
ref = H.oracle_out(w, ko, vo)
for P in (64, 512, 1024, 8192):
    out, k, v, err = H.gpu_step(w, 2, partition_size=P)
    assert err == 0, (P, err)
    H.assert_attention_close(out, ref, "ring {ring} partition %d" % P)
for P in (64, 512, 8192):
    out, kq, vq, ko8, vo8, err = H.fp8_step(w, partition_size=P)
    assert err == 0, (P, err)
    H.assert_attention_close(out, H.fp8_ref(w, ko8, vo8), "ring {ring} E4M3 partition %d" % P)
print("ok")
"""


@pytest.mark.parametrize("ring", ["3x2", "4x2", "2x3", "8x2", "4x4", "4x3", "2x2", "2x4", "3x3"])
def test_ring_shape(ring):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, PKV_MMA_RING=ring)
    r = subprocess.run([sys.executable, "-c", SCRIPT.format(root=ROOT, here=HERE, ring=ring)],
                       env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]
