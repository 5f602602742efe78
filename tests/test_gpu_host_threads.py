"""Calls from several host threads at once, each on its own stream with its own
workspace, in a fresh process (so the library's first-call set-up -- kernel attributes,
occupancy, tensor maps -- runs concurrently): every result matches the oracle."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

SCRIPT = r"""
import sys, threading
sys.path.insert(0, {root!r}); sys.path.insert(0, {here!r})
import numpy as np, torch
import gpu_helpers as H
from paged_kv_cache_272_gb300 import workloads
o = H.ops()
ws_ = [workloads.build("threads-%d" % i, [40 + 300 * i, 1100, 2000 - 100 * i, 700], 16, 2, 128,
                       seed=300 + i, device="cuda") for i in range(4)]
refs = []
for w in ws_:
    ko, vo = H.oracle_caches(w)
    refs.append(H.oracle_out(w, ko, vo))
outs = [None] * 4
barrier = threading.Barrier(4)
def run(i):
    w = ws_[i]
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        d = H.to_cuda(w)
        st.synchronize()
        barrier.wait()  # first library calls of every thread at the same time
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        o.paged_kv_write(d["k_new"], d["v_new"], d["slots"], d["k"], d["v"], err_flag=err, stream=st)
        S, Hq, D = d["q"].shape
        out = torch.empty((S, Hq, D), dtype=torch.bfloat16, device="cuda")
        ws = o.alloc_workspace(S, Hq, D, w.max_context_len)
        o.paged_attention_decode(out, d["q"], d["k"], d["v"], d["bt"], d["ctx"], w.scale,
                                 w.max_context_len, ws, err_flag=err, stream=st)
        st.synchronize()
        outs[i] = (out, int(err.item()))
ts = [threading.Thread(target=run, args=(i,)) for i in range(4)]
for t in ts: t.start()
for t in ts: t.join()
for i in range(4):
    out, err = outs[i]
    assert err == 0, (i, err)
    H.assert_attention_close(out, refs[i], "thread %d" % i)
print("ok")
"""


def test_concurrent_first_calls_from_threads():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    r = subprocess.run([sys.executable, "-c", SCRIPT.format(root=ROOT, here=HERE)],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]
