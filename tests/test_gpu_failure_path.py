"""The kernels' failure path, exercised without a fault: a bounded wait that nothing
completes gives up after its limit, ORs PKV_DEV_TIMEOUT into the error word and returns;
the context stays usable (an attention call afterwards matches the oracle)."""
import pytest
import torch

import gpu_helpers as H
from paged_kv_cache_272_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("spin", [False, True])
def test_bounded_wait_gives_up_and_reports(spin):
    o = H.ops()
    limit = 2_000_000  # clock cycles, about a millisecond
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    res = torch.full((3,), -1, dtype=torch.int64, device="cuda")
    o.selftest_bounded_wait(err, res, limit, use_spin=spin)
    torch.cuda.synchronize()
    ok, cycles, abort = res.tolist()
    assert ok == 0 and abort == 1
    assert cycles >= limit
    assert int(err.item()) & o.DEV_TIMEOUT
    # the context is still usable
    w = workloads.build("after-timeout", [5, 300, 1200], 16, 2, 128, seed=77, device="cuda")
    out, k, v, e2 = H.gpu_step(w, 2)
    assert e2 == 0
    ko, vo = H.oracle_caches(w)
    H.assert_attention_close(out, H.oracle_out(w, ko, vo), "attention after a timeout")
