"""Failure detection on the GPU without a fault: the bounded-wait self-test kernel waits on a
barrier that nothing completes; the wait gives up after about a second and raises the device
error word, kda_device_status reports 40008 once and clears it, and the context stays usable
(a decode step afterwards matches the oracle)."""

import time

import pytest
import torch

from gated_delta_rule_scan_gb300 import inputs
from tests.gpu_util import TOL, oracle_forward, rel_linf, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield


def test_bounded_wait_times_out_and_reports():
    from gated_delta_rule_scan_gb300 import kda, mixer
    assert kda.kda_device_status() == 0
    t0 = time.perf_counter()
    kda.kda_selftest_wait_timeout()
    assert kda.kda_device_status() == 40008
    elapsed = time.perf_counter() - t0
    assert 0.01 < elapsed < 60.0, elapsed
    assert kda.kda_device_status() == 0        # read once, then cleared
    inp = inputs.decode_step(N=2, T=1, H=2, seed=9)
    out = mixer.kda_decode(N=2, T=1, H=2, **to_dev(inp))
    torch.cuda.synchronize()
    ref = oracle_forward(inp)
    assert rel_linf(out["y"], ref["y"]) <= TOL
    assert kda.kda_device_status() == 0
