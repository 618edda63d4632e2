"""GPU tests of mixer.HostPrefillStream: batches held in pinned host memory, copied in, run
through kda_prefill and copied out on three pipelined streams.  Every batch's results must equal,
bit for bit, those of a plain kda_prefill on the same inputs (same kernels, same order), whatever
the number of batches in flight; one batch is also checked against the f64 oracle."""

import dataclasses

import numpy as np
import pytest
import torch

from gated_delta_rule_scan_gb300 import inputs
from tests.gpu_util import TOL, gpu_prefill, oracle_forward, rel_linf

pytestmark = pytest.mark.gpu

WEIGHTS = ("conv_w", "dt_bias", "a_log", "norm_w")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    from gated_delta_rule_scan_gb300 import kda
    assert kda.kda_device_status() == 0


def _batches(n, N, T, H, gate_mode=0):
    """n seeded batches sharing the first one's weights (the weights are model parameters)."""
    base = inputs.make_inputs(300, H=H, N=N, T=T, raw_dtype="bf16", conv=True, ring="randn",
                              state="randn", epilogue=True, gate_mode=gate_mode)
    out = [base]
    for i in range(1, n):
        b = inputs.make_inputs(300 + i, H=H, N=N, T=T, raw_dtype="bf16", conv=True,
                               ring="randn", state="randn", epilogue=True, gate_mode=gate_mode)
        out.append(dataclasses.replace(b, **{k: getattr(base, k) for k in WEIGHTS}))
    return out


def _pinned(t):
    return t.contiguous().pin_memory()


@pytest.mark.parametrize("slots,gate_mode", [(2, 0), (3, 0), (2, 1)])
def test_host_stream_matches_prefill(slots, gate_mode):
    from gated_delta_rule_scan_gb300 import mixer
    N, T, H, n = 2, 203, 3, 5
    batches = _batches(n, N, T, H, gate_mode)
    w = {k: getattr(batches[0], k).cuda() for k in WEIGHTS}
    host_in = [{k: _pinned(getattr(b, k)) for k in mixer.HostPrefillStream.BATCH_KEYS}
               for b in batches]
    pipe = mixer.HostPrefillStream(like=host_in[0], H=H, N=N, T=T, K=batches[0].K,
                                   gate_mode=gate_mode, slots=slots, **w)
    host_out = [dict(y=torch.empty(N * T, H * 128).pin_memory(),
                     state_out=torch.empty_like(h["state_in"]).pin_memory(),
                     ring_out=torch.empty_like(h["ring_in"]).pin_memory()) for h in host_in]
    for hi, ho in zip(host_in, host_out):
        pipe.submit(hi, ho)
    done = torch.cuda.Event()
    pipe.record_done(done)
    done.synchronize()
    assert pipe.submitted == n
    assert pipe.h2d_bytes_per_batch == sum(t.numel() * t.element_size()
                                           for t in host_in[0].values())
    for b, ho in zip(batches, host_out):
        ref = gpu_prefill(b)
        for k in ("y", "state_out", "ring_out"):
            assert torch.equal(ho[k], ref[k].cpu()), k
    ora = oracle_forward(batches[-1])
    assert rel_linf(host_out[-1]["y"], ora["y"]) <= TOL
    assert rel_linf(host_out[-1]["state_out"], ora["state_out"]) <= TOL
    assert np.array_equal(host_out[-1]["ring_out"].double().numpy(), ora["ring_out"])


def test_host_stream_without_conv():
    """A mixer without the short conv: no ring buffer is copied either way."""
    from gated_delta_rule_scan_gb300 import mixer
    N, T, H = 1, 100, 2
    b = inputs.make_inputs(310, H=H, N=N, T=T, raw_dtype="bf16", conv=False, state="randn",
                           epilogue=True)
    keys = [k for k in mixer.HostPrefillStream.BATCH_KEYS if k != "ring_in"]
    hi = {k: _pinned(getattr(b, k)) for k in keys}
    pipe = mixer.HostPrefillStream(like=hi, conv_w=None, dt_bias=b.dt_bias.cuda(),
                                   a_log=b.a_log.cuda(), norm_w=b.norm_w.cuda(), H=H, N=N, T=T)
    ho = dict(y=torch.empty(N * T, H * 128).pin_memory(),
              state_out=torch.empty_like(hi["state_in"]).pin_memory())
    for _ in range(3):      # the same batch three times: identical results each time
        pipe.submit(hi, ho)
    pipe.synchronize()
    ref = gpu_prefill(b)
    assert torch.equal(ho["y"], ref["y"].cpu())
    assert torch.equal(ho["state_out"], ref["state_out"].cpu())
