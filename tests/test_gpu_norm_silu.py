"""GPU parity of the SiLU-gated RMSNorm mode (GDN's gated_rmsnorm: y = rmsnorm(o) * w * SiLU(z))
against the f64 oracle: the standalone kernel, the fused decode of a full GDN mixer (per-head
gate + SiLU norm) and the fused prefill; the fused prefill equals the staged chunked path with the
standalone SiLU norm bit for bit."""

import numpy as np
import pytest
import torch

from gated_delta_rule_scan_gb300 import inputs
from tests.gpu_util import TOL, gpu_forward, gpu_prefill, oracle_forward, rel_linf, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    from gated_delta_rule_scan_gb300 import kda
    assert kda.kda_device_status() == 0


def test_standalone_silu_norm_vs_oracle():
    from gated_delta_rule_scan_gb300 import kda
    from oracle import oracle as orc
    rng = np.random.default_rng(3)
    rows, D = 1000, 128
    o = rng.standard_normal((rows, D)).astype(np.float32)
    w = (1 + 0.1 * rng.standard_normal(D)).astype(np.float32)
    z = (3 * rng.standard_normal((rows, D))).astype(np.float32)
    y = torch.empty(rows, D, device="cuda")
    kda.kda_gated_rmsnorm_silu_out(torch.from_numpy(o).cuda(), torch.from_numpy(w).cuda(),
                                   torch.from_numpy(z).cuda(), y, rows=rows)
    torch.cuda.synchronize()
    ref = orc.gated_rmsnorm(o, w, z, 1e-6, gate="silu")
    assert rel_linf(y, ref) <= 1e-5
    # and the sigmoid kernel differs from it by exactly the factor z (to rounding)
    y_sig = torch.empty_like(y)
    kda.kda_gated_rmsnorm_out(torch.from_numpy(o).cuda(), torch.from_numpy(w).cuda(),
                              torch.from_numpy(z).cuda(), y_sig, rows=rows)
    torch.cuda.synchronize()
    assert rel_linf(y_sig.cpu().double().numpy() * z, ref) <= 1e-5


@pytest.mark.parametrize("T", [1, 3])
def test_gdn_mixer_decode_silu_norm(T):
    """A full GDN decode step: per-head gate, SiLU-gated norm."""
    from gated_delta_rule_scan_gb300 import mixer
    N, H = 6, 4
    inp = inputs.make_inputs(55 + T, H=H, N=N, T=T, raw_dtype="bf16", conv=True, ring="randn",
                             gate_mode=1, state="randn", epilogue=True)
    out = mixer.kda_decode(N=N, T=T, H=H, gate_mode=1, norm_gate="silu", **to_dev(inp))
    torch.cuda.synchronize()
    ref = oracle_forward(inp, norm_gate="silu")
    assert rel_linf(out["y"], ref["y"]) <= TOL
    assert rel_linf(out["state_out"], ref["state_out"]) <= TOL
    assert np.array_equal(out["ring_out"].cpu().double().numpy(), ref["ring_out"])
    # the sigmoid-gated output is a different one
    sig = mixer.kda_decode(N=N, T=T, H=H, gate_mode=1, **to_dev(inp))
    torch.cuda.synchronize()
    assert rel_linf(sig["y"], ref["y"]) > 1e-2


@pytest.mark.parametrize("gate_mode", [0, 1])
def test_prefill_fused_silu_norm(gate_mode):
    inp = inputs.make_inputs(66 + gate_mode, H=3, N=2, T=150, raw_dtype="bf16", conv=True,
                             ring="randn", gate_mode=gate_mode, state="randn", epilogue=True)
    fused = gpu_prefill(inp, norm_gate="silu")
    ref = oracle_forward(inp, norm_gate="silu")
    assert rel_linf(fused["y"], ref["y"]) <= TOL
    assert rel_linf(fused["state_out"], ref["state_out"]) <= TOL
    staged = gpu_forward(inp, algo=2, norm_gate="silu")
    assert torch.equal(fused["y"], staged["y"])
    assert torch.equal(fused["state_out"], staged["state_out"])
