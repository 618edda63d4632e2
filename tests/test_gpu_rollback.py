"""GPU tests of kda_verify_rollback: after a T-token verify round, each sequence keeps its first
keep[n] tokens; the rolled-back state and ring must equal keep[n] chained one-token decode calls
from the pre-round state and ring, bit for bit, and the kept y rows must equal the verify's own
rows.  Rows past keep[n] are left as they were."""

import numpy as np
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
    from gated_delta_rule_scan_gb300 import kda
    assert kda.kda_device_status() == 0


def _chain(d, N, T, H, keep):
    """keep[n] one-token decode calls per sequence (all sequences stepped together; a sequence
    past its keep count keeps its state and ring)."""
    from gated_delta_rule_scan_gb300 import mixer
    state, ring = d["state_in"].clone(), d["ring_in"].clone()
    for t in range(max(keep)):
        rows = torch.arange(N, device="cuda") * T + t
        step = {k: d[k] for k in ("conv_w", "dt_bias", "a_log", "norm_w")}
        for k in ("q_raw", "k_raw", "v_raw", "f_raw", "beta_raw", "gate_raw"):
            step[k] = d[k][rows].contiguous()
        r = mixer.kda_decode(N=N, T=1, H=H, state_in=state, ring_in=ring, **step)
        live = torch.tensor([t < k for k in keep], device="cuda")
        state = torch.where(live.view(N, 1, 1, 1), r["state_out"], state)
        ring = torch.where(live.view(N, 1, 1), r["ring_out"], ring)
    return state, ring


@pytest.mark.parametrize("T", [2, 4, 16])
def test_rollback_equals_chained_decode(T):
    from gated_delta_rule_scan_gb300 import kda, mixer
    N, H = 8, 16
    C = H * 128
    inp = inputs.decode_step(N=N, T=T, H=H, seed=40 + T)
    d = to_dev(inp)
    rng = np.random.default_rng(T)
    keep = [0, T] + [int(x) for x in rng.integers(0, T + 1, size=N - 2)]
    full = mixer.kda_decode(N=N, T=T, H=H, **d)              # the verify round
    torch.cuda.synchronize()
    keep_d = torch.tensor(keep, dtype=torch.int32, device="cuda")
    state_out = torch.empty_like(d["state_in"])
    ring_out = torch.empty_like(d["ring_in"])
    sentinel = 12345.0
    y = torch.full((N * T, C), sentinel, device="cuda")
    kda.kda_verify_rollback(d["q_raw"], d["k_raw"], d["v_raw"], d["conv_w"], d["ring_in"],
                            ring_out, d["f_raw"], d["dt_bias"], d["a_log"], d["beta_raw"],
                            d["state_in"], state_out, d["norm_w"], d["gate_raw"], y, keep_d,
                            N=N, T=T, H=H)
    torch.cuda.synchronize()
    state_ref, ring_ref = _chain(d, N, T, H, keep)
    assert torch.equal(state_out, state_ref)
    assert torch.equal(ring_out, ring_ref)
    yv, fv = y.view(N, T, C), full["y"].view(N, T, C)
    for n, k in enumerate(keep):
        assert torch.equal(yv[n, :k], fv[n, :k])
        assert bool((yv[n, k:] == sentinel).all())
    # a full accept is the verify itself; keep = 0 returns the pre-round state and ring
    n_full, n_none = 1, 0
    assert torch.equal(state_out[n_full], full["state_out"][n_full])
    assert torch.equal(ring_out[n_full], full["ring_out"][n_full])
    assert torch.equal(state_out[n_none], d["state_in"][n_none])
    assert torch.equal(ring_out[n_none], d["ring_in"][n_none])


def test_rollback_in_place_ring_against_oracle():
    """Ring rolled in place (ring_out is the pre-round copy), one kept prefix per sequence,
    checked against the f64 oracle run on the kept rows alone."""
    from gated_delta_rule_scan_gb300 import kda
    N, T, H = 4, 8, 8
    inp = inputs.decode_step(N=N, T=T, H=H, seed=77)
    d = to_dev(inp)
    keep = [3, 8, 1, 5]
    ring = d["ring_in"].clone()
    state_out = torch.empty_like(d["state_in"])
    y = torch.zeros(N * T, H * 128, device="cuda")
    kda.kda_verify_rollback(d["q_raw"], d["k_raw"], d["v_raw"], d["conv_w"], ring, ring,
                            d["f_raw"], d["dt_bias"], d["a_log"], d["beta_raw"], d["state_in"],
                            state_out, d["norm_w"], d["gate_raw"], y,
                            torch.tensor(keep, dtype=torch.int32, device="cuda"), N=N, T=T, H=H)
    torch.cuda.synchronize()
    # the oracle on the kept rows only: a varlen batch of lengths keep
    rows = np.concatenate([np.arange(n * T, n * T + k) for n, k in enumerate(keep)])
    sub = inputs.make_inputs(77, H=H, N=N, T=T, raw_dtype="bf16", conv=True, ring="randn",
                             gate_mode=0, state="randn", epilogue=True)
    for name in ("q_raw", "k_raw", "v_raw", "f_raw", "beta_raw", "gate_raw"):
        setattr(sub, name, getattr(inp, name)[torch.from_numpy(rows)])
    sub.cu_seqlens = np.concatenate([[0], np.cumsum(keep)]).astype(np.int64)
    ref = oracle_forward(sub)
    assert rel_linf(state_out, ref["state_out"]) <= TOL
    assert np.array_equal(ring.cpu().double().numpy(), ref["ring_out"])
    y_kept = y[torch.from_numpy(rows).cuda()]
    assert rel_linf(y_kept, ref["y"]) <= TOL
