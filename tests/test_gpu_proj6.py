"""GPU parity of kda_proj6, stage 1 of the mixer: the six projections of the layer input x by bf16
weights ("memra_engine/kda.rs", kda_core_gated stage 1 and Engine::kda_proj_fused6), through the
C ABI, against the f64 oracle on the same seeded inputs.

Bar: relative L-inf <= 1e-3 per output (the tensor-core products see the weights exactly and x
split into bf16 hi + lo, so the error is ~1e-6; a tighter 2e-5 check guards that split).  A token
row's outputs do not depend on the other rows of the call (bit-equal to a one-row call), and the
projections feed kda_decode_fused directly.
"""

import numpy as np
import pytest
import torch

from tests.gpu_util import TOL, rel_linf

pytestmark = pytest.mark.gpu

D = 128


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    from gated_delta_rule_scan_gb300 import kda
    assert kda.kda_device_status() == 0


def _weights(seed, H, in_f):
    """Random synthetic bf16 weights of the layer's shapes, std 1/sqrt(in_f), and x ~ N(0, 1)."""
    rng = np.random.default_rng(seed)
    dims = (H * D, H * D, H * D, D, D, H)
    ws = [torch.from_numpy((rng.standard_normal((r, in_f)) / np.sqrt(in_f)).astype(np.float32))
          .to(torch.bfloat16) for r in dims]
    return ws, dims


def _x(seed, t, in_f):
    rng = np.random.default_rng(seed + 1000)
    return torch.from_numpy(rng.standard_normal((t, in_f)).astype(np.float32))


def _gpu_proj(x, ws, dims, H):
    from gated_delta_rule_scan_gb300 import kda
    dev = torch.device("cuda")
    t, in_f = x.shape
    outs = [torch.full((t, r), float("nan"), device=dev) for r in dims]
    wd = [w.to(dev) for w in ws]
    kda.kda_proj6(x.to(dev), *wd, *outs, kda.proj6_workspace(t, in_f, dev), H=H)
    torch.cuda.synchronize()
    return outs


@pytest.mark.parametrize("t,H,in_f", [(1, 2, 256), (3, 2, 384), (16, 4, 512), (64, 3, 256),
                                      (17, 1, 128), (256, 1, 128)])
def test_proj6_vs_oracle(t, H, in_f):
    """Ragged token counts (padded to the MMA's N), partial weight tiles (beta: H < 128 rows),
    several K-stages, and the largest batch of 256 rows."""
    from oracle import oracle as orc
    ws, dims = _weights(t * 7 + H, H, in_f)
    x = _x(t * 7 + H, t, in_f)
    outs = _gpu_proj(x, ws, dims, H)
    refs = orc.proj6(x, *ws)
    for o, r in zip(outs, refs):
        assert torch.isfinite(o).all()
        e = rel_linf(o, r)
        assert e <= TOL and e <= 2e-5, e


def test_proj6_rows_independent():
    """Each token row of a 16-row call equals a one-row call on that row, bit for bit."""
    H, in_f, t = 2, 512, 16
    ws, dims = _weights(5, H, in_f)
    x = _x(5, t, in_f)
    full = _gpu_proj(x, ws, dims, H)
    for s in (0, 7, 15):
        one = _gpu_proj(x[s:s + 1].contiguous(), ws, dims, H)
        for a, b in zip(full, one):
            assert torch.equal(a[s:s + 1], b)


@pytest.mark.slow
def test_proj6_full_size():
    """The decode batch's projections: 64 token rows, 64 heads (q/k/v 8192 wide), hidden 6144."""
    from oracle import oracle as orc
    H, in_f, t = 64, 6144, 64
    ws, dims = _weights(9, H, in_f)
    x = _x(9, t, in_f)
    outs = _gpu_proj(x, ws, dims, H)
    refs = orc.proj6(x, *ws)
    for o, r in zip(outs, refs):
        assert rel_linf(o, r) <= TOL


def test_proj6_feeds_decode():
    """The projections as the decode kernel's raw q/k/v and beta (f32 raw rows): y, state and
    ring equal the oracle's mixer run on the oracle's own projections of the same x."""
    from gated_delta_rule_scan_gb300 import inputs, mixer
    from oracle import oracle as orc
    from tests.gpu_util import to_dev
    N, H, in_f = 4, 2, 256
    ws, dims = _weights(11, H, in_f)
    x = _x(11, N, in_f)                        # one token per sequence
    q, k, v, _, _, b = _gpu_proj(x, ws, dims, H)
    dec = inputs.decode_step(N=N, T=1, H=H, seed=12)
    d = to_dev(dec)
    d.update(q_raw=q, k_raw=k, v_raw=v, beta_raw=b)
    out = mixer.kda_decode(N=N, T=1, H=H, **d)
    torch.cuda.synchronize()
    rq, rk, rv, _, _, rb = orc.proj6(x, *ws)
    ref = orc.forward(q_raw=rq, k_raw=rk, v_raw=rv, beta_raw=rb, f_raw=dec.f_raw,
                      dt_bias=dec.dt_bias, a_log=dec.a_log, state_in=dec.state_in, H=H, D=D,
                      conv_w=dec.conv_w, ring_in=dec.ring_in, cu_seqlens=dec.cu_seqlens,
                      norm_w=dec.norm_w, gate_raw=dec.gate_raw)
    for key in ("y", "state_out"):
        assert rel_linf(out[key], ref[key]) <= TOL, key
    # the ring holds the projected raw rows themselves: f32 GPU values against f64 oracle values
    assert rel_linf(out["ring_out"], ref["ring_out"]) <= 2e-5


def test_proj6_contract():
    from gated_delta_rule_scan_gb300 import kda
    H, in_f, t = 1, 128, 2
    ws, dims = _weights(13, H, in_f)
    dev = torch.device("cuda")
    wd = [w.to(dev) for w in ws]
    outs = [torch.empty((t, r), device=dev) for r in dims]
    x = _x(13, t, in_f).to(dev)
    wsp = kda.proj6_workspace(t, in_f, dev)
    with pytest.raises(kda.KdaError) as e:
        kda.kda_proj6(x, *wd, *outs, wsp[:16], H=H)
    assert e.value.status == 40009
    with pytest.raises(kda.KdaError) as e:
        kda.kda_proj6(x[:, :100].contiguous(), *wd, *outs, wsp, H=H)
    assert e.value.status == 40005
