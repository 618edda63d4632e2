"""GPU parity of the grouped-query scans (kda_scan_gqa, kda_scan_varlen_gqa): q and k hold Hk
heads and value head h reads q/k head h % Hk.  By that definition the result is the ordinary scan
on q/k re-indexed to H heads, so (1) the f64 oracle on the re-indexed inputs is the reference and
(2) kda_scan on the re-indexed inputs must agree bit for bit (the same arithmetic per head), in
the sequential and the chunked form, per-channel and per-head gate."""

import numpy as np
import pytest
import torch

from gated_delta_rule_scan_gb300 import inputs
from tests.gpu_util import TOL, rel_linf

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    from gated_delta_rule_scan_gb300 import kda
    assert kda.kda_device_status() == 0


def _planes(seed, rows, H, Hk, gate_mode):
    rng = np.random.default_rng(seed)
    D = 128

    def unit(h):
        x = rng.standard_normal((rows, h, D))
        return (x / np.linalg.norm(x, axis=-1, keepdims=True)).reshape(rows, h * D)
    q, k = unit(Hk), unit(Hk)
    v = rng.standard_normal((rows, H * D))
    g = -5.0 / (1 + np.exp(-rng.standard_normal((rows, H * D if gate_mode == 0 else H))))
    beta = 1 / (1 + np.exp(-rng.standard_normal((rows, H))))
    return q, k, v, g, beta


def _expand(x, H, Hk):
    """q/k of Hk heads -> H heads, head h = head h % Hk."""
    rows = x.shape[0]
    x = x.reshape(rows, Hk, 128)
    return np.ascontiguousarray(x[:, np.arange(H) % Hk]).reshape(rows, H * 128)


@pytest.mark.parametrize("algo", [1, 2])
@pytest.mark.parametrize("H,Hk,gate_mode", [(4, 2, 0), (6, 3, 1), (5, 2, 0), (3, 1, 1)])
def test_gqa_scan(algo, H, Hk, gate_mode):
    from gated_delta_rule_scan_gb300 import kda
    from oracle import oracle as orc
    N, T = 2, 70
    rows = N * T
    q, k, v, g, beta = _planes(H * 10 + Hk + algo, rows, H, Hk, gate_mode)
    rng = np.random.default_rng(5)
    s0 = 0.02 * rng.standard_normal((N, H, 128, 128))
    f32 = lambda x: torch.from_numpy(np.asarray(x, dtype=np.float32)).cuda().contiguous()  # noqa: E731
    ws = kda.scan_workspace(N, rows, H, "cuda", algo)
    st, o = torch.empty(N, H, 128, 128, device="cuda"), torch.empty(rows, H * 128, device="cuda")
    kda.kda_scan_gqa(f32(q), f32(k), f32(v), f32(g), f32(beta), f32(s0), st, o, N=N, T=T, H=H,
                     Hk=Hk, gate_mode=gate_mode, algo=algo, workspace=ws)
    qe, ke = _expand(q, H, Hk), _expand(k, H, Hk)
    st2, o2 = torch.empty_like(st), torch.empty_like(o)
    kda.kda_scan(f32(qe), f32(ke), f32(v), f32(g), f32(beta), f32(s0), st2, o2, N=N, T=T, H=H,
                 gate_mode=gate_mode, algo=algo, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(o, o2)
    assert torch.equal(st, st2)
    cu = np.arange(N + 1, dtype=np.int64) * T
    shp = (rows, H, 128)
    gg = g.reshape(shp) if gate_mode == 0 else np.repeat(g.reshape(rows, H, 1), 128, axis=2)
    ref_o, ref_s = orc.scan_kda(qe.astype(np.float32).astype(np.float64).reshape(shp),
                                ke.astype(np.float32).astype(np.float64).reshape(shp),
                                v.astype(np.float32).astype(np.float64).reshape(shp),
                                gg.astype(np.float32).astype(np.float64),
                                beta.astype(np.float32).astype(np.float64),
                                s0.astype(np.float32).astype(np.float64), cu, None)
    assert rel_linf(o, ref_o.reshape(rows, H * 128)) <= TOL
    assert rel_linf(st, ref_s) <= TOL


def test_gqa_varlen_and_contract():
    from gated_delta_rule_scan_gb300 import kda
    H, Hk = 4, 2
    lengths = [0, 33, 5, 96]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32)
    rows = int(cu[-1])
    q, k, v, g, beta = _planes(21, rows, H, Hk, 0)
    f32 = lambda x: torch.from_numpy(np.asarray(x, dtype=np.float32)).cuda().contiguous()  # noqa: E731
    s0 = torch.zeros(len(lengths), H, 128, 128, device="cuda")
    ws = kda.scan_workspace(len(lengths), rows, H, "cuda", 2)
    outs = []
    for qq, kk, fn in ((q, k, "gqa"), (_expand(q, H, Hk), _expand(k, H, Hk), "plain")):
        st, o = torch.empty_like(s0), torch.empty(rows, H * 128, device="cuda")
        if fn == "gqa":
            kda.kda_scan_varlen_gqa(f32(qq), f32(kk), f32(v), f32(g), f32(beta), s0, st, o,
                                    cu.cuda(), cu, H=H, Hk=Hk, algo=2, workspace=ws)
        else:
            kda.kda_scan_varlen(f32(qq), f32(kk), f32(v), f32(g), f32(beta), s0, st, o, cu.cuda(),
                                cu, H=H, algo=2, workspace=ws)
        torch.cuda.synchronize()
        outs.append((st, o))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    with pytest.raises(kda.KdaError) as e:
        kda.kda_scan_gqa(f32(q), f32(k), f32(v), f32(g), f32(beta), s0, s0.clone(),
                         torch.empty(rows, H * 128, device="cuda"), N=1, T=rows, H=H, Hk=0)
    assert e.value.status == 40005
