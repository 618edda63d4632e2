"""GPU parity of a value head wider than the key head (kda_conv_l2norm_prep_dv, kda_scan_dv,
their varlen forms, and the gated RMSNorm over rows of Dv values): the GDN page's separate
head_k_dim and head_v_dim (aprender-serve gdn_ops.rs `gdn_delta_rule_into` doc), with a
head_v_dim x head_k_dim state per value head.

(1) The staged mixer against the oracle's rectangular-state mixer, in the sequential and the
chunked form, per-channel and per-head gate, with and without grouped queries, uniform and packed
sequences.  (2) By the recurrence, value column block b of value head h is an ordinary 128-wide
head that reads value head h's gate, beta and q/k head, so kda_scan_dv must equal kda_scan with
H * Dv / 128 heads on inputs re-indexed that way, bit for bit (the same arithmetic per unit)."""

import numpy as np
import pytest
import torch

from gated_delta_rule_scan_gb300 import inputs
from tests.gpu_util import check_all_heads, gpu_forward

pytestmark = pytest.mark.gpu

MIX = ("y", "o", "state_out", "ring_out", "v_hat", "beta")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    from gated_delta_rule_scan_gb300 import kda
    assert kda.kda_device_status() == 0


@pytest.mark.parametrize("algo", [1, 2])
@pytest.mark.parametrize("H,Hk,Dv,gate_mode,raw", [(2, None, 256, 0, "bf16"),
                                                  (3, None, 256, 1, "f32"),
                                                  (2, 1, 384, 0, "bf16"),
                                                  (4, 2, 256, 1, "bf16"),
                                                  (1, None, 1024, 0, "f32")])
def test_value_width_mixer(algo, H, Hk, Dv, gate_mode, raw):
    """Two sequences of 75 tokens (a ragged last chunk), random state and ring; the GDN gate
    with the SiLU-gated norm, the KDA gate with the sigmoid-gated norm."""
    inp = inputs.make_inputs(300 + 7 * H + Dv // 128 + algo, H=H, N=2, T=75, raw_dtype=raw,
                             conv=True, ring="randn", gate_mode=gate_mode, state="randn",
                             epilogue=True, Hk=Hk, Dv=Dv)
    ng = "silu" if gate_mode == 1 else "sigmoid"
    out = gpu_forward(inp, algo=algo, norm_gate=ng, gate_exp=False)
    check_all_heads(out, inp, MIX + ("g",), norm_gate=ng)


@pytest.mark.parametrize("algo", [1, 2])
def test_value_width_varlen_edges(algo):
    """Packed sequences with empty ones, lengths below the conv window and around the chunk."""
    lengths = [5, 0, 1, 2, 33, 64, 70]
    H, Hk, Dv = 3, 1, 256
    cu = np.concatenate([[0], np.cumsum(lengths)])
    rows = int(cu[-1])
    inp = inputs.make_inputs(331, H=H, N=len(lengths), lengths=(0, 1), raw_dtype="bf16",
                             conv=True, ring="randn", state="randn", epilogue=True, Hk=Hk, Dv=Dv)
    rng = np.random.default_rng(1331)

    def draw(shape):
        return torch.from_numpy(rng.standard_normal(shape).astype(np.float32))
    inp.q_raw = draw((rows, Hk * 128)).to(torch.bfloat16)
    inp.k_raw = draw((rows, Hk * 128)).to(torch.bfloat16)
    inp.v_raw = draw((rows, H * Dv)).to(torch.bfloat16)
    inp.f_raw = draw((rows, H * 128))
    inp.beta_raw = draw((rows, H))
    inp.gate_raw = draw((rows, H * Dv))
    inp.cu_seqlens = cu
    out = gpu_forward(inp, varlen=True, algo=algo)
    check_all_heads(out, inp, ("y", "state_out", "ring_out"))


@pytest.mark.parametrize("algo", [1, 2])
@pytest.mark.parametrize("gate_mode", [0, 1])
def test_value_width_scan_is_column_blocks(algo, gate_mode):
    """kda_scan_dv == kda_scan over the value column blocks as heads, bit for bit."""
    from gated_delta_rule_scan_gb300 import kda
    H, Hk, Dv, N, T = 3, 1, 384, 2, 90
    m, rows = Dv // 128, N * T
    rng = np.random.default_rng(41 + gate_mode)

    def unit(h):
        x = rng.standard_normal((rows, h, 128))
        return (x / np.linalg.norm(x, axis=-1, keepdims=True)).reshape(rows, h * 128)
    q, k = unit(Hk), unit(Hk)
    v = rng.standard_normal((rows, H * Dv))
    gw = H * 128 if gate_mode == 0 else H
    g = -5.0 / (1 + np.exp(-rng.standard_normal((rows, gw))))
    beta = 1 / (1 + np.exp(-rng.standard_normal((rows, H))))
    s0 = 0.02 * rng.standard_normal((N, H, Dv, 128))
    f32 = lambda x: torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()  # noqa: E731
    ws = kda.scan_workspace(N, rows, H * m, "cuda", algo)
    st = torch.empty(N, H, Dv, 128, device="cuda")
    o = torch.empty(rows, H * Dv, device="cuda")
    kda.kda_scan_dv(f32(q), f32(k), f32(v), f32(g), f32(beta), f32(s0), st, o, N=N, T=T, H=H,
                    Hk=Hk, Dv=Dv, gate_mode=gate_mode, algo=algo, workspace=ws)
    # unit u = h * m + b reads q/k head h % Hk, the gate and beta of value head h
    unit_head = np.arange(H * m) // m
    qe = q.reshape(rows, Hk, 128)[:, unit_head % Hk].reshape(rows, H * m * 128)
    ke = k.reshape(rows, Hk, 128)[:, unit_head % Hk].reshape(rows, H * m * 128)
    ge = (g.reshape(rows, H, 128)[:, unit_head].reshape(rows, H * m * 128) if gate_mode == 0
          else g[:, unit_head])
    be = beta[:, unit_head]
    st2 = torch.empty(N, H * m, 128, 128, device="cuda")
    o2 = torch.empty(rows, H * m * 128, device="cuda")
    kda.kda_scan(f32(qe), f32(ke), f32(v), f32(ge), f32(be), f32(s0).reshape(N, H * m, 128, 128),
                 st2, o2, N=N, T=T, H=H * m, gate_mode=gate_mode, algo=algo, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(o, o2)
    assert torch.equal(st.reshape(N, H * m, 128, 128), st2)


def test_value_width_norm_rows():
    """The gated RMSNorm over rows of 256 and 1024 values against the oracle's norm."""
    from gated_delta_rule_scan_gb300 import kda
    from oracle import oracle as orc
    from tests.gpu_util import rel_linf
    rng = np.random.default_rng(77)
    for width, rows, silu in ((256, 37, False), (1024, 9, True), (512, 1, False)):
        o = rng.standard_normal((rows, width)).astype(np.float32)
        w = (1 + 0.1 * rng.standard_normal(width)).astype(np.float32)
        z = rng.standard_normal((rows, width)).astype(np.float32)
        y = torch.empty(rows, width, device="cuda")
        fn = kda.kda_gated_rmsnorm_silu_out if silu else kda.kda_gated_rmsnorm_out
        fn(torch.from_numpy(o).cuda(), torch.from_numpy(w).cuda(), torch.from_numpy(z).cuda(), y,
           rows=rows, D=width)
        torch.cuda.synchronize()
        ref = orc.gated_rmsnorm(o, w, z, 1e-6, gate="silu" if silu else "sigmoid")
        assert rel_linf(y, ref) <= 1e-5, width
