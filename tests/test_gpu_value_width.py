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
from tests.gpu_util import check_all_heads, gpu_forward, rel_linf

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


# ---- the fused entries: prefill (prep + chunked scan + RMSNorm over Dv) and decode / verify /
#      rollback (a value head = a thread-block cluster of Dv / 128 CTAs) ---------------------------

from tests.gpu_util import gpu_prefill, to_dev  # noqa: E402

FUSED = ("y", "state_out", "ring_out")


@pytest.mark.parametrize("H,Hk,Dv,gate_mode,raw,K", [(2, None, 256, 0, "bf16", 4),
                                                    (2, 1, 384, 1, "bf16", 4),
                                                    (3, 3, 256, 0, "bf16", 4),
                                                    (2, 1, 256, 0, "f32", 4),
                                                    (2, 2, 256, 1, "bf16", 6)])
def test_value_width_fused_prefill(H, Hk, Dv, gate_mode, raw, K):
    """kda_prefill_fused_dv against the oracle and bit-equal to the staged chunked path (prep_dv,
    scan_dv, the RMSNorm over Dv); two sequences of 75 tokens, random state and ring; bf16 raw
    rows (staged by TMA) and f32 raw rows (loaded directly), conv widths 4 and 6."""
    inp = inputs.make_inputs(400 + 7 * H + Dv // 128 + K, H=H, N=2, T=75, raw_dtype=raw,
                             conv=True, ring="randn", gate_mode=gate_mode, state="randn",
                             epilogue=True, Hk=Hk, Dv=Dv, K=K)
    fused = gpu_prefill(inp)
    check_all_heads(fused, inp, FUSED)
    staged = gpu_forward(inp, algo=2)
    for k in FUSED:
        assert torch.equal(fused[k], staged[k]), k


def test_value_width_fused_prefill_varlen():
    """Packed sequences with empty ones and lengths around the conv window and the chunk."""
    lengths = [5, 0, 1, 2, 33, 64, 70]
    H, Hk, Dv = 2, 1, 256
    cu = np.concatenate([[0], np.cumsum(lengths)])
    rows = int(cu[-1])
    inp = inputs.make_inputs(431, H=H, N=len(lengths), lengths=(0, 1), raw_dtype="bf16",
                             conv=True, ring="randn", state="randn", epilogue=True, Hk=Hk, Dv=Dv)
    rng = np.random.default_rng(1431)

    def draw(shape):
        return torch.from_numpy(rng.standard_normal(shape).astype(np.float32))
    inp.q_raw = draw((rows, Hk * 128)).to(torch.bfloat16)
    inp.k_raw = draw((rows, Hk * 128)).to(torch.bfloat16)
    inp.v_raw = draw((rows, H * Dv)).to(torch.bfloat16)
    inp.f_raw = draw((rows, H * 128))
    inp.beta_raw = draw((rows, H))
    inp.gate_raw = draw((rows, H * Dv))
    inp.cu_seqlens = cu
    fused = gpu_prefill(inp, varlen=True)
    check_all_heads(fused, inp, FUSED)
    staged = gpu_forward(inp, varlen=True, algo=2)
    for k in FUSED:
        assert torch.equal(fused[k], staged[k]), k


def _decode_step(d, N, T, t, H, Hk, Dv, state, ring, norm_gate="sigmoid", gate_mode=0, K=4):
    from gated_delta_rule_scan_gb300 import mixer
    rows = torch.arange(N, device="cuda") * T + t
    step = {k: d[k] for k in ("conv_w", "dt_bias", "a_log", "norm_w")}
    for k in ("q_raw", "k_raw", "v_raw", "f_raw", "beta_raw", "gate_raw"):
        step[k] = d[k][rows].contiguous()
    return mixer.kda_decode(N=N, T=1, H=H, Hk=Hk, Dv=Dv, K=K, state_in=state, ring_in=ring,
                            norm_gate=norm_gate, gate_mode=gate_mode, **step)


@pytest.mark.parametrize("H,Hk,Dv,T,gate_mode,raw,K", [(2, 1, 256, 1, 0, "bf16", 4),
                                                       (3, 3, 256, 4, 0, "bf16", 4),
                                                       (2, 2, 512, 4, 1, "bf16", 4),
                                                       (1, 1, 1024, 2, 0, "bf16", 4),
                                                       (2, 1, 256, 3, 0, "f32", 6)])
def test_value_width_decode_verify(H, Hk, Dv, T, gate_mode, raw, K):
    """kda_decode_fused_dv against the oracle; a T-token call bit-equal to T chained one-token
    calls; the staged sequential path (prep_dv, scan_dv, RMSNorm over Dv) equal to f32 rounding,
    the ring bit for bit (the two scans sum the key dimension over different lane groupings)."""
    from gated_delta_rule_scan_gb300 import mixer
    N = 5
    ng = "silu" if gate_mode == 1 else "sigmoid"
    inp = inputs.make_inputs(440 + T + Dv // 128, H=H, N=N, T=T, raw_dtype=raw, conv=True,
                             ring="randn", gate_mode=gate_mode, state="randn", epilogue=True,
                             Hk=Hk, Dv=Dv, K=K)
    d = to_dev(inp)
    full = mixer.kda_decode(N=N, T=T, H=H, Hk=Hk, Dv=Dv, K=K, norm_gate=ng, gate_mode=gate_mode,
                            **d)
    torch.cuda.synchronize()
    check_all_heads(full, inp, FUSED, norm_gate=ng)
    staged = gpu_forward(inp, algo=1, norm_gate=ng)
    assert torch.equal(full["ring_out"], staged["ring_out"])
    for k in ("y", "state_out"):
        assert rel_linf(full[k], staged[k]) <= 1e-5, k
    state, ring = d["state_in"], d["ring_in"]
    ys = []
    for t in range(T):
        r = _decode_step(d, N, T, t, H, Hk, Dv, state, ring, ng, gate_mode, K)
        state, ring = r["state_out"], r["ring_out"]
        ys.append(r["y"].view(N, 1, -1))
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(ys, dim=1).view(N * T, -1), full["y"])
    assert torch.equal(state, full["state_out"])
    assert torch.equal(ring, full["ring_out"])


def test_value_width_rollback_and_in_place_refusal():
    """kda_verify_rollback_dv equals keep[n] chained one-token decodes; rolling the ring in place
    is refused when a value head spans several units (40003)."""
    from gated_delta_rule_scan_gb300 import kda, mixer
    N, H, Hk, Dv, T = 4, 2, 2, 256, 4
    inp = inputs.make_inputs(450, H=H, N=N, T=T, raw_dtype="bf16", conv=True, ring="randn",
                             state="randn", epilogue=True, Hk=Hk, Dv=Dv)
    d = to_dev(inp)
    keep_h = np.array([0, 1, 3, 4], dtype=np.int32)
    keep = torch.from_numpy(keep_h).cuda()
    rb = mixer.kda_verify_rollback(N=N, T=T, H=H, Hk=Hk, Dv=Dv, keep=keep, **d)
    torch.cuda.synchronize()
    for n in range(N):
        state = d["state_in"][n:n + 1]
        ring = d["ring_in"][n:n + 1]
        for t in range(int(keep_h[n])):
            row = slice(n * T + t, n * T + t + 1)
            step = {k: d[k] for k in ("conv_w", "dt_bias", "a_log", "norm_w")}
            for k in ("q_raw", "k_raw", "v_raw", "f_raw", "beta_raw", "gate_raw"):
                step[k] = d[k][row].contiguous()
            r = mixer.kda_decode(N=1, T=1, H=H, Hk=Hk, Dv=Dv, state_in=state, ring_in=ring,
                                 **step)
            assert torch.equal(r["y"], rb["y"][row])
            state, ring = r["state_out"], r["ring_out"]
        torch.cuda.synchronize()
        assert torch.equal(state, rb["state_out"][n:n + 1])
        assert torch.equal(ring, rb["ring_out"][n:n + 1])
    ring = d["ring_in"].clone()
    with pytest.raises(kda.KdaError) as e:
        mixer.kda_decode(N=N, T=T, H=H, Hk=Hk, Dv=Dv, ring_out=ring, **dict(d, ring_in=ring))
    assert e.value.status == 40003
