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


# ------------------------------------------------------------------------------------------
# grouped queries through the whole mixer: prep, fused prefill, fused decode / verify, rollback
# ------------------------------------------------------------------------------------------

from tests.gpu_util import check_all_heads, gpu_forward, gpu_prefill, to_dev  # noqa: E402

MIX = ("y", "state_out", "ring_out")


@pytest.mark.parametrize("H,Hk,gate_mode,raw", [(4, 2, 0, "bf16"), (6, 3, 1, "bf16"),
                                                (5, 2, 0, "bf16"), (3, 1, 0, "bf16"),
                                                (4, 2, 0, "f32")])
def test_gqa_mixer_staged_and_fused(H, Hk, gate_mode, raw):
    """The staged mixer (prep_gqa -> scan_gqa -> RMSNorm, sequential and chunked) and the fused
    prefill against the oracle's grouped-query mixer; the fused prefill bit-equal to the staged
    chunked path.  Two sequences with a ragged last chunk, random state and ring; bf16 raw rows
    (staged into shared memory by TMA) and f32 raw rows (loaded directly)."""
    inp = inputs.make_inputs(200 + 10 * H + Hk, H=H, N=2, T=75, raw_dtype=raw, conv=True,
                             ring="randn", gate_mode=gate_mode, state="randn", epilogue=True,
                             Hk=Hk)
    seq = gpu_forward(inp, algo=1)
    check_all_heads(seq, inp, MIX + ("o",))
    chunk = gpu_forward(inp, algo=2)
    check_all_heads(chunk, inp, MIX + ("o",))
    fused = gpu_prefill(inp)
    check_all_heads(fused, inp, MIX)
    for k in MIX:
        assert torch.equal(fused[k], chunk[k]), k


def test_gqa_prefill_varlen_edges():
    """Packed sequences with empty ones, lengths below the conv window and around the chunk."""
    lengths = [5, 0, 1, 2, 3, 33, 64, 70]
    inp = inputs.make_inputs(231, H=4, N=len(lengths), lengths=(0, 1), raw_dtype="bf16",
                             conv=True, ring="randn", state="randn", epilogue=True, Hk=2)
    cu = np.concatenate([[0], np.cumsum(lengths)])
    rows = int(cu[-1])
    rng = np.random.default_rng(1231)
    for k, w in (("q_raw", 2), ("k_raw", 2), ("v_raw", 4)):
        setattr(inp, k, torch.from_numpy(rng.standard_normal((rows, w * 128)).astype(np.float32))
                .to(torch.bfloat16))
    inp.f_raw = torch.from_numpy(rng.standard_normal((rows, 4 * 128)).astype(np.float32))
    inp.beta_raw = torch.from_numpy(rng.standard_normal((rows, 4)).astype(np.float32))
    inp.gate_raw = torch.from_numpy(rng.standard_normal((rows, 4 * 128)).astype(np.float32))
    inp.cu_seqlens = cu
    fused = gpu_prefill(inp, varlen=True)
    check_all_heads(fused, inp, MIX)
    staged = gpu_forward(inp, varlen=True, algo=2)
    for k in MIX:
        assert torch.equal(fused[k], staged[k]), k


@pytest.mark.parametrize("H,Hk,T", [(4, 2, 1), (6, 3, 4), (4, 1, 16)])
def test_gqa_decode_verify(H, Hk, T):
    """The fused decode / verify kernel with grouped queries against the oracle, and a T-token
    call bit-equal to T chained one-token calls."""
    from gated_delta_rule_scan_gb300 import mixer
    N = 5
    inp = inputs.make_inputs(240 + T, H=H, N=N, T=T, raw_dtype="bf16", conv=True, ring="randn",
                             state="randn", epilogue=True, Hk=Hk)
    d = to_dev(inp)
    full = mixer.kda_decode(N=N, T=T, H=H, Hk=Hk, **d)
    torch.cuda.synchronize()
    check_all_heads(full, inp, MIX)
    state, ring = d["state_in"], d["ring_in"]
    ys = []
    for t in range(T):
        rows = torch.arange(N, device="cuda") * T + t
        step = {k: d[k] for k in ("conv_w", "dt_bias", "a_log", "norm_w")}
        for k in ("q_raw", "k_raw", "v_raw", "f_raw", "beta_raw", "gate_raw"):
            step[k] = d[k][rows].contiguous()
        r = mixer.kda_decode(N=N, T=1, H=H, Hk=Hk, state_in=state, ring_in=ring, **step)
        state, ring = r["state_out"], r["ring_out"]
        ys.append(r["y"].view(N, 1, -1))
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(ys, dim=1).view(N * T, -1), full["y"])
    assert torch.equal(state, full["state_out"])
    assert torch.equal(ring, full["ring_out"])


def test_gqa_rollback_and_in_place_refusal():
    """Rollback with grouped queries equals keep[n] chained one-token decodes; rolling the ring in
    place is refused when several value heads share a q/k head (40003)."""
    from gated_delta_rule_scan_gb300 import kda, mixer
    N, H, Hk, T = 4, 4, 2, 4
    inp = inputs.make_inputs(250, H=H, N=N, T=T, raw_dtype="bf16", conv=True, ring="randn",
                             state="randn", epilogue=True, Hk=Hk)
    d = to_dev(inp)
    keep_h = np.array([0, 1, 3, 4], dtype=np.int32)
    keep = torch.from_numpy(keep_h).cuda()
    rb = mixer.kda_verify_rollback(N=N, T=T, H=H, Hk=Hk, keep=keep, **d)
    torch.cuda.synchronize()
    for n in range(N):
        state = d["state_in"][n:n + 1]
        ring = d["ring_in"][n:n + 1]
        for t in range(int(keep_h[n])):
            row = slice(n * T + t, n * T + t + 1)
            step = {k: d[k] for k in ("conv_w", "dt_bias", "a_log", "norm_w")}
            for k in ("q_raw", "k_raw", "v_raw", "f_raw", "beta_raw", "gate_raw"):
                step[k] = d[k][row].contiguous()
            r = mixer.kda_decode(N=1, T=1, H=H, Hk=Hk, state_in=state, ring_in=ring, **step)
            assert torch.equal(r["y"], rb["y"][row])
            state, ring = r["state_out"], r["ring_out"]
        torch.cuda.synchronize()
        assert torch.equal(state, rb["state_out"][n:n + 1])
        assert torch.equal(ring, rb["ring_out"][n:n + 1])
    ring = d["ring_in"].clone()
    with pytest.raises(kda.KdaError) as e:
        mixer.kda_decode(N=N, T=T, H=H, Hk=Hk, ring_out=ring, **dict(d, ring_in=ring))
    assert e.value.status == 40003
