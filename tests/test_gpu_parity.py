"""GPU parity: the CUDA path through the C ABI against the f64 oracle on the same seeded inputs.

Bar: relative L-inf (max|gpu - ref| / max|ref|, per output tensor) <= 1e-3 for every f32
output; the conv ring is exact copies of raw samples, so it must be bit-equal; decode vs verify
and chained one-token scans vs one T-token scan must be bit-equal.
"""

import numpy as np
import pytest
import torch

from gated_delta_rule_scan_gb300 import inputs
from tests.gpu_util import TOL, check_all_heads, gpu_forward, oracle_forward, rel_linf, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    from gated_delta_rule_scan_gb300 import kda
    assert kda.kda_device_status() == 0


def _assert_close(out, ref, keys, tol=TOL, ring_exact=True):
    errs = {}
    for k in keys:
        if k == "ring_out" and ring_exact:
            g = out[k].cpu().double().numpy()
            assert np.array_equal(g, ref[k]), "ring_out not bit-equal to the raw samples"
            errs[k] = 0.0
        else:
            errs[k] = rel_linf(out[k], ref[k])
    assert max(errs.values()) <= tol, errs
    return errs


# ------------------------------------------------------------------------------------------
# tiny KDA scan: 1 x 64 tokens, 4 heads, f32, no conv
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("algo", [1, 2], ids=["seq", "chunk"])
def test_tiny_scan_full_path(algo):
    inp = inputs.tiny_scan()
    out = gpu_forward(inp, algo=algo)
    ref = oracle_forward(inp)
    _assert_close(out, ref, ("o", "state_out"))


def test_tiny_scan_identical_inputs():
    """Scan only: both sides read the same f32 q, k, v, g, beta (made by the oracle's own prologue
    and rounded to f32), so the difference is the scan alone."""
    from gated_delta_rule_scan_gb300 import kda
    from oracle import oracle as orc
    inp = inputs.tiny_scan()
    ref = oracle_forward(inp)
    T, H, D = 64, 4, 128
    f32 = {k: torch.from_numpy(ref[k]).float() for k in ("q_hat", "k_hat", "v_hat", "g", "beta")}
    o_ref, s_ref = orc.scan_kda(*(f32[k].double().numpy().reshape(T, H, -1)
                                  for k in ("q_hat", "k_hat", "v_hat", "g")),
                                f32["beta"].double().numpy(), np.zeros((1, H, D, D)))
    dev = {k: v.cuda() for k, v in f32.items()}
    s_in = torch.zeros(1, H, D, D, device="cuda")
    s_out = torch.empty_like(s_in)
    o = torch.empty(T, H * D, device="cuda")
    kda.kda_scan(dev["q_hat"], dev["k_hat"], dev["v_hat"], dev["g"], dev["beta"], s_in, s_out, o,
                 N=1, T=T, H=H, algo=kda.ALGO_SEQ)
    torch.cuda.synchronize()
    assert rel_linf(o, o_ref.reshape(T, H * D)) <= 1e-4
    assert rel_linf(s_out, s_ref) <= 1e-4


# ------------------------------------------------------------------------------------------
# decode and verify: 64 sequences x H=64, fused kernel
# ------------------------------------------------------------------------------------------

DEC_KEYS = ("q_raw", "k_raw", "v_raw", "conv_w", "ring_in", "f_raw", "dt_bias", "a_log",
            "beta_raw", "state_in", "norm_w", "gate_raw")


def _decode(inp, T, **kw):
    from gated_delta_rule_scan_gb300 import mixer
    d = to_dev(inp)
    out = mixer.kda_decode(N=inp.N, T=T, H=inp.H, **d, **kw)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("N,H", [(3, 2), (64, 64)])
def test_decode_fused_vs_oracle(N, H):
    inp = inputs.decode_step(N=N, T=1, H=H)
    out = _decode(inp, 1)
    check_all_heads(out, inp, ("y", "state_out", "ring_out"))


@pytest.mark.parametrize("T", [2, 4, 16])
def test_verify_equals_chained_decode_bitwise(T):
    """A T-token fused call equals T chained one-token fused calls, bit for bit."""
    N, H = 8, 64
    inp = inputs.decode_step(N=N, T=T, H=H, seed=11)
    full = _decode(inp, T)
    d = to_dev(inp)
    C = H * 128
    state, ring = d["state_in"], d["ring_in"]
    ys = []
    from gated_delta_rule_scan_gb300 import mixer
    for t in range(T):
        rows = torch.arange(N, device="cuda") * T + t
        step = {k: d[k] for k in ("conv_w", "dt_bias", "a_log", "norm_w")}
        for k in ("q_raw", "k_raw", "v_raw", "f_raw", "beta_raw", "gate_raw"):
            step[k] = d[k][rows].contiguous()
        r = mixer.kda_decode(N=N, T=1, H=H, state_in=state, ring_in=ring, **step)
        state, ring = r["state_out"], r["ring_out"]
        ys.append(r["y"].view(N, 1, C))
    torch.cuda.synchronize()
    y_chain = torch.cat(ys, dim=1).view(N * T, C)
    assert torch.equal(y_chain, full["y"])
    assert torch.equal(state, full["state_out"])
    assert torch.equal(ring, full["ring_out"])
    # and the verify call itself matches the oracle on every head
    check_all_heads(full, inp, ("y", "state_out", "ring_out"))


def test_decode_fused_equals_unfused():
    """The fused kernel and prep -> scan -> gated RMSNorm agree: the ring bit for bit (pure copies),
    y and the state to f32 rounding (the two scans reduce over different lane groupings)."""
    inp = inputs.decode_step(N=16, T=4, H=8, seed=12)
    fused = _decode(inp, 4)
    for gate_exp in (False, True):
        unf = gpu_forward(inp, varlen=False, algo=1, gate_exp=gate_exp)
        assert torch.equal(fused["ring_out"], unf["ring_out"])
        for k in ("y", "state_out"):
            assert rel_linf(fused[k], unf[k]) <= 1e-5, (k, gate_exp)


def test_decode_in_place_ring():
    inp = inputs.decode_step(N=4, T=3, H=4, seed=13)
    d = to_dev(inp)
    from gated_delta_rule_scan_gb300 import mixer
    sep = mixer.kda_decode(N=4, T=3, H=4, **d)
    ring = d["ring_in"].clone()
    d2 = dict(d, ring_in=ring)
    inpl = mixer.kda_decode(N=4, T=3, H=4, ring_out=ring, **d2)
    torch.cuda.synchronize()
    assert torch.equal(inpl["y"], sep["y"])
    assert torch.equal(ring, sep["ring_out"])


# ------------------------------------------------------------------------------------------
# prefill
# ------------------------------------------------------------------------------------------

def test_prefill_small_ragged():
    """T = 4096-shaped workload shrunk to T=203 (ragged against the 16-token blocks), H=6."""
    inp = inputs.prefill(T=203, H=6)
    out = gpu_forward(inp, algo=1, gate_exp=False)
    ref = oracle_forward(inp)
    _assert_close(out, ref, ("y", "o", "state_out", "ring_out"))
    _assert_close(out, ref, ("q_hat", "k_hat", "v_hat", "g", "beta"))
    # the decay-factor hand-off computes the same bits, and its g is exp of the log-decay
    out2 = gpu_forward(inp, algo=1, gate_exp=True)
    for k in ("y", "o", "state_out", "ring_out", "q_hat", "k_hat", "v_hat", "beta"):
        assert torch.equal(out[k], out2[k]), k
    assert rel_linf(out2["g"], np.exp(ref["g"])) <= TOL


@pytest.mark.parametrize("T", [1, 15, 16, 17, 203])
def test_prefill_chunked_ragged(T):
    """The chunked tensor-core form against the oracle: T below, at and above one 16-token chunk,
    and many chunks with a ragged tail; random initial state and ring."""
    inp = inputs.make_inputs(30 + T, H=3, N=2, T=T, raw_dtype="bf16", conv=True, ring="randn",
                             state="randn", epilogue=True)
    out = gpu_forward(inp, algo=2)
    ref = oracle_forward(inp)
    _assert_close(out, ref, ("y", "o", "state_out", "ring_out"))
    out_e = gpu_forward(inp, algo=2, gate_exp=True)
    _assert_close(out_e, ref, ("y", "o", "state_out"))


@pytest.mark.slow
@pytest.mark.parametrize("algo", [1, 2], ids=["seq", "chunk"])
def test_prefill_full_size(algo):
    """T=4096, H=64 (the prefill benchmark workload), every head against the oracle."""
    inp = inputs.prefill()
    out = gpu_forward(inp, algo=algo)
    check_all_heads(out, inp, ("y", "o", "state_out", "ring_out"))


def test_scan_chain_bitwise():
    """kda_scan over T tokens equals T chained one-token kda_scan calls, bit for bit."""
    from gated_delta_rule_scan_gb300 import kda
    inp = inputs.decode_step(N=2, T=37, H=3, seed=14)
    out = gpu_forward(inp, varlen=False, algo=1, gate_exp=False)
    N, T, H = 2, 37, 3
    C = H * 128
    q, k, v, g, b = (out[x].view(N, T, -1) for x in ("q_hat", "k_hat", "v_hat", "g", "beta"))
    state = inp.state_in.cuda()
    for t in range(T):
        nxt = torch.empty_like(state)
        o = torch.empty(N, C, device="cuda")
        kda.kda_scan(q[:, t].contiguous(), k[:, t].contiguous(), v[:, t].contiguous(),
                     g[:, t].contiguous(), b[:, t].contiguous(), state, nxt, o, N=N, T=1, H=H,
                     algo=kda.ALGO_SEQ)
        assert torch.equal(o, out["o"].view(N, T, C)[:, t]), t
        state = nxt
    torch.cuda.synchronize()
    assert torch.equal(state, out["state_out"])


# ------------------------------------------------------------------------------------------
# varlen
# ------------------------------------------------------------------------------------------

def _varlen_inputs(lengths, seed, H=4):
    inp = inputs.make_inputs(seed, H=H, N=len(lengths), lengths=(0, 1), raw_dtype="bf16",
                             conv=True, ring="randn", state="randn", epilogue=True)
    # re-draw with the exact lengths: the generator takes a range, so pin it via cu_seqlens
    L = np.array(lengths, dtype=np.int64)
    cu = np.concatenate([[0], np.cumsum(L)])
    rows = int(cu[-1])
    rng = np.random.default_rng(seed + 1000)
    C = H * 128

    def nrm(shape, std=1.0):
        return torch.from_numpy((rng.standard_normal(shape) * std).astype(np.float32))
    inp.cu_seqlens = cu
    inp.q_raw, inp.k_raw, inp.v_raw = (nrm((rows, C)).to(torch.bfloat16) for _ in range(3))
    inp.f_raw = nrm((rows, C))
    inp.beta_raw = nrm((rows, H))
    inp.gate_raw = nrm((rows, C))
    return inp


@pytest.mark.parametrize("algo", [1, 2], ids=["seq", "chunk"])
def test_varlen_edge_lengths(algo):
    """Empty sequences, lengths below the conv window (1, 2), a length equal to it (3), lengths
    straddling the 16-row tiles and blocks."""
    inp = _varlen_inputs([5, 0, 1, 2, 3, 17, 0, 33, 16], seed=21)
    out = gpu_forward(inp, varlen=True, algo=algo)
    ref = oracle_forward(inp)
    _assert_close(out, ref, ("y", "o", "state_out", "ring_out"))


@pytest.mark.parametrize("algo", [1, 2], ids=["seq", "chunk"])
def test_varlen_split_resume_state_carry(algo):
    """Run each sequence's prefix, then its suffix from the saved (state, ring): the result
    matches the unsplit run (GPU vs GPU) and the oracle."""
    inp = inputs.varlen_prefill(N=6, lo=20, hi=300, H=4, seed=22)
    full = gpu_forward(inp, varlen=True, algo=algo)
    cu = inp.cu_seqlens
    P = inp.split_points
    L = np.diff(cu)

    def sub(rows_of):
        sel = np.concatenate([np.arange(cu[n], cu[n + 1])[rows_of(n)] for n in range(inp.N)])
        cu2 = np.concatenate([[0], np.cumsum([len(np.arange(L[n])[rows_of(n)])
                                               for n in range(inp.N)])])
        return torch.from_numpy(sel), cu2

    import copy
    sel_a, cu_a = sub(lambda n: slice(0, P[n]))
    sel_b, cu_b = sub(lambda n: slice(P[n], None))
    a = copy.copy(inp)
    for k in ("q_raw", "k_raw", "v_raw", "f_raw", "beta_raw", "gate_raw"):
        setattr(a, k, getattr(inp, k)[sel_a])
    a.cu_seqlens = cu_a
    out_a = gpu_forward(a, varlen=True, algo=algo)
    b = copy.copy(inp)
    for k in ("q_raw", "k_raw", "v_raw", "f_raw", "beta_raw", "gate_raw"):
        setattr(b, k, getattr(inp, k)[sel_b])
    b.cu_seqlens = cu_b
    b.state_in = out_a["state_out"].cpu()
    b.ring_in = out_a["ring_out"].cpu()
    out_b = gpu_forward(b, varlen=True, algo=algo)
    y_split = torch.empty_like(full["y"])
    y_split[sel_a.cuda()] = out_a["y"]
    y_split[sel_b.cuda()] = out_b["y"]
    assert rel_linf(y_split, full["y"]) <= TOL
    assert rel_linf(out_b["state_out"], full["state_out"]) <= TOL
    assert torch.equal(out_b["ring_out"], full["ring_out"])
    ref = oracle_forward(inp)
    _assert_close(full, ref, ("y", "state_out", "ring_out"))


@pytest.mark.slow
@pytest.mark.parametrize("algo", [1, 2], ids=["seq", "chunk"])
def test_varlen_full_size(algo):
    """16 sequences with lengths U[256, 8192] at H=64, every head against the oracle."""
    inp = inputs.varlen_prefill()
    out = gpu_forward(inp, varlen=True, algo=algo)
    check_all_heads(out, inp, ("y", "o", "state_out", "ring_out"))


# ------------------------------------------------------------------------------------------
# Gated DeltaNet special case
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("algo", [1, 2], ids=["seq", "chunk"])
@pytest.mark.parametrize("T,H", [(300, 4), pytest.param(16384, 32, marks=pytest.mark.slow)])
def test_gdn_vs_both_oracles(T, H, algo):
    inp = inputs.gdn_long(T=T, H=H)
    out = gpu_forward(inp, algo=algo)
    check_all_heads(out, inp, ("o", "state_out"))
    check_all_heads(out, inp, ("o", "state_out"), scalar_scan=True)


# ------------------------------------------------------------------------------------------
# edge cases and contract through the C ABI on device pointers
# ------------------------------------------------------------------------------------------

def test_zero_tokens_copies_state():
    from gated_delta_rule_scan_gb300 import kda
    s_in = torch.randn(2, 3, 128, 128, device="cuda")
    s_out = torch.zeros_like(s_in)
    e = torch.empty(0, device="cuda")
    kda.kda_scan(e, e, e, e, e, s_in, s_out, e, N=2, T=0, H=3, algo=kda.ALGO_SEQ)
    torch.cuda.synchronize()
    assert torch.equal(s_in, s_out)


def test_contract_errors_on_device_pointers():
    from gated_delta_rule_scan_gb300 import kda
    lib = kda.library()
    s = torch.zeros(1, 1, 128, 128, device="cuda")
    x = torch.zeros(4, 128, device="cuda")
    b = torch.zeros(4, 1, device="cuda")
    p = lambda t: t.data_ptr()  # noqa: E731
    # aliased states
    assert lib.kda_scan(p(x), p(x), p(x), p(x), 0, p(b), p(s), p(s), p(x), 1, 4, 1, 128, 1.0, 1,
                        None, 0, None) == 40003
    # misaligned state
    s2 = torch.zeros(1 * 128 * 128 + 1, device="cuda")
    assert lib.kda_scan(p(x), p(x), p(x), p(x), 0, p(b), s2.data_ptr() + 4, p(s), p(x), 1, 4, 1,
                        128, 1.0, 1, None, 0, None) == 40010
    torch.cuda.synchronize()


@pytest.mark.parametrize("N,T,form", [(1, 95, "seq"), (1, 96, "chunk"), (4, 64, "seq"),
                                      (8, 63, "seq"), (8, 64, "chunk")])
def test_auto_form_follows_the_crossover(N, T, form):
    """KDA_ALGO_AUTO with a workspace large enough for either form takes the chunked one from 96
    tokens per sequence, or from 64 when sequences x heads >= 512 (H = 64), else the sequential
    one: the kernels that ran (the library's kernel timer) show which."""
    from gated_delta_rule_scan_gb300 import kda
    H, D, dev = 64, 128, "cuda"
    rows, C = N * T, H * D
    gen = torch.Generator(device=dev).manual_seed(7)
    unit = lambda: torch.nn.functional.normalize(  # noqa: E731
        torch.randn(rows, H, D, device=dev, generator=gen), dim=-1).reshape(rows, C)
    q, k = unit(), unit()
    v = torch.randn(rows, C, device=dev, generator=gen)
    g = -5.0 * torch.sigmoid(torch.randn(rows, C, device=dev, generator=gen))
    beta = torch.sigmoid(torch.randn(rows, H, device=dev, generator=gen))
    s0 = torch.zeros(N, H, D, D, device=dev)
    s1, o = torch.empty_like(s0), torch.empty(rows, C, device=dev)
    ws = kda.scan_workspace(N, rows, H, dev, algo=kda.ALGO_CHUNK)
    kda.kernel_timing(True)
    try:
        kda.kda_scan(q, k, v, g, beta, s0, s1, o, N=N, T=T, H=H, algo=kda.ALGO_AUTO, workspace=ws)
        torch.cuda.synchronize()
        ran = kda.kernel_times()
    finally:
        kda.kernel_timing(False)
    assert ("kda_chunk_inter_kernel" in ran) == (form == "chunk"), ran
    assert ("kda_scan_seq_kernel" in ran) == (form == "seq"), ran
