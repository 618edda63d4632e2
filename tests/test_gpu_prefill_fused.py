"""GPU parity of the fused prefill (kda_prefill_fused[_varlen]): conv + SiLU, l2 norm, gates,
chunked scan and gated RMSNorm in one call, with the readout fed straight into the norm.

Against the f64 oracle: relative L-inf <= 1e-3 on y and the state, the ring bit-equal.  Against
the stage-by-stage path with the chunked scan (the same kernels in the same order): y, state and
ring bit-equal.
"""

import numpy as np
import pytest
import torch

from gated_delta_rule_scan_gb300 import inputs
from tests.gpu_util import TOL, check_all_heads, gpu_forward, gpu_prefill, rel_linf

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    from gated_delta_rule_scan_gb300 import kda
    assert kda.kda_device_status() == 0


def _check(fused, inp, varlen=None):
    keys = ("y", "state_out") + (("ring_out",) if fused.get("ring_out") is not None else ())
    check_all_heads(fused, inp, keys)
    unf = gpu_forward(inp, varlen=varlen, algo=2)
    assert torch.equal(fused["state_out"], unf["state_out"])
    if fused.get("ring_out") is not None:
        assert torch.equal(fused["ring_out"], unf["ring_out"])
    assert torch.equal(fused["y"], unf["y"])


@pytest.mark.parametrize("T", [1, 17, 32, 203])
def test_prefill_fused_ragged(T):
    """One chunk or less, exactly one chunk, and many chunks with a ragged tail; two sequences,
    random state and ring (the uniform layout's ragged chunk is followed by the next sequence)."""
    inp = inputs.make_inputs(60 + T, H=3, N=2, T=T, raw_dtype="bf16", conv=True, ring="randn",
                             state="randn", epilogue=True)
    _check(gpu_prefill(inp), inp)


def test_prefill_fused_varlen_edges():
    """Packed sequences with empty ones, lengths below the conv window and around the chunk."""
    lengths = [5, 0, 1, 2, 3, 17, 0, 33, 64, 70]
    inp = inputs.make_inputs(71, H=4, N=len(lengths), lengths=(0, 1), raw_dtype="bf16",
                             conv=True, ring="randn", state="randn", epilogue=True)
    cu = np.concatenate([[0], np.cumsum(lengths)])
    rows = int(cu[-1])
    rng = np.random.default_rng(1071)
    C = inp.H * 128
    for k in ("q_raw", "k_raw", "v_raw"):
        setattr(inp, k, torch.from_numpy(rng.standard_normal((rows, C)).astype(np.float32))
                .to(torch.bfloat16))
    inp.f_raw = torch.from_numpy(rng.standard_normal((rows, C)).astype(np.float32))
    inp.beta_raw = torch.from_numpy(rng.standard_normal((rows, inp.H)).astype(np.float32))
    inp.gate_raw = torch.from_numpy(rng.standard_normal((rows, C)).astype(np.float32))
    inp.cu_seqlens = cu
    _check(gpu_prefill(inp, varlen=True), inp, varlen=True)


@pytest.mark.parametrize("varlen", [False, True])
def test_prefill_nonfinite_rows_after_a_ragged_chunk(varlen):
    """A sequence's ragged last chunk is staged together with the rows that follow it (the next
    sequence's); when those rows hold inf and NaN (the next sequence's own data), the first
    sequence must not see them: its readout, state and ring equal the oracle's on it alone (and
    stay finite) through the fused prefill, the staged chunked path and the sequential scan."""
    import dataclasses
    T, H = 45, 2
    inp = inputs.make_inputs(74, H=H, N=2, T=T, raw_dtype="bf16", conv=True, ring="randn",
                             state="randn", epilogue=True)
    bad = slice(T, T + 19)                       # the rows that share the ragged chunk's tile
    for name, val in (("q_raw", float("inf")), ("k_raw", float("nan")), ("v_raw", -float("inf")),
                      ("f_raw", float("nan")), ("beta_raw", float("nan")),
                      ("gate_raw", float("inf"))):
        t = getattr(inp, name).clone()
        t[bad] = val
        setattr(inp, name, t)
    first = dataclasses.replace(
        inp, N=1, cu_seqlens=inp.cu_seqlens[:2].copy(),
        **{k: getattr(inp, k)[:T] for k in ("q_raw", "k_raw", "v_raw", "f_raw", "beta_raw",
                                            "gate_raw")},
        ring_in=inp.ring_in[:1], state_in=inp.state_in[:1])
    if varlen:
        inp = dataclasses.replace(inp, cu_seqlens=np.array([0, T, 2 * T], dtype=np.int64))
    runs = [gpu_prefill(inp, varlen=varlen)] + [gpu_forward(inp, varlen=varlen, algo=a)
                                                for a in (1, 2)]
    for out in runs:
        mine = {"y": out["y"][:T], "state_out": out["state_out"][:1], "ring_out": out["ring_out"][:1]}
        for k, v in mine.items():
            assert torch.isfinite(v).all(), k
        check_all_heads(mine, first, ("y", "state_out", "ring_out"))


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("norm_gate,gate_mode", [("sigmoid", 0), ("silu", 1)])
def test_prefill_folded_norm(norm_gate, gate_mode):
    """With (sequence, head) chains on every SM the inter kernel writes y through the
    gated RMSNorm itself (no RMSNorm launch): packed sequences with ragged last chunks, one
    shorter than a chunk and one empty; y, state and ring equal the staged path's (chunked scan,
    then the RMSNorm kernel) bit for bit, and the oracle's on every head."""
    from gated_delta_rule_scan_gb300 import kda
    H = 64
    lengths = [40, 90, 0, 17, 75]
    N = -(-_sms() // H) + 1                      # N * H >= the SM count
    lengths = (lengths * N)[:N]
    inp = inputs.make_inputs(76 + gate_mode, H=H, N=N, lengths=(0, 1), raw_dtype="bf16",
                             conv=True, ring="randn", gate_mode=gate_mode, state="randn",
                             epilogue=True)
    cu = np.concatenate([[0], np.cumsum(lengths)])
    rows, C = int(cu[-1]), H * 128
    rng = np.random.default_rng(1076)
    for k in ("q_raw", "k_raw", "v_raw"):
        setattr(inp, k, torch.from_numpy(rng.standard_normal((rows, C)).astype(np.float32))
                .to(torch.bfloat16))
    inp.f_raw = torch.from_numpy(rng.standard_normal((rows, C if gate_mode == 0 else H))
                                 .astype(np.float32))
    inp.beta_raw = torch.from_numpy(rng.standard_normal((rows, H)).astype(np.float32))
    inp.gate_raw = torch.from_numpy(rng.standard_normal((rows, C)).astype(np.float32))
    inp.cu_seqlens = cu
    kda.kernel_timing(True)
    try:
        fused = gpu_prefill(inp, varlen=True, norm_gate=norm_gate)
        times = kda.kernel_times()
    finally:
        kda.kernel_timing(False)
    assert "kda_gated_rmsnorm_kernel" not in times and "kda_chunk_inter_kernel" in times, times
    unf = gpu_forward(inp, varlen=True, algo=2, norm_gate=norm_gate)
    for k in ("y", "state_out", "ring_out"):
        assert torch.equal(fused[k], unf[k]), k
    check_all_heads(fused, inp, ("y", "state_out", "ring_out"), norm_gate=norm_gate)


@pytest.mark.parametrize("raw,gate_mode", [("f32", 1), ("f32", 0), ("bf16", 1)])
def test_prefill_fused_repeatable(raw, gate_mode):
    """Repeated fused prefills of a sequence whose last chunk holds 12 tokens (whole warps of the
    chunk past the end) give the same bits every time, and the staged path's: the values computed
    for tokens past the end are fixed zeros or finite, never left over from an earlier task."""
    inp = inputs.make_inputs(75, H=4, N=1, T=300, raw_dtype=raw, conv=True, ring="randn",
                             gate_mode=gate_mode, state="randn", epilogue=True)
    unf = gpu_forward(inp, algo=2)
    for _ in range(6):
        fused = gpu_prefill(inp)
        for k in ("y", "state_out", "ring_out"):
            assert torch.equal(fused[k], unf[k]), k


def test_prefill_fused_gdn():
    """The per-head (Gated DeltaNet) gate through the fused path."""
    inp = inputs.make_inputs(72, H=4, N=1, T=300, raw_dtype="f32", conv=True, ring="randn",
                             gate_mode=1, state="randn", epilogue=True)
    _check(gpu_prefill(inp), inp)


@pytest.mark.parametrize("raw,gate_mode,conv,K", [("bf16", 1, True, 4), ("bf16", 0, True, 6),
                                                  ("bf16", 1, False, 4), ("f32", 0, True, 4),
                                                  ("bf16", 0, True, 2)])
def test_prefill_fused_variants(raw, gate_mode, conv, K):
    """Each kernel variant: bf16 raw rows staged in shared memory (with the conv weights for up
    to 4 taps, loaded directly for more) or f32 rows loaded directly; per-channel or per-head
    gate; with or without the conv.  Many chunks per sequence, so every persistent CTA runs
    several tasks and stages the next one's inputs."""
    inp = inputs.make_inputs(90 + K, H=5, N=3, T=333, K=K, raw_dtype=raw, conv=conv,
                             ring="randn", gate_mode=gate_mode, state="randn", epilogue=True)
    _check(gpu_prefill(inp), inp)


@pytest.mark.slow
def test_prefill_fused_full_size():
    """T=4096, H=64 (the prefill benchmark workload), every head against the oracle."""
    inp = inputs.prefill()
    _check(gpu_prefill(inp), inp)


def _split_rows(inp, first):
    """The workload cut at each sequence's split point: the first parts (first=True) or the rest,
    as packed inputs of their own, and the rows of the original they came from."""
    import copy
    cu, P = inp.cu_seqlens, inp.split_points
    parts = [np.arange(cu[n], cu[n] + P[n]) if first else np.arange(cu[n] + P[n], cu[n + 1])
             for n in range(inp.N)]
    sel = torch.from_numpy(np.concatenate(parts))
    sub = copy.copy(inp)
    for k in ("q_raw", "k_raw", "v_raw", "f_raw", "beta_raw", "gate_raw"):
        setattr(sub, k, getattr(inp, k)[sel])
    sub.cu_seqlens = np.concatenate([[0], np.cumsum([len(p) for p in parts])])
    return sub, sel


@pytest.mark.slow
def test_prefill_varlen_full_size_split_resume():
    """The packed varlen workload at its stated size (16 sequences, lengths U[256, 8192], H=64,
    random states and rings): the fused prefill against the oracle on every head and bit-equal to
    the staged chunked path; then each sequence cut at its seeded split point, the prefix run,
    and the suffix resumed from the saved (state, ring) -- through the fused prefill and through
    the staged chunked path -- matches the unsplit run within the tolerance, the ring bit for
    bit."""
    inp = inputs.varlen_prefill()
    full = gpu_prefill(inp, varlen=True)
    _check(full, inp, varlen=True)
    a, sel_a = _split_rows(inp, True)
    b, sel_b = _split_rows(inp, False)
    for run in (lambda x: gpu_prefill(x, varlen=True), lambda x: gpu_forward(x, varlen=True, algo=2)):
        out_a = run(a)
        b.state_in = out_a["state_out"].cpu()
        b.ring_in = out_a["ring_out"].cpu()
        out_b = run(b)
        y = torch.empty_like(full["y"])
        y[sel_a.cuda()] = out_a["y"]
        y[sel_b.cuda()] = out_b["y"]
        assert rel_linf(y, full["y"]) <= TOL
        assert rel_linf(out_b["state_out"], full["state_out"]) <= TOL
        assert torch.equal(out_b["ring_out"], full["ring_out"])
        del out_a, out_b, y


def test_prefill_fused_contract():
    """Contract errors through the C ABI: the decay-factor flag, a short workspace, no output."""
    from gated_delta_rule_scan_gb300 import kda
    inp = inputs.make_inputs(73, H=2, N=1, T=40, raw_dtype="bf16", conv=True, ring="randn",
                             state="randn", epilogue=True)
    from tests.gpu_util import to_dev
    d = to_dev(inp)
    y = torch.empty(40, 256, device="cuda")
    s_out = torch.empty_like(d["state_in"])
    r_out = torch.empty_like(d["ring_in"])
    ws = kda.prefill_workspace(1, 40, 2, "cuda")
    args = [d["q_raw"], d["k_raw"], d["v_raw"], d["conv_w"], d["ring_in"], r_out, d["f_raw"],
            d["dt_bias"], d["a_log"], d["beta_raw"], d["state_in"], s_out, d["norm_w"],
            d["gate_raw"], y, ws]
    with pytest.raises(kda.KdaError) as e:
        kda.kda_prefill_fused(*args, N=1, T=40, H=2, gate_mode=kda.GATE_EXP)
    assert e.value.status == 40007
    short = args.copy()
    short[-1] = ws[: ws.numel() // 4]   # the query is an upper bound: cut well below the need
    with pytest.raises(kda.KdaError) as e:
        kda.kda_prefill_fused(*short, N=1, T=40, H=2)
    assert e.value.status == 40009
    none_y = args.copy()
    none_y[-2] = None
    with pytest.raises(kda.KdaError) as e:
        kda.kda_prefill_fused(*none_y, N=1, T=40, H=2)
    assert e.value.status == 40004


def test_kernel_timer_counts_fused_launches():
    """With timing on, one fused prefill of two packed sequences records exactly its kernels:
    chunk offsets, the fused prep + intra-chunk kernel, inter (which also rolls the conv ring)
    and the RMSNorm, once each (no separate prep or ring-roll kernel): with (sequence, head)
    chains on fewer than two thirds of the SMs the RMSNorm runs as a kernel of its own."""
    from gated_delta_rule_scan_gb300 import kda
    inp = inputs.make_inputs(74, H=2, N=2, lengths=(40, 90), raw_dtype="bf16", conv=True,
                             ring="randn", state="randn", epilogue=True)
    kda.kernel_timing(True)
    try:
        gpu_prefill(inp, varlen=True)
        times = kda.kernel_times()
    finally:
        kda.kernel_timing(False)
    assert set(times) == {"kda_chunk_offsets_kernel", "kda_chunk_prep_intra_kernel",
                          "kda_chunk_inter_kernel", "kda_gated_rmsnorm_kernel"}, times
    assert all(n == 1 and ms > 0 for n, ms in times.values()), times
