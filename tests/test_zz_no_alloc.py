"""kda_scan_varlen_static (the chunked scan on the library's fixed device scratch) against
kda_scan_varlen's chunked form with a caller workspace, through the C ABI.

The static form exists for callers that may not allocate device memory during a call -- a server
that has reserved its whole HBM budget up front, or C code without an allocator -- so the test
also checks that a call claims no device memory.

Two static calls in a row -- different sequence lengths, head counts and gate kinds, so the second
reuses scratch the first left full -- must each equal the workspace path bit for bit.  The file
name sorts last so the test also runs after every other GPU test; it passes alone as well."""

import pytest
import torch

from gated_delta_rule_scan_gb300 import kda

pytestmark = pytest.mark.gpu

D = 128


def _case(seed, lengths, H, gate_mode, dev):
    gen = torch.Generator().manual_seed(seed)
    total, N, C = sum(lengths), len(lengths), H * D

    def unit(rows):
        x = torch.randn(rows, H, D, generator=gen, dtype=torch.float64)
        return (x / x.norm(dim=-1, keepdim=True)).reshape(rows, C).float()

    q, k = unit(total), unit(total)
    v = torch.randn(total, C, generator=gen)
    if gate_mode == kda.GATE_PER_CHANNEL:
        g = -5.0 * torch.sigmoid(torch.randn(total, C, generator=gen))
    else:
        g = -2.0 * torch.rand(total, H, generator=gen)
    beta = torch.sigmoid(torch.randn(total, H, generator=gen))
    s0 = 0.1 * torch.randn(N, H, D, D, generator=gen)
    cu = torch.tensor([0] + torch.tensor(lengths).cumsum(0).tolist(), dtype=torch.int32)
    c = {name: t.to(dev) for name, t in
         dict(q=q, k=k, v=v, g=g, beta=beta, s0=s0, cu=cu).items()}
    c.update(cu_host=cu, H=H, gate_mode=gate_mode, N=N, total=total)
    for arm in ("static", "ws"):
        c["o_" + arm] = torch.full((total, C), float("nan"), device=dev)
        c["s_" + arm] = torch.full((N, H, D, D), float("nan"), device=dev)
    c["ws"] = kda.scan_workspace(N, total, H, dev, algo=kda.ALGO_CHUNK)
    return c


def _static(c, arm="static"):
    kda.kda_scan_varlen_static(c["q"], c["k"], c["v"], c["g"], c["beta"], c["s0"], c["s_" + arm],
                               c["o_" + arm], c["cu"], c["cu_host"], H=c["H"],
                               gate_mode=c["gate_mode"])


def test_static_scratch_equals_workspace_path():
    dev = torch.device("cuda:0")
    cases = [_case(21, [45, 300, 7, 64], 4, kda.GATE_PER_CHANNEL, dev),
             _case(22, [200, 1, 33, 0, 129], 6, kda.GATE_PER_HEAD, dev)]
    for c in cases:                                  # two calls in a row on the shared scratch
        _static(c)
    torch.cuda.synchronize()
    assert kda.kda_device_status() == 0
    for c in cases:
        kda.kda_scan_varlen(c["q"], c["k"], c["v"], c["g"], c["beta"], c["s0"], c["s_ws"],
                            c["o_ws"], c["cu"], c["cu_host"], H=c["H"], gate_mode=c["gate_mode"],
                            algo=kda.ALGO_CHUNK, workspace=c["ws"])
    torch.cuda.synchronize()
    assert kda.kda_device_status() == 0
    for c in cases:
        assert torch.isfinite(c["o_static"]).all() and c["o_static"].abs().max() > 0
        assert torch.equal(c["o_static"], c["o_ws"])
        assert torch.equal(c["s_static"], c["s_ws"])

    # a repeat of the first call, after the second overwrote the scratch: same result, and no
    # device memory claimed by the call
    c = cases[0]
    c["o_static"].fill_(float("nan"))
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info(dev)[0]
    _static(c)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info(dev)[0] == free_before
    assert torch.equal(c["o_static"], c["o_ws"])


def test_static_scratch_limit():
    dev = torch.device("cuda:0")
    over = kda.STATIC_SCRATCH_BYTES // kda.chunk_block_bytes() + 1   # one block past the limit
    c = _case(23, [32 * over], 1, kda.GATE_PER_CHANNEL, dev)
    with pytest.raises(kda.KdaError) as err:
        _static(c)
    assert err.value.status == 40011
    assert torch.isnan(c["o_static"]).all()          # nothing launched


def test_static_scratch_exactly_at_limit():
    """A problem that needs exactly the largest number of (32-token chunk, head) blocks the fixed
    array holds -- one head, one sequence whose last chunk is ragged -- is accepted and equals the
    workspace path bit for bit (an off-by-one in the size check, or a write past the array's end,
    would show here)."""
    dev = torch.device("cuda:0")
    cap_blocks = (kda.STATIC_SCRATCH_BYTES - 256) // kda.chunk_block_bytes()
    c = _case(24, [32 * cap_blocks - 5], 1, kda.GATE_PER_CHANNEL, dev)
    _static(c)
    kda.kda_scan_varlen(c["q"], c["k"], c["v"], c["g"], c["beta"], c["s0"], c["s_ws"], c["o_ws"],
                        c["cu"], c["cu_host"], H=1, gate_mode=kda.GATE_PER_CHANNEL,
                        algo=kda.ALGO_CHUNK, workspace=c["ws"])
    torch.cuda.synchronize()
    assert kda.kda_device_status() == 0
    assert torch.isfinite(c["o_static"]).all()
    assert torch.equal(c["o_static"], c["o_ws"])
    assert torch.equal(c["s_static"], c["s_ws"])
