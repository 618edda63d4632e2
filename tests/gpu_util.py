"""Helpers shared by the GPU tests: move a seeded workload to the device, run it through the
library, run the oracle on the same inputs (optionally on a subset of heads, which is exact
because heads are independent), and measure relative L-infinity error."""

from __future__ import annotations

import numpy as np
import torch

from gated_delta_rule_scan_gb300.inputs import KdaInputs

TOL = 1e-3  # relative L-inf bound for f32 state (max|gpu - ref| / max|ref| per output tensor)


def rel_linf(gpu, ref) -> float:
    g = gpu.detach().double().cpu().numpy() if isinstance(gpu, torch.Tensor) else np.asarray(gpu)
    r = ref.detach().double().cpu().numpy() if isinstance(ref, torch.Tensor) else np.asarray(ref)
    assert g.shape == r.shape, (g.shape, r.shape)
    den = np.abs(r).max()
    num = np.abs(g - r).max()
    return float(num / den) if den > 0 else float(num)


def to_dev(inp: KdaInputs, dev="cuda"):
    d = {}
    for name in ("q_raw", "k_raw", "v_raw", "conv_w", "ring_in", "f_raw", "dt_bias", "a_log",
                 "beta_raw", "state_in", "norm_w", "gate_raw"):
        t = getattr(inp, name)
        d[name] = None if t is None else t.to(dev).contiguous()
    return d


def gpu_forward(inp: KdaInputs, *, varlen=None, algo=0, **kw):
    from gated_delta_rule_scan_gb300 import mixer
    d = to_dev(inp)
    T = inp.uniform_T
    if varlen is None:
        varlen = T is None
    if varlen:
        cu_h = torch.from_numpy(inp.cu_seqlens.astype(np.int32))
        extra = dict(cu_seqlens=cu_h.to("cuda"), cu_seqlens_host=cu_h)
    else:
        extra = dict(N=inp.N, T=T)
    out = mixer.kda_forward(H=inp.H, K=inp.K, gate_mode=inp.gate_mode, algo=algo, **d, **extra,
                            **kw)
    torch.cuda.synchronize()
    return out


def gpu_prefill(inp: KdaInputs, *, varlen=None, **kw):
    """The fused prefill entry point (kda_prefill_fused[_varlen]) on the workload."""
    from gated_delta_rule_scan_gb300 import mixer
    d = to_dev(inp)
    T = inp.uniform_T
    if varlen is None:
        varlen = T is None
    if varlen:
        cu_h = torch.from_numpy(inp.cu_seqlens.astype(np.int32))
        extra = dict(cu_seqlens=cu_h.to("cuda"), cu_seqlens_host=cu_h)
    else:
        extra = dict(N=inp.N, T=T)
    out = mixer.kda_prefill(H=inp.H, K=inp.K, gate_mode=inp.gate_mode, **d, **extra, **kw)
    torch.cuda.synchronize()
    return out


def head_channels(heads, D=128):
    return np.concatenate([np.arange(h * D, (h + 1) * D) for h in heads])


def oracle_forward(inp: KdaInputs, heads=None, **kw):
    """The f64 oracle on the workload (all heads, or the listed ones)."""
    from oracle import oracle as orc
    H, D = inp.H, inp.D
    heads = list(range(H)) if heads is None else list(heads)
    ch = head_channels(heads, D)
    C = H * D

    def cols(t, idx):
        return None if t is None else t[:, idx]

    ring_in = conv_w = None
    if inp.conv_w is not None:
        prow = np.concatenate([p * C + ch for p in range(3)])
        conv_w = inp.conv_w[prow]
        ring_in = inp.ring_in[:, prow]
    gm = inp.gate_mode
    return orc.forward(
        q_raw=cols(inp.q_raw, ch), k_raw=cols(inp.k_raw, ch), v_raw=cols(inp.v_raw, ch),
        f_raw=cols(inp.f_raw, ch) if gm == 0 else cols(inp.f_raw, heads),
        dt_bias=inp.dt_bias[ch] if gm == 0 else inp.dt_bias[heads],
        a_log=inp.a_log[heads], beta_raw=cols(inp.beta_raw, heads),
        state_in=inp.state_in[:, heads], H=len(heads), D=D, conv_w=conv_w, ring_in=ring_in,
        cu_seqlens=inp.cu_seqlens, gate_mode=gm, norm_w=inp.norm_w,
        gate_raw=cols(inp.gate_raw, ch), **kw)


def gpu_heads(out, inp: KdaInputs, heads):
    """The GPU outputs restricted to the listed heads (same layout as oracle_forward's)."""
    ch = torch.from_numpy(head_channels(heads, inp.D))
    C = inp.H * inp.D
    res = dict(state_out=out["state_out"].cpu()[:, heads])
    if out.get("o") is not None:
        res["o"] = out["o"].cpu()[:, ch]
    if out.get("y") is not None:
        res["y"] = out["y"].cpu()[:, ch]
    if out.get("ring_out") is not None:
        prow = torch.cat([p * C + ch for p in range(3)])
        res["ring_out"] = out["ring_out"].cpu()[:, prow]
    return res
