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
    if inp.Hk is not None:
        kw = dict(kw, Hk=inp.Hk)
    if inp.Dv is not None:
        kw = dict(kw, Dv=inp.Dv)
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
    if inp.Hk is not None:
        kw = dict(kw, Hk=inp.Hk)
    if inp.Dv is not None:
        kw = dict(kw, Dv=inp.Dv)
    out = mixer.kda_prefill(H=inp.H, K=inp.K, gate_mode=inp.gate_mode, **d, **extra, **kw)
    torch.cuda.synchronize()
    return out


def head_channels(heads, D=128):
    return np.concatenate([np.arange(h * D, (h + 1) * D) for h in heads])


def oracle_forward(inp: KdaInputs, heads=None, **kw):
    """The f64 oracle on the workload (all heads, or the listed ones; grouped-query and
    value-width workloads run on all heads)."""
    from oracle import oracle as orc
    H, D = inp.H, inp.D
    if inp.Hk is not None or inp.Dv is not None:
        assert heads is None or list(heads) == list(range(H)), "grouped queries: all heads"
        return orc.forward(
            q_raw=inp.q_raw, k_raw=inp.k_raw, v_raw=inp.v_raw, f_raw=inp.f_raw,
            dt_bias=inp.dt_bias, a_log=inp.a_log, beta_raw=inp.beta_raw, state_in=inp.state_in,
            H=H, D=D, conv_w=inp.conv_w, ring_in=inp.ring_in, cu_seqlens=inp.cu_seqlens,
            gate_mode=inp.gate_mode, norm_w=inp.norm_w, gate_raw=inp.gate_raw, Hk=inp.Hk,
            Dv=inp.Dv, **kw)
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


def check_all_heads(out, inp: KdaInputs, keys, tol=TOL, ring_exact=True, budget=2 << 30, **kw):
    """Every head of the GPU outputs against the oracle.  The oracle runs a few heads at a time
    (heads are independent, so each group is exact) so that its f64 planes stay within about
    `budget` bytes of host memory; the relative L-inf error is taken over the whole tensor
    (max |gpu - ref| over all heads / max |ref| over all heads).  The conv ring must be
    bit-equal.  Returns the errors per key."""
    H, D = inp.H, inp.D
    rows = max(inp.rows, 1)
    host = {}
    for k in keys:
        host[k] = out[k].detach().cpu() if isinstance(out[k], torch.Tensor) else out[k]
    if inp.Hk is not None or inp.Dv is not None:   # one oracle run over every head
        ref = oracle_forward(inp, **kw)
        errs = {}
        for k in keys:
            g = host[k].double().numpy()
            assert g.shape == ref[k].shape, (k, g.shape, ref[k].shape)
            if k == "ring_out" and ring_exact:
                assert np.array_equal(g, ref[k]), "ring_out not bit-equal"
                errs[k] = 0.0
            else:
                errs[k] = rel_linf(g, ref[k])
        assert max(errs.values()) <= tol, errs
        return errs
    per_head = rows * D * 8 * 16            # about sixteen f64 [rows, D] planes per head
    group = max(1, min(H, budget // per_head))
    num = {k: 0.0 for k in keys}
    den = {k: 0.0 for k in keys}
    C = H * D
    for h0 in range(0, H, group):
        heads = list(range(h0, min(H, h0 + group)))
        ref = oracle_forward(inp, heads=heads, **kw)
        ch = torch.from_numpy(head_channels(heads, D))
        for k in keys:
            if k == "state_out":
                g = host[k][:, heads]
            elif k == "ring_out":
                prow = torch.cat([p * C + ch for p in range(3)])
                g = host[k][:, prow]
            else:
                g = host[k][:, ch]
            g = g.double().numpy()
            r = ref[k]
            assert g.shape == r.shape, (k, g.shape, r.shape)
            if k == "ring_out" and ring_exact:
                assert np.array_equal(g, r), f"ring_out not bit-equal (heads {heads})"
                continue
            num[k] = max(num[k], float(np.abs(g - r).max()) if g.size else 0.0)
            den[k] = max(den[k], float(np.abs(r).max()) if r.size else 0.0)
        del ref
    errs = {k: (num[k] / den[k] if den[k] > 0 else num[k]) for k in keys}
    assert max(errs.values()) <= tol, errs
    return errs
