"""Whole-mixer convenience calls over the C ABI: allocate the intermediate and output buffers
with torch on the inputs' device and run the entry points in the mixer's stage order
(prep -> scan -> gated RMSNorm, or the single fused decode/verify launch).  Plumbing only: every
value is computed by the library's kernels.
"""

from __future__ import annotations

import torch

from . import kda


def _empty(shape, like):
    return torch.empty(shape, dtype=torch.float32, device=like.device)


def kda_forward(*, q_raw, k_raw, v_raw, f_raw, dt_bias, a_log, beta_raw, state_in, H,
                conv_w=None, ring_in=None, norm_w=None, gate_raw=None, cu_seqlens=None,
                cu_seqlens_host=None, N=None, T=None, K=4, gate_mode=0, gate_lb=-5.0,
                l2_eps=1e-6, rms_eps=1e-6, scale=None, algo=kda.ALGO_AUTO, state_out=None,
                ring_out=None, out=None, gate_exp=None, workspace=None, stream=None):
    """Run the mixer on device tensors.  Either (N, T) for N sequences of T tokens, or
    cu_seqlens (int32 device) + cu_seqlens_host (int32 CPU) for packed sequences.
    gate_exp: hand the gate from the prep to the scan as decay factors exp(log-decay) (the
    prep takes the exp once per element instead of every sequential-scan CTA taking it); the
    returned g then holds decay factors.  Default: on for the sequential form, off otherwise (the
    chunked form consumes log-decays).
    workspace: scratch for the chunked form; allocated here when algo is AUTO or CHUNK and none
    is given.
    Returns a dict with q_hat, k_hat, v_hat, g, beta, o, y (None without an epilogue),
    state_out and ring_out."""
    D = kda.HEAD_DIM
    C = H * D
    rows = q_raw.shape[0]
    varlen = cu_seqlens is not None
    if not varlen:
        assert N is not None and T is not None and N * T == rows
    n_seq = (cu_seqlens_host.numel() - 1) if varlen else N
    buf = out if out is not None else {}

    def take(name, shape):
        t = buf.get(name)
        return t if t is not None else _empty(shape, q_raw)
    q_hat = take("q_hat", (rows, C))
    k_hat = take("k_hat", (rows, C))
    v_hat = take("v_hat", (rows, C))
    g = take("g", (rows, C) if gate_mode == 0 else (rows, H))
    beta = take("beta", (rows, H))
    o = take("o", (rows, C))
    if state_out is None:
        state_out = torch.empty_like(state_in)
    if conv_w is not None and ring_out is None:
        ring_out = torch.empty_like(ring_in)
    if workspace is None and algo != kda.ALGO_SEQ:
        workspace = kda.scan_workspace(n_seq, rows, H, q_raw.device, algo)
    if gate_exp is None:
        gate_exp = algo == kda.ALGO_SEQ
    gm = gate_mode | (kda.GATE_EXP if gate_exp else 0)
    common = dict(H=H, K=K, gate_mode=gm, gate_lb=gate_lb, l2_eps=l2_eps, stream=stream)
    if varlen:
        kda.kda_conv_l2norm_prep_varlen(q_raw, k_raw, v_raw, conv_w, ring_in, ring_out, f_raw,
                                        dt_bias, a_log, beta_raw, q_hat, k_hat, v_hat, g, beta,
                                        cu_seqlens, cu_seqlens_host, **common)
        kda.kda_scan_varlen(q_hat, k_hat, v_hat, g, beta, state_in, state_out, o, cu_seqlens,
                            cu_seqlens_host, H=H, gate_mode=gm, scale=scale, algo=algo,
                            workspace=workspace, stream=stream)
    else:
        kda.kda_conv_l2norm_prep(q_raw, k_raw, v_raw, conv_w, ring_in, ring_out, f_raw, dt_bias,
                                 a_log, beta_raw, q_hat, k_hat, v_hat, g, beta, N=N, T=T,
                                 **common)
        kda.kda_scan(q_hat, k_hat, v_hat, g, beta, state_in, state_out, o, N=N, T=T, H=H,
                     gate_mode=gm, scale=scale, algo=algo, workspace=workspace, stream=stream)
    y = None
    if norm_w is not None:
        y = take("y", (rows, C))
        kda.kda_gated_rmsnorm_out(o, norm_w, gate_raw, y, rows=rows * H, eps=rms_eps,
                                  stream=stream)
    return dict(q_hat=q_hat, k_hat=k_hat, v_hat=v_hat, g=g, beta=beta, o=o, y=y,
                state_out=state_out, ring_out=ring_out, n_seq=n_seq)


def kda_prefill(*, q_raw, k_raw, v_raw, f_raw, dt_bias, a_log, beta_raw, state_in, H, conv_w,
                ring_in, norm_w, gate_raw, cu_seqlens=None, cu_seqlens_host=None, N=None, T=None,
                K=4, gate_mode=0, gate_lb=-5.0, l2_eps=1e-6, rms_eps=1e-6, scale=None,
                state_out=None, ring_out=None, y=None, workspace=None, stream=None):
    """The whole mixer for a prefill in one library call (kda_prefill_fused[_varlen]): conv +
    SiLU, l2 norm, gates, the chunked scan and the gated RMSNorm, the intermediates kept in the
    workspace.  Either (N, T) or cu_seqlens (int32 device) + cu_seqlens_host (int32
    CPU).  workspace: from kda.prefill_workspace (allocated here when None).
    Returns a dict with y, state_out and ring_out."""
    C = H * kda.HEAD_DIM
    rows = q_raw.shape[0]
    varlen = cu_seqlens is not None
    if not varlen:
        assert N is not None and T is not None and N * T == rows
    n_seq = (cu_seqlens_host.numel() - 1) if varlen else N
    if y is None:
        y = _empty((rows, C), q_raw)
    if state_out is None:
        state_out = torch.empty_like(state_in)
    if ring_out is None and conv_w is not None:
        ring_out = torch.empty_like(ring_in)
    if workspace is None:
        workspace = kda.prefill_workspace(n_seq, rows, H, q_raw.device, gate_mode)
    args = (q_raw, k_raw, v_raw, conv_w, ring_in, ring_out, f_raw, dt_bias, a_log, beta_raw,
            state_in, state_out, norm_w, gate_raw, y, workspace)
    common = dict(H=H, K=K, gate_mode=gate_mode, gate_lb=gate_lb, l2_eps=l2_eps, scale=scale,
                  rms_eps=rms_eps, stream=stream)
    if varlen:
        kda.kda_prefill_fused_varlen(*args, cu_seqlens, cu_seqlens_host, **common)
    else:
        kda.kda_prefill_fused(*args, N=N, T=T, **common)
    return dict(y=y, state_out=state_out, ring_out=ring_out, n_seq=n_seq)


def kda_decode(*, q_raw, k_raw, v_raw, conv_w, ring_in, f_raw, dt_bias, a_log, beta_raw,
               state_in, norm_w, gate_raw, N, T, H, K=4, gate_mode=0, gate_lb=-5.0,
               l2_eps=1e-6, rms_eps=1e-6, scale=None, state_out=None, ring_out=None, y=None,
               stream=None):
    """One fused decode (T=1) or T-token verify launch.  ring_out may be ring_in (in place)."""
    if state_out is None:
        state_out = torch.empty_like(state_in)
    if ring_out is None:
        ring_out = torch.empty_like(ring_in)
    if y is None:
        y = _empty((q_raw.shape[0], H * kda.HEAD_DIM), q_raw)
    kda.kda_decode_fused(q_raw, k_raw, v_raw, conv_w, ring_in, ring_out, f_raw, dt_bias, a_log,
                         beta_raw, state_in, state_out, norm_w, gate_raw, y, N=N, T=T, H=H, K=K,
                         gate_mode=gate_mode, gate_lb=gate_lb, l2_eps=l2_eps, scale=scale,
                         rms_eps=rms_eps, stream=stream)
    return dict(y=y, state_out=state_out, ring_out=ring_out)
