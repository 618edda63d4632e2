"""Whole-mixer convenience calls over the C ABI: allocate the intermediate and output buffers
with torch on the inputs' device and run the entry points in the mixer's stage order
(prep -> scan -> gated RMSNorm, or the single fused decode/verify launch).  Plumbing only: every
value is computed by the library's kernels.
"""

from __future__ import annotations

import torch

from . import kda


def _norm_flag(norm_gate):
    if norm_gate not in ("sigmoid", "silu"):
        raise ValueError(norm_gate)
    return kda.NORM_SILU if norm_gate == "silu" else 0


def _empty(shape, like):
    return torch.empty(shape, dtype=torch.float32, device=like.device)


def kda_forward(*, q_raw, k_raw, v_raw, f_raw, dt_bias, a_log, beta_raw, state_in, H,
                conv_w=None, ring_in=None, norm_w=None, gate_raw=None, cu_seqlens=None,
                cu_seqlens_host=None, N=None, T=None, K=4, gate_mode=0, gate_lb=-5.0,
                l2_eps=1e-6, rms_eps=1e-6, scale=None, algo=kda.ALGO_AUTO, state_out=None,
                ring_out=None, out=None, gate_exp=None, workspace=None, stream=None,
                norm_gate="sigmoid", Hk=None, Dv=None):
    """Run the mixer on device tensors.  Either (N, T) for N sequences of T tokens, or
    cu_seqlens (int32 device) + cu_seqlens_host (int32 CPU) for packed sequences.
    gate_exp: hand the gate from the prep to the scan as decay factors exp(log-decay) (the
    prep takes the exp once per element instead of every sequential-scan CTA taking it); the
    returned g then holds decay factors.  Default: on for the sequential form, off otherwise (the
    chunked form consumes log-decays).
    workspace: scratch for the chunked form; allocated here when algo is AUTO or CHUNK and none
    is given.
    norm_gate: the RMSNorm's gate, "sigmoid" (KDA) or "silu" (GDN's gated_rmsnorm).
    Hk: grouped queries (q_raw / k_raw of Hk heads, value head h reads q/k head h % Hk).
    Dv: value heads Dv wide (a multiple of 128; q/k heads stay 128 wide; state [N, H, Dv, 128]).
    Returns a dict with q_hat, k_hat, v_hat, g, beta, o, y (None without an epilogue),
    state_out and ring_out."""
    D = kda.HEAD_DIM
    wide = Dv is not None
    Dv = D if Dv is None else Dv
    C = H * Dv
    Cg = H * D                      # per-channel gate rows: the key dim of every value head
    Cq = (H if Hk is None else Hk) * D
    rows = q_raw.shape[0]
    varlen = cu_seqlens is not None
    if not varlen:
        assert N is not None and T is not None and N * T == rows
    n_seq = (cu_seqlens_host.numel() - 1) if varlen else N
    buf = out if out is not None else {}

    def take(name, shape):
        t = buf.get(name)
        return t if t is not None else _empty(shape, q_raw)
    q_hat = take("q_hat", (rows, Cq))
    k_hat = take("k_hat", (rows, Cq))
    v_hat = take("v_hat", (rows, C))
    g = take("g", (rows, Cg) if gate_mode == 0 else (rows, H))
    beta = take("beta", (rows, H))
    o = take("o", (rows, C))
    if state_out is None:
        state_out = torch.empty_like(state_in)
    if conv_w is not None and ring_out is None:
        ring_out = torch.empty_like(ring_in)
    if workspace is None and algo != kda.ALGO_SEQ:
        workspace = kda.scan_workspace(n_seq, rows, H * Dv // D, q_raw.device, algo)
    if gate_exp is None:
        gate_exp = algo == kda.ALGO_SEQ
    gm = gate_mode | (kda.GATE_EXP if gate_exp else 0)
    common = dict(H=H, K=K, gate_mode=gm, gate_lb=gate_lb, l2_eps=l2_eps, stream=stream, Hk=Hk)
    scan_kw = dict(H=H, gate_mode=gm, scale=scale, algo=algo, workspace=workspace, stream=stream)
    if wide:
        common.update(Dv=Dv)
        scan_kw.update(Hk=Hk, Dv=Dv)
        if varlen:
            kda.kda_conv_l2norm_prep_varlen_dv(q_raw, k_raw, v_raw, conv_w, ring_in, ring_out,
                                               f_raw, dt_bias, a_log, beta_raw, q_hat, k_hat,
                                               v_hat, g, beta, cu_seqlens, cu_seqlens_host,
                                               **common)
            kda.kda_scan_varlen_dv(q_hat, k_hat, v_hat, g, beta, state_in, state_out, o,
                                   cu_seqlens, cu_seqlens_host, **scan_kw)
        else:
            kda.kda_conv_l2norm_prep_dv(q_raw, k_raw, v_raw, conv_w, ring_in, ring_out, f_raw,
                                        dt_bias, a_log, beta_raw, q_hat, k_hat, v_hat, g, beta,
                                        N=N, T=T, **common)
            kda.kda_scan_dv(q_hat, k_hat, v_hat, g, beta, state_in, state_out, o, N=N, T=T,
                            **scan_kw)
    elif varlen:
        kda.kda_conv_l2norm_prep_varlen(q_raw, k_raw, v_raw, conv_w, ring_in, ring_out, f_raw,
                                        dt_bias, a_log, beta_raw, q_hat, k_hat, v_hat, g, beta,
                                        cu_seqlens, cu_seqlens_host, **common)
        scan_args = (q_hat, k_hat, v_hat, g, beta, state_in, state_out, o, cu_seqlens,
                     cu_seqlens_host)
        if Hk is None:
            kda.kda_scan_varlen(*scan_args, **scan_kw)
        else:
            kda.kda_scan_varlen_gqa(*scan_args, Hk=Hk, **scan_kw)
    else:
        kda.kda_conv_l2norm_prep(q_raw, k_raw, v_raw, conv_w, ring_in, ring_out, f_raw, dt_bias,
                                 a_log, beta_raw, q_hat, k_hat, v_hat, g, beta, N=N, T=T,
                                 **common)
        scan_args = (q_hat, k_hat, v_hat, g, beta, state_in, state_out, o)
        if Hk is None:
            kda.kda_scan(*scan_args, N=N, T=T, **scan_kw)
        else:
            kda.kda_scan_gqa(*scan_args, N=N, T=T, Hk=Hk, **scan_kw)
    y = None
    if norm_w is not None:
        y = take("y", (rows, C))
        _norm_flag(norm_gate)
        norm = kda.kda_gated_rmsnorm_silu_out if norm_gate == "silu" else kda.kda_gated_rmsnorm_out
        norm(o, norm_w, gate_raw, y, rows=rows * H, eps=rms_eps, D=Dv, stream=stream)
    return dict(q_hat=q_hat, k_hat=k_hat, v_hat=v_hat, g=g, beta=beta, o=o, y=y,
                state_out=state_out, ring_out=ring_out, n_seq=n_seq)


def kda_prefill(*, q_raw, k_raw, v_raw, f_raw, dt_bias, a_log, beta_raw, state_in, H, conv_w,
                ring_in, norm_w, gate_raw, cu_seqlens=None, cu_seqlens_host=None, N=None, T=None,
                K=4, gate_mode=0, gate_lb=-5.0, l2_eps=1e-6, rms_eps=1e-6, scale=None,
                state_out=None, ring_out=None, y=None, workspace=None, stream=None,
                norm_gate="sigmoid", Hk=None, Dv=None):
    """The whole mixer for a prefill in one library call (kda_prefill_fused[_varlen]): conv +
    SiLU, l2 norm, gates, the chunked scan and the gated RMSNorm, the intermediates kept in the
    workspace.  Either (N, T) or cu_seqlens (int32 device) + cu_seqlens_host (int32
    CPU).  workspace: from kda.prefill_workspace (allocated here when None).
    norm_gate: the RMSNorm's gate, "sigmoid" (KDA) or "silu" (GDN's gated_rmsnorm).
    Dv: value heads Dv wide (the _dv entries; the workspace counts H * Dv / 128 units).
    Returns a dict with y, state_out and ring_out."""
    units = H if Dv is None else H * Dv // kda.HEAD_DIM
    C = units * kda.HEAD_DIM
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
        workspace = kda.prefill_workspace(n_seq, rows, units, q_raw.device, gate_mode)
    args = (q_raw, k_raw, v_raw, conv_w, ring_in, ring_out, f_raw, dt_bias, a_log, beta_raw,
            state_in, state_out, norm_w, gate_raw, y, workspace)
    common = dict(H=H, K=K, gate_mode=gate_mode | _norm_flag(norm_gate), gate_lb=gate_lb,
                  l2_eps=l2_eps, scale=scale, rms_eps=rms_eps, stream=stream, Hk=Hk, Dv=Dv)
    if varlen:
        kda.kda_prefill_fused_varlen(*args, cu_seqlens, cu_seqlens_host, **common)
    else:
        kda.kda_prefill_fused(*args, N=N, T=T, **common)
    return dict(y=y, state_out=state_out, ring_out=ring_out, n_seq=n_seq)


def kda_decode(*, q_raw, k_raw, v_raw, conv_w, ring_in, f_raw, dt_bias, a_log, beta_raw,
               state_in, norm_w, gate_raw, N, T, H, K=4, gate_mode=0, gate_lb=-5.0,
               l2_eps=1e-6, rms_eps=1e-6, scale=None, state_out=None, ring_out=None, y=None,
               stream=None, norm_gate="sigmoid", Hk=None, Dv=None):
    """One fused decode (T=1) or T-token verify launch.  ring_out may be ring_in and state_out
    state_in (in place).  norm_gate: "sigmoid" (KDA) or "silu" (GDN's gated_rmsnorm).
    Dv: value heads Dv wide (kda_decode_fused_dv)."""
    if state_out is None:
        state_out = torch.empty_like(state_in)
    if ring_out is None:
        ring_out = torch.empty_like(ring_in)
    if y is None:
        y = _empty((q_raw.shape[0], H * (kda.HEAD_DIM if Dv is None else Dv)), q_raw)
    kda.kda_decode_fused(q_raw, k_raw, v_raw, conv_w, ring_in, ring_out, f_raw, dt_bias, a_log,
                         beta_raw, state_in, state_out, norm_w, gate_raw, y, N=N, T=T, H=H, K=K,
                         gate_mode=gate_mode | _norm_flag(norm_gate), gate_lb=gate_lb,
                         l2_eps=l2_eps, scale=scale,
                         rms_eps=rms_eps, stream=stream, Hk=Hk, Dv=Dv)
    return dict(y=y, state_out=state_out, ring_out=ring_out)


def kda_verify_rollback(*, q_raw, k_raw, v_raw, conv_w, ring_in, f_raw, dt_bias, a_log,
                        beta_raw, state_in, norm_w, gate_raw, keep, N, T, H, K=4, gate_mode=0,
                        gate_lb=-5.0, l2_eps=1e-6, rms_eps=1e-6, scale=None, state_out=None,
                        ring_out=None, y=None, stream=None, norm_gate="sigmoid", Hk=None,
                        Dv=None):
    """Roll a T-token verify round back to the accepted prefixes: keep (int32 device [N]) tokens
    of each sequence, from the pre-round state_in and ring_in.  ring_out may be ring_in."""
    if state_out is None:
        state_out = torch.empty_like(state_in)
    if ring_out is None:
        ring_out = torch.empty_like(ring_in)
    if y is None:
        y = torch.zeros((q_raw.shape[0], H * (kda.HEAD_DIM if Dv is None else Dv)),
                        dtype=torch.float32, device=q_raw.device)
    kda.kda_verify_rollback(q_raw, k_raw, v_raw, conv_w, ring_in, ring_out, f_raw, dt_bias,
                            a_log, beta_raw, state_in, state_out, norm_w, gate_raw, y, keep,
                            N=N, T=T, H=H, K=K, gate_mode=gate_mode | _norm_flag(norm_gate),
                            gate_lb=gate_lb, l2_eps=l2_eps, scale=scale, rms_eps=rms_eps,
                            stream=stream, Hk=Hk, Dv=Dv)
    return dict(y=y, state_out=state_out, ring_out=ring_out)


class HostPrefillStream:
    """Prefill over batches that live in pinned host memory, pipelined over three CUDA streams:
    while batch i runs kda_prefill on the device, batch i+1 is copied in and the results of
    batch i-1 are copied out (the host<->device link is full duplex, so the two copies overlap
    each other as well as the kernels).  Every batch moves its own inputs and results; nothing is
    cached between batches.

    Layout: `slots` (default 2) device copies of the per-batch inputs and outputs, used in turn;
    one prefill workspace, since the prefills run in order on one stream.  The weights (conv_w,
    dt_bias, a_log, norm_w) are model parameters and stay resident on the device.
    Fixed-length batches only: every batch has the N, T, H given here.

    submit(host_in, host_out) queues one batch and returns at once.  host_in maps BATCH_KEYS to
    pinned CPU tensors (ring_in only when the mixer has a conv); host_out maps y, state_out and
    (with a conv) ring_out to pinned CPU tensors that receive the results.  Neither may be
    touched by the host until synchronize() returns.  Ordering: a slot's inputs are overwritten
    only after the prefill that read them finished, and its outputs only after they were copied
    out (CUDA events on the streams; the host never blocks in submit)."""

    BATCH_KEYS = ("q_raw", "k_raw", "v_raw", "f_raw", "beta_raw", "gate_raw", "state_in",
                  "ring_in")

    def __init__(self, *, like, conv_w, dt_bias, a_log, norm_w, H, N, T, K=4, gate_mode=0,
                 gate_lb=-5.0, l2_eps=1e-6, rms_eps=1e-6, scale=None, slots=2):
        dev = dt_bias.device
        if dev.type != "cuda":
            raise ValueError("HostPrefillStream: the weights must be CUDA tensors")
        self.keys = tuple(k for k in self.BATCH_KEYS
                          if not (k == "ring_in" and conv_w is None))
        self.weights = dict(conv_w=conv_w, dt_bias=dt_bias, a_log=a_log, norm_w=norm_w)
        self.params = dict(H=H, N=N, T=T, K=K, gate_mode=gate_mode, gate_lb=gate_lb,
                           l2_eps=l2_eps, rms_eps=rms_eps, scale=scale)
        rows, C = N * T, H * kda.HEAD_DIM
        self.slots = []
        for _ in range(slots):
            din = {k: torch.empty(like[k].shape, dtype=like[k].dtype, device=dev)
                   for k in self.keys}
            dout = dict(y=torch.empty(rows, C, dtype=torch.float32, device=dev),
                        state_out=torch.empty_like(din["state_in"]))
            if conv_w is not None:
                dout["ring_out"] = torch.empty_like(din["ring_in"])
            self.slots.append((din, dout, dict(copied=torch.cuda.Event(),
                                               ran=torch.cuda.Event(),
                                               drained=torch.cuda.Event())))
        self.workspace = kda.prefill_workspace(N, rows, H, dev, gate_mode)
        self.copy_in = torch.cuda.Stream(dev)
        self.run = torch.cuda.Stream(dev)
        self.copy_out = torch.cuda.Stream(dev)
        self.submitted = 0
        # the buffers live on the default stream's pool but are used on the three streams: the
        # allocator keeps their memory until work queued there has finished, even if this
        # object is dropped early
        for din, dout, _ in self.slots:
            for t in (*din.values(), *dout.values()):
                for st in (self.copy_in, self.run, self.copy_out):
                    t.record_stream(st)
        self.workspace.record_stream(self.run)

    @property
    def h2d_bytes_per_batch(self) -> int:
        din = self.slots[0][0]
        return sum(t.numel() * t.element_size() for t in din.values())

    @property
    def d2h_bytes_per_batch(self) -> int:
        dout = self.slots[0][1]
        return sum(t.numel() * t.element_size() for t in dout.values())

    def submit(self, host_in, host_out):
        din, dout, ev = self.slots[self.submitted % len(self.slots)]
        reused = self.submitted >= len(self.slots)
        if reused:                          # the slot's previous prefill has read its inputs
            self.copy_in.wait_event(ev["ran"])
        with torch.cuda.stream(self.copy_in):
            for k in self.keys:
                din[k].copy_(host_in[k], non_blocking=True)
        ev["copied"].record(self.copy_in)
        self.run.wait_event(ev["copied"])
        if reused:                          # the slot's previous results have been copied out
            self.run.wait_event(ev["drained"])
        kda_prefill(**{"ring_in": None, **din}, **self.weights, **self.params, y=dout["y"],
                    state_out=dout["state_out"], ring_out=dout.get("ring_out"),
                    workspace=self.workspace, stream=self.run)
        ev["ran"].record(self.run)
        self.copy_out.wait_event(ev["ran"])
        with torch.cuda.stream(self.copy_out):
            for k, t in dout.items():
                host_out[k].copy_(t, non_blocking=True)
        ev["drained"].record(self.copy_out)
        self.submitted += 1

    def record_done(self, event):
        """Record `event` on the copy-out stream: it completes once every batch submitted so far
        has been copied in, run and copied out."""
        event.record(self.copy_out)

    def synchronize(self):
        self.copy_out.synchronize()
        self.run.synchronize()
        self.copy_in.synchronize()

    def close(self):
        """Wait for every submitted batch; the host buffers given to submit() are then free."""
        self.synchronize()
