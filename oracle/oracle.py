"""Python face of the f64 CPU oracle (``kda_oracle.c``).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's CPU-baseline leg
are the only callers.  The product path (the CUDA library and its binding) never imports this
module.  It shares no code with the CUDA path; the only thing both sides use is the seeded input
generator module, which holds none of the method's arithmetic.

Each wrapper converts its arguments to contiguous float64 numpy arrays, calls the matching C
routine, and returns float64 arrays.  Method sources are cited in ``kda_oracle.c``.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle into ``oracle/_build/libkda_oracle.so`` (plain gcc, OpenMP when the
    compiler has it).  ``-ffp-contract=off`` keeps every multiply and add separately rounded, so
    the oracle computes the same bits on x86 and Arm hosts.  ``src``/``out`` let the mutation
    tests build a deliberately broken copy elsewhere."""
    out_dir = os.path.dirname(out)
    os.makedirs(out_dir, exist_ok=True)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    base = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-ffp-contract=off", src, "-lm"]
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=out_dir)
    os.close(fd)
    try:
        try:
            subprocess.run(base[:-1] + ["-fopenmp", "-o", tmp, "-lm"], check=True,
                           capture_output=True)
        except subprocess.CalledProcessError:
            subprocess.run(base + ["-o", tmp], check=True, capture_output=True)
        os.replace(tmp, out)
    finally:
        if os.path.exists(tmp):
            os.remove(tmp)
    return out


def _bind(path: str):
    """Open one build of the oracle and declare its C signatures."""
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    lp = ctypes.POINTER(ctypes.c_int64)
    L, I, D = ctypes.c_long, ctypes.c_int, ctypes.c_double
    lib.orc_num_threads.restype = I
    lib.orc_conv_silu.argtypes = [dp, L, dp, dp, dp, L, dp, I, I, I]
    lib.orc_l2norm.argtypes = [dp, dp, L, I, D]
    lib.orc_gate_kda.argtypes = [dp, dp, dp, D, dp, L, I, I]
    lib.orc_gate_gdn.argtypes = [dp, dp, dp, dp, L, I]
    lib.orc_sigmoid.argtypes = [dp, dp, L]
    for fn in (lib.orc_scan_kda, lib.orc_scan_gdn):
        fn.argtypes = [dp, dp, dp, dp, dp, lp, I, I, I, dp, dp, dp, D]
    lib.orc_gated_rmsnorm.argtypes = [dp, dp, dp, dp, L, I, D, I]
    lib.orc_matvec_rows.argtypes = [dp, dp, dp, L, L, I]
    lib.orc_scan_kda_rect.argtypes = [dp, dp, dp, dp, dp, lp, I, I, I, I, dp, dp, dp, D]
    lib.orc_scan_kda_rect.restype = None
    for name in ("orc_conv_silu", "orc_l2norm", "orc_gate_kda", "orc_gate_gdn",
                 "orc_sigmoid", "orc_scan_kda", "orc_scan_gdn", "orc_gated_rmsnorm",
                 "orc_matvec_rows"):
        getattr(lib, name).restype = None
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
    return _lib


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor: exact upcast (bf16 / f32 -> f64)
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def num_threads() -> int:
    """OpenMP threads the oracle's parallel loops use."""
    return int(_load().orc_num_threads())


# ------------------------------------------------------------------------------------------
# single steps
# ------------------------------------------------------------------------------------------

def conv_silu(x, w, ring_in):
    """a1 + a2 for one sequence and one set of channels.

    x: [T, Cch] raw rows, w: [Cch, K] or None (no conv: y = x), ring_in: [Cch, K-1].
    Returns (y [T, Cch], ring_out [Cch, K-1] or None).
    """
    lib = _load()
    x = _f64(x)
    T, Cch = x.shape
    y = np.empty((T, Cch))
    if w is None:
        lib.orc_conv_silu(_p(x), Cch, None, None, _p(y), Cch, None, T, Cch, 0)
        return y, None
    w = _f64(w)
    K = w.shape[1]
    ring_in = _f64(ring_in).reshape(Cch, K - 1)
    ring_out = np.empty((Cch, K - 1))
    lib.orc_conv_silu(_p(x), Cch, _p(w), _p(ring_in), _p(y), Cch, _p(ring_out), T, Cch, K)
    return y, ring_out


def l2norm(x, D: int, eps: float = 1e-6):
    """a3 over rows of length D (any leading shape whose size is a multiple of D)."""
    x = _f64(x)
    y = np.empty_like(x)
    _load().orc_l2norm(_p(x), _p(y), x.size // D, D, eps)
    return y


def gate_kda(f, dt_bias, a_log, lb: float = -5.0):
    """a4, KDA per-channel gate.  f: [rows, H*D], dt_bias: [H*D], a_log: [H]."""
    f, dt_bias, a_log = _f64(f), _f64(dt_bias), _f64(a_log)
    H = a_log.size
    D = dt_bias.size // H
    rows = f.size // (H * D)
    g = np.empty_like(f)
    _load().orc_gate_kda(_p(f), _p(dt_bias), _p(a_log), lb, _p(g), rows, H, D)
    return g


def gate_gdn(alpha, dt_bias, a_log):
    """a4, GDN per-head gate.  alpha: [rows, H], dt_bias: [H], a_log: [H]."""
    alpha, dt_bias, a_log = _f64(alpha), _f64(dt_bias), _f64(a_log)
    H = a_log.size
    g = np.empty_like(alpha)
    _load().orc_gate_gdn(_p(alpha), _p(dt_bias), _p(a_log), _p(g), alpha.size // H, H)
    return g


def sigmoid(x):
    x = _f64(x)
    y = np.empty_like(x)
    _load().orc_sigmoid(_p(x), _p(y), x.size)
    return y


def _cu(cu_seqlens, rows):
    if cu_seqlens is None:
        return np.array([0, rows], dtype=np.int64)
    return np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))


def scan_kda(q, k, v, g, beta, state_in, cu_seqlens=None, scale=None):
    """a5, KDA scan.  q, k, v, g: [rows, H, D]; beta: [rows, H]; state_in: [N, H, D, D] in the
    M[j][i] = S[i][j] layout.  Returns (o [rows, H, D], state_out [N, H, D, D])."""
    q, k, v, g, beta = (_f64(a) for a in (q, k, v, g, beta))
    state_in = _f64(state_in)
    N, H, D, _ = state_in.shape
    rows = q.size // (H * D)
    cu = _cu(cu_seqlens, rows)
    assert cu.size == N + 1 and cu[-1] == rows
    scale = D ** -0.5 if scale is None else float(scale)
    o = np.empty((rows, H, D))
    st = np.empty_like(state_in)
    _load().orc_scan_kda(_p(q), _p(k), _p(v), _p(g), _p(beta),
                         cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), N, H, D,
                         _p(state_in), _p(st), _p(o), scale)
    return o, st


def scan_kda_rect(q, k, v, g, beta, state_in, cu_seqlens=None, scale=None):
    """a5 with a value width of its own: q, k, g [rows, H, Dk]; v [rows, H, Dv]; beta [rows, H];
    state_in [N, H, Dv, Dk] (M[j][i] = S[i][j]).  Returns (o [rows, H, Dv], state_out)."""
    q, k, v, g, beta = (_f64(a) for a in (q, k, v, g, beta))
    state_in = _f64(state_in)
    N, H, Dv, Dk = state_in.shape
    rows = q.size // (H * Dk)
    cu = _cu(cu_seqlens, rows)
    assert cu.size == N + 1 and cu[-1] == rows
    scale = Dk ** -0.5 if scale is None else float(scale)
    o = np.empty((rows, H, Dv))
    st = np.empty_like(state_in)
    _load().orc_scan_kda_rect(_p(q), _p(k), _p(v), _p(g), _p(beta),
                              cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), N, H, Dk, Dv,
                              _p(state_in), _p(st), _p(o), scale)
    return o, st


def scan_gdn(q, k, v, g, beta, state_in, cu_seqlens=None, scale=None):
    """a5, separate scalar-gate GDN scan.  g: [rows, H] (one log-decay per token and head)."""
    q, k, v, g, beta = (_f64(a) for a in (q, k, v, g, beta))
    state_in = _f64(state_in)
    N, H, D, _ = state_in.shape
    rows = q.size // (H * D)
    cu = _cu(cu_seqlens, rows)
    assert cu.size == N + 1 and cu[-1] == rows
    scale = D ** -0.5 if scale is None else float(scale)
    o = np.empty((rows, H, D))
    st = np.empty_like(state_in)
    _load().orc_scan_gdn(_p(q), _p(k), _p(v), _p(g), _p(beta),
                         cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), N, H, D,
                         _p(state_in), _p(st), _p(o), scale)
    return o, st


def gated_rmsnorm(o, w, z, eps: float = 1e-6, gate: str = "sigmoid"):
    """a6 over rows of length D = w.size; gate "sigmoid" (KDA) or "silu" (GDN's
    gated_rmsnorm)."""
    if gate not in ("sigmoid", "silu"):
        raise ValueError(gate)
    o, w, z = _f64(o), _f64(w), _f64(z)
    D = w.size
    y = np.empty_like(o)
    _load().orc_gated_rmsnorm(_p(o), _p(w), _p(z), _p(y), o.size // D, D, eps,
                              1 if gate == "silu" else 0)
    return y


def matvec_rows(w, x):
    """One projection of token rows: out[s][r] = sum_k w[r][k] x[s][k] (terms k ascending, f64).
    w: [rows, in_f] (bf16 weights are upcast exactly), x: [t, in_f].  Returns [t, rows]."""
    w, x = _f64(w), _f64(x)
    rows, in_f = w.shape
    x = x.reshape(-1, in_f)
    t = x.shape[0]
    out = np.empty((t, rows))
    if t and rows:
        _load().orc_matvec_rows(_p(w), _p(x), _p(out), rows, in_f, t)
    return out


def proj6(x, w_q, w_k, w_v, w_fa, w_ga, w_b):
    """Stage 1 of the mixer: the six projections of the layer input x [t, hidden], in the pages'
    output order [q, k, v, forget_down, gate_down, beta_raw]."""
    return [matvec_rows(w, x) for w in (w_q, w_k, w_v, w_fa, w_ga, w_b)]


# ------------------------------------------------------------------------------------------
# the whole mixer, a1 .. a6
# ------------------------------------------------------------------------------------------

def forward(*, q_raw, k_raw, v_raw, f_raw, dt_bias, a_log, beta_raw, state_in, H, D,
            conv_w=None, ring_in=None, cu_seqlens=None, gate_mode=0, gate_lb=-5.0,
            norm_w=None, gate_raw=None, l2_eps=1e-6, rms_eps=1e-6, scale=None,
            scalar_scan=False, norm_gate="sigmoid", Hk=None, Dv=None):
    """The mixer from projected channels to the gated output, in the pages' stage order
    (conv+SiLU -> ring roll -> l2 norm -> gates -> scan -> gated RMSNorm).

    q_raw/k_raw/v_raw: [rows, C] raw (pre-conv) channels, C = H*D.
    Hk: grouped queries (gdn_ops.rs `gdn_delta_rule_into` doc): q_raw and k_raw hold Hk heads
        ([rows, Hk*D]) and value head h reads query/key head h % Hk; None means Hk = H.  The conv
        planes and the ring then hold Hk*D q channels, Hk*D k channels and C v channels.
    Dv: the value head width when it differs from the key width D (gdn_ops.rs
        `gdn_delta_rule_into` doc: head_k_dim and head_v_dim are separate): v_raw, gate_raw and y
        are [rows, H*Dv], state_in [N, H, Dv, D], norm_w [Dv], and the v conv plane and ring rows
        hold H*Dv channels.  None means Dv = D.
    conv_w: [2*Hk*D + H*Dv, K] fused q,k,v conv weights or None (then no conv / SiLU and no ring).
    ring_in: [N, 2*Hk*D + H*Dv, K-1].
    f_raw: [rows, C] (gate_mode 0, KDA) or [rows, H] (gate_mode 1, GDN).
    dt_bias: [C] (KDA) or [H] (GDN); a_log: [H]; beta_raw: [rows, H].
    state_in: [N, H, D, D] (M[j][i] layout).
    norm_w: [D] and gate_raw: [rows, C], or None for no epilogue.
    scalar_scan: run the separate scalar-gate routine (gate_mode 1 only).
    norm_gate: the RMSNorm's gate, "sigmoid" (KDA) or "silu" (GDN's gated_rmsnorm).
    Returns a dict with q_hat, k_hat, v_hat, g, beta, o, y (or None), state_out, ring_out.
    """
    C = H * D
    Hk = H if Hk is None else Hk
    Cq = Hk * D
    Dv = D if Dv is None else Dv
    Cv = H * Dv
    q_raw, k_raw, v_raw = _f64(q_raw), _f64(k_raw), _f64(v_raw)
    rows = q_raw.shape[0]
    cu = _cu(cu_seqlens, rows)
    N = cu.size - 1
    planes = [q_raw, k_raw, v_raw]
    widths = [Cq, Cq, Cv]                     # channels of the q, k and v planes
    offs = [0, Cq, 2 * Cq]                    # their first row in conv_w and the ring
    conv = [np.empty((rows, w)) for w in widths]
    ring_out = None
    if conv_w is not None:
        conv_w = _f64(conv_w)
        K = conv_w.shape[1]
        ring_in = _f64(ring_in).reshape(N, 2 * Cq + Cv, K - 1)
        ring_out = np.empty_like(ring_in)
    for n in range(N):
        r0, r1 = int(cu[n]), int(cu[n + 1])
        for p in range(3):
            if conv_w is None:
                y, _ = conv_silu(planes[p][r0:r1], None, None)
            else:
                sl = slice(offs[p], offs[p] + widths[p])
                y, ro = conv_silu(planes[p][r0:r1], conv_w[sl], ring_in[n, sl])
                ring_out[n, sl] = ro
            conv[p][r0:r1] = y
    q_hat = l2norm(conv[0], D, l2_eps)
    k_hat = l2norm(conv[1], D, l2_eps)
    v_hat = conv[2]
    # value head h reads query/key head h % Hk (the tiled order of gdn_delta_rule_into)
    qk_head = np.arange(H) % Hk
    q_scan = q_hat.reshape(rows, Hk, D)[:, qk_head]
    k_scan = k_hat.reshape(rows, Hk, D)[:, qk_head]
    if gate_mode == 0:
        g = gate_kda(f_raw, dt_bias, a_log, gate_lb)
    else:
        g = gate_gdn(f_raw, dt_bias, a_log)
    beta = sigmoid(beta_raw).reshape(rows, H)
    shp = (rows, H, D)
    if Dv != D:                               # separate value width: the rectangular routine
        assert not scalar_scan, "the scalar-gate routine is square"
        gk = g.reshape(shp) if gate_mode == 0 else np.repeat(g.reshape(rows, H, 1), D, axis=2)
        o, st = scan_kda_rect(q_scan, k_scan, v_hat.reshape(rows, H, Dv), gk, beta, state_in,
                              cu, scale)
    elif gate_mode == 0:
        o, st = scan_kda(q_scan, k_scan, v_hat.reshape(shp), g.reshape(shp), beta, state_in, cu,
                         scale)
    elif scalar_scan:
        o, st = scan_gdn(q_scan, k_scan, v_hat.reshape(shp), g.reshape(rows, H), beta, state_in,
                         cu, scale)
    else:  # the KDA routine with the per-head gate broadcast over the key dim
        gb = np.repeat(g.reshape(rows, H, 1), D, axis=2)
        o, st = scan_kda(q_scan, k_scan, v_hat.reshape(shp), gb, beta, state_in, cu, scale)
    y = None
    if norm_w is not None:
        y = gated_rmsnorm(o.reshape(rows, Cv), norm_w, gate_raw, rms_eps,
                          norm_gate).reshape(rows, Cv)
    return dict(q_hat=q_hat.reshape(rows, Cq), k_hat=k_hat.reshape(rows, Cq),
                v_hat=v_hat.reshape(rows, Cv), g=g, beta=beta, o=o.reshape(rows, Cv), y=y,
                state_out=st, ring_out=ring_out)
