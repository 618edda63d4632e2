"""ctypes binding of libkda (include/kda.h): argument marshalling only.

Each function has the name of the C entry point it calls and takes torch tensors where the C call
takes device pointers; it passes ``tensor.data_ptr()``, the shape integers and the CUDA stream
(default: torch's current stream on the tensors' device), and raises ``KdaError`` on a non-zero
status.  No step of the method runs here: every value is computed by the CUDA kernels behind the
ABI.  Importing this module loads the library and fails loudly when it is missing.
"""

from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkda.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"libkda.so not found at {LIB_PATH}; build it first "
        "(python -c 'import __graft_entry__ as g; g.build()')")
_lib = ctypes.CDLL(LIB_PATH)

DTYPE_F32, DTYPE_BF16 = 0, 1
GATE_PER_CHANNEL, GATE_PER_HEAD = 0, 1
GATE_EXP = 2  # flag: g holds decay factors exp(log-decay)
NORM_SILU = 4  # flag (fused entries): the RMSNorm gates with SiLU(z) instead of sigmoid(z)
ALGO_AUTO, ALGO_SEQ, ALGO_CHUNK = 0, 1, 2
HEAD_DIM = 128
DECODE_MAX_T = 16
STATIC_SCRATCH_BYTES = 32 << 20  # kda_scan_varlen_static's fixed device scratch

_P, _I, _F, _L, _Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_long, ctypes.c_size_t

_lib.kda_abi_version.restype = _I
_lib.kda_status_string.restype = ctypes.c_char_p
_lib.kda_status_string.argtypes = [_I]
_lib.kda_conv_l2norm_prep.restype = _I
_lib.kda_conv_l2norm_prep.argtypes = [_P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _I, _F, _P, _P, _P,
                                      _P, _P, _P, _I, _I, _I, _I, _I, _F, _P]
_lib.kda_conv_l2norm_prep_varlen.restype = _I
_lib.kda_conv_l2norm_prep_varlen.argtypes = [_P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _I, _F, _P,
                                             _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F,
                                             _P]
_lib.kda_scan_workspace_bytes.restype = _Z
_lib.kda_scan_workspace_bytes.argtypes = [_I, _I, _I, _I, _I, _I]
_lib.kda_scan.restype = _I
_lib.kda_scan.argtypes = [_P, _P, _P, _P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P, _Z, _P]
_lib.kda_scan_varlen.restype = _I
_lib.kda_scan_varlen.argtypes = [_P, _P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _F,
                                 _I, _P, _Z, _P]
_lib.kda_gated_rmsnorm_out.restype = _I
_lib.kda_scan_varlen_static.restype = _I
_lib.kda_scan_varlen_static.argtypes = [_P, _P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _I, _I, _I,
                                        _I, _F, _P]
_lib.kda_gated_rmsnorm_out.argtypes = [_P, _P, _P, _P, _L, _I, _F, _P]
_lib.kda_gated_rmsnorm_silu_out.restype = _I
_lib.kda_gated_rmsnorm_silu_out.argtypes = [_P, _P, _P, _P, _L, _I, _F, _P]
_lib.kda_decode_fused.restype = _I
_lib.kda_prefill_workspace_bytes.restype = _Z
_lib.kda_prefill_workspace_bytes.argtypes = [_I, _I, _I, _I, _I]
_lib.kda_prefill_fused.restype = _I
_lib.kda_prefill_fused.argtypes = [_P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _I, _F, _P, _P, _P, _P,
                                   _P, _P, _I, _I, _I, _I, _I, _F, _F, _F, _P, _Z, _P]
_lib.kda_prefill_fused_varlen.restype = _I
_lib.kda_prefill_fused_varlen.argtypes = [_P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _I, _F, _P, _P,
                                          _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _F, _F,
                                          _P, _Z, _P]
_lib.kda_kernel_timing.restype = _I
_lib.kda_kernel_timing.argtypes = [_I]
_lib.kda_kernel_times.restype = _I
_lib.kda_kernel_times.argtypes = [_I, _P, _P]
_lib.kda_kernel_name.restype = ctypes.c_char_p
_lib.kda_kernel_name.argtypes = [_I]
_lib.kda_decode_fused.argtypes = [_P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _I, _F, _P, _P, _P, _P,
                                  _P, _P, _I, _I, _I, _I, _I, _F, _F, _F, _P]
_lib.kda_verify_rollback.restype = _I
_lib.kda_verify_rollback.argtypes = [_P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _I, _F, _P, _P, _P,
                                     _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _F, _F, _P]
_lib.kda_device_status.restype = _I
_lib.kda_device_status.argtypes = [_P]
_lib.kda_scan_gqa.restype = _I
_lib.kda_scan_gqa.argtypes = [_P, _P, _P, _P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P,
                              _Z, _P]
_lib.kda_scan_varlen_gqa.restype = _I
_lib.kda_scan_varlen_gqa.argtypes = [_P, _P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I,
                                     _I, _F, _I, _P, _Z, _P]
_lib.kda_conv_l2norm_prep_gqa.restype = _I
_lib.kda_conv_l2norm_prep_gqa.argtypes = [_P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _I, _F, _P, _P,
                                          _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P]
_lib.kda_conv_l2norm_prep_varlen_gqa.restype = _I
_lib.kda_conv_l2norm_prep_varlen_gqa.argtypes = [_P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _I, _F,
                                                 _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I,
                                                 _I, _I, _F, _P]
_lib.kda_prefill_fused_gqa.restype = _I
_lib.kda_prefill_fused_gqa.argtypes = [_P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _I, _F, _P, _P, _P,
                                       _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _F, _F, _P, _Z, _P]
_lib.kda_prefill_fused_varlen_gqa.restype = _I
_lib.kda_prefill_fused_varlen_gqa.argtypes = [_P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _I, _F, _P,
                                              _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                                              _F, _F, _F, _P, _Z, _P]
_lib.kda_decode_fused_gqa.restype = _I
_lib.kda_decode_fused_gqa.argtypes = [_P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _I, _F, _P, _P, _P,
                                      _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _F, _F, _P]
_lib.kda_verify_rollback_gqa.restype = _I
_lib.kda_verify_rollback_gqa.argtypes = [_P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _I, _F, _P, _P,
                                         _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _F, _F,
                                         _P]
_lib.kda_proj6_workspace_bytes.restype = _Z
_lib.kda_proj6_workspace_bytes.argtypes = [_I, _I]
_lib.kda_proj6.restype = _I
_lib.kda_proj6.argtypes = [_P, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _P,
                           _Z, _P]
_lib.kda_conv_l2norm_prep_dv.restype = _I
_lib.kda_conv_l2norm_prep_dv.argtypes = [_P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _I, _F, _P, _P,
                                         _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P]
_lib.kda_conv_l2norm_prep_varlen_dv.restype = _I
_lib.kda_conv_l2norm_prep_varlen_dv.argtypes = [_P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _I, _F,
                                                _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I,
                                                _I, _I, _I, _F, _P]
_lib.kda_scan_dv.restype = _I
_lib.kda_scan_dv.argtypes = [_P, _P, _P, _P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I,
                             _P, _Z, _P]
_lib.kda_scan_varlen_dv.restype = _I
_lib.kda_scan_varlen_dv.argtypes = [_P, _P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I,
                                    _I, _I, _F, _I, _P, _Z, _P]
_lib.kda_prefill_fused_dv.restype = _I
_lib.kda_prefill_fused_dv.argtypes = [_P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _I, _F, _P, _P, _P,
                                      _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _F, _F, _P, _Z,
                                      _P]
_lib.kda_prefill_fused_varlen_dv.restype = _I
_lib.kda_prefill_fused_varlen_dv.argtypes = [_P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _I, _F, _P,
                                             _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                                             _I, _F, _F, _F, _P, _Z, _P]
_lib.kda_decode_fused_dv.restype = _I
_lib.kda_decode_fused_dv.argtypes = [_P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _I, _F, _P, _P, _P,
                                     _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _F, _F, _P]
_lib.kda_verify_rollback_dv.restype = _I
_lib.kda_verify_rollback_dv.argtypes = [_P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _I, _F, _P, _P,
                                        _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _F,
                                        _F, _P]
_lib.kda_selftest_wait_timeout.restype = _I
_lib.kda_selftest_wait_timeout.argtypes = [_P]

# every symbol include/kda.h declares
EXPORTED = ("kda_abi_version", "kda_status_string", "kda_conv_l2norm_prep",
            "kda_conv_l2norm_prep_varlen", "kda_scan_workspace_bytes", "kda_scan",
            "kda_scan_varlen", "kda_gated_rmsnorm_out", "kda_decode_fused", "kda_device_status",
            "kda_scan_varlen_static", "kda_prefill_workspace_bytes", "kda_prefill_fused",
            "kda_prefill_fused_varlen", "kda_kernel_timing", "kda_kernel_times",
            "kda_kernel_name", "kda_verify_rollback", "kda_gated_rmsnorm_silu_out",
            "kda_selftest_wait_timeout", "kda_scan_gqa", "kda_scan_varlen_gqa",
            "kda_proj6_workspace_bytes", "kda_proj6", "kda_conv_l2norm_prep_gqa",
            "kda_conv_l2norm_prep_varlen_gqa", "kda_prefill_fused_gqa",
            "kda_prefill_fused_varlen_gqa", "kda_decode_fused_gqa", "kda_verify_rollback_gqa",
            "kda_conv_l2norm_prep_dv", "kda_conv_l2norm_prep_varlen_dv", "kda_scan_dv",
            "kda_scan_varlen_dv", "kda_prefill_fused_dv", "kda_prefill_fused_varlen_dv",
            "kda_decode_fused_dv", "kda_verify_rollback_dv")


class KdaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: status {status} ({status_string(status)})")


def status_string(status: int) -> str:
    return _lib.kda_status_string(int(status)).decode()


def abi_version() -> int:
    return int(_lib.kda_abi_version())


def library():
    """The ctypes handle (for callers that pass raw pointers, e.g. host-side contract tests)."""
    return _lib


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream, *tensors) -> int | None:
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    for t in tensors:
        if isinstance(t, torch.Tensor) and t.is_cuda:
            return torch.cuda.current_stream(t.device).cuda_stream
    return None


def _check(fn: str, status: int):
    if status != 0:
        raise KdaError(fn, status)


def _call(fn: str, like, *args):
    """Call C entry ``fn`` with the device of tensor ``like`` current: the library keys its
    per-device lookups by the current device and requires the stream to belong to it (40012)."""
    if isinstance(like, torch.Tensor) and like.is_cuda:
        with torch.cuda.device(like.device):
            status = getattr(_lib, fn)(*args)
    else:
        status = getattr(_lib, fn)(*args)
    _check(fn, status)


def _raw_dtype(t) -> int:
    return DTYPE_BF16 if t.dtype == torch.bfloat16 else DTYPE_F32


def _heads(H, Hk, D, Dv=None):
    """(name suffix, head arguments before K) of an entry point: the plain form (H, D), the _gqa
    form (H, Hk, D) when Hk is given, the _dv form (H, Hk, Dk = D, Dv) when Dv is given."""
    if Dv is not None:
        return "_dv", (H, H if Hk is None else Hk, D, Dv)
    return ("", (H, D)) if Hk is None else ("_gqa", (H, Hk, D))


def kda_conv_l2norm_prep(q_raw, k_raw, v_raw, conv_w, ring_in, ring_out, f_raw, dt_bias, a_log,
                         beta_raw, q_hat, k_hat, v_hat, g, beta, *, N, T, H, K=4, gate_mode=0,
                         gate_lb=-5.0, l2_eps=1e-6, D=HEAD_DIM, stream=None, Hk=None):
    """Hk: grouped queries (q/k planes of Hk heads; kda_conv_l2norm_prep_gqa)."""
    st = _stream(stream, q_hat)
    sfx, heads = _heads(H, Hk, D)
    _call("kda_conv_l2norm_prep" + sfx, q_hat,
        _ptr(q_raw), _ptr(k_raw), _ptr(v_raw), _raw_dtype(q_raw), _ptr(conv_w), _ptr(ring_in),
        _ptr(ring_out), _ptr(f_raw), _ptr(dt_bias), _ptr(a_log), gate_mode, gate_lb,
        _ptr(beta_raw), _ptr(q_hat), _ptr(k_hat), _ptr(v_hat), _ptr(g), _ptr(beta), N, T, *heads,
        K, l2_eps, st)


def kda_conv_l2norm_prep_varlen(q_raw, k_raw, v_raw, conv_w, ring_in, ring_out, f_raw, dt_bias,
                                a_log, beta_raw, q_hat, k_hat, v_hat, g, beta, cu_seqlens,
                                cu_seqlens_host, *, H, K=4, gate_mode=0, gate_lb=-5.0,
                                l2_eps=1e-6, D=HEAD_DIM, stream=None, Hk=None):
    """cu_seqlens: int32 device tensor [N+1]; cu_seqlens_host: int32 CPU tensor [N+1]."""
    N = cu_seqlens_host.numel() - 1
    total = int(cu_seqlens_host[-1])
    st = _stream(stream, q_hat)
    sfx, heads = _heads(H, Hk, D)
    _call("kda_conv_l2norm_prep_varlen" + sfx, q_hat,
        _ptr(q_raw), _ptr(k_raw), _ptr(v_raw), _raw_dtype(q_raw), _ptr(conv_w), _ptr(ring_in),
        _ptr(ring_out), _ptr(f_raw), _ptr(dt_bias), _ptr(a_log), gate_mode, gate_lb,
        _ptr(beta_raw), _ptr(q_hat), _ptr(k_hat), _ptr(v_hat), _ptr(g), _ptr(beta),
        _ptr(cu_seqlens), _ptr(cu_seqlens_host), N, total, *heads, K, l2_eps, st)


def kda_scan_workspace_bytes(N, total_T, H, gate_mode=0, algo=ALGO_AUTO, D=HEAD_DIM) -> int:
    return int(_lib.kda_scan_workspace_bytes(N, total_T, H, D, gate_mode, algo))


def chunk_block_bytes() -> int:
    """Workspace bytes of one (32-token chunk, head) block of the chunked form: a one-head,
    one-chunk varlen problem is sized for two blocks (a sequence may straddle one more chunk) plus
    the 256-byte header of chunk offsets."""
    return (kda_scan_workspace_bytes(1, 32, 1, algo=ALGO_CHUNK) - 256) // 2


def scan_workspace(N, total_T, H, device, algo=ALGO_AUTO):
    """A device byte buffer large enough for kda_scan / kda_scan_varlen (None when none is
    needed)."""
    nbytes = kda_scan_workspace_bytes(N, total_T, H, algo=algo)
    return None if nbytes == 0 else torch.empty(nbytes, dtype=torch.uint8, device=device)


def kda_scan(q_hat, k_hat, v_hat, g, beta, state_in, state_out, o, *, N, T, H, gate_mode=0,
             scale=None, algo=ALGO_AUTO, workspace=None, D=HEAD_DIM, stream=None):
    scale = D ** -0.5 if scale is None else scale
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = _stream(stream, state_out)
    _call("kda_scan", state_out,
        _ptr(q_hat), _ptr(k_hat), _ptr(v_hat), _ptr(g), gate_mode, _ptr(beta), _ptr(state_in),
        _ptr(state_out), _ptr(o), N, T, H, D, scale, algo, _ptr(workspace), ws_bytes, st)


def kda_scan_gqa(q_hat, k_hat, v_hat, g, beta, state_in, state_out, o, *, N, T, H, Hk,
                 gate_mode=0, scale=None, algo=ALGO_AUTO, workspace=None, D=HEAD_DIM, stream=None):
    """kda_scan with grouped queries: q_hat / k_hat have Hk heads, value head h reads h % Hk."""
    scale = D ** -0.5 if scale is None else scale
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = _stream(stream, state_out)
    _call("kda_scan_gqa", state_out,
        _ptr(q_hat), _ptr(k_hat), _ptr(v_hat), _ptr(g), gate_mode, _ptr(beta), _ptr(state_in),
        _ptr(state_out), _ptr(o), N, T, H, Hk, D, scale, algo, _ptr(workspace), ws_bytes, st)


def kda_scan_varlen_gqa(q_hat, k_hat, v_hat, g, beta, state_in, state_out, o, cu_seqlens,
                        cu_seqlens_host, *, H, Hk, gate_mode=0, scale=None, algo=ALGO_AUTO,
                        workspace=None, D=HEAD_DIM, stream=None):
    """kda_scan_varlen with grouped queries (see kda_scan_gqa)."""
    N = cu_seqlens_host.numel() - 1
    total = int(cu_seqlens_host[-1])
    scale = D ** -0.5 if scale is None else scale
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = _stream(stream, state_out)
    _call("kda_scan_varlen_gqa", state_out,
        _ptr(q_hat), _ptr(k_hat), _ptr(v_hat), _ptr(g), gate_mode, _ptr(beta), _ptr(state_in),
        _ptr(state_out), _ptr(o), _ptr(cu_seqlens), _ptr(cu_seqlens_host), N, total, H, Hk, D,
        scale, algo, _ptr(workspace), ws_bytes, st)


def kda_scan_varlen(q_hat, k_hat, v_hat, g, beta, state_in, state_out, o, cu_seqlens,
                    cu_seqlens_host, *, H, gate_mode=0, scale=None, algo=ALGO_AUTO,
                    workspace=None, D=HEAD_DIM, stream=None):
    N = cu_seqlens_host.numel() - 1
    total = int(cu_seqlens_host[-1])
    scale = D ** -0.5 if scale is None else scale
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = _stream(stream, state_out)
    _call("kda_scan_varlen", state_out,
        _ptr(q_hat), _ptr(k_hat), _ptr(v_hat), _ptr(g), gate_mode, _ptr(beta), _ptr(state_in),
        _ptr(state_out), _ptr(o), _ptr(cu_seqlens), _ptr(cu_seqlens_host), N, total, H, D, scale,
        algo, _ptr(workspace), ws_bytes, st)


def kda_conv_l2norm_prep_dv(q_raw, k_raw, v_raw, conv_w, ring_in, ring_out, f_raw, dt_bias,
                            a_log, beta_raw, q_hat, k_hat, v_hat, g, beta, *, N, T, H, Dv,
                            Hk=None, K=4, gate_mode=0, gate_lb=-5.0, l2_eps=1e-6, Dk=HEAD_DIM,
                            stream=None):
    """The prep with value heads Dv wide (a multiple of 128) and q/k heads Dk = 128 wide."""
    st = _stream(stream, q_hat)
    _call("kda_conv_l2norm_prep_dv", q_hat,
        _ptr(q_raw), _ptr(k_raw), _ptr(v_raw), _raw_dtype(q_raw), _ptr(conv_w), _ptr(ring_in),
        _ptr(ring_out), _ptr(f_raw), _ptr(dt_bias), _ptr(a_log), gate_mode, gate_lb,
        _ptr(beta_raw), _ptr(q_hat), _ptr(k_hat), _ptr(v_hat), _ptr(g), _ptr(beta), N, T, H,
        H if Hk is None else Hk, Dk, Dv, K, l2_eps, st)


def kda_conv_l2norm_prep_varlen_dv(q_raw, k_raw, v_raw, conv_w, ring_in, ring_out, f_raw,
                                   dt_bias, a_log, beta_raw, q_hat, k_hat, v_hat, g, beta,
                                   cu_seqlens, cu_seqlens_host, *, H, Dv, Hk=None, K=4,
                                   gate_mode=0, gate_lb=-5.0, l2_eps=1e-6, Dk=HEAD_DIM,
                                   stream=None):
    """kda_conv_l2norm_prep_dv over packed sequences."""
    N = cu_seqlens_host.numel() - 1
    total = int(cu_seqlens_host[-1])
    st = _stream(stream, q_hat)
    _call("kda_conv_l2norm_prep_varlen_dv", q_hat,
        _ptr(q_raw), _ptr(k_raw), _ptr(v_raw), _raw_dtype(q_raw), _ptr(conv_w), _ptr(ring_in),
        _ptr(ring_out), _ptr(f_raw), _ptr(dt_bias), _ptr(a_log), gate_mode, gate_lb,
        _ptr(beta_raw), _ptr(q_hat), _ptr(k_hat), _ptr(v_hat), _ptr(g), _ptr(beta),
        _ptr(cu_seqlens), _ptr(cu_seqlens_host), N, total, H, H if Hk is None else Hk, Dk, Dv, K,
        l2_eps, st)


def kda_scan_dv(q_hat, k_hat, v_hat, g, beta, state_in, state_out, o, *, N, T, H, Dv, Hk=None,
                gate_mode=0, scale=None, algo=ALGO_AUTO, workspace=None, Dk=HEAD_DIM,
                stream=None):
    """kda_scan with a Dk x Dv state per value head (state [N, H, Dv, Dk])."""
    scale = Dk ** -0.5 if scale is None else scale
    st = _stream(stream, state_out)
    _call("kda_scan_dv", state_out,
        _ptr(q_hat), _ptr(k_hat), _ptr(v_hat), _ptr(g), gate_mode, _ptr(beta), _ptr(state_in),
        _ptr(state_out), _ptr(o), N, T, H, H if Hk is None else Hk, Dk, Dv, scale, algo,
        _ptr(workspace), _ws_bytes(workspace), st)


def kda_scan_varlen_dv(q_hat, k_hat, v_hat, g, beta, state_in, state_out, o, cu_seqlens,
                       cu_seqlens_host, *, H, Dv, Hk=None, gate_mode=0, scale=None,
                       algo=ALGO_AUTO, workspace=None, Dk=HEAD_DIM, stream=None):
    """kda_scan_dv over packed sequences."""
    N = cu_seqlens_host.numel() - 1
    total = int(cu_seqlens_host[-1])
    scale = Dk ** -0.5 if scale is None else scale
    st = _stream(stream, state_out)
    _call("kda_scan_varlen_dv", state_out,
        _ptr(q_hat), _ptr(k_hat), _ptr(v_hat), _ptr(g), gate_mode, _ptr(beta), _ptr(state_in),
        _ptr(state_out), _ptr(o), _ptr(cu_seqlens), _ptr(cu_seqlens_host), N, total, H,
        H if Hk is None else Hk, Dk, Dv, scale, algo, _ptr(workspace), _ws_bytes(workspace), st)


def kda_scan_varlen_static(q_hat, k_hat, v_hat, g, beta, state_in, state_out, o, cu_seqlens,
                           cu_seqlens_host, *, H, gate_mode=0, scale=None, D=HEAD_DIM,
                           stream=None):
    """kda_scan_varlen's chunked form on the library's fixed device scratch (no allocation)."""
    N = cu_seqlens_host.numel() - 1
    total = int(cu_seqlens_host[-1])
    scale = D ** -0.5 if scale is None else scale
    st = _stream(stream, state_out)
    _call("kda_scan_varlen_static", state_out,
        _ptr(q_hat), _ptr(k_hat), _ptr(v_hat), _ptr(g), gate_mode, _ptr(beta), _ptr(state_in),
        _ptr(state_out), _ptr(o), _ptr(cu_seqlens), _ptr(cu_seqlens_host), N, total, H, D, scale,
        st)


def kda_gated_rmsnorm_out(o, norm_w, gate_raw, y, *, rows, eps=1e-6, D=HEAD_DIM, stream=None):
    st = _stream(stream, y)
    _call("kda_gated_rmsnorm_out", y,
        _ptr(o), _ptr(norm_w), _ptr(gate_raw), _ptr(y), rows, D, eps, st)


def kda_gated_rmsnorm_silu_out(o, norm_w, gate_raw, y, *, rows, eps=1e-6, D=HEAD_DIM,
                               stream=None):
    st = _stream(stream, y)
    _call("kda_gated_rmsnorm_silu_out", y,
        _ptr(o), _ptr(norm_w), _ptr(gate_raw), _ptr(y), rows, D, eps, st)


def kda_decode_fused(q_raw, k_raw, v_raw, conv_w, ring_in, ring_out, f_raw, dt_bias, a_log,
                     beta_raw, state_in, state_out, norm_w, gate_raw, y, *, N, T, H, K=4,
                     gate_mode=0, gate_lb=-5.0, l2_eps=1e-6, scale=None, rms_eps=1e-6,
                     D=HEAD_DIM, stream=None, Hk=None, Dv=None):
    scale = D ** -0.5 if scale is None else scale
    st = _stream(stream, y)
    sfx, heads = _heads(H, Hk, D, Dv)
    _call("kda_decode_fused" + sfx, y,
        _ptr(q_raw), _ptr(k_raw), _ptr(v_raw), _raw_dtype(q_raw), _ptr(conv_w), _ptr(ring_in),
        _ptr(ring_out), _ptr(f_raw), _ptr(dt_bias), _ptr(a_log), gate_mode, gate_lb,
        _ptr(beta_raw), _ptr(state_in), _ptr(state_out), _ptr(norm_w), _ptr(gate_raw), _ptr(y),
        N, T, *heads, K, l2_eps, scale, rms_eps, st)


def kda_verify_rollback(q_raw, k_raw, v_raw, conv_w, ring_in, ring_out, f_raw, dt_bias, a_log,
                        beta_raw, state_in, state_out, norm_w, gate_raw, y, keep, *, N, T, H, K=4,
                        gate_mode=0, gate_lb=-5.0, l2_eps=1e-6, scale=None, rms_eps=1e-6,
                        D=HEAD_DIM, stream=None, Hk=None, Dv=None):
    """keep: int32 device tensor [N], tokens accepted per sequence of the T-token verify batch."""
    scale = D ** -0.5 if scale is None else scale
    st = _stream(stream, y)
    sfx, heads = _heads(H, Hk, D, Dv)
    _call("kda_verify_rollback" + sfx, y,
        _ptr(q_raw), _ptr(k_raw), _ptr(v_raw), _raw_dtype(q_raw), _ptr(conv_w), _ptr(ring_in),
        _ptr(ring_out), _ptr(f_raw), _ptr(dt_bias), _ptr(a_log), gate_mode, gate_lb,
        _ptr(beta_raw), _ptr(state_in), _ptr(state_out), _ptr(norm_w), _ptr(gate_raw), _ptr(y),
        _ptr(keep), N, T, *heads, K, l2_eps, scale, rms_eps, st)


def kda_prefill_workspace_bytes(N, total_T, H, gate_mode=0, D=HEAD_DIM) -> int:
    return int(_lib.kda_prefill_workspace_bytes(N, total_T, H, D, gate_mode))


def prefill_workspace(N, total_T, H, device, gate_mode=0):
    """A device byte buffer large enough for kda_prefill_fused / kda_prefill_fused_varlen."""
    nbytes = kda_prefill_workspace_bytes(N, total_T, H, gate_mode)
    return torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)


def _ws_bytes(workspace):
    return 0 if workspace is None else workspace.numel() * workspace.element_size()


def kda_prefill_fused(q_raw, k_raw, v_raw, conv_w, ring_in, ring_out, f_raw, dt_bias, a_log,
                      beta_raw, state_in, state_out, norm_w, gate_raw, y, workspace, *, N, T, H,
                      K=4, gate_mode=0, gate_lb=-5.0, l2_eps=1e-6, scale=None, rms_eps=1e-6,
                      D=HEAD_DIM, stream=None, Hk=None, Dv=None):
    scale = D ** -0.5 if scale is None else scale
    st = _stream(stream, y)
    sfx, heads = _heads(H, Hk, D, Dv)
    _call("kda_prefill_fused" + sfx, y,
        _ptr(q_raw), _ptr(k_raw), _ptr(v_raw), _raw_dtype(q_raw), _ptr(conv_w), _ptr(ring_in),
        _ptr(ring_out), _ptr(f_raw), _ptr(dt_bias), _ptr(a_log), gate_mode, gate_lb,
        _ptr(beta_raw), _ptr(state_in), _ptr(state_out), _ptr(norm_w), _ptr(gate_raw), _ptr(y),
        N, T, *heads, K, l2_eps, scale, rms_eps, _ptr(workspace), _ws_bytes(workspace), st)


def kda_prefill_fused_varlen(q_raw, k_raw, v_raw, conv_w, ring_in, ring_out, f_raw, dt_bias,
                             a_log, beta_raw, state_in, state_out, norm_w, gate_raw, y,
                             workspace, cu_seqlens, cu_seqlens_host, *, H, K=4, gate_mode=0,
                             gate_lb=-5.0, l2_eps=1e-6, scale=None, rms_eps=1e-6, D=HEAD_DIM,
                             stream=None, Hk=None, Dv=None):
    N = cu_seqlens_host.numel() - 1
    total = int(cu_seqlens_host[-1])
    scale = D ** -0.5 if scale is None else scale
    st = _stream(stream, y)
    sfx, heads = _heads(H, Hk, D, Dv)
    _call("kda_prefill_fused_varlen" + sfx, y,
        _ptr(q_raw), _ptr(k_raw), _ptr(v_raw), _raw_dtype(q_raw), _ptr(conv_w), _ptr(ring_in),
        _ptr(ring_out), _ptr(f_raw), _ptr(dt_bias), _ptr(a_log), gate_mode, gate_lb,
        _ptr(beta_raw), _ptr(state_in), _ptr(state_out), _ptr(norm_w), _ptr(gate_raw), _ptr(y),
        _ptr(cu_seqlens), _ptr(cu_seqlens_host), N, total, *heads, K, l2_eps, scale, rms_eps,
        _ptr(workspace), _ws_bytes(workspace), st)


PROJ_MAX_T = 256


def kda_proj6_workspace_bytes(t, in_f) -> int:
    return int(_lib.kda_proj6_workspace_bytes(t, in_f))


def proj6_workspace(t, in_f, device):
    """A device byte buffer large enough for kda_proj6 over t token rows of width in_f."""
    return torch.empty(max(kda_proj6_workspace_bytes(t, in_f), 16), dtype=torch.uint8,
                       device=device)


def kda_proj6(x, w_q, w_k, w_v, w_fa, w_ga, w_b, q_raw, k_raw, v_raw, f_down, g_down, beta_raw,
              workspace, *, H, D=HEAD_DIM, stream=None):
    """The six projections of x [t, in_f] (f32) by bf16 weights into f32 outputs."""
    t, in_f = x.shape
    st = _stream(stream, q_raw)
    _call("kda_proj6", q_raw,
          _ptr(x), t, in_f, _ptr(w_q), _ptr(w_k), _ptr(w_v), _ptr(w_fa), _ptr(w_ga), _ptr(w_b),
          _ptr(q_raw), _ptr(k_raw), _ptr(v_raw), _ptr(f_down), _ptr(g_down), _ptr(beta_raw), H, D,
          _ptr(workspace), _ws_bytes(workspace), st)


def kernel_timing(enable: bool) -> bool:
    """Turn per-kernel event timing on (clearing the totals) or off; returns the old setting."""
    return bool(_lib.kda_kernel_timing(1 if enable else 0))


def kernel_times() -> dict:
    """{kernel name: (launches, total ms)} since the last read, for kernels launched at least once
    (waits for the recorded launches)."""
    n = 16
    launches = (ctypes.c_long * n)()
    ms = (ctypes.c_double * n)()
    k = _lib.kda_kernel_times(n, launches, ms)
    if k < 0:
        raise KdaError("kda_kernel_times", -k)
    out = {}
    for i in range(min(k, n)):
        if launches[i]:
            out[_lib.kda_kernel_name(i).decode()] = (int(launches[i]), float(ms[i]))
    return out


def kda_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error word status."""
    if stream is None and torch.cuda.is_available():
        stream = torch.cuda.current_stream().cuda_stream
    elif stream is not None and not isinstance(stream, int):
        stream = stream.cuda_stream
    return int(_lib.kda_device_status(stream))


def kda_selftest_wait_timeout(stream=None):
    """Launch the bounded-wait self-test (a wait that nothing completes gives up after about a
    second); a following kda_device_status() returns 40008."""
    if stream is None and torch.cuda.is_available():
        stream = torch.cuda.current_stream().cuda_stream
    elif stream is not None and not isinstance(stream, int):
        stream = stream.cuda_stream
    _check("kda_selftest_wait_timeout", _lib.kda_selftest_wait_timeout(stream))
