"""Seeded synthetic inputs for the KDA mixer, shared by the tests, the benchmark and the oracle's
callers.

This module draws random numbers and rounds them to the storage dtype; it holds none of the
method's arithmetic (no conv, norm, gate or scan).  Every workload is drawn from
``numpy.random.default_rng(seed)`` in one fixed order, so a (workload, seed) pair names one exact
set of tensors on every machine:

  1. lengths (varlen only)   integers in [lo, hi]
  2. q_raw, k_raw, v_raw     N(0, 1), [rows, C]            (rounded to bf16 when raw_dtype is bf16)
  3. conv_w                  N(0, 0.5^2), [3C, K]          (conv on)
  4. ring_in                 N(0, 1) or zero, [N, 3C, K-1] (conv on)
  5. f_raw                   N(0, 1), [rows, C] (KDA) or [rows, H] (GDN)
  6. dt_bias                 N(0, 0.5^2), [C] (KDA) or [H] (GDN)
  7. a_log                   log U[1, 16), [H]
  8. beta_raw                N(0, 1), [rows, H]
  9. state_in                N(0, 0.02^2) or zero, [N, H, D, D]
 10. norm_w                  1 + N(0, 0.1^2), [D]          (epilogue on)
 11. gate_raw (z)            N(0, 1), [rows, C]            (epilogue on)
 12. split points            integers in [1, L-1] per sequence (varlen only)

A value head width Dv (a multiple of D) widens the v plane, its conv/ring rows, gate_raw and norm_w
to Dv per head and the state to [N, H, Dv, D]; the gate stays D (the key dim) per head.  With Dv = D
the draws are the ones above, value for value.

Tensors come back as CPU torch tensors (f32, or bf16 for the raw q/k/v planes when asked);
callers move them to the device themselves.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

D_HEAD = 128
CONV_K = 4


@dataclass
class KdaInputs:
    N: int
    H: int
    D: int
    K: int
    cu_seqlens: np.ndarray            # int64 [N+1]
    q_raw: torch.Tensor
    k_raw: torch.Tensor
    v_raw: torch.Tensor
    conv_w: torch.Tensor | None
    ring_in: torch.Tensor | None
    f_raw: torch.Tensor
    dt_bias: torch.Tensor
    a_log: torch.Tensor
    beta_raw: torch.Tensor
    state_in: torch.Tensor
    norm_w: torch.Tensor | None
    gate_raw: torch.Tensor | None
    gate_mode: int                    # 0 = per-channel (KDA), 1 = per-head (GDN)
    split_points: np.ndarray | None = None
    meta: dict = field(default_factory=dict)
    Hk: int | None = None             # grouped queries: q/k planes of Hk heads (None: H)
    Dv: int | None = None             # value head width (None: D)

    @property
    def rows(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def C(self) -> int:
        return self.H * (self.D if self.Dv is None else self.Dv)

    @property
    def uniform_T(self) -> int | None:
        """T when every sequence has the same length, else None."""
        L = np.diff(self.cu_seqlens)
        return int(L[0]) if L.size and np.all(L == L[0]) else None


def _normal(rng, shape, std=1.0):
    x = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return torch.from_numpy(x)


def make_inputs(seed: int, *, H: int, N: int = 1, T: int | None = None,
                lengths: tuple[int, int] | None = None, D: int = D_HEAD, K: int = CONV_K,
                raw_dtype: str = "f32", conv: bool = True, ring: str = "zero",
                gate_mode: int = 0, state: str = "zero", epilogue: bool = True,
                split: bool = False, Hk: int | None = None,
                Dv: int | None = None) -> KdaInputs:
    """Draw one workload.  Exactly one of ``T`` (N sequences of T tokens) and ``lengths``
    (N sequence lengths drawn uniformly from [lo, hi], packed with cu_seqlens) is given.
    ``Hk``: grouped queries -- the q and k planes (and their conv weight and ring rows) hold Hk
    heads, v and everything per value head H.  ``Dv``: value heads Dv wide (q/k stay D)."""
    rng = np.random.default_rng(seed)
    Cg = H * D                                  # per-channel gate: the key dim of each value head
    C = H * (D if Dv is None else Dv)           # the v plane, gate_raw, y
    Cq = Cg if Hk is None else Hk * D
    if lengths is not None:
        L = rng.integers(lengths[0], lengths[1], size=N, endpoint=True).astype(np.int64)
    else:
        L = np.full(N, int(T), dtype=np.int64)
    cu = np.zeros(N + 1, dtype=np.int64)
    cu[1:] = np.cumsum(L)
    rows = int(cu[-1])

    planes = [_normal(rng, (rows, w)) for w in (Cq, Cq, C)]
    if raw_dtype == "bf16":
        planes = [p.to(torch.bfloat16) for p in planes]
    elif raw_dtype != "f32":
        raise ValueError(raw_dtype)
    conv_w = ring_in = None
    if conv:
        conv_w = _normal(rng, (2 * Cq + C, K), 0.5)
        ring_in = (_normal(rng, (N, 2 * Cq + C, K - 1)) if ring == "randn"
                   else torch.zeros(N, 2 * Cq + C, K - 1))
    if gate_mode == 0:
        f_raw = _normal(rng, (rows, Cg))
        dt_bias = _normal(rng, (Cg,), 0.5)
    else:
        f_raw = _normal(rng, (rows, H))
        dt_bias = _normal(rng, (H,), 0.5)
    a_log = torch.from_numpy(np.log(rng.uniform(1.0, 16.0, size=H)).astype(np.float32))
    beta_raw = _normal(rng, (rows, H))
    Dvw = D if Dv is None else Dv
    state_in = (_normal(rng, (N, H, Dvw, D), 0.02) if state == "randn"
                else torch.zeros(N, H, Dvw, D))
    norm_w = gate_raw = None
    if epilogue:
        norm_w = 1.0 + _normal(rng, (Dvw,), 0.1)
        gate_raw = _normal(rng, (rows, C))
    splits = None
    if split:
        splits = np.array([rng.integers(1, max(int(l) - 1, 1), endpoint=True) for l in L],
                          dtype=np.int64)
    return KdaInputs(N=N, H=H, D=D, K=K, cu_seqlens=cu, q_raw=planes[0], k_raw=planes[1],
                     v_raw=planes[2], conv_w=conv_w, ring_in=ring_in, f_raw=f_raw,
                     dt_bias=dt_bias, a_log=a_log, beta_raw=beta_raw, state_in=state_in,
                     norm_w=norm_w, gate_raw=gate_raw, gate_mode=gate_mode, split_points=splits,
                     meta=dict(seed=seed, raw_dtype=raw_dtype), Hk=Hk, Dv=Dv)


# ------------------------------------------------------------------------------------------
# the five named workloads (shapes and distributions of the pages' geometry: 64 heads x 128)
# ------------------------------------------------------------------------------------------

def tiny_scan(T: int = 64, H: int = 4, seed: int = 0) -> KdaInputs:
    """Tiny KDA scan: 1 sequence, T=64, H=4, f32 raw q/k/v (no conv), zero state."""
    return make_inputs(seed, H=H, N=1, T=T, raw_dtype="f32", conv=False, gate_mode=0,
                       state="zero", epilogue=False)


def decode_step(N: int = 64, T: int = 1, H: int = 64, seed: int = 1) -> KdaInputs:
    """Decode (T=1) or multi-token verify (T>1): N sequences with random states and rings,
    bf16 raw q/k/v, conv + gated-RMSNorm epilogue."""
    return make_inputs(seed, H=H, N=N, T=T, raw_dtype="bf16", conv=True, ring="randn",
                       gate_mode=0, state="randn", epilogue=True)


def prefill(T: int = 4096, H: int = 64, seed: int = 2) -> KdaInputs:
    """Single-sequence prefill from a zero state and zero ring, full fused path."""
    return make_inputs(seed, H=H, N=1, T=T, raw_dtype="bf16", conv=True, ring="zero",
                       gate_mode=0, state="zero", epilogue=True)


def varlen_prefill(N: int = 16, lo: int = 256, hi: int = 8192, H: int = 64,
                   seed: int = 3) -> KdaInputs:
    """Packed varlen prefill: N sequences with lengths U[lo, hi], random states and rings, and a
    random split point per sequence for the state-carry check."""
    return make_inputs(seed, H=H, N=N, lengths=(lo, hi), raw_dtype="bf16", conv=True,
                       ring="randn", gate_mode=0, state="randn", epilogue=True, split=True)


def gdn_long(T: int = 16384, H: int = 32, seed: int = 4) -> KdaInputs:
    """Gated DeltaNet special case: per-(token, head) scalar gate, f32 raw q/k/v, no conv."""
    return make_inputs(seed, H=H, N=1, T=T, raw_dtype="f32", conv=False, gate_mode=1,
                       state="zero", epilogue=False)
