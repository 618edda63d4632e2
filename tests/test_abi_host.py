"""Host-side checks of the C ABI (no GPU): the library loads, exports every entry point that
include/kda.h declares, and rejects contract violations before touching the device."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kda():
    from gated_delta_rule_scan_gb300 import _build
    _build.build()
    from gated_delta_rule_scan_gb300 import kda as mod
    return mod


def _declared():
    text = open(os.path.join(ROOT, "include", "kda.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(kda):
    names = _declared()
    assert len(names) >= 10
    for n in names:
        assert hasattr(kda.library(), n), n
    assert sorted(kda.EXPORTED) == names


def test_status_strings(kda):
    assert kda.abi_version() == 1
    for code in (0, 40001, 40002, 40003, 40004, 40005, 40006, 40007, 40008, 40009, 40010, 40011,
                 40012):
        assert kda.status_string(code) not in ("unknown status",)
    assert kda.status_string(10000 + 2) == "CUDA error"


# The calls below carry fake (never dereferenced) pointers; every one violates a contract that
# is checked on the host before any CUDA call, so none reaches the device.
FAKE = 0x10000  # 16-byte aligned dummy address


def test_scan_contract(kda):
    lib = kda.library()
    args = [FAKE] * 4 + [0, FAKE, FAKE, FAKE * 2, FAKE * 3]

    def scan(**kw):
        a = dict(N=1, T=4, H=2, D=128, scale=1.0, algo=1, gate_mode=0)
        a.update(kw)
        base = list(args)
        base[4] = a["gate_mode"]
        return lib.kda_scan(*base, a["N"], a["T"], a["H"], a["D"], ctypes.c_float(a["scale"]),
                            a["algo"], None, 0, None)
    assert scan(D=64) == 40001
    assert scan(H=0) == 40005
    assert scan(N=-1) == 40005
    assert scan(T=-3) == 40005
    assert scan(gate_mode=4) == 40007
    assert scan(algo=7) == 40007
    # state_in == state_out
    a2 = [FAKE] * 4 + [0, FAKE, FAKE, FAKE, FAKE]
    assert lib.kda_scan(*a2, 1, 4, 2, 128, ctypes.c_float(1.0), 1, None, 0, None) == 40003
    # misaligned state
    a3 = [FAKE] * 4 + [0, FAKE, FAKE + 4, FAKE * 8, FAKE]
    assert lib.kda_scan(*a3, 1, 4, 2, 128, ctypes.c_float(1.0), 1, None, 0, None) == 40010
    # null inputs with tokens present
    a4 = [None] * 4 + [0, None, FAKE, FAKE * 8, None]
    assert lib.kda_scan(*a4, 1, 4, 2, 128, ctypes.c_float(1.0), 1, None, 0, None) == 40004


def test_varlen_cu_seqlens_contract(kda):
    lib = kda.library()
    a = [FAKE] * 4 + [0, FAKE, FAKE, FAKE * 8, FAKE]
    for cu, total in (([1, 3, 5], 5), ([0, 3, 2], 2), ([0, 3, 5], 6)):
        arr = (ctypes.c_int * len(cu))(*cu)
        rc = lib.kda_scan_varlen(*a, FAKE, ctypes.cast(arr, ctypes.c_void_p), len(cu) - 1, total,
                                 2, 128, ctypes.c_float(1.0), 1, None, 0, None)
        assert rc == 40006, (cu, rc)
    rc = lib.kda_scan_varlen(*a, None, None, 2, 5, 2, 128, ctypes.c_float(1.0), 1, None, 0, None)
    assert rc == 40004


def test_prep_and_decode_contract(kda):
    lib = kda.library()
    F = ctypes.c_float
    prep = lambda **kw: lib.kda_conv_l2norm_prep(  # noqa: E731
        FAKE, FAKE, FAKE, kw.get("dtype", 1), FAKE, FAKE, FAKE * 2, FAKE, FAKE, FAKE,
        kw.get("gm", 0), F(-5.0), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 2, kw.get("D", 128),
        kw.get("K", 4), F(1e-6), None)
    assert prep(D=96) == 40001
    assert prep(K=1) == 40002
    assert prep(K=9) == 40002
    assert prep(dtype=5) == 40007
    assert prep(gm=4) == 40007
    dec = lambda **kw: lib.kda_decode_fused(  # noqa: E731
        FAKE, FAKE, FAKE, 1, FAKE, FAKE, FAKE * 2, FAKE, FAKE, FAKE, 0, F(-5.0), FAKE, FAKE,
        FAKE * 64, FAKE, FAKE, FAKE, 2, kw.get("T", 1), 2, 128, kw.get("K", 4), F(1e-6), F(0.1),
        F(1e-6), None)
    assert dec(T=0) == 40005
    assert dec(T=17) == 40005
    assert dec(K=12) == 40002
    rb = lambda keep, **kw: lib.kda_verify_rollback(  # noqa: E731
        FAKE, FAKE, FAKE, 1, FAKE, FAKE, FAKE * 2, FAKE, FAKE, FAKE, 0, F(-5.0), FAKE, FAKE,
        FAKE * 64, FAKE, FAKE, FAKE, keep, 2, kw.get("T", 4), 2, 128, 4, F(1e-6), F(0.1),
        F(1e-6), None)
    assert rb(None) == 40004                 # keep is required
    # in place is fine for decode (it launches, so only a partial overlap is checked here)
    partial = lib.kda_decode_fused(
        FAKE, FAKE, FAKE, 1, FAKE, FAKE, FAKE * 2, FAKE, FAKE, FAKE, 0, F(-5.0), FAKE, FAKE * 64,
        FAKE * 64 + 16, FAKE, FAKE, FAKE, 2, 1, 2, 128, 4, F(1e-6), F(0.1), F(1e-6), None)
    assert partial == 40003
    assert rb(FAKE, T=17) == 40005
    assert rb(FAKE, T=0) == 40005
    norm = lib.kda_gated_rmsnorm_out(FAKE, FAKE + 8, FAKE, FAKE, ctypes.c_long(4), 128, F(1e-6),
                                     None)
    assert norm == 40010


def test_prefill_contract(kda):
    """kda_prefill_fused takes bf16 raw rows only at 16-byte alignment (the staged prep accepts
    8), and refuses the decay-factor gate flag, before any device call."""
    lib = kda.library()
    F = ctypes.c_float

    def call(q=FAKE, gm=0, dtype=1):
        return lib.kda_prefill_fused(q, FAKE, FAKE, dtype, FAKE, FAKE, FAKE * 2, FAKE, FAKE, FAKE,
                                     gm, F(-5.0), FAKE, FAKE, FAKE * 4, FAKE, FAKE, FAKE, 1, 64, 2,
                                     128, 4, F(1e-6), F(0.1), F(1e-6), FAKE, 0, None)
    assert call(q=FAKE + 8) == 40010
    assert call(q=FAKE + 8, dtype=0) == 40010
    assert call(gm=2) == 40007
    assert call() == 40009          # aligned and valid up to the (zero-byte) workspace


def test_static_scan_contract(kda):
    """kda_scan_varlen_static refuses, before any device call, a problem whose chunked scratch
    exceeds KDA_STATIC_SCRATCH_BYTES, besides kda_scan_varlen's own contract."""
    lib = kda.library()
    a = [FAKE] * 4 + [0, FAKE, FAKE, FAKE * 8, FAKE]
    per_block = kda.chunk_block_bytes()
    assert per_block == 43520
    cap_blocks = (kda.STATIC_SCRATCH_BYTES - 256) // per_block

    def call(cu, H, D=128):
        arr = (ctypes.c_int * len(cu))(*cu)
        return lib.kda_scan_varlen_static(*a, FAKE, ctypes.cast(arr, ctypes.c_void_p),
                                          len(cu) - 1, cu[-1], H, D, ctypes.c_float(1.0), None)
    assert call([0, 32 * (cap_blocks + 1)], 1) == 40011
    # exactly the cap (ragged tail) passes the size check; with no device the call then stops
    # at its first CUDA query, never with the limit's code
    assert call([0, 32 * cap_blocks - 5], 1) not in (0, 40011)
    assert call([0, 32 * (cap_blocks // 2 + 1) - 5, 32 * (cap_blocks + 2) - 10], 2) == 40011
    assert call([0, 3, 2], 1) == 40006
    assert call([0, 64], 1, D=64) == 40001
    assert call([0, 64], 0) == 40005
    assert kda.status_string(40011) != "unknown status"


def test_kernel_timer_host(kda):
    """The timing switch and the read work without a device: nothing pending reads as zeros."""
    lib = kda.library()
    assert kda.kernel_timing(True) in (False, True)
    assert kda.kernel_times() == {}
    assert kda.kernel_timing(False) is True
    n = lib.kda_kernel_times(0, None, None)
    assert n >= 8
    names = [lib.kda_kernel_name(i).decode() for i in range(n)]
    assert "kda_chunk_inter_kernel" in names and "kda_prep_kernel" in names
    assert lib.kda_kernel_name(n) is None and lib.kda_kernel_name(-1) is None


def test_proj6_contract(kda):
    """kda_proj6 refuses bad shapes, null or misaligned pointers and a short workspace on the host,
    before any device call."""
    lib = kda.library()
    ws_need = kda.kda_proj6_workspace_bytes(3, 256)
    assert ws_need == 2 * 16 * 256 * 2               # hi and lo images of 16 padded rows
    assert kda.kda_proj6_workspace_bytes(0, 256) == 0
    assert kda.kda_proj6_workspace_bytes(257, 256) == 0
    assert kda.kda_proj6_workspace_bytes(4, 100) == 0

    def call(x=FAKE, t=3, in_f=256, w0=FAKE, H=2, D=128, ws=FAKE, wsb=None):
        return lib.kda_proj6(x, t, in_f, w0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                             FAKE, FAKE, H, D, ws, ws_need if wsb is None else wsb, None)
    assert call(D=64) == 40001
    assert call(t=0) == 40005
    assert call(t=257) == 40005
    assert call(in_f=100) == 40005
    assert call(H=0) == 40005
    assert call(x=None) == 40004
    assert call(w0=None) == 40004
    assert call(w0=FAKE + 8) == 40010
    assert call(x=FAKE + 4) == 40010
    assert call(wsb=ws_need - 1) == 40009
    assert call(ws=None) == 40009


def test_value_width_contract(kda):
    """The value-width entries take Dk = 128 and Dv = 128 * m (m = 1..8), 1 <= Hk <= H."""
    lib = kda.library()
    F = ctypes.c_float
    scan = lambda **kw: lib.kda_scan_dv(  # noqa: E731
        FAKE, FAKE, FAKE, FAKE, 0, FAKE, FAKE, FAKE * 8, FAKE, 1, 4, kw.get("H", 2),
        kw.get("Hk", 1), kw.get("Dk", 128), kw.get("Dv", 256), F(0.1), 1, None, 0, None)
    for dv in (0, 64, 192, 1152, -128):
        assert scan(Dv=dv) == 40001, dv
    assert scan(Dk=64) == 40001
    assert scan(Hk=3) == 40005
    assert scan(Hk=0) == 40005
    assert scan(H=0) == 40005
    prep = lambda **kw: lib.kda_conv_l2norm_prep_dv(  # noqa: E731
        FAKE, FAKE, FAKE, 1, FAKE, FAKE, FAKE * 2, FAKE, FAKE, FAKE, 0, F(-5.0), FAKE, FAKE, FAKE,
        FAKE, FAKE, FAKE, 1, 4, 2, kw.get("Hk", 2), 128, kw.get("Dv", 256), kw.get("K", 4),
        F(1e-6), None)
    assert prep(Dv=320) == 40001
    assert prep(Hk=5) == 40005
    assert prep(K=1) == 40002
    cu = (ctypes.c_int * 3)(0, 3, 2)
    rc = lib.kda_scan_varlen_dv(FAKE, FAKE, FAKE, FAKE, 0, FAKE, FAKE, FAKE * 8, FAKE, FAKE,
                                ctypes.cast(cu, ctypes.c_void_p), 2, 2, 2, 2, 128, 256, F(0.1), 1,
                                None, 0, None)
    assert rc == 40006
    for d in (192, 1152, 0):
        norm = lib.kda_gated_rmsnorm_out(FAKE, FAKE, FAKE, FAKE, ctypes.c_long(4), d, F(1e-6),
                                         None)
        assert norm == 40001, d


def test_value_width_fused_contract(kda):
    """The fused value-width entries check Dk, Dv and Hk on the host."""
    lib = kda.library()
    F = ctypes.c_float
    pre = lambda **kw: lib.kda_prefill_fused_dv(  # noqa: E731
        FAKE, FAKE, FAKE, 1, FAKE, FAKE, FAKE * 2, FAKE, FAKE, FAKE, 0, F(-5.0), FAKE, FAKE,
        FAKE * 64, FAKE, FAKE, FAKE, 1, 4, 2, kw.get("Hk", 1), kw.get("Dk", 128),
        kw.get("Dv", 256), 4, F(1e-6), F(0.1), F(1e-6), None, 0, None)
    assert pre(Dv=192) == 40001
    assert pre(Dk=256) == 40001
    assert pre(Hk=3) == 40005
    dec = lambda **kw: lib.kda_decode_fused_dv(  # noqa: E731
        FAKE, FAKE, FAKE, 1, FAKE, FAKE, FAKE * 2, FAKE, FAKE, FAKE, 0, F(-5.0), FAKE, FAKE,
        FAKE * 64, FAKE, FAKE, FAKE, 2, kw.get("T", 1), 2, kw.get("Hk", 1), 128,
        kw.get("Dv", 256), 4, F(1e-6), F(0.1), F(1e-6), None)
    assert dec(Dv=2048) == 40001
    assert dec(Hk=0) == 40005
    assert dec(T=17) == 40005
    rb = lib.kda_verify_rollback_dv(
        FAKE, FAKE, FAKE, 1, FAKE, FAKE, FAKE * 2, FAKE, FAKE, FAKE, 0, F(-5.0), FAKE, FAKE,
        FAKE * 64, FAKE, FAKE, FAKE, None, 2, 4, 2, 1, 128, 256, 4, F(1e-6), F(0.1), F(1e-6),
        None)
    assert rb == 40004                       # keep is required
