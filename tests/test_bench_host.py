"""Host checks of the benchmark's bookkeeping (no GPU): the method bytes behind each roofline
fraction equal the per-unit figures of the prefill workload worked out by hand (T = 4096 tokens,
H = 64 heads, D = 128, conv K = 4), the library's intermediate traffic (128 chunks of 32 tokens,
43,520-byte workspace blocks) is counted apart from them, and every kernel the benchmark reports
has its source list on disk."""

import importlib.util
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    sys.argv = ["bench.py"]
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_prefill_method_bytes(bench):
    """The method's own I/O per prefill step, attributed to the fused kernels, adds up to the
    step's inputs read once and outputs written once; no workspace byte is counted in it."""
    mb = bench._method_bytes(4096, 64)
    MB = 1 << 20
    raw = 3 * 4096 * 8192 * 2               # 192 MiB of bf16 q, k, v
    plane = 4096 * 8192 * 4                 # 128 MiB per f32 [T, C] plane (f, z, y)
    assert raw == 192 * MB and plane == 128 * MB
    beta = 4096 * 64 * 4
    conv = 3 * 8192 * 4 * 4
    ring = 3 * 8192 * 3 * 4                 # one direction
    state = 64 * 128 * 128 * 4              # one direction
    params = 8192 * 4 + 64 * 4 + 128 * 4    # dt_bias, A_log, norm weight
    assert mb["kda_chunk_prep_intra_kernel"] == raw + plane + beta + conv + ring + 8192 * 4 + 64 * 4
    # the fused prefill's inter kernel writes y itself: z, the norm weight and y are its bytes
    assert mb["kda_chunk_inter_kernel"] == 2 * state + ring + 2 * plane + 128 * 4
    step = mb["kda_chunk_prep_intra_kernel"] + mb["kda_chunk_inter_kernel"]
    assert step == raw + 3 * plane + beta + conv + 2 * ring + 2 * state + params == 614_433_536
    # with the RMSNorm as a kernel of its own, the same total split three ways
    mu = bench._method_bytes(4096, 64, norm_folded=False)
    assert mu["kda_chunk_inter_kernel"] == 2 * state + ring
    assert mu["kda_gated_rmsnorm_kernel"] == 2 * plane + 128 * 4
    assert sum(mu[k] for k in ("kda_chunk_prep_intra_kernel", "kda_chunk_inter_kernel",
                               "kda_gated_rmsnorm_kernel")) == step


def test_prefill_impl_bytes(bench):
    """The library's own intermediates, reported apart: the chunk workspace (one 43,520-byte
    block per (32-token chunk, head)), and the readout plane o only where the RMSNorm runs as a
    kernel of its own."""
    ib = bench._impl_bytes(4096, 64, 43520, 128)
    blocks = 128 * 64 * 43520
    plane = 4096 * 8192 * 4
    assert blocks == 356_515_840
    assert ib["kda_chunk_prep_intra_kernel"] == blocks
    assert ib["kda_chunk_inter_kernel"] == blocks
    iu = bench._impl_bytes(4096, 64, 43520, 128, norm_folded=False)
    assert iu["kda_chunk_inter_kernel"] == blocks + plane
    assert iu["kda_gated_rmsnorm_kernel"] == plane


def test_chunk_flops(bench):
    """The chunked form's tensor-core products per (32-token chunk, head), one pass each."""
    f = bench._chunk_flops(4096, 64)
    per = 128 * 64
    assert f["kda_chunk_prep_intra_kernel"] == per * (2 * 64 * 128 * 32 + 2 * 32 * 32 * 256)
    assert f["kda_chunk_inter_kernel"] == per * (2 * 128 * 128 * 64 + 2 * 128 * 32 * 160)


def test_kernel_sources_exist(bench):
    csrc = os.path.join(ROOT, "gated_delta_rule_scan_gb300", "csrc")
    for kernel, files in bench.KERNEL_SOURCES.items():
        for f in files:
            assert os.path.exists(os.path.join(csrc, f)), (kernel, f)
