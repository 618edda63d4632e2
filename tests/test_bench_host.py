"""Host checks of the benchmark's bookkeeping (no GPU): the algorithmic bytes behind each
roofline fraction equal the per-unit figures of the prefill workload worked out by hand (T = 4096
tokens, H = 64 heads, D = 128, conv K = 4, 128 chunks of 32 tokens, 70,144-byte workspace
blocks), and every kernel the benchmark reports has its source list on disk."""

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


def test_prefill_kernel_bytes(bench):
    kb = bench._kernel_bytes(4096, 64, 70144, 128)
    MB = 1 << 20
    raw = 3 * 4096 * 8192 * 2               # 192 MiB of bf16 q, k, v
    plane = 4096 * 8192 * 4                 # 128 MiB per f32 [T, C] plane
    blocks = 128 * 64 * 70144               # the workspace: one block per (chunk, head)
    assert raw == 192 * MB and plane == 128 * MB and blocks == 574_619_648
    small = 4096 * 64 * 4 + 3 * 8192 * 4 * 4 + 3 * 8192 * 3 * 4   # beta in, conv weights, ring in
    assert kb["kda_chunk_prep_intra_kernel"] == raw + plane + small + blocks == 911_900_672
    ring = 3 * 8192 * 3 * (2 + 4 + 4)       # raw tail rows in, ring in, ring out
    assert kb["kda_chunk_inter_kernel"] == blocks + 2 * 64 * 128 * 128 * 4 + plane + ring
    assert kb["kda_gated_rmsnorm_kernel"] == 3 * plane + 128 * 4        # o, z in; y out; weight


def test_kernel_sources_exist(bench):
    csrc = os.path.join(ROOT, "gated_delta_rule_scan_gb300", "csrc")
    for kernel, files in bench.KERNEL_SOURCES.items():
        for f in files:
            assert os.path.exists(os.path.join(csrc, f)), (kernel, f)
