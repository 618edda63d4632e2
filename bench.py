"""Benchmark of the KDA mixer on one GB300 (or N replicas, one per GPU).

One step = one pass of the whole mixer (conv+SiLU, ring roll, l2 norm, gates, scan, gated
RMSNorm) over the prefill workload: 1 sequence x 4096 tokens, 64 heads x 128, bf16 projected
q/k/v channels, zero initial state and ring (seeded synthetic data).  The same run also measures
the decode step: 64 sequences x 1 token, 64 heads, random states (4 MiB each), through the fused
decode kernel, state buffers ping-ponged between steps.

Printed JSON line (rank 0):
  value       prefill tokens/s, all ranks, inputs resident in HBM, CUDA events
  e2e         the same through the public API with inputs copied from pinned host memory and the
              result (y, final state, ring) read back every step
  roofline    the step's dominant kernel (by device time, from the library's per-kernel CUDA-event
              timer over the timed region) against measured HBM bandwidth, with its
              algorithmic bytes per launch; "kernels" lists every kernel the same way.  With
              --scan-algo seq (the staged sequential path) the scan against the FP32-pipe peak.
  decode      decode state GB/s, total GB/s and its roofline against measured HBM bandwidth
  cpu_baseline  the f64 oracle on a bounded sample of the prefill workload, host cores
--impl reference times that oracle alone as the reference arm.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KDA prefill tokens/s (H=64,d=128); decode state HBM GB/s vs peak"
D = 128
PREFILL_T, PREFILL_H = 4096, 64
RB_T = 4                         # verify width of the rollback workload
VER_T = 4                        # tokens per sequence of the verify leg
PROJ_HIDDEN = 6144               # layer width of the projection leg (synthetic weights; the pages
                                 # do not state it, 6144 is a multiple of 128 as they require)
DEC_N, DEC_H = 64, 64
FLOP_PER_TOKEN_HEAD = 7 * D * D   # decay D^2 + S^T k 2D^2 + rank-1 update 2D^2 + S^T q 2D^2
FP32_LANES, SM_MAX_MHZ = 128, 2070.0


def _peaks():
    """Roofline denominators: the measured copy bandwidth and bf16 GEMM rates of this machine's
    GB300s when MEASURED_PEAKS.json is present, else the recipe's fallback figures."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm_gbs=float(d["hbm_gbs"]), src="measured",
                    bf16_tflops=float(d.get("bf16_tflops", 1900.0)),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", 1700.0)),
                    sm_max_mhz=float(d.get("sm_max_mhz", SM_MAX_MHZ)))
    return dict(hbm_gbs=6800.0, src="fallback", bf16_tflops=1900.0,
                bf16_tflops_sustained=1700.0, sm_max_mhz=SM_MAX_MHZ)


def _fp32_peak_tflops(sms, mhz):
    """FP32 FMA peak: SMs x 128 lanes x 2 flop x clock."""
    return sms * FP32_LANES * 2 * mhz * 1e6 / 1e12


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class Replicas:
    """The N > 1 plumbing: one process per GPU, each running an independent replica of the
    workload (the (sequence, head) units shard with no exchange step, so there is no data-path
    collective).  barrier() brackets the timed region (and synchronises the device);
    max_over_ranks() takes the slowest rank's time; whole_job() turns it into throughput over the
    units all ranks processed.  World size 1 needs no process group."""

    def __init__(self, ws, rank, device, backend="nccl"):
        import torch
        import torch.distributed as dist
        self.ws, self.rank, self.device = ws, rank, torch.device(device)
        self._dist = dist
        if ws > 1 and not dist.is_initialized():
            dist.init_process_group(backend)

    def barrier(self):
        import torch
        if self.ws > 1:
            self._dist.barrier()
        if self.device.type == "cuda":
            torch.cuda.synchronize(self.device)

    def max_over_ranks(self, x):
        import torch
        if self.ws == 1:
            return x
        t = torch.tensor([x], dtype=torch.float64, device=self.device)
        self._dist.all_reduce(t, op=self._dist.ReduceOp.MAX)
        return float(t.item())

    def whole_job(self, units_per_rank, ms):
        """Units per second over all ranks: every rank processed units_per_rank in at most ms."""
        return self.ws * units_per_rank / (ms / 1e3)

    def close(self):
        if self.ws > 1 and self._dist.is_initialized():
            self._dist.destroy_process_group()


# ------------------------------------------------------------------------------------------
# clocks
# ------------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.remove(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        load = [r for r in rows if (num(r[3]) or 0) > 200.0] or rows
        sm = [num(r[1]) for r in load if num(r[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in load for i in range(4)
                          if r[5 + i].lower() in ("active", "1", "yes")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": num(load[0][2]), "samples": len(rows),
                "samples_under_load": len(load), "reasons": reasons}


# ------------------------------------------------------------------------------------------
# our arm
# ------------------------------------------------------------------------------------------

def _kernel_hash(files):
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, "gated_delta_rule_scan_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


# the sources each kernel is built from: profiles/traffic.json holds DRAM traffic keyed by their
# hash, reported only while they are unchanged
KERNEL_SOURCES = {
    "kda_chunk_intra_kernel": ["kda_scan_chunk.cu", "kda_chunk_common.cuh", "kda_tc.cuh",
                               "kda_device.cuh", "kda_internal.h", "kda_ring.cuh"],
    "kda_chunk_prep_intra_kernel": ["kda_chunk_prep.cu", "kda_chunk_common.cuh", "kda_tc.cuh",
                                    "kda_device.cuh", "kda_internal.h"],
    "kda_chunk_inter_kernel": ["kda_scan_chunk.cu", "kda_chunk_common.cuh", "kda_tc.cuh",
                               "kda_device.cuh", "kda_internal.h", "kda_ring.cuh"],
    "kda_gated_rmsnorm_kernel": ["kda_epilogue.cu", "kda_device.cuh", "kda_internal.h"],
    "kda_prep_kernel": ["kda_prep.cu", "kda_device.cuh", "kda_internal.h", "kda_ring.cuh"],
    "kda_decode_fused_kernel": ["kda_decode.cu", "kda_scan_core.cuh", "kda_device.cuh",
                                "kda_internal.h"],
    "kda_scan_seq_kernel": ["kda_scan_seq.cu", "kda_scan_core.cuh", "kda_device.cuh",
                            "kda_internal.h"],
    "kda_proj6_kernel": ["kda_proj.cu", "kda_tc.cuh", "kda_device.cuh", "kda_internal.h"],
}


def _traffic(kernel, files):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel)
    if not d or d.get("source_hash") != _kernel_hash(files):
        return None
    return d.get("dram_bytes_per_launch")


def _method_bytes(T, H, K=4, norm_folded=True):
    """The method's own HBM bytes per prefill step (T tokens, H heads, one sequence, conv K taps,
    bf16 raw q/k/v), split by the kernel that moves them: every input read once, every output
    written once, no intermediate.  norm_folded: the fused prefill's inter kernel writes y itself
    (128-wide value heads, N * H at least two thirds of the SM count), so z, the norm weight and
    y are its bytes; otherwise, and on the staged path, they are the RMSNorm kernel's.  What the
    library writes and reads back between its own kernels (the chunk workspace, the readout
    plane o, the staged path's prepared planes) is implementation traffic, reported apart by
    _impl_bytes."""
    C = H * D
    f32, bf16 = 4, 2
    plane = T * C * f32
    raw = 3 * T * C * bf16
    small = C * f32 + H * f32                       # dt_bias, A_log
    conv = 3 * C * K * f32
    ring = 3 * C * (K - 1) * f32                    # one direction
    state = H * D * D * f32                         # one direction
    beta = T * H * f32
    norm = plane + D * f32                          # z read (y written: plane below)
    return {
        # fused path: raw q, k, v, f, beta, conv weights, ring in, gate parameters
        "kda_chunk_prep_intra_kernel": raw + plane + beta + conv + ring + small,
        # state in and out, the rolled ring out (and, folded, the RMSNorm's z and weight in, y out)
        "kda_chunk_inter_kernel": 2 * state + ring + (norm + plane if norm_folded else 0),
        # z and the norm weight in, y out
        "kda_gated_rmsnorm_kernel": norm + plane,
        # staged path: prep reads what the fused prep reads and writes the ring; the scan moves
        # the state (its q, k, v, g, beta in and o out are intermediates)
        "kda_prep_kernel": raw + plane + beta + conv + 2 * ring + small,
        "kda_ring_roll_kernel": 0,
        "kda_chunk_intra_kernel": 0,
        "kda_scan_seq_kernel": 2 * state,
        "kda_chunk_offsets_kernel": 0,
    }


def _impl_bytes(T, H, blk_bytes, chunks, K=4, norm_folded=True):
    """Intermediate bytes each kernel of the prefill step writes or reads back (not the method's
    I/O): the chunk workspace (one block per (chunk, head)), the readout plane o between the scan
    and the RMSNorm (none when the inter kernel writes y itself), and the staged path's prepared
    q, k, v, g, beta planes."""
    C = H * D
    plane = T * C * 4
    ws = chunks * H * blk_bytes
    prepared = 4 * plane + T * H * 4
    return {
        "kda_chunk_prep_intra_kernel": ws,
        "kda_chunk_inter_kernel": ws + (0 if norm_folded else plane),
        "kda_gated_rmsnorm_kernel": plane,
        "kda_prep_kernel": prepared,
        "kda_ring_roll_kernel": 3 * C * (K - 1) * (2 + 4 + 4),
        "kda_chunk_intra_kernel": prepared + ws,
        "kda_scan_seq_kernel": prepared + plane,
        "kda_chunk_offsets_kernel": 0,
    }


def _chunk_flops(T, H):
    """Products the chunked form's tensor cores compute per launch (one pass, i.e. before the
    operand splits: bf16 x3 in the intra-chunk products, f16 x2 in the state chain's), for
    32-token chunks: intra = A and Aqk ([K;Q] (64 x 128) times K^T) plus [W | U] = Tm times
    [beta K e^G | beta V] (32 x 32 x 256);
    inter = MMA-1 (S^T, 128 x 128, times 64 rows) plus MMA-2 (U'^T, 128 x 32, times 160 rows)."""
    chunks_h = (T + 31) // 32 * H
    intra = 2 * 64 * 128 * 32 + 2 * 32 * 32 * 256
    inter = 2 * 128 * 128 * 64 + 2 * 128 * 32 * 160
    return {"kda_chunk_prep_intra_kernel": chunks_h * intra,
            "kda_chunk_intra_kernel": chunks_h * intra,
            "kda_chunk_inter_kernel": chunks_h * inter}


def _prefill_e2e(args, d, buf, state_out, ring_out, stream, barrier, max_over_ranks, mixer,
                 algo, ws, T, H, C, workspace, fused, gate_mode):
    """Prefill through the public API with every step's inputs copied from pinned host memory and
    its y, final state and ring read back.  Fused path: mixer.HostPrefillStream, which overlaps
    one step's host->device copy, the previous step's prefill and the device->host copy of the
    one before on three streams (weights resident).  Sequential path: one stream, in order."""
    import torch

    if fused:
        host_in = {k: d[k].cpu().pin_memory() for k in mixer.HostPrefillStream.BATCH_KEYS}
        host_out = dict(y=torch.empty(T, C, dtype=torch.float32).pin_memory(),
                        state_out=torch.empty_like(host_in["state_in"]).pin_memory(),
                        ring_out=torch.empty_like(host_in["ring_in"]).pin_memory())
        pipe = mixer.HostPrefillStream(like=host_in, conv_w=d["conv_w"], dt_bias=d["dt_bias"],
                                       a_log=d["a_log"], norm_w=d["norm_w"], H=H, N=1, T=T,
                                       gate_mode=gate_mode)
        h2d_bytes, d2h_bytes = pipe.h2d_bytes_per_batch, pipe.d2h_bytes_per_batch

        def e2e_step():
            pipe.submit(host_in, host_out)

        def e2e_start(ev):
            ev.record(pipe.copy_in)

        def e2e_stop(ev):
            pipe.record_done(ev)
    else:
        host = {k: v.cpu().pin_memory() for k, v in d.items() if v is not None}
        dev_in = {k: torch.empty_like(v) for k, v in d.items() if v is not None}
        y_host = torch.empty(T, C, dtype=torch.float32).pin_memory()
        st_host = torch.empty_like(d["state_in"], device="cpu").pin_memory()
        ring_host = torch.empty_like(d["ring_in"], device="cpu").pin_memory()
        h2d_bytes = sum(v.numel() * v.element_size() for v in host.values())
        d2h_bytes = sum(v.numel() * v.element_size() for v in (y_host, st_host, ring_host))

        def e2e_step():
            for k, v in host.items():
                dev_in[k].copy_(v, non_blocking=True)
            out = mixer.kda_forward(H=H, N=1, T=T, algo=algo, out=buf, state_out=state_out,
                                    ring_out=ring_out, workspace=workspace, **dev_in)
            y_host.copy_(out["y"], non_blocking=True)
            st_host.copy_(out["state_out"], non_blocking=True)
            ring_host.copy_(out["ring_out"], non_blocking=True)

        def e2e_start(ev):
            ev.record(stream)

        def e2e_stop(ev):
            ev.record(stream)

    for _ in range(max(3, args.warmup // 4)):
        e2e_step()
    barrier()
    # at least 20 steps and at least a second of timed work (the warm-up sets the estimate)
    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_start(w0)
    for _ in range(3):
        e2e_step()
    e2e_stop(w1)
    barrier()
    est_ms = max(w0.elapsed_time(w1) / 3, 1e-3)
    Ke = max(20, args.steps // 10, int(1000.0 / est_ms) + 1)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_start(e0)
    for _ in range(Ke):
        e2e_step()
    e2e_stop(e1)
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1)) / Ke
    out = {"value": ws * T / (e2e_ms / 1e3), "unit": "tokens/s", "ms_per_step": e2e_ms,  # all ranks
           "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes,
           "pipeline": ("three streams: copy-in, prefill, copy-out" if fused else "one stream")}
    if fused:
        # the host link alone: the same pinned inputs copied in, nothing else on the device
        for k in host_in:
            pipe.slots[0][0][k].copy_(host_in[k], non_blocking=True)
        barrier()
        l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        l0.record(stream)
        for _ in range(Ke):
            for k in host_in:
                pipe.slots[0][0][k].copy_(host_in[k], non_blocking=True)
        l1.record(stream)
        barrier()
        link_ms = max_over_ranks(l0.elapsed_time(l1)) / Ke
        out["link"] = {"h2d_gbs": h2d_bytes / (link_ms / 1e3) / 1e9,
                       "h2d_ms_per_step": link_ms,
                       "frac": link_ms / e2e_ms,
                       "note": "the step's host->device copy alone over the measured link; "
                               "frac = that time / the pipelined end-to-end step"}
    return out


def run_ours(args):
    import torch

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    rep = Replicas(ws, rank, dev)
    import __graft_entry__
    __graft_entry__.build()
    from gated_delta_rule_scan_gb300 import inputs, kda, mixer

    peaks = _peaks()
    stream = torch.cuda.current_stream()

    barrier, max_over_ranks = rep.barrier, rep.max_over_ranks

    # ---------------- prefill workload (resident) ----------------
    H, T = args.heads, PREFILL_T
    pre = inputs.prefill(T=T, H=H)
    C = H * D
    d = {k: (None if getattr(pre, k) is None else getattr(pre, k).to(dev)) for k in
         ("q_raw", "k_raw", "v_raw", "conv_w", "ring_in", "f_raw", "dt_bias", "a_log",
          "beta_raw", "state_in", "norm_w", "gate_raw")}
    f32 = lambda *s: torch.empty(*s, dtype=torch.float32, device=dev)  # noqa: E731
    buf = dict(q_hat=f32(T, C), k_hat=f32(T, C), v_hat=f32(T, C), g=f32(T, C), beta=f32(T, H),
               o=f32(T, C), y=f32(T, C))
    state_out = torch.empty_like(d["state_in"])
    ring_out = torch.empty_like(d["ring_in"])
    algo = {"auto": kda.ALGO_AUTO, "seq": kda.ALGO_SEQ, "chunk": kda.ALGO_CHUNK}[args.scan_algo]
    # auto / chunk: one kda_prefill_fused call per step (prep, chunked scan with the RMSNorm
    # epilogue); seq: the staged calls with the sequential scan
    fused = algo != kda.ALGO_SEQ
    # the sequential form consumes decay factors, the chunked form log-decays
    gate_mode = kda.GATE_PER_CHANNEL | (kda.GATE_EXP if algo == kda.ALGO_SEQ else 0)
    if fused:
        workspace = kda.prefill_workspace(1, T, H, dev)
    else:
        workspace = kda.scan_workspace(1, T, H, dev, algo)
    chunks = (T + 31) // 32
    blk_bytes = (kda.kda_scan_workspace_bytes(1, T, H, algo=kda.ALGO_CHUNK) - 256) // ((chunks + 1) * H)

    def prefill_step(timed_scan=None):
        if fused:
            kda.kda_prefill_fused(d["q_raw"], d["k_raw"], d["v_raw"], d["conv_w"], d["ring_in"],
                                  ring_out, d["f_raw"], d["dt_bias"], d["a_log"], d["beta_raw"],
                                  d["state_in"], state_out, d["norm_w"], d["gate_raw"], buf["y"],
                                  workspace, N=1, T=T, H=H)
            return
        kda.kda_conv_l2norm_prep(d["q_raw"], d["k_raw"], d["v_raw"], d["conv_w"], d["ring_in"],
                                 ring_out, d["f_raw"], d["dt_bias"], d["a_log"], d["beta_raw"],
                                 buf["q_hat"], buf["k_hat"], buf["v_hat"], buf["g"],
                                 buf["beta"], N=1, T=T, H=H, gate_mode=gate_mode)
        if timed_scan is not None:
            timed_scan[0].record(stream)
        kda.kda_scan(buf["q_hat"], buf["k_hat"], buf["v_hat"], buf["g"], buf["beta"],
                     d["state_in"], state_out, buf["o"], N=1, T=T, H=H, gate_mode=gate_mode,
                     algo=algo, workspace=workspace)
        if timed_scan is not None:
            timed_scan[1].record(stream)
        kda.kda_gated_rmsnorm_out(buf["o"], d["norm_w"], d["gate_raw"], buf["y"], rows=T * H)

    kda.kernel_timing(True)     # CUDA events around every library launch
    for _ in range(args.warmup):
        prefill_step()
    barrier()
    kda.kernel_times()          # drop the warm-up launches
    K = args.steps
    scan_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier()
        t0.record(stream)
        for i in range(K):
            prefill_step(None if fused else scan_ev[i])
        t1.record(stream)
        barrier()
    clocks = clk.summary()
    ktimes = kda.kernel_times()
    kda.kernel_timing(False)
    ms = max_over_ranks(t0.elapsed_time(t1))
    ms_step = ms / K
    tokens_per_s = rep.whole_job(T, ms_step)
    if fused:
        scan_ms = sum(ktimes[k][1] for k in ("kda_chunk_prep_intra_kernel", "kda_chunk_intra_kernel",
                                             "kda_chunk_inter_kernel", "kda_chunk_offsets_kernel")
                      if k in ktimes) / K
    else:
        scan_ms = statistics.mean(a.elapsed_time(b) for a, b in scan_ev)
    scan_flop = FLOP_PER_TOKEN_HEAD * T * H
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    fp32_peak = _fp32_peak_tflops(sms, peaks["sm_max_mhz"])
    scan_tflops = scan_flop / (scan_ms / 1e3) / 1e12
    assert kda.kda_device_status() == 0

    # ---------------- prefill end to end from pinned host memory ----------------
    e2e = None
    if not args.skip_e2e:
        e2e = _prefill_e2e(args, d, buf, state_out, ring_out, stream, barrier, max_over_ranks,
                           mixer, algo, ws, T, H, C, workspace, fused, gate_mode)

    # ---------------- decode step (fused kernel) ----------------
    dec = inputs.decode_step(N=DEC_N, T=1, H=DEC_H)
    dd = {k: getattr(dec, k).to(dev) for k in
          ("q_raw", "k_raw", "v_raw", "conv_w", "ring_in", "f_raw", "dt_bias", "a_log",
           "beta_raw", "state_in", "norm_w", "gate_raw")}
    states = [dd["state_in"], torch.empty_like(dd["state_in"])]
    ring = dd["ring_in"]
    y_dec = torch.empty(DEC_N, DEC_H * D, device=dev)

    def decode_step(i):
        kda.kda_decode_fused(dd["q_raw"], dd["k_raw"], dd["v_raw"], dd["conv_w"], ring, ring,
                             dd["f_raw"], dd["dt_bias"], dd["a_log"], dd["beta_raw"],
                             states[i & 1], states[(i + 1) & 1], dd["norm_w"], dd["gate_raw"],
                             y_dec, N=DEC_N, T=1, H=DEC_H)

    for i in range(max(args.warmup, 3)):
        decode_step(i)
    barrier()
    Kd = max(K, 10)
    d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    d0.record(stream)
    for i in range(Kd):
        decode_step(i)
    d1.record(stream)
    barrier()
    dec_ms = max_over_ranks(d0.elapsed_time(d1)) / Kd
    C1 = DEC_H * D
    state_bytes = DEC_N * DEC_H * D * D * 4 * 2
    per_seq = (DEC_H * D * D * 4 * 2 + 3 * C1 * 3 * 4 * 2 + 3 * C1 * 2 + C1 * 4 * 3 + DEC_H * 4)
    dec_bytes = DEC_N * per_seq + 3 * C1 * 4 * 4 + C1 * 4 + DEC_H * 4 + D * 4
    dec_gbs = dec_bytes / (dec_ms / 1e3) / 1e9
    assert kda.kda_device_status() == 0

    # the same step in place (state and ring), captured once in a CUDA graph and replayed
    g_state, g_ring = dd["state_in"].clone(), dd["ring_in"].clone()
    g_y = torch.empty_like(y_dec)

    def decode_in_place():
        kda.kda_decode_fused(dd["q_raw"], dd["k_raw"], dd["v_raw"], dd["conv_w"], g_ring, g_ring,
                             dd["f_raw"], dd["dt_bias"], dd["a_log"], dd["beta_raw"], g_state,
                             g_state, dd["norm_w"], dd["gate_raw"], g_y, N=DEC_N, T=1, H=DEC_H)

    decode_in_place()
    barrier()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        decode_in_place()
    for _ in range(max(args.warmup, 3)):
        graph.replay()
    barrier()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(Kd):
        graph.replay()
    g1.record(stream)
    barrier()
    dec_graph_ms = max_over_ranks(g0.elapsed_time(g1)) / Kd
    assert kda.kda_device_status() == 0

    # ---------------- 4-token verify of the decode batch (the same kernel, T = 4) -------------
    ver4 = inputs.decode_step(N=DEC_N, T=VER_T, H=DEC_H)
    dv4 = {k: getattr(ver4, k).to(dev) for k in
           ("q_raw", "k_raw", "v_raw", "conv_w", "ring_in", "f_raw", "dt_bias", "a_log",
            "beta_raw", "state_in", "norm_w", "gate_raw")}
    v_states = [dv4["state_in"], torch.empty_like(dv4["state_in"])]
    v_ring = dv4["ring_in"]
    y_ver = torch.empty(DEC_N * VER_T, DEC_H * D, device=dev)

    def verify_step(i):
        kda.kda_decode_fused(dv4["q_raw"], dv4["k_raw"], dv4["v_raw"], dv4["conv_w"], v_ring,
                             v_ring, dv4["f_raw"], dv4["dt_bias"], dv4["a_log"],
                             dv4["beta_raw"], v_states[i & 1], v_states[(i + 1) & 1],
                             dv4["norm_w"], dv4["gate_raw"], y_ver, N=DEC_N, T=VER_T, H=DEC_H)

    for i in range(max(args.warmup, 3)):
        verify_step(i)
    barrier()
    v0, v1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    v0.record(stream)
    for i in range(Kd):
        verify_step(i)
    v1.record(stream)
    barrier()
    ver_ms = max_over_ranks(v0.elapsed_time(v1)) / Kd
    # state and ring read + written once per call; per token raw q/k/v in, f, beta, z in, y out
    ver_bytes = (DEC_N * (DEC_H * D * D * 4 * 2 + 3 * C1 * 3 * 4 * 2)
                 + DEC_N * VER_T * (3 * C1 * 2 + C1 * 4 * 3 + DEC_H * 4)
                 + 3 * C1 * 4 * 4 + C1 * 4 + DEC_H * 4 + D * 4)
    assert kda.kda_device_status() == 0
    del dv4, v_states, y_ver

    # ---------------- verify rollback (the decode kernel on accepted prefixes) ----------------
    import numpy as np
    ver = inputs.decode_step(N=DEC_N, T=RB_T, H=DEC_H, seed=5)
    dv = {k: getattr(ver, k).to(dev) for k in
          ("q_raw", "k_raw", "v_raw", "conv_w", "ring_in", "f_raw", "dt_bias", "a_log",
           "beta_raw", "state_in", "norm_w", "gate_raw")}
    keep_h = np.random.default_rng(6).integers(1, RB_T, size=DEC_N, endpoint=False)
    keep_d = torch.from_numpy(keep_h.astype(np.int32)).to(dev)
    rb_state = torch.empty_like(dv["state_in"])
    rb_ring = torch.empty_like(dv["ring_in"])
    y_rb = torch.empty(DEC_N * RB_T, DEC_H * D, device=dev)

    def rollback():
        kda.kda_verify_rollback(dv["q_raw"], dv["k_raw"], dv["v_raw"], dv["conv_w"], dv["ring_in"],
                                rb_ring, dv["f_raw"], dv["dt_bias"], dv["a_log"], dv["beta_raw"],
                                dv["state_in"], rb_state, dv["norm_w"], dv["gate_raw"], y_rb,
                                keep_d, N=DEC_N, T=RB_T, H=DEC_H)

    for _ in range(max(args.warmup, 3)):
        rollback()
    barrier()
    r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    r0.record(stream)
    for _ in range(Kd):
        rollback()
    r1.record(stream)
    barrier()
    rb_ms = max_over_ranks(r0.elapsed_time(r1)) / Kd
    kept = int(keep_h.sum())
    # state and ring read + written once per sequence; raw q/k/v, f, beta, z read and y written
    # for the kept rows only
    rb_bytes = (DEC_N * (DEC_H * D * D * 4 * 2 + 3 * C1 * 3 * 4 * 2)
                + kept * (3 * C1 * 2 + C1 * 4 * 3 + DEC_H * 4) + 3 * C1 * 4 * 4 + C1 * 4 + D * 4)
    assert kda.kda_device_status() == 0

    # ---------------- stage 1: the six projections of the decode batch's layer input ----------
    import numpy as np_
    prng = np_.random.default_rng(7)
    pdims = (DEC_H * D, DEC_H * D, DEC_H * D, D, D, DEC_H)
    pw = [torch.from_numpy((prng.standard_normal((r, PROJ_HIDDEN), dtype=np_.float32)
                            / np_.float32(np_.sqrt(PROJ_HIDDEN)))).to(torch.bfloat16).to(dev)
          for r in pdims]
    px = torch.from_numpy(prng.standard_normal((DEC_N, PROJ_HIDDEN), dtype=np_.float32)).to(dev)
    pouts = [torch.empty(DEC_N, r, device=dev) for r in pdims]
    pws = kda.proj6_workspace(DEC_N, PROJ_HIDDEN, dev)

    def proj_step():
        kda.kda_proj6(px, *pw, *pouts, pws, H=DEC_H)

    for _ in range(max(args.warmup, 3)):
        proj_step()
    barrier()
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0.record(stream)
    for _ in range(Kd):
        proj_step()
    p1.record(stream)
    barrier()
    proj_ms = max_over_ranks(p0.elapsed_time(p1)) / Kd
    # per-kernel times from a separate short loop: the timer's events between the two launches
    # would serialise the projection kernel behind its split pre-pass
    kda.kernel_timing(True)
    for _ in range(10):
        proj_step()
    barrier()
    proj_kt = kda.kernel_times()
    kda.kernel_timing(False)
    proj_w_bytes = sum(r * PROJ_HIDDEN * 2 for r in pdims)
    proj_bytes = proj_w_bytes + DEC_N * PROJ_HIDDEN * 4 + DEC_N * sum(pdims) * 4
    assert kda.kda_device_status() == 0
    del pw, px, pouts, pws

    rep.close()
    if rank != 0:
        return None

    cpu = None if args.skip_cpu else cpu_baseline(pre, args.cpu_sample_heads)
    # the fused prefill normalises inside its inter kernel (no RMSNorm launch in the step)
    folded = fused and "kda_gated_rmsnorm_kernel" not in ktimes
    mbytes = _method_bytes(T, H, norm_folded=folded)
    ibytes = _impl_bytes(T, H, blk_bytes, chunks, norm_folded=folded)
    cflops = _chunk_flops(T, H)
    tensor_peak = peaks["bf16_tflops_sustained"]
    total_kms = sum(v[1] for v in ktimes.values())
    kernels = []
    for name, (n, kms) in sorted(ktimes.items(), key=lambda kv: -kv[1][1]):
        per = kms / n
        ent = {"kernel": name, "launches": n, "ms_per_launch": per, "share": kms / total_kms,
               "traffic": _traffic(name, KERNEL_SOURCES.get(name, []))}
        if name in mbytes:
            gbs = mbytes[name] / (per / 1e3) / 1e9
            ent.update(bytes_per_launch=mbytes[name], gbs=gbs, frac_hbm=gbs / peaks["hbm_gbs"],
                       impl_bytes_per_launch=ibytes[name],
                       impl_gbs=ibytes[name] / (per / 1e3) / 1e9)
        if name in cflops:
            tf = cflops[name] / (per / 1e3) / 1e12
            ent.update(tensor_flop_per_launch=cflops[name], tensor_tflops=tf,
                       frac_tensor=tf / tensor_peak)
        kernels.append(ent)
    step_bytes = sum(mbytes[k] for k in ("kda_chunk_prep_intra_kernel", "kda_chunk_inter_kernel")
                     + (() if folded else ("kda_gated_rmsnorm_kernel",)))
    method_tflops = scan_flop / (ms_step / 1e3) / 1e12
    step = {"method_bytes": step_bytes, "method_gbs": step_bytes / (ms_step / 1e3) / 1e9,
            "frac_hbm": step_bytes / (ms_step / 1e3) / 1e9 / peaks["hbm_gbs"],
            "method_flop": scan_flop, "method_tflops": method_tflops,
            "note": "the whole step: the method's I/O (raw q/k/v, f, beta, z, conv weights, ring "
                    "and state in and out, y) and its 7*D^2 flop per token-head over the step "
                    "time"}
    if fused:
        top = kernels[0]
        roofline = {"bound": "hbm", "kernel": top["kernel"], "achieved": top.get("gbs"),
                    "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": top.get("frac_hbm"),
                    "traffic": _traffic(top["kernel"], KERNEL_SOURCES.get(top["kernel"], [])),
                    "bytes_per_launch": top.get("bytes_per_launch"),
                    "impl_bytes_per_launch": top.get("impl_bytes_per_launch"),
                    "ms_per_launch": top["ms_per_launch"],
                    "peak_src": f"{peaks['src']} hbm_gbs (copy bandwidth)",
                    "bytes": "the method's I/O this kernel moves (raw q/k/v, f, beta, conv "
                             "weights, ring in); its workspace writes are impl_bytes_per_launch",
                    "timing": "library CUDA-event timer around each launch, timed region"}
        # the prefill's fraction of the tensor-pipe roofline: the method's flop over the step
        roofline_tensor = {"bound": "tensor", "kernel": "whole step (prep + intra, inter + "
                                                        "RMSNorm)",
                           "achieved": method_tflops, "peak": tensor_peak, "unit": "TFLOP/s",
                           "frac": method_tflops / tensor_peak,
                           "flop_per_step": scan_flop,
                           "peak_src": f"{peaks['src']} bf16_tflops_sustained (cuBLAS bf16 GEMM "
                                       "over seconds)"}
    else:
        roofline = {"bound": "alu", "kernel": "kda_scan_seq_kernel", "achieved": scan_tflops,
                    "peak": fp32_peak, "unit": "TFLOP/s", "frac": scan_tflops / fp32_peak,
                    "traffic": _traffic("kda_scan_seq_kernel",
                                        KERNEL_SOURCES["kda_scan_seq_kernel"]),
                    "ms_per_launch": scan_ms, "flop_per_launch": scan_flop,
                    "peak_src": f"{sms} SMs x 128 FP32 lanes x 2 x {peaks['sm_max_mhz']:.0f} MHz"}
        roofline_tensor = None
    return {
        "metric": METRIC, "value": tokens_per_s, "unit": "tokens/s", "n_gpus": ws,
        "steps": K, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": ("f32 state and elementwise; tensor-core products with f32 accumulate: "
                  "intra-chunk bf16 x3 (hi*hi + hi*lo + lo*hi), state chain f16 x2 (state and "
                  "U' split f16 hi + lo against single f16 images); bf16 raw q/k/v" if fused
                  else "f32 (FP32 FMA scan); bf16 raw q/k/v"),
        "data": "synthetic (seeded numpy default_rng; bf16 raw q/k/v, f32 gates, state, norm)",
        "config": {"workload": f"prefill: 1 sequence x 4096 tokens, H={H}, head_dim=128, conv K=4,"
                               " zero state and ring, whole mixer per step",
                   "path": "kda_prefill_fused (prep, chunked scan, gated RMSNorm)" if fused
                           else "staged calls, sequential scan",
                   "global_batch": ws, "seq_len": T, "heads": H, "head_dim": D,
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                   "scan_algo": args.scan_algo,
                   "l2": "inputs larger than L2 (470 MB read per step)"},
        "gpu_launches": sum(v[0] for v in ktimes.values()),
        "roofline": roofline,
        "roofline_tensor": roofline_tensor,
        "step": step,
        "kernels": kernels,
        "scan_ms_per_step": scan_ms,
        "e2e": e2e,
        "decode": {"workload": "64 sequences x 1 token, H=64, fused decode kernel, states "
                               "ping-ponged (512 MiB working set)",
                   "ms_per_step": dec_ms, "seq_per_s": ws * DEC_N / (dec_ms / 1e3),
                   "state_gbs": state_bytes / (dec_ms / 1e3) / 1e9,
                   "roofline": {"bound": "hbm", "kernel": "kda_decode_fused_kernel",
                                "achieved": dec_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                "frac": dec_gbs / peaks["hbm_gbs"],
                                "peak_src": f"{peaks['src']} hbm_gbs",
                                "traffic": _traffic("kda_decode_fused_kernel",
                                                    KERNEL_SOURCES["kda_decode_fused_kernel"]),
                                "bytes_per_launch": dec_bytes}},
        "decode_graph": {"workload": "the decode step in place (state and ring), captured once "
                                     "in a CUDA graph and replayed",
                         "ms_per_step": dec_graph_ms,
                         "roofline": {"bound": "hbm", "kernel": "kda_decode_fused_kernel",
                                      "achieved": dec_bytes / (dec_graph_ms / 1e3) / 1e9,
                                      "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                      "frac": dec_bytes / (dec_graph_ms / 1e3) / 1e9
                                      / peaks["hbm_gbs"], "bytes_per_launch": dec_bytes}},
        "verify": {"workload": f"{DEC_N} sequences x {VER_T} tokens, H={DEC_H}, one "
                               "kda_decode_fused launch (the decode kernel at T = 4), states "
                               "ping-ponged",
                   "ms_per_step": ver_ms, "tokens_per_s": ws * DEC_N * VER_T / (ver_ms / 1e3),
                   "roofline": {"bound": "hbm", "kernel": "kda_decode_fused_kernel",
                                "achieved": ver_bytes / (ver_ms / 1e3) / 1e9,
                                "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                "frac": ver_bytes / (ver_ms / 1e3) / 1e9 / peaks["hbm_gbs"],
                                "bytes_per_launch": ver_bytes}},
        "rollback": {"workload": f"{DEC_N} sequences, verify width {RB_T}, H={DEC_H}, accepted "
                                 f"prefixes U[1, {RB_T - 1}] ({kept} rows kept), one "
                                 "kda_verify_rollback launch",
                     "ms_per_step": rb_ms,
                     "roofline": {"bound": "hbm", "kernel": "kda_decode_fused_kernel",
                                  "achieved": rb_bytes / (rb_ms / 1e3) / 1e9,
                                  "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                  "frac": rb_bytes / (rb_ms / 1e3) / 1e9 / peaks["hbm_gbs"],
                                  "bytes_per_launch": rb_bytes}},
        "proj6": {"workload": f"the six projections of a {DEC_N}-row decode batch: hidden "
                              f"{PROJ_HIDDEN} -> q, k, v ({DEC_H * D} each), forget/gate down "
                              f"({D} each), beta ({DEC_H}); bf16 weights, f32 x and outputs; "
                              "kda_proj6 (x split + one tcgen05 launch)",
                  "ms_per_step": proj_ms,
                  "kernels": {k: {"launches": v[0], "ms_per_launch": v[1] / v[0]}
                              for k, v in proj_kt.items()},
                  "kernels_note": "per-kernel times from 10 extra calls with an event around each "
                                  "launch (serialised); ms_per_step is the timed loop without",
                  "roofline": {"bound": "hbm", "kernel": "kda_proj6_kernel + kda_proj_split_kernel",
                               "achieved": proj_bytes / (proj_ms / 1e3) / 1e9,
                               "peak": peaks["hbm_gbs"], "unit": "GB/s",
                               "frac": proj_bytes / (proj_ms / 1e3) / 1e9 / peaks["hbm_gbs"],
                               "bytes_per_launch": proj_bytes,
                               "weight_bytes": proj_w_bytes,
                               "traffic": _traffic("kda_proj6_kernel",
                                                   KERNEL_SOURCES["kda_proj6_kernel"]),
                               "bytes": "bf16 weights read once, x read and the six outputs "
                                        "written once (the x hi/lo images are intermediates)"}},
        "clocks": clocks,
        "cpu_baseline": cpu,
    }


# ------------------------------------------------------------------------------------------
# oracle (CPU baseline and reference arm)
# ------------------------------------------------------------------------------------------

def _oracle_sample(pre, heads):
    """The oracle on the prefill workload restricted to `heads` (heads are independent, so this
    is the exact work of those heads).  Returns seconds."""
    import numpy as np

    from oracle import oracle as orc
    ch = np.concatenate([np.arange(h * D, (h + 1) * D) for h in heads])
    C = pre.H * D
    prow = np.concatenate([p * C + ch for p in range(3)])
    args = dict(q_raw=pre.q_raw[:, ch], k_raw=pre.k_raw[:, ch], v_raw=pre.v_raw[:, ch],
                f_raw=pre.f_raw[:, ch], dt_bias=pre.dt_bias[ch], a_log=pre.a_log[heads],
                beta_raw=pre.beta_raw[:, heads], state_in=pre.state_in[:, heads],
                conv_w=pre.conv_w[prow], ring_in=pre.ring_in[:, prow], norm_w=pre.norm_w,
                gate_raw=pre.gate_raw[:, ch], H=len(heads), D=D, cu_seqlens=pre.cu_seqlens)
    t = time.perf_counter()
    orc.forward(**args)
    return time.perf_counter() - t


def cpu_baseline(pre, n_heads, min_secs=10.0):
    """The oracle as it stands on the host cores: the prefill workload restricted to n_heads heads
    (all 64 by default, i.e. the whole workload), repeated until at least min_secs have passed."""
    from oracle import oracle as orc
    orc.build()
    heads = list(range(n_heads))
    secs = []
    while sum(secs) < min_secs and len(secs) < 100:
        secs.append(_oracle_sample(pre, heads))
    total = sum(secs)
    tokens = PREFILL_T * (n_heads / pre.H) * len(secs)
    return {"value": tokens / total, "unit": "tokens/s",
            "cores": min(orc.num_threads(), n_heads), "kind": "oracle",
            "sample": f"prefill workload, heads 0..{n_heads - 1} of {pre.H} (all {PREFILL_T} "
                      f"tokens, full mixer) x {len(secs)} runs, {total:.1f} s"
                      + ("" if n_heads == pre.H else ", scaled to all heads"),
            "host_cpus": os.cpu_count()}


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return None
    from gated_delta_rule_scan_gb300 import inputs
    from oracle import oracle as orc
    orc.build()
    pre = inputs.prefill(T=PREFILL_T, H=PREFILL_H)
    heads = list(range(args.cpu_sample_heads))
    for _ in range(args.warmup if args.warmup < 2 else 1):
        _oracle_sample(pre, heads)
    ref_steps = min(args.steps, args.ref_steps)
    secs = [_oracle_sample(pre, heads) for _ in range(ref_steps)]
    frac = len(heads) / PREFILL_H
    s = statistics.mean(secs)
    value = PREFILL_T * frac / s
    cores = min(orc.num_threads(), len(heads))
    sample = (f"prefill workload, heads 0..{len(heads) - 1} of 64 per step (all 4096 tokens, "
              f"full mixer), mean of {ref_steps} steps, scaled to 64 heads")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": ws, "steps": ref_steps, "warmup": args.warmup,
            "ms_per_step": s * 1e3 / frac, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "prefill: 1 sequence x 4096 tokens, H=64, head_dim=128",
                       "seq_len": PREFILL_T, "heads": PREFILL_H},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def run_configs(args):
    """The other configurations of the workload table (the headline is the prefill): the 4-token
    verify, the packed varlen prefill and the long GDN scan, each through the public API on
    resident inputs larger than L2, one JSON line each (mean of --steps calls after 3 warm-up
    calls)."""
    import numpy as np
    import torch

    import __graft_entry__
    __graft_entry__.build()
    from gated_delta_rule_scan_gb300 import inputs, kda, mixer
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peaks = _peaks()
    K = max(args.steps, 5)

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(K):
            fn()
        e1.record()
        torch.cuda.synchronize()
        assert kda.kda_device_status() == 0
        return e0.elapsed_time(e1) / K

    def to_dev(inp):
        return {k: (None if getattr(inp, k) is None else getattr(inp, k).to(dev)) for k in
                ("q_raw", "k_raw", "v_raw", "conv_w", "ring_in", "f_raw", "dt_bias", "a_log",
                 "beta_raw", "state_in", "norm_w", "gate_raw")}

    # 1' verify: 64 sequences x 4 tokens, one fused launch
    ver = inputs.decode_step(N=DEC_N, T=4, H=DEC_H)
    dv = to_dev(ver)
    vout = dict(state_out=torch.empty_like(dv["state_in"]), ring_out=torch.empty_like(dv["ring_in"]),
                y=torch.empty(DEC_N * 4, DEC_H * D, device=dev))
    ms = timed(lambda: mixer.kda_decode(N=DEC_N, T=4, H=DEC_H, **dv, **vout))
    C1 = DEC_H * D
    vbytes = DEC_N * (DEC_H * D * D * 4 * 2 + 3 * C1 * 3 * 4 * 2 + 4 * (3 * C1 * 2 + C1 * 4 * 3
                                                                      + DEC_H * 4))
    print(json.dumps({"config": "verify: 64 sequences x 4 tokens, H=64, fused decode kernel",
                      "ms_per_call": ms, "tokens_per_s": DEC_N * 4 / (ms / 1e3),
                      "hbm_gbs": vbytes / (ms / 1e3) / 1e9,
                      "frac_hbm": vbytes / (ms / 1e3) / 1e9 / peaks["hbm_gbs"]}), flush=True)
    del dv, vout

    # 3 varlen: 16 packed sequences, lengths U[256, 8192], fused prefill
    var = inputs.varlen_prefill()
    dvl = to_dev(var)
    cu_h = torch.from_numpy(var.cu_seqlens.astype(np.int32))
    cu_d = cu_h.to(dev)
    total = int(cu_h[-1])
    ws = kda.prefill_workspace(var.N, total, var.H, dev)
    vout = dict(state_out=torch.empty_like(dvl["state_in"]), ring_out=torch.empty_like(dvl["ring_in"]),
                y=torch.empty(total, var.H * D, device=dev))
    ms = timed(lambda: mixer.kda_prefill(H=var.H, cu_seqlens=cu_d, cu_seqlens_host=cu_h,
                                         workspace=ws, **dvl, **vout))
    print(json.dumps({"config": f"varlen: {var.N} sequences, lengths U[256, 8192] "
                                f"({total} tokens), H={var.H}, fused prefill",
                      "ms_per_call": ms, "tokens_per_s": total / (ms / 1e3)}), flush=True)
    del dvl, vout, ws

    # 4 GDN long: 1 x 16384 tokens, H=32, per-head gate, f32, prep + scan (no conv, no norm)
    gdn = inputs.gdn_long()
    dg = to_dev(gdn)
    rows = gdn.rows
    ws = kda.scan_workspace(1, rows, gdn.H, dev, kda.ALGO_AUTO)
    f32 = lambda *sh: torch.empty(*sh, device=dev)  # noqa: E731
    C4 = gdn.H * D
    gbuf = dict(q_hat=f32(rows, C4), k_hat=f32(rows, C4), v_hat=f32(rows, C4), g=f32(rows, gdn.H),
                beta=f32(rows, gdn.H), o=f32(rows, C4))
    st = torch.empty_like(dg["state_in"])
    ms = timed(lambda: mixer.kda_forward(H=gdn.H, N=1, T=rows, gate_mode=1, out=gbuf,
                                         state_out=st, workspace=ws,
                                         **{k: v for k, v in dg.items()
                                            if k not in ("norm_w", "gate_raw")}))
    print(json.dumps({"config": f"GDN long: 1 x {rows} tokens, H={gdn.H}, per-head gate, f32, "
                                "prep + scan (AUTO: chunked)",
                      "ms_per_call": ms, "tokens_per_s": rows / (ms / 1e3)}), flush=True)


def run_crossover(args):
    """The sequential and the chunked scan (kda_scan, q/k/v/g resident) over a grid of sequence
    counts and lengths at H = 64: one JSON line per point with both times.  The library's AUTO
    rule is set from this table."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    from gated_delta_rule_scan_gb300 import kda
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    gen = torch.Generator(device=dev).manual_seed(5)

    def timed(N, T, H, algo):
        C, rows = H * D, N * T
        unit = lambda: torch.nn.functional.normalize(  # noqa: E731
            torch.randn(rows, H, D, device=dev, generator=gen), dim=-1).reshape(rows, C)
        q, k = unit(), unit()
        v = torch.randn(rows, C, device=dev, generator=gen)
        gl = -5.0 * torch.sigmoid(torch.randn(rows, C, device=dev, generator=gen))
        seq = algo == kda.ALGO_SEQ
        g = torch.exp(gl) if seq else gl
        beta = torch.sigmoid(torch.randn(rows, H, device=dev, generator=gen))
        s0 = torch.zeros(N, H, D, D, device=dev)
        s1, o = torch.empty_like(s0), torch.empty(rows, C, device=dev)
        ws = kda.scan_workspace(N, rows, H, dev, algo)
        gm = kda.GATE_EXP if seq else 0

        def f():
            kda.kda_scan(q, k, v, g, beta, s0, s1, o, N=N, T=T, H=H, gate_mode=gm, algo=algo,
                         workspace=ws)
        for _ in range(3):
            f()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            f()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / args.steps * 1e3

    for N in (1, 16, 64):
        for T in (16, 32, 48, 64, 96, 128, 256, 512, 1024):
            s_us = timed(N, T, PREFILL_H, kda.ALGO_SEQ)
            c_us = timed(N, T, PREFILL_H, kda.ALGO_CHUNK)
            print(json.dumps({"N": N, "T": T, "H": PREFILL_H, "seq_us": round(s_us, 1),
                              "chunk_us": round(c_us, 1),
                              "faster": "chunk" if c_us < s_us else "seq"}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--cpu-sample-heads", type=int, default=64)
    ap.add_argument("--ref-steps", type=int, default=5)
    ap.add_argument("--scan-algo", choices=("auto", "seq", "chunk"), default="auto",
                    help="prefill scan form (auto = the library's choice for the shape)")
    ap.add_argument("--skip-e2e", action="store_true", help="profiling runs: no host-copy leg")
    ap.add_argument("--skip-cpu", action="store_true", help="profiling runs: no oracle timing")
    ap.add_argument("--configs", action="store_true",
                    help="time the verify, varlen and GDN-long configurations, one JSON line each")
    ap.add_argument("--crossover", action="store_true",
                    help="time the sequential vs the chunked scan over lengths and exit")
    ap.add_argument("--heads", type=int, default=PREFILL_H,
                    help="profiling runs: a smaller prefill of the same kernels (default 64)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.configs:
        run_configs(args)
        return
    if args.crossover:
        run_crossover(args)
        return
    res = run_reference(args) if args.impl == "reference" else run_ours(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
