// kda_decode.cu -- fused decode / multi-token verify: prologue + scan + epilogue in one launch.
//
// Method ("memra_engine/kda.rs", memra-engine 0.125.0): kda_core_gated stages 2-6 for T new
// tokens per sequence (T = 1 is a decode step; T > 1 is a speculative verify whose rows must equal
// T chained decode steps, the decode==verify law the module doc states).  Steps per token:
// conv + SiLU over the ring and the new rows, ring roll, l2 norm of q and k, the KDA (or GDN) gate
// and beta, the delta-rule recurrence, the sigmoid-gated RMSNorm.
//
// GB300 layout.  Decode is bound by the 64 KiB state read + write per (sequence, head), so one CTA
// owns one (sequence, head) and issues its whole state column block as streaming 128-bit loads at
// entry, before the prologue runs, so the HBM latency overlaps the conv / norm / gate work.  256
// threads; 8 lanes share 4 value columns with 16 key-dim elements each, and the per-token step is
// the sequential prefill scan's (kda_scan_core.cuh), instruction for instruction.
// The prologue and epilogue use the same device functions as the prep and epilogue kernels, so
// this kernel's outputs equal prep + scan + gated-RMSNorm launched separately to f32 rounding (the
// standalone sequential scan groups 16 lanes per column, this kernel 8, so their key-dimension
// sums round differently; the ring is bit-equal), and a T-token launch equals T one-token
// launches bit for bit.
#include "kda_scan_core.cuh"

namespace kda {

constexpr int kDecThreads = 256;

// Asynchronous 4- or 8-byte copies global -> shared (cp.async, completion waited per thread).
__device__ __forceinline__ void cp_async_4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(src))
                 : "memory");
}
__device__ __forceinline__ void cp_async_8(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(src))
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit_wait() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_all;" ::: "memory");
}

// Thread-block cluster barrier (every thread of every CTA of the cluster arrives; release /
// acquire order the shared-memory writes before it with the remote reads after it).
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// A float in the shared memory of the cluster's CTA `rank`, at the address of `local` there.
__device__ __forceinline__ float ld_cluster_f32(const float* local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

// KW: register window width of the conv (4 when K <= 4, else 8).  WIDE: value heads of
// a.vsub > 1 units, launched as clusters of a.vsub CTAs.
template <bool BF16, int GATE_MODE, int KW, bool WIDE>
__global__ void __launch_bounds__(kDecThreads, 2) kda_decode_fused_kernel(DecodeArgs a) {
    __shared__ __align__(16) float qh[kDecodeMaxT][kHeadDim];
    __shared__ __align__(16) float kh[kDecodeMaxT][kHeadDim];
    __shared__ __align__(16) float av[kDecodeMaxT][kHeadDim];
    __shared__ __align__(16) float vh[kDecodeMaxT][kHeadDim];
    __shared__ __align__(16) float os[kDecodeMaxT][kHeadDim];
    __shared__ float beta_s[kDecodeMaxT];
    __shared__ float ascal[kDecodeMaxT];
    __shared__ float part[2][2][kDecodeMaxT];
    __shared__ float inv_s[2][kDecodeMaxT];
    __shared__ float nss[kDecodeMaxT];           // this unit's RMSNorm sums of squares (vs > 1)

    // unit h: value column block h % vs of value head gh = h / vs, whose gate and beta it reads,
    // and q/k head hq = gh % Hk (vs = 1: the value head itself)
    const int h = blockIdx.x, n = blockIdx.y;
    const int vs = WIDE ? a.vsub : 1;
    const int gh = WIDE ? h / vs : h;
    const int tid = threadIdx.x;
    const int H = a.H, K = a.K, R = a.K - 1;
    const long C = (long)H * kHeadDim;
    const int Hg = H / vs;                       // value heads
    const long Cg = (long)Hg * kHeadDim;         // per-channel gate rows
    const int Hkq = prep_qk_heads(Hg, a.Hk);
    const int hq = gh < Hkq ? gh : gh % Hkq;
    const long row0 = (long)n * a.T;             // rows of sequence n: stride T in every mode
    // tokens taken: all T, or (rollback) the first keep[n]
    const int T = a.keep != nullptr ? min(max(a.keep[n], 0), a.T) : a.T;
    const int warp = tid >> 5, lane = tid & 31;
    const int grp = lane >> 3, r = lane & 7;

    // ---- the prologue's inputs first, so that they return ahead of the state stream and the
    //      conv / norm / gate work overlaps the state transfer: conv weights and ring slots into
    //      registers; every token's raw q / k / v (and gate input) channel pair copied into the
    //      slot its result will take (qh / kh / vh, av); beta and the scalar gate inputs.
    //      64 threads per task, each on a channel pair (2i, 2i+1): threads 0-63 q plane, 64-127
    //      k plane, 128-191 v plane (+ beta), 192-255 the gate.  Grouped queries: the q and k
    //      planes hold Hk heads and this value head reads q/k head h % Hk; only the CTAs of heads
    //      h < Hk write those heads' ring rows.
    const int task = tid >> 6, i0 = 2 * (tid & 63);
    const int cg = gh * kHeadDim + i0;           // channel pair in the gate rows
    float wr[2][KW], win[2][KW];
    long ring_row = 0;
    bool ring_owner = false;
    float braw = 0.0f, fgate = 0.0f, dtb = 0.0f, alog = 0.0f;
    float2 dt = make_float2(0.0f, 0.0f);
    if (task < 3) {
        const void* raw = task == 0 ? a.q_raw : (task == 1 ? a.k_raw : a.v_raw);
        const long Cp = plane_width(H, a.Hk, task);        // row width of this plane
        const int cp = (task < 2 ? hq : h) * kHeadDim + i0;
        // the q / k ring rows of head hq are rolled by one unit: the first of value head hq
        ring_owner = task == 2 || (h == gh * vs && gh < Hkq);
        ring_row = ((long)n * ring_channels(H, a.Hk) + plane_offset(H, a.Hk, task) + cp) * R;
#pragma unroll
        for (int m = 0; m < KW; ++m) {
            const int jj = m - (KW - K);
            const int d = KW - m;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                wr[e][m] = jj >= 0 ? a.conv_w[(plane_offset(H, a.Hk, task) + cp + e) * K + jj] : 0.0f;
                win[e][m] = d <= R ? a.ring_in[ring_row + e * R + (R - d)] : 0.0f;
            }
        }
        float (*dst)[kHeadDim] = task == 0 ? qh : (task == 1 ? kh : vh);
        for (int t = 0; t < T; ++t) {
            if (BF16)
                cp_async_4(&dst[t][i0], reinterpret_cast<const __nv_bfloat16*>(raw) + (row0 + t) * Cp + cp);
            else
                cp_async_8(&dst[t][i0], reinterpret_cast<const float*>(raw) + (row0 + t) * Cp + cp);
        }
        if (task == 2 && (tid & 63) < T) {
            const long rw = (row0 + (tid & 63)) * Hg + gh;
            braw = a.beta_raw[rw];
            if (GATE_MODE == 1) {
                fgate = a.f_raw[rw];
                dtb = a.dt_bias[gh];
                alog = a.a_log[gh];
            }
        }
    } else if (GATE_MODE == 0) {
        alog = a.a_log[gh];
        dt = *reinterpret_cast<const float2*>(a.dt_bias + cg);
        for (int t = 0; t < T; ++t) cp_async_8(&av[t][i0], a.f_raw + (row0 + t) * Cg + cg);
    }

    // ---- then the state loads: 4 columns x 16 elements per lane -----------------------------
    const int cw = warp * 16 + grp * 4;      // the group's first column
    const long col0 = (((long)n * H + h) * kHeadDim + cw) * kHeadDim;
    Col4 S;
    col4_load(S, a.state_in + col0, r);

    // ---- prologue: conv + SiLU and the ring roll, beta, the gate -------------------------------
    if (task < 3) {
        float (*dst)[kHeadDim] = task == 0 ? qh : (task == 1 ? kh : vh);
        cp_async_commit_wait();
        for (int t = 0; t < T; ++t) {
            float2 x;
            if (BF16) x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&dst[t][i0]));
            else x = *reinterpret_cast<const float2*>(&dst[t][i0]);
            window_push(win[0], x.x);
            window_push(win[1], x.y);
            *reinterpret_cast<float2*>(&dst[t][i0]) =
                make_float2(silu_f(conv_taps_f(wr[0], win[0], K)), silu_f(conv_taps_f(wr[1], win[1], K)));
        }
#pragma unroll
        for (int m = 0; m < KW; ++m) {
            const int d = KW - 1 - m;  // win[m] = sample d steps before the last one
            if (d < R && ring_owner) {
                a.ring_out[ring_row + (R - 1 - d)] = win[0][m];
                a.ring_out[ring_row + R + (R - 1 - d)] = win[1][m];
            }
        }
        if (task == 2 && (tid & 63) < T) {
            const int t = tid & 63;
            beta_s[t] = sigmoid_f(braw);
            if (GATE_MODE == 1) ascal[t] = decay_f(gdn_gate_f(fgate, dtb, alog));
        }
    } else if (GATE_MODE == 0) {
        const float rate = expf(alog);
        cp_async_commit_wait();
        for (int t = 0; t < T; ++t) {
            const float2 f = *reinterpret_cast<const float2*>(&av[t][i0]);
            *reinterpret_cast<float2*>(&av[t][i0]) =
                make_float2(decay_f(kda_gate_f(f.x, dt.x, rate, a.gate_lb)),
                            decay_f(kda_gate_f(f.y, dt.y, rate, a.gate_lb)));
        }
    }
    __syncthreads();
    // ---- l2 norm of q (warps 0-1) and k (warps 2-3) ----------------------------------------
    if (task < 2) {
        // four tokens' butterflies at a time, so their shuffles overlap (each value still goes
        // through its own warp_sum, so the bits do not depend on the grouping)
        float (*x)[kHeadDim] = task == 0 ? qh : kh;
        for (int t0 = 0; t0 < T; t0 += 4) {
            float ssum[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                ssum[j] = 0.0f;
                if (t0 + j < T) {
                    const float2 v = *reinterpret_cast<const float2*>(&x[t0 + j][i0]);
                    ssum[j] = pair_sumsq(v.x, v.y);
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) ssum[j] = warp_sum(ssum[j]);
            if (lane == 0) {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (t0 + j < T) part[task][warp & 1][t0 + j] = ssum[j];
            }
        }
    }
    __syncthreads();
    if (tid < 2 * kDecodeMaxT) {
        const int pl = tid / kDecodeMaxT, t = tid % kDecodeMaxT;
        if (t < T) inv_s[pl][t] = l2_inv_f(part[pl][0][t] + part[pl][1][t], a.l2_eps);
    }
    __syncthreads();
    if (task < 2) {
        float (*x)[kHeadDim] = task == 0 ? qh : kh;
        for (int t = 0; t < T; ++t) {
            const float2 v = *reinterpret_cast<const float2*>(&x[t][i0]);
            *reinterpret_cast<float2*>(&x[t][i0]) =
                make_float2(__fmul_rn(v.x, inv_s[task][t]), __fmul_rn(v.y, inv_s[task][t]));
        }
    }
    __syncthreads();

    // ---- the recurrence, token by token ---------------------------------------------------
    {
        TokView vw;
        vw.k = &kh[0][0];
        vw.a = &av[0][0];
        vw.q = &qh[0][0];
        vw.a_scal = ascal;
        vw.v = &vh[0][0];
        vw.beta = beta_s;
        vw.out = &os[0][0];
        vw.row_stride = kHeadDim;
        vw.v_stride = kHeadDim;
        vw.v_col0 = cw;
        vw.out_stride = kHeadDim;
        vw.out_col0 = cw;
        col4_tokens<GATE_MODE == 0, false>(S, T, vw, a.scale, r, lane);
    }
    // the epilogue's first gate row and the norm weight are requested before the state stores go
    // out, so their latency overlaps the stores and the barrier
    // (the unit's column block of the norm weight: blockIdx.x % vsub, from the launch parameters)
    const float4 w4 = *reinterpret_cast<const float4*>(
        a.norm_w + (WIDE ? (int)blockIdx.x % a.vsub : 0) * kHeadDim + 4 * lane);
    float4 z_first = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (warp < T)
        z_first = *reinterpret_cast<const float4*>(a.gate_raw + (row0 + warp) * C + h * kHeadDim + 4 * lane);
    col4_store(S, a.state_out + col0, r);
    __syncthreads();
    // ---- epilogue: gated RMSNorm, one warp per token row -----------------------------------
    // A value head of vs units: each unit's sum of squares of a row goes to its shared memory,
    // and after a cluster barrier every unit adds the vs sums in unit order (the order of the
    // standalone RMSNorm over rows of vs * 128), for the mean over the whole value row.
    if constexpr (WIDE) {
        for (int t = warp; t < T; t += kDecThreads / 32) {
            const float4 o4 = *reinterpret_cast<const float4*>(&os[t][4 * lane]);
            float ss = __fmul_rn(o4.x, o4.x);
            ss = ss + __fmul_rn(o4.y, o4.y);
            ss = ss + __fmul_rn(o4.z, o4.z);
            ss = ss + __fmul_rn(o4.w, o4.w);
            ss = warp_sum(ss);
            if (lane == 0) nss[t] = ss;
        }
        cluster_sync_all();
    }
    for (int t = warp; t < T; t += kDecThreads / 32) {
        const float4 o4 = *reinterpret_cast<const float4*>(&os[t][4 * lane]);
        float inv;
        if constexpr (WIDE) {
            float tot = 0.0f;
            for (int b = 0; b < a.vsub; ++b) tot = tot + ld_cluster_f32(&nss[t], (uint32_t)b);
            inv = rms_inv_w(tot, a.rms_eps, a.vsub * kHeadDim);
        } else {
            float ss = __fmul_rn(o4.x, o4.x);
            ss = ss + __fmul_rn(o4.y, o4.y);
            ss = ss + __fmul_rn(o4.z, o4.z);
            ss = ss + __fmul_rn(o4.w, o4.w);
            inv = rms_inv_f(warp_sum(ss), a.rms_eps);
        }
        const long base = (row0 + t) * C + h * kHeadDim + 4 * lane;
        const float4 z4 = t == warp ? z_first : *reinterpret_cast<const float4*>(a.gate_raw + base);
        float4 y4;
        if (a.norm_silu) {
            y4.x = gated_norm_f<true>(o4.x, inv, w4.x, z4.x);
            y4.y = gated_norm_f<true>(o4.y, inv, w4.y, z4.y);
            y4.z = gated_norm_f<true>(o4.z, inv, w4.z, z4.z);
            y4.w = gated_norm_f<true>(o4.w, inv, w4.w, z4.w);
        } else {
            y4.x = gated_norm_f(o4.x, inv, w4.x, z4.x);
            y4.y = gated_norm_f(o4.y, inv, w4.y, z4.y);
            y4.z = gated_norm_f(o4.z, inv, w4.z, z4.z);
            y4.w = gated_norm_f(o4.w, inv, w4.w, z4.w);
        }
        *reinterpret_cast<float4*>(a.y + base) = y4;
    }
    if constexpr (WIDE) cluster_sync_all();      // the other units have read this unit's sums
}

// A value head of vsub > 1 units is one thread-block cluster of vsub CTAs along x.
template <typename Kern>
static cudaError_t launch_dec_kernel(Kern kernel, const DecodeArgs& a, cudaStream_t s) {
    dim3 grid((unsigned)a.H, (unsigned)a.N);
    if (a.vsub <= 1) {
        kernel<<<grid, kDecThreads, 0, s>>>(a);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kDecThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)a.vsub;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

template <bool BF16, int GM>
static cudaError_t launch_dec_t(const DecodeArgs& a, cudaStream_t s) {
    KernelTimer kt(kKDecode, s);
    if (a.vsub > 1) {
        if (a.K <= 4) return launch_dec_kernel(kda_decode_fused_kernel<BF16, GM, 4, true>, a, s);
        return launch_dec_kernel(kda_decode_fused_kernel<BF16, GM, kMaxConvK, true>, a, s);
    }
    if (a.K <= 4) return launch_dec_kernel(kda_decode_fused_kernel<BF16, GM, 4, false>, a, s);
    return launch_dec_kernel(kda_decode_fused_kernel<BF16, GM, kMaxConvK, false>, a, s);
}

cudaError_t launch_decode_fused(const DecodeArgs& a, cudaStream_t s) {
    if (a.N == 0 || a.T == 0) return cudaSuccess;
    if (a.raw_bf16)
        return a.gate_mode == 0 ? launch_dec_t<true, 0>(a, s) : launch_dec_t<true, 1>(a, s);
    return a.gate_mode == 0 ? launch_dec_t<false, 0>(a, s) : launch_dec_t<false, 1>(a, s);
}

}  // namespace kda
