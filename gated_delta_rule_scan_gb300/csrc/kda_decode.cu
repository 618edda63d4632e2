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
// this kernel's outputs equal prep + scan + gated-RMSNorm launched separately, bit for bit, and a
// T-token launch equals T one-token launches bit for bit.
#include "kda_scan_core.cuh"

namespace kda {

constexpr int kDecThreads = 256;

template <bool BF16, int GATE_MODE>
__global__ void __launch_bounds__(kDecThreads, 2) kda_decode_fused_kernel(DecodeArgs a) {
    __shared__ __align__(16) float qh[kDecodeMaxT][kHeadDim];
    __shared__ __align__(16) float kh[kDecodeMaxT][kHeadDim];
    __shared__ __align__(16) float av[kDecodeMaxT][kHeadDim];
    __shared__ __align__(16) float vh[kDecodeMaxT][kHeadDim];
    __shared__ __align__(16) float os[kDecodeMaxT][kHeadDim];
    __shared__ float beta_s[kDecodeMaxT];
    __shared__ float ascal[kDecodeMaxT];
    __shared__ float part[2][4][kDecodeMaxT];
    __shared__ float inv_s[2][kDecodeMaxT];

    const int h = blockIdx.x, n = blockIdx.y;
    const int tid = threadIdx.x;
    const int H = a.H, T = a.T, K = a.K, R = a.K - 1;
    const long C = (long)H * kHeadDim;
    const long row0 = (long)n * T;
    const int warp = tid >> 5, lane = tid & 31;
    const int grp = lane >> 3, r = lane & 7;

    // ---- issue the state loads first: 4 columns x 16 elements per lane -------------------
    const int cw = warp * 16 + grp * 4;      // the group's first column
    const int own = cw + ((r >> 1) & 3);     // the column this lane reduces and writes
    const long col0 = (((long)n * H + h) * kHeadDim + cw) * kHeadDim;
    Col4 S;
    col4_load(S, a.state_in + col0, r);

    // ---- prologue, q and k planes: thread = (plane tid/128, channel tid%128) ----------------
    {
        const int p = tid >> 7, i = tid & 127;
        const int c = h * kHeadDim + i;
        const void* raw = p == 0 ? a.q_raw : a.k_raw;
        float wr[kMaxConvK], win[kMaxConvK];
        const long ring_row = ((long)n * 3 * C + p * C + c) * R;
#pragma unroll
        for (int m = 0; m < kMaxConvK; ++m) {
            const int jj = m - (kMaxConvK - K);
            const int d = kMaxConvK - m;
            wr[m] = jj >= 0 ? a.conv_w[(p * C + c) * K + jj] : 0.0f;
            win[m] = d <= R ? a.ring_in[ring_row + (R - d)] : 0.0f;
        }
        float (*dst)[kHeadDim] = p == 0 ? qh : kh;
        for (int t = 0; t < T; ++t) {
            window_push(win, load_raw<BF16>(raw, (row0 + t) * C + c));
            dst[t][i] = silu_f(conv_taps_f(wr, win, K));
        }
#pragma unroll
        for (int m = 0; m < kMaxConvK; ++m) {
            const int d = kMaxConvK - 1 - m;  // win[m] = sample d steps before the last one
            if (d < R) a.ring_out[ring_row + (R - 1 - d)] = win[m];
        }
    }
    // ---- v plane (threads 0..127) and the gate (threads 128..255) -------------------------
    if (tid < kHeadDim) {
        const int i = tid, c = h * kHeadDim + i;
        float wr[kMaxConvK], win[kMaxConvK];
        const long ring_row = ((long)n * 3 * C + 2 * C + c) * R;
#pragma unroll
        for (int m = 0; m < kMaxConvK; ++m) {
            const int jj = m - (kMaxConvK - K);
            const int d = kMaxConvK - m;
            wr[m] = jj >= 0 ? a.conv_w[(2 * C + c) * K + jj] : 0.0f;
            win[m] = d <= R ? a.ring_in[ring_row + (R - d)] : 0.0f;
        }
        for (int t = 0; t < T; ++t) {
            window_push(win, load_raw<BF16>(a.v_raw, (row0 + t) * C + c));
            vh[t][i] = silu_f(conv_taps_f(wr, win, K));
        }
#pragma unroll
        for (int m = 0; m < kMaxConvK; ++m) {
            const int d = kMaxConvK - 1 - m;
            if (d < R) a.ring_out[ring_row + (R - 1 - d)] = win[m];
        }
        if (i < T) {
            beta_s[i] = sigmoid_f(a.beta_raw[(row0 + i) * H + h]);
            if (GATE_MODE == 1)
                ascal[i] = expf(gdn_gate_f(a.f_raw[(row0 + i) * H + h], a.dt_bias[h], a.a_log[h]));
        }
    } else if (GATE_MODE == 0) {
        const int i = tid - kHeadDim, c = h * kHeadDim + i;
        const float rate = expf(a.a_log[h]);
        const float dt = a.dt_bias[c];
        for (int t = 0; t < T; ++t)
            av[t][i] = expf(kda_gate_f(a.f_raw[(row0 + t) * C + c], dt, rate, a.gate_lb));
    }
    __syncthreads();
    // ---- l2 norm of q (warps 0-3) and k (warps 4-7) ----------------------------------------
    {
        const int p = tid >> 7, i = tid & 127;
        float (*x)[kHeadDim] = p == 0 ? qh : kh;
        for (int t = 0; t < T; ++t) {
            const float v = x[t][i];
            const float ssum = warp_sum(__fmul_rn(v, v));
            if (lane == 0) part[p][warp & 3][t] = ssum;
        }
        __syncthreads();
        if (tid < 2 * kDecodeMaxT) {
            const int pl = tid / kDecodeMaxT, t = tid % kDecodeMaxT;
            if (t < T) {
                const float p4[4] = {part[pl][0][t], part[pl][1][t], part[pl][2][t], part[pl][3][t]};
                inv_s[pl][t] = l2_inv_f(head_sum4(p4), a.l2_eps);
            }
        }
        __syncthreads();
        for (int t = 0; t < T; ++t) x[t][i] = __fmul_rn(x[t][i], inv_s[p][t]);
        __syncthreads();
    }

    // ---- the recurrence, token by token ---------------------------------------------------
    for (int t = 0; t < T; ++t) {
        const float dq = col4_token<GATE_MODE == 0>(S, &kh[t][0], &av[t][0], ascal[t], &qh[t][0],
                                                    vh[t][own], beta_s[t], r, lane);
        if ((r & 1) == 0) os[t][own] = __fmul_rn(a.scale, dq);
    }
    col4_store(S, a.state_out + col0, r);
    __syncthreads();
    // ---- epilogue: gated RMSNorm, one warp per token row -----------------------------------
    for (int t = warp; t < T; t += kDecThreads / 32) {
        const float4 o4 = *reinterpret_cast<const float4*>(&os[t][4 * lane]);
        float ss = __fmul_rn(o4.x, o4.x);
        ss = ss + __fmul_rn(o4.y, o4.y);
        ss = ss + __fmul_rn(o4.z, o4.z);
        ss = ss + __fmul_rn(o4.w, o4.w);
        const float inv = rms_inv_f(warp_sum(ss), a.rms_eps);
        const long base = (row0 + t) * C + h * kHeadDim + 4 * lane;
        const float4 w4 = *reinterpret_cast<const float4*>(a.norm_w + 4 * lane);
        const float4 z4 = *reinterpret_cast<const float4*>(a.gate_raw + base);
        float4 y4;
        y4.x = gated_norm_f(o4.x, inv, w4.x, z4.x);
        y4.y = gated_norm_f(o4.y, inv, w4.y, z4.y);
        y4.z = gated_norm_f(o4.z, inv, w4.z, z4.z);
        y4.w = gated_norm_f(o4.w, inv, w4.w, z4.w);
        *reinterpret_cast<float4*>(a.y + base) = y4;
    }
}

cudaError_t launch_decode_fused(const DecodeArgs& a, cudaStream_t s) {
    if (a.N == 0 || a.T == 0) return cudaSuccess;
    dim3 grid((unsigned)a.H, (unsigned)a.N);
    if (a.raw_bf16) {
        if (a.gate_mode == 0) kda_decode_fused_kernel<true, 0><<<grid, kDecThreads, 0, s>>>(a);
        else kda_decode_fused_kernel<true, 1><<<grid, kDecThreads, 0, s>>>(a);
    } else {
        if (a.gate_mode == 0) kda_decode_fused_kernel<false, 0><<<grid, kDecThreads, 0, s>>>(a);
        else kda_decode_fused_kernel<false, 1><<<grid, kDecThreads, 0, s>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace kda
