// kda_prep.cu -- the scan's prologue over projected channels, prefill form.
//
// Method ("memra_engine/kda.rs", memra-engine 0.125.0, kda_core_gated stages 2-4):
//   stage 2  per plane p in (q, k, v) and channel c: y_t = silu(sum_j w[c][j] * xt[t+j]), where
//            xt is the conv ring (oldest first) followed by the call's raw rows; the ring then
//            rolls to the last K-1 raw samples (Engine::kda_conv_silu / kda_conv_ring_roll;
//            shift-left-append orientation as in gdn_ops.rs gdn_causal_conv1d_silu_into).
//   stage 3  q, k: x / sqrt(sum_i x_i^2 + 1e-6) over each head's 128 channels (KDA_L2_EPS doc).
//   stage 4  g = lb * sigmoid(exp(A_log[h]) * (f + dt_bias[c])) per channel (Engine::kda_gate),
//            or the GDN per-head g = -exp(A_log[h]) * softplus(alpha + dt_bias[h])
//            (gdn_ops.rs gdn_gates_into); beta = sigmoid(beta_raw) per (token, head).
//
// Layout: one warp walks a run of kRun consecutive packed rows of one head; lane l owns channels
// 4l..4l+3 of the head in all three planes and keeps their conv weights and a sliding window of
// the last K raw samples in registers, so every raw sample is read once (plus the K-1 halo rows
// of the run), as 8-byte bf16x4 (or 16-byte f32x4) vectors, one row ahead of its use.  The l2
// norm is one warp butterfly per row; every output row is a 512-byte coalesced store.  A run may
// straddle sequence boundaries (varlen): the window restarts from the next sequence's ring.  The
// ring is rewritten by a second, tiny kernel launched after this one on the same stream, so
// ring_in and ring_out may be the same buffer.
#include "kda_device.cuh"
#include "kda_internal.h"
#include "kda_ring.cuh"

namespace kda {

constexpr int kRun = 16;               // rows per warp
constexpr int kPrepWarps = 8;          // warps (runs) per CTA
constexpr int kPrepThreads = 32 * kPrepWarps;

// Sequence holding packed row r: index n, first row begin, one-past-last row end.
__device__ __forceinline__ void seq_of_row(const SeqLayout& L, long r, int& n, long& begin,
                                           long& end) {
    if (L.cu_seqlens == nullptr) {
        n = (int)(r / L.T_uniform);
        begin = (long)n * L.T_uniform;
        end = begin + L.T_uniform;
        return;
    }
    int lo = 0, hi = L.N;  // largest n with cu[n] <= r: its sequence is non-empty and holds r
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if ((long)L.cu_seqlens[mid] <= r) lo = mid; else hi = mid;
    }
    n = lo;
    begin = L.cu_seqlens[lo];
    end = L.cu_seqlens[lo + 1];
}

template <bool BF16>
__device__ __forceinline__ float4 load_raw4(const void* base, long idx) {
    if constexpr (BF16) {
        const uint2 u = *reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(base) + idx);
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
        return make_float4(a.x, a.y, b.x, b.y);
    } else {
        return *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(base) + idx);
    }
}

// Register state of one plane for this lane's 4 channels: weights and window, aligned to the end
// (slot KW-1 = the current sample).
template <int KW>
struct PlaneWin {
    float w[4][KW];
    float x[4][KW];
};

template <int KW>
__device__ __forceinline__ void pw_push(PlaneWin<KW>& P, const float4& v) {
#pragma unroll
    for (int e = 0; e < 4; ++e)
#pragma unroll
        for (int m = 0; m < KW - 1; ++m) P.x[e][m] = P.x[e][m + 1];
    P.x[0][KW - 1] = v.x; P.x[1][KW - 1] = v.y; P.x[2][KW - 1] = v.z; P.x[3][KW - 1] = v.w;
}

template <int KW>
__device__ __forceinline__ float4 pw_conv_silu(const PlaneWin<KW>& P, int K) {
    return make_float4(silu_f(conv_taps_f(P.w[0], P.x[0], K)), silu_f(conv_taps_f(P.w[1], P.x[1], K)),
                       silu_f(conv_taps_f(P.w[2], P.x[2], K)), silu_f(conv_taps_f(P.w[3], P.x[3], K)));
}

// Fill the window with the K-1 samples preceding position p of the sequence that starts at row
// begin: slot KW-d holds the sample at p-d (raw rows when p-d >= 0, else the ring, oldest first).
template <bool BF16, int KW>
__device__ __forceinline__ void pw_fill(PlaneWin<KW>& P, const void* raw, long C, int c,
                                        const float* ring_in, long ring_row0, int R, long begin,
                                        long p) {
#pragma unroll
    for (int m = 0; m < KW; ++m) {
        const int d = KW - m;
        float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (d <= R) {
            const long pos = p - d;
            if (pos >= 0) {
                v = load_raw4<BF16>(raw, (begin + pos) * C + c);
            } else {
                const long s2 = R + pos;
                v = make_float4(ring_in[ring_row0 + s2], ring_in[ring_row0 + R + s2],
                                ring_in[ring_row0 + 2 * R + s2], ring_in[ring_row0 + 3 * R + s2]);
            }
        }
        P.x[0][m] = v.x; P.x[1][m] = v.y; P.x[2][m] = v.z; P.x[3][m] = v.w;
    }
}

// EXP: write the decay factor exp(g) instead of the log-decay g.  KW: compile-time bound on K.
template <bool BF16, int GATE_MODE, bool CONV, bool EXP, int KW>
__global__ void __launch_bounds__(kPrepThreads) kda_prep_kernel(PrepArgs a) {
    const int h = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long r0 = ((long)blockIdx.x * kPrepWarps + warp) * kRun;
    const long rows = a.seq.total_rows;
    if (r0 >= rows) return;
    const int nr = (int)min((long)kRun, rows - r0);
    const int H = a.H;
    const long C = (long)H * kHeadDim;
    // grouped queries: the q and k planes hold Hk heads (rows Cq wide); the CTAs of heads h < Hk
    // also compute q/k head h, the others only their v head, gate and beta
    const long Cq = plane_width(H, a.Hk, 0);
    const bool has_qk = h < prep_qk_heads(H, a.Hk);
    // value heads wider than 128 (H counts 128-wide sub-heads): the CTAs of heads h < Hg also
    // compute value head h's gate and beta, whose rows are Cg = Hg * 128 (or Hg) wide
    const int Hg = prep_gate_heads(a);
    const bool has_gate = h < Hg;
    const long Cg = (long)Hg * kHeadDim;
    const long RC = ring_channels(H, a.Hk);
    const int c = h * kHeadDim + 4 * lane;     // first of this lane's 4 channels in a plane
    const int K = a.K, R = a.K - 1;

    PlaneWin<KW> pq, pk, pv;
    int n = 0;
    long begin = 0, end = 0;
    if constexpr (CONV) {
#pragma unroll
        for (int e = 0; e < 4; ++e)
#pragma unroll
            for (int m = 0; m < KW; ++m) {
                const int j = m - (KW - K);
                pq.w[e][m] = j >= 0 && has_qk ? a.conv_w[(0 * Cq + c + e) * K + j] : 0.0f;
                pk.w[e][m] = j >= 0 && has_qk ? a.conv_w[(1 * Cq + c + e) * K + j] : 0.0f;
                pv.w[e][m] = j >= 0 ? a.conv_w[(2 * Cq + c + e) * K + j] : 0.0f;
            }
        seq_of_row(a.seq, r0, n, begin, end);
        const long rr = (long)n * RC * R;
        if (has_qk) {
            pw_fill<BF16, KW>(pq, a.q_raw, Cq, c, a.ring_in, rr + (0 * Cq + c) * R, R, begin, r0 - begin);
            pw_fill<BF16, KW>(pk, a.k_raw, Cq, c, a.ring_in, rr + (1 * Cq + c) * R, R, begin, r0 - begin);
        }
        pw_fill<BF16, KW>(pv, a.v_raw, C, c, a.ring_in, rr + (2 * Cq + c) * R, R, begin, r0 - begin);
    }
    float rate = 0.0f;
    float4 dt = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (GATE_MODE == 0 && has_gate) {
        rate = expf(a.a_log[h]);
        dt = *reinterpret_cast<const float4*>(a.dt_bias + c);
    }

    // row-ahead prefetch of the raw samples and f
    const float4 z4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    float4 nq = has_qk ? load_raw4<BF16>(a.q_raw, r0 * Cq + c) : z4;
    float4 nk = has_qk ? load_raw4<BF16>(a.k_raw, r0 * Cq + c) : z4;
    float4 nv = load_raw4<BF16>(a.v_raw, r0 * C + c);
    float4 nf = GATE_MODE == 0 && has_gate ? *reinterpret_cast<const float4*>(a.f_raw + r0 * Cg + c)
                               : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int i = 0; i < nr; ++i) {
        const long r = r0 + i;
        const float4 cq = nq, ck = nk, cv = nv, cf = nf;
        if (i + 1 < nr) {
            if (has_qk) {
                nq = load_raw4<BF16>(a.q_raw, (r + 1) * Cq + c);
                nk = load_raw4<BF16>(a.k_raw, (r + 1) * Cq + c);
            }
            nv = load_raw4<BF16>(a.v_raw, (r + 1) * C + c);
            if (GATE_MODE == 0 && has_gate)
                nf = *reinterpret_cast<const float4*>(a.f_raw + (r + 1) * Cg + c);
        }
        float4 xq, xk, xv;
        if constexpr (CONV) {
            if (r >= end) {  // entered the next non-empty sequence: restart the windows
                seq_of_row(a.seq, r, n, begin, end);
                const long rr = (long)n * RC * R;
                if (has_qk) {
                    pw_fill<BF16, KW>(pq, a.q_raw, Cq, c, a.ring_in, rr + (0 * Cq + c) * R, R, begin, 0);
                    pw_fill<BF16, KW>(pk, a.k_raw, Cq, c, a.ring_in, rr + (1 * Cq + c) * R, R, begin, 0);
                }
                pw_fill<BF16, KW>(pv, a.v_raw, C, c, a.ring_in, rr + (2 * Cq + c) * R, R, begin, 0);
            }
            xq = xk = z4;
            if (has_qk) {
                pw_push(pq, cq);
                pw_push(pk, ck);
                xq = pw_conv_silu(pq, K);
                xk = pw_conv_silu(pk, K);
            }
            pw_push(pv, cv);
            xv = pw_conv_silu(pv, K);
        } else {
            xq = cq;
            xk = ck;
            xv = cv;
        }
        *reinterpret_cast<float4*>(a.v_hat + r * C + c) = xv;
        if (has_qk) {
            float sq = __fmul_rn(xq.x, xq.x);
            sq = fmaf(xq.y, xq.y, sq); sq = fmaf(xq.z, xq.z, sq); sq = fmaf(xq.w, xq.w, sq);
            float sk = __fmul_rn(xk.x, xk.x);
            sk = fmaf(xk.y, xk.y, sk); sk = fmaf(xk.z, xk.z, sk); sk = fmaf(xk.w, xk.w, sk);
            const float iq = l2_inv_f(warp_sum(sq), a.l2_eps);
            const float ik = l2_inv_f(warp_sum(sk), a.l2_eps);
            *reinterpret_cast<float4*>(a.q_hat + r * Cq + c) =
                make_float4(xq.x * iq, xq.y * iq, xq.z * iq, xq.w * iq);
            *reinterpret_cast<float4*>(a.k_hat + r * Cq + c) =
                make_float4(xk.x * ik, xk.y * ik, xk.z * ik, xk.w * ik);
        }
        if (GATE_MODE == 0 && has_gate) {
            float4 g = make_float4(kda_gate_f(cf.x, dt.x, rate, a.gate_lb), kda_gate_f(cf.y, dt.y, rate, a.gate_lb),
                                   kda_gate_f(cf.z, dt.z, rate, a.gate_lb), kda_gate_f(cf.w, dt.w, rate, a.gate_lb));
            if (EXP) g = make_float4(decay_f(g.x), decay_f(g.y), decay_f(g.z), decay_f(g.w));
            *reinterpret_cast<float4*>(a.g + r * Cg + c) = g;
        }
    }
    if (lane < nr && has_gate) {
        const long r = r0 + lane;
        a.beta[r * Hg + h] = sigmoid_f(a.beta_raw[r * Hg + h]);
        if constexpr (GATE_MODE == 1) {
            const float gl = gdn_gate_f(a.f_raw[r * Hg + h], a.dt_bias[h], a.a_log[h]);
            a.g[r * Hg + h] = EXP ? decay_f(gl) : gl;
        }
    }
}

// Ring roll, one thread per (sequence, fused channel) (kda_ring.cuh).
template <bool BF16>
__global__ void __launch_bounds__(256) kda_ring_roll_kernel(PrepArgs a) {
    const long Cq = plane_width(a.H, a.Hk, 0);
    const long idx = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= ring_channels(a.H, a.Hk)) return;
    const int p = idx < Cq ? 0 : (idx < 2 * Cq ? 1 : 2);
    ring_roll_one<BF16>(a, blockIdx.y, p, idx - plane_offset(a.H, a.Hk, p));
}

cudaError_t launch_ring_roll(const PrepArgs& a, cudaStream_t s) {
    if (a.conv_w == nullptr || a.seq.N == 0) return cudaSuccess;
    const long C3 = ring_channels(a.H, a.Hk);
    dim3 grid((unsigned)((C3 + 255) / 256), (unsigned)a.seq.N);
    KernelTimer kt(kKRingRoll, s);
    if (a.raw_bf16) kda_ring_roll_kernel<true><<<grid, 256, 0, s>>>(a);
    else kda_ring_roll_kernel<false><<<grid, 256, 0, s>>>(a);
    return cudaGetLastError();
}

template <bool BF16, int GM, bool CONV, bool EXP>
static cudaError_t launch_prep_t(const PrepArgs& a, cudaStream_t s) {
    const long tiles = (a.seq.total_rows + (long)kRun * kPrepWarps - 1) / ((long)kRun * kPrepWarps);
    if (tiles > 0) {
        dim3 grid((unsigned)tiles, (unsigned)a.H);
        KernelTimer kt(kKPrep, s);
        if (a.K <= 4) kda_prep_kernel<BF16, GM, CONV, EXP, 4><<<grid, kPrepThreads, 0, s>>>(a);
        else kda_prep_kernel<BF16, GM, CONV, EXP, kMaxConvK><<<grid, kPrepThreads, 0, s>>>(a);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (CONV) return launch_ring_roll(a, s);
    return cudaSuccess;
}

template <bool BF16, int GM, bool EXP>
static cudaError_t launch_prep_c(const PrepArgs& a, cudaStream_t s) {
    return a.conv_w != nullptr ? launch_prep_t<BF16, GM, true, EXP>(a, s)
                               : launch_prep_t<BF16, GM, false, EXP>(a, s);
}

template <bool BF16>
static cudaError_t launch_prep_b(const PrepArgs& a, cudaStream_t s) {
    switch (a.gate_mode) {
        case 0: return launch_prep_c<BF16, 0, false>(a, s);
        case 1: return launch_prep_c<BF16, 1, false>(a, s);
        case 2: return launch_prep_c<BF16, 0, true>(a, s);
        default: return launch_prep_c<BF16, 1, true>(a, s);
    }
}

cudaError_t launch_prep(const PrepArgs& a, cudaStream_t s) {
    return a.raw_bf16 ? launch_prep_b<true>(a, s) : launch_prep_b<false>(a, s);
}

}  // namespace kda
