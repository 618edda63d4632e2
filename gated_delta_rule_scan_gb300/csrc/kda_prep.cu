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
// Layout: one CTA per (tile of kTileRows consecutive packed rows, head); 64 threads, each owning
// the channel pair (2i, 2i+1) of the head in all three planes, carrying the planes' conv windows
// in registers while it walks the tile, so each raw sample is read once per tile (plus K-1 halo
// rows).  Raw rows are read as bf16x2 / float2 pairs and kPrefetch rows of loads are issued
// before any of them is used, so each thread keeps several loads in flight.  A tile may straddle
// sequence boundaries (varlen): the windows restart from the next sequence's ring.  The ring is
// rewritten by a second, tiny kernel launched after this one on the same stream, so ring_in and
// ring_out may be the same buffer.
#include "kda_device.cuh"
#include "kda_internal.h"

namespace kda {

constexpr int kTileRows = 32;
constexpr int kPrepThreads = kHeadDim / 2;  // one channel pair per thread
constexpr int kPrefetch = 8;                // rows of loads issued ahead

struct SeqCursor {
    int n;        // sequence index
    long begin;   // first packed row of the sequence
    long end;     // one past its last row
};

// Sequence containing packed row r (rows of empty sequences are skipped).
__device__ __forceinline__ SeqCursor seq_of_row(const SeqLayout& L, long r) {
    SeqCursor s;
    if (L.cu_seqlens == nullptr) {
        s.n = (int)(r / L.T_uniform);
        s.begin = (long)s.n * L.T_uniform;
        s.end = s.begin + L.T_uniform;
        return s;
    }
    // largest n with cu[n] <= r: its sequence is non-empty and contains r
    int lo = 0, hi = L.N;  // invariant: cu[lo] <= r < cu[hi]
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if ((long)L.cu_seqlens[mid] <= r) lo = mid; else hi = mid;
    }
    s.n = lo;
    s.begin = L.cu_seqlens[lo];
    s.end = L.cu_seqlens[lo + 1];
    return s;
}

__device__ __forceinline__ SeqCursor seq_next(const SeqLayout& L, SeqCursor s) {
    SeqCursor t;
    t.n = s.n + 1;
    if (L.cu_seqlens == nullptr) {
        t.begin = s.end;
        t.end = s.end + L.T_uniform;
    } else {
        t.begin = L.cu_seqlens[t.n];
        t.end = L.cu_seqlens[t.n + 1];
    }
    return t;
}

// Fill the windows of one plane's channel pair with the K-1 samples that precede position p of
// sequence s: win[KW - d] = sample at position p - d (d = 1..R), from the raw rows when
// p - d >= 0 and from the ring (oldest slot first) otherwise.  window_push then appends p.
template <bool BF16, int KW>
__device__ __forceinline__ void window_fill2(float (&w0)[KW], float (&w1)[KW], const void* raw,
                                             long C, int c, const float* ring_in, long ring_row0,
                                             int R, SeqCursor s, long p) {
#pragma unroll
    for (int m = 0; m < KW; ++m) {
        const int d = KW - m;
        float2 x = make_float2(0.0f, 0.0f);
        if (d <= R) {
            const long pos = p - d;
            if (pos >= 0) {
                x = load_raw2<BF16>(raw, (s.begin + pos) * C + c);
            } else {
                x.x = ring_in[ring_row0 + (R + pos)];
                x.y = ring_in[ring_row0 + R + (R + pos)];
            }
        }
        w0[m] = x.x;
        w1[m] = x.y;
    }
}

// EXP: write the decay factor exp(g) instead of the log-decay g.  KW: register window width
// (4 when K <= 4, else 8).
template <bool BF16, int GATE_MODE, bool CONV, bool EXP, int KW>
__global__ void __launch_bounds__(kPrepThreads) kda_prep_kernel(PrepArgs a) {
    __shared__ __align__(16) float xs[2][kTileRows][kHeadDim];   // pre-norm q, k of the tile
    __shared__ float part[2][2][kTileRows];
    __shared__ float inv_s[2][kTileRows];

    const int h = blockIdx.y;
    const int tid = threadIdx.x;
    const int i0 = 2 * tid;                   // channel pair within the head
    const int H = a.H;
    const long C = (long)H * kHeadDim;
    const int c = h * kHeadDim + i0;          // first channel of the pair within a plane
    const long r0 = (long)blockIdx.x * kTileRows;
    const int nt = (int)min((long)kTileRows, a.seq.total_rows - r0);
    const int K = a.K, R = a.K - 1;
    const int warp = tid >> 5, lane = tid & 31;

    float wq[2][KW], wk[2][KW], wv[2][KW];
    float winq[2][KW], wink[2][KW], winv[2][KW];
#pragma unroll
    for (int m = 0; m < KW; ++m)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            wq[e][m] = wk[e][m] = wv[e][m] = 0.0f;
            winq[e][m] = wink[e][m] = winv[e][m] = 0.0f;
        }
    SeqCursor s = seq_of_row(a.seq, r0);
    const bool single = s.end >= r0 + nt;     // the whole tile lies in one sequence
    auto fill = [&](long p) {
        const long rr = (long)s.n * 3 * C * R;
        window_fill2<BF16, KW>(winq[0], winq[1], a.q_raw, C, c, a.ring_in, rr + (0 * C + c) * R, R, s, p);
        window_fill2<BF16, KW>(wink[0], wink[1], a.k_raw, C, c, a.ring_in, rr + (1 * C + c) * R, R, s, p);
        window_fill2<BF16, KW>(winv[0], winv[1], a.v_raw, C, c, a.ring_in, rr + (2 * C + c) * R, R, s, p);
    };
    if constexpr (CONV) {
#pragma unroll
        for (int m = 0; m < KW; ++m) {
            const int j = m - (KW - K);
            if (j >= 0) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    wq[e][m] = a.conv_w[(0 * C + c + e) * K + j];
                    wk[e][m] = a.conv_w[(1 * C + c + e) * K + j];
                    wv[e][m] = a.conv_w[(2 * C + c + e) * K + j];
                }
            }
        }
        fill(r0 - s.begin);
    }
    float rate = 0.0f;
    float2 dtb = make_float2(0.0f, 0.0f);
    if constexpr (GATE_MODE == 0) {
        rate = expf(a.a_log[h]);
        dtb = *reinterpret_cast<const float2*>(a.dt_bias + c);
    }

    for (int t0 = 0; t0 < nt; t0 += kPrefetch) {
        float2 rq[kPrefetch], rk[kPrefetch], rv[kPrefetch], fr[kPrefetch];
#pragma unroll
        for (int u = 0; u < kPrefetch; ++u) {
            if (t0 + u < nt) {
                const long r = r0 + t0 + u;
                rq[u] = load_raw2<BF16>(a.q_raw, r * C + c);
                rk[u] = load_raw2<BF16>(a.k_raw, r * C + c);
                rv[u] = load_raw2<BF16>(a.v_raw, r * C + c);
                if (GATE_MODE == 0) fr[u] = *reinterpret_cast<const float2*>(a.f_raw + r * C + c);
            }
        }
#pragma unroll
        for (int u = 0; u < kPrefetch; ++u) {
            const int t = t0 + u;
            if (t < nt) {
                const long r = r0 + t;
                float2 xq, xk, xv;
                if constexpr (CONV) {
                    if (!single && r >= s.end) {  // next non-empty sequence: restart the windows
                        do { s = seq_next(a.seq, s); } while (s.end <= r);
                        fill(0);
                    }
                    window_push(winq[0], rq[u].x); window_push(winq[1], rq[u].y);
                    window_push(wink[0], rk[u].x); window_push(wink[1], rk[u].y);
                    window_push(winv[0], rv[u].x); window_push(winv[1], rv[u].y);
                    xq = make_float2(silu_f(conv_taps_f(wq[0], winq[0], K)),
                                     silu_f(conv_taps_f(wq[1], winq[1], K)));
                    xk = make_float2(silu_f(conv_taps_f(wk[0], wink[0], K)),
                                     silu_f(conv_taps_f(wk[1], wink[1], K)));
                    xv = make_float2(silu_f(conv_taps_f(wv[0], winv[0], K)),
                                     silu_f(conv_taps_f(wv[1], winv[1], K)));
                } else {
                    xq = rq[u];
                    xk = rk[u];
                    xv = rv[u];
                }
                *reinterpret_cast<float2*>(a.v_hat + r * C + c) = xv;
                *reinterpret_cast<float2*>(&xs[0][t][i0]) = xq;
                *reinterpret_cast<float2*>(&xs[1][t][i0]) = xk;
                if constexpr (GATE_MODE == 0) {
                    float g0 = kda_gate_f(fr[u].x, dtb.x, rate, a.gate_lb);
                    float g1 = kda_gate_f(fr[u].y, dtb.y, rate, a.gate_lb);
                    if (EXP) { g0 = decay_f(g0); g1 = decay_f(g1); }
                    *reinterpret_cast<float2*>(a.g + r * C + c) = make_float2(g0, g1);
                }
            }
        }
    }
    if (tid < nt) {
        const long r = r0 + tid;
        a.beta[r * H + h] = sigmoid_f(a.beta_raw[r * H + h]);
        if constexpr (GATE_MODE == 1) {
            const float gl = gdn_gate_f(a.f_raw[r * H + h], a.dt_bias[h], a.a_log[h]);
            a.g[r * H + h] = EXP ? decay_f(gl) : gl;
        }
    }
    __syncthreads();

    // l2 norm of q and k over the head's 128 channels, one reduction per token
    for (int t = 0; t < nt; ++t) {
        const float2 xq = *reinterpret_cast<const float2*>(&xs[0][t][i0]);
        const float2 xk = *reinterpret_cast<const float2*>(&xs[1][t][i0]);
        const float sq = warp_sum(pair_sumsq(xq.x, xq.y));
        const float sk = warp_sum(pair_sumsq(xk.x, xk.y));
        if (lane == 0) { part[0][warp][t] = sq; part[1][warp][t] = sk; }
    }
    __syncthreads();
    {
        const int pl = tid / kTileRows, t = tid % kTileRows;   // 64 threads = 2 planes x 32 rows
        if (t < nt) inv_s[pl][t] = l2_inv_f(part[pl][0][t] + part[pl][1][t], a.l2_eps);
    }
    __syncthreads();
    for (int t = 0; t < nt; ++t) {
        const long r = r0 + t;
        const float2 xq = *reinterpret_cast<const float2*>(&xs[0][t][i0]);
        const float2 xk = *reinterpret_cast<const float2*>(&xs[1][t][i0]);
        *reinterpret_cast<float2*>(a.q_hat + r * C + c) =
            make_float2(__fmul_rn(xq.x, inv_s[0][t]), __fmul_rn(xq.y, inv_s[0][t]));
        *reinterpret_cast<float2*>(a.k_hat + r * C + c) =
            make_float2(__fmul_rn(xk.x, inv_s[1][t]), __fmul_rn(xk.y, inv_s[1][t]));
    }
}

// Ring roll: ring_out[n][pc][s] = xt[L_n + s], xt = (ring_in[n][pc][0..R-1], raw rows of n).
// One thread per (sequence, fused channel); each reads all its old slots before writing, so the
// roll is safe in place.
template <bool BF16>
__global__ void __launch_bounds__(256) kda_ring_roll_kernel(PrepArgs a) {
    const long C = (long)a.H * kHeadDim;
    const long idx = (long)blockIdx.x * blockDim.x + threadIdx.x;
    const int n = blockIdx.y;
    if (idx >= 3 * C) return;
    const int p = (int)(idx / C);
    const long c = idx % C;
    const int R = a.K - 1;
    long begin, end;
    if (a.seq.cu_seqlens == nullptr) {
        begin = (long)n * a.seq.T_uniform;
        end = begin + a.seq.T_uniform;
    } else {
        begin = a.seq.cu_seqlens[n];
        end = a.seq.cu_seqlens[n + 1];
    }
    const long Ln = end - begin;
    const void* raw = p == 0 ? a.q_raw : (p == 1 ? a.k_raw : a.v_raw);
    const long base = ((long)n * 3 * C + idx) * R;
    float old[kMaxConvK - 1];
#pragma unroll
    for (int s2 = 0; s2 < kMaxConvK - 1; ++s2) old[s2] = s2 < R ? a.ring_in[base + s2] : 0.0f;
#pragma unroll
    for (int s2 = 0; s2 < kMaxConvK - 1; ++s2) {
        if (s2 < R) {
            const long pos = Ln + s2;  // index into xt
            float x;
            if (pos < R) {
                x = 0.0f;
#pragma unroll
                for (int m = 0; m < kMaxConvK - 1; ++m) if (m == pos) x = old[m];
            } else {
                x = load_raw<BF16>(raw, (begin + pos - R) * C + c);
            }
            a.ring_out[base + s2] = x;
        }
    }
}

template <bool BF16, int GM, bool CONV, bool EXP>
static cudaError_t launch_prep_t(const PrepArgs& a, cudaStream_t s) {
    const long tiles = (a.seq.total_rows + kTileRows - 1) / kTileRows;
    if (tiles > 0) {
        dim3 grid((unsigned)tiles, (unsigned)a.H);
        if (a.K <= 4) kda_prep_kernel<BF16, GM, CONV, EXP, 4><<<grid, kPrepThreads, 0, s>>>(a);
        else kda_prep_kernel<BF16, GM, CONV, EXP, kMaxConvK><<<grid, kPrepThreads, 0, s>>>(a);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (CONV && a.seq.N > 0) {
        const long C3 = 3L * a.H * kHeadDim;
        dim3 grid((unsigned)((C3 + 255) / 256), (unsigned)a.seq.N);
        kda_ring_roll_kernel<BF16><<<grid, 256, 0, s>>>(a);
        return cudaGetLastError();
    }
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
