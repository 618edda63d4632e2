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
// Layout: one CTA per (tile of kTileRows consecutive packed rows, head); one thread per channel
// of the head, carrying the three planes' conv windows in registers while it walks the tile, so
// each raw sample is read once per tile (plus K-1 halo rows).  A tile may straddle sequence
// boundaries (varlen): the window restarts from the next sequence's ring.  The ring itself is
// rewritten by a second, tiny kernel launched after this one on the same stream, so ring_in and
// ring_out may be the same buffer.
#include "kda_device.cuh"
#include "kda_internal.h"

namespace kda {

constexpr int kTileRows = 16;
constexpr int kPrepThreads = kHeadDim;  // one thread per channel of the head

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
    // largest n with cu[n] <= r, then skip empty sequences forward
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

// Fill the window of one plane with the K-1 samples that precede position p of sequence s:
// win[kMaxConvK - d] = sample at position p - d (d = 1..R), from the raw rows when p - d >= 0 and
// from the ring (oldest slot first) otherwise.  The next window_push appends position p.
template <bool BF16>
__device__ __forceinline__ void window_fill(float (&win)[kMaxConvK], const void* raw, long C,
                                            int c_plane, const float* ring_in, long ring_row,
                                            int R, SeqCursor s, long p) {
#pragma unroll
    for (int m = 0; m < kMaxConvK; ++m) {
        const int d = kMaxConvK - m;
        float x = 0.0f;
        if (d <= R) {
            const long pos = p - d;
            x = pos >= 0 ? load_raw<BF16>(raw, (s.begin + pos) * C + c_plane)
                         : ring_in[ring_row + (R + pos)];
        }
        win[m] = x;
    }
}

// EXP: write the decay factor exp(g) instead of the log-decay g.
template <bool BF16, int GATE_MODE, bool CONV, bool EXP>
__global__ void __launch_bounds__(kPrepThreads) kda_prep_kernel(PrepArgs a) {
    __shared__ float xs[2][kTileRows][kHeadDim];   // pre-norm q, k of the tile
    __shared__ float part[2][kPrepThreads / 32][kTileRows];
    __shared__ float inv_s[2][kTileRows];

    const int h = blockIdx.y;
    const int i = threadIdx.x;              // channel within the head
    const int H = a.H;
    const long C = (long)H * kHeadDim;
    const int c = h * kHeadDim + i;         // channel within a plane
    const long r0 = (long)blockIdx.x * kTileRows;
    const long rows = a.seq.total_rows;
    const int nt = (int)min((long)kTileRows, rows - r0);
    const int K = a.K, R = a.K - 1;
    const int warp = i >> 5, lane = i & 31;

    // conv weights of this channel for the three planes, aligned to the window's end
    float wq[kMaxConvK], wk[kMaxConvK], wv[kMaxConvK];
    float winq[kMaxConvK], wink[kMaxConvK], winv[kMaxConvK];
#pragma unroll
    for (int m = 0; m < kMaxConvK; ++m) {
        wq[m] = wk[m] = wv[m] = 0.0f;
        winq[m] = wink[m] = winv[m] = 0.0f;
    }
    SeqCursor s = seq_of_row(a.seq, r0);
    if constexpr (CONV) {
#pragma unroll
        for (int m = 0; m < kMaxConvK; ++m) {
            const int j = m - (kMaxConvK - K);
            if (j >= 0) {
                wq[m] = a.conv_w[(0 * C + c) * K + j];
                wk[m] = a.conv_w[(1 * C + c) * K + j];
                wv[m] = a.conv_w[(2 * C + c) * K + j];
            }
        }
        const long p = r0 - s.begin;
        const long rr = (long)s.n * 3 * C * R;
        window_fill<BF16>(winq, a.q_raw, C, c, a.ring_in, rr + (0 * C + c) * R, R, s, p);
        window_fill<BF16>(wink, a.k_raw, C, c, a.ring_in, rr + (1 * C + c) * R, R, s, p);
        window_fill<BF16>(winv, a.v_raw, C, c, a.ring_in, rr + (2 * C + c) * R, R, s, p);
    }
    float rate = 0.0f;
    if constexpr (GATE_MODE == 0) rate = expf(a.a_log[h]);

    for (int t = 0; t < nt; ++t) {
        const long r = r0 + t;
        float xq, xk;
        if constexpr (CONV) {
            if (r >= s.end) {  // crossed into the next non-empty sequence: restart the windows
                do { s = seq_next(a.seq, s); } while (s.end <= r);
                const long rr = (long)s.n * 3 * C * R;
                window_fill<BF16>(winq, a.q_raw, C, c, a.ring_in, rr + (0 * C + c) * R, R, s, 0);
                window_fill<BF16>(wink, a.k_raw, C, c, a.ring_in, rr + (1 * C + c) * R, R, s, 0);
                window_fill<BF16>(winv, a.v_raw, C, c, a.ring_in, rr + (2 * C + c) * R, R, s, 0);
            }
            window_push(winq, load_raw<BF16>(a.q_raw, r * C + c));
            window_push(wink, load_raw<BF16>(a.k_raw, r * C + c));
            window_push(winv, load_raw<BF16>(a.v_raw, r * C + c));
            xq = silu_f(conv_taps_f(wq, winq, K));
            xk = silu_f(conv_taps_f(wk, wink, K));
            a.v_hat[r * C + c] = silu_f(conv_taps_f(wv, winv, K));
        } else {
            xq = load_raw<BF16>(a.q_raw, r * C + c);
            xk = load_raw<BF16>(a.k_raw, r * C + c);
            a.v_hat[r * C + c] = load_raw<BF16>(a.v_raw, r * C + c);
        }
        xs[0][t][i] = xq;
        xs[1][t][i] = xk;
        if constexpr (GATE_MODE == 0) {
            const float gl = kda_gate_f(a.f_raw[r * C + c], a.dt_bias[c], rate, a.gate_lb);
            a.g[r * C + c] = EXP ? expf(gl) : gl;
        }
    }
    if (i < nt) {
        const long r = r0 + i;
        a.beta[r * H + h] = sigmoid_f(a.beta_raw[r * H + h]);
        if constexpr (GATE_MODE == 1) {
            const float gl = gdn_gate_f(a.f_raw[r * H + h], a.dt_bias[h], a.a_log[h]);
            a.g[r * H + h] = EXP ? expf(gl) : gl;
        }
    }

    // l2 norm of q and k over the head's 128 channels, one reduction per token
    for (int t = 0; t < nt; ++t) {
        const float xq = xs[0][t][i], xk = xs[1][t][i];
        const float sq = warp_sum(__fmul_rn(xq, xq));
        const float sk = warp_sum(__fmul_rn(xk, xk));
        if (lane == 0) { part[0][warp][t] = sq; part[1][warp][t] = sk; }
    }
    __syncthreads();
    if (i < 2 * kTileRows) {
        const int pl = i / kTileRows, t = i % kTileRows;
        const float p4[4] = {part[pl][0][t], part[pl][1][t], part[pl][2][t], part[pl][3][t]};
        inv_s[pl][t] = l2_inv_f(head_sum4(p4), a.l2_eps);
    }
    __syncthreads();
    for (int t = 0; t < nt; ++t) {
        const long r = r0 + t;
        a.q_hat[r * C + c] = __fmul_rn(xs[0][t][i], inv_s[0][t]);
        a.k_hat[r * C + c] = __fmul_rn(xs[1][t][i], inv_s[1][t]);
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
        kda_prep_kernel<BF16, GM, CONV, EXP><<<grid, kPrepThreads, 0, s>>>(a);
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
