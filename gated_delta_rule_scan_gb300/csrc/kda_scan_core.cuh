// kda_scan_core.cuh -- one token of the gated delta rule for four value columns per lane.
//
// Per token and value column j ("memra_engine/kda.rs", memra-engine 0.125.0, module doc and
// kda_core_gated stage 5):
//     S[:, j] <- a * S[:, j]              (a = exp(g): per key-dim channel, or one scalar for GDN)
//     u_j      = v_j - S[:, j] . k
//     S[:, j] <- S[:, j] + k * (beta u_j)
//     o_j      = S[:, j] . q              (the caller applies the readout scale)
//
// Lane layout (shared by the sequential prefill scan and the fused decode/verify kernel, so the
// two compute the same bits).  lane = 8 * grp + r.  The 8 lanes of a group own the same 4 value
// columns c = 0..3; lane r holds key-dim elements i = 4r + 32m + e (m, e = 0..3) of each, as
// float2 pairs S.s[c][2m + h] = (S[i], S[i+1]) with i = 4r + 32m + 2h.  Every k / decay / q value
// a lane loads from shared memory therefore serves 4 columns, which keeps the shared-memory data
// path below the FP32 pipe (one load per 4 x 4 flops instead of per 4 flops).  The elementwise
// work uses Blackwell's paired f32x2 FMA/MUL (one instruction, two lanes of arithmetic).
//
// The dot products reduce over the 8 lanes with a transposed butterfly (reduce8_group8): one
// reduction per token completes that token's S^T k for the 4 columns and the previous token's
// S^T q, so the readout reduction is off the recurrence's critical path.
#pragma once

#include "kda_device.cuh"

namespace kda {

struct Col4 {
    float2 s[4][8];
};

__device__ __forceinline__ float2 lo2(const float4& v) { return make_float2(v.x, v.y); }
__device__ __forceinline__ float2 hi2(const float4& v) { return make_float2(v.z, v.w); }

// Load / store the 4 columns of this lane's group.  col0 points at element i = 0 of column c = 0
// (state layout [.., j, i], so columns are kHeadDim floats apart).
__device__ __forceinline__ void col4_load(Col4& S, const float* col0, int r) {
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const float4 x = __ldcs(reinterpret_cast<const float4*>(col0 + c * kHeadDim + 4 * r + 32 * m));
            S.s[c][2 * m] = lo2(x);
            S.s[c][2 * m + 1] = hi2(x);
        }
}

__device__ __forceinline__ void col4_store(const Col4& S, float* col0, int r) {
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const float4 x = make_float4(S.s[c][2 * m].x, S.s[c][2 * m].y, S.s[c][2 * m + 1].x,
                                         S.s[c][2 * m + 1].y);
            __stcs(reinterpret_cast<float4*>(col0 + c * kHeadDim + 4 * r + 32 * m), x);
        }
}

// Transposed butterfly over the 8 lanes of a group for 8 values per lane: exchanging across
// xor 4, xor 2 and xor 1 halves the values each lane keeps, so lane r ends with the full sum of
// value index r.  Each index is summed over the same lanes in the same order whatever the other
// indices hold.
__device__ __forceinline__ float reduce8_group8(const float (&v)[8], int r) {
    const bool b2 = (r & 4) != 0, b1 = (r & 2) != 0, b0 = (r & 1) != 0;
    float k4[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const float y = __shfl_xor_sync(0xffffffffu, b2 ? v[m] : v[4 + m], 4);
        k4[m] = (b2 ? v[4 + m] : v[m]) + y;
    }
    float k2[2];
#pragma unroll
    for (int m = 0; m < 2; ++m) {
        const float y = __shfl_xor_sync(0xffffffffu, b1 ? k4[m] : k4[2 + m], 2);
        k2[m] = (b1 ? k4[2 + m] : k4[m]) + y;
    }
    const float y = __shfl_xor_sync(0xffffffffu, b0 ? k2[0] : k2[1], 1);
    return (b0 ? k2[1] : k2[0]) + y;
}

__device__ __forceinline__ float sum4(const float2& a, const float2& b) {
    return (a.x + a.y) + (b.x + b.y);
}

// The rows of one token that a lane reads: its 16 key-dim elements of k and of the decay.
struct TokRows {
    float4 k[4];
    float4 a[4];
};

template <bool PER_CHANNEL>
__device__ __forceinline__ void load_rows(TokRows& R, const float* k_row, const float* a_row,
                                          float a_scalar, int r) {
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        R.k[m] = *reinterpret_cast<const float4*>(k_row + 4 * r + 32 * m);
        R.a[m] = PER_CHANNEL ? *reinterpret_cast<const float4*>(a_row + 4 * r + 32 * m)
                             : make_float4(a_scalar, a_scalar, a_scalar, a_scalar);
    }
}

// Token-sequence view of shared memory for col4_tokens: row t of k / decay / q is at
// k + t * row_stride (etc.), v of the group's column c at v + t * v_stride + v_col0 + c,
// beta at beta[t], scalar decay at a_scal[t] (per-head gate), and the readout of column c goes
// to out[t * out_stride + out_col0 + c] (already multiplied by scale).
struct TokView {
    const float* k;
    const float* a;
    const float* q;
    const float* a_scal;
    const float* v;
    const float* beta;
    float* out;
    int row_stride, v_stride, v_col0, out_stride, out_col0;
};

// Runs tokens 0..nt-1 of the view through the recurrence for the 4 columns of this lane's group.
// Per token: decay and S^T k partial sums; one 8-value reduction that completes this token's
// S^T k together with the previous token's S^T q; w = beta (v - S^T k) from the lane owning each
// column, shuffled to the group; rank-1 update and the S^T q partial sums.  The last token's
// readout is completed by the same reduction with zeros in the key slots, so the bits of every
// output depend only on the token, not on how a sequence is split into calls.
// PREFETCH: load the next token's rows during the update (more registers, same values).
template <bool PER_CHANNEL, bool PREFETCH>
__device__ __forceinline__ void col4_tokens(Col4& S, int nt, const TokView& vw, float scale,
                                            int r, int lane) {
    if (nt <= 0) return;
    const int c_own = r & 3;
    const bool key_lane = r < 4;
    float dqp[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    TokRows cur;
    load_rows<PER_CHANNEL>(cur, vw.k, vw.a, PER_CHANNEL ? 0.0f : vw.a_scal[0], r);
    for (int t = 0; t < nt; ++t) {
        float2 acc[4][2];
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[c][0] = acc[c][1] = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const float2 alo = lo2(cur.a[m]), ahi = hi2(cur.a[m]);
            const float2 klo = lo2(cur.k[m]), khi = hi2(cur.k[m]);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                S.s[c][2 * m] = __fmul2_rn(alo, S.s[c][2 * m]);
                S.s[c][2 * m + 1] = __fmul2_rn(ahi, S.s[c][2 * m + 1]);
                acc[c][0] = __ffma2_rn(S.s[c][2 * m], klo, acc[c][0]);
                acc[c][1] = __ffma2_rn(S.s[c][2 * m + 1], khi, acc[c][1]);
            }
        }
        float v8[8];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            v8[c] = sum4(acc[c][0], acc[c][1]);
            v8[4 + c] = dqp[c];
        }
        const float red = reduce8_group8(v8, r);
        if (t > 0 && !key_lane)
            vw.out[(t - 1) * vw.out_stride + vw.out_col0 + c_own] = __fmul_rn(scale, red);
        const float vt = vw.v[t * vw.v_stride + vw.v_col0 + c_own];
        const float w = __fmul_rn(vw.beta[t], vt - red);   // meaningful in key lanes 0..3
        float2 w2[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const float wc = __shfl_sync(0xffffffffu, w, (lane & ~7) | c);
            w2[c] = make_float2(wc, wc);
            acc[c][0] = acc[c][1] = make_float2(0.0f, 0.0f);
        }
        const float4* qrow = reinterpret_cast<const float4*>(vw.q + t * vw.row_stride + 4 * r);
        TokRows nxt;
        if (PREFETCH && t + 1 < nt)
            load_rows<PER_CHANNEL>(nxt, vw.k + (t + 1) * vw.row_stride,
                                   vw.a + (t + 1) * vw.row_stride,
                                   PER_CHANNEL ? 0.0f : vw.a_scal[t + 1], r);
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const float4 q4 = qrow[8 * m];
            const float2 klo = lo2(cur.k[m]), khi = hi2(cur.k[m]);
            const float2 qlo = lo2(q4), qhi = hi2(q4);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                S.s[c][2 * m] = __ffma2_rn(klo, w2[c], S.s[c][2 * m]);
                S.s[c][2 * m + 1] = __ffma2_rn(khi, w2[c], S.s[c][2 * m + 1]);
                acc[c][0] = __ffma2_rn(S.s[c][2 * m], qlo, acc[c][0]);
                acc[c][1] = __ffma2_rn(S.s[c][2 * m + 1], qhi, acc[c][1]);
            }
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) dqp[c] = sum4(acc[c][0], acc[c][1]);
        if (t + 1 < nt) {
            if (PREFETCH)
                cur = nxt;
            else
                load_rows<PER_CHANNEL>(cur, vw.k + (t + 1) * vw.row_stride,
                                       vw.a + (t + 1) * vw.row_stride,
                                       PER_CHANNEL ? 0.0f : vw.a_scal[t + 1], r);
        }
    }
    float v8[8];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        v8[c] = 0.0f;
        v8[4 + c] = dqp[c];
    }
    const float red = reduce8_group8(v8, r);
    if (!key_lane) vw.out[(nt - 1) * vw.out_stride + vw.out_col0 + c_own] = __fmul_rn(scale, red);
}


// ------------------------------------------------------------------------------------------
// The same recurrence with G lanes per group (G = 8 or 16): lane = G * grp + r holds key-dim
// elements i = 4r + 4G m + e (m < 32 / G, e = 0..3) of the group's 4 columns.  G = 16 halves the
// elements per lane (more warps for the same state) while every shared-memory load still feeds
// 4 columns.  The 8-value transposed reduction runs over log2(G) butterfly steps and leaves value
// index r * 8 / G in lane r.
// ------------------------------------------------------------------------------------------

template <int G>
struct ColG {
    float2 s[4][32 / G * 2];
};

template <int G>
__device__ __forceinline__ void colg_load(ColG<G>& S, const float* col0, int r) {
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int m = 0; m < 32 / G; ++m) {
            const float4 x = __ldcs(reinterpret_cast<const float4*>(col0 + c * kHeadDim + 4 * r + 4 * G * m));
            S.s[c][2 * m] = lo2(x);
            S.s[c][2 * m + 1] = hi2(x);
        }
}

template <int G>
__device__ __forceinline__ void colg_store(const ColG<G>& S, float* col0, int r) {
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int m = 0; m < 32 / G; ++m)
            __stcs(reinterpret_cast<float4*>(col0 + c * kHeadDim + 4 * r + 4 * G * m),
                   make_float4(S.s[c][2 * m].x, S.s[c][2 * m].y, S.s[c][2 * m + 1].x,
                               S.s[c][2 * m + 1].y));
}

template <int G>
__device__ __forceinline__ float reduce8_groupG(const float (&v)[8], int r) {
    if constexpr (G == 8) {
        return reduce8_group8(v, r);
    } else {
        const bool b3 = (r & 8) != 0, b2 = (r & 4) != 0, b1 = (r & 2) != 0;
        float k4[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const float y = __shfl_xor_sync(0xffffffffu, b3 ? v[m] : v[4 + m], 8);
            k4[m] = (b3 ? v[4 + m] : v[m]) + y;
        }
        float k2[2];
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            const float y = __shfl_xor_sync(0xffffffffu, b2 ? k4[m] : k4[2 + m], 4);
            k2[m] = (b2 ? k4[2 + m] : k4[m]) + y;
        }
        const float y = __shfl_xor_sync(0xffffffffu, b1 ? k2[0] : k2[1], 2);
        float s1 = (b1 ? k2[1] : k2[0]) + y;
        s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
        return s1;
    }
}

template <bool PER_CHANNEL, int G>
__device__ __forceinline__ void load_rows_g(float4 (&k)[32 / G], float4 (&a)[32 / G],
                                            const float* k_row, const float* a_row,
                                            float a_scalar, int r) {
#pragma unroll
    for (int m = 0; m < 32 / G; ++m) {
        k[m] = *reinterpret_cast<const float4*>(k_row + 4 * r + 4 * G * m);
        a[m] = PER_CHANNEL ? *reinterpret_cast<const float4*>(a_row + 4 * r + 4 * G * m)
                           : make_float4(a_scalar, a_scalar, a_scalar, a_scalar);
    }
}

// col4_tokens with G lanes per group (see above); same contract.
template <bool PER_CHANNEL, bool PREFETCH, int G>
__device__ __forceinline__ void colg_tokens(ColG<G>& S, int nt, const TokView& vw, float scale,
                                            int r, int lane) {
    if (nt <= 0) return;
    constexpr int MC = 32 / G;
    const int idx = r * 8 / G;               // the reduced value this lane ends with
    const int c_own = idx & 3;
    const bool key_lane = idx < 4;
    const bool write_lane = !key_lane && ((r & (G / 8 - 1)) == 0);
    float dqp[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    float4 ck[MC], ca[MC];
    load_rows_g<PER_CHANNEL, G>(ck, ca, vw.k, vw.a, PER_CHANNEL ? 0.0f : vw.a_scal[0], r);
    for (int t = 0; t < nt; ++t) {
        float2 acc[4][2];
#pragma unroll
        for (int m = 0; m < MC; ++m) {
            const float2 alo = lo2(ca[m]), ahi = hi2(ca[m]);
            const float2 klo = lo2(ck[m]), khi = hi2(ck[m]);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                S.s[c][2 * m] = __fmul2_rn(alo, S.s[c][2 * m]);
                S.s[c][2 * m + 1] = __fmul2_rn(ahi, S.s[c][2 * m + 1]);
                if (m == 0) {
                    acc[c][0] = __fmul2_rn(S.s[c][0], klo);
                    acc[c][1] = __fmul2_rn(S.s[c][1], khi);
                } else {
                    acc[c][0] = __ffma2_rn(S.s[c][2 * m], klo, acc[c][0]);
                    acc[c][1] = __ffma2_rn(S.s[c][2 * m + 1], khi, acc[c][1]);
                }
            }
        }
        float v8[8];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            v8[c] = sum4(acc[c][0], acc[c][1]);
            v8[4 + c] = dqp[c];
        }
        const float red = reduce8_groupG<G>(v8, r);
        if (t > 0 && write_lane)
            vw.out[(t - 1) * vw.out_stride + vw.out_col0 + c_own] = __fmul_rn(scale, red);
        const float vt = vw.v[t * vw.v_stride + vw.v_col0 + c_own];
        const float w = __fmul_rn(vw.beta[t], vt - red);   // meaningful in key lanes
        float2 w2[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const float wc = __shfl_sync(0xffffffffu, w, (lane & ~(G - 1)) | (c * G / 8));
            w2[c] = make_float2(wc, wc);
        }
        float4 nk[MC], na[MC];
        if (PREFETCH && t + 1 < nt)
            load_rows_g<PER_CHANNEL, G>(nk, na, vw.k + (t + 1) * vw.row_stride,
                                        vw.a + (t + 1) * vw.row_stride,
                                        PER_CHANNEL ? 0.0f : vw.a_scal[t + 1], r);
#pragma unroll
        for (int m = 0; m < MC; ++m) {
            const float4 q4 = *reinterpret_cast<const float4*>(vw.q + t * vw.row_stride + 4 * r + 4 * G * m);
            const float2 klo = lo2(ck[m]), khi = hi2(ck[m]);
            const float2 qlo = lo2(q4), qhi = hi2(q4);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                S.s[c][2 * m] = __ffma2_rn(klo, w2[c], S.s[c][2 * m]);
                S.s[c][2 * m + 1] = __ffma2_rn(khi, w2[c], S.s[c][2 * m + 1]);
                if (m == 0) {
                    acc[c][0] = __fmul2_rn(S.s[c][0], qlo);
                    acc[c][1] = __fmul2_rn(S.s[c][1], qhi);
                } else {
                    acc[c][0] = __ffma2_rn(S.s[c][2 * m], qlo, acc[c][0]);
                    acc[c][1] = __ffma2_rn(S.s[c][2 * m + 1], qhi, acc[c][1]);
                }
            }
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) dqp[c] = sum4(acc[c][0], acc[c][1]);
        if (t + 1 < nt) {
            if (PREFETCH) {
#pragma unroll
                for (int m = 0; m < MC; ++m) { ck[m] = nk[m]; ca[m] = na[m]; }
            } else {
                load_rows_g<PER_CHANNEL, G>(ck, ca, vw.k + (t + 1) * vw.row_stride,
                                            vw.a + (t + 1) * vw.row_stride,
                                            PER_CHANNEL ? 0.0f : vw.a_scal[t + 1], r);
            }
        }
    }
    float v8[8];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        v8[c] = 0.0f;
        v8[4 + c] = dqp[c];
    }
    const float red = reduce8_groupG<G>(v8, r);
    if (write_lane) vw.out[(nt - 1) * vw.out_stride + vw.out_col0 + c_own] = __fmul_rn(scale, red);
}

}  // namespace kda
