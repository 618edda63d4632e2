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
// The two dot products reduce over the 8 lanes with a transposed butterfly: after exchanging
// across xor 4 and xor 2 each lane keeps one column's partial sum, and xor 1 completes it, so
// lanes 2c and 2c+1 of a group hold column c's full sum (4 shuffles instead of 12).
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

// Transposed butterfly over the 8 lanes of a group: d[c] are this lane's partial sums of the 4
// columns; returns the full sum of column (r >> 1) & 3.
__device__ __forceinline__ float reduce4_group8(const float (&d)[4], int r) {
    const bool b2 = (r & 4) != 0, b1 = (r & 2) != 0;
    const float x0 = b2 ? d[0] : d[2];
    const float x1 = b2 ? d[1] : d[3];
    const float y0 = __shfl_xor_sync(0xffffffffu, x0, 4);
    const float y1 = __shfl_xor_sync(0xffffffffu, x1, 4);
    const float k0 = (b2 ? d[2] : d[0]) + y0;
    const float k1 = (b2 ? d[3] : d[1]) + y1;
    const float x = b1 ? k0 : k1;
    const float y = __shfl_xor_sync(0xffffffffu, x, 2);
    float s = (b1 ? k1 : k0) + y;
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    return s;
}

__device__ __forceinline__ float sum4(const float2& a, const float2& b) {
    return (a.x + a.y) + (b.x + b.y);
}

// One token.  k_row, q_row: the token's 128 key-dim values (shared memory, 16-byte aligned);
// a_row: its 128 decay factors (PER_CHANNEL) or ignored (a_scalar used instead); v_own: v of the
// lane's own column (r >> 1) & 3; beta: the token's beta.  Returns S^T q (unscaled) of the own
// column; lanes 2c and 2c+1 of a group return the same bits for column c.
template <bool PER_CHANNEL>
__device__ __forceinline__ float col4_token(Col4& S, const float* k_row, const float* a_row,
                                            float a_scalar, const float* q_row, float v_own,
                                            float beta, int r, int lane) {
    float4 k4[4];
    float2 acc[4][2];
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[c][0] = acc[c][1] = make_float2(0.0f, 0.0f);
    // decay, then S^T k with the decayed state
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        k4[m] = *reinterpret_cast<const float4*>(k_row + 4 * r + 32 * m);
        float2 alo, ahi;
        if (PER_CHANNEL) {
            const float4 a4 = *reinterpret_cast<const float4*>(a_row + 4 * r + 32 * m);
            alo = lo2(a4);
            ahi = hi2(a4);
        } else {
            alo = ahi = make_float2(a_scalar, a_scalar);
        }
        const float2 klo = lo2(k4[m]), khi = hi2(k4[m]);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            S.s[c][2 * m] = __fmul2_rn(alo, S.s[c][2 * m]);
            S.s[c][2 * m + 1] = __fmul2_rn(ahi, S.s[c][2 * m + 1]);
            acc[c][0] = __ffma2_rn(S.s[c][2 * m], klo, acc[c][0]);
            acc[c][1] = __ffma2_rn(S.s[c][2 * m + 1], khi, acc[c][1]);
        }
    }
    float d[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) d[c] = sum4(acc[c][0], acc[c][1]);
    const float dk = reduce4_group8(d, r);
    const float w = __fmul_rn(beta, v_own - dk);
    // every lane of the group needs the 4 columns' w: column c's is held by lane 2c of the group
    float2 w2[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const float wc = __shfl_sync(0xffffffffu, w, (lane & ~7) | (2 * c));
        w2[c] = make_float2(wc, wc);
        acc[c][0] = acc[c][1] = make_float2(0.0f, 0.0f);
    }
    // rank-1 update, then S^T q with the updated state
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const float4 q4 = *reinterpret_cast<const float4*>(q_row + 4 * r + 32 * m);
        const float2 klo = lo2(k4[m]), khi = hi2(k4[m]);
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
    for (int c = 0; c < 4; ++c) d[c] = sum4(acc[c][0], acc[c][1]);
    return reduce4_group8(d, r);
}

}  // namespace kda
