#pragma once
// kda_chunk_common.cuh -- shared by the chunked (UT / WY) form of the per-channel gated delta rule on the
// tcgen05 tensor cores: a parallel intra-chunk kernel and a sequential inter-chunk kernel.
//
// Method: "memra_engine/kda.rs" (memra-engine 0.125.0) module doc, the chunked twin: KDA's decay
// is per channel, so the chunk form carries a per-channel cumulative log gate Gcum[t][i] with k
// scaled by exp(-Gcum) and q by exp(+Gcum).  For one chunk of C tokens with start state S0
// (rows = key dim), inclusive cumulative gate G_t = sum_{s<=t} g_s (per channel) and
// Gamma_t = exp(G_t), the C sequential steps
//     S <- Diag(e^{g_t}) S;  u_t = v_t - S^T k_t;  S <- S + beta_t k_t u_t^T;  o_t = scale S^T q_t
// are reproduced exactly (up to rounding) by
//     A[t][s]   = beta_t (k_t * Gamma_t) . (k_s / Gamma_s)       s < t   (strictly lower)
//     Aqk[t][s] = (q_t * Gamma_t) . (k_s / Gamma_s)              s <= t
//     Tm        = (I + A)^{-1}
//     W         = Tm diag(beta) (K * Gamma),   U = Tm diag(beta) V
//     U'        = U - W S0
//     O         = scale [ (Q * Gamma) S0 + Aqk U' ]
//     S_C       = Diag(Gamma_C) S0 + (K * Gamma_C / Gamma)^T U'
// (the algebra is pinned against the sequential oracle at every chunk size by the test suite).
//
// GB300 design.  Chunks are kCc = 32 tokens.  Everything that does not depend on the state -- A,
// Aqk, Tm, W, U and the decayed k / q -- is computed by kda_chunk_intra_kernel for every
// (chunk, head) at once, in parallel over the whole GPU, and written to the caller's workspace as
// ready-to-use tensor-core operand images.  kda_chunk_inter_kernel then walks each (sequence,
// head)'s chunks in order with only two dependent MMA stages per chunk:
//     [O1^T | X^T]  = S^T   (Q e^G | W)^T          M=128 (value rows), N=64,  K=128
//     U'^T          = U^T - X^T
//     [dS^T | O2^T] = U'^T  (K e^{G_C-G} | Aqk)    M=128,              N=160, K=32
//     S^T <- S^T Diag(e^{G_C}) + dS^T,   o = scale (O1 + O2)
// with S^T and U'^T held in tensor memory as the MMAs' A operands and the state row kept in f32
// registers.  Precision.  The intra kernel's products (A, Aqk, W, U) take both operands as bf16
// hi + lo and sum hi*hi + hi*lo + lo*hi (about 16 significant bits).  The chain's two MMAs take
// the f32 state and U' split as f16 hi + lo (22 bits) against single f16 images of their other
// operand (11 bits): two products per K-step instead of three, 20 MMA instructions per chunk
// instead of 30.  The chain's error is then the f16 rounding of (Q e^G | W) and
// (K e^{G_C-G} | Aqk), a few 1e-4 relative at every length (measured 2.4e-4 .. 4.8e-4 on the
// stated workloads, inside the 1e-3 parity bound), where bf16 images there gave 2e-3 .. 3e-3.
// Every operand of those images is at most 1 in magnitude (e^{G} <= 1, l2-normalised q and k)
// or a small multiple (W); the state and U' must stay below f16's 65504.  Shared-memory operands
// are K-major, no swizzle, 8-row x 16-byte core matrices (kda_tc.cuh).
//
// Range.  The intra-chunk products pair k_t e^{G_t - c} with k_s e^{c - G_s}, c = half the
// chunk's total gate per channel, so each factor stays below e^{|G_C|/2}.  For the per-channel
// gate the chunk's total log-decay must stay above -170 on every channel (the KDA gate's lower
// bound of -5 per token gives -160 over 32 tokens); beyond that the kernel raises the device error
// word.  The per-head (GDN) gate forms A and Aqk from unscaled k and q and applies the scalar
// e^{G_t - G_s} <= 1 after the MMA, so it has no range limit.
#include "kda_internal.h"
#include "kda_tc.cuh"

namespace kda {

constexpr int kCc = 32;                  // tokens per chunk
constexpr int kThr = 128;                // both kernels: thread = TMEM lane
constexpr uint32_t kSbo128 = 2048;       // 8-row group stride, K = 128 bf16 image
constexpr uint32_t kSbo32 = 512;         // 8-row group stride, K = 32 bf16 image
// The same for MMA-b's B operand in shared memory, padded by 16 bytes so that the column images'
// 8-byte stores from 32 lanes (rows 4 apart) spread over the banks instead of landing on two.
constexpr uint32_t kSboKt = 528;
constexpr int kDevErrRange = 2;          // device error word bit: chunk gate outside f32 range

// ---- workspace block of one (chunk, head) ----------------------------------------------------
// The inter kernel's two B operands are single f16 images (its MMAs pair them with the state and
// U' split into f16 hi + lo, two products per K-step); U and e^{G_C} are f32.
constexpr int kQWBytes = 64 * 128 * 2;             // [Q e^G (32 rows) ; W (32 rows)] x 128 k, f16
constexpr int kB2Bytes = (128 + kCc) * kCc * 2;    // [(K e^{G_C-G})^T (128 rows) ; Aqk (32)] x 32, f16
constexpr int kUTBytes = 128 * kCc * 4;            // U f32 [32 t][128 v]
constexpr int kEGBytes = 128 * 4;                  // e^{G_C} f32 [128]
constexpr int kOffQW = 0;
constexpr int kOffB2 = kQWBytes;
constexpr int kOffUT = kOffB2 + kB2Bytes;
constexpr int kOffEG = kOffUT + kUTBytes;
constexpr int kBlkBytes = kOffEG + kEGBytes;       // 43520
static_assert(kBlkBytes % 128 == 0, "workspace blocks stay 128-byte aligned");
static_assert(kBlkBytes == kChunkBlockBytes, "the workspace sizing uses the same block size");
constexpr int kHeaderAlign = 256;

// store 8 values (one 16-byte core-matrix row) as f16 at byte offset off of an image
__device__ __forceinline__ void put8h(unsigned char* img, uint32_t off, const float (&x)[8]) {
    *reinterpret_cast<uint4*>(img + off) =
        make_uint4(f16x2_rn(x[0], x[1]), f16x2_rn(x[2], x[3]), f16x2_rn(x[4], x[5]),
                   f16x2_rn(x[6], x[7]));
}

// store 8 values (one 16-byte core-matrix row) as bf16 hi / lo at byte offset off of two images
__device__ __forceinline__ void put8x(unsigned char* hi_img, unsigned char* lo_img, uint32_t off,
                                      const float (&x)[8]) {
    uint4 hi, lo;
    split_bf16x2(x[0], x[1], hi.x, lo.x);
    split_bf16x2(x[2], x[3], hi.y, lo.y);
    split_bf16x2(x[4], x[5], hi.z, lo.z);
    split_bf16x2(x[6], x[7], hi.w, lo.w);
    *reinterpret_cast<uint4*>(hi_img + off) = hi;
    *reinterpret_cast<uint4*>(lo_img + off) = lo;
}

__device__ __forceinline__ void put1x(unsigned char* hi_img, unsigned char* lo_img, uint32_t off,
                                      float x) {
    __nv_bfloat16 h, l;
    split_bf16(x, h, l);
    *reinterpret_cast<__nv_bfloat16*>(hi_img + off) = h;
    *reinterpret_cast<__nv_bfloat16*>(lo_img + off) = l;
}

// D (+)= A * B^T, bf16x3, both operands in shared memory
__device__ __forceinline__ void mma3_ss(uint32_t d, uint64_t a_hi, uint64_t a_lo, uint64_t b_hi,
                                        uint64_t b_lo, int nks, uint32_t idesc) {
    const uint64_t as[3] = {a_hi, a_hi, a_lo};
    const uint64_t bs[3] = {b_hi, b_lo, b_hi};
#pragma unroll
    for (int p = 0; p < 3; ++p)
        for (int ks = 0; ks < nks; ++ks)
            tc_mma_ss(d, tc_desc_advance(as[p], 256 * ks), tc_desc_advance(bs[p], 256 * ks), idesc,
                      p > 0 || ks > 0);
}

// D[tmem] (+)= A[tmem] * B[smem desc]^T, issued by one thread
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                         uint32_t idesc, bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate)
        : "memory");
}

// D = A * B^T, f16 x 2: A in tensor memory split as hi (at a_hi) + lo (at a_lo), 8 columns per
// K-step of 16; B one f16 image in shared memory; the first product starts the sum
__device__ __forceinline__ void mma2_ts(uint32_t d, uint32_t a_hi, uint32_t a_lo, uint64_t b,
                                        int nks, uint32_t idesc) {
    for (int ks = 0; ks < nks; ++ks) {
        tc_mma_ts(d, a_hi + 8 * ks, tc_desc_advance(b, 256 * ks), idesc, ks > 0);
        tc_mma_ts(d, a_lo + 8 * ks, tc_desc_advance(b, 256 * ks), idesc, true);
    }
}

__device__ __forceinline__ void seq_range(const SeqLayout& L, int n, long& begin, long& end) {
    if (L.cu_seqlens == nullptr) {
        begin = (long)n * L.T_uniform;
        end = begin + L.T_uniform;
    } else {
        begin = L.cu_seqlens[n];
        end = L.cu_seqlens[n + 1];
    }
}

// first global chunk index of sequence n
__device__ __forceinline__ long chunk_base(const SeqLayout& L, const int* chunk_off, int n) {
    if (L.cu_seqlens == nullptr) return (long)n * ((L.T_uniform + kCc - 1) / kCc);
    return chunk_off[n];
}

struct __align__(128) IntraSmem {
    // MMA-a A operand [K e^{G-c} ; Q e^{G-c}] (64 rows, K = 128 channels).  Its 128-row
    // descriptor reads rows 64..127 from the 16 KB that follow (bia[1] after bia[0], kb after
    // bia[1]); those accumulator rows are discarded.
    // After MMA-a its first 16 KB hold the MMA-b A operand: Tm in four copies [4 x 32 t x 32 s],
    // hi then lo (8 KB each).
    unsigned char bia[2][64 * 128 * 2];
    unsigned char kb[2][kCc * 128 * 2];          // K e^{c-G}            [32 s x 128 k]  MMA-a B
    unsigned char ktv[2][256 / 8 * kSboKt];      // [(beta K e^G)^T ; (beta V)^T] [256 x 32 s]  MMA-b B
    float scr[kCc * 128];                        // G [32 t][128 k]; after MMA-a: A, Tm, products
    float beta[kCc];
    float gs[kCc];                               // per-head log-gate per token (GDN)
    float gsc[kCc];                              // its running sum (GDN)
    float cref[128];                             // intra kernel: c = G_C / 2 per channel
    float ecr[128];                              // intra kernel: e^c
    float gcs[128];                              // the chunk's total gate per channel (fused prep)
    uint64_t bar;
    uint32_t tmem_base;
};
constexpr int kLd = kCc + 1;                     // row stride of the 32 x 32 f32 matrices in scr
constexpr int kTmBytes = 128 * kCc * 2;          // one (hi or lo) four-copy Tm image
static_assert(2 * kTmBytes <= 64 * 128 * 2, "Tm fits in bia[0]");

// The part of the intra-chunk computation that follows the operand images, shared by the
// chunked scan's intra kernel and the fused prefill kernel: MMA-a (A and Aqk), the blocked
// inverse Tm = (I + A)^{-1}, MMA-b (W and U) and the workspace epilogue.  On entry every thread
// has written its share of sm.bia, sm.kb, sm.ktv, the QG and K^T images in blk and blk's EG row
// (the fused kernel: the column images may still be on their way, see PRE_A below); sm.beta (and
// for GDN sm.gsc, the running per-head gate) are set; warp 0 holds sm.tmem_base (256 columns) and
// sm.bar is initialised; phase is sm.bar's current parity (updated).  Once MMA-a has completed
// (sm.bia[1] and sm.kb are then free for the rest of the tail), every thread calls after_a();
// once the Tm image is written (sm.scr is then free), after_tm().  Ends after a barrier that
// also agrees on the result, the TMEM still allocated; returns false (in every thread) if a
// bounded wait gave up.  NT = threads of the CTA, 128 or 256 (warps w and w+4 share TMEM lane
// quarter w and split the epilogue's columns).
struct NoHook {
    __device__ void operator()() const {}
};

// MMA-a, issued by one thread once sm.bia and sm.kb hold the row images (and a proxy fence and a
// barrier have made them visible): D[r][s] = (K e^{G-c} ; Q e^{G-c})_r . (K e^{c-G})_s, committed
// to sm.bar.
__device__ __forceinline__ void intra_mma_a_issue(IntraSmem& sm) {
    mma3_ss(sm.tmem_base, tc_smem_desc(smem_u32(sm.bia[0]), 128, kSbo128),
            tc_smem_desc(smem_u32(sm.bia[1]), 128, kSbo128),
            tc_smem_desc(smem_u32(sm.kb[0]), 128, kSbo128),
            tc_smem_desc(smem_u32(sm.kb[1]), 128, kSbo128), 8, tc_idesc_bf16(128, kCc));
    tc_commit(&sm.bar);
}

// PRE_A: the caller has issued MMA-a already (intra_mma_a_issue after the row images) and wrote
// the column images while it ran; the tail starts by waiting for it.  The caller may have thread 0
// bulk-store from sm.scr meanwhile: in this mode the tail lets those copies read sm.scr before it
// writes there.
template <int GATE_MODE, int NT, bool PRE_A = false, typename AfterA = NoHook,
          typename AfterTm = NoHook>
__device__ __forceinline__ bool intra_mma_tail(IntraSmem& sm, int* err, unsigned char* blk,
                                               uint32_t& phase, AfterA after_a = AfterA(),
                                               AfterTm after_tm = AfterTm(),
                                               const CUtensorMap* umap = nullptr, int ublock = 0) {
    static_assert(NT == 128 || NT == 256, "128 or 256 threads");
    static_assert(!PRE_A || NT == 256, "the staged epilogue takes 32 columns per warp");
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (!PRE_A) {
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    const uint32_t tbase = sm.tmem_base;
    const uint32_t tlane = tbase + ((uint32_t)(32 * (warp & 3)) << 16);
    bool ok = true;
    float* am = sm.scr;                          // A (strictly lower), f32 [32][kLd]
    float* ti = sm.scr + kCc * kLd;              // Tm
    float* pb = sm.scr + 2 * kCc * kLd;          // block products
    unsigned char* tmh = sm.bia[0];              // Tm image, written once MMA-a has completed
    unsigned char* tml = sm.bia[0] + kTmBytes;

    // ---- MMA-a: D[r][s] = (K e^{G-c} ; Q e^{G-c})_r . (K e^{c-G})_s ---------------------------
    if (!PRE_A && tid == 0) intra_mma_a_issue(sm);
    if (!PRE_A)
        for (int i = tid; i < kCc * kLd; i += NT) ti[i] = 0.0f;   // G is dead: scr is free
    ok = mbar_wait_bounded(&sm.bar, phase, err);
    phase ^= 1u;
    tc_fence_after();
    if (PRE_A && tid == 0) bulk_wait_read0();   // the caller's copies out of sm.scr have read it
    if (__syncthreads_or(!ok)) goto done;
    if (PRE_A)
        for (int i = tid; i < kCc * kLd; i += NT) ti[i] = 0.0f;
    after_a();

    // ---- A (warp 0, lane t = row t) and Aqk (warp 1, lane t) -----------------------------------
    if (warp < 2) {
        float d[kCc];
        tmem_ld16(tlane, *reinterpret_cast<float(*)[16]>(&d[0]));
        tmem_ld16(tlane + 16, *reinterpret_cast<float(*)[16]>(&d[16]));
        tmem_ld_wait();
        const int t = lane;
        const float Gt = GATE_MODE == 1 ? sm.gsc[t] : 0.0f;
        if (warp == 0) {
            const float bt = sm.beta[t];
#pragma unroll
            for (int s = 0; s < kCc; ++s) {
                const float fac = GATE_MODE == 1 ? __expf(fminf(Gt - sm.gsc[s], 0.0f)) : 1.0f;
                am[t * kLd + s] = s < t ? bt * d[s] * fac : 0.0f;
            }
        } else {
            unsigned char* b2 = blk + kOffB2;
#pragma unroll
            for (int sb = 0; sb < kCc / 8; ++sb) {
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int s = 8 * sb + e;
                    const float fac = GATE_MODE == 1 ? __expf(fminf(Gt - sm.gsc[s], 0.0f)) : 1.0f;
                    x[e] = s <= t ? d[s] * fac : 0.0f;
                }
                put8h(b2, tc_offset(128 + t, 8 * sb, kSbo32), x);
            }
        }
    }
    __syncthreads();

    // ---- Tm = (I + A)^{-1}: 8x8 diagonal blocks by substitution, then two doubling steps of
    //      [T11 0; T21 T22] with T21 = -T22 A21 T11 ------------------------------------------
    if (tid < kCc) {
        const int b8 = (tid >> 3) * 8, j = tid & 7;
        float x[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            float acc = r == j ? 1.0f : 0.0f;
#pragma unroll
            for (int m = 0; m < r; ++m) acc = fmaf(-am[(b8 + r) * kLd + b8 + m], x[m], acc);
            x[r] = acc;
            ti[(b8 + r) * kLd + b8 + j] = acc;
        }
    }
    __syncthreads();
    {
        const int p = (tid >> 6) & 1, r = (tid & 63) >> 3, cc = tid & 7;   // threads 0..127
        const int r0 = 16 * p + 8, c0 = 16 * p;
        if (tid < 128) {
            float acc = 0.0f;
#pragma unroll
            for (int m = 0; m < 8; ++m) acc = fmaf(am[(r0 + r) * kLd + c0 + m], ti[(c0 + m) * kLd + c0 + cc], acc);
            pb[(r0 + r) * kLd + c0 + cc] = acc;
        }
        __syncthreads();
        if (tid < 128) {
            float acc = 0.0f;
#pragma unroll
            for (int m = 0; m < 8; ++m) acc = fmaf(ti[(r0 + r) * kLd + r0 + m], pb[(r0 + m) * kLd + c0 + cc], acc);
            ti[(r0 + r) * kLd + c0 + cc] = -acc;
        }
        __syncthreads();
    }
#pragma unroll
    for (int e = tid; e < 256; e += NT) {
        const int r = e >> 4, cc = e & 15;
        float acc = 0.0f;
#pragma unroll
        for (int m = 0; m < 16; ++m) acc = fmaf(am[(16 + r) * kLd + m], ti[m * kLd + cc], acc);
        pb[(16 + r) * kLd + cc] = acc;
    }
    __syncthreads();
#pragma unroll
    for (int e = tid; e < 256; e += NT) {
        const int r = e >> 4, cc = e & 15;
        float acc = 0.0f;
#pragma unroll
        for (int m = 0; m < 16; ++m) acc = fmaf(ti[(16 + r) * kLd + 16 + m], pb[(16 + m) * kLd + cc], acc);
        ti[(16 + r) * kLd + cc] = -acc;
    }
    __syncthreads();
    if (tid < 128) {   // Tm image, four copies (rows t, 32+t, 64+t, 96+t): one per lane quarter
        const int t = tid >> 2, s0 = (tid & 3) * 8;
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = ti[t * kLd + s0 + e];
#pragma unroll
        for (int r = 0; r < 4; ++r) put8x(tmh, tml, tc_offset(32 * r + t, s0, kSbo32), x);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    after_tm();

    // ---- MMA-b: [W | U] = Tm [(beta K e^G) | (beta V)], every warp's 32 lanes = tokens --------
    if (tid == 0) {
        mma3_ss(tbase, tc_smem_desc(smem_u32(tmh), 128, kSbo32), tc_smem_desc(smem_u32(tml), 128, kSbo32),
                tc_smem_desc(smem_u32(sm.ktv[0]), 128, kSboKt),
                tc_smem_desc(smem_u32(sm.ktv[1]), 128, kSboKt), 2, tc_idesc_bf16(128, 256));
        tc_commit(&sm.bar);
    }
    // every thread observes MMA-b's completion itself; whether every wait succeeded is agreed at
    // the final barrier below (the epilogue runs either way, its bulk copies only on success)
    ok = mbar_wait_bounded(&sm.bar, phase, err);
    phase ^= 1u;
    tc_fence_after();
    {
        // warp w: columns CW*w .. CW*w+CW-1 of [W | U] (W: 0..127, U: 128..255) for token t = lane
        constexpr int CW = 256 / (NT / 32);
        const int t = lane, col0 = CW * warp;
        float x[CW];
#pragma unroll
        for (int q = 0; q < CW / 16; ++q)
            tmem_ld16(tlane + col0 + 16 * q, *reinterpret_cast<float(*)[16]>(&x[16 * q]));
        tmem_ld_wait();
        if (PRE_A) {        // staged in sm.ktv (free once MMA-b has completed), copied out in bulk
            if (col0 < 128) {   // W row t: rows 0..31 of an f16 image of 32 rows
#pragma unroll
                for (int cb = 0; cb < CW / 8; ++cb)
                    put8h(sm.ktv[1], tc_offset(t, col0 + 8 * cb, kSbo128),
                          *reinterpret_cast<const float(*)[8]>(&x[8 * cb]));
            } else {            // U row t: a [32 t][32 v] f32 tile, 16-byte pieces 128B-swizzled
                unsigned char* tile = sm.ktv[0] + (col0 - 128) * 128;   // 1024-byte aligned
#pragma unroll
                for (int q = 0; q < CW / 4; ++q)
                    *reinterpret_cast<float4*>(tile + t * 128 + ((q ^ (t & 7)) << 4)) =
                        make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
            }
        } else if (col0 < 128) {   // W row t, channels col0 .. : QW image rows 32 + t
            unsigned char* qw = blk + kOffQW;
#pragma unroll
            for (int cb = 0; cb < CW / 8; ++cb)
                put8h(qw, tc_offset(kCc + t, col0 + 8 * cb, kSbo128),
                      *reinterpret_cast<const float(*)[8]>(&x[8 * cb]));
        } else {            // U row t, values col0 - 128 .. : f32 [32 t][128 v]
            float4* ut = reinterpret_cast<float4*>(blk + kOffUT) + t * 32 + (col0 - 128) / 4;
#pragma unroll
            for (int q = 0; q < CW / 4; ++q) ut[q] = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
        }
    }
done:
    tc_fence_before();
    if (PRE_A) fence_proxy_async_smem();
    ok = __syncthreads_or(!ok) == 0;
    if (PRE_A && ok && tid == 0) {   // W: QW rows 32..63; U: four [32 t][32 v] tiles
        constexpr uint32_t kW = kCc * kSbo128 / 8;   // 8 KB: 4 groups of 8 rows
        bulk_store(blk + kOffQW + kW, sm.ktv[1], kW);
#pragma unroll
        for (int j = 0; j < 4; ++j) tma_store_3d(umap, sm.ktv[0] + 4096 * j, 32 * j, 0, ublock);
        bulk_commit();
    }
    return ok;
}

// Opt a kernel into `bytes` of dynamic shared memory once per device; `done` is the caller's own
// per-device flag array (one per template instantiation).
template <typename K>
inline cudaError_t set_smem(K kernel, size_t bytes, PerDevice<int>& done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const bool cached = dev >= 0 && dev < kMaxDevices;
    if (cached && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess && cached) done[dev].store(1, std::memory_order_release);
    return e;
}

}  // namespace kda
