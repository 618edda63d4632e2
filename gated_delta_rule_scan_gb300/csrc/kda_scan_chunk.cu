// kda_scan_chunk.cu -- the chunked (UT / WY) form of the per-channel gated delta rule on the
// tcgen05 tensor cores.
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
// GB300 design.  One CTA (128 threads) owns one (sequence, head) and walks its chunks of kCc = 16
// tokens; thread i is TMEM lane i and, depending on the phase, key channel k = i or value row
// v = i.  The state is kept transposed (S^T, value rows) in that thread's registers, f32, for the
// whole sequence.  Every contraction runs on tcgen05 (M = 128, f32 accumulators in TMEM) with
// bf16 operands written by the threads into shared memory in the K-major core-matrix layout;
// each operand is split x = hi + lo (bf16 each) and every product is hi*hi + hi*lo + lo*hi, which
// keeps ~16 significant bits (relative error ~1e-5, far inside the 1e-3 parity bound; one bf16
// pass is ~4e-3).  Per chunk:
//   MMA-a   [A/beta | Aqk]^T  = (K e^{c-G}) (K e^{G-c} | Q e^{G-c})^T      M=128 (16 used), N=32
//           (c = half the chunk's total gate per channel, so every exponent stays inside f32)
//   Tm      forward substitution on 16 lanes
//   MMA-b   [W^T | U^T]       = (beta K e^G | beta V)^T Tm^T                  M=128, N=16+16, K=16
//   MMA-1   [O1^T | X^T]      = S^T (Q e^G | W)^T                             M=128, N=32, K=128
//   U'^T = U^T - X^T                                                         (registers)
//   MMA-2   [dS^T | O2^T]     = U'^T (K e^{G_C-G} | Aqk)                      M=128, N=144, K=16
//   S^T <- S^T Diag(e^{G_C}) + dS^T,  o = scale (O1 + O2)                    (registers)
// The per-token q, k, v, g rows stream in by 2-D TMA, double-buffered, with bounded mbarrier
// waits; MMA completion is tracked by tcgen05.commit on an mbarrier.  For the per-head (GDN) gate
// the decay factors are scalars per token, so A and Aqk are formed from unscaled k, q and scaled
// after the MMA, which removes any range limit on the gate.  For the per-channel gate the chunk's
// total log-decay must stay above -170 on every channel (the KDA gate is bounded below by -5 per
// token, so 16 tokens stay above -80); otherwise the kernel raises the device error word.
#include "kda_tc.cuh"

namespace kda {

constexpr int kCc = 16;
constexpr int kChThreads = 128;
constexpr uint32_t kSboK128 = 2048;  // 8-row group stride of a K = 128 bf16 image
constexpr uint32_t kSboK16 = 256;    // 8-row group stride of a K = 16 bf16 image
constexpr int kDevErrRange = 2;      // device error word bit: chunk gate outside the f32 range

constexpr int kImgA1 = 128 * 128 * 2;  // S^T            [128 v  x 128 k]
constexpr int kImgKB = kCc * 128 * 2;  // K e^{c-G}      [16 s   x 128 k]  (descriptor spans 32 KB)
constexpr int kImgBI = 64 * 128 * 2;   // K e^{G-c} ; Q e^{G-c} ; Q e^G ; W   [64 x 128 k]
constexpr int kImgKT = 128 * kCc * 2;  // (beta K e^G)^T [128 k  x 16 s]
constexpr int kImgVT = 128 * kCc * 2;  // (beta V)^T     [128 v  x 16 s]
constexpr int kImgTM = kCc * kCc * 2;  // Tm             [16 t   x 16 s]
constexpr int kImgB2 = 144 * kCc * 2;  // (K e^{G_C-G})^T ; Aqk  [144 x 16]
constexpr int kImgA2 = 128 * kCc * 2;  // U'^T           [128 v  x 16 t]

// TMEM columns of the four accumulators (256 allocated)
constexpr uint32_t kTmA = 0, kTmB = 32, kTm1 = 64, kTm2 = 96;

struct __align__(1024) ChunkSmem {
    // operand images, [0] = hi, [1] = lo; kb is followed by a1 so that kb's 128-row descriptor
    // (only its first 16 rows are used) stays inside this allocation
    unsigned char kb[2][kImgKB];
    unsigned char a1[2][kImgA1];
    unsigned char bi[2][kImgBI];
    unsigned char kt[2][kImgKT];
    unsigned char vt[2][kImgVT];
    unsigned char tm[2][kImgTM];
    unsigned char b2[2][kImgB2];
    unsigned char a2[2][kImgA2];
    // staged chunk rows (TMA, double-buffered); g is turned into the cumulative gate in place
    float q[2][kCc][128];
    float k[2][kCc][128];
    float v[2][kCc][128];
    float g[2][kCc][128];
    float beta[2][kCc];
    float gs[2][kCc];            // per-head gate of the chunk (GDN), cumulative after phase 1
    float cref[128];             // per-channel reference: half the chunk's total log-decay
    float ecr[128];              // e^{cref}
    float egc[128];              // e^{G_C}: the chunk's total decay per channel
    float amat[kCc][kCc];        // beta_t A[t][s], strictly lower
    uint64_t bar_tma[2];
    uint64_t bar_mma;
    uint32_t tmem_base;
};

// byte offset of element (row, col) in a bf16 image with 8-row group stride sbo
__device__ __forceinline__ uint32_t img_off(int row, int col, uint32_t sbo) {
    return tc_offset(row, col, sbo);
}

// store x at byte offset off of an image pair (hi, lo)
template <int BYTES>
__device__ __forceinline__ void put1(unsigned char (&im)[2][BYTES], uint32_t off, float x) {
    __nv_bfloat16 hi, lo;
    split_bf16(x, hi, lo);
    *reinterpret_cast<__nv_bfloat16*>(&im[0][off]) = hi;
    *reinterpret_cast<__nv_bfloat16*>(&im[1][off]) = lo;
}

// store 8 consecutive-k values (one 16-byte core-matrix row) at byte offset off
template <int BYTES>
__device__ __forceinline__ void put8(unsigned char (&im)[2][BYTES], uint32_t off, const float (&x)[8]) {
    uint4 hi, lo;
    split_bf16x2(x[0], x[1], hi.x, lo.x);
    split_bf16x2(x[2], x[3], hi.y, lo.y);
    split_bf16x2(x[4], x[5], hi.z, lo.z);
    split_bf16x2(x[6], x[7], hi.w, lo.w);
    *reinterpret_cast<uint4*>(&im[0][off]) = hi;
    *reinterpret_cast<uint4*>(&im[1][off]) = lo;
}

// A pair of descriptors (hi, lo) of one operand image.
struct DescPair {
    uint64_t hi, lo;
};

template <int BYTES>
__device__ __forceinline__ DescPair desc_pair(unsigned char (&im)[2][BYTES], uint32_t byte_off,
                                              uint32_t sbo) {
    return {tc_smem_desc(smem_u32(im[0]) + byte_off, 128, sbo),
            tc_smem_desc(smem_u32(im[1]) + byte_off, 128, sbo)};
}

// D (+)= A * B^T in bf16x3: hi*hi + hi*lo + lo*hi, nks K-steps of 16 (256 bytes each).
__device__ __forceinline__ void mma_x3(uint32_t d, DescPair A, DescPair B, int nks,
                                       uint32_t idesc) {
    const uint64_t as[3] = {A.hi, A.hi, A.lo};
    const uint64_t bs[3] = {B.hi, B.lo, B.hi};
#pragma unroll
    for (int p = 0; p < 3; ++p)
        for (int ks = 0; ks < nks; ++ks)
            tc_mma_ss(d, tc_desc_advance(as[p], 256 * ks), tc_desc_advance(bs[p], 256 * ks), idesc,
                      p > 0 || ks > 0);
}

// GATE_MODE 0 per-channel, 1 per-head; EXP: g holds decay factors (take log first)
template <int GATE_MODE, bool EXP>
__global__ void __launch_bounds__(kChThreads, 1)
kda_scan_chunk_kernel(ScanArgs a, const __grid_constant__ CUtensorMap tq,
                      const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                      const __grid_constant__ CUtensorMap tg) {
    extern __shared__ unsigned char smem_raw[];
    ChunkSmem& sm = *reinterpret_cast<ChunkSmem*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.x;
    const int n = a.order ? a.order[blockIdx.y] : (int)blockIdx.y;
    const int H = a.H;
    const long C = (long)H * kHeadDim;
    long begin, end;
    if (a.seq.cu_seqlens == nullptr) {
        begin = (long)n * a.seq.T_uniform;
        end = begin + a.seq.T_uniform;
    } else {
        begin = a.seq.cu_seqlens[n];
        end = a.seq.cu_seqlens[n + 1];
    }
    const long L = end - begin;
    const int nch = (int)((L + kCc - 1) / kCc);

    if (warp == 0) {
        tmem_alloc(&sm.tmem_base, 256);
        tmem_relinquish();
    }
    if (tid == 0) {
        prefetch_tensormap(&tq);
        prefetch_tensormap(&tk);
        prefetch_tensormap(&tv);
        if (GATE_MODE == 0) prefetch_tensormap(&tg);
        mbar_init(&sm.bar_tma[0], 1);
        mbar_init(&sm.bar_tma[1], 1);
        mbar_init(&sm.bar_mma, 1);
        fence_mbar_init();
    }
    // this thread's state row S^T[v = tid][0..127]
    float srow[128];
    const float* sin = a.state_in + (((long)n * H + h) * kHeadDim + tid) * kHeadDim;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const float4 x = __ldcs(reinterpret_cast<const float4*>(sin) + j);
        srow[4 * j] = x.x; srow[4 * j + 1] = x.y; srow[4 * j + 2] = x.z; srow[4 * j + 3] = x.w;
    }
    auto write_a1 = [&]() {
#pragma unroll
        for (int c8 = 0; c8 < 16; ++c8) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = srow[8 * c8 + e];
            put8(sm.a1, img_off(tid, 8 * c8, kSboK128), x);
        }
    };
    write_a1();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = sm.tmem_base;
    const uint32_t tlane = tbase + ((uint32_t)(32 * warp) << 16);

    constexpr uint32_t kTx = (GATE_MODE == 0 ? 4u : 3u) * kCc * 128 * 4;
    auto issue = [&](int c, int st) {
        const int row = (int)(begin + (long)c * kCc);
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&sm.bar_tma[st], kTx);
        tma_load_2d(&sm.q[st][0][0], &tq, h * kHeadDim, row, &sm.bar_tma[st]);
        tma_load_2d(&sm.k[st][0][0], &tk, h * kHeadDim, row, &sm.bar_tma[st]);
        tma_load_2d(&sm.v[st][0][0], &tv, h * kHeadDim, row, &sm.bar_tma[st]);
        if (GATE_MODE == 0) tma_load_2d(&sm.g[st][0][0], &tg, h * kHeadDim, row, &sm.bar_tma[st]);
    };
    if (tid == 0 && nch > 0) issue(0, 0);
    float bpre = 0.0f, gpre = 0.0f;
    if (tid < kCc && tid < L) {
        bpre = a.beta[(begin + tid) * H + h];
        if (GATE_MODE == 1) gpre = a.g[(begin + tid) * H + h];
    }

    const uint32_t idA = tc_idesc_bf16(128, 32), idB = tc_idesc_bf16(128, 16);
    const uint32_t id2 = tc_idesc_bf16(128, 144);
    const DescPair dKB = desc_pair(sm.kb, 0, kSboK128), dBI0 = desc_pair(sm.bi, 0, kSboK128);
    const DescPair dBI32 = desc_pair(sm.bi, 4 * kSboK128, kSboK128);
    const DescPair dA1 = desc_pair(sm.a1, 0, kSboK128);
    const DescPair dKT = desc_pair(sm.kt, 0, kSboK16), dVT = desc_pair(sm.vt, 0, kSboK16);
    const DescPair dTM = desc_pair(sm.tm, 0, kSboK16), dB2 = desc_pair(sm.b2, 0, kSboK16);
    const DescPair dA2 = desc_pair(sm.a2, 0, kSboK16);
    uint32_t mma_phase = 0;
    bool failed = false;
    auto mma_wait = [&]() -> bool {
        const bool ok = mbar_wait_bounded(&sm.bar_mma, mma_phase, a.err);
        if (ok) mma_phase ^= 1u;
        tc_fence_after();
        return ok;
    };
    auto sync_images = [&]() {  // thread-written operand images -> visible to the tensor cores
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    };

    for (int c = 0; c < nch && !failed; ++c) {
        const int st = c & 1;
        const long row0 = begin + (long)c * kCc;
        const int nt = (int)min((long)kCc, L - (long)c * kCc);
        if (tid < kCc) {
            sm.beta[st][tid] = tid < nt ? bpre : 0.0f;
            if (GATE_MODE == 1) {
                float gl = tid < nt ? gpre : 0.0f;
                if (EXP && tid < nt) gl = logf(gpre);
                sm.gs[st][tid] = gl;
            }
            const long rn = row0 + kCc + tid;
            if (rn < end) {
                bpre = a.beta[rn * H + h];
                if (GATE_MODE == 1) gpre = a.g[rn * H + h];
            }
        }
        const bool arrived = mbar_wait_bounded(&sm.bar_tma[st], (uint32_t)((c >> 1) & 1), a.err);
        if (__syncthreads_or(!arrived)) { failed = true; break; }
        if (tid == 0 && c + 1 < nch) issue(c + 1, st ^ 1);

        // ---- phase 1: cumulative gate over the chunk ------------------------------------------
        if (GATE_MODE == 0) {
            float G = 0.0f;
            for (int t = 0; t < kCc; ++t) {
                float x = 0.0f;
                if (t < nt) {
                    x = sm.g[st][t][tid];
                    if (EXP) x = logf(x);
                }
                G += x;
                sm.g[st][t][tid] = G;
            }
            sm.cref[tid] = 0.5f * G;
            sm.ecr[tid] = __expf(0.5f * G);
            sm.egc[tid] = decay_f(G);
            if (G < -170.0f && a.err) atomicOr(a.err, kDevErrRange);
        } else if (tid == 0) {
            float G = 0.0f;
            for (int t = 0; t < kCc; ++t) {
                G += sm.gs[st][t];
                sm.gs[st][t] = G;
            }
            sm.cref[0] = G;
        }
        __syncthreads();
        if (GATE_MODE == 1) sm.egc[tid] = decay_f(sm.cref[0]);

        // ---- phase 2: operand images --------------------------------------------------------
        // row images: item = (token t, channels k0..k0+7); one exp pair feeds all four images
        for (int it = tid; it < kCc * 16; it += kChThreads) {
            const int t = it >> 4, k0 = (it & 15) * 8;
            float xb[8], xk[8], xq[8], xg[8];
            if (t < nt) {
                const float4* K4 = reinterpret_cast<const float4*>(&sm.k[st][t][k0]);
                const float4* Q4 = reinterpret_cast<const float4*>(&sm.q[st][t][k0]);
                const float kv[8] = {K4[0].x, K4[0].y, K4[0].z, K4[0].w, K4[1].x, K4[1].y, K4[1].z, K4[1].w};
                const float qv[8] = {Q4[0].x, Q4[0].y, Q4[0].z, Q4[0].w, Q4[1].x, Q4[1].y, Q4[1].z, Q4[1].w};
                if (GATE_MODE == 0) {
                    const float4* G4 = reinterpret_cast<const float4*>(&sm.g[st][t][k0]);
                    const float4* C4 = reinterpret_cast<const float4*>(&sm.cref[k0]);
                    const float4* E4 = reinterpret_cast<const float4*>(&sm.ecr[k0]);
                    const float gv[8] = {G4[0].x, G4[0].y, G4[0].z, G4[0].w, G4[1].x, G4[1].y, G4[1].z, G4[1].w};
                    const float cv[8] = {C4[0].x, C4[0].y, C4[0].z, C4[0].w, C4[1].x, C4[1].y, C4[1].z, C4[1].w};
                    const float ev[8] = {E4[0].x, E4[0].y, E4[0].z, E4[0].w, E4[1].x, E4[1].y, E4[1].z, E4[1].w};
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float ef = __expf(gv[e] - cv[e]);   // e^{G-c}
                        const float eb = __expf(cv[e] - gv[e]);   // e^{c-G}
                        xb[e] = kv[e] * eb;
                        xk[e] = kv[e] * ef;
                        xq[e] = qv[e] * ef;
                        xg[e] = qv[e] * (ef * ev[e]);             // Q e^{G}
                    }
                } else {
                    const float eg = __expf(sm.gs[st][t]);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        xb[e] = kv[e];
                        xk[e] = kv[e];
                        xq[e] = qv[e];
                        xg[e] = qv[e] * eg;
                    }
                }
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) xb[e] = xk[e] = xq[e] = xg[e] = 0.0f;
            }
            put8(sm.kb, img_off(t, k0, kSboK128), xb);
            put8(sm.bi, img_off(t, k0, kSboK128), xk);
            put8(sm.bi, img_off(16 + t, k0, kSboK128), xq);
            put8(sm.bi, img_off(32 + t, k0, kSboK128), xg);
        }
        // column images: item = (channel kk, tokens t0..t0+7)
        for (int it = tid; it < 128 * 2; it += kChThreads) {
            const int kk = it >> 1, t0 = (it & 1) * 8;
            float xt[8], xv[8], xc[8];
            const float GC = GATE_MODE == 0 ? sm.g[st][kCc - 1][kk] : sm.gs[st][kCc - 1];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int t = t0 + e;
                if (t < nt) {
                    const float G = GATE_MODE == 0 ? sm.g[st][t][kk] : sm.gs[st][t];
                    const float kv = sm.k[st][t][kk];
                    const float bt = sm.beta[st][t];
                    xt[e] = bt * kv * __expf(G);          // beta K e^{G}
                    xv[e] = bt * sm.v[st][t][kk];         // beta V
                    xc[e] = kv * __expf(GC - G);          // K e^{G_C - G}
                } else {
                    xt[e] = xv[e] = xc[e] = 0.0f;
                }
            }
            put8(sm.kt, img_off(kk, t0, kSboK16), xt);
            put8(sm.vt, img_off(kk, t0, kSboK16), xv);
            put8(sm.b2, img_off(kk, t0, kSboK16), xc);
        }
        sync_images();

        // ---- MMA-a: [A/beta | Aqk]^T, rows s --------------------------------------------------
        if (tid == 0) {
            mma_x3(tbase + kTmA, dKB, dBI0, 8, idA);
            tc_commit(&sm.bar_mma);
        }
        if (__syncthreads_or(!mma_wait())) { failed = true; break; }

        // ---- phase 4: A, Aqk, Tm on warp 0 ---------------------------------------------------
        if (warp == 0) {
            float d[32];
            tmem_ld16(tlane + kTmA, *reinterpret_cast<float(*)[16]>(&d[0]));
            tmem_ld16(tlane + kTmA + 16, *reinterpret_cast<float(*)[16]>(&d[16]));  // rows s
            tmem_ld_wait();
            const int s = lane;
            if (s < kCc) {
                const float Gs = GATE_MODE == 1 ? sm.gs[st][s] : 0.0f;
#pragma unroll
                for (int t = 0; t < kCc; ++t) {
                    float fac = 1.0f;
                    if (GATE_MODE == 1) fac = __expf(fminf(sm.gs[st][t] - Gs, 0.0f));
                    sm.amat[t][s] = t > s ? sm.beta[st][t] * d[t] * fac : 0.0f;
                    const float aqk = t >= s ? d[16 + t] * fac : 0.0f;
                    put1(sm.b2, img_off(128 + t, s, kSboK16), aqk);
                }
            }
            __syncwarp();
            if (s < kCc) {
                float x[kCc];
#pragma unroll
                for (int t = 0; t < kCc; ++t) {
                    float acc = t == s ? 1.0f : 0.0f;
#pragma unroll
                    for (int j = 0; j < t; ++j) acc = fmaf(-sm.amat[t][j], x[j], acc);
                    x[t] = acc;
                    put1(sm.tm, img_off(t, s, kSboK16), acc);
                }
            }
        }
        sync_images();

        // ---- MMA-b: [W^T | U^T] = (beta K e^G | beta V)^T Tm^T --------------------------------
        if (tid == 0) {
            mma_x3(tbase + kTmB, dKT, dTM, 1, idB);
            mma_x3(tbase + kTmB + 16, dVT, dTM, 1, idB);
            tc_commit(&sm.bar_mma);
        }
        if (__syncthreads_or(!mma_wait())) { failed = true; break; }
        float urow[kCc];
        {
            float d[16];
            tmem_ld16(tlane + kTmB, d);              // W[t][k = tid]
            tmem_ld16(tlane + kTmB + 16, urow);      // U^T[v = tid][t]
            tmem_ld_wait();
#pragma unroll
            for (int t = 0; t < kCc; ++t) put1(sm.bi, img_off(48 + t, tid, kSboK128), d[t]);
        }
        sync_images();

        // ---- MMA-1: [O1^T | X^T] = S^T (Q e^G | W)^T ---------------------------------------
        if (tid == 0) {
            mma_x3(tbase + kTm1, dA1, dBI32, 8, idA);
            tc_commit(&sm.bar_mma);
        }
        if (__syncthreads_or(!mma_wait())) { failed = true; break; }
        float o1[kCc];
        {
            float xr[16];
            tmem_ld16(tlane + kTm1, o1);
            tmem_ld16(tlane + kTm1 + 16, xr);
            tmem_ld_wait();
            float up[16];
#pragma unroll
            for (int t = 0; t < kCc; ++t) up[t] = urow[t] - xr[t];
            float lo8[8], hi8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) { lo8[e] = up[e]; hi8[e] = up[8 + e]; }
            put8(sm.a2, img_off(tid, 0, kSboK16), lo8);
            put8(sm.a2, img_off(tid, 8, kSboK16), hi8);
        }
        sync_images();

        // ---- MMA-2: [dS^T | O2^T] = U'^T (K e^{G_C-G} | Aqk) -------------------------------
        if (tid == 0) {
            mma_x3(tbase + kTm2, dA2, dB2, 1, id2);
            tc_commit(&sm.bar_mma);
        }
        if (__syncthreads_or(!mma_wait())) { failed = true; break; }
        {
#pragma unroll
            for (int c16 = 0; c16 < 8; ++c16) {
                float d[16];
                tmem_ld16(tlane + kTm2 + 16 * c16, d);
                tmem_ld_wait();
                const float4* E4 = reinterpret_cast<const float4*>(&sm.egc[16 * c16]);
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const float4 e4 = E4[q4];
                    const int kk = 16 * c16 + 4 * q4;
                    srow[kk] = fmaf(srow[kk], e4.x, d[4 * q4]);
                    srow[kk + 1] = fmaf(srow[kk + 1], e4.y, d[4 * q4 + 1]);
                    srow[kk + 2] = fmaf(srow[kk + 2], e4.z, d[4 * q4 + 2]);
                    srow[kk + 3] = fmaf(srow[kk + 3], e4.w, d[4 * q4 + 3]);
                }
            }
            float o2[16];
            tmem_ld16(tlane + kTm2 + 128, o2);
            tmem_ld_wait();
            float* orow = a.o + row0 * C + h * kHeadDim + tid;
#pragma unroll
            for (int t = 0; t < kCc; ++t)
                if (t < nt) orow[(long)t * C] = __fmul_rn(a.scale, o1[t] + o2[t]);
        }
        write_a1();
        sync_images();
    }
    if (!failed) {
        float* sout = a.state_out + (((long)n * H + h) * kHeadDim + tid) * kHeadDim;
#pragma unroll
        for (int j = 0; j < 32; ++j)
            __stcs(reinterpret_cast<float4*>(sout) + j,
                   make_float4(srow[4 * j], srow[4 * j + 1], srow[4 * j + 2], srow[4 * j + 3]));
    } else {
        // let in-flight MMAs finish (bounded) before the tensor memory is released
        mbar_wait_bounded(&sm.bar_mma, mma_phase, nullptr);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, 256);
}

template <int GM, bool EXP>
static cudaError_t launch_chunk_t(const ScanArgs& a, cudaStream_t s) {
    const long C = (long)a.H * kHeadDim;
    const long rows = a.seq.total_rows;
    CUtensorMap tq, tk, tv, tg;
    if (!make_tensor_map_2d(&tq, a.q, rows, C, kHeadDim, kCc) ||
        !make_tensor_map_2d(&tk, a.k, rows, C, kHeadDim, kCc) ||
        !make_tensor_map_2d(&tv, a.v, rows, C, kHeadDim, kCc))
        return cudaErrorInvalidValue;
    if (GM == 0) {
        if (!make_tensor_map_2d(&tg, a.g, rows, C, kHeadDim, kCc)) return cudaErrorInvalidValue;
    } else {
        tg = tq;
    }
    const size_t smem = sizeof(ChunkSmem) + 1024;
    static int attr_done[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !attr_done[dev]) {
        e = cudaFuncSetAttribute(kda_scan_chunk_kernel<GM, EXP>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_done[dev] = 1;
    }
    dim3 grid((unsigned)a.H, (unsigned)a.seq.N);
    kda_scan_chunk_kernel<GM, EXP><<<grid, kChThreads, smem, s>>>(a, tq, tk, tv, tg);
    return cudaGetLastError();
}

size_t chunk_smem_bytes() { return sizeof(ChunkSmem) + 1024; }

cudaError_t launch_scan_chunk(const ScanArgs& a, cudaStream_t s) {
    if (a.seq.N == 0) return cudaSuccess;
    if (a.seq.total_rows == 0) {
        const size_t bytes = (size_t)a.seq.N * a.H * kHeadDim * kHeadDim * sizeof(float);
        return cudaMemcpyAsync(a.state_out, a.state_in, bytes, cudaMemcpyDeviceToDevice, s);
    }
    const bool exp_done = (a.gate_mode & 2) != 0;
    if ((a.gate_mode & 1) == 0) return exp_done ? launch_chunk_t<0, true>(a, s) : launch_chunk_t<0, false>(a, s);
    return exp_done ? launch_chunk_t<1, true>(a, s) : launch_chunk_t<1, false>(a, s);
}

}  // namespace kda
