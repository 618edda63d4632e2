// kda_scan_chunk.cu -- the chunked (UT / WY) form of the per-channel gated delta rule on the
// tcgen05 tensor cores: the per-sequence chunk offsets, the intra-chunk kernel over the prepared
// q, k, v, g planes and the sequential inter-chunk kernel, with their launchers.  The method,
// the workspace layout and the shared device code are in kda_chunk_common.cuh.
#include <cstring>
#include <type_traits>

#include "kda_chunk_common.cuh"
#include "kda_ring.cuh"

namespace kda {

// ============================================================================================
// kernel 0: per-sequence chunk offsets (varlen): chunk_off[n] = sum_{m<n} ceil(L_m / kCc)
// ============================================================================================
__global__ void __launch_bounds__(1024) kda_chunk_offsets_kernel(const int* cu, int N, int* out) {
    __shared__ long part[1024];
    const int tid = threadIdx.x;
    const int per = (N + 1023) / 1024;
    const int b = min(N, tid * per), e = min(N, b + per);
    long sum = 0;
    for (int n = b; n < e; ++n) sum += (cu[n + 1] - cu[n] + kCc - 1) / kCc;
    part[tid] = sum;
    __syncthreads();
    if (tid == 0) {
        long acc = 0;
        for (int i = 0; i < 1024; ++i) { const long x = part[i]; part[i] = acc; acc += x; }
        out[N] = (int)acc;
    }
    __syncthreads();
    long acc = part[tid];
    for (int n = b; n < e; ++n) {
        out[n] = (int)acc;
        acc += (cu[n + 1] - cu[n] + kCc - 1) / kCc;
    }
}

// ============================================================================================
// kernel 1: intra-chunk quantities, one CTA per (chunk, head)
// ============================================================================================

template <int GATE_MODE, bool EXP>
__global__ void __launch_bounds__(kThr, 2)
kda_chunk_intra_kernel(ScanArgs a, const int* chunk_off, unsigned char* ws) {
    extern __shared__ unsigned char smem_raw[];
    IntraSmem& sm = *reinterpret_cast<IntraSmem*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    const int tid = threadIdx.x, warp = tid >> 5;
    const int h = blockIdx.y;
    const long gid = blockIdx.x;                 // global chunk index
    const int H = a.H;
    const long C = (long)H * kHeadDim;

    // chunk -> (sequence n, chunk c within it)
    int n;
    if (a.seq.cu_seqlens == nullptr) {
        const long per = (a.seq.T_uniform + kCc - 1) / kCc;
        n = (int)(gid / per);
    } else {
        int lo = 0, hi = a.seq.N;                // largest n with chunk_off[n] <= gid
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if ((long)chunk_off[mid] <= gid) lo = mid; else hi = mid;
        }
        n = lo;
    }
    long begin, end;
    seq_range(a.seq, n, begin, end);
    const long c = gid - chunk_base(a.seq, chunk_off, n);
    const long row0 = begin + c * kCc;
    const int nt = (int)min((long)kCc, end - row0);
    unsigned char* blk = ws + ((long)gid * H + h) * kBlkBytes;
    const long hoff = row0 * C + (long)h * kHeadDim;
    const long Ck = (long)qk_heads(a) * kHeadDim;     // q and k rows: the head (h / vsub) % Hk
    const long qkoff = row0 * Ck + (long)unit_qk_head(a, h) * kHeadDim;
    const int gh = gate_head(a, h), Hg = gate_heads(a);   // the value head: gate and beta
    const long Cg = (long)Hg * kHeadDim;
    const long goff = row0 * Cg + (long)gh * kHeadDim;

    // ---- every global load of the chunk is issued before any store ---------------------------
    // column role: channel tid over the chunk's 32 tokens
    float kc[kCc], vc[kCc], gc[kCc];
#pragma unroll
    for (int t = 0; t < kCc; ++t) {
        const bool live = t < nt;
        kc[t] = live ? __ldg(a.k + qkoff + t * Ck + tid) : 0.0f;
        vc[t] = live ? __ldg(a.v + hoff + t * C + tid) : 0.0f;
        if (GATE_MODE == 0) gc[t] = live ? __ldg(a.g + goff + t * Cg + tid) : (EXP ? 1.0f : 0.0f);
    }
    // row role: tokens tr + 8j (j = 0..3), channels k0 .. k0+7
    const int tr = tid >> 4, k0 = (tid & 15) * 8;
    float4 kr[4][2], qr[4][2];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int t = tr + 8 * j;
        if (t < nt) {
            const float4* kp = reinterpret_cast<const float4*>(a.k + qkoff + t * Ck + k0);
            const float4* qp = reinterpret_cast<const float4*>(a.q + qkoff + t * Ck + k0);
            kr[j][0] = __ldg(kp); kr[j][1] = __ldg(kp + 1);
            qr[j][0] = __ldg(qp); qr[j][1] = __ldg(qp + 1);
        } else {
            kr[j][0] = kr[j][1] = qr[j][0] = qr[j][1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    if (tid < kCc) {
        const bool live = tid < nt;
        sm.beta[tid] = live ? a.beta[(row0 + tid) * Hg + gh] : 0.0f;
        if (GATE_MODE == 1) {
            const float x = live ? a.g[(row0 + tid) * Hg + gh] : (EXP ? 1.0f : 0.0f);
            sm.gs[tid] = EXP ? logf(x) : x;
        }
    }

    if (warp == 0) {
        tmem_alloc(&sm.tmem_base, 256);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&sm.bar, 1);
        fence_mbar_init();
    }

    // ---- cumulative gate: gc[t] = G_t of channel tid (KDA) or of the head (GDN) ---------------
    // KDA, blocked: tokens in blocks of 4, each block summed in order from 0; the running total
    // of the blocks before (in order, from 0) is added to every token of the block
    if (GATE_MODE == 0) {
        float G = 0.0f;                          // total of the blocks so far
#pragma unroll
        for (int b = 0; b < kCc / 4; ++b) {
            float run = 0.0f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int t = 4 * b + i;
                run += EXP ? logf(gc[t]) : gc[t];
                gc[t] = run;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int t = 4 * b + i;
                gc[t] = G + gc[t];
                sm.scr[t * 128 + tid] = gc[t];
            }
            G = G + run;
        }
        sm.cref[tid] = 0.5f * G;
        sm.ecr[tid] = __expf(0.5f * G);
        reinterpret_cast<float*>(blk + kOffEG)[tid] = decay_f(G);
        if (G < -170.0f && a.err) atomicOr(a.err, kDevErrRange);
    }
    __syncthreads();
    if (GATE_MODE == 1) {
        float G = 0.0f;
#pragma unroll
        for (int t = 0; t < kCc; ++t) {
            G += sm.gs[t];
            gc[t] = G;
        }
        if (tid < kCc) {
            float Gt = 0.0f;
            for (int t = 0; t <= tid; ++t) Gt += sm.gs[t];   // same summation order as gc
            sm.gsc[tid] = Gt;
        }
        reinterpret_cast<float*>(blk + kOffEG)[tid] = decay_f(G);
    }

    // ---- column images: channel tid, tokens 8j .. 8j+7 ----------------------------------------
    {
        const float GC = gc[kCc - 1];
        float bv[kCc];                           // loaded before the image stores (see below)
#pragma unroll
        for (int q = 0; q < kCc / 4; ++q) {
            const float4 b4 = *reinterpret_cast<const float4*>(&sm.beta[4 * q]);
            bv[4 * q] = b4.x; bv[4 * q + 1] = b4.y; bv[4 * q + 2] = b4.z; bv[4 * q + 3] = b4.w;
        }
#pragma unroll
        for (int j = 0; j < kCc / 8; ++j) {
            float xt[8], xv[8], xc[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int t = 8 * j + e;
                const float bt = bv[t];
                xt[e] = bt * kc[t] * __expf(gc[t]);
                xv[e] = bt * vc[t];
                xc[e] = kc[t] * __expf(GC - gc[t]);
            }
            put8x(sm.ktv[0], sm.ktv[1], tc_offset(tid, 8 * j, kSboKt), xt);
            put8x(sm.ktv[0], sm.ktv[1], tc_offset(128 + tid, 8 * j, kSboKt), xv);
            put8h(blk + kOffB2, tc_offset(tid, 8 * j, kSbo32), xc);
        }
    }
    if (GATE_MODE == 1) __syncthreads();          // gsc

    // ---- row images: token t = tr + 8j, channels k0 .. k0+7 -----------------------------------
    // the shared-memory operands of all four items first (the image stores below are byte
    // stores that could alias them, so loads after a store would wait for it)
    float gtv[4][8], crv[8], ecv[8];
    if (GATE_MODE == 0) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float4 a0 = *reinterpret_cast<const float4*>(&sm.scr[(tr + 8 * j) * 128 + k0]);
            const float4 a1 = *reinterpret_cast<const float4*>(&sm.scr[(tr + 8 * j) * 128 + k0 + 4]);
            gtv[j][0] = a0.x; gtv[j][1] = a0.y; gtv[j][2] = a0.z; gtv[j][3] = a0.w;
            gtv[j][4] = a1.x; gtv[j][5] = a1.y; gtv[j][6] = a1.z; gtv[j][7] = a1.w;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) { crv[e] = sm.cref[k0 + e]; ecv[e] = sm.ecr[k0 + e]; }
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) gtv[j][0] = sm.gsc[tr + 8 * j];
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int t = tr + 8 * j;
        const float kv[8] = {kr[j][0].x, kr[j][0].y, kr[j][0].z, kr[j][0].w,
                             kr[j][1].x, kr[j][1].y, kr[j][1].z, kr[j][1].w};
        const float qv[8] = {qr[j][0].x, qr[j][0].y, qr[j][0].z, qr[j][0].w,
                             qr[j][1].x, qr[j][1].y, qr[j][1].z, qr[j][1].w};
        float xb[8], xk[8], xq[8], xg[8];
        if (GATE_MODE == 0) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float gt = gtv[j][e], cr = crv[e];
                const float ef = __expf(gt - cr), eb = __expf(cr - gt);
                xb[e] = kv[e] * eb;
                xk[e] = kv[e] * ef;
                xq[e] = qv[e] * ef;
                xg[e] = qv[e] * (ef * ecv[e]);
            }
        } else {
            const float eg = __expf(gtv[j][0]);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                xb[e] = kv[e];
                xk[e] = kv[e];
                xq[e] = qv[e];
                xg[e] = qv[e] * eg;
            }
        }
        put8x(sm.kb[0], sm.kb[1], tc_offset(t, k0, kSbo128), xb);
        put8x(sm.bia[0], sm.bia[1], tc_offset(t, k0, kSbo128), xk);
        put8x(sm.bia[0], sm.bia[1], tc_offset(kCc + t, k0, kSbo128), xq);
        put8h(blk + kOffQW, tc_offset(t, k0, kSbo128), xg);
    }
    uint32_t phase = 0;
    intra_mma_tail<GATE_MODE, kThr>(sm, a.err, blk, phase);
    if (warp == 0) tmem_dealloc(sm.tmem_base, 256);
}

// ============================================================================================
// kernel 2: the state recurrence over chunks, one CTA per (sequence, head)
// ============================================================================================

constexpr int kInterStages = 3;                  // workspace blocks in flight per CTA (2: 271 us,
                                                 // 3: 254 us, 4: 266 us at full size)

struct __align__(128) InterSmem {
    unsigned char blk[kInterStages][kBlkBytes];
    float otile[3][kCc][128];                    // chunks' o rows on their way out (c % 3)
    float ztile[kCc][128];                       // NORM: the RMSNorm gate z of the next o rows
    uint64_t bar_ld[kInterStages];
    uint64_t bar_mma;                            // MMA-1, then MMA-2
    uint32_t tmem_base;
};

// TMEM columns
constexpr uint32_t kTA1 = 0;      // S^T hi (64) then lo (64)
constexpr uint32_t kTA2 = 128;    // U'^T hi (16) then lo (16)
constexpr uint32_t kTD1 = 160;    // [O1^T | X^T]  64
constexpr uint32_t kTD2 = 224;    // [dS^T | O2^T] 160

// Write NV f32 values (NV = 4, 8, 16 or a multiple of 32) as packed f16 hi words at col_hi and
// lo words at col_lo: the inter kernel's A operands (the state S^T, U'^T) in TMEM.
template <int NV>
__device__ __forceinline__ void tmem_put_split_n(uint32_t col_hi, uint32_t col_lo, const float* v) {
    if constexpr (NV == 4) {
        uint32_t hw[2], lw[2];
        split_f16x2(v[0], v[1], hw[0], lw[0]);
        split_f16x2(v[2], v[3], hw[1], lw[1]);
        tmem_st2(col_hi, hw);
        tmem_st2(col_lo, lw);
    } else if constexpr (NV == 8) {
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) split_f16x2(v[2 * i], v[2 * i + 1], hw[i], lw[i]);
        tmem_st4(col_hi, hw);
        tmem_st4(col_lo, lw);
    } else if constexpr (NV == 16) {
        uint32_t hw[8], lw[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) split_f16x2(v[2 * i], v[2 * i + 1], hw[i], lw[i]);
        tmem_st8(col_hi, hw);
        tmem_st8(col_lo, lw);
    } else {
#pragma unroll
        for (int b = 0; b < NV / 32; ++b) {
            float hw[16], lw[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                uint32_t hu, lu;
                split_f16x2(v[32 * b + 2 * i], v[32 * b + 2 * i + 1], hu, lu);
                hw[i] = __uint_as_float(hu);
                lw[i] = __uint_as_float(lu);
            }
            tmem_st16(col_hi + 16 * b, hw);
            tmem_st16(col_lo + 16 * b, lw);
        }
    }
}

// N = 4, 8 or a multiple of 16 consecutive columns of this thread's lane
template <int N>
__device__ __forceinline__ void tmem_ld_n(uint32_t taddr, float* v) {
    if constexpr (N == 4) {
        tmem_ld4(taddr, *reinterpret_cast<float(*)[4]>(v));
    } else if constexpr (N == 8) {
        tmem_ld8(taddr, *reinterpret_cast<float(*)[8]>(v));
    } else {
#pragma unroll
        for (int b = 0; b < N / 16; ++b)
            tmem_ld16(taddr + 16 * b, *reinterpret_cast<float(*)[16]>(v + 16 * b));
    }
}

// Threads: 128 * kInterKq.  Thread (key group qf = tid / 128, value row v = tid % 128) owns TMEM
// lane v (warps w, w + 4, ... share lane quarter w % 4); with KPP = 64 / kInterKq it keeps key
// columns KPP qf .. KPP qf + KPP - 1 and 64 + KPP qf .. of state row v in registers and handles
// tokens TPT qf .. TPT qf + TPT - 1 (TPT = 32 / kInterKq) of each chunk's U' and o.  The state
// update runs in two passes, keys 0..63 then 64..127, so that the next chunk's MMA-1 takes its
// first four K-steps while the second pass runs.  More threads per value row shorten each
// thread's share of the chunk's dependent register / TMEM work.  Thread 0 issues the MMAs,
// thread 32 the workspace loads, and the lanes of warp 2 the o rows' bulk stores.  With NORM (the
// fused prefill, 128-wide value heads) no o row leaves: while MMA-2 of chunk c runs, each warp
// turns two o rows of chunk c-1 into y rows of the gated RMSNorm, their z rows copied into shared
// memory (cp.async) a chunk ahead.
constexpr int kInterKq = 4;
constexpr int kThrInter = 128 * kInterKq;

template <int GATE_MODE, bool NORM>
__global__ void __launch_bounds__(kThrInter, 1)
kda_chunk_inter_kernel(ScanArgs a, const int* chunk_off, const unsigned char* ws,
                       const __grid_constant__ CUtensorMap tmo, const __grid_constant__ PrepArgs ring) {
    extern __shared__ unsigned char smem_raw[];
    InterSmem& sm = *reinterpret_cast<InterSmem*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    constexpr int KPP = 64 / kInterKq;           // keys per thread and pass
    constexpr int TPT = kCc / kInterKq;          // tokens per thread
    const int tid = threadIdx.x, warp = tid >> 5;
    const int v = tid & 127, qf = tid >> 7;
    const int h = blockIdx.x;
    const int n = a.order ? a.order[blockIdx.y] : (int)blockIdx.y;
    const int H = a.H;
    const long C = (long)H * kHeadDim;
    long begin, end;
    seq_range(a.seq, n, begin, end);
    const long L = end - begin;
    const int nch = (int)((L + kCc - 1) / kCc);
    const long gbase = chunk_base(a.seq, chunk_off, n);

    if (warp == 0) {
        tmem_alloc(&sm.tmem_base, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < kInterStages; ++i) mbar_init(&sm.bar_ld[i], 1);
        mbar_init(&sm.bar_mma, 1);
        fence_mbar_init();
    }
    float srow[2 * KPP];             // keys 64 pass + KPP qf + j at srow[KPP pass + j]
    {
        const float* srow_in = a.state_in + (((long)n * H + h) * kHeadDim + v) * kHeadDim;
#pragma unroll
        for (int pass = 0; pass < 2; ++pass)
#pragma unroll
            for (int j = 0; j < KPP / 4; ++j) {
                const float4 x = __ldcs(reinterpret_cast<const float4*>(
                    srow_in + 64 * pass + KPP * qf + 4 * j));
                float* d = srow + KPP * pass + 4 * j;
                d[0] = x.x; d[1] = x.y; d[2] = x.z; d[3] = x.w;
            }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = sm.tmem_base;
    const uint32_t tl = tbase + ((uint32_t)(32 * (warp & 3)) << 16);
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
        const int k0 = 64 * pass + KPP * qf;
        tmem_put_split_n<KPP>(tl + kTA1 + k0 / 2, tl + kTA1 + 64 + k0 / 2, srow + KPP * pass);
    }
    tmem_st_wait();

    auto issue = [&](int c, int st) {
        const unsigned char* src = ws + ((gbase + c) * H + h) * (long)kBlkBytes;
        mbar_arrive_expect_tx(&sm.bar_ld[st], kBlkBytes);
        bulk_load(&sm.blk[st][kOffQW], src + kOffQW, kQWBytes, &sm.bar_ld[st]);
        bulk_load(&sm.blk[st][kOffB2], src + kOffB2, kB2Bytes, &sm.bar_ld[st]);
        bulk_load(&sm.blk[st][kOffUT], src + kOffUT, kUTBytes + kEGBytes, &sm.bar_ld[st]);
    };
    const uint32_t id1 = tc_idesc_f16(128, 2 * kCc), id2 = tc_idesc_f16(128, 160);
    // MMA-1: [O1^T | X^T] = S^T (Q e^G | W)^T for the chunk in stage st, K-steps ks0 .. ks0+3
    // (keys 16 ks0 ..), S^T as f16 hi + lo against the f16 image per K-step; the first product of
    // K-step 0 starts the sum.  (One N = 64 group: the tensor pipe's cost here follows the
    // instruction count, so two N = 32 groups are slower.)
    auto mma1_half = [&](int st, int ks0) {
        const unsigned char* B = sm.blk[st];
        const uint64_t bq = tc_smem_desc(smem_u32(B + kOffQW), 128, kSbo128);
#pragma unroll
        for (int ks = ks0; ks < ks0 + 4; ++ks) {
            const uint32_t ah = tbase + kTA1 + 8 * ks, al = tbase + kTA1 + 64 + 8 * ks;
            tc_mma_ts(tbase + kTD1, ah, tc_desc_advance(bq, 256 * ks), id1, ks > 0);
            tc_mma_ts(tbase + kTD1, al, tc_desc_advance(bq, 256 * ks), id1, true);
        }
    };
    auto mma1 = [&](int st) {
        mma1_half(st, 0);
        mma1_half(st, 4);
        tc_commit(&sm.bar_mma);
    };
    // the state is in TMEM (the barrier orders every thread's stores before the first MMA-1); the
    // first chunk's MMA-1 goes out as soon as its block lands
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0 && nch > 0) {
        for (int i = 0; i < kInterStages && i < nch; ++i) issue(i, i);
        tc_fence_before();
        if (mbar_wait_bounded(&sm.bar_ld[0], 0, a.err)) {
            tc_fence_after();
            mma1(0);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // the fused prefill's conv ring roll of this (sequence, head) while the first MMA-1 runs (the
    // prep kernel that read ring_in has finished)
    if (ring.conv_w != nullptr) {
        // grouped queries: the q and k ring rows of head h exist (and are rolled here) only for
        // h < Hk; every value head rolls its v rows
        const int p0 = h < prep_qk_heads(ring.H, ring.Hk) ? 0 : 2;
        for (int i = tid + p0 * kHeadDim; i < 3 * kHeadDim; i += kThrInter) {
            const int p = i / kHeadDim;
            const long c = (long)h * kHeadDim + i % kHeadDim;
            if (ring.raw_bf16) ring_roll_one<true>(ring, n, p, c);
            else ring_roll_one<false>(ring, n, p, c);
        }
    }

    uint32_t mph = 0;
    bool failed = false;
    bool late_fail = false;          // an MMA-2 wait gave up: ends the loop at its next barrier
    const float scale = a.scale;
    const bool ostore_lane = warp == 2;
    const int olane = tid & 31;
    // store the o rows of chunk cp (staged in otile[cp % 3]) -- warp 2 only.  A full chunk (or
    // one whose overhang lies past the last row of the tensor) goes out as one TMA tile store;
    // the ragged last chunk of a sequence followed by another is copied row by row.
    auto flush_o = [&](int cp) {
        const long r0 = begin + (long)cp * kCc;
        const int ntp = (int)min((long)kCc, L - (long)cp * kCc);
        if (ntp == kCc || end == a.seq.total_rows) {
            if (olane == 0) tma_store_2d(&tmo, sm.otile[cp % 3], h * kHeadDim, (int)r0);
        } else {
            for (int t = 0; t < ntp; ++t)
                reinterpret_cast<float4*>(a.o + (r0 + t) * C + h * kHeadDim)[olane] =
                    reinterpret_cast<const float4*>(sm.otile[cp % 3][t])[olane];
        }
        bulk_commit();
    };
    // NORM: the gated RMSNorm of chunk cp's o rows (staged in otile[cp % 3]), rows 2 warp and
    // 2 warp + 1, one float4 per lane -- the RMSNorm kernel's arithmetic on the same o values,
    // so y has the bits that storing o and normalising it there gives.  Each lane reads back
    // only the z float4s it copied itself (load_z), so its own wait suffices.
    constexpr int kRowsPerWarp = kCc / (kThrInter / 32);
    auto norm_rows = [&](int cp, auto silu) {
        const long r0 = begin + (long)cp * kCc;
        const int ntp = (int)min((long)kCc, L - (long)cp * kCc);
        const float4 w4 = *reinterpret_cast<const float4*>(a.norm_w + 4 * olane);
        cp_async_wait_all();
#pragma unroll
        for (int j = 0; j < kRowsPerWarp; ++j) {
            const int t = kRowsPerWarp * warp + j;
            if (t >= ntp) break;
            const float4 o4 = reinterpret_cast<const float4*>(sm.otile[cp % 3][t])[olane];
            float ss = __fmul_rn(o4.x, o4.x);
            ss = ss + __fmul_rn(o4.y, o4.y);
            ss = ss + __fmul_rn(o4.z, o4.z);
            ss = ss + __fmul_rn(o4.w, o4.w);
            const float inv = rms_inv_f(warp_sum(ss), a.norm_eps);
            const long base = (r0 + t) * C + h * kHeadDim + 4 * olane;
            const float4 z4 = reinterpret_cast<const float4*>(sm.ztile[t])[olane];
            constexpr bool SILU = decltype(silu)::value;
            float4 y4;
            y4.x = gated_norm_f<SILU>(o4.x, inv, w4.x, z4.x);
            y4.y = gated_norm_f<SILU>(o4.y, inv, w4.y, z4.y);
            y4.z = gated_norm_f<SILU>(o4.z, inv, w4.z, z4.z);
            y4.w = gated_norm_f<SILU>(o4.w, inv, w4.w, z4.w);
            __stcs(reinterpret_cast<float4*>(a.norm_y + base), y4);
        }
    };
    auto norm_chunk = [&](int cp) {
        if (a.norm_silu) norm_rows(cp, std::true_type{});
        else norm_rows(cp, std::false_type{});
    };
    // NORM: chunk c's z rows (this warp's two) into ztile, a chunk before norm_rows reads them;
    // issued after the lane's reads of the previous rows there
    auto load_z = [&](int c) {
        const long r0 = begin + (long)c * kCc;
        const int ntp = (int)min((long)kCc, L - (long)c * kCc);
#pragma unroll
        for (int j = 0; j < kRowsPerWarp; ++j) {
            const int t = kRowsPerWarp * warp + j;
            if (t < ntp)
                cp_async16(reinterpret_cast<float4*>(sm.ztile[t]) + olane,
                           a.norm_z + (r0 + t) * C + h * kHeadDim + 4 * olane);
        }
        cp_async_commit();
    };
    if (NORM && nch > 0) load_z(0);
    for (int c = 0; c < nch; ++c) {
        const int st = c % kInterStages;
        const unsigned char* B = sm.blk[st];
        // the block landed before thread 0 issued this chunk's MMA-1; each thread still observes
        // its barrier before reading it, and MMA-1's completion itself (no barrier here: a wait
        // that gave up is agreed on at the U' barrier below)
        bool ok = mbar_wait_bounded(&sm.bar_ld[st], (uint32_t)((c / kInterStages) & 1), a.err);
        ok = ok && mbar_wait_bounded(&sm.bar_mma, mph, a.err);
        if (ok) mph ^= 1u;
        tc_fence_after();
        // O1 and X for tokens TPT qf ..; O1 stays in registers until the chunk's o rows are
        // formed; U' = U - X into TMEM as MMA-2's A operand.  (The U rows are read from shared
        // memory before the TMEM wait, which orders every memory access after it.)
        float* ot = &sm.otile[c % 3][TPT * qf][v];
        float o1[TPT];
        {
            const float* ut = reinterpret_cast<const float*>(B + kOffUT) + (TPT * qf) * 128 + v;
            float up[TPT];
#pragma unroll
            for (int t = 0; t < TPT; ++t) up[t] = ut[t * 128];
            float x[TPT];
            tmem_ld_n<TPT>(tl + kTD1 + TPT * qf, o1);
            tmem_ld_n<TPT>(tl + kTD1 + 32 + TPT * qf, x);
            tmem_ld_wait();
#pragma unroll
            for (int t = 0; t < TPT; ++t) up[t] -= x[t];
            tmem_put_split_n<TPT>(tl + kTA2 + TPT / 2 * qf, tl + kTA2 + 16 + TPT / 2 * qf, up);
            tmem_st_wait();
        }
        tc_fence_before();
        if (__syncthreads_or(!ok || late_fail)) { failed = true; break; }
        tc_fence_after();
        if (!NORM && ostore_lane) {
            if (c > 0) flush_o(c - 1);           // its o rows were written before the barrier
            bulk_wait_read1();                   // only that store may still read its tile: the
                                                 // one of chunk c-3 (tile c % 3) is free
        }
        // MMA-2: [dS^T | O2^T] = U'^T (K e^{G_C-G} | Aqk)
        if (tid == 0) {
            mma2_ts(tbase + kTD2, tbase + kTA2, tbase + kTA2 + 16,
                    tc_smem_desc(smem_u32(B + kOffB2), 128, kSbo32), 2, id2);
            tc_commit(&sm.bar_mma);
        }
        if constexpr (NORM) {                    // while MMA-2 runs: its o rows were written
            if (c > 0) {                         // before the barrier above
                norm_chunk(c - 1);
                load_z(c);
            }
        }
        // every thread observes MMA-2's completion itself (no barrier needed for the TMEM reads
        // below); a wait that gave up is carried to the next barrier that can end the loop
        {
            const bool ok2 = mbar_wait_bounded(&sm.bar_mma, mph, a.err);
            if (ok2) mph ^= 1u;
            late_fail = late_fail || !ok2;
        }
        tc_fence_after();
        float o2[TPT];
        bool next_ok = false;            // thread 0: the next chunk's block landed, MMA-1 going
        // S <- S e^{G_C} + dS, keys 0..63 (srow[0..31]) then 64..127 (srow[32..63]); after the
        // first pass thread 0 starts the next chunk's MMA-1 on keys 0..63
        const float4* eg4 = reinterpret_cast<const float4*>(B + kOffEG);
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {
            const int k0 = 64 * pass + KPP * qf;     // this thread's first key of the pass
            float d[KPP];
            tmem_ld_n<KPP>(tl + kTD2 + k0, d);
            if (pass == 1) tmem_ld_n<TPT>(tl + kTD2 + 128 + TPT * qf, o2);
            tmem_ld_wait();
            float* sr = srow + KPP * pass;
#pragma unroll
            for (int q = 0; q < KPP / 4; ++q) {
                const float4 e4 = eg4[k0 / 4 + q];
                sr[4 * q] = fmaf(sr[4 * q], e4.x, d[4 * q]);
                sr[4 * q + 1] = fmaf(sr[4 * q + 1], e4.y, d[4 * q + 1]);
                sr[4 * q + 2] = fmaf(sr[4 * q + 2], e4.z, d[4 * q + 2]);
                sr[4 * q + 3] = fmaf(sr[4 * q + 3], e4.w, d[4 * q + 3]);
            }
            tmem_put_split_n<KPP>(tl + kTA1 + k0 / 2, tl + kTA1 + 64 + k0 / 2, sr);
            tmem_st_wait();
            tc_fence_before();
            __syncthreads();   // pass 1: block st consumed; S^T in place for the next MMA-1
            tc_fence_after();
            if (tid == 0 && c + 1 < nch) {
                const int s1 = (c + 1) % kInterStages;
                if (pass == 0)
                    next_ok = mbar_wait_bounded(&sm.bar_ld[s1], (uint32_t)(((c + 1) / kInterStages) & 1),
                                                a.err);
                if (next_ok) {
                    tc_fence_after();
                    mma1_half(s1, 4 * pass);
                    if (pass == 1) tc_commit(&sm.bar_mma);
                }
            }
        }
        if (tid == 32 && c + kInterStages < nch) issue(c + kInterStages, st);
        // the chunk's o rows into the staging tile while the next MMA-1 runs
#pragma unroll
        for (int t = 0; t < TPT; ++t) ot[t * 128] = __fmul_rn(scale, o1[t] + o2[t]);
        fence_proxy_async_smem();
    }
    failed = __syncthreads_or(failed || late_fail) != 0;
    if (!NORM && ostore_lane) {
        if (!failed && nch > 0) flush_o(nch - 1);
        bulk_wait_all();
    }
    if (NORM && !failed && nch > 0) norm_chunk(nch - 1);
    if (NORM) cp_async_wait_all();               // no copy may land after the CTA has left
    if (!failed) {
        float* srow_out = a.state_out + (((long)n * H + h) * kHeadDim + v) * kHeadDim;
#pragma unroll
        for (int pass = 0; pass < 2; ++pass)
#pragma unroll
            for (int j = 0; j < KPP / 4; ++j) {
                const float* x = srow + KPP * pass + 4 * j;
                __stcs(reinterpret_cast<float4*>(srow_out + 64 * pass + KPP * qf + 4 * j),
                       make_float4(x[0], x[1], x[2], x[3]));
            }
    } else {
        mbar_wait_bounded(&sm.bar_mma, mph, nullptr);   // let in-flight MMAs drain (bounded)
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, 512);
}

// ============================================================================================
// host side
// ============================================================================================

long chunk_count(const SeqLayout& s, const int* cu_host) {
    if (s.cu_seqlens == nullptr) return (long)s.N * ((s.T_uniform + kCc - 1) / kCc);
    long total = 0;
    for (int n = 0; n < s.N; ++n) total += (cu_host[n + 1] - cu_host[n] + kCc - 1) / kCc;
    return total;
}

size_t chunk_workspace_bytes(const SeqLayout& s, const int* cu_host, int H) {
    const size_t header =
        s.cu_seqlens ? (((size_t)(s.N + 1) * 4 + kHeaderAlign - 1) / kHeaderAlign) * kHeaderAlign : 0;
    return header + (size_t)chunk_count(s, cu_host) * H * kBlkBytes;
}

cudaError_t launch_chunk_offsets(const SeqLayout& seq, void* workspace, int** chunk_off,
                                 unsigned char** blocks, cudaStream_t s) {
    *chunk_off = nullptr;
    *blocks = static_cast<unsigned char*>(workspace);
    if (seq.cu_seqlens == nullptr) return cudaSuccess;
    *chunk_off = reinterpret_cast<int*>(workspace);
    *blocks += ((size_t)(seq.N + 1) * 4 + kHeaderAlign - 1) / kHeaderAlign * kHeaderAlign;
    KernelTimer kt(kKChunkOffsets, s);
    kda_chunk_offsets_kernel<<<1, 1024, 0, s>>>(seq.cu_seqlens, seq.N, *chunk_off);
    return cudaGetLastError();
}

template <int GM, bool NORM>
static cudaError_t launch_inter_t(const ScanArgs& a, const int* chunk_off,
                                  const unsigned char* blocks, const PrepArgs& ring, cudaStream_t s) {
    const size_t smem2 = sizeof(InterSmem) + 128;
    static PerDevice<int> done2;
    cudaError_t e = set_smem(kda_chunk_inter_kernel<GM, NORM>, smem2, done2);
    if (e != cudaSuccess) return e;
    dim3 g2((unsigned)a.H, (unsigned)a.seq.N);
    CUtensorMap tmo;
    if (!make_tensor_map_2d(&tmo, a.o, a.seq.total_rows, (long)a.H * kHeadDim, kHeadDim, kCc))
        return cudaErrorInvalidValue;
    KernelTimer kt(kKChunkInter, s);
    kda_chunk_inter_kernel<GM, NORM><<<g2, kThrInter, smem2, s>>>(a, chunk_off, blocks, tmo, ring);
    return cudaGetLastError();
}

cudaError_t launch_chunk_inter(const ScanArgs& a, const int* chunk_off,
                               const unsigned char* blocks, cudaStream_t s, const PrepArgs* ring) {
    PrepArgs none;
    std::memset(&none, 0, sizeof(none));
    const PrepArgs& r = ring != nullptr ? *ring : none;
    if (a.norm_y != nullptr)
        return (a.gate_mode & 1) == 0 ? launch_inter_t<0, true>(a, chunk_off, blocks, r, s)
                                      : launch_inter_t<1, true>(a, chunk_off, blocks, r, s);
    return (a.gate_mode & 1) == 0 ? launch_inter_t<0, false>(a, chunk_off, blocks, r, s)
                                  : launch_inter_t<1, false>(a, chunk_off, blocks, r, s);
}

template <int GM, bool EXP>
static cudaError_t launch_chunk_t(const ScanArgs& a, const int* cu_host, void* workspace,
                                  cudaStream_t s) {
    const long nchunks = chunk_count(a.seq, cu_host);
    int* chunk_off = nullptr;
    unsigned char* ws = nullptr;
    cudaError_t e = launch_chunk_offsets(a.seq, workspace, &chunk_off, &ws, s);
    if (e != cudaSuccess) return e;
    if (nchunks > 0) {
        const size_t smem1 = sizeof(IntraSmem) + 128;
        static PerDevice<int> done1;
        e = set_smem(kda_chunk_intra_kernel<GM, EXP>, smem1, done1);
        if (e != cudaSuccess) return e;
        dim3 g1((unsigned)nchunks, (unsigned)a.H);
        KernelTimer kt(kKChunkIntra, s);
        kda_chunk_intra_kernel<GM, EXP><<<g1, kThr, smem1, s>>>(a, chunk_off, ws);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return launch_chunk_inter(a, chunk_off, ws, s);
}

cudaError_t launch_scan_chunk(const ScanArgs& a, const int* cu_host, void* workspace,
                              cudaStream_t s) {
    if (a.seq.N == 0) return cudaSuccess;
    if (a.seq.total_rows == 0) {
        const size_t bytes = (size_t)a.seq.N * a.H * kHeadDim * kHeadDim * sizeof(float);
        return cudaMemcpyAsync(a.state_out, a.state_in, bytes, cudaMemcpyDeviceToDevice, s);
    }
    const bool exp_done = (a.gate_mode & 2) != 0;
    if ((a.gate_mode & 1) == 0)
        return exp_done ? launch_chunk_t<0, true>(a, cu_host, workspace, s)
                        : launch_chunk_t<0, false>(a, cu_host, workspace, s);
    return exp_done ? launch_chunk_t<1, true>(a, cu_host, workspace, s)
                    : launch_chunk_t<1, false>(a, cu_host, workspace, s);
}

}  // namespace kda
