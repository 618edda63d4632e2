// kda_chunk_prep.cu -- the fused prefill's first kernel: stages 2-4 of kda_core_gated (conv +
// SiLU, l2 norm, gates, beta; "memra_engine/kda.rs", memra-engine 0.125.0) computed straight
// into the chunked form's intra-chunk operand images, so the prepared q, k, v and gate planes never
// reach memory.  Persistent CTAs (two per SM) loop over (32-token chunk, head) tasks; from the
// images on, a task runs the same MMA tail as the chunked scan's intra kernel
// (kda_chunk_common.cuh), and while it runs the next task's inputs are copied into shared memory.
//
// Layout: 256 threads; warp w takes tokens 4w .. 4w+3 of the chunk and lane l channels 4l .. 4l+3
// of the head, the prep kernel's lane-to-channel map, so every per-token quantity is computed
// with the prep's arithmetic: conv taps oldest first over a window that starts K-1 samples back
// (from the ring for the first chunk of a sequence), SiLU, the l2 sum of squares reduced over the
// warp (a transposed butterfly that adds the same pairs as the prep's per-row butterfly), gates
// and beta.  The column images (consecutive tokens of one channel) are written from a thread's
// registers as 8-byte half rows of their 16-byte core-matrix rows; the row images (8 consecutive
// channels of one token) pair lane l with l^1 by shuffles.  The per-channel running sum of the
// gate passes from warp to warp through shared memory in token order, the order of the chunked
// scan's own intra kernel.  The output blocks therefore equal those of the prep kernel followed
// by the intra kernel bit for bit in the rows of live tokens; the rows of tokens past a sequence's
// end (zero beta and gates, so zero U' rows, and readout rows that are never stored) may differ,
// and the results (readout, state, ring) are equal.
#include <cstddef>
#include <cstring>

#include "kda_chunk_common.cuh"

namespace kda {

constexpr int kTokW = 4;      // tokens per warp: 8 warps cover one 32-token chunk
constexpr int kThrF = 256;    // threads of the fused kernel

template <bool BF16>
struct RawVec;
template <>
struct RawVec<true> { using T = uint2; };     // 4 bf16 channels
template <>
struct RawVec<false> { using T = float4; };   // 4 f32 channels

template <bool BF16>
__device__ __forceinline__ typename RawVec<BF16>::T raw_ld(const void* base, long idx) {
    if constexpr (BF16) {
        return __ldg(reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(base) + idx));
    } else {
        return __ldg(reinterpret_cast<const float4*>(reinterpret_cast<const float*>(base) + idx));
    }
}

template <bool BF16>
__device__ __forceinline__ typename RawVec<BF16>::T raw_zero() {
    if constexpr (BF16) return make_uint2(0u, 0u);
    else return make_float4(0.0f, 0.0f, 0.0f, 0.0f);
}

template <bool BF16>
__device__ __forceinline__ float4 raw_unpack(const typename RawVec<BF16>::T& u) {
    if constexpr (BF16) {
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
        return make_float4(a.x, a.y, b.x, b.y);
    } else {
        return u;
    }
}

__device__ __forceinline__ float f4c(const float4& v, int e) {
    return e == 0 ? v.x : (e == 1 ? v.y : (e == 2 ? v.z : v.w));
}

// One plane's raw samples for this lane's 4 channels: the KW-1 samples before the warp's first
// token (halo, f32) and the warp's 4 tokens (raw, packed).
template <bool BF16, int KW>
struct PlaneRaw {
    float4 halo[KW - 1];
    typename RawVec<BF16>::T cur[kTokW];
};

// Issue the loads of one plane.  pos0 = position of the warp's first token in its sequence;
// ring_base = this plane's ring row of channel c4 (channel e at + e*R).
template <bool BF16, bool CONV, int KW>
__device__ __forceinline__ void plane_load(PlaneRaw<BF16, KW>& P, const void* raw, long C, long c4,
                                           long begin, long pos0, int ntok, const float* ring_in,
                                           long ring_base, int R) {
#pragma unroll
    for (int i = 0; i < kTokW; ++i)
        P.cur[i] = i < ntok ? raw_ld<BF16>(raw, (begin + pos0 + i) * C + c4) : raw_zero<BF16>();
#pragma unroll
    for (int m = 0; m < KW - 1; ++m) P.halo[m] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (CONV && ntok > 0) {                       // (a warp past the sequence end loads nothing)
#pragma unroll
        for (int m = 0; m < KW - 1; ++m) {
            const int d = KW - 1 - m;                 // samples back from the first token
            const long pos = pos0 - d;
            float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (d <= R) {
                if (pos >= 0) {
                    v = raw_unpack<BF16>(raw_ld<BF16>(raw, (begin + pos) * C + c4));
                } else {
                    const long s2 = R + pos;
                    v = make_float4(ring_in[ring_base + s2], ring_in[ring_base + R + s2],
                                    ring_in[ring_base + 2 * R + s2], ring_in[ring_base + 3 * R + s2]);
                }
            }
            P.halo[m] = v;
        }
    }
}

// conv + SiLU of one plane for the warp's 4 tokens (or the raw samples without a conv).
template <bool BF16, bool CONV, int KW>
__device__ __forceinline__ void plane_conv(const PlaneRaw<BF16, KW>& P, const float (&w)[4][KW],
                                           float (&y)[kTokW][4]) {
    float4 cur[kTokW];
#pragma unroll
    for (int i = 0; i < kTokW; ++i) cur[i] = raw_unpack<BF16>(P.cur[i]);
#pragma unroll
    for (int i = 0; i < kTokW; ++i) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if constexpr (CONV) {
                float win[KW];
#pragma unroll
                for (int m = 0; m < KW; ++m) {
                    const int idx = i + m;            // window slot m = sample at token i-(KW-1)+m
                    win[m] = idx < KW - 1 ? f4c(P.halo[idx], e) : f4c(cur[idx - (KW - 1)], e);
                }
                // a K-tap conv (K < KW) meets zero weights and zero samples in its first KW - K
                // slots, so every slot runs unpredicated, adding exact zeros: the same sum as the
                // prep kernel's K taps, without a per-tap test
                float acc = 0.0f;
#pragma unroll
                for (int m = 0; m < KW; ++m) acc = fmaf(w[e][m], win[m], acc);
                y[i][e] = silu_f(acc);
            } else {
                y[i][e] = f4c(cur[i], e);
            }
        }
    }
}

// The staged (transposed) weights of channels kq .. kq+3: one 16-byte load per tap slot (tap j of
// a K-tap conv sits in slot j + KW - K, the slots before it hold zeros).
template <int KW>
__device__ __forceinline__ void plane_weights_t(const float* wt, int kq, float (&w)[4][KW]) {
#pragma unroll
    for (int m = 0; m < KW; ++m) {
        const float4 x = *reinterpret_cast<const float4*>(wt + m * kHeadDim + kq);
        w[0][m] = x.x; w[1][m] = x.y; w[2][m] = x.z; w[3][m] = x.w;
    }
}

template <int KW>
__device__ __forceinline__ void plane_weights(const float* conv_w, long row, int K, float (&w)[4][KW]) {
#pragma unroll
    for (int e = 0; e < 4; ++e)
#pragma unroll
        for (int m = 0; m < KW; ++m) {
            const int j = m - (KW - K);
            w[e][m] = j >= 0 ? conv_w[(row + e) * K + j] : 0.0f;
        }
}

// Sum 8 per-lane values over the warp with 9 shuffles: on return lanes 4j .. 4j+3 hold the total
// of value j.  Each step adds a lane's own partial and its partner's, the pairs of a per-value
// butterfly (xor 16, 8, 4, 2, 1), so the totals equal warp_sum's bit for bit.
__device__ __forceinline__ float warp_sum8(float (&x)[8]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int w = 4; w >= 1; w >>= 1) {
        const int off = 4 * w;
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < w; ++i) {
            const float send = upper ? x[i] : x[i + w];
            const float keep = upper ? x[i + w] : x[i];
            x[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
    float t = x[0] + __shfl_xor_sync(0xffffffffu, x[0], 2);
    return t + __shfl_xor_sync(0xffffffffu, t, 1);
}

// the chunk of global index gid: its sequence n and rows, the chunk's first row and its tokens
__device__ __forceinline__ void chunk_task(const SeqLayout& L, const int* chunk_off, long gid,
                                           int& n, long& begin, long& end, long& row0, int& nt) {
    if (L.cu_seqlens == nullptr) {          // gid < 2^31 (host check)
        n = (int)((unsigned)gid / (unsigned)((L.T_uniform + kCc - 1) / kCc));
    } else {
        int lo = 0, hi = L.N;                    // largest n with chunk_off[n] <= gid
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if ((long)chunk_off[mid] <= gid) lo = mid; else hi = mid;
        }
        n = lo;
    }
    seq_range(L, n, begin, end);
    row0 = begin + (gid - chunk_base(L, chunk_off, n)) * kCc;
    nt = (int)min((long)kCc, end - row0);
}

// A task of the persistent kernel: (global chunk gid, head h), task = h * nchunks + gid, and the
// chunk's sequence n, rows and token count.  The host keeps h * nchunks + gid below 2^31.  h is
// a 128-wide value unit: with value heads vs * 128 wide it is column block h % vs of value head
// gh = h / vs, whose gate, beta and q/k head hq = gh % Hk it reads.
struct TaskPos {
    long begin, end, row0, gid;
    int n, h, nt;
    int gh, hq;
};

__device__ __forceinline__ TaskPos task_pos(const SeqLayout& L, const int* chunk_off, long task,
                                            long nchunks, int vs, int Hk) {
    TaskPos t;
    const unsigned tk = (unsigned)task, nc = (unsigned)nchunks;
    t.h = (int)(tk / nc);
    t.gid = (long)(tk - (unsigned)t.h * nc);
    t.gh = vs == 1 ? t.h : t.h / vs;
    t.hq = t.gh < Hk ? t.gh : t.gh % Hk;
    chunk_task(L, chunk_off, t.gid, t.n, t.begin, t.end, t.row0, t.nt);
    return t;
}

// Staged bf16 raw rows of one task: [plane][row][128 channels], row r = chunk token r - (KW-1)
// (the conv halo first).  Lives in sm.bia[1] + sm.kb (32 KB), free from the end of one task's
// MMA-a to the next task's conv.
template <int KW>
struct RawStage {
    static constexpr int kRows = kCc + KW - 1;
    __nv_bfloat16 v[3][kRows][kHeadDim];
};

// 4 f32 values as bf16 hi / lo at byte offset off (8-byte aligned) of two images: half of a
// 16-byte core-matrix row.
__device__ __forceinline__ void put4x(unsigned char* hi_img, unsigned char* lo_img, uint32_t off,
                                      const float (&x)[4]) {
    uint2 hi, lo;
    split_bf16x2(x[0], x[1], hi.x, lo.x);
    split_bf16x2(x[2], x[3], hi.y, lo.y);
    *reinterpret_cast<uint2*>(hi_img + off) = hi;
    *reinterpret_cast<uint2*>(lo_img + off) = lo;
}

// One 8-channel row of this lane's half of the warp's tokens (even lane: tokens 0-1, odd lane:
// tokens 2-3): own 4 channels plus the partner lane's 4, in channel order.  Row j is token j ^ sw
// of the half (sw is the same for both lanes of a pair), so that lanes with sw set write their two
// rows in the other order and a 16-byte store of the warp touches four row slots of the core
// matrices instead of two.  One row at a time: the row images then fit in 128 registers without
// a spill (both rows at once spilled, and measured 2 % slower).
__device__ __forceinline__ void pair_row(const float (&x)[kTokW][4], float (&row)[8], bool sw, int j) {
    const bool odd = (threadIdx.x & 1) != 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float lo_t = sw ? x[1 - j][e] : x[j][e];          // token j ^ sw
        const float hi_t = sw ? x[3 - j][e] : x[2 + j][e];      // token 2 + (j ^ sw)
        const float send = odd ? lo_t : hi_t;
        const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
        row[e] = odd ? recv : lo_t;
        row[4 + e] = odd ? hi_t : recv;
    }
}

// Tensor maps of the raw rows: q, k [rows, Cq] and v [rows, C] bf16 with a [kRows, 128] box, and
// (KDA) the gate input f [rows, Cg] f32 with a [32, 128] box.
struct RawMaps {
    CUtensorMap q, k, v, f;
    CUtensorMap ut;              // the workspace blocks' U rows (the MMA tail's epilogue)
};

// Issued by one thread: TMA tile loads of task tp's raw q, k, v rows (the chunk's tokens and the
// KW-1 rows before them) into the stage, counted on bar.  Rows before the tensor or past its end
// read as zeros; rows of a neighbouring sequence are loaded but never read (the conv takes the
// halo from the ring before the sequence start, and tokens past the chunk end are masked).
template <int KW>
__device__ __forceinline__ void stage_raw(RawStage<KW>& st, const RawMaps& m, const TaskPos& tp,
                                          uint64_t* bar) {
    mbar_arrive_expect_tx(bar, 3u * RawStage<KW>::kRows * kHeadDim * sizeof(__nv_bfloat16));
    const int xq = tp.hq * kHeadDim, x = tp.h * kHeadDim, y = (int)tp.row0 - (KW - 1);
    tma_load_2d(&st.v[0][0][0], &m.q, xq, y, bar);
    tma_load_2d(&st.v[1][0][0], &m.k, xq, y, bar);
    tma_load_2d(&st.v[2][0][0], &m.v, x, y, bar);
}

// Issued by one thread: the TMA tile load of task tp's gate-input rows (KDA: [32 tokens][128]
// f32) into sm.scr, free from the end of one task's Tm image to the next task's gate step.
__device__ __forceinline__ void stage_f(float* dst, const RawMaps& m, const TaskPos& tp,
                                        uint64_t* bar) {
    mbar_arrive_expect_tx(bar, kCc * kHeadDim * sizeof(float));
    tma_load_2d(dst, &m.f, tp.gh * kHeadDim, (int)tp.row0, bar);
}

__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(src))
                 : "memory");
}

// Staged small inputs of one task: the head's conv weights (K <= 4 taps, transposed to
// [plane][tap slot][channel] so a lane reads its 4 channels' tap as one conflict-free 16-byte load;
// tap j in slot j + 4 - K, the leading slots zeroed once per CTA),
// dt_bias (KDA: the head's 128 channels; GDN: one value), A_log of the head, and the chunk's raw
// beta and (GDN) gate inputs.  Filled during the previous task's MMA tail, so that the front half
// waits on no global load; a region of its own, read only by the front half.
struct ParamStage {
    float w[3][4 * kHeadDim];
    float dt[kHeadDim];
    float braw[kCc];
    float fraw[kCc];
    float alog;
};

struct __align__(128) PrepIntraSmem {
    IntraSmem in;
    ParamStage ps;
    alignas(128) float gtot[kThrF / 32][kHeadDim];   // the warps' 4-token gate totals (KDA),
                                                     // read and written as float4
    uint64_t bar_raw, bar_f;                     // TMA completion of the raw rows, the gate input
};
// TMA destinations and sources inside the layout (its base aligned to 1024 bytes): the raw-row
// stage at sm.bia[1] and the gate input at sm.scr (128-byte aligned), the epilogue's swizzled U
// tiles at sm.ktv[0] (1024-byte aligned).
static_assert(offsetof(IntraSmem, bia) + sizeof(IntraSmem::bia[0]) == 16384, "stage at 16 KB");
static_assert(offsetof(IntraSmem, ktv) % 1024 == 0, "U tiles 1024-byte aligned");
static_assert(offsetof(IntraSmem, scr) % 128 == 0, "gate input 128-byte aligned");
// 16-byte vector accesses into the parameter stage and the gate totals
static_assert(offsetof(PrepIntraSmem, ps) % 16 == 0 && offsetof(ParamStage, dt) % 16 == 0,
              "dt_bias stage 16-byte aligned");
static_assert(offsetof(PrepIntraSmem, gtot) % 16 == 0, "gate totals 16-byte aligned");
// the dynamic allocation: the layout plus room to align it to 1024 bytes (128-byte swizzled tiles)
constexpr size_t kPrepIntraSmemBytes = sizeof(PrepIntraSmem) + 1024;
// two resident CTAs per SM: 228 KB of shared memory per SM, 1 KB of it reserved per CTA
static_assert(2 * (kPrepIntraSmemBytes + 1024) <= 228 * 1024, "two CTAs per SM");

// Issue the cp.async copies of task tp's small inputs into the parameter stage (H units, Hg gate
// heads).
template <int GATE_MODE, bool CONV, int KW>
__device__ __forceinline__ void stage_params(ParamStage& ps, const PrepArgs& p, int H, int Hg,
                                             const TaskPos& tp) {
    const int tid = threadIdx.x, h = tp.h, gh = tp.gh, nt = tp.nt;
    const long row0 = tp.row0;
    if constexpr (CONV) {
        const int K = p.K, per = kHeadDim * K;   // one plane's rows of this head, contiguous
        const int hq = tp.hq;                    // the q and k planes' head
#pragma unroll 1
        for (int pl = 0; pl < 3; ++pl) {
            const float* src =
                p.conv_w + (plane_offset(H, p.Hk, pl) + (long)(pl < 2 ? hq : h) * kHeadDim) * K;
            for (int r = tid; r < per; r += kThrF) {
                const int ch = K == 4 ? r >> 2 : r / K, j = r - ch * K;
                cp_async4(&ps.w[pl][(j + KW - K) * kHeadDim + ch], src + r);
            }
        }
    }
    if (GATE_MODE == 0) {
        if (tid < kHeadDim / 4) cp_async16(&ps.dt[4 * tid], p.dt_bias + (long)gh * kHeadDim + 4 * tid);
    } else if (tid == kThrF - 1) {
        cp_async4(&ps.dt[0], p.dt_bias + gh);
    }
    if (tid == kThrF - 2) cp_async4(&ps.alog, p.a_log + gh);
    if (tid < nt) {
        cp_async4(&ps.braw[tid], p.beta_raw + (row0 + tid) * Hg + gh);
        if (GATE_MODE == 1) cp_async4(&ps.fraw[tid], p.f_raw + (row0 + tid) * Hg + gh);
    }
    cp_async_commit();
}

// The staged samples of one plane for this lane's 4 channels: the halo (from the stage, or the
// ring before the sequence start) and the warp's tokens, in the PlaneRaw form the conv reads.
template <int KW>
__device__ __forceinline__ void plane_from_stage(PlaneRaw<true, KW>& P, const RawStage<KW>& st,
                                                 int pl, int t0, int kq, long pos0, int R,
                                                 const float* ring_in, long ring_base) {
#pragma unroll
    for (int i = 0; i < kTokW; ++i)
        P.cur[i] = *reinterpret_cast<const uint2*>(&st.v[pl][t0 + i + KW - 1][kq]);
    if (pos0 >= KW - 1 && R == KW - 1) {        // the whole window inside the sequence
#pragma unroll
        for (int m = 0; m < KW - 1; ++m)
            P.halo[m] = raw_unpack<true>(*reinterpret_cast<const uint2*>(&st.v[pl][t0 + m][kq]));
        return;
    }
#pragma unroll
    for (int m = 0; m < KW - 1; ++m) {
        const int d = KW - 1 - m;
        const long pos = pos0 - d;
        float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (d <= R) {
            if (pos >= 0) {
                v = raw_unpack<true>(*reinterpret_cast<const uint2*>(&st.v[pl][t0 + m][kq]));
            } else {
                const long s2 = R + pos;
                v = make_float4(ring_in[ring_base + s2], ring_in[ring_base + R + s2],
                                ring_in[ring_base + 2 * R + s2], ring_in[ring_base + 3 * R + s2]);
            }
        }
        P.halo[m] = v;
    }
}

// Persistent: CTA b takes tasks b, b + gridDim.x, ... (task = head * nchunks + chunk).  With bf16
// raw input the next task's raw rows, gate input and small inputs are copied into shared memory
// while this task's MMA tail runs (PF); f32 raw rows do not fit the free space and are loaded
// directly, as are conv weights of more than 4 taps.
template <bool BF16, int GATE_MODE, bool CONV, int KW>
__global__ void __launch_bounds__(kThrF, 2)
kda_chunk_prep_intra_kernel(PrepArgs p, ScanArgs a, const int* chunk_off, unsigned char* ws,
                            long nchunks, const __grid_constant__ RawMaps maps) {
    constexpr bool PF = BF16;
    constexpr bool PW = PF && CONV && KW <= 4;   // conv weights from the parameter stage
    extern __shared__ unsigned char smem_raw[];
    PrepIntraSmem& smf = *reinterpret_cast<PrepIntraSmem*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    IntraSmem& sm = smf.in;
    ParamStage& ps = smf.ps;
    RawStage<KW>& stage = *reinterpret_cast<RawStage<KW>*>(sm.bia[1]);
    static_assert(sizeof(RawStage<KW>) <= sizeof(sm.bia[1]) + sizeof(sm.kb), "stage fits");
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.H;
    const long C = (long)H * kHeadDim;
    // grouped queries: the q and k planes hold Hk heads ([rows, Cq]); task head h reads q/k head
    // h % Hk, and the conv weights and ring rows are [q | k | v] = [Cq | Cq | C]
    const int Hk = prep_qk_heads(H, p.Hk);
    const long Cq = (long)Hk * kHeadDim;
    // value heads wider than 128: H counts 128-wide units, vs of them per value head; the gate
    // rows (KDA) are Cg = Hg * 128 wide and beta (and the GDN gate) Hg per row
    const int vs = value_sub(a);
    const int Hg = prep_gate_heads(p);
    const long Cg = (long)Hg * kHeadDim;
    const long ntasks = nchunks * H;
    const int kq = 4 * lane;                     // first of this lane's channels within the head
    const int t0 = kTokW * warp;                 // the warp's first token within the chunk
    const int K = p.K, R = p.K - 1;

    if (warp == 0) {
        tmem_alloc(&sm.tmem_base, 256);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&sm.bar, 1);
        mbar_init(&smf.bar_raw, 1);
        mbar_init(&smf.bar_f, 1);
        fence_mbar_init();
    }
    uint32_t phase = 0, ph_ld = 0;               // MMA commits; staged loads (one per task)
    bool ld_pending = false;                     // a task's loads issued and not yet waited on
    if constexpr (PW) {                          // leading weight slots of a conv shorter than KW
        for (int i = tid; i < 3 * (KW - K) * kHeadDim; i += kThrF)
            ps.w[i / ((KW - K) * kHeadDim)][i % ((KW - K) * kHeadDim)] = 0.0f;
    }
    if (PF && (long)blockIdx.x < ntasks) {
        const TaskPos tp = task_pos(a.seq, chunk_off, blockIdx.x, nchunks, vs, Hk);
        if (tid == 0) {
            prefetch_tensormap(&maps.q);
            prefetch_tensormap(&maps.k);
            prefetch_tensormap(&maps.v);
            stage_raw<KW>(stage, maps, tp, &smf.bar_raw);
            if (GATE_MODE == 0) stage_f(sm.scr, maps, tp, &smf.bar_f);
        }
        stage_params<GATE_MODE, PW, KW>(ps, p, H, Hg, tp);
    }
    __syncthreads();

    for (long task = blockIdx.x; task < ntasks; task += gridDim.x) {
    const TaskPos tp = task_pos(a.seq, chunk_off, task, nchunks, vs, Hk);
    const long gid = tp.gid;                     // global chunk index
    const int h = tp.h, gh = tp.gh, n = tp.n, nt = tp.nt;
    const long begin = tp.begin, row0 = tp.row0;
    const long c = (row0 - begin) / kCc;
    unsigned char* blk = ws + ((long)gid * H + h) * kBlkBytes;
    const long c4 = (long)h * kHeadDim + kq;     // this lane's first channel within the v plane
    const long cq4 = (long)tp.hq * kHeadDim + kq;   // ... and within the q and k planes
    const long cg4 = (long)gh * kHeadDim + kq;      // ... and within the gate rows
    const int ntok = max(0, min(kTokW, nt - t0));

    // ---- loads: the gate input and beta; raw q, k, v (staged, or direct) -----------------------
    float4 fr[kTokW];
    if (GATE_MODE == 0 && !PF) {
#pragma unroll
        for (int i = 0; i < kTokW; ++i)
            fr[i] = i < ntok ? __ldg(reinterpret_cast<const float4*>(p.f_raw + (row0 + t0 + i) * Cg + cg4))
                             : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
    if (!PF && tid < kCc) {
        const bool live = tid < nt;
        sm.beta[tid] = live ? sigmoid_f(p.beta_raw[(row0 + tid) * Hg + gh]) : 0.0f;
        if (GATE_MODE == 1)
            sm.gs[tid] = live ? gdn_gate_f(p.f_raw[(row0 + tid) * Hg + gh], p.dt_bias[gh], p.a_log[gh]) : 0.0f;
    }
    const long pos0 = c * kCc + t0;
    const long rr = (long)n * (2 * Cq + C) * R;
    PlaneRaw<BF16, KW> rq, rk, rv;               // direct loads (no staging)
    if constexpr (PF) {
        bool ld_ok = mbar_wait_bounded(&smf.bar_raw, ph_ld, a.err);
        if (GATE_MODE == 0) ld_ok = mbar_wait_bounded(&smf.bar_f, ph_ld, a.err) && ld_ok;
        ph_ld ^= 1u;
        ld_pending = false;
        cp_async_wait_all();
        if (nt < kCc && ld_ok) {
            // a ragged chunk: its stage rows past the last token (the next sequence's rows, or
            // zeros past the tensor) are cleared, so that whatever they held, every value computed
            // for a token past the end stays finite (those tokens meet zero beta and zero gates)
            constexpr int kPieces = kHeadDim / 4;        // 8-byte pieces of a stage row
            const int dead = kCc - nt;
            for (int i = tid; i < 3 * dead * kPieces; i += kThrF) {
                const int pl = i / (dead * kPieces), r = (i / kPieces) % dead, c = i % kPieces;
                *reinterpret_cast<uint2*>(&stage.v[pl][KW - 1 + nt + r][4 * c]) = make_uint2(0u, 0u);
            }
        }
        if (__syncthreads_or(!ld_ok)) break;     // every piece of the stage has landed
        if (tid < kCc) {
            const bool live = tid < nt;
            sm.beta[tid] = live ? sigmoid_f(ps.braw[tid]) : 0.0f;
            if (GATE_MODE == 1)
                sm.gs[tid] = live ? gdn_gate_f(ps.fraw[tid], ps.dt[0], ps.alog) : 0.0f;
        }
        if (GATE_MODE == 0) {                    // (rows past the end: their gates are masked)
#pragma unroll
            for (int i = 0; i < kTokW; ++i)
                fr[i] = *reinterpret_cast<const float4*>(&sm.scr[(t0 + i) * kHeadDim + kq]);
        }
    } else {
        plane_load<BF16, CONV, KW>(rq, p.q_raw, Cq, cq4, begin, pos0, ntok, p.ring_in, rr + (0 * Cq + cq4) * R, R);
        plane_load<BF16, CONV, KW>(rk, p.k_raw, Cq, cq4, begin, pos0, ntok, p.ring_in, rr + (1 * Cq + cq4) * R, R);
        plane_load<BF16, CONV, KW>(rv, p.v_raw, C, c4, begin, pos0, ntok, p.ring_in, rr + (2 * Cq + c4) * R, R);
    }

    // ---- conv + SiLU; l2 norm of q and k over the head (one warp = one token group) ------------
    float v[kTokW][4], k[kTokW][4], q[kTokW][4];
    {
        float w[4][KW];
        if constexpr (PF) {                      // one plane's samples live at a time
            const int Rr = CONV ? R : 0;
#pragma unroll
            for (int pl = 2; pl >= 0; --pl) {
                PlaneRaw<true, KW> pr;
                const long crow = pl * Cq + (pl < 2 ? cq4 : c4);   // conv / ring row of channel
                plane_from_stage<KW>(pr, stage, pl, t0, kq, pos0, Rr, p.ring_in, rr + crow * R);
                if constexpr (PW) plane_weights_t<KW>(ps.w[pl], kq, w);
                else if constexpr (CONV) plane_weights<KW>(p.conv_w, crow, K, w);
                plane_conv<true, CONV, KW>(pr, w, pl == 2 ? v : (pl == 1 ? k : q));
            }
        } else {
            if constexpr (CONV) plane_weights<KW>(p.conv_w, 2 * Cq + c4, K, w);
            plane_conv<BF16, CONV, KW>(rv, w, v);
            if constexpr (CONV) plane_weights<KW>(p.conv_w, 1 * Cq + cq4, K, w);
            plane_conv<BF16, CONV, KW>(rk, w, k);
            if constexpr (CONV) plane_weights<KW>(p.conv_w, 0 * Cq + cq4, K, w);
            plane_conv<BF16, CONV, KW>(rq, w, q);
        }
    }
    {
        float ss[2 * kTokW];
#pragma unroll
        for (int i = 0; i < kTokW; ++i) {
            float s = __fmul_rn(q[i][0], q[i][0]);
            s = fmaf(q[i][1], q[i][1], s); s = fmaf(q[i][2], q[i][2], s); s = fmaf(q[i][3], q[i][3], s);
            ss[i] = s;
            s = __fmul_rn(k[i][0], k[i][0]);
            s = fmaf(k[i][1], k[i][1], s); s = fmaf(k[i][2], k[i][2], s); s = fmaf(k[i][3], k[i][3], s);
            ss[kTokW + i] = s;
        }
        const float part = warp_sum8(ss);
#pragma unroll
        for (int i = 0; i < kTokW; ++i) {
            const float iq = l2_inv_f(__shfl_sync(0xffffffffu, part, 4 * i), p.l2_eps);
            const float ik = l2_inv_f(__shfl_sync(0xffffffffu, part, 4 * (kTokW + i)), p.l2_eps);
            // a token past the sequence end keeps its (finite) values: its beta and gates are zero,
            // so it adds nothing to A, W, U or the state, and its readout rows are never stored
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                q[i][e] *= iq;
                k[i][e] *= ik;
            }
        }
    }

    // ---- running gate sum G (per channel, KDA) in token order, warp to warp --------------------
    float G[kTokW][4];
    float GCh = 0.0f;                            // per-head gate: the chunk's total
    float cref_l[4], ecr_l[4];                   // KDA: c = G_C / 2 and e^c of this lane's channels
    if (GATE_MODE == 0) {
        const float rate = expf(PF ? ps.alog : p.a_log[gh]);
        const float4 dt = PF ? *reinterpret_cast<const float4*>(&ps.dt[kq])
                             : *reinterpret_cast<const float4*>(p.dt_bias + cg4);
        const float dtv[4] = {dt.x, dt.y, dt.z, dt.w};
        float g[kTokW][4];
#pragma unroll
        for (int i = 0; i < kTokW; ++i)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                g[i][e] = i < ntok ? kda_gate_f(f4c(fr[i], e), dtv[e], rate, p.gate_lb) : 0.0f;
        // blocked running sum (the chunked intra kernel's order): each warp sums its 4 tokens in
        // order from 0, the warps' totals go through shared memory, and warp w adds the totals
        // of warps 0 .. w-1 in order, starting from 0
        float run[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int i = 0; i < kTokW; ++i)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                run[e] += g[i][e];
                G[i][e] = run[e];
            }
        float* gtot = &smf.gtot[0][0];
        *reinterpret_cast<float4*>(&gtot[warp * kHeadDim + kq]) = make_float4(run[0], run[1], run[2], run[3]);
        __syncthreads();
        // one pass over the warps' totals in order from 0: the prefix before this warp (pre) and,
        // in every warp from the same additions as warp 7's last token (so the same bits), the
        // chunk total -- the reference c = G_C / 2 and e^c of this lane's channels, for the row
        // images without another barrier
        float pre[4] = {0.0f, 0.0f, 0.0f, 0.0f}, tot[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int w2 = 0; w2 < kThrF / 32; ++w2) {
            const float4 t4 = *reinterpret_cast<const float4*>(&gtot[w2 * kHeadDim + kq]);
            if (w2 == warp) { pre[0] = tot[0]; pre[1] = tot[1]; pre[2] = tot[2]; pre[3] = tot[3]; }
            tot[0] += t4.x; tot[1] += t4.y; tot[2] += t4.z; tot[3] += t4.w;
        }
#pragma unroll
        for (int i = 0; i < kTokW; ++i)
#pragma unroll
            for (int e = 0; e < 4; ++e) G[i][e] = pre[e] + G[i][e];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            cref_l[e] = 0.5f * tot[e];
            ecr_l[e] = __expf(0.5f * tot[e]);
        }
        if (warp == kThrF / 32 - 1) {            // published for the column images and the block
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                sm.gcs[kq + e] = tot[e];
                reinterpret_cast<float*>(blk + kOffEG)[kq + e] = decay_f(tot[e]);
                if (tot[e] < -170.0f && a.err) atomicOr(a.err, kDevErrRange);
            }
        }
#pragma unroll
        for (int i = 0; i < kTokW; ++i)
            *reinterpret_cast<float4*>(&sm.scr[(t0 + i) * 128 + kq]) =
                make_float4(G[i][0], G[i][1], G[i][2], G[i][3]);
        __syncwarp();                            // the row images read this warp's own G rows
    } else {
        __syncthreads();                         // sm.gs
        float run = 0.0f;                        // the running sum in token order
        for (int t = 0; t < t0; ++t) run += sm.gs[t];
#pragma unroll
        for (int i = 0; i < kTokW; ++i) {
            run += sm.gs[t0 + i];
#pragma unroll
            for (int e = 0; e < 4; ++e) G[i][e] = run;
        }
        for (int t = t0 + kTokW; t < kCc; ++t) run += sm.gs[t];
        GCh = run;
        if (tid < kCc) {
            float Gt = 0.0f;
            for (int t = 0; t <= tid; ++t) Gt += sm.gs[t];    // same summation order as G
            sm.gsc[tid] = Gt;
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) reinterpret_cast<float*>(blk + kOffEG)[kq + e] = decay_f(GCh);
        __syncthreads();                         // gsc
    }

    // ---- row images: tokens t0 + 2*(lane&1) + (j ^ sw), channels k0 .. k0+7 --------------------
    {
        const bool sw = ((lane >> 1) & 1) != 0;
        const int k0 = 8 * (lane >> 1);
        const int tb = t0 + 2 * (lane & 1);
        const int tj[2] = {tb + (sw ? 1 : 0), tb + (sw ? 0 : 1)};
        float crv[8], ecv[8];
        if (GATE_MODE == 0) {
            // channels k0 .. k0+7 = this lane pair's: the even lane's 4 then the odd lane's 4
            const bool odd = (lane & 1) != 0;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float oc = __shfl_xor_sync(0xffffffffu, cref_l[e], 1);
                const float oe = __shfl_xor_sync(0xffffffffu, ecr_l[e], 1);
                crv[e] = odd ? oc : cref_l[e];
                crv[4 + e] = odd ? cref_l[e] : oc;
                ecv[e] = odd ? oe : ecr_l[e];
                ecv[4 + e] = odd ? ecr_l[e] : oe;
            }
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {            // one token row at a time
            const int t = tj[j];
            float kr[8], qr[8];
            pair_row(k, kr, sw, j);
            pair_row(q, qr, sw, j);
            float xb[8], xk[8], xq[8], xg[8];
            if (GATE_MODE == 0) {
                const float4 a0 = *reinterpret_cast<const float4*>(&sm.scr[t * 128 + k0]);
                const float4 a1 = *reinterpret_cast<const float4*>(&sm.scr[t * 128 + k0 + 4]);
                const float gtv[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float gt = gtv[e], cr = crv[e];
                    const float ef = __expf(gt - cr), eb = __expf(cr - gt);
                    xb[e] = kr[e] * eb;
                    xk[e] = kr[e] * ef;
                    xq[e] = qr[e] * ef;
                    xg[e] = qr[e] * (ef * ecv[e]);
                }
            } else {
                const float eg = __expf(sm.gsc[t]);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    xb[e] = kr[e];
                    xk[e] = kr[e];
                    xq[e] = qr[e];
                    xg[e] = qr[e] * eg;
                }
            }
            put8x(sm.kb[0], sm.kb[1], tc_offset(t, k0, kSbo128), xb);
            put8x(sm.bia[0], sm.bia[1], tc_offset(t, k0, kSbo128), xk);
            put8x(sm.bia[0], sm.bia[1], tc_offset(kCc + t, k0, kSbo128), xq);
            put8h(blk + kOffQW, tc_offset(t, k0, kSbo128), xg);
        }
    }
    // ---- MMA-a on the row images ---------------------------------------------------------------
    if (tid == 0) bulk_wait_read0();             // the last epilogue's copies have read sm.ktv
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) intra_mma_a_issue(sm);

    // ---- column images (while MMA-a runs): channel kq+e, tokens t0 .. t0+3 ----------------------
    // K e^{G} beta and V beta into sm.ktv (MMA-b's B operand); K e^{G_C-G} staged in sm.scr (the G
    // tile is dead once the row images are written) and copied to the workspace in bulk.
    unsigned char* b2s = reinterpret_cast<unsigned char*>(sm.scr);
    constexpr uint32_t kB2KBytes = kHeadDim * kCc * 2;
    {
        float bv[kTokW];
#pragma unroll
        for (int i = 0; i < kTokW; ++i) bv[i] = sm.beta[t0 + i];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            float xt[kTokW], xv[kTokW], xc[kTokW];
            const float GCe = GATE_MODE == 0 ? sm.gcs[kq + e] : GCh;
#pragma unroll
            for (int i = 0; i < kTokW; ++i) {
                const float Gi = G[i][e];
                xt[i] = bv[i] * k[i][e] * __expf(Gi);
                xv[i] = bv[i] * v[i][e];
                xc[i] = k[i][e] * __expf(GCe - Gi);
            }
            put4x(sm.ktv[0], sm.ktv[1], tc_offset(kq + e, t0, kSboKt), xt);
            put4x(sm.ktv[0], sm.ktv[1], tc_offset(128 + kq + e, t0, kSboKt), xv);
            *reinterpret_cast<uint2*>(b2s + tc_offset(kq + e, t0, kSbo32)) =
                make_uint2(f16x2_rn(xc[0], xc[1]), f16x2_rn(xc[2], xc[3]));
        }
    }
    // the first 128 rows of the B2 image (K e^{G_C-G}, f16) leave in one bulk copy
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
        bulk_store(blk + kOffB2, b2s, kB2KBytes);
        bulk_commit();
    }

    const long next = task + gridDim.x;
    const bool ok = intra_mma_tail<GATE_MODE, kThrF, true>(sm, a.err, blk, phase, [&]() {
        if (PF && next < ntasks) {
            const TaskPos np = task_pos(a.seq, chunk_off, next, nchunks, vs, Hk);
            ld_pending = true;
            // issued from warp 7, idle here, not from thread 0, whose warp extracts A next (a
            // clock-stamped probe saw thread 0 spend ~2,900 cycles in this hook)
            if (tid == kThrF - 32) stage_raw<KW>(stage, maps, np, &smf.bar_raw);
            stage_params<GATE_MODE, PW, KW>(ps, p, H, Hg, np);
        }
    }, [&]() {
        if (PF && GATE_MODE == 0 && next < ntasks && tid == kThrF - 32)
            stage_f(sm.scr, maps, task_pos(a.seq, chunk_off, next, nchunks, vs, Hk), &smf.bar_f);
    }, &maps.ut, (int)(gid * H + h));
    if (!ok) break;
    }   // task loop
    if (PF && ld_pending) {                      // left early: let the next task's loads land
        mbar_wait_bounded(&smf.bar_raw, ph_ld, a.err);
        if (GATE_MODE == 0) mbar_wait_bounded(&smf.bar_f, ph_ld, a.err);
    }
    if (PF) cp_async_wait_all();                 // no copy may land after the CTA has left
    if (tid == 0) bulk_wait_all();               // nor leave unfinished
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(sm.tmem_base, 256);
}

template <bool BF16, int GM, bool CONV, int KW>
static cudaError_t launch_prep_intra_t(const PrepArgs& p, const ScanArgs& a, const int* chunk_off,
                                       unsigned char* blocks, long nchunks, cudaStream_t s) {
    const size_t smem = kPrepIntraSmemBytes;
    static PerDevice<int> done;
    cudaError_t e = set_smem(kda_chunk_prep_intra_kernel<BF16, GM, CONV, KW>, smem, done);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const long ntasks = nchunks * a.H;
    if (ntasks >= (1L << 31)) return cudaErrorInvalidValue;   // tasks split with 32-bit division
    const long ctas = min(ntasks, 2L * sms);     // two resident CTAs per SM, persistent
    RawMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    if (!make_tensor_map_blocks_ut(&maps.ut, blocks + kOffUT, ntasks, kBlkBytes))
        return cudaErrorInvalidValue;
    if (BF16) {                                  // the staged form reads through tensor maps
        const long rows = a.seq.total_rows, C = (long)a.H * kHeadDim;
        const long Cq = plane_width(a.H, p.Hk, 0);
        constexpr int kRows = RawStage<KW>::kRows;
        if (!make_tensor_map_2d_any(&maps.q, p.q_raw, true, rows, Cq, kHeadDim, kRows) ||
            !make_tensor_map_2d_any(&maps.k, p.k_raw, true, rows, Cq, kHeadDim, kRows) ||
            !make_tensor_map_2d_any(&maps.v, p.v_raw, true, rows, C, kHeadDim, kRows) ||
            (GM == 0 && !make_tensor_map_2d_any(&maps.f, p.f_raw, false, rows,
                                                (long)prep_gate_heads(p) * kHeadDim, kHeadDim, kCc)))
            return cudaErrorInvalidValue;
    }
    KernelTimer kt(kKPrepIntra, s);
    kda_chunk_prep_intra_kernel<BF16, GM, CONV, KW><<<(unsigned)ctas, kThrF, smem, s>>>(
        p, a, chunk_off, blocks, nchunks, maps);
    return cudaGetLastError();
}

template <bool BF16, int GM>
static cudaError_t launch_prep_intra_c(const PrepArgs& p, const ScanArgs& a, const int* chunk_off,
                                       unsigned char* blocks, long nchunks, cudaStream_t s) {
    if (p.conv_w == nullptr)
        return launch_prep_intra_t<BF16, GM, false, 4>(p, a, chunk_off, blocks, nchunks, s);
    if (p.K <= 4) return launch_prep_intra_t<BF16, GM, true, 4>(p, a, chunk_off, blocks, nchunks, s);
    return launch_prep_intra_t<BF16, GM, true, kMaxConvK>(p, a, chunk_off, blocks, nchunks, s);
}

cudaError_t launch_prefill_chunk(const PrepArgs& p, const ScanArgs& a, const int* cu_host,
                                 void* workspace, cudaStream_t s) {
    if (a.seq.N == 0) return cudaSuccess;
    cudaError_t e;
    if (a.seq.total_rows == 0) {
        const size_t bytes = (size_t)a.seq.N * a.H * kHeadDim * kHeadDim * sizeof(float);
        e = cudaMemcpyAsync(a.state_out, a.state_in, bytes, cudaMemcpyDeviceToDevice, s);
        if (e != cudaSuccess) return e;
        return launch_ring_roll(p, s);
    }
    int* chunk_off = nullptr;
    unsigned char* blocks = nullptr;
    e = launch_chunk_offsets(a.seq, workspace, &chunk_off, &blocks, s);
    if (e != cudaSuccess) return e;
    const long nchunks = chunk_count(a.seq, cu_host);
    if (nchunks > 0) {
        const bool gm1 = (a.gate_mode & 1) != 0;
        if (p.raw_bf16) e = gm1 ? launch_prep_intra_c<true, 1>(p, a, chunk_off, blocks, nchunks, s)
                                : launch_prep_intra_c<true, 0>(p, a, chunk_off, blocks, nchunks, s);
        else e = gm1 ? launch_prep_intra_c<false, 1>(p, a, chunk_off, blocks, nchunks, s)
                     : launch_prep_intra_c<false, 0>(p, a, chunk_off, blocks, nchunks, s);
        if (e != cudaSuccess) return e;
    }
    // the inter kernel also rolls the conv ring (after the kernel above has read ring_in)
    return launch_chunk_inter(a, chunk_off, blocks, s, p.conv_w != nullptr ? &p : nullptr);
}

}  // namespace kda
