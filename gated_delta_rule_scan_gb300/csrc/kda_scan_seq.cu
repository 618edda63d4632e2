// kda_scan_seq.cu -- the per-channel gated delta-rule scan, sequential form.
//
// Method ("memra_engine/kda.rs", memra-engine 0.125.0: module doc and kda_core_gated stage 5,
// Engine::kda_scan "the per-channel-decay delta-rule scan"), per (sequence, head), per token t:
//     S <- Diag(exp g_t) S        (decay along the key dim i)
//     u  = v_t - S^T k_t
//     S <- S + beta_t k_t u^T
//     o_t = scale * S^T q_t       (readout from the updated state)
// The state buffers hold M[j][i] = S[i][j] (value column j, key dim i contiguous).
//
// GB300 layout.  Every value column j of S is an independent 128-vector recurrence, so the kernel
// parallelises over (sequence, head, column) and keeps each column in registers for the whole
// sequence.  A CTA (4 warps) owns 32 columns of one head; within a warp, 16 lanes share 4 columns
// and each lane holds 8 key-dim elements of all 4 (kda_scan_core.cuh), so each k / decay / q
// value a lane loads from shared memory feeds 4 columns, and a 4096-token, 64-head prefill runs
// about two warps per scheduler.  The per-token inputs every column of
// the head shares (q, k, g rows: 512 B each) and the CTA's 32 v values are staged by 2-D TMA
// tensor-map loads into a double-buffered shared-memory ring of kScanTB-token blocks, completion
// tracked by mbarriers (bounded waits); the next block streams in while the current one is
// scanned.  beta (and the GDN scalar gate) are register-prefetched one block ahead.  Outputs are
// buffered per block in shared memory and written back as coalesced 128-byte rows.
//
// The in-kernel token loop is the chained one-token program: a T-token launch and T one-token
// launches run the same instruction sequence per token, so their results are bit-identical.
#include "kda_scan_core.cuh"

namespace kda {

constexpr int kScanG = 16;                      // lanes per column group (kda_scan_core.cuh)
constexpr int kScanWarps = 4;
constexpr int kScanThreads = 32 * kScanWarps;
constexpr int kScanCols = (32 / kScanG) * 4 * kScanWarps;   // value columns per CTA
constexpr int kScanTB = 16;                     // tokens per staged block
constexpr int kColBlocks = kHeadDim / kScanCols;

struct __align__(128) ScanSmem {
    float q[2][kScanTB][kHeadDim];
    float k[2][kScanTB][kHeadDim];
    float g[2][kScanTB][kHeadDim];      // per-channel gate (log-decay, or decay factor)
    float v[2][kScanTB][kScanCols];
    float a[kScanTB][kHeadDim];         // exp(g) of the block being scanned (log-decay input)
    float obuf[kScanTB][kScanCols];
    float beta[2][kScanTB];
    float ascal[2][kScanTB];            // per-head decay factor (gate mode 1)
    uint64_t bar[2];
};

// GATE_MODE: 0 per-channel g [rows, C], 1 per-head g [rows, H].  EXP_DONE: g already holds the
// decay factor exp(log-decay), so no exp is taken here.
template <int GATE_MODE, bool EXP_DONE>
__global__ void __launch_bounds__(kScanThreads)
kda_scan_seq_kernel(ScanArgs a, const __grid_constant__ CUtensorMap tq,
                    const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tg,
                    const __grid_constant__ CUtensorMap tv) {
    extern __shared__ unsigned char smem_raw[];
    ScanSmem& sm = *reinterpret_cast<ScanSmem*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31, grp = lane / kScanG, r = lane % kScanG;
    const int cb = blockIdx.x % kColBlocks;
    const int h = blockIdx.x / kColBlocks;
    const int n = a.order ? a.order[blockIdx.y] : (int)blockIdx.y;
    const int cw = (warp * (32 / kScanG) + grp) * 4;   // first of the group's 4 columns in the CTA
    const int H = a.H;
    const long C = (long)H * kHeadDim;
    const int gh = gate_head(a, h);             // the value head: its gate and beta
    const int Hg = gate_heads(a);
    const int kh = unit_qk_head(a, h);          // the q / k head this value head reads

    long begin, end;
    if (a.seq.cu_seqlens == nullptr) {
        begin = (long)n * a.seq.T_uniform;
        end = begin + a.seq.T_uniform;
    } else {
        begin = a.seq.cu_seqlens[n];
        end = a.seq.cu_seqlens[n + 1];
    }
    const long L = end - begin;
    const int nblk = (int)((L + kScanTB - 1) / kScanTB);

    ColG<kScanG> S;
    const long col0 = (((long)n * H + h) * kHeadDim + cb * kScanCols + cw) * kHeadDim;
    colg_load<kScanG>(S, a.state_in + col0, r);

    constexpr uint32_t kTxBytes =
        (GATE_MODE == 0 ? 3u : 2u) * kScanTB * kHeadDim * 4u + kScanTB * kScanCols * 4u;
    if (tid == 0) {
        prefetch_tensormap(&tq);
        prefetch_tensormap(&tk);
        if (GATE_MODE == 0) prefetch_tensormap(&tg);
        prefetch_tensormap(&tv);
        mbar_init(&sm.bar[0], 1);
        mbar_init(&sm.bar[1], 1);
        fence_mbar_init();
    }
    __syncthreads();

    auto issue = [&](int b, int st) {
        const int row = (int)(begin + (long)b * kScanTB);
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&sm.bar[st], kTxBytes);
        tma_load_2d(&sm.q[st][0][0], &tq, kh * kHeadDim, row, &sm.bar[st]);
        tma_load_2d(&sm.k[st][0][0], &tk, kh * kHeadDim, row, &sm.bar[st]);
        if (GATE_MODE == 0) tma_load_2d(&sm.g[st][0][0], &tg, gh * kHeadDim, row, &sm.bar[st]);
        tma_load_2d(&sm.v[st][0][0], &tv, h * kHeadDim + cb * kScanCols, row, &sm.bar[st]);
    };
    if (tid == 0 && nblk > 0) issue(0, 0);

    float bpre = 0.0f, gpre = 0.0f;
    if (tid < kScanTB && tid < L) {
        bpre = a.beta[(begin + tid) * Hg + gh];
        if (GATE_MODE == 1) gpre = a.g[(begin + tid) * Hg + gh];
    }

    for (int b = 0; b < nblk; ++b) {
        const int st = b & 1;
        const long row0 = begin + (long)b * kScanTB;
        const int nt = (int)min((long)kScanTB, L - (long)b * kScanTB);
        if (tid < kScanTB) {
            sm.beta[st][tid] = bpre;
            if (GATE_MODE == 1) sm.ascal[st][tid] = EXP_DONE ? gpre : decay_f(gpre);
            const long rn = row0 + kScanTB + tid;
            if (rn < end) {
                bpre = a.beta[rn * Hg + gh];
                if (GATE_MODE == 1) gpre = a.g[rn * Hg + gh];
            }
        }
        const bool arrived = mbar_wait_bounded(&sm.bar[st], (uint32_t)((b >> 1) & 1), a.err);
        if (__syncthreads_or(!arrived)) return;  // device error word already raised
        if (tid == 0 && b + 1 < nblk) issue(b + 1, st ^ 1);
        if (GATE_MODE == 0 && !EXP_DONE) {
            for (int e = tid; e < nt * kHeadDim; e += kScanThreads)
                (&sm.a[0][0])[e] = decay_f((&sm.g[st][0][0])[e]);
        }
        __syncthreads();

        TokView vw;
        vw.k = &sm.k[st][0][0];
        vw.a = EXP_DONE ? &sm.g[st][0][0] : &sm.a[0][0];
        vw.q = &sm.q[st][0][0];
        vw.a_scal = &sm.ascal[st][0];
        vw.v = &sm.v[st][0][0];
        vw.beta = &sm.beta[st][0];
        vw.out = &sm.obuf[0][0];
        vw.row_stride = kHeadDim;
        vw.v_stride = kScanCols;
        vw.v_col0 = cw;
        vw.out_stride = kScanCols;
        vw.out_col0 = cw;
        colg_tokens<GATE_MODE == 0, true, kScanG>(S, nt, vw, a.scale, r, lane);
        __syncthreads();
        for (int e = tid; e < nt * (kScanCols / 4); e += kScanThreads) {
            const int t = e / (kScanCols / 4), c4 = e % (kScanCols / 4);
            *reinterpret_cast<float4*>(a.o + (row0 + t) * C + h * kHeadDim + cb * kScanCols + 4 * c4) =
                *reinterpret_cast<const float4*>(&sm.obuf[t][4 * c4]);
        }
    }
    colg_store<kScanG>(S, a.state_out + col0, r);
}

// ------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn lookup_encode_fn() {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        return reinterpret_cast<EncodeTiledFn>(p);
    return nullptr;
}

// the driver's tensor-map encoder, looked up once (a function-local static: thread-safe)
static EncodeTiledFn encode_fn() {
    static const EncodeTiledFn fn = lookup_encode_fn();
    return fn;
}

bool make_tensor_map_2d_any(CUtensorMap* m, const void* base, bool bf16, long rows, long cols,
                            int box_cols, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const size_t es_bytes = bf16 ? 2 : 4;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * es_bytes};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
              const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tensor_map_blocks_ut(CUtensorMap* m, void* base, long nblocks, size_t block_bytes) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {128, 32, (cuuint64_t)nblocks};
    cuuint64_t strides[2] = {128 * sizeof(float), (cuuint64_t)block_bytes};
    cuuint32_t box[3] = {32, 32, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tensor_map_2d_bf16_sw128(CUtensorMap* m, const void* base, long rows, long cols,
                                   int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};      // 64 bf16 = one 128-byte swizzle row
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
              es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tensor_map_2d(CUtensorMap* m, const float* base, long rows, long cols, int box_cols,
                        int box_rows) {
    return make_tensor_map_2d_any(m, base, false, rows, cols, box_cols, box_rows);
}

template <int GM, bool EXP>
static cudaError_t launch_t(const ScanArgs& a, cudaStream_t s) {
    const long C = (long)a.H * kHeadDim;
    const long Ck = (long)qk_heads(a) * kHeadDim;
    const long rows = a.seq.total_rows;
    CUtensorMap tq, tk, tg, tv;
    if (!make_tensor_map_2d(&tq, a.q, rows, Ck, kHeadDim, kScanTB) ||
        !make_tensor_map_2d(&tk, a.k, rows, Ck, kHeadDim, kScanTB) ||
        !make_tensor_map_2d(&tv, a.v, rows, C, kScanCols, kScanTB))
        return cudaErrorInvalidValue;
    if (GM == 0) {
        const long Cg = (long)gate_heads(a) * kHeadDim;   // gate rows: the value heads
        if (!make_tensor_map_2d(&tg, a.g, rows, Cg, kHeadDim, kScanTB)) return cudaErrorInvalidValue;
    } else {
        tg = tq;  // unused
    }
    const size_t smem = sizeof(ScanSmem) + 128;
    static PerDevice<int> attr_done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const bool cached = dev >= 0 && dev < kMaxDevices;
    if (!cached || !attr_done[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(kda_scan_seq_kernel<GM, EXP>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        if (cached) attr_done[dev].store(1, std::memory_order_release);
    }
    dim3 grid((unsigned)(a.H * kColBlocks), (unsigned)a.seq.N);
    KernelTimer kt(kKScanSeq, s);
    kda_scan_seq_kernel<GM, EXP><<<grid, kScanThreads, smem, s>>>(a, tq, tk, tg, tv);
    return cudaGetLastError();
}

cudaError_t launch_scan_seq(const ScanArgs& a, cudaStream_t s) {
    if (a.seq.N == 0) return cudaSuccess;
    if (a.seq.total_rows == 0) {
        // no tokens at all: the state passes through unchanged
        const size_t bytes = (size_t)a.seq.N * a.H * kHeadDim * kHeadDim * sizeof(float);
        return cudaMemcpyAsync(a.state_out, a.state_in, bytes, cudaMemcpyDeviceToDevice, s);
    }
    const bool exp_done = (a.gate_mode & 2) != 0;
    if ((a.gate_mode & 1) == 0) return exp_done ? launch_t<0, true>(a, s) : launch_t<0, false>(a, s);
    return exp_done ? launch_t<1, true>(a, s) : launch_t<1, false>(a, s);
}

}  // namespace kda
