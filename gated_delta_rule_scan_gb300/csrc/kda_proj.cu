// kda_proj.cu -- stage 1 of the KDA mixer: the six projections that read the layer input x (the
// docs.rs page "memra_engine/kda.rs", memra-engine 0.125.0: `kda_core_gated` stage 1, the
// `KdaAttnLayer` field docs for the shapes, `Engine::kda_proj_fused6` for the one-launch form).
//
//     out_i[s][r] = sum_k W_i[r][k] * x[s][k]      i = q, k, v, forget-down, gate-down, beta
//
// with W_q, W_k, W_v [H*D, in_f], W_fa, W_ga [D, in_f], W_b [H, in_f] in bf16 and x [t, in_f] f32.
//
// GB300 design.  For a decode or verify batch t is small (1..256) and the weights (hundreds of MB)
// are read once, so the launch is bound by HBM; the products still run on the tcgen05 tensor
// cores so that the FP32 pipe never becomes the limit as t grows.  The weights are the MMA's A
// operand as they are (K-major bf16, TMA-loaded in the 128-byte swizzle); x is split once into
// bf16 hi + lo images (x = hi + lo to about 16 significant bits) by a small pre-pass, and every
// K-step takes two MMAs, W * hi + W * lo, accumulating in f32 in TMEM.  The weights' bf16 values
// are exact in the product, so the result carries only the f32 accumulation and the split's
// ~2^-17 relative residue.
//
// Two CTAs per 128-row tile of one weight, each on half of K (the six weights' tiles in one grid),
// launched as a programmatic dependent of the split pre-pass so that its set-up and first weight
// loads overlap the split: warp 0's lane 0 streams K-stages of 64 (16 KB of weights plus the x
// images) through a ring of mbarrier-guarded shared-memory slots, warp 1's lane 0 issues the MMAs
// and frees each slot with a commit, and all four warps read the accumulator back (TMEM lane =
// weight row, column = token) and add it into the outputs (zeroed by the pre-pass), each warp
// covering 32 consecutive floats per token.  Exactly two partial sums meet in each output and
// float addition is commutative, so the result is deterministic.  A CTA's ring stays near 66 KB
// for t <= 64, so three CTAs share an SM and the grid (390 CTAs at 64 heads) is resident at once.
// Every wait is bounded; a wait that gives up raises the device error word.
#include <cuda_bf16.h>

#include "kda_device.cuh"
#include "kda_internal.h"
#include "kda_tc.cuh"

namespace kda {

namespace {

constexpr int kPRows = 128;                    // weight rows per tile = MMA M = TMEM lanes
constexpr int kPK = 64;                        // K per stage: one 128-byte swizzle row of bf16
constexpr int kPThreads = 128;
constexpr int kPStageW = kPRows * kPK * 2;     // 16 KB of weights per stage
constexpr int kPSmemTarget = 66 * 1024;        // stage ring budget: three CTAs per SM up to t = 64
constexpr int kPKSplit = 2;                    // CTAs per weight tile, each on half of K

struct Proj6Maps {
    CUtensorMap w[6];
    CUtensorMap xh, xl;
};

struct Proj6Params {
    float* out[6];
    int rows[6];
    int tile_start[7];      // first tile of each weight; tile_start[6] = the tiles
    int t, t_pad, in_f;
    int stages;
    uint32_t tmem_cols;
    int* err;
};

// x [t, in_f] f32 -> hi, lo [t_pad, in_f] bf16 with hi + lo ~= x; rows t .. t_pad-1 are zero.
// Also zeroes the six outputs, which the projection kernel's two K halves then add into.
__global__ void __launch_bounds__(256) kda_proj_split_kernel(const float* __restrict__ x,
                                                             __nv_bfloat16* __restrict__ hi,
                                                             __nv_bfloat16* __restrict__ lo,
                                                             const __grid_constant__ Proj6Params p) {
    // the projection kernel may start now: it loads weights until it needs these images
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const long n4 = (long)p.t_pad * p.in_f / 4;
    const long live4 = (long)p.t * p.in_f / 4;
    const long stride = (long)gridDim.x * blockDim.x;
    const long i0 = blockIdx.x * (long)blockDim.x + threadIdx.x;
    for (long i = i0; i < n4; i += stride) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i < live4) v = __ldg(reinterpret_cast<const float4*>(x) + i);
        uint2 h, l;
        split_bf16x2(v.x, v.y, h.x, l.x);
        split_bf16x2(v.z, v.w, h.y, l.y);
        reinterpret_cast<uint2*>(hi)[i] = h;
        reinterpret_cast<uint2*>(lo)[i] = l;
    }
#pragma unroll 1
    for (int w = 0; w < 6; ++w) {
        const long n = (long)p.t * p.rows[w];
        for (long i = i0; i < n; i += stride) p.out[w][i] = 0.0f;
    }
}

__global__ void __launch_bounds__(kPThreads, 1)
kda_proj6_kernel(const __grid_constant__ Proj6Maps maps, const __grid_constant__ Proj6Params p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* base = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int stage_x = p.t_pad * kPK * 2;                  // one x image per stage
    const int stage_bytes = kPStageW + 2 * stage_x;
    uint64_t* full = reinterpret_cast<uint64_t*>(base + p.stages * stage_bytes);
    uint64_t* empty = full + p.stages;
    uint64_t* done = empty + p.stages;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);

    // CTA pair (2 tile, 2 tile + 1): the tile's two K halves
    const int tile = (int)blockIdx.x / kPKSplit, half = (int)blockIdx.x % kPKSplit;
    int wi = 0;
    while (wi < 5 && tile >= p.tile_start[wi + 1]) ++wi;
    const int row0 = (tile - p.tile_start[wi]) * kPRows;
    const int nk = p.in_f / kPK / kPKSplit;       // K-stages of this CTA
    const int kb0 = half * nk;                     // its first K-stage of the weight rows

    if (warp == 0) {
        tmem_alloc(tmem_slot, p.tmem_cols);
        tmem_relinquish();
    }
    if (tid == 32) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(done, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;

    if (tid == 0) {
        // producer: K-stage kb into slot kb % stages once the MMAs of kb - stages have read it.
        // The first ring of weight tiles goes out before the x images exist: the split kernel
        // launched just before this one may still be running (programmatic dependent launch);
        // griddepcontrol.wait returns once it has finished and its writes are visible.
        prefetch_tensormap(&maps.w[wi]);
        prefetch_tensormap(&maps.xh);
        prefetch_tensormap(&maps.xl);
        const int first = nk < p.stages ? nk : p.stages;
        for (int kb = 0; kb < first; ++kb) {
            mbar_arrive_expect_tx(&full[kb], (uint32_t)stage_bytes);
            tma_load_2d(base + kb * stage_bytes, &maps.w[wi], (kb0 + kb) * kPK, row0, &full[kb]);
        }
        asm volatile("griddepcontrol.wait;" ::: "memory");
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % p.stages;
            unsigned char* st = base + s * stage_bytes;
            const int kx = (kb0 + kb) * kPK;
            if (kb >= first) {
                if (!mbar_wait_bounded(&empty[s], (uint32_t)(((kb / p.stages) & 1) ^ 1), p.err))
                    break;
                mbar_arrive_expect_tx(&full[s], (uint32_t)stage_bytes);
                tma_load_2d(st, &maps.w[wi], kx, row0, &full[s]);
            }
            tma_load_2d(st + kPStageW, &maps.xh, kx, 0, &full[s]);
            tma_load_2d(st + kPStageW + stage_x, &maps.xl, kx, 0, &full[s]);
        }
    } else if (tid == 32) {
        // MMA issuer: D[row][token] += W[row][k] * (hi + lo)[token][k], four K-steps per stage
        const uint32_t idesc = tc_idesc_bf16(kPRows, p.t_pad);
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % p.stages;
            if (!mbar_wait_bounded(&full[s], (uint32_t)((kb / p.stages) & 1), p.err)) break;
            tc_fence_after();
            const uint32_t st = smem_u32(base + s * stage_bytes);
#pragma unroll
            for (int ks = 0; ks < kPK / 16; ++ks) {
                const uint64_t a = tc_smem_desc_sw128(st + 32 * ks);
                const uint64_t bh = tc_smem_desc_sw128(st + kPStageW + 32 * ks);
                const uint64_t bl = tc_smem_desc_sw128(st + kPStageW + stage_x + 32 * ks);
                tc_mma_ss(tbase, a, bh, idesc, kb > 0 || ks > 0);
                tc_mma_ss(tbase, a, bl, idesc, true);
            }
            tc_commit(&empty[s]);
        }
        tc_commit(done);      // arrives once every MMA issued above has completed
    }
    __syncwarp();
    const bool ok = mbar_wait_bounded(done, 0, p.err);
    tc_fence_after();

    // epilogue: thread (warp w, lane l) owns weight row row0 + 32 w + l and adds its K half's
    // partial sums into the zeroed outputs.  Two partials meet in each output element, and
    // (0 + a) + b == (0 + b) + a exactly, so the result does not depend on which half lands first.
    const int rows = p.rows[wi];
    const int row = row0 + 32 * warp + lane;
    float* out = p.out[wi];
    const uint32_t tl = tbase + ((uint32_t)(32 * warp) << 16);
    for (int n0 = 0; n0 < p.t_pad; n0 += 16) {
        float v[16];
        tmem_ld16(tl + n0, v);
        tmem_ld_wait();
        if (ok && row < rows) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
                if (n0 + j < p.t) atomicAdd(out + (long)(n0 + j) * rows + row, v[j]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, p.tmem_cols);
}

}  // namespace

cudaError_t launch_proj6(const Proj6Args& a, cudaStream_t s) {
    const int t_pad = proj_t_pad(a.t);
    __nv_bfloat16* xh = static_cast<__nv_bfloat16*>(a.ws);
    __nv_bfloat16* xl = xh + (size_t)t_pad * a.in_f;
    Proj6Maps maps;
    Proj6Params p{};
    int tiles = 0;
    for (int i = 0; i < 6; ++i) {
        p.out[i] = a.out[i];
        p.rows[i] = a.rows[i];
        p.tile_start[i] = tiles;
        tiles += (a.rows[i] + kPRows - 1) / kPRows;
        if (!make_tensor_map_2d_bf16_sw128(&maps.w[i], a.w[i], a.rows[i], a.in_f, kPRows))
            return cudaErrorInvalidValue;
    }
    p.tile_start[6] = tiles;
    if (!make_tensor_map_2d_bf16_sw128(&maps.xh, xh, t_pad, a.in_f, t_pad) ||
        !make_tensor_map_2d_bf16_sw128(&maps.xl, xl, t_pad, a.in_f, t_pad))
        return cudaErrorInvalidValue;
    p.t = a.t;
    p.t_pad = t_pad;
    p.in_f = a.in_f;
    p.err = a.err;
    const int stage_bytes = kPStageW + 2 * t_pad * kPK * 2;
    int stages = kPSmemTarget / stage_bytes;
    stages = stages < 2 ? 2 : (stages > 6 ? 6 : stages);
    if (stages > a.in_f / kPK / kPKSplit) stages = a.in_f / kPK / kPKSplit < 2 ? 2 : a.in_f / kPK / kPKSplit;
    p.stages = stages;
    uint32_t cols = 32;
    while ((int)cols < t_pad) cols <<= 1;
    p.tmem_cols = cols;
    const size_t smem = 1024 + (size_t)stages * stage_bytes + (2 * stages + 1) * 8 + 16;

    {
        const long n4 = (long)t_pad * a.in_f / 4;
        const int blocks = (int)((n4 + 255) / 256 < 1024 ? (n4 + 255) / 256 : 1024);
        KernelTimer kt(kKProjSplit, s);
        kda_proj_split_kernel<<<blocks, 256, 0, s>>>(a.x, xh, xl, p);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    static PerDevice<int> smem_set_for;    // the largest dynamic shared memory opted into so far
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const bool cached = dev >= 0 && dev < kMaxDevices;
    if (!cached || smem_set_for[dev].load(std::memory_order_acquire) < (int)smem) {
        e = cudaFuncSetAttribute(kda_proj6_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        if (cached) {
            int cur = smem_set_for[dev].load(std::memory_order_acquire);
            while (cur < (int)smem &&
                   !smem_set_for[dev].compare_exchange_weak(cur, (int)smem,
                                                            std::memory_order_acq_rel)) {
            }
        }
    }
    // launched as a programmatic dependent of the split kernel: its CTAs may start (and stream
    // weights) while the split is still running
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(tiles * kPKSplit));
    cfg.blockDim = dim3(kPThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    KernelTimer kt(kKProj6, s);
    return cudaLaunchKernelEx(&cfg, kda_proj6_kernel, maps, p);
}

}  // namespace kda
