// kda_epilogue.cu -- sigmoid-gated RMSNorm over head_dim.
//
// Method ("memra_engine/kda.rs", memra-engine 0.125.0, kda_core_gated stage 6 and
// Engine::kda_gated_rmsnorm): per (token, head) row of 128 values,
//     y_i = o_i / sqrt(mean_i o_i^2 + eps) * w_i * sigmoid(z_i)
// with w shared by all heads and the gate z not normalised (gdn_ops.rs gdn_gated_rmsnorm_into).
//
// One warp per row, one float4 per lane: a 512-byte coalesced load of o and z and store of y, a
// 5-step butterfly for the mean square.  Rows wider than 128 (a value head wider than the key
// head) take m float4s per lane.  The arithmetic is the fused decode kernel's epilogue,
// instruction for instruction.
#include "kda_device.cuh"
#include "kda_internal.h"

namespace kda {

template <bool SILU>
__global__ void __launch_bounds__(256) kda_gated_rmsnorm_kernel(NormArgs a) {
    const long row = (long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= a.rows) return;
    const long base = row * kHeadDim + 4 * lane;
    const float4 o4 = __ldcs(reinterpret_cast<const float4*>(a.o + base));
    float ss = __fmul_rn(o4.x, o4.x);
    ss = ss + __fmul_rn(o4.y, o4.y);
    ss = ss + __fmul_rn(o4.z, o4.z);
    ss = ss + __fmul_rn(o4.w, o4.w);
    const float inv = rms_inv_f(warp_sum(ss), a.eps);
    const float4 w4 = *reinterpret_cast<const float4*>(a.w + 4 * lane);
    const float4 z4 = __ldcs(reinterpret_cast<const float4*>(a.z + base));
    float4 y4;
    y4.x = gated_norm_f<SILU>(o4.x, inv, w4.x, z4.x);
    y4.y = gated_norm_f<SILU>(o4.y, inv, w4.y, z4.y);
    y4.z = gated_norm_f<SILU>(o4.z, inv, w4.z, z4.z);
    y4.w = gated_norm_f<SILU>(o4.w, inv, w4.w, z4.w);
    __stcs(reinterpret_cast<float4*>(a.y + base), y4);
}

// Rows of m * 128 values (a value head wider than the key head): one warp per row, lane l on the
// float4s at 4l + 128 j (j < m).  The sum of squares of each 128-block is the square kernel's
// (four products, then the butterfly); the blocks' sums are added in block order from 0, the
// order in which the fused decode's thread-block cluster adds its CTAs' sums; the mean is over the
// whole row.
template <bool SILU>
__global__ void __launch_bounds__(256) kda_gated_rmsnorm_wide_kernel(NormArgs a, int m) {
    const long row = (long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= a.rows) return;
    const long base = row * (long)a.width + 4 * lane;
    float tot = 0.0f;
    for (int j = 0; j < m; ++j) {
        const float4 o4 = __ldcs(reinterpret_cast<const float4*>(a.o + base + kHeadDim * j));
        float ss = __fmul_rn(o4.x, o4.x);
        ss = ss + __fmul_rn(o4.y, o4.y);
        ss = ss + __fmul_rn(o4.z, o4.z);
        ss = ss + __fmul_rn(o4.w, o4.w);
        tot = tot + warp_sum(ss);
    }
    const float inv = rms_inv_w(tot, a.eps, a.width);
    for (int j = 0; j < m; ++j) {
        const long off = base + kHeadDim * j;
        const float4 o4 = __ldcs(reinterpret_cast<const float4*>(a.o + off));
        const float4 w4 = *reinterpret_cast<const float4*>(a.w + 4 * lane + kHeadDim * j);
        const float4 z4 = __ldcs(reinterpret_cast<const float4*>(a.z + off));
        float4 y4;
        y4.x = gated_norm_f<SILU>(o4.x, inv, w4.x, z4.x);
        y4.y = gated_norm_f<SILU>(o4.y, inv, w4.y, z4.y);
        y4.z = gated_norm_f<SILU>(o4.z, inv, w4.z, z4.z);
        y4.w = gated_norm_f<SILU>(o4.w, inv, w4.w, z4.w);
        __stcs(reinterpret_cast<float4*>(a.y + off), y4);
    }
}

cudaError_t launch_gated_rmsnorm(const NormArgs& a, cudaStream_t s) {
    if (a.rows == 0) return cudaSuccess;
    const long blocks = (a.rows + 7) / 8;
    const int m = a.width > kHeadDim ? a.width / kHeadDim : 1;
    KernelTimer kt(kKRmsNorm, s);
    if (m > 1) {
        if (a.silu) kda_gated_rmsnorm_wide_kernel<true><<<(unsigned)blocks, 256, 0, s>>>(a, m);
        else kda_gated_rmsnorm_wide_kernel<false><<<(unsigned)blocks, 256, 0, s>>>(a, m);
    } else if (a.silu) {
        kda_gated_rmsnorm_kernel<true><<<(unsigned)blocks, 256, 0, s>>>(a);
    } else {
        kda_gated_rmsnorm_kernel<false><<<(unsigned)blocks, 256, 0, s>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace kda
