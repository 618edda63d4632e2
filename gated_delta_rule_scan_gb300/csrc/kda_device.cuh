// kda_device.cuh -- device-side helpers shared by every KDA kernel.
//
// The scalar maths here is written once and used by the prep kernel, the fused decode/verify
// kernel, the sequential scan and the epilogue, so that every path that must agree bit for bit
// (decode vs multi-token verify, chained T=1 scans vs one T-token scan) runs the same instruction
// sequence.  All products that feed a reduction use explicit fmaf/__fmul_rn so the compiler has
// no contraction freedom between call sites.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_internal.h"

namespace kda {

constexpr int kWaitSpinLimit = 1 << 22;  // bounded mbarrier wait: ~1 s with the back-off below

// device error word codes (written by kernels, read by kda_device_status)
constexpr int kDevErrTimeout = 1;

// ------------------------------------------------------------------------------------------
// scalar maths (f32).  The elementwise prologue / epilogue functions use the hardware
// exponential and reciprocal intrinsics (a few ulp; far inside the 1e-3 parity bound); the decay
// factor exp(g) that the recurrence multiplies by uses the full-precision expf.
// ------------------------------------------------------------------------------------------

__device__ __forceinline__ float sigmoid_f(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }

__device__ __forceinline__ float silu_f(float x) { return __fmul_rn(x, sigmoid_f(x)); }

// log(1 + e^x) without overflow: max(x, 0) + log1p(e^-|x|)
__device__ __forceinline__ float softplus_f(float x) {
    return fmaxf(x, 0.0f) + log1pf(__expf(-fabsf(x)));
}

// KDA per-channel forget gate as a raw log-decay: lb * sigmoid(rate * (f + dt_bias)),
// rate = exp(A_log[h]) computed once per head by the caller.  decay_f turns it into the factor
// the recurrence multiplies the state by.
__device__ __forceinline__ float kda_gate_f(float f, float dt_bias, float rate, float lb) {
    return __fmul_rn(lb, sigmoid_f(__fmul_rn(rate, f + dt_bias)));
}

// GDN per-head log-decay: -exp(A_log[h]) * softplus(alpha + dt_bias[h]).
__device__ __forceinline__ float gdn_gate_f(float alpha, float dt_bias, float a_log) {
    return -__fmul_rn(expf(a_log), softplus_f(alpha + dt_bias));
}

__device__ __forceinline__ float decay_f(float g) { return expf(g); }

// 1 / sqrt(sum of squares + eps): the l2-norm scale (eps inside the sqrt, on the SUM).
__device__ __forceinline__ float l2_inv_f(float ss, float eps) { return rsqrtf(ss + eps); }

// 1 / sqrt(mean of squares + eps) over 128 values: the RMSNorm scale.
__device__ __forceinline__ float rms_inv_f(float ss, float eps) {
    return rsqrtf(__fmul_rn(ss, 1.0f / kHeadDim) + eps);
}

// the same over a row of `width` values (equal to rms_inv_f at width 128)
__device__ __forceinline__ float rms_inv_w(float ss, float eps, int width) {
    return rsqrtf(__fmul_rn(ss, 1.0f / (float)width) + eps);
}

// one gated-RMSNorm output element: ((o * inv) * w) * gate(z), gate = sigmoid (KDA) or SiLU
// (GDN's gated_rmsnorm)
template <bool SILU = false>
__device__ __forceinline__ float gated_norm_f(float o, float inv, float w, float z) {
    return __fmul_rn(__fmul_rn(__fmul_rn(o, inv), w), SILU ? silu_f(z) : sigmoid_f(z));
}

// Causal conv taps over a register window win[0..KW-1] whose last K slots hold the K samples
// oldest first (win[KW-1] = current token), weights wr likewise aligned to the end.  Taps are
// accumulated oldest first, one fmaf each, starting from 0; the result does not depend on KW.
template <int KW>
__device__ __forceinline__ float conv_taps_f(const float (&wr)[KW], const float (&win)[KW], int K) {
    float acc = 0.0f;
#pragma unroll
    for (int m = 0; m < KW; ++m)
        if (m >= KW - K) acc = fmaf(wr[m], win[m], acc);
    return acc;
}

template <int KW>
__device__ __forceinline__ void window_push(float (&win)[KW], float x) {
#pragma unroll
    for (int m = 0; m < KW - 1; ++m) win[m] = win[m + 1];
    win[KW - 1] = x;
}

// Sum of squares of a 128-channel head held as channel pairs (2i, 2i+1) by 64 consecutive
// threads (two warps): each thread adds its pair, each warp reduces by butterfly, and the two
// warp partials are added.  Both the prep and the fused decode kernel use this grouping.
__device__ __forceinline__ float pair_sumsq(float x0, float x1) {
    return __fmul_rn(x0, x0) + __fmul_rn(x1, x1);
}

// ------------------------------------------------------------------------------------------
// reductions
// ------------------------------------------------------------------------------------------

// Butterfly sum over all 32 lanes; every lane ends with the same bits (a + b == b + a).
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
    return x;
}

// Butterfly sum over aligned groups of 8 lanes (xor 1, 2, 4).
__device__ __forceinline__ float group8_sum(float x) {
    x += __shfl_xor_sync(0xffffffffu, x, 1);
    x += __shfl_xor_sync(0xffffffffu, x, 2);
    x += __shfl_xor_sync(0xffffffffu, x, 4);
    return x;
}


// ------------------------------------------------------------------------------------------
// loads
// ------------------------------------------------------------------------------------------

template <bool BF16>
__device__ __forceinline__ float load_raw(const void* base, long idx) {
    if constexpr (BF16) {
        return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[idx]);
    } else {
        return reinterpret_cast<const float*>(base)[idx];
    }
}

// Two adjacent raw channels (idx even): one 4-byte bf16x2 or 8-byte float2 load.
template <bool BF16>
__device__ __forceinline__ float2 load_raw2(const void* base, long idx) {
    if constexpr (BF16) {
        return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(
            reinterpret_cast<const __nv_bfloat16*>(base) + idx));
    } else {
        return *reinterpret_cast<const float2*>(reinterpret_cast<const float*>(base) + idx);
    }
}

// ------------------------------------------------------------------------------------------
// mbarrier + TMA (inline PTX, sm_90+ forms valid on sm_103a)
// ------------------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait on an mbarrier phase.  try_wait itself suspends the thread for a while before it
// reports "not yet", so the loop does not spin hot; after kWaitSpinLimit tries (seconds) it
// gives up, raises the device error word and returns false, and the caller stops issuing work.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, int* err) {
    for (int it = 0; it < kWaitSpinLimit; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if (it > 1024) __nanosleep(64);
    }
    if (err) atomicOr(err, kDevErrTimeout);
    return false;
}

// 2D tiled TMA load global -> shared, completion counted on an mbarrier (bytes).
// c0 = innermost (element) coordinate, c1 = row coordinate.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

// 2D tiled TMA store shared -> global into the issuing thread's current bulk group; rows or
// columns outside the tensor are not written.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int c0, int c1) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(smem_u32(src))
                 : "memory");
}

// 1D bulk copy global -> shared (16-byte aligned ends, size a multiple of 16), completion counted
// on an mbarrier (bytes).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// 1D bulk copy shared -> global into the issuing thread's current bulk group (16-byte aligned
// ends, size a multiple of 16).  The shared source must be made visible to the async proxy first
// (fence_proxy_async_smem by the writing threads, then a barrier).
__device__ __forceinline__ void bulk_store(void* dst, const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                     reinterpret_cast<uint64_t>(dst)),
                 "r"(smem_u32(src)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// wait until at most one committed group still reads its shared-memory source
__device__ __forceinline__ void bulk_wait_read1() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// wait until no committed group still reads its shared-memory source
__device__ __forceinline__ void bulk_wait_read0() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// wait until every committed group has completed its writes
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// 3D tiled TMA store shared -> global into the issuing thread's current bulk group.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int c0, int c1,
                                             int c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(src))
                 : "memory");
}

// 16 bytes global -> shared, asynchronous (both addresses 16-byte aligned); a thread sees its
// own copies after cp_async_wait_all
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(src))
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

}  // namespace kda
