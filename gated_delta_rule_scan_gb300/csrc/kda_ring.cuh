// kda_ring.cuh -- the conv ring roll of one (sequence, plane, channel): stage 2 of kda_core_gated
// ("memra_engine/kda.rs", memra-engine 0.125.0) keeps the last K-1 raw samples of every fused
// q/k/v channel for the next call.  Used by the standalone ring-roll kernel (after the staged
// prep) and by the chunked scan's inter kernel (the fused prefill's roll, in its prologue).
#pragma once

#include "kda_device.cuh"
#include "kda_internal.h"

namespace kda {

// ring_out[n][off_p + c][s] = xt[L_n + s] for s < K-1, where xt = (ring_in[n][off_p + c][0 .. K-2],
// plane p's raw rows of sequence n), L_n its length and off_p the plane's first ring row (q, k of
// Hk heads, then v of H heads).  Every old slot is read before any is written, so the roll is safe
// in place (ring_out == ring_in).
template <bool BF16>
__device__ __forceinline__ void ring_roll_one(const PrepArgs& a, int n, int p, long c) {
    const long C = plane_width(a.H, a.Hk, p);          // row width of plane p's raw rows
    const int R = a.K - 1;
    long begin, end;
    if (a.seq.cu_seqlens == nullptr) {
        begin = (long)n * a.seq.T_uniform;
        end = begin + a.seq.T_uniform;
    } else {
        begin = a.seq.cu_seqlens[n];
        end = a.seq.cu_seqlens[n + 1];
    }
    const long Ln = end - begin;
    const void* raw = p == 0 ? a.q_raw : (p == 1 ? a.k_raw : a.v_raw);
    const long base = ((long)n * ring_channels(a.H, a.Hk) + plane_offset(a.H, a.Hk, p) + c) * R;
    float old[kMaxConvK - 1];
#pragma unroll
    for (int s2 = 0; s2 < kMaxConvK - 1; ++s2) old[s2] = s2 < R ? a.ring_in[base + s2] : 0.0f;
#pragma unroll
    for (int s2 = 0; s2 < kMaxConvK - 1; ++s2) {
        if (s2 < R) {
            const long pos = Ln + s2;  // index into xt
            float x;
            if (pos < R) {
                x = 0.0f;
#pragma unroll
                for (int m = 0; m < kMaxConvK - 1; ++m) if (m == pos) x = old[m];
            } else {
                x = load_raw<BF16>(raw, (begin + pos - R) * C + c);
            }
            a.ring_out[base + s2] = x;
        }
    }
}

}  // namespace kda
