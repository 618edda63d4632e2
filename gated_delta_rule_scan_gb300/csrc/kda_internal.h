// kda_internal.h -- host-side launch interface between the C ABI (kda_api.cu) and the kernels.
// Every launcher assumes its arguments already passed the ABI's contract checks and returns the
// cudaError_t of its launch(es).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace kda {

constexpr int kHeadDim = 128;      // the only head width the kernels are built for
constexpr int kMaxConvK = 8;       // conv window held in registers (taps 2..8)
constexpr int kMaxDevices = 64;    // per-device caches (symbol addresses, function attributes)

// A value looked up once per device (a symbol address, an attribute that was set).  Every slot
// is an atomic, so host threads that make their first call on one device at the same time each
// look the value up and store the same result: no data race.  The cache is not invalidated by
// cudaDeviceReset; a process that resets a device must not call the library on it afterwards.
template <typename T>
using PerDevice = std::atomic<T>[kMaxDevices];

// Row ranges of the packed token-major arrays.  When cu_seqlens is null every sequence has
// T_uniform tokens and sequence n owns rows [n*T, (n+1)*T).
struct SeqLayout {
    const int* cu_seqlens;   // device int32 [N+1] or null
    int T_uniform;
    int N;
    long total_rows;
};

struct PrepArgs {
    const void* q_raw; const void* k_raw; const void* v_raw; int raw_bf16;
    const float* conv_w;                 // [3C, K] or null (no conv, no SiLU)
    const float* ring_in; float* ring_out;  // [N, 3C, K-1]
    const float* f_raw; const float* dt_bias; const float* a_log; int gate_mode; float gate_lb;
    const float* beta_raw;
    float* q_hat; float* k_hat; float* v_hat; float* g; float* beta;
    SeqLayout seq;
    int H; int K; float l2_eps;
    int Hk;                  // heads of the q and k planes (grouped queries: value head h reads
                             // q/k head h % Hk); 0 means H
    int Hg;                  // heads of the gate and beta (a value head wider than 128 is H / Hg
                             // 128-wide sub-heads that share them); 0 means H
};

// Gate / beta heads of a prep call (the value heads); H counts 128-wide value sub-heads.
__host__ __device__ inline int prep_gate_heads(const PrepArgs& a) { return a.Hg > 0 ? a.Hg : a.H; }

// Channel layout of the three conv planes under grouped queries: q and k hold Hk heads, v holds H;
// conv_w rows and ring rows are [q | k | v] = [Hk*D | Hk*D | H*D] (gdn_ops.rs gdn_delta_rule_into
// doc: q, k are [num_k_heads * head_k_dim], v is [num_v_heads * head_v_dim]).
__host__ __device__ inline int prep_qk_heads(int H, int Hk) { return Hk > 0 ? Hk : H; }
__host__ __device__ inline long plane_width(int H, int Hk, int p) {
    return (long)(p < 2 ? prep_qk_heads(H, Hk) : H) * kHeadDim;
}
__host__ __device__ inline long plane_offset(int H, int Hk, int p) {
    return (long)p * prep_qk_heads(H, Hk) * kHeadDim;
}
__host__ __device__ inline long ring_channels(int H, int Hk) {
    return (2L * prep_qk_heads(H, Hk) + H) * kHeadDim;
}

struct ScanArgs {
    const float* q; const float* k; const float* v; const float* g; int gate_mode;
    const float* beta;
    const float* state_in; float* state_out; float* o;
    SeqLayout seq;
    int H; float scale;
    const int* order;        // device-side order of sequences (longest first) or null
    int* err;                // device error word
    int Hk;                  // heads of q and k (grouped queries: value head h reads q/k head
                             // h % Hk; rows of q and k are Hk * D wide); 0 means H
    int vsub;                // 128-wide sub-heads per value head (value width vsub * 128): unit h
                             // is value head h / vsub, which owns the gate and beta and reads q/k
                             // head (h / vsub) % Hk; 0 means 1
    // the gated RMSNorm folded into the chunked scan's readout (fused prefill, 128-wide value
    // heads): with norm_y set the chunk kernel writes y = rmsnorm(o) * w * gate(z) in place of o
    const float* norm_w; const float* norm_z; float* norm_y; float norm_eps;
    int norm_silu;           // gate: 0 sigmoid (KDA), 1 SiLU (GDN's gated_rmsnorm)
};

// the heads of q and k, and the one value head h reads
__host__ __device__ inline int qk_heads(const ScanArgs& a) { return a.Hk > 0 ? a.Hk : a.H; }
__host__ __device__ inline int value_sub(const ScanArgs& a) { return a.vsub > 0 ? a.vsub : 1; }
// the value head (gate and beta head) of unit h, the number of such heads, and the q/k head
__host__ __device__ inline int gate_head(const ScanArgs& a, int h) { return h / value_sub(a); }
__host__ __device__ inline int gate_heads(const ScanArgs& a) { return a.H / value_sub(a); }
__host__ __device__ inline int unit_qk_head(const ScanArgs& a, int h) {
    return gate_head(a, h) % qk_heads(a);
}

struct NormArgs {
    const float* o; const float* w; const float* z; float* y; long rows; float eps;
    int silu;                // gate: 0 sigmoid (KDA), 1 SiLU (GDN's gated_rmsnorm)
    int width;               // row length, a multiple of 128 (0 means 128)
};

struct DecodeArgs {
    const void* q_raw; const void* k_raw; const void* v_raw; int raw_bf16;
    const float* conv_w; const float* ring_in; float* ring_out;
    const float* f_raw; const float* dt_bias; const float* a_log; int gate_mode; float gate_lb;
    const float* beta_raw;
    const float* state_in; float* state_out;
    const float* norm_w; const float* gate_raw; float* y;
    int N; int T; int H; int K; float l2_eps; float scale; float rms_eps;
    const int* keep;         // rollback: tokens of sequence n to take (device [N], clamped to
                             // 0..T; rows keep their stride T), or null for all T
    int Hk;                  // heads of the q and k planes (grouped queries); 0 means H
    int norm_silu;           // RMSNorm gate: 0 sigmoid (KDA), 1 SiLU (GDN's gated_rmsnorm)
    int* err;                // device error word (bounded waits)
    int vsub;                // 128-wide units per value head (H counts units); 0 means 1.  A
                             // value head's units run as one thread-block cluster, which sums the
                             // RMSNorm's squares over the whole value row
};

cudaError_t launch_prep(const PrepArgs& a, cudaStream_t s);
cudaError_t launch_wait_selftest(int* err, cudaStream_t s);
cudaError_t launch_scan_seq(const ScanArgs& a, cudaStream_t s);
cudaError_t launch_scan_chunk(const ScanArgs& a, const int* cu_host, void* workspace,
                              cudaStream_t s);
// exact workspace the chunked scan needs for this layout (cu_host: host copy of cu_seqlens)
size_t chunk_workspace_bytes(const SeqLayout& s, const int* cu_host, int H);
long chunk_count(const SeqLayout& s, const int* cu_host);
// pieces of the chunked form for the fused prefill (kda_scan_chunk.cu): the varlen chunk offsets
// at the head of the workspace (blocks = where the per-(chunk, head) blocks start), and the
// inter-chunk kernel over filled blocks
cudaError_t launch_chunk_offsets(const SeqLayout& seq, void* workspace, int** chunk_off,
                                 unsigned char** blocks, cudaStream_t s);
cudaError_t launch_chunk_inter(const ScanArgs& a, const int* chunk_off,
                               const unsigned char* blocks, cudaStream_t s,
                               const PrepArgs* ring = nullptr);
// the fused prefill's prep + intra-chunk kernel, then the ring roll (kda_chunk_prep.cu)
cudaError_t launch_prefill_chunk(const PrepArgs& p, const ScanArgs& a, const int* cu_host,
                                 void* workspace, cudaStream_t s);
// the conv ring roll alone (kda_prep.cu)
cudaError_t launch_ring_roll(const PrepArgs& a, cudaStream_t s);

// Fixed device scratch for kda_scan_varlen_static (kda_scan_static.cu): its byte size, and the
// address of this device's copy (looked up once per device, on the first call with it current).
constexpr size_t kStaticScratchBytes = (size_t)32 << 20;
cudaError_t static_scratch(void** ptr);
constexpr int kChunkTokens = 32;        // tokens per chunk of the chunked scan
constexpr size_t kChunkBlockBytes = 43520;  // workspace bytes per (chunk, head)

// 2-D f32 tensor map over [rows, cols] (row stride = cols), box [box_rows, box_cols], no swizzle.
bool make_tensor_map_2d(CUtensorMap* m, const float* base, long rows, long cols, int box_cols,
                        int box_rows);
// The same over bf16 (bf16 = true) or f32 elements.
bool make_tensor_map_2d_any(CUtensorMap* m, const void* base, bool bf16, long rows, long cols,
                            int box_cols, int box_rows);
// The U rows of the chunked scan's workspace blocks: f32 [nblocks][32 tokens][128 values] at
// `base` (the first block's U region), block stride block_bytes; box [1][32][32], 128-byte swizzle.
bool make_tensor_map_blocks_ut(CUtensorMap* m, void* base, long nblocks, size_t block_bytes);
// The layer input's six projections (kda_proj.cu).  Weights are bf16 [rows_i, in_f]; outputs f32
// [t, rows_i]; x f32 [t, in_f]; ws holds x split into bf16 hi / lo images of t_pad rows.
struct Proj6Args {
    const float* x;
    const void* w[6];
    float* out[6];
    int rows[6];
    int t; int in_f;
    void* ws;
    int* err;
};
constexpr int kProjMaxT = 256;          // token rows per call: the MMA's N
constexpr int kProjKAlign = 128;        // in_f must be a multiple of this
inline int proj_t_pad(int t) { return (t + 15) / 16 * 16; }
inline size_t proj_workspace_bytes(int t, int in_f) {
    return 2 * (size_t)proj_t_pad(t) * (size_t)in_f * 2;   // x hi and x lo, bf16
}
cudaError_t launch_proj6(const Proj6Args& a, cudaStream_t s);
// 2-D bf16 tensor map over [rows, cols] with a [box_rows][64] box in the 128-byte swizzle
bool make_tensor_map_2d_bf16_sw128(CUtensorMap* m, const void* base, long rows, long cols,
                                   int box_rows);
cudaError_t launch_gated_rmsnorm(const NormArgs& a, cudaStream_t s);
cudaError_t launch_decode_fused(const DecodeArgs& a, cudaStream_t s);

constexpr int kDecodeMaxT = 16;   // tokens one fused decode/verify call may carry

// ---- optional per-kernel timing (kda_timer.cu): a KernelTimer scoped around a launch records a
// CUDA event before and after it on the launch stream while timing is enabled.
enum KernelId {
    kKPrep, kKRingRoll, kKScanSeq, kKChunkOffsets, kKChunkIntra, kKChunkInter, kKRmsNorm,
    kKDecode, kKPrepIntra, kKProjSplit, kKProj6, kKernelCount
};
class KernelTimer {
public:
    KernelTimer(int id, cudaStream_t s);
    ~KernelTimer();
    KernelTimer(const KernelTimer&) = delete;
    KernelTimer& operator=(const KernelTimer&) = delete;
private:
    int id_; cudaStream_t s_; bool on_;
};

}  // namespace kda
