/*
 * kda.h -- C ABI of libkda: the Kimi Delta Attention (KDA) gated delta-rule mixer and its
 * scalar-gate special case, Gated DeltaNet (GDN), on one NVIDIA GB300 (sm_103a).
 *
 * The method is the one the docs.rs page "memra_engine/kda.rs" (memra-engine 0.125.0) describes
 * in its module doc and in kda_core_gated stages 2-6; GDN semantics follow the page
 * "aprender-serve 0.70.2 src/cuda/executor/gdn_ops.rs".  Conventions follow the C-ABI launcher
 * pattern of the page "memra_engine/mla_ffi.rs" (memra-engine 0.124.0), module doc:
 *
 *   - Every entry returns 0 on success, 10000 + cudaError_t when a CUDA call fails, and
 *     40000 + n for a contract violation (codes below).  Contract checks run on the host before
 *     anything is launched; a violating call launches nothing and touches no buffer.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).  Every call
 *     is asynchronous on that stream; outputs are ready when the stream reaches the call.  The
 *     stream must belong to the CURRENT device (cudaSetDevice), whose memory the pointers refer
 *     to: the library keys its per-device lookups by the current device, so a stream of another
 *     device returns 40012 and launches nothing.  (While a stream is being captured into a CUDA
 *     graph the runtime refuses that query, and the call cannot check: the caller must keep the
 *     capturing stream's device current.)
 *   - The caller owns all memory.  The library allocates no device memory.  It keeps no state
 *     between calls except one device-side error word (see kda_device_status) and, per device,
 *     cached symbol addresses and function attributes.  The first call on a device may load the
 *     library's module there and set function attributes; after that, with kernel timing off,
 *     calls allocate no host memory either (kernel timing, kda_kernel_timing, creates CUDA events
 *     and grows host-side lists while it is on).  The per-device caches are filled thread-safely;
 *     a device that the process resets (cudaDeviceReset) must not be used with the library again.
 *   - Pointers are device pointers unless the name ends in _host.  Pointers marked [16B] must be
 *     16-byte aligned (40010 otherwise).
 *
 * Notation: N sequences, T tokens per sequence (or total_T packed rows for the varlen entries),
 * H heads, D = head_dim = 128 (the only width built), C = H*D channels, K conv taps (2..8),
 * R = K-1 ring slots.  Channel c = h*D + i is the (head, dim) pair ("Geometry" in the module doc),
 * so every per-token tensor is token-major [rows, C] = [rows, H, D] with no repacking.
 *   state  [N, H, D, D] f32, element [n][h][j][i] = S[i][j]: S has rows i = key dim and columns
 *          j = value dim; the buffer stores it transposed, one value column per 512-byte row
 *          (the "M[col][i]" layout of kda_core's doc).
 *   ring   [N, 3C, R] f32, planes q, k, v at rows 0, C, 2C; slot 0 is the oldest raw sample.
 *   conv_w [3C, K] f32, same plane order; tap K-1 multiplies the current token.
 */
#ifndef KDA_H
#define KDA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
#define KDA_OK 0
#define KDA_ERR_CUDA_BASE 10000       /* 10000 + cudaError_t */
#define KDA_ERR_HEAD_DIM 40001        /* D != 128 */
#define KDA_ERR_CONV_K 40002          /* K outside 2..8 while conv_w != NULL */
#define KDA_ERR_STATE_ALIAS 40003     /* state (or ring) buffers overlap; decode and rollback
                                         accept the very same buffer (in place) */
#define KDA_ERR_NULL 40004            /* a required pointer is NULL */
#define KDA_ERR_SHAPE 40005           /* negative size, H == 0, N or H > 65535, T too large */
#define KDA_ERR_CU_SEQLENS 40006      /* cu_seqlens_host[0] != 0, decreasing, or last != total_T */
#define KDA_ERR_ENUM 40007            /* unknown raw_dtype, gate_mode or algo */
#define KDA_ERR_TIMEOUT 40008         /* a kernel gave up a bounded device wait (kda_device_status) */
#define KDA_ERR_WORKSPACE 40009       /* workspace NULL or smaller than kda_scan_workspace_bytes */
#define KDA_ERR_ALIGN 40010           /* a [16B] pointer is not 16-byte aligned */
#define KDA_ERR_SCRATCH_LIMIT 40011   /* kda_scan_varlen_static: problem needs more scratch than
                                         KDA_STATIC_SCRATCH_BYTES */
#define KDA_ERR_STREAM_DEVICE 40012   /* the stream belongs to a device other than the current one */

/* enums */
#define KDA_DTYPE_F32 0
#define KDA_DTYPE_BF16 1
#define KDA_GATE_PER_CHANNEL 0        /* KDA: g is [rows, C] */
#define KDA_GATE_PER_HEAD 1           /* GDN: g is [rows, H], broadcast over the key dim */
#define KDA_GATE_EXP 2                /* flag, or-ed into gate_mode: g holds the decay factor
                                         exp(log-decay) instead of the log-decay itself */
#define KDA_NORM_SILU 4               /* flag, or-ed into gate_mode of the fused entries
                                         (kda_prefill_fused[_varlen], kda_decode_fused,
                                         kda_verify_rollback): the RMSNorm gates with
                                         SiLU(z) = z * sigmoid(z), the GDN form, instead of
                                         sigmoid(z) (Engine::kda_gated_rmsnorm doc).  The
                                         prep and scan entries have no norm: 40007 there */
#define KDA_ALGO_AUTO 0
#define KDA_ALGO_SEQ 1
#define KDA_ALGO_CHUNK 2

#define KDA_HEAD_DIM 128
#define KDA_STATIC_SCRATCH_BYTES 33554432u  /* kda_scan_varlen_static's fixed scratch (32 MiB) */
#define KDA_DECODE_MAX_T 16

/* ABI revision of this header; bumped on any signature change. */
int kda_abi_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char* kda_status_string(int status);

/*
 * kda_conv_l2norm_prep -- stages 2-4 of kda_core_gated: the scan's inputs from projected
 * channels, for N sequences of T tokens each (rows = N*T, sequence n owns rows n*T .. n*T+T-1).
 *
 *   conv (Engine::kda_conv_silu, stage 2): for plane p and channel c, with xt = the ring slots of
 *     (n, p, c) oldest first followed by the sequence's raw rows,
 *         x_t = silu( sum_{j<K} conv_w[p*C+c][j] * xt[t+j] ), taps summed j ascending;
 *   roll (Engine::kda_conv_ring_roll): ring_out = the last R entries of xt (raw values);
 *   l2   (stage 3, constant KDA_L2_EPS): q_hat, k_hat = x / sqrt(sum_i x_i^2 + l2_eps) per (t, h);
 *        v_hat = x (no norm);
 *   gate (stage 4, Engine::kda_gate): gate_mode 0: g[t][c] = gate_lb * sigmoid(exp(a_log[h]) *
 *        (f_raw[t][c] + dt_bias[c])); gate_mode 1 (gdn_ops.rs gdn_gates_into):
 *        g[t][h] = -exp(a_log[h]) * softplus(f_raw[t][h] + dt_bias[h]); gate_lb is ignored;
 *   beta = sigmoid(beta_raw) per (t, h).
 *   With KDA_GATE_EXP or-ed into gate_mode, g receives exp() of the gate above (the per-step
 *   decay factor in (0, 1]), the form kda_scan consumes without taking exp itself.
 *
 * q_raw, k_raw, v_raw  [rows, C] in raw_dtype (KDA_DTYPE_F32 / KDA_DTYPE_BF16), read only;
 *                      8-byte aligned (bf16) or 16-byte aligned (f32).
 * conv_w               [3C, K] f32, or NULL: no conv and no SiLU (x = raw), rings unused.
 * ring_in, ring_out    [N, 3C, R] f32 (ignored when conv_w is NULL).  They may be the same
 *                      buffer (in-place roll); otherwise they must not overlap.
 * f_raw                [rows, C] (gate_mode 0, [16B]) or [rows, H] (gate_mode 1) f32.
 * dt_bias              [C] (gate_mode 0, [16B]) or [H] (gate_mode 1) f32;  a_log [H] f32.
 * beta_raw             [rows, H] f32.
 * q_hat, k_hat, v_hat  [rows, C] f32 outputs [16B];  g: [rows, C] or [rows, H] f32 output [16B];
 * beta                 [rows, H] f32 output.
 * Returns 40001/40002/40004/40005/40007/40010 on contract violations.
 */
int kda_conv_l2norm_prep(const void* q_raw, const void* k_raw, const void* v_raw, int raw_dtype,
                         const float* conv_w, const float* ring_in, float* ring_out,
                         const float* f_raw, const float* dt_bias, const float* a_log,
                         int gate_mode, float gate_lb, const float* beta_raw, float* q_hat,
                         float* k_hat, float* v_hat, float* g, float* beta, int N, int T, int H,
                         int D, int K, float l2_eps, void* stream);

/*
 * kda_conv_l2norm_prep_varlen -- kda_conv_l2norm_prep over N packed sequences of different
 * lengths: sequence n owns rows cu_seqlens[n] .. cu_seqlens[n+1]-1 of every [rows, ...] array,
 * and ring row n.  cu_seqlens is int32 [N+1] on the device (read by the kernels);
 * cu_seqlens_host is the same array in host memory (validated: starts at 0, non-decreasing, ends
 * at total_T; 40006 otherwise).  Empty sequences are allowed: their ring rows pass through.
 */
int kda_conv_l2norm_prep_varlen(const void* q_raw, const void* k_raw, const void* v_raw,
                                int raw_dtype, const float* conv_w, const float* ring_in,
                                float* ring_out, const float* f_raw, const float* dt_bias,
                                const float* a_log, int gate_mode, float gate_lb,
                                const float* beta_raw, float* q_hat, float* k_hat, float* v_hat,
                                float* g, float* beta, const int* cu_seqlens,
                                const int* cu_seqlens_host, int N, int total_T, int H, int D,
                                int K, float l2_eps, void* stream);

/*
 * Workspace bytes that suffice for kda_scan / kda_scan_varlen over N sequences holding total_T
 * tokens in all (an upper bound for any split of total_T into N lengths): 0 for KDA_ALGO_SEQ,
 * else the chunked form's scratch, about 1.4 KB per (token, head).  Returns 0 for invalid
 * arguments.
 */
size_t kda_scan_workspace_bytes(int N, int total_T, int H, int D, int gate_mode, int algo);

/*
 * kda_scan -- stage 5 of kda_core_gated (Engine::kda_scan, "the per-channel-decay delta-rule
 * scan"; module doc): for each sequence n and head h, for t = 0..T-1:
 *     S <- Diag(exp g_t) S;   u = v_t - S^T k_t;   S <- S + beta_t k_t u^T;   o_t = scale S^T q_t
 * starting from state_in[n][h] and leaving the final state in state_out[n][h].  With gate_mode 1
 * the scalar g[t][h] decays every key-dim row alike (Gated DeltaNet).
 *
 * q_hat, k_hat, v_hat  [N*T, C] f32 [16B] (q_hat, k_hat normally l2-normalised).
 * g                    [N*T, C] f32 [16B] (gate_mode 0) or [N*T, H] f32 (gate_mode 1): raw
 *                      log-decay; the scan applies exp.  With KDA_GATE_EXP or-ed into gate_mode,
 *                      g already holds the decay factors exp(log-decay) (as the prep emits them
 *                      under the same flag) and the scan uses them as they are.
 * beta                 [N*T, H] f32.
 * state_in, state_out  [N, H, D, D] f32 [16B], distinct, non-overlapping buffers (40003).
 * o                    [N*T, C] f32 output [16B].
 * scale                readout scale, normally 1/sqrt(D) (the reference's query scale, applied to
 *                      the readout only).
 * algo                 KDA_ALGO_SEQ: register-resident sequential scan; the T-token call equals T
 *                      chained one-token calls bit for bit.  KDA_ALGO_CHUNK: the chunked (UT/WY)
 *                      form on the tensor cores (module doc's chunked twin); needs workspace;
 *                      for the per-channel gate every 32-token chunk's total log-decay must stay
 *                      above -170 per channel (a bounded gate such as KDA's >= -5 per token
 *                      satisfies it), otherwise kda_device_status reports 40008.  Precision: the
 *                      intra-chunk products are bf16 x 3 (about 16 significant bits); the state
 *                      chain pairs the state and U' = U - W S, split into f16 hi + lo, with f16
 *                      images of its other operands (about 11 bits), so results carry a
 *                      relative error of a few 1e-4 of their scale (inside the 1e-3 parity
 *                      bound), and state and U' entries must stay below 65504 in magnitude.
 *                      KDA_ALGO_AUTO takes the chunked form when a large-enough workspace is given
 *                      and the longest sequence has at least 96 tokens (64 when N * H >= 512),
 *                      else the sequential one: the measured crossover on GB300.
 * workspace            device scratch [16B], at least kda_scan_workspace_bytes(...) bytes for
 *                      KDA_ALGO_CHUNK (40009 otherwise), or NULL.  Its contents are overwritten;
 *                      calls that share a workspace must not overlap on the GPU.
 * T == 0 copies state_in to state_out.
 */
int kda_scan(const float* q_hat, const float* k_hat, const float* v_hat, const float* g,
             int gate_mode, const float* beta, const float* state_in, float* state_out,
             float* o, int N, int T, int H, int D, float scale, int algo, void* workspace,
             size_t workspace_bytes, void* stream);

/*
 * kda_scan_varlen -- kda_scan over N packed sequences (rows cu_seqlens[n] .. cu_seqlens[n+1]-1,
 * state row n); cu_seqlens / cu_seqlens_host as in kda_conv_l2norm_prep_varlen.  An empty
 * sequence copies its state through.
 */
int kda_scan_varlen(const float* q_hat, const float* k_hat, const float* v_hat, const float* g,
                    int gate_mode, const float* beta, const float* state_in, float* state_out,
                    float* o, const int* cu_seqlens, const int* cu_seqlens_host, int N,
                    int total_T, int H, int D, float scale, int algo, void* workspace,
                    size_t workspace_bytes, void* stream);

/*
 * kda_scan_gqa, kda_scan_varlen_gqa -- kda_scan / kda_scan_varlen with grouped queries: q_hat
 * and k_hat hold Hk heads ([rows, Hk*D] f32 [16B]) and value head h reads q/k head h % Hk (the
 * tiled order of `gdn_delta_rule_into` / delta_rule_recurrence_gqa, aprender-serve gdn_ops.rs);
 * v_hat, g, beta, the state and o keep H heads.  Hk >= 1 (40005 otherwise); Hk == H is kda_scan
 * itself.  Same workspace as kda_scan_workspace_bytes(N, total_T, H, ...).
 */
int kda_scan_gqa(const float* q_hat, const float* k_hat, const float* v_hat, const float* g,
                 int gate_mode, const float* beta, const float* state_in, float* state_out,
                 float* o, int N, int T, int H, int Hk, int D, float scale, int algo,
                 void* workspace, size_t workspace_bytes, void* stream);
int kda_scan_varlen_gqa(const float* q_hat, const float* k_hat, const float* v_hat,
                        const float* g, int gate_mode, const float* beta, const float* state_in,
                        float* state_out, float* o, const int* cu_seqlens,
                        const int* cu_seqlens_host, int N, int total_T, int H, int Hk, int D,
                        float scale, int algo, void* workspace, size_t workspace_bytes,
                        void* stream);

/*
 * kda_scan_varlen_static -- kda_scan_varlen with algo KDA_ALGO_CHUNK, except that the chunked
 * form's scratch is a fixed array of KDA_STATIC_SCRATCH_BYTES (32 MiB) inside the library rather
 * than a caller workspace: the call allocates no device memory (no cudaMalloc, no allocating
 * library routine), and after its first call on a device, with kernel timing off, no host memory.  The KDA pages have no counterpart to this entry point.  It is for
 * callers that must not allocate device memory while they run: a serving process that reserves its
 * whole HBM budget at start-up and turns allocation off afterwards (an allocation then fails, or
 * stalls the device in the middle of a step), or plain C code with no allocator at hand.  The
 * array is held on every GPU where the library's scratch module is loaded, until the process exits.
 *
 * Arguments, layouts, results and errors as in kda_scan_varlen (algo and workspace are implied).
 * The results equal kda_scan_varlen with KDA_ALGO_CHUNK bit for bit.
 * Size limit: the problem's chunked scratch -- kda_scan_workspace_bytes for its exact lengths,
 * a 256-byte header plus 43,520 bytes per (32-token chunk, head), about
 * H * sum_n ceil(len_n / 32) <= 771 -- must fit KDA_STATIC_SCRATCH_BYTES; a larger problem
 * returns 40011 and launches nothing.
 * Setup: the first call on each device looks up the array's address once, with that device
 * current (a failure returns 10000 + its cudaError_t); the stream must belong to that device
 * (40012 otherwise), so the kernels never see another device's array.  Make that first call
 * before any stream capture begins.
 * Zeroing: nothing in the scratch has to start at zero; every byte the call reads it has first
 * written itself, so no clearing happens between calls.
 * Concurrency: the array is one per device and shared by every call on it.  Calls that may run
 * at the same time on the GPU (different streams, or several host threads) race on it and
 * corrupt one another's results; serialise them on one stream.
 */
int kda_scan_varlen_static(const float* q_hat, const float* k_hat, const float* v_hat,
                           const float* g, int gate_mode, const float* beta,
                           const float* state_in, float* state_out, float* o,
                           const int* cu_seqlens, const int* cu_seqlens_host, int N, int total_T,
                           int H, int D, float scale, void* stream);

/*
 * kda_gated_rmsnorm_out -- stage 6 of kda_core_gated (Engine::kda_gated_rmsnorm): per row of D
 * values, y_i = o_i / sqrt(mean_i o_i^2 + eps) * norm_w[i] * sigmoid(gate_raw_i).  KDA gates with
 * sigmoid; the gate is not normalised.
 * o, gate_raw, y   [rows, D] f32 [16B] (rows = tokens * heads);  norm_w [D] f32 [16B], shared by
 * all heads.  y may alias o.
 * D                the value head width: 128 * m for m = 1..8 (40001 otherwise); the mean runs over
 *                  the whole row of D values.
 */
int kda_gated_rmsnorm_out(const float* o, const float* norm_w, const float* gate_raw, float* y,
                          long rows, int D, float eps, void* stream);

/*
 * kda_gated_rmsnorm_silu_out -- the same with the SiLU gate of GDN's gated_rmsnorm
 * (Engine::kda_gated_rmsnorm doc: GDN gates with SiLU, KDA with sigmoid):
 * y_i = o_i / sqrt(mean_i o_i^2 + eps) * norm_w[i] * gate_raw_i * sigmoid(gate_raw_i).
 * Arguments as in kda_gated_rmsnorm_out.
 */
int kda_gated_rmsnorm_silu_out(const float* o, const float* norm_w, const float* gate_raw,
                               float* y, long rows, int D, float eps, void* stream);

/*
 * kda_prefill_workspace_bytes -- device scratch that suffices for kda_prefill_fused /
 * kda_prefill_fused_varlen over N sequences holding total_T tokens in all: a readout plane
 * (4 bytes per (token, channel); used by kda_prefill_fused_dv with Dv > 128, whose RMSNorm spans
 * several 128-wide blocks) plus the chunked scan's scratch (kda_scan_workspace_bytes with
 * KDA_ALGO_CHUNK).  Returns 0 for invalid arguments.
 */
size_t kda_prefill_workspace_bytes(int N, int total_T, int H, int D, int gate_mode);

/*
 * kda_prefill_fused -- a prefill of N sequences of T tokens in one call: stages 2-6 of
 * kda_core_gated (conv + SiLU, l2 norm, gates and beta, the chunked scan, gated RMSNorm), the
 * same computation as kda_conv_l2norm_prep + kda_scan with KDA_ALGO_CHUNK +
 * kda_gated_rmsnorm_out with the same arguments.  The prepared q, k, v and gates are computed
 * inside the chunked scan's first kernel and never reach memory.  With N * H at least two thirds
 * of the device's SM count the readout is normalised inside the chunked scan's second kernel as
 * it leaves (the RMSNorm of a row needs only that row); with fewer (sequence, head) pairs it
 * passes through the workspace to the RMSNorm kernel.  y is the same either way.
 * Arguments and layouts as in those three calls, except that bf16 q_raw, k_raw and v_raw must be
 * [16B] here (40010 otherwise; the staged prep needs 8 bytes); gate_mode is KDA_GATE_PER_CHANNEL
 * or KDA_GATE_PER_HEAD (the KDA_GATE_EXP flag is not accepted, 40007); norm_w [D] f32 [16B];
 * gate_raw and y [N*T, C] f32 [16B].  The chunked form's range condition applies (every
 * 32-token chunk's total log-decay above -170 per channel, else kda_device_status reports 40008).
 * workspace   device scratch [16B] of at least kda_prefill_workspace_bytes(...) bytes (40009
 *             otherwise); its contents are overwritten, so calls sharing it must not overlap.
 * y, state_out and ring_out equal those of the three calls bit for bit.
 */
int kda_prefill_fused(const void* q_raw, const void* k_raw, const void* v_raw, int raw_dtype,
                      const float* conv_w, const float* ring_in, float* ring_out,
                      const float* f_raw, const float* dt_bias, const float* a_log, int gate_mode,
                      float gate_lb, const float* beta_raw, const float* state_in,
                      float* state_out, const float* norm_w, const float* gate_raw, float* y,
                      int N, int T, int H, int D, int K, float l2_eps, float scale,
                      float rms_eps, void* workspace, size_t workspace_bytes, void* stream);

/*
 * kda_prefill_fused_varlen -- kda_prefill_fused over N packed sequences (rows cu_seqlens[n] ..
 * cu_seqlens[n+1]-1, state and ring row n); cu_seqlens / cu_seqlens_host as in
 * kda_conv_l2norm_prep_varlen.
 */
int kda_prefill_fused_varlen(const void* q_raw, const void* k_raw, const void* v_raw,
                             int raw_dtype, const float* conv_w, const float* ring_in,
                             float* ring_out, const float* f_raw, const float* dt_bias,
                             const float* a_log, int gate_mode, float gate_lb,
                             const float* beta_raw, const float* state_in, float* state_out,
                             const float* norm_w, const float* gate_raw, float* y,
                             const int* cu_seqlens, const int* cu_seqlens_host, int N,
                             int total_T, int H, int D, int K, float l2_eps, float scale,
                             float rms_eps, void* workspace, size_t workspace_bytes,
                             void* stream);

/*
 * Per-kernel timing (support, for measurement; not part of the method).
 * kda_kernel_timing(1) makes every kernel launch of the library record a CUDA event before and
 * after it on its stream, and clears the totals; kda_kernel_timing(0) stops.  Returns the previous
 * setting.  Off by default, when it costs nothing measurable.
 * kda_kernel_times waits for the recorded launches, writes for kernel ids 0 .. max_kernels-1 the
 * number of launches and their summed device time in milliseconds since the last read (either
 * array may be NULL), clears them, and returns the number of kernel ids, or -(10000 + cudaError_t)
 * on a CUDA error.  kda_kernel_name(id) is that kernel's name, NULL outside the range.
 */
int kda_kernel_timing(int enable);
int kda_kernel_times(int max_kernels, long* launches, double* total_ms);
const char* kda_kernel_name(int id);

/*
 * kda_decode_fused -- one decode step (T = 1) or a T-token speculative verify (2 <= T <= 16) of
 * N sequences in ONE launch: kda_conv_l2norm_prep + kda_scan + kda_gated_rmsnorm_out with the
 * same arguments, computed without round-tripping the intermediates through memory.  Its outputs
 * equal those three calls to f32 rounding (the ring bit for bit; the two scans sum the key
 * dimension over different lane groupings), and a T-token call equals T chained one-token calls
 * bit for bit (the decode == verify identity of the KDA module doc).
 * Argument meanings and layouts as in the three calls; rows = N*T; conv_w must not be NULL.
 * ring_in / ring_out may be the same buffer, and so may state_in / state_out (an in-place step:
 * with stable pointers a decode step can be captured once in a CUDA graph and replayed); buffers
 * that overlap without being the same return 40003.
 * norm_w [D] [16B], gate_raw and y [rows, C] f32 [16B].  T outside 1..16 returns 40005.
 */
int kda_decode_fused(const void* q_raw, const void* k_raw, const void* v_raw, int raw_dtype,
                     const float* conv_w, const float* ring_in, float* ring_out,
                     const float* f_raw, const float* dt_bias, const float* a_log, int gate_mode,
                     float gate_lb, const float* beta_raw, const float* state_in,
                     float* state_out, const float* norm_w, const float* gate_raw, float* y,
                     int N, int T, int H, int D, int K, float l2_eps, float scale, float rms_eps,
                     void* stream);

/*
 * kda_verify_rollback -- the rollback of a speculative verify round (kda_verify_rollback_rows,
 * memra_engine/kda.rs, memra-engine 0.125.0: restore the pre-round conv ring, re-roll the kept
 * raw rows, replay the scan at T = keep from the pre-round state): from the state and ring BEFORE
 * a T-token verify, take only the first keep[n] rows of each sequence n of the same verify batch
 * and produce the state, ring and y rows that keep[n] chained one-token kda_decode_fused calls
 * would, bit for bit (the decode == verify identity applied to the accepted prefix).  One launch;
 * the prep of the kept rows is recomputed from the raw rows with the verify's own arithmetic.
 * Arguments as in kda_decode_fused, plus
 * keep        device int32 [N]: tokens accepted per sequence, clamped to 0..T on the device
 *             (keep[n] = 0 leaves state and ring of sequence n as they were).  NULL returns 40004.
 * The raw rows, f, beta and gate_raw keep the verify batch's layout: row n*T + t.  ring_in must
 * hold the ring from before the round (the verify call may not have rolled it in place, or the
 * caller keeps a copy); state_in the state from before the round (the verify ran out of place,
 * or the caller keeps a copy).  y rows n*T + t are written for t < keep[n] only.
 */
int kda_verify_rollback(const void* q_raw, const void* k_raw, const void* v_raw, int raw_dtype,
                        const float* conv_w, const float* ring_in, float* ring_out,
                        const float* f_raw, const float* dt_bias, const float* a_log,
                        int gate_mode, float gate_lb, const float* beta_raw,
                        const float* state_in, float* state_out, const float* norm_w,
                        const float* gate_raw, float* y, const int* keep, int N, int T, int H,
                        int D, int K, float l2_eps, float scale, float rms_eps, void* stream);

/*
 * Grouped queries through the whole mixer (the GDN page's head mapping, aprender-serve gdn_ops.rs
 * `gdn_delta_rule_into` doc: q and k hold num_k_heads heads and value head h reads query/key head
 * h % num_k_heads; beta and the gate are per value head).  Each entry equals the entry without the
 * suffix, with Hk (1 <= Hk <= H, 40005 otherwise) q/k heads:
 *   q_raw, k_raw  [rows, Hk*D] (the staged prep's q_hat, k_hat outputs likewise; they feed
 *                 kda_scan_gqa / kda_scan_varlen_gqa);
 *   v_raw, f_raw, gate_raw, y, the state, beta: H value heads as before;
 *   conv_w        [2*Hk*D + H*D, K], rows [q | k | v];  ring [N, 2*Hk*D + H*D, K-1], same order.
 * Hk == H is the entry without the suffix.  kda_decode_fused_gqa and kda_verify_rollback_gqa with
 * Hk < H cannot roll the ring in place (several value heads read one q/k ring row that only one of
 * them rewrites): ring_in == ring_out returns 40003 there.
 */
int kda_conv_l2norm_prep_gqa(const void* q_raw, const void* k_raw, const void* v_raw,
                             int raw_dtype, const float* conv_w, const float* ring_in,
                             float* ring_out, const float* f_raw, const float* dt_bias,
                             const float* a_log, int gate_mode, float gate_lb,
                             const float* beta_raw, float* q_hat, float* k_hat, float* v_hat,
                             float* g, float* beta, int N, int T, int H, int Hk, int D, int K,
                             float l2_eps, void* stream);
int kda_conv_l2norm_prep_varlen_gqa(const void* q_raw, const void* k_raw, const void* v_raw,
                                    int raw_dtype, const float* conv_w, const float* ring_in,
                                    float* ring_out, const float* f_raw, const float* dt_bias,
                                    const float* a_log, int gate_mode, float gate_lb,
                                    const float* beta_raw, float* q_hat, float* k_hat,
                                    float* v_hat, float* g, float* beta, const int* cu_seqlens,
                                    const int* cu_seqlens_host, int N, int total_T, int H,
                                    int Hk, int D, int K, float l2_eps, void* stream);
int kda_prefill_fused_gqa(const void* q_raw, const void* k_raw, const void* v_raw, int raw_dtype,
                          const float* conv_w, const float* ring_in, float* ring_out,
                          const float* f_raw, const float* dt_bias, const float* a_log,
                          int gate_mode, float gate_lb, const float* beta_raw,
                          const float* state_in, float* state_out, const float* norm_w,
                          const float* gate_raw, float* y, int N, int T, int H, int Hk, int D,
                          int K, float l2_eps, float scale, float rms_eps, void* workspace,
                          size_t workspace_bytes, void* stream);
int kda_prefill_fused_varlen_gqa(const void* q_raw, const void* k_raw, const void* v_raw,
                                 int raw_dtype, const float* conv_w, const float* ring_in,
                                 float* ring_out, const float* f_raw, const float* dt_bias,
                                 const float* a_log, int gate_mode, float gate_lb,
                                 const float* beta_raw, const float* state_in, float* state_out,
                                 const float* norm_w, const float* gate_raw, float* y,
                                 const int* cu_seqlens, const int* cu_seqlens_host, int N,
                                 int total_T, int H, int Hk, int D, int K, float l2_eps,
                                 float scale, float rms_eps, void* workspace,
                                 size_t workspace_bytes, void* stream);
int kda_decode_fused_gqa(const void* q_raw, const void* k_raw, const void* v_raw, int raw_dtype,
                         const float* conv_w, const float* ring_in, float* ring_out,
                         const float* f_raw, const float* dt_bias, const float* a_log,
                         int gate_mode, float gate_lb, const float* beta_raw,
                         const float* state_in, float* state_out, const float* norm_w,
                         const float* gate_raw, float* y, int N, int T, int H, int Hk, int D, int K,
                         float l2_eps, float scale, float rms_eps, void* stream);
int kda_verify_rollback_gqa(const void* q_raw, const void* k_raw, const void* v_raw,
                            int raw_dtype, const float* conv_w, const float* ring_in,
                            float* ring_out, const float* f_raw, const float* dt_bias,
                            const float* a_log, int gate_mode, float gate_lb,
                            const float* beta_raw, const float* state_in, float* state_out,
                            const float* norm_w, const float* gate_raw, float* y, const int* keep,
                            int N, int T, int H, int Hk, int D, int K, float l2_eps, float scale,
                            float rms_eps, void* stream);

/*
 * A value head wider than the key head (the GDN page's head dims, aprender-serve gdn_ops.rs
 * `gdn_delta_rule_into` doc: q and k are num_k_heads * head_k_dim wide, v num_v_heads *
 * head_v_dim, and the state of one value head is head_v_dim x head_k_dim).  Dk = 128 and
 * Dv = 128 * m, m = 1..8 (40001 otherwise); H value heads, Hk q/k heads (1 <= Hk <= H, value head
 * h reads q/k head h % Hk; 40005 otherwise).  Layouts, row-major f32 unless stated:
 *   q_raw, k_raw, q_hat, k_hat  [rows, Hk*Dk];  v_raw, v_hat, o  [rows, H*Dv];
 *   f_raw, g   [rows, H*Dk] (gate_mode 0: the decay is over the key dim) or [rows, H] (mode 1);
 *   dt_bias    [H*Dk] (mode 0) or [H];  a_log, beta_raw rows, beta rows  [H] per row;
 *   conv_w     [2*Hk*Dk + H*Dv, K], rows [q | k | v];  ring [N, 2*Hk*Dk + H*Dv, K-1];
 *   state      [N, H, Dv, Dk] f32 [16B]: state[n][h][j][i] couples value column j and key row i.
 * The scan is kda_scan's recurrence with a Dk x Dv state per value head, run as m independent
 * 128-wide value column blocks (column block b of value head h is unit h*m + b of a kda_scan with
 * H*m heads, sharing value head h's gate, beta and q/k head: the recurrence's columns never mix).
 * The workspace for the chunked form is kda_scan_workspace_bytes(N, total_T, H*m, 128, ...).
 * The gated RMSNorm over rows of Dv values is kda_gated_rmsnorm_out / _silu_out with D = Dv.
 * The fused entries take the same layouts, plus
 *   norm_w     [Dv];  gate_raw, y  [rows, H*Dv];  the RMSNorm's mean over the whole Dv row.
 *   kda_prefill_fused_dv / _varlen_dv: workspace of kda_prefill_workspace_bytes(N, total_T, H*m,
 *   128, gate_mode) bytes; outputs equal kda_conv_l2norm_prep_dv + kda_scan_dv (KDA_ALGO_CHUNK)
 *   + kda_gated_rmsnorm_out(D = Dv) bit for bit.
 *   kda_decode_fused_dv / kda_verify_rollback_dv: one launch in which each value head is a
 *   thread-block cluster of m CTAs (one per 128-wide column block) that sum the RMSNorm's squares
 *   across the cluster; decode == verify bit for bit and the staged path to f32 rounding, as for
 *   Dv = 128.  With
 *   m > 1 or Hk < H the ring cannot be rolled in place (ring_in == ring_out returns 40003).
 */
int kda_conv_l2norm_prep_dv(const void* q_raw, const void* k_raw, const void* v_raw,
                            int raw_dtype, const float* conv_w, const float* ring_in,
                            float* ring_out, const float* f_raw, const float* dt_bias,
                            const float* a_log, int gate_mode, float gate_lb,
                            const float* beta_raw, float* q_hat, float* k_hat, float* v_hat,
                            float* g, float* beta, int N, int T, int H, int Hk, int Dk, int Dv,
                            int K, float l2_eps, void* stream);
int kda_conv_l2norm_prep_varlen_dv(const void* q_raw, const void* k_raw, const void* v_raw,
                                   int raw_dtype, const float* conv_w, const float* ring_in,
                                   float* ring_out, const float* f_raw, const float* dt_bias,
                                   const float* a_log, int gate_mode, float gate_lb,
                                   const float* beta_raw, float* q_hat, float* k_hat,
                                   float* v_hat, float* g, float* beta, const int* cu_seqlens,
                                   const int* cu_seqlens_host, int N, int total_T, int H, int Hk,
                                   int Dk, int Dv, int K, float l2_eps, void* stream);
int kda_scan_dv(const float* q_hat, const float* k_hat, const float* v_hat, const float* g,
                int gate_mode, const float* beta, const float* state_in, float* state_out,
                float* o, int N, int T, int H, int Hk, int Dk, int Dv, float scale, int algo,
                void* workspace, size_t workspace_bytes, void* stream);
int kda_scan_varlen_dv(const float* q_hat, const float* k_hat, const float* v_hat,
                       const float* g, int gate_mode, const float* beta, const float* state_in,
                       float* state_out, float* o, const int* cu_seqlens,
                       const int* cu_seqlens_host, int N, int total_T, int H, int Hk, int Dk,
                       int Dv, float scale, int algo, void* workspace, size_t workspace_bytes,
                       void* stream);
int kda_prefill_fused_dv(const void* q_raw, const void* k_raw, const void* v_raw, int raw_dtype,
                         const float* conv_w, const float* ring_in, float* ring_out,
                         const float* f_raw, const float* dt_bias, const float* a_log,
                         int gate_mode, float gate_lb, const float* beta_raw,
                         const float* state_in, float* state_out, const float* norm_w,
                         const float* gate_raw, float* y, int N, int T, int H, int Hk, int Dk,
                         int Dv, int K, float l2_eps, float scale, float rms_eps, void* workspace,
                         size_t workspace_bytes, void* stream);
int kda_prefill_fused_varlen_dv(const void* q_raw, const void* k_raw, const void* v_raw,
                                int raw_dtype, const float* conv_w, const float* ring_in,
                                float* ring_out, const float* f_raw, const float* dt_bias,
                                const float* a_log, int gate_mode, float gate_lb,
                                const float* beta_raw, const float* state_in, float* state_out,
                                const float* norm_w, const float* gate_raw, float* y,
                                const int* cu_seqlens, const int* cu_seqlens_host, int N,
                                int total_T, int H, int Hk, int Dk, int Dv, int K, float l2_eps,
                                float scale, float rms_eps, void* workspace,
                                size_t workspace_bytes, void* stream);
int kda_decode_fused_dv(const void* q_raw, const void* k_raw, const void* v_raw, int raw_dtype,
                        const float* conv_w, const float* ring_in, float* ring_out,
                        const float* f_raw, const float* dt_bias, const float* a_log,
                        int gate_mode, float gate_lb, const float* beta_raw,
                        const float* state_in, float* state_out, const float* norm_w,
                        const float* gate_raw, float* y, int N, int T, int H, int Hk, int Dk,
                        int Dv, int K, float l2_eps, float scale, float rms_eps, void* stream);
int kda_verify_rollback_dv(const void* q_raw, const void* k_raw, const void* v_raw,
                           int raw_dtype, const float* conv_w, const float* ring_in,
                           float* ring_out, const float* f_raw, const float* dt_bias,
                           const float* a_log, int gate_mode, float gate_lb,
                           const float* beta_raw, const float* state_in, float* state_out,
                           const float* norm_w, const float* gate_raw, float* y, const int* keep,
                           int N, int T, int H, int Hk, int Dk, int Dv, int K, float l2_eps,
                           float scale, float rms_eps, void* stream);

/*
 * kda_proj6 -- stage 1 of kda_core_gated: the six projections of the layer input that the mixer
 * reads, in one call (Engine::kda_proj_fused6, its bf16-weight arm; the shapes are the
 * KdaAttnLayer field docs of "memra_engine/kda.rs"): for every token row s < t,
 *     out[s][r] = sum_{k < in_f} W[r][k] * x[s][k]
 * for W = w_q, w_k, w_v [H*D, in_f] -> q_raw, k_raw, v_raw [t, H*D]; W = w_fa, w_ga [D, in_f] ->
 * f_down, g_down [t, D] (the forget and output gates' down-projections, which the layer's own
 * low-rank up-projections widen to [t, H*D]); W = w_b [H, in_f] -> beta_raw [t, H].  The outputs
 * are what kda_decode_fused / kda_prefill_fused take as q_raw, k_raw, v_raw (raw_dtype f32) and
 * beta_raw.
 *
 * x            [t, in_f] f32 [16B], t = 1..256 token rows (a decode or verify batch), in_f a
 *              multiple of 128 (40005 otherwise).
 * w_*          bf16 (raw 16-bit patterns), row-major [rows, in_f] [16B].
 * outputs      f32 row-major, written for the t rows only.
 * H heads, D = 128 (40001 otherwise).
 * workspace    device scratch [16B] of at least kda_proj6_workspace_bytes(t, in_f) bytes (40009
 *              otherwise): x split into bf16 hi + lo images.  Calls sharing it must not overlap.
 * Precision: the weights' bf16 values enter the products exactly; x enters as hi + lo (about 16
 * significant bits); the sums accumulate in f32.  One token row's result does not depend on the
 * other rows of the call.
 */
size_t kda_proj6_workspace_bytes(int t, int in_f);
int kda_proj6(const float* x, int t, int in_f, const void* w_q, const void* w_k, const void* w_v,
              const void* w_fa, const void* w_ga, const void* w_b, float* q_raw, float* k_raw,
              float* v_raw, float* f_down, float* g_down, float* beta_raw, int H, int D,
              void* workspace, size_t workspace_bytes, void* stream);

/*
 * kda_selftest_wait_timeout -- a self-test of failure detection (no counterpart in the pages):
 * launches one kernel whose single thread waits, with the bounded wait every kernel here uses,
 * on a barrier that nothing completes.  The wait gives up after about a second, raises the device
 * error word and the kernel ends; a following kda_device_status(stream) returns 40008 (and
 * clears the word).  Nothing faults or hangs; the context stays usable.  Returns 0, or
 * 10000 + cudaError_t if the launch fails.
 */
int kda_selftest_wait_timeout(void* stream);

/*
 * kda_device_status -- synchronises `stream`, then reports and clears the device error word on
 * the current device: 0, or 40008 when a kernel gave up a bounded device wait since the last
 * check (its outputs are then incomplete), or 10000 + cudaError_t.
 */
int kda_device_status(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H */
