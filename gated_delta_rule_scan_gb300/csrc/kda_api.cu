// kda_api.cu -- the extern "C" boundary of libkda: host-side contract checks, then dispatch to
// the kernel launchers.  Status bands follow the launcher pattern of "memra_engine/mla_ffi.rs"
// (memra-engine 0.124.0): 0 ok, 10000 + cudaError_t, 40000 + contract code.  No check touches
// the GPU, so a violating call launches nothing.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"
#include "kda_internal.h"

namespace {

using namespace kda;

// one device error word per device, raised by kernels that give up a bounded wait
__device__ int g_kda_dev_err;

constexpr int kMaxGridY = 65535;  // sequences (and heads) map to gridDim.y
constexpr int kMaxValueWidth = 1024;   // widest value head: 8 sub-heads of 128

// the current device's error word (its address is looked up once per device)
int* dev_err_ptr() {
    static PerDevice<int*> ptrs;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    int* p = ptrs[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        void* q = nullptr;
        if (cudaGetSymbolAddress(&q, g_kda_dev_err) != cudaSuccess) return nullptr;
        p = static_cast<int*>(q);
        ptrs[dev].store(p, std::memory_order_release);
    }
    return p;
}

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA_BASE + (int)e; }

// The kernels run on the stream's device, while the per-device lookups (the error word, the fixed
// scratch, function attributes) follow the current device: a stream of another device is a
// contract violation (40012).  The legacy and per-thread default streams always belong to the
// current device.  Only host-side queries; nothing is launched.  The runtime refuses the stream's
// device query while the stream is being captured into a graph (error 900), so a capturing stream
// is not checked: the caller then answers for the match itself.
int check_stream_device(void* stream) {
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (s == nullptr || s == cudaStreamLegacy || s == cudaStreamPerThread) return KDA_OK;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(s, &cs);
    if (e != cudaSuccess) return cuda_status(e);
    if (cs != cudaStreamCaptureStatusNone) return KDA_OK;
    int sdev = -1, cur = -1;
    e = cudaStreamGetDevice(s, &sdev);
    if (e != cudaSuccess) return cuda_status(e);
    e = cudaGetDevice(&cur);
    if (e != cudaSuccess) return cuda_status(e);
    return sdev == cur ? KDA_OK : KDA_ERR_STREAM_DEVICE;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline bool overlap(const void* a, const void* b, size_t bytes) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + bytes && y < x + bytes;
}

int check_cu(const int* cu_host, int N, long total) {
    if (cu_host == nullptr) return KDA_ERR_NULL;
    if (cu_host[0] != 0) return KDA_ERR_CU_SEQLENS;
    for (int n = 0; n < N; ++n)
        if (cu_host[n + 1] < cu_host[n]) return KDA_ERR_CU_SEQLENS;
    if ((long)cu_host[N] != total) return KDA_ERR_CU_SEQLENS;
    return KDA_OK;
}

// Contract checks of the prep stages and their argument block.  planes: the call writes the
// q, k, v, g, beta planes (the fused prefill does not, and passes them as NULL).
int prep_build(const void* q_raw, const void* k_raw, const void* v_raw, int raw_dtype,
               const float* conv_w, const float* ring_in, float* ring_out, const float* f_raw,
               const float* dt_bias, const float* a_log, int gate_mode, float gate_lb,
               const float* beta_raw, float* q_hat, float* k_hat, float* v_hat, float* g,
               float* beta, const SeqLayout& seq, int H, int D, int K, float l2_eps,
               bool planes, PrepArgs& a, int Hk = 0, int Hg = 0) {
    a = PrepArgs{};
    a.seq = seq;
    if (D != kHeadDim) return KDA_ERR_HEAD_DIM;
    if (seq.N < 0 || seq.N > kMaxGridY || seq.total_rows < 0 || H <= 0 || H > kMaxGridY)
        return KDA_ERR_SHAPE;
    if (Hg == 0) Hg = H;                      // H: 128-wide value sub-heads; Hg: value heads
    if (Hg < 1 || Hg > H || H % Hg != 0) return KDA_ERR_SHAPE;
    if (Hk == 0) Hk = Hg;
    if (Hk < 1 || Hk > Hg) return KDA_ERR_SHAPE;
    if (raw_dtype != KDA_DTYPE_F32 && raw_dtype != KDA_DTYPE_BF16) return KDA_ERR_ENUM;
    if (gate_mode < 0 || gate_mode > (KDA_GATE_PER_HEAD | KDA_GATE_EXP)) return KDA_ERR_ENUM;
    if (conv_w != nullptr && (K < 2 || K > kMaxConvK)) return KDA_ERR_CONV_K;
    if (seq.N == 0) return KDA_OK;
    if (conv_w != nullptr && (ring_in == nullptr || ring_out == nullptr)) return KDA_ERR_NULL;
    if (seq.total_rows > 0) {
        if (!q_raw || !k_raw || !v_raw || !f_raw || !dt_bias || !a_log || !beta_raw)
            return KDA_ERR_NULL;
        if (planes && (!q_hat || !k_hat || !v_hat || !g || !beta)) return KDA_ERR_NULL;
        if (planes && (!aligned16(q_hat) || !aligned16(k_hat) || !aligned16(v_hat) || !aligned16(g)))
            return KDA_ERR_ALIGN;
        // raw rows are read 4 channels at a time: 8-byte bf16x4 or 16-byte f32x4
        const uintptr_t rmask = raw_dtype == KDA_DTYPE_BF16 ? 7u : 15u;
        if (((reinterpret_cast<uintptr_t>(q_raw) | reinterpret_cast<uintptr_t>(k_raw) |
              reinterpret_cast<uintptr_t>(v_raw)) & rmask) != 0)
            return KDA_ERR_ALIGN;
        if ((gate_mode & KDA_GATE_PER_HEAD) == 0 && (!aligned16(f_raw) || !aligned16(dt_bias)))
            return KDA_ERR_ALIGN;
    }
    if (conv_w != nullptr && ring_in != ring_out) {
        const size_t rb = (size_t)seq.N * ring_channels(H, Hk) * (K - 1) * sizeof(float);
        if (overlap(ring_in, ring_out, rb)) return KDA_ERR_STATE_ALIAS;
    }
    a.Hk = Hk;
    a.q_raw = q_raw; a.k_raw = k_raw; a.v_raw = v_raw; a.raw_bf16 = raw_dtype == KDA_DTYPE_BF16;
    a.conv_w = conv_w; a.ring_in = ring_in; a.ring_out = ring_out;
    a.f_raw = f_raw; a.dt_bias = dt_bias; a.a_log = a_log; a.gate_mode = gate_mode;
    a.gate_lb = gate_lb; a.beta_raw = beta_raw;
    a.q_hat = q_hat; a.k_hat = k_hat; a.v_hat = v_hat; a.g = g; a.beta = beta;
    a.seq = seq; a.H = H; a.K = conv_w ? K : 1; a.l2_eps = l2_eps;
    a.Hk = Hk;
    a.Hg = Hg;
    return KDA_OK;
}

int prep_impl(const void* q_raw, const void* k_raw, const void* v_raw, int raw_dtype,
              const float* conv_w, const float* ring_in, float* ring_out, const float* f_raw,
              const float* dt_bias, const float* a_log, int gate_mode, float gate_lb,
              const float* beta_raw, float* q_hat, float* k_hat, float* v_hat, float* g,
              float* beta, const SeqLayout& seq, int H, int D, int K, float l2_eps,
              void* stream, int Hk = 0, int Hg = 0) {
    PrepArgs a;
    const int rc = prep_build(q_raw, k_raw, v_raw, raw_dtype, conv_w, ring_in, ring_out, f_raw,
                              dt_bias, a_log, gate_mode, gate_lb, beta_raw, q_hat, k_hat, v_hat,
                              g, beta, seq, H, D, K, l2_eps, true, a, Hk, Hg);
    if (rc != KDA_OK || seq.N == 0) return rc;
    if (const int sd = check_stream_device(stream)) return sd;
    return cuda_status(launch_prep(a, static_cast<cudaStream_t>(stream)));
}

// AUTO takes the chunked form when the longest sequence has at least kAutoChunkMinLen tokens, or
// at least kAutoChunkMinLenWide when there are kAutoWidePairs or more (sequence, head) pairs.
// Measured on GB300 (H = 64): one sequence crosses over at about 96 tokens, 16 or more sequences
// between 32 and 64 (the chunked form's margin below 64 is within the spread between boxes).
constexpr long kAutoChunkMinLen = 96;
constexpr long kAutoChunkMinLenWide = 64;
constexpr long kAutoWidePairs = 512;

long max_len(const SeqLayout& seq, const int* cu_host) {
    if (seq.cu_seqlens == nullptr) return seq.T_uniform;
    long m = 0;
    for (int n = 0; n < seq.N; ++n) m = cu_host[n + 1] - cu_host[n] > m ? cu_host[n + 1] - cu_host[n] : m;
    return m;
}

int scan_impl(const float* q, const float* k, const float* v, const float* g, int gate_mode,
              const float* beta, const float* state_in, float* state_out, float* o,
              const SeqLayout& seq, const int* cu_host, int H, int D, float scale, int algo,
              void* workspace, size_t workspace_bytes, void* stream, int Hk = 0, int vsub = 1) {
    if (D != kHeadDim) return KDA_ERR_HEAD_DIM;
    if (seq.N < 0 || seq.N > kMaxGridY || seq.total_rows < 0 || H <= 0) return KDA_ERR_SHAPE;
    if (vsub < 1 || H % vsub != 0) return KDA_ERR_SHAPE;
    if (Hk == 0) Hk = H / vsub;
    if (Hk < 1 || Hk > kMaxGridY) return KDA_ERR_SHAPE;
    if (gate_mode < 0 || gate_mode > (KDA_GATE_PER_HEAD | KDA_GATE_EXP)) return KDA_ERR_ENUM;
    if (algo != KDA_ALGO_AUTO && algo != KDA_ALGO_SEQ && algo != KDA_ALGO_CHUNK) return KDA_ERR_ENUM;
    if (seq.total_rows >= (1L << 31)) return KDA_ERR_SHAPE;
    if (seq.N == 0) return KDA_OK;
    if (!state_in || !state_out) return KDA_ERR_NULL;
    if (!aligned16(state_in) || !aligned16(state_out)) return KDA_ERR_ALIGN;
    const size_t sb = (size_t)seq.N * H * kHeadDim * kHeadDim * sizeof(float);
    if (overlap(state_in, state_out, sb)) return KDA_ERR_STATE_ALIAS;
    if (seq.total_rows > 0) {
        if (!q || !k || !v || !g || !beta || !o) return KDA_ERR_NULL;
        if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
            ((gate_mode & KDA_GATE_PER_HEAD) == 0 && !aligned16(g)))
            return KDA_ERR_ALIGN;
    }
    ScanArgs a{};
    a.Hk = Hk;
    a.vsub = vsub;
    a.q = q; a.k = k; a.v = v; a.g = g; a.gate_mode = gate_mode; a.beta = beta;
    a.state_in = state_in; a.state_out = state_out; a.o = o;
    a.seq = seq; a.H = H; a.scale = scale; a.order = nullptr;
    const size_t need = chunk_workspace_bytes(seq, cu_host, H);
    const bool ws_ok = workspace != nullptr && workspace_bytes >= need && aligned16(workspace);
    bool chunk = algo == KDA_ALGO_CHUNK;
    if (chunk && !ws_ok) return workspace && !aligned16(workspace) ? KDA_ERR_ALIGN : KDA_ERR_WORKSPACE;
    if (algo == KDA_ALGO_AUTO) {
        const long ml = max_len(seq, cu_host);
        const bool wide = (long)seq.N * H >= kAutoWidePairs;
        chunk = ws_ok && (ml >= kAutoChunkMinLen || (wide && ml >= kAutoChunkMinLenWide));
    }
    if (const int sd = check_stream_device(stream)) return sd;
    a.err = dev_err_ptr();  // null only if the symbol lookup failed: waits then report nothing
    return cuda_status(chunk ? launch_scan_chunk(a, cu_host, workspace, static_cast<cudaStream_t>(stream))
                             : launch_scan_seq(a, static_cast<cudaStream_t>(stream)));
}

// Byte offsets of the pieces of kda_prefill_fused's workspace: the scan's readout o (written only
// when the RMSNorm kernel reads it back: value heads wider than 128, or (sequence, head) chains
// on fewer than two thirds of the SMs; otherwise the chunk kernel normalises it as it leaves),
// then the chunked
// scan's scratch (the prepared q, k, v, g never leave the chunk kernel).
struct PrefillLayout {
    size_t o, chunk;
};

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

PrefillLayout prefill_layout(long rows, int H) {
    PrefillLayout L;
    L.o = 0;
    L.chunk = align256((size_t)rows * H * kHeadDim * sizeof(float));
    return L;
}

int prefill_impl(const void* q_raw, const void* k_raw, const void* v_raw, int raw_dtype,
                 const float* conv_w, const float* ring_in, float* ring_out, const float* f_raw,
                 const float* dt_bias, const float* a_log, int gate_mode, float gate_lb,
                 const float* beta_raw, const float* state_in, float* state_out,
                 const float* norm_w, const float* gate_raw, float* y, const SeqLayout& seq,
                 const int* cu_host, int H, int D, int K, float l2_eps, float scale,
                 float norm_eps, void* workspace, size_t workspace_bytes, void* stream,
                 int Hk = 0, int Hg = 0) {
    // H: 128-wide value units; Hg: value heads (H / Hg units each), 0 meaning H
    if (D != kHeadDim) return KDA_ERR_HEAD_DIM;
    if (seq.N < 0 || seq.N > kMaxGridY || seq.total_rows < 0 || H <= 0 || H > kMaxGridY)
        return KDA_ERR_SHAPE;
    if (seq.total_rows >= (1L << 31)) return KDA_ERR_SHAPE;
    const bool norm_silu = (gate_mode & KDA_NORM_SILU) != 0;
    gate_mode &= ~KDA_NORM_SILU;
    if (gate_mode != KDA_GATE_PER_CHANNEL && gate_mode != KDA_GATE_PER_HEAD) return KDA_ERR_ENUM;
    if (seq.N == 0) return KDA_OK;
    if (seq.total_rows > 0) {
        if (!norm_w || !gate_raw || !y) return KDA_ERR_NULL;
        if (!aligned16(norm_w) || !aligned16(gate_raw) || !aligned16(y)) return KDA_ERR_ALIGN;
    }
    PrepArgs pa;
    int rc = prep_build(q_raw, k_raw, v_raw, raw_dtype, conv_w, ring_in, ring_out, f_raw, dt_bias,
                        a_log, gate_mode, gate_lb, beta_raw, nullptr, nullptr, nullptr, nullptr,
                        nullptr, seq, H, D, K, l2_eps, false, pa, Hk, Hg);
    if (rc != KDA_OK) return rc;
    const int vsub = H / pa.Hg;                  // prep_build checked that Hg divides H
    // the fused kernel copies bf16 raw rows into shared memory 16 bytes at a time
    if (seq.total_rows > 0 && pa.raw_bf16 &&
        (!aligned16(q_raw) || !aligned16(k_raw) || !aligned16(v_raw)))
        return KDA_ERR_ALIGN;
    if (!state_in || !state_out) return KDA_ERR_NULL;
    if (!aligned16(state_in) || !aligned16(state_out)) return KDA_ERR_ALIGN;
    if (overlap(state_in, state_out, (size_t)seq.N * H * kHeadDim * kHeadDim * sizeof(float)))
        return KDA_ERR_STATE_ALIAS;
    const PrefillLayout L = prefill_layout(seq.total_rows, H);
    const size_t need = L.chunk + chunk_workspace_bytes(seq, cu_host, H);
    if (workspace == nullptr || workspace_bytes < need) return KDA_ERR_WORKSPACE;
    if (!aligned16(workspace)) return KDA_ERR_ALIGN;
    if (const int sd = check_stream_device(stream)) return sd;
    unsigned char* w = static_cast<unsigned char*>(workspace);
    float* oh = reinterpret_cast<float*>(w + L.o);
    ScanArgs a{};
    a.Hk = pa.Hk;
    a.vsub = vsub;
    a.gate_mode = gate_mode; a.state_in = state_in; a.state_out = state_out; a.o = oh;
    a.seq = seq; a.H = H; a.scale = scale; a.order = nullptr; a.err = dev_err_ptr();
    // 128-wide value heads and (sequence, head) chains on at least two thirds of the SMs: the
    // chunk kernel writes y itself (the RMSNorm of a row needs only that row; its ~200
    // instructions a row, spread over most SMs, cost less than the readout's round trip through
    // HBM; measured at full length: 64 chains on 152 SMs 6 % slower folded, 128 to 1,024 chains
    // 1-3 % faster but for 192, one wave and a small second, 1 % slower).  With fewer chains they
    // would lengthen each chain on the SMs it has, and value heads wider than 128 need the whole
    // row: there the RMSNorm kernel runs apart.
    bool fold_norm = false;
    if (vsub == 1) {
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
            fold_norm = sms > 0 && 3 * (long)seq.N * H >= 2L * sms;
    }
    if (fold_norm) {
        a.norm_w = norm_w; a.norm_z = gate_raw; a.norm_y = y; a.norm_eps = norm_eps;
        a.norm_silu = norm_silu ? 1 : 0;
    }
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    rc = cuda_status(launch_prefill_chunk(pa, a, cu_host, w + L.chunk, st));
    if (rc != KDA_OK || seq.total_rows == 0 || fold_norm) return rc;
    NormArgs na{oh, norm_w, gate_raw, y, seq.total_rows * pa.Hg, norm_eps, norm_silu ? 1 : 0,
                vsub * kHeadDim};
    return cuda_status(launch_gated_rmsnorm(na, static_cast<cudaStream_t>(stream)));
}

int norm_impl(const float* o, const float* norm_w, const float* gate_raw, float* y, long rows,
              int D, float eps, bool silu, void* stream) {
    // D: the value head width, a multiple of 128 up to kMaxValueWidth
    if (D <= 0 || D % kHeadDim != 0 || D > kMaxValueWidth) return KDA_ERR_HEAD_DIM;
    if (rows < 0) return KDA_ERR_SHAPE;
    if (rows == 0) return KDA_OK;
    if (!o || !norm_w || !gate_raw || !y) return KDA_ERR_NULL;
    if (!aligned16(o) || !aligned16(norm_w) || !aligned16(gate_raw) || !aligned16(y))
        return KDA_ERR_ALIGN;
    if (const int sd = check_stream_device(stream)) return sd;
    NormArgs a{o, norm_w, gate_raw, y, rows, eps, silu ? 1 : 0, D};
    return cuda_status(launch_gated_rmsnorm(a, static_cast<cudaStream_t>(stream)));
}

int decode_impl(const void* q_raw, const void* k_raw, const void* v_raw, int raw_dtype,
                const float* conv_w, const float* ring_in, float* ring_out, const float* f_raw,
                const float* dt_bias, const float* a_log, int gate_mode, float gate_lb,
                const float* beta_raw, const float* state_in, float* state_out,
                const float* norm_w, const float* gate_raw, float* y, int N, int T, int H, int D,
                int K, float l2_eps, float scale, float rms_eps, const int* keep, bool rollback,
                void* stream, int Hk = 0, int Hg = 0) {
    // H: 128-wide value units; Hg: value heads of H / Hg units each (0 meaning H)
    if (D != kHeadDim) return KDA_ERR_HEAD_DIM;
    if (N < 0 || N > kMaxGridY || H <= 0 || H > kMaxGridY || T < 1 || T > kDecodeMaxT)
        return KDA_ERR_SHAPE;
    if (Hg == 0) Hg = H;
    if (Hg < 1 || Hg > H || H % Hg != 0 || H / Hg > kMaxValueWidth / kHeadDim)
        return KDA_ERR_SHAPE;
    if (Hk == 0) Hk = Hg;
    if (Hk < 1 || Hk > Hg) return KDA_ERR_SHAPE;
    if ((long)N * H >= (1L << 31)) return KDA_ERR_SHAPE;
    if (raw_dtype != KDA_DTYPE_F32 && raw_dtype != KDA_DTYPE_BF16) return KDA_ERR_ENUM;
    const bool norm_silu = (gate_mode & KDA_NORM_SILU) != 0;
    gate_mode &= ~KDA_NORM_SILU;
    if (gate_mode != KDA_GATE_PER_CHANNEL && gate_mode != KDA_GATE_PER_HEAD) return KDA_ERR_ENUM;
    if (K < 2 || K > kMaxConvK) return KDA_ERR_CONV_K;
    if (N == 0) return KDA_OK;
    if (!q_raw || !k_raw || !v_raw || !conv_w || !ring_in || !ring_out || !f_raw || !dt_bias ||
        !a_log || !beta_raw || !state_in || !state_out || !norm_w || !gate_raw || !y)
        return KDA_ERR_NULL;
    if (!aligned16(state_in) || !aligned16(state_out) || !aligned16(norm_w) ||
        !aligned16(gate_raw) || !aligned16(y))
        return KDA_ERR_ALIGN;
    const size_t sb = (size_t)N * H * kHeadDim * kHeadDim * sizeof(float);
    // in place (state_out == state_in) is allowed: every thread loads its part of its (sequence,
    // head) block before it stores the same elements; a partial overlap is not
    if (state_in != state_out && overlap(state_in, state_out, sb)) return KDA_ERR_STATE_ALIAS;
    if (ring_in != ring_out) {
        const size_t rb = (size_t)N * ring_channels(H, Hk) * (K - 1) * sizeof(float);
        if (overlap(ring_in, ring_out, rb)) return KDA_ERR_STATE_ALIAS;
    } else if (Hk < H) {
        // grouped queries or value heads of several units: several units read one q/k ring row
        // that only one of them rewrites, so the ring cannot be rolled in place
        return KDA_ERR_STATE_ALIAS;
    }
    DecodeArgs a{};
    a.Hk = Hk;
    a.vsub = H / Hg;
    a.q_raw = q_raw; a.k_raw = k_raw; a.v_raw = v_raw; a.raw_bf16 = raw_dtype == KDA_DTYPE_BF16;
    a.conv_w = conv_w; a.ring_in = ring_in; a.ring_out = ring_out;
    a.f_raw = f_raw; a.dt_bias = dt_bias; a.a_log = a_log; a.gate_mode = gate_mode;
    a.gate_lb = gate_lb; a.beta_raw = beta_raw; a.state_in = state_in; a.state_out = state_out;
    a.norm_w = norm_w; a.gate_raw = gate_raw; a.y = y;
    a.N = N; a.T = T; a.H = H; a.K = K; a.l2_eps = l2_eps; a.scale = scale; a.rms_eps = rms_eps;
    if (rollback && keep == nullptr) return KDA_ERR_NULL;
    a.keep = keep;
    a.norm_silu = norm_silu ? 1 : 0;
    if (const int sd = check_stream_device(stream)) return sd;
    a.err = dev_err_ptr();
    return cuda_status(launch_decode_fused(a, static_cast<cudaStream_t>(stream)));
}


}  // namespace

extern "C" {

int kda_abi_version(void) { return 1; }

const char* kda_status_string(int s) {
    switch (s) {
        case KDA_OK: return "ok";
        case KDA_ERR_HEAD_DIM: return "head_dim must be 128";
        case KDA_ERR_CONV_K: return "conv kernel width K must be in 2..8";
        case KDA_ERR_STATE_ALIAS: return "state_in/state_out (or ring_in/ring_out) overlap";
        case KDA_ERR_NULL: return "a required pointer is NULL";
        case KDA_ERR_SHAPE: return "bad shape (negative size, H == 0, or T out of range)";
        case KDA_ERR_CU_SEQLENS: return "bad cu_seqlens (must start at 0, not decrease, end at total_T)";
        case KDA_ERR_ENUM: return "unknown raw_dtype, gate_mode or algo";
        case KDA_ERR_TIMEOUT: return "a kernel gave up a bounded device wait";
        case KDA_ERR_WORKSPACE: return "workspace missing or too small";
        case KDA_ERR_ALIGN: return "a pointer that must be 16-byte aligned is not";
        case KDA_ERR_SCRATCH_LIMIT:
            return "the chunked scratch this call needs exceeds KDA_STATIC_SCRATCH_BYTES";
        case KDA_ERR_STREAM_DEVICE:
            return "the stream belongs to a device other than the current one";
        default:
            if (s >= KDA_ERR_CUDA_BASE && s < KDA_ERR_CUDA_BASE + 10000) return "CUDA error";
            return "unknown status";
    }
}

int kda_conv_l2norm_prep(const void* q_raw, const void* k_raw, const void* v_raw, int raw_dtype,
                         const float* conv_w, const float* ring_in, float* ring_out,
                         const float* f_raw, const float* dt_bias, const float* a_log,
                         int gate_mode, float gate_lb, const float* beta_raw, float* q_hat,
                         float* k_hat, float* v_hat, float* g, float* beta, int N, int T, int H,
                         int D, int K, float l2_eps, void* stream) {
    if (N < 0 || T < 0) return KDA_ERR_SHAPE;
    SeqLayout seq{nullptr, T, N, (long)N * T};
    if (T == 0 && N > 0) seq.T_uniform = 0;
    return prep_impl(q_raw, k_raw, v_raw, raw_dtype, conv_w, ring_in, ring_out, f_raw, dt_bias,
                     a_log, gate_mode, gate_lb, beta_raw, q_hat, k_hat, v_hat, g, beta, seq, H,
                     D, K, l2_eps, stream);
}

int kda_conv_l2norm_prep_varlen(const void* q_raw, const void* k_raw, const void* v_raw,
                                int raw_dtype, const float* conv_w, const float* ring_in,
                                float* ring_out, const float* f_raw, const float* dt_bias,
                                const float* a_log, int gate_mode, float gate_lb,
                                const float* beta_raw, float* q_hat, float* k_hat, float* v_hat,
                                float* g, float* beta, const int* cu_seqlens,
                                const int* cu_seqlens_host, int N, int total_T, int H, int D,
                                int K, float l2_eps, void* stream) {
    if (N < 0 || total_T < 0) return KDA_ERR_SHAPE;
    if (N > 0) {
        if (cu_seqlens == nullptr) return KDA_ERR_NULL;
        const int rc = check_cu(cu_seqlens_host, N, total_T);
        if (rc) return rc;
    }
    SeqLayout seq{cu_seqlens, 0, N, (long)total_T};
    return prep_impl(q_raw, k_raw, v_raw, raw_dtype, conv_w, ring_in, ring_out, f_raw, dt_bias,
                     a_log, gate_mode, gate_lb, beta_raw, q_hat, k_hat, v_hat, g, beta, seq, H,
                     D, K, l2_eps, stream);
}

size_t kda_scan_workspace_bytes(int N, int total_T, int H, int D, int gate_mode, int algo) {
    (void)gate_mode;
    if (N < 0 || total_T < 0 || H <= 0 || D != kHeadDim) return 0;
    if (algo == KDA_ALGO_SEQ) return 0;
    // every sequence contributes ceil(L / kChunkTokens) chunks <= L / kChunkTokens + 1, plus the
    // varlen header of chunk offsets
    const size_t chunks = (size_t)(total_T + kChunkTokens - 1) / kChunkTokens + (size_t)N;
    const size_t header = (((size_t)N + 1) * 4 + 255) / 256 * 256;
    return header + chunks * (size_t)H * kChunkBlockBytes;
}

size_t kda_prefill_workspace_bytes(int N, int total_T, int H, int D, int gate_mode) {
    if (N < 0 || total_T < 0 || H <= 0 || D != kHeadDim) return 0;
    gate_mode &= ~KDA_NORM_SILU;
    if (gate_mode != KDA_GATE_PER_CHANNEL && gate_mode != KDA_GATE_PER_HEAD) return 0;
    return prefill_layout(total_T, H).chunk +
           kda_scan_workspace_bytes(N, total_T, H, D, gate_mode, KDA_ALGO_CHUNK);
}

int kda_prefill_fused(const void* q_raw, const void* k_raw, const void* v_raw, int raw_dtype,
                      const float* conv_w, const float* ring_in, float* ring_out,
                      const float* f_raw, const float* dt_bias, const float* a_log, int gate_mode,
                      float gate_lb, const float* beta_raw, const float* state_in,
                      float* state_out, const float* norm_w, const float* gate_raw, float* y,
                      int N, int T, int H, int D, int K, float l2_eps, float scale,
                      float rms_eps, void* workspace, size_t workspace_bytes, void* stream) {
    if (N < 0 || T < 0) return KDA_ERR_SHAPE;
    SeqLayout seq{nullptr, T, N, (long)N * T};
    return prefill_impl(q_raw, k_raw, v_raw, raw_dtype, conv_w, ring_in, ring_out, f_raw, dt_bias,
                        a_log, gate_mode, gate_lb, beta_raw, state_in, state_out, norm_w, gate_raw,
                        y, seq, nullptr, H, D, K, l2_eps, scale, rms_eps, workspace,
                        workspace_bytes, stream);
}

int kda_prefill_fused_varlen(const void* q_raw, const void* k_raw, const void* v_raw,
                             int raw_dtype, const float* conv_w, const float* ring_in,
                             float* ring_out, const float* f_raw, const float* dt_bias,
                             const float* a_log, int gate_mode, float gate_lb,
                             const float* beta_raw, const float* state_in, float* state_out,
                             const float* norm_w, const float* gate_raw, float* y,
                             const int* cu_seqlens, const int* cu_seqlens_host, int N,
                             int total_T, int H, int D, int K, float l2_eps, float scale,
                             float rms_eps, void* workspace, size_t workspace_bytes,
                             void* stream) {
    if (N < 0 || total_T < 0) return KDA_ERR_SHAPE;
    if (N > 0) {
        if (cu_seqlens == nullptr) return KDA_ERR_NULL;
        const int rc = check_cu(cu_seqlens_host, N, total_T);
        if (rc) return rc;
    }
    SeqLayout seq{cu_seqlens, 0, N, (long)total_T};
    return prefill_impl(q_raw, k_raw, v_raw, raw_dtype, conv_w, ring_in, ring_out, f_raw, dt_bias,
                        a_log, gate_mode, gate_lb, beta_raw, state_in, state_out, norm_w, gate_raw,
                        y, seq, cu_seqlens_host, H, D, K, l2_eps, scale, rms_eps, workspace,
                        workspace_bytes, stream);
}

int kda_scan(const float* q_hat, const float* k_hat, const float* v_hat, const float* g,
             int gate_mode, const float* beta, const float* state_in, float* state_out,
             float* o, int N, int T, int H, int D, float scale, int algo, void* workspace,
             size_t workspace_bytes, void* stream) {
    if (N < 0 || T < 0) return KDA_ERR_SHAPE;
    SeqLayout seq{nullptr, T, N, (long)N * T};
    return scan_impl(q_hat, k_hat, v_hat, g, gate_mode, beta, state_in, state_out, o, seq, nullptr,
                     H, D, scale, algo, workspace, workspace_bytes, stream);
}

int kda_scan_varlen(const float* q_hat, const float* k_hat, const float* v_hat, const float* g,
                    int gate_mode, const float* beta, const float* state_in, float* state_out,
                    float* o, const int* cu_seqlens, const int* cu_seqlens_host, int N,
                    int total_T, int H, int D, float scale, int algo, void* workspace,
                    size_t workspace_bytes, void* stream) {
    if (N < 0 || total_T < 0) return KDA_ERR_SHAPE;
    if (N > 0) {
        if (cu_seqlens == nullptr) return KDA_ERR_NULL;
        const int rc = check_cu(cu_seqlens_host, N, total_T);
        if (rc) return rc;
    }
    SeqLayout seq{cu_seqlens, 0, N, (long)total_T};
    return scan_impl(q_hat, k_hat, v_hat, g, gate_mode, beta, state_in, state_out, o, seq,
                     cu_seqlens_host, H, D, scale, algo, workspace, workspace_bytes, stream);
}

int kda_scan_gqa(const float* q_hat, const float* k_hat, const float* v_hat, const float* g,
                 int gate_mode, const float* beta, const float* state_in, float* state_out,
                 float* o, int N, int T, int H, int Hk, int D, float scale, int algo,
                 void* workspace, size_t workspace_bytes, void* stream) {
    if (N < 0 || T < 0 || Hk <= 0) return KDA_ERR_SHAPE;
    SeqLayout seq{nullptr, T, N, (long)N * T};
    return scan_impl(q_hat, k_hat, v_hat, g, gate_mode, beta, state_in, state_out, o, seq, nullptr,
                     H, D, scale, algo, workspace, workspace_bytes, stream, Hk);
}

int kda_scan_varlen_gqa(const float* q_hat, const float* k_hat, const float* v_hat,
                        const float* g, int gate_mode, const float* beta, const float* state_in,
                        float* state_out, float* o, const int* cu_seqlens,
                        const int* cu_seqlens_host, int N, int total_T, int H, int Hk, int D,
                        float scale, int algo, void* workspace, size_t workspace_bytes,
                        void* stream) {
    if (N < 0 || total_T < 0 || Hk <= 0) return KDA_ERR_SHAPE;
    if (N > 0) {
        if (cu_seqlens == nullptr) return KDA_ERR_NULL;
        const int rc = check_cu(cu_seqlens_host, N, total_T);
        if (rc) return rc;
    }
    SeqLayout seq{cu_seqlens, 0, N, (long)total_T};
    return scan_impl(q_hat, k_hat, v_hat, g, gate_mode, beta, state_in, state_out, o, seq,
                     cu_seqlens_host, H, D, scale, algo, workspace, workspace_bytes, stream, Hk);
}

int kda_gated_rmsnorm_out(const float* o, const float* norm_w, const float* gate_raw, float* y,
                          long rows, int D, float eps, void* stream) {
    return norm_impl(o, norm_w, gate_raw, y, rows, D, eps, false, stream);
}

int kda_gated_rmsnorm_silu_out(const float* o, const float* norm_w, const float* gate_raw,
                               float* y, long rows, int D, float eps, void* stream) {
    return norm_impl(o, norm_w, gate_raw, y, rows, D, eps, true, stream);
}


int kda_decode_fused(const void* q_raw, const void* k_raw, const void* v_raw, int raw_dtype,
                     const float* conv_w, const float* ring_in, float* ring_out,
                     const float* f_raw, const float* dt_bias, const float* a_log, int gate_mode,
                     float gate_lb, const float* beta_raw, const float* state_in,
                     float* state_out, const float* norm_w, const float* gate_raw, float* y,
                     int N, int T, int H, int D, int K, float l2_eps, float scale, float rms_eps,
                     void* stream) {
    return decode_impl(q_raw, k_raw, v_raw, raw_dtype, conv_w, ring_in, ring_out, f_raw, dt_bias,
                       a_log, gate_mode, gate_lb, beta_raw, state_in, state_out, norm_w, gate_raw,
                       y, N, T, H, D, K, l2_eps, scale, rms_eps, nullptr, false, stream);
}

int kda_verify_rollback(const void* q_raw, const void* k_raw, const void* v_raw, int raw_dtype,
                        const float* conv_w, const float* ring_in, float* ring_out,
                        const float* f_raw, const float* dt_bias, const float* a_log,
                        int gate_mode, float gate_lb, const float* beta_raw,
                        const float* state_in, float* state_out, const float* norm_w,
                        const float* gate_raw, float* y, const int* keep, int N, int T, int H,
                        int D, int K, float l2_eps, float scale, float rms_eps, void* stream) {
    return decode_impl(q_raw, k_raw, v_raw, raw_dtype, conv_w, ring_in, ring_out, f_raw, dt_bias,
                       a_log, gate_mode, gate_lb, beta_raw, state_in, state_out, norm_w, gate_raw,
                       y, N, T, H, D, K, l2_eps, scale, rms_eps, keep, true, stream);
}

int kda_conv_l2norm_prep_gqa(const void* q_raw, const void* k_raw, const void* v_raw,
                             int raw_dtype, const float* conv_w, const float* ring_in,
                             float* ring_out, const float* f_raw, const float* dt_bias,
                             const float* a_log, int gate_mode, float gate_lb,
                             const float* beta_raw, float* q_hat, float* k_hat, float* v_hat,
                             float* g, float* beta, int N, int T, int H, int Hk, int D, int K,
                             float l2_eps, void* stream) {
    if (N < 0 || T < 0 || Hk <= 0) return KDA_ERR_SHAPE;
    SeqLayout seq{nullptr, T, N, (long)N * T};
    return prep_impl(q_raw, k_raw, v_raw, raw_dtype, conv_w, ring_in, ring_out, f_raw, dt_bias,
                     a_log, gate_mode, gate_lb, beta_raw, q_hat, k_hat, v_hat, g, beta, seq, H,
                     D, K, l2_eps, stream, Hk);
}

int kda_conv_l2norm_prep_varlen_gqa(const void* q_raw, const void* k_raw, const void* v_raw,
                                    int raw_dtype, const float* conv_w, const float* ring_in,
                                    float* ring_out, const float* f_raw, const float* dt_bias,
                                    const float* a_log, int gate_mode, float gate_lb,
                                    const float* beta_raw, float* q_hat, float* k_hat,
                                    float* v_hat, float* g, float* beta, const int* cu_seqlens,
                                    const int* cu_seqlens_host, int N, int total_T, int H,
                                    int Hk, int D, int K, float l2_eps, void* stream) {
    if (N < 0 || total_T < 0 || Hk <= 0) return KDA_ERR_SHAPE;
    if (N > 0) {
        if (cu_seqlens == nullptr) return KDA_ERR_NULL;
        const int rc = check_cu(cu_seqlens_host, N, total_T);
        if (rc) return rc;
    }
    SeqLayout seq{cu_seqlens, 0, N, (long)total_T};
    return prep_impl(q_raw, k_raw, v_raw, raw_dtype, conv_w, ring_in, ring_out, f_raw, dt_bias,
                     a_log, gate_mode, gate_lb, beta_raw, q_hat, k_hat, v_hat, g, beta, seq, H,
                     D, K, l2_eps, stream, Hk);
}

int kda_prefill_fused_gqa(const void* q_raw, const void* k_raw, const void* v_raw, int raw_dtype,
                          const float* conv_w, const float* ring_in, float* ring_out,
                          const float* f_raw, const float* dt_bias, const float* a_log,
                          int gate_mode, float gate_lb, const float* beta_raw,
                          const float* state_in, float* state_out, const float* norm_w,
                          const float* gate_raw, float* y, int N, int T, int H, int Hk, int D,
                          int K, float l2_eps, float scale, float rms_eps, void* workspace,
                          size_t workspace_bytes, void* stream) {
    if (N < 0 || T < 0 || Hk <= 0) return KDA_ERR_SHAPE;
    SeqLayout seq{nullptr, T, N, (long)N * T};
    return prefill_impl(q_raw, k_raw, v_raw, raw_dtype, conv_w, ring_in, ring_out, f_raw, dt_bias,
                        a_log, gate_mode, gate_lb, beta_raw, state_in, state_out, norm_w, gate_raw,
                        y, seq, nullptr, H, D, K, l2_eps, scale, rms_eps, workspace,
                        workspace_bytes, stream, Hk);
}

int kda_prefill_fused_varlen_gqa(const void* q_raw, const void* k_raw, const void* v_raw,
                                 int raw_dtype, const float* conv_w, const float* ring_in,
                                 float* ring_out, const float* f_raw, const float* dt_bias,
                                 const float* a_log, int gate_mode, float gate_lb,
                                 const float* beta_raw, const float* state_in, float* state_out,
                                 const float* norm_w, const float* gate_raw, float* y,
                                 const int* cu_seqlens, const int* cu_seqlens_host, int N,
                                 int total_T, int H, int Hk, int D, int K, float l2_eps,
                                 float scale, float rms_eps, void* workspace,
                                 size_t workspace_bytes, void* stream) {
    if (N < 0 || total_T < 0 || Hk <= 0) return KDA_ERR_SHAPE;
    if (N > 0) {
        if (cu_seqlens == nullptr) return KDA_ERR_NULL;
        const int rc = check_cu(cu_seqlens_host, N, total_T);
        if (rc) return rc;
    }
    SeqLayout seq{cu_seqlens, 0, N, (long)total_T};
    return prefill_impl(q_raw, k_raw, v_raw, raw_dtype, conv_w, ring_in, ring_out, f_raw, dt_bias,
                        a_log, gate_mode, gate_lb, beta_raw, state_in, state_out, norm_w, gate_raw,
                        y, seq, cu_seqlens_host, H, D, K, l2_eps, scale, rms_eps, workspace,
                        workspace_bytes, stream, Hk);
}

int kda_decode_fused_gqa(const void* q_raw, const void* k_raw, const void* v_raw, int raw_dtype,
                         const float* conv_w, const float* ring_in, float* ring_out,
                         const float* f_raw, const float* dt_bias, const float* a_log,
                         int gate_mode, float gate_lb, const float* beta_raw,
                         const float* state_in, float* state_out, const float* norm_w,
                         const float* gate_raw, float* y, int N, int T, int H, int Hk, int D, int K,
                         float l2_eps, float scale, float rms_eps, void* stream) {
    if (Hk <= 0) return KDA_ERR_SHAPE;
    return decode_impl(q_raw, k_raw, v_raw, raw_dtype, conv_w, ring_in, ring_out, f_raw, dt_bias,
                       a_log, gate_mode, gate_lb, beta_raw, state_in, state_out, norm_w, gate_raw,
                       y, N, T, H, D, K, l2_eps, scale, rms_eps, nullptr, false, stream, Hk);
}

int kda_verify_rollback_gqa(const void* q_raw, const void* k_raw, const void* v_raw,
                            int raw_dtype, const float* conv_w, const float* ring_in,
                            float* ring_out, const float* f_raw, const float* dt_bias,
                            const float* a_log, int gate_mode, float gate_lb,
                            const float* beta_raw, const float* state_in, float* state_out,
                            const float* norm_w, const float* gate_raw, float* y, const int* keep,
                            int N, int T, int H, int Hk, int D, int K, float l2_eps, float scale,
                            float rms_eps, void* stream) {
    if (Hk <= 0) return KDA_ERR_SHAPE;
    return decode_impl(q_raw, k_raw, v_raw, raw_dtype, conv_w, ring_in, ring_out, f_raw, dt_bias,
                       a_log, gate_mode, gate_lb, beta_raw, state_in, state_out, norm_w, gate_raw,
                       y, N, T, H, D, K, l2_eps, scale, rms_eps, keep, true, stream, Hk);
}

// a value head width Dv = m * 128 (m = 1..8) with a key width of 128: the number of 128-wide
// value sub-heads, or 0 for a width that is not built
static int value_subheads(int Dk, int Dv) {
    if (Dk != kHeadDim || Dv <= 0 || Dv % kHeadDim != 0 || Dv > kMaxValueWidth) return 0;
    return Dv / kHeadDim;
}

int kda_conv_l2norm_prep_dv(const void* q_raw, const void* k_raw, const void* v_raw,
                            int raw_dtype, const float* conv_w, const float* ring_in,
                            float* ring_out, const float* f_raw, const float* dt_bias,
                            const float* a_log, int gate_mode, float gate_lb,
                            const float* beta_raw, float* q_hat, float* k_hat, float* v_hat,
                            float* g, float* beta, int N, int T, int H, int Hk, int Dk, int Dv,
                            int K, float l2_eps, void* stream) {
    const int m = value_subheads(Dk, Dv);
    if (m == 0) return KDA_ERR_HEAD_DIM;
    if (N < 0 || T < 0 || H <= 0 || Hk <= 0 || Hk > H || (long)H * m > kMaxGridY) return KDA_ERR_SHAPE;
    SeqLayout seq{nullptr, T, N, (long)N * T};
    return prep_impl(q_raw, k_raw, v_raw, raw_dtype, conv_w, ring_in, ring_out, f_raw, dt_bias,
                     a_log, gate_mode, gate_lb, beta_raw, q_hat, k_hat, v_hat, g, beta, seq,
                     H * m, kHeadDim, K, l2_eps, stream, Hk, H);
}

int kda_conv_l2norm_prep_varlen_dv(const void* q_raw, const void* k_raw, const void* v_raw,
                                   int raw_dtype, const float* conv_w, const float* ring_in,
                                   float* ring_out, const float* f_raw, const float* dt_bias,
                                   const float* a_log, int gate_mode, float gate_lb,
                                   const float* beta_raw, float* q_hat, float* k_hat,
                                   float* v_hat, float* g, float* beta, const int* cu_seqlens,
                                   const int* cu_seqlens_host, int N, int total_T, int H, int Hk,
                                   int Dk, int Dv, int K, float l2_eps, void* stream) {
    const int m = value_subheads(Dk, Dv);
    if (m == 0) return KDA_ERR_HEAD_DIM;
    if (N < 0 || total_T < 0 || H <= 0 || Hk <= 0 || Hk > H || (long)H * m > kMaxGridY)
        return KDA_ERR_SHAPE;
    if (N > 0) {
        if (cu_seqlens == nullptr) return KDA_ERR_NULL;
        const int rc = check_cu(cu_seqlens_host, N, total_T);
        if (rc) return rc;
    }
    SeqLayout seq{cu_seqlens, 0, N, (long)total_T};
    return prep_impl(q_raw, k_raw, v_raw, raw_dtype, conv_w, ring_in, ring_out, f_raw, dt_bias,
                     a_log, gate_mode, gate_lb, beta_raw, q_hat, k_hat, v_hat, g, beta, seq,
                     H * m, kHeadDim, K, l2_eps, stream, Hk, H);
}

int kda_scan_dv(const float* q_hat, const float* k_hat, const float* v_hat, const float* g,
                int gate_mode, const float* beta, const float* state_in, float* state_out,
                float* o, int N, int T, int H, int Hk, int Dk, int Dv, float scale, int algo,
                void* workspace, size_t workspace_bytes, void* stream) {
    const int m = value_subheads(Dk, Dv);
    if (m == 0) return KDA_ERR_HEAD_DIM;
    if (N < 0 || T < 0 || H <= 0 || Hk <= 0 || Hk > H || (long)H * m > kMaxGridY) return KDA_ERR_SHAPE;
    SeqLayout seq{nullptr, T, N, (long)N * T};
    return scan_impl(q_hat, k_hat, v_hat, g, gate_mode, beta, state_in, state_out, o, seq,
                     nullptr, H * m, kHeadDim, scale, algo, workspace, workspace_bytes, stream, Hk,
                     m);
}

int kda_scan_varlen_dv(const float* q_hat, const float* k_hat, const float* v_hat,
                       const float* g, int gate_mode, const float* beta, const float* state_in,
                       float* state_out, float* o, const int* cu_seqlens,
                       const int* cu_seqlens_host, int N, int total_T, int H, int Hk, int Dk,
                       int Dv, float scale, int algo, void* workspace, size_t workspace_bytes,
                       void* stream) {
    const int m = value_subheads(Dk, Dv);
    if (m == 0) return KDA_ERR_HEAD_DIM;
    if (N < 0 || total_T < 0 || H <= 0 || Hk <= 0 || Hk > H || (long)H * m > kMaxGridY)
        return KDA_ERR_SHAPE;
    if (N > 0) {
        if (cu_seqlens == nullptr) return KDA_ERR_NULL;
        const int rc = check_cu(cu_seqlens_host, N, total_T);
        if (rc) return rc;
    }
    SeqLayout seq{cu_seqlens, 0, N, (long)total_T};
    return scan_impl(q_hat, k_hat, v_hat, g, gate_mode, beta, state_in, state_out, o, seq,
                     cu_seqlens_host, H * m, kHeadDim, scale, algo, workspace, workspace_bytes,
                     stream, Hk, m);
}

int kda_prefill_fused_dv(const void* q_raw, const void* k_raw, const void* v_raw, int raw_dtype,
                         const float* conv_w, const float* ring_in, float* ring_out,
                         const float* f_raw, const float* dt_bias, const float* a_log,
                         int gate_mode, float gate_lb, const float* beta_raw,
                         const float* state_in, float* state_out, const float* norm_w,
                         const float* gate_raw, float* y, int N, int T, int H, int Hk, int Dk,
                         int Dv, int K, float l2_eps, float scale, float rms_eps, void* workspace,
                         size_t workspace_bytes, void* stream) {
    const int m = value_subheads(Dk, Dv);
    if (m == 0) return KDA_ERR_HEAD_DIM;
    if (N < 0 || T < 0 || H <= 0 || Hk <= 0 || Hk > H || (long)H * m > kMaxGridY)
        return KDA_ERR_SHAPE;
    SeqLayout seq{nullptr, T, N, (long)N * T};
    return prefill_impl(q_raw, k_raw, v_raw, raw_dtype, conv_w, ring_in, ring_out, f_raw, dt_bias,
                        a_log, gate_mode, gate_lb, beta_raw, state_in, state_out, norm_w, gate_raw,
                        y, seq, nullptr, H * m, kHeadDim, K, l2_eps, scale, rms_eps, workspace,
                        workspace_bytes, stream, Hk, H);
}

int kda_prefill_fused_varlen_dv(const void* q_raw, const void* k_raw, const void* v_raw,
                                int raw_dtype, const float* conv_w, const float* ring_in,
                                float* ring_out, const float* f_raw, const float* dt_bias,
                                const float* a_log, int gate_mode, float gate_lb,
                                const float* beta_raw, const float* state_in, float* state_out,
                                const float* norm_w, const float* gate_raw, float* y,
                                const int* cu_seqlens, const int* cu_seqlens_host, int N,
                                int total_T, int H, int Hk, int Dk, int Dv, int K, float l2_eps,
                                float scale, float rms_eps, void* workspace,
                                size_t workspace_bytes, void* stream) {
    const int m = value_subheads(Dk, Dv);
    if (m == 0) return KDA_ERR_HEAD_DIM;
    if (N < 0 || total_T < 0 || H <= 0 || Hk <= 0 || Hk > H || (long)H * m > kMaxGridY)
        return KDA_ERR_SHAPE;
    if (N > 0) {
        if (cu_seqlens == nullptr) return KDA_ERR_NULL;
        const int rc = check_cu(cu_seqlens_host, N, total_T);
        if (rc) return rc;
    }
    SeqLayout seq{cu_seqlens, 0, N, (long)total_T};
    return prefill_impl(q_raw, k_raw, v_raw, raw_dtype, conv_w, ring_in, ring_out, f_raw, dt_bias,
                        a_log, gate_mode, gate_lb, beta_raw, state_in, state_out, norm_w, gate_raw,
                        y, seq, cu_seqlens_host, H * m, kHeadDim, K, l2_eps, scale, rms_eps,
                        workspace, workspace_bytes, stream, Hk, H);
}

int kda_decode_fused_dv(const void* q_raw, const void* k_raw, const void* v_raw, int raw_dtype,
                        const float* conv_w, const float* ring_in, float* ring_out,
                        const float* f_raw, const float* dt_bias, const float* a_log,
                        int gate_mode, float gate_lb, const float* beta_raw,
                        const float* state_in, float* state_out, const float* norm_w,
                        const float* gate_raw, float* y, int N, int T, int H, int Hk, int Dk,
                        int Dv, int K, float l2_eps, float scale, float rms_eps, void* stream) {
    const int m = value_subheads(Dk, Dv);
    if (m == 0) return KDA_ERR_HEAD_DIM;
    if (H <= 0 || Hk <= 0 || Hk > H || (long)H * m > kMaxGridY) return KDA_ERR_SHAPE;
    return decode_impl(q_raw, k_raw, v_raw, raw_dtype, conv_w, ring_in, ring_out, f_raw, dt_bias,
                       a_log, gate_mode, gate_lb, beta_raw, state_in, state_out, norm_w, gate_raw,
                       y, N, T, H * m, kHeadDim, K, l2_eps, scale, rms_eps, nullptr, false, stream,
                       Hk, H);
}

int kda_verify_rollback_dv(const void* q_raw, const void* k_raw, const void* v_raw,
                           int raw_dtype, const float* conv_w, const float* ring_in,
                           float* ring_out, const float* f_raw, const float* dt_bias,
                           const float* a_log, int gate_mode, float gate_lb,
                           const float* beta_raw, const float* state_in, float* state_out,
                           const float* norm_w, const float* gate_raw, float* y, const int* keep,
                           int N, int T, int H, int Hk, int Dk, int Dv, int K, float l2_eps,
                           float scale, float rms_eps, void* stream) {
    const int m = value_subheads(Dk, Dv);
    if (m == 0) return KDA_ERR_HEAD_DIM;
    if (H <= 0 || Hk <= 0 || Hk > H || (long)H * m > kMaxGridY) return KDA_ERR_SHAPE;
    return decode_impl(q_raw, k_raw, v_raw, raw_dtype, conv_w, ring_in, ring_out, f_raw, dt_bias,
                       a_log, gate_mode, gate_lb, beta_raw, state_in, state_out, norm_w, gate_raw,
                       y, N, T, H * m, kHeadDim, K, l2_eps, scale, rms_eps, keep, true, stream,
                       Hk, H);
}

int kda_selftest_wait_timeout(void* stream) {
    if (const int sd = check_stream_device(stream)) return sd;
    int* p = dev_err_ptr();
    if (p == nullptr) return cuda_status(cudaErrorUnknown);
    return cuda_status(launch_wait_selftest(p, static_cast<cudaStream_t>(stream)));
}

int kda_device_status(void* stream) {
    if (const int sd = check_stream_device(stream)) return sd;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_status(e);
    int* p = dev_err_ptr();
    if (p == nullptr) return cuda_status(cudaErrorUnknown);
    int v = 0;
    e = cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_status(e);
    if (v != 0) {
        const int zero = 0;
        e = cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_status(e);
        return KDA_ERR_TIMEOUT;
    }
    return KDA_OK;
}

size_t kda_proj6_workspace_bytes(int t, int in_f) {
    if (t < 1 || t > kProjMaxT || in_f <= 0 || in_f % kProjKAlign != 0) return 0;
    return proj_workspace_bytes(t, in_f);
}

int kda_proj6(const float* x, int t, int in_f, const void* w_q, const void* w_k, const void* w_v,
              const void* w_fa, const void* w_ga, const void* w_b, float* q_raw, float* k_raw,
              float* v_raw, float* f_down, float* g_down, float* beta_raw, int H, int D,
              void* workspace, size_t workspace_bytes, void* stream) {
    if (D != kHeadDim) return KDA_ERR_HEAD_DIM;
    if (t < 1 || t > kProjMaxT || H <= 0 || H > kMaxGridY || in_f <= 0 ||
        in_f % kProjKAlign != 0)
        return KDA_ERR_SHAPE;
    const void* w[6] = {w_q, w_k, w_v, w_fa, w_ga, w_b};
    float* out[6] = {q_raw, k_raw, v_raw, f_down, g_down, beta_raw};
    if (!x) return KDA_ERR_NULL;
    for (int i = 0; i < 6; ++i)
        if (!w[i] || !out[i]) return KDA_ERR_NULL;
    if (!aligned16(x)) return KDA_ERR_ALIGN;
    for (int i = 0; i < 6; ++i)
        if (!aligned16(w[i])) return KDA_ERR_ALIGN;
    if (workspace == nullptr || workspace_bytes < proj_workspace_bytes(t, in_f))
        return KDA_ERR_WORKSPACE;
    if (!aligned16(workspace)) return KDA_ERR_ALIGN;
    if (const int sd = check_stream_device(stream)) return sd;
    Proj6Args a{};
    a.x = x;
    const int rows[6] = {H * kHeadDim, H * kHeadDim, H * kHeadDim, kHeadDim, kHeadDim, H};
    for (int i = 0; i < 6; ++i) {
        a.w[i] = w[i];
        a.out[i] = out[i];
        a.rows[i] = rows[i];
    }
    a.t = t;
    a.in_f = in_f;
    a.ws = workspace;
    a.err = dev_err_ptr();
    return cuda_status(launch_proj6(a, static_cast<cudaStream_t>(stream)));
}

int kda_scan_varlen_static(const float* q_hat, const float* k_hat, const float* v_hat,
                           const float* g, int gate_mode, const float* beta,
                           const float* state_in, float* state_out, float* o,
                           const int* cu_seqlens, const int* cu_seqlens_host, int N, int total_T,
                           int H, int D, float scale, void* stream) {
    // every contract check that does not need the device comes before the scratch setup
    if (D != kHeadDim) return KDA_ERR_HEAD_DIM;
    if (N < 0 || total_T < 0 || N > kMaxGridY || H <= 0) return KDA_ERR_SHAPE;
    if (N == 0) return KDA_OK;
    if (cu_seqlens == nullptr) return KDA_ERR_NULL;
    const int rc = check_cu(cu_seqlens_host, N, total_T);
    if (rc) return rc;
    const SeqLayout seq{cu_seqlens, 0, N, (long)total_T};
    if (chunk_workspace_bytes(seq, cu_seqlens_host, H) > kStaticScratchBytes)
        return KDA_ERR_SCRATCH_LIMIT;
    if (const int sd = check_stream_device(stream)) return sd;
    void* scratch = nullptr;
    const cudaError_t e = static_scratch(&scratch);
    if (e != cudaSuccess) return cuda_status(e);
    return scan_impl(q_hat, k_hat, v_hat, g, gate_mode, beta, state_in, state_out, o, seq,
                     cu_seqlens_host, H, D, scale, KDA_ALGO_CHUNK, scratch, kStaticScratchBytes,
                     stream);
}

}  // extern "C"
