// kda_timer.cu -- optional per-kernel timing: while enabled, every kernel the library launches is
// bracketed by a pair of CUDA events recorded on its stream; a read waits for the pending pairs and
// returns, per kernel, the number of launches and the summed device time.  Disabled (the default)
// it costs one relaxed atomic load per launch.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "../../include/kda.h"
#include "kda_internal.h"

namespace kda {

namespace {

constexpr int kMaxDev = 64;

struct Pending {
    int id; int dev; cudaEvent_t a, b;
};

std::atomic<bool> g_on{false};
std::mutex g_mu;
std::vector<Pending> g_pending;
std::vector<cudaEvent_t> g_free[kMaxDev];   // recycled events, per device
double g_ms[kKernelCount];
long g_launches[kKernelCount];
thread_local cudaEvent_t t_open[kKernelCount];
thread_local int t_open_dev[kKernelCount];

cudaEvent_t take_event(int dev) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_free[dev].empty()) {
        cudaEvent_t e = g_free[dev].back();
        g_free[dev].pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

const char* const kNames[kKernelCount] = {
    "kda_prep_kernel",        "kda_ring_roll_kernel",   "kda_scan_seq_kernel",
    "kda_chunk_offsets_kernel", "kda_chunk_intra_kernel", "kda_chunk_inter_kernel",
    "kda_gated_rmsnorm_kernel", "kda_decode_fused_kernel", "kda_chunk_prep_intra_kernel",
    "kda_proj_split_kernel",  "kda_proj6_kernel"};

}  // namespace

KernelTimer::KernelTimer(int id, cudaStream_t s) : id_(id), s_(s), on_(false) {
    if (!g_on.load(std::memory_order_relaxed)) return;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return;
    cudaEvent_t e = take_event(dev);
    if (e == nullptr || cudaEventRecord(e, s) != cudaSuccess) return;
    t_open[id] = e;
    t_open_dev[id] = dev;
    on_ = true;
}

KernelTimer::~KernelTimer() {
    if (!on_) return;
    const int dev = t_open_dev[id_];
    cudaEvent_t e = take_event(dev);
    if (e == nullptr || cudaEventRecord(e, s_) != cudaSuccess) return;
    std::lock_guard<std::mutex> lk(g_mu);
    g_pending.push_back({id_, dev, t_open[id_], e});
}

}  // namespace kda

using namespace kda;

extern "C" {

int kda_kernel_timing(int enable) {
    std::lock_guard<std::mutex> lk(g_mu);
    const bool was = g_on.exchange(enable != 0);
    if (enable) {
        for (int i = 0; i < kKernelCount; ++i) { g_ms[i] = 0.0; g_launches[i] = 0; }
    }
    return was ? 1 : 0;
}

int kda_kernel_times(int max_kernels, long* launches, double* total_ms) {
    std::lock_guard<std::mutex> lk(g_mu);
    int prev = -1;
    for (const Pending& p : g_pending) {
        if (p.dev != prev) {
            if (cudaSetDevice(p.dev) != cudaSuccess) return -(KDA_ERR_CUDA_BASE);
            prev = p.dev;
        }
        float ms = 0.0f;
        cudaError_t e = cudaEventSynchronize(p.b);
        if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, p.a, p.b);
        if (e != cudaSuccess) return -(KDA_ERR_CUDA_BASE + (int)e);
        g_ms[p.id] += ms;
        g_launches[p.id] += 1;
        g_free[p.dev].push_back(p.a);
        g_free[p.dev].push_back(p.b);
    }
    g_pending.clear();
    const int n = max_kernels < kKernelCount ? max_kernels : kKernelCount;
    for (int i = 0; i < n; ++i) {
        if (launches) launches[i] = g_launches[i];
        if (total_ms) total_ms[i] = g_ms[i];
        g_launches[i] = 0;
        g_ms[i] = 0.0;
    }
    return kKernelCount;
}

const char* kda_kernel_name(int id) { return id >= 0 && id < kKernelCount ? kNames[id] : nullptr; }

}  // extern "C"
