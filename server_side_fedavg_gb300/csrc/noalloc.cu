// fa_aggregate_noalloc: weighted aggregation of one tensor that allocates no
// memory at all, for callers that cannot let a library call cudaMalloc --
// e.g. a process whose device memory is owned by another allocator (a
// framework's caching pool, a server that reserves its memory at start-up)
// or that forbids allocation on its request path.
//
// Its device state lives in fixed arrays of this library's device image, which
// every GPU that loads the library keeps until the process exits: the fp32
// running sum (FA_NOALLOC_MAX_ELEMS floats, 16 MiB) and an error word of its own
// (read and cleared by fa_aggregate_noalloc_status); the finalize kernel's one-entry
// segment table travels in its launch's parameters.  Host code cannot use
// these names as device addresses: on the first call on each device the entry
// point looks the addresses up with cudaGetSymbolAddress (with that device
// current) and caches them; that first call should therefore come before any
// stream capture.  All calls share the arrays and they keep the last call's
// contents: the first client's launch overwrites every element of the sum it
// uses (no clearing is needed), and calls that overlap on the GPU race on it.
#include <fedavg.h>

#include <cuda_runtime.h>

#include <chrono>
#include <cmath>
#include <cstring>
#include <mutex>
#include <thread>

#include "kernels.cuh"

namespace {

__device__ __align__(256) float g_noalloc_sum[FA_NOALLOC_MAX_ELEMS];
__device__ unsigned int g_noalloc_error;

constexpr int kMaxDevices = 64;

struct DeviceSetup {
    bool ready = false;
    float* sum = nullptr;            // device address of g_noalloc_sum on this device
    unsigned int* err = nullptr;     // ... of g_noalloc_error
    fa::LaunchShape shape;
};

std::mutex g_setup_mu;
DeviceSetup g_setup[kMaxDevices];

// Once per device, with that device current.
cudaError_t setup_for(int dev, DeviceSetup** out) {
    std::lock_guard<std::mutex> lk(g_setup_mu);
    DeviceSetup& d = g_setup[dev];
    if (!d.ready) {
        void* sum = nullptr;
        void* err = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&sum, g_noalloc_sum);
        if (e == cudaSuccess) e = cudaGetSymbolAddress(&err, g_noalloc_error);
        if (e == cudaSuccess) e = fa::query_launch_shape(&d.shape);
        if (e != cudaSuccess) return e;
        d.sum = static_cast<float*>(sum);
        d.err = static_cast<unsigned int*>(err);
        d.ready = true;
    }
    *out = &d;
    return cudaSuccess;
}


// Memory of device `dev`; managed memory only where plain stores touch it (the output):
// inputs are read with bulk copies, which are kept off pages that may sit on the host.
bool is_device_memory(const void* p, int dev, bool allow_managed) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return (at.type == cudaMemoryTypeDevice && at.device == dev) ||
           (allow_managed && at.type == cudaMemoryTypeManaged);
}

}  // namespace

extern "C" fa_status fa_aggregate_noalloc(uint32_t n_clients, const double* weights,
                                          const void* const* client_ptrs, uint64_t numel,
                                          fa_dtype dtype_in, fa_dtype dtype_out, void* out,
                                          void* stream) {
    if ((dtype_in != FA_F32 && dtype_in != FA_BF16) || (dtype_out != FA_F32 && dtype_out != FA_BF16))
        return FA_ERR_DTYPE;
    if (numel > FA_NOALLOC_MAX_ELEMS) return FA_ERR_RANGE;
    if (n_clients == 0 || numel == 0) return FA_OK;
    if (weights == nullptr || client_ptrs == nullptr || out == nullptr) return FA_ERR_ARG;
    double total = 0.0;
    for (uint32_t j = 0; j < n_clients; ++j) {
        const double w = weights[j];
        if (!std::isfinite(w) || w < 0.0 || w > 16777216.0) return FA_ERR_WEIGHT;
        total += w;
    }
    if (total == 0.0) return FA_OK;   // no weight: out is left as it was

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
    for (uint32_t j = 0; j < n_clients; ++j)
        if (client_ptrs[j] == nullptr || !is_device_memory(client_ptrs[j], dev, false)) return FA_ERR_ARG;
    if (!is_device_memory(out, dev, true)) return FA_ERR_ARG;
    DeviceSetup* d = nullptr;
    if (setup_for(dev, &d) != cudaSuccess) return FA_ERR_CUDA;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int din = dtype_in == FA_F32 ? 0 : 1;
    // clients in batches of 16, 8, 4, 2, 1, in index order; the first batch
    // starts the sum (stores its first product), so no clearing is needed
    uint32_t done = 0;
    while (done < n_clients) {
        uint32_t left = n_clients - done, jb = 16;
        while (jb > left) jb >>= 1;
        fa::AccArgs a;
        std::memset(&a, 0, sizeof a);
        bool aligned = true;
        for (uint32_t j = 0; j < jb; ++j) {
            a.x[j] = client_ptrs[done + j];
            a.w[j] = static_cast<float>(weights[done + j]);
            aligned = aligned && (reinterpret_cast<uintptr_t>(a.x[j]) & 15u) == 0;
        }
        a.acc = d->sum;
        a.acc_lo = nullptr;
        a.err = d->err;
        a.J = jb;
        a.nseg = 1;
        a.vec_ok = aligned ? 1ull : 0ull;
        a.seg[0].x = a.x[0];
        a.seg[0].x_off = 0;
        a.seg[0].acc_idx = 0;
        a.seg[0].len = numel;
        a.seg[0].first = done == 0 ? 1u : 0u;
        if (fa::launch_accumulate(a, din, d->shape, s) != cudaSuccess) return FA_ERR_CUDA;
        done += jb;
    }
    // the finalize step: the library's tiled finalize kernel, its one-entry segment table
    // in the launch's parameters
    static thread_local fa::FinArgs fin;
    fin.segs = nullptr;
    fin.acc = d->sum;
    fin.acc_lo = nullptr;
    fin.nseg = 1;
    fin.ntiles = static_cast<uint32_t>((numel + fa::kTile - 1) / fa::kTile);
    fa::FinSeg& seg = fin.seg[0];
    std::memset(&seg, 0, sizeof seg);
    seg.acc_idx = 0;
    seg.len = numel;
    seg.out = out;
    seg.base = nullptr;
    seg.div = fa::make_divisor(total);
    seg.tile0 = 0;
    const cudaError_t fe = fa::launch_finalize(fin, dtype_out == FA_F32 ? 0 : 1, false, 1.0f, false, d->shape, s);
    return fe == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

extern "C" fa_status fa_aggregate_noalloc_status(void* stream, uint32_t timeout_ms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
    DeviceSetup* d = nullptr;
    if (setup_for(dev, &d) != cudaSuccess) return FA_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // wait, bounded, for the work queued on `stream` (polling: never blocks without bound)
    const auto t0 = std::chrono::steady_clock::now();
    const uint32_t limit = timeout_ms ? timeout_ms : 60000u;
    for (uint32_t spins = 0;; ++spins) {
        const cudaError_t q = cudaStreamQuery(s);
        if (q == cudaSuccess) break;
        if (q != cudaErrorNotReady) return FA_ERR_CUDA;
        const auto ms = std::chrono::duration_cast<std::chrono::milliseconds>(
                            std::chrono::steady_clock::now() - t0).count();
        if (ms > static_cast<long long>(limit)) return FA_ERR_TIMEOUT;
        if (spins < 64)
            std::this_thread::yield();
        else
            std::this_thread::sleep_for(std::chrono::microseconds(50));
    }
    // the stream is idle: read the word (a 4-byte copy into this stack variable) and clear it
    unsigned int word = 0;
    // (a copy into pageable memory returns once it has completed)
    if (cudaMemcpyAsync(&word, d->err, sizeof word, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return FA_ERR_CUDA;
    if (word == 0) return FA_OK;
    if (cudaMemsetAsync(d->err, 0, sizeof word, s) != cudaSuccess) return FA_ERR_CUDA;
    return FA_ERR_INTERNAL;
}
