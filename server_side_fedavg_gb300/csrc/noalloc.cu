// fa_aggregate_noalloc: weighted aggregation of one tensor that allocates no
// memory at all, for callers that cannot let a library call cudaMalloc --
// e.g. a process whose device memory is owned by another allocator (a
// framework's caching pool, a server that reserves its memory at start-up)
// or that forbids allocation on its request path.
//
// The fp32 running sum lives in a fixed array in this library's device image
// (FA_NOALLOC_MAX_ELEMS floats, 16 MiB), which every GPU that loads the
// library keeps until the process exits.  Host code cannot use the array's
// name as a device address: on the first call on each device the entry point
// looks the address up with cudaGetSymbolAddress (with that device current)
// and caches it; that first call should therefore come before any stream
// capture.  All calls share the array and it keeps the last call's contents:
// the first client's launch overwrites every element it uses (no clearing is
// needed), and calls that overlap on the GPU race on it.
#include <fedavg.h>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "kernels.cuh"

namespace {

__device__ __align__(256) float g_noalloc_sum[FA_NOALLOC_MAX_ELEMS];

constexpr int kMaxDevices = 64;

struct DeviceSetup {
    bool ready = false;
    float* sum = nullptr;       // device address of g_noalloc_sum on this device
    fa::LaunchShape shape;
};

std::mutex g_setup_mu;
DeviceSetup g_setup[kMaxDevices];

// Once per device, with that device current.
cudaError_t setup_for(int dev, DeviceSetup** out) {
    std::lock_guard<std::mutex> lk(g_setup_mu);
    DeviceSetup& d = g_setup[dev];
    if (!d.ready) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_sum);
        if (e != cudaSuccess) return e;
        e = fa::query_launch_shape(&d.shape);
        if (e != cudaSuccess) return e;
        d.sum = static_cast<float*>(p);
        d.ready = true;
    }
    *out = &d;
    return cudaSuccess;
}

// The finalize step over the fixed array: out[i] = RNE(sum[i] / N), the same
// IEEE division and cast as the regular finalize kernel.
template <typename Tout>
__global__ void finalize_noalloc_kernel(uint64_t n, float divisor, Tout* __restrict__ out) {
    const uint64_t stride = static_cast<uint64_t>(gridDim.x) * blockDim.x;
    for (uint64_t i = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
        const float q = __fdiv_rn(g_noalloc_sum[i], divisor);
        if constexpr (sizeof(Tout) == 4) {
            out[i] = q;
        } else {
            out[i] = __bfloat16_as_ushort(__float2bfloat16_rn(q));
        }
    }
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
    const float divisor = static_cast<float>(total);
    const int per = d->shape.fin_ctas_per_sm[0][dtype_out == FA_F32 ? 0 : 1];
    uint64_t want = (numel + fa::kBlock - 1) / fa::kBlock;
    uint64_t cap = static_cast<uint64_t>(d->shape.sms > 0 ? d->shape.sms : 1) * (per > 0 ? per : 1);
    const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
    if (dtype_out == FA_F32)
        finalize_noalloc_kernel<float><<<grid, fa::kBlock, 0, s>>>(numel, divisor, static_cast<float*>(out));
    else
        finalize_noalloc_kernel<uint16_t><<<grid, fa::kBlock, 0, s>>>(numel, divisor, static_cast<uint16_t*>(out));
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
