// Seeded synthetic client updates: device side.  Input creation only.
// Same definition as synth.c, operation for operation: integer SplitMix64
// draws, the Irwin-Hall(12) integer sum, and single IEEE double operations
// written with explicit round-to-nearest intrinsics so that nothing is
// contracted into an fma.  A GPU test checks these bits against synth.c.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ULL;

__host__ __device__ __forceinline__ uint64_t mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

__host__ __device__ __forceinline__ uint64_t draw(uint64_t key, uint64_t c) {
    return mix(key + (c + 1) * kGamma);
}

__device__ __forceinline__ long long ih12(uint64_t key, uint64_t c0) {
    long long s = 0;
#pragma unroll
    for (int d = 0; d < 3; ++d) {
        uint64_t r = draw(key, c0 + d);
        s += (long long)(r & 0xFFFF) + (long long)((r >> 16) & 0xFFFF) +
             (long long)((r >> 32) & 0xFFFF) + (long long)(r >> 48);
    }
    return s - 393210;
}

__device__ __forceinline__ float value_f32(uint64_t key, int dist, double sigma, uint64_t i) {
    double v;
    if (dist == 0) {
        double z = __dmul_rn((double)ih12(key, 3 * i), 0x1p-16);
        v = __dmul_rn(sigma, z);
    } else {
        long long s0 = ih12(key, 12 * i);
        long long s1 = ih12(key, 12 * i + 3);
        long long s2 = ih12(key, 12 * i + 6);
        long long s3 = ih12(key, 12 * i + 9);
        long long vi = s1 * s1 + s2 * s2 + s3 * s3;
        if (vi == 0) vi = 1;
        double vv = __dmul_rn((double)vi, 0x1p-32);
        double q = __ddiv_rn(vv, 3.0);
        double r = __dsqrt_rn(q);
        double t = __ddiv_rn(__dmul_rn((double)s0, 0x1p-16), r);
        v = __dmul_rn(sigma, t);
    }
    return __double2float_rn(v);
}

__global__ void fill_kernel(uint64_t key, int dist, double sigma, int dtype,
                            uint64_t first, uint64_t n, void* out) {
    uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t j = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; j < n; j += stride) {
        float f = value_f32(key, dist, sigma, first + j);
        if (dtype == 0) {
            static_cast<float*>(out)[j] = f;
        } else {
            static_cast<uint16_t*>(out)[j] = (uint16_t)(__float_as_uint(f) >> 16);
        }
    }
}

}  // namespace

extern "C" int synth_dev_fill(uint64_t seed, uint64_t client, int dist, double sigma,
                              int dtype, uint64_t first, uint64_t n, void* out,
                              void* stream) {
    if (n == 0) return 0;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    uint64_t want = (n + 255) / 256;
    uint64_t cap = (uint64_t)sms * 8;
    unsigned grid = (unsigned)(want < cap ? want : cap);
    fill_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        draw(seed, client), dist, sigma, dtype, first, n, out);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}
