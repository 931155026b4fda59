// Finalize kernel (see kernels.cuh for the operation and device.cuh for the shared
// conventions): the running sum read with 128-bit loads, divided by each key's weight
// total, rounded to the output type (RNE for bf16) and written with 128-bit stores;
// delta rounds add server_lr times that mean to a base model with one rounding.
#include "device.cuh"

namespace fa {

namespace {

template <typename Tout>
struct LoadBase;

template <>
struct LoadBase<float> {
    static __device__ __forceinline__ void vec(const void* b, uint64_t e, float (&v)[8]) {
        const float* p = static_cast<const float*>(b) + e;
        const uint4 a = ld_stream_v4(p), c = ld_stream_v4(p + 4);
        v[0] = __uint_as_float(a.x); v[1] = __uint_as_float(a.y);
        v[2] = __uint_as_float(a.z); v[3] = __uint_as_float(a.w);
        v[4] = __uint_as_float(c.x); v[5] = __uint_as_float(c.y);
        v[6] = __uint_as_float(c.z); v[7] = __uint_as_float(c.w);
    }
    static __device__ __forceinline__ float one(const void* b, uint64_t e) {
        return static_cast<const float*>(b)[e];
    }
};

template <>
struct LoadBase<uint16_t> {
    static __device__ __forceinline__ void vec(const void* b, uint64_t e, float (&v)[8]) {
        const uint4 r = ld_stream_v4(static_cast<const uint16_t*>(b) + e);
        v[0] = bf16_lo(r.x); v[1] = bf16_hi(r.x);
        v[2] = bf16_lo(r.y); v[3] = bf16_hi(r.y);
        v[4] = bf16_lo(r.z); v[5] = bf16_hi(r.z);
        v[6] = bf16_lo(r.w); v[7] = bf16_hi(r.w);
    }
    static __device__ __forceinline__ float one(const void* b, uint64_t e) {
        return __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(b)[e]) << 16);
    }
};

// Segments whose first tiles a searching finalize CTA keeps in shared memory (16 KB).
constexpr uint32_t kFinSegCache = 4096;

// q = sum / N; delta rounds then add server_lr * q to the base with one rounding (fma).
template <typename Tout, bool kApply, bool kComp>
__device__ __forceinline__ void fin_vec(const FinSeg& sg, uint64_t e, const float* s,
                                        const float* sl, float lr) {
    float hi[8], lo[8] = {}, q[8];
    ld8f(s, hi);
    if constexpr (kComp) ld8f(sl, lo);
#pragma unroll
    for (int i = 0; i < 8; ++i)
        q[i] = kApply ? quotient<kComp>(hi[i], lo[i], sg.div) : quotient_out<kComp, Tout>(hi[i], lo[i], sg.div);
    if constexpr (kApply) {
        float b[8];
        LoadBase<Tout>::vec(sg.base, e, b);
#pragma unroll
        for (int i = 0; i < 8; ++i) q[i] = __fmaf_rn(lr, q[i], b[i]);
    }
    store8_global<Tout>(sg.out, e, q);
}

template <typename Tout, bool kApply, bool kComp>
__device__ __forceinline__ void fin_one(const FinSeg& sg, uint64_t e, const float* s,
                                        const float* sl, float lr) {
    float q = kApply ? quotient<kComp>(*s, kComp ? *sl : 0.0f, sg.div)
                     : quotient_out<kComp, Tout>(*s, kComp ? *sl : 0.0f, sg.div);
    if constexpr (kApply) q = __fmaf_rn(lr, q, LoadBase<Tout>::one(sg.base, e));
    store_one<Tout>(sg.out, e, q);
}

// kSearch: the layout has many keys per grid stride (small keys), so each CTA keeps the
// segments' first tiles in shared memory (up to kFinSegCache of them) and finds a tile's
// segment by binary search; otherwise the table is walked in global memory, one step per
// segment boundary crossed, which for large keys is rarely more than one step per tile.
template <typename Tout, bool kApply, bool kComp, bool kSearch>
__global__ void __launch_bounds__(kBlock) finalize_kernel(const __grid_constant__ FinArgs a, float lr) {
    const FinSeg* segs = a.segs ? a.segs : a.seg;   // device memory or these parameters
    const uint32_t nseg = a.nseg, ntiles = a.ntiles;
    const float* __restrict__ acc = a.acc;
    const float* __restrict__ acc_lo = a.acc_lo;
    constexpr int kVecPerTile = kTile / kVec;
    constexpr int kUnroll = kVecPerTile / kBlock;
    uint32_t si = 0;
    uint32_t next0 = nseg > 1 ? segs[1].tile0 : 0xFFFFFFFFu;   // first tile of segment si + 1
    [[maybe_unused]] uint32_t* t0s = nullptr;
    [[maybe_unused]] bool cached = false;
    if constexpr (kSearch) {
        __shared__ uint32_t t0_cache[kFinSegCache];
        t0s = t0_cache;
        cached = nseg <= kFinSegCache;
        if (cached) {
            for (uint32_t i = threadIdx.x; i < nseg; i += kBlock) t0s[i] = segs[i].tile0;
            __syncthreads();
        }
    }
    for (uint32_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
        if constexpr (kSearch) {
            if (t >= next0) {
                // the last segment whose first tile is at or before t, in (si, nseg)
                uint32_t lo = si + 1, hi = nseg;
                while (hi - lo > 1) {
                    const uint32_t mid = (lo + hi) / 2;
                    if ((cached ? t0s[mid] : segs[mid].tile0) <= t) lo = mid; else hi = mid;
                }
                si = lo;
                next0 = si + 1 < nseg ? (cached ? t0s[si + 1] : segs[si + 1].tile0) : 0xFFFFFFFFu;
            }
        } else {
            while (t >= next0) {
                ++si;
                next0 = si + 1 < nseg ? segs[si + 1].tile0 : 0xFFFFFFFFu;
            }
        }
        const FinSeg sg = segs[si];
        const uint64_t e0 = static_cast<uint64_t>(t - sg.tile0) * kTile;
        const uint64_t rem = sg.len - e0;
        const uint32_t cnt = rem < kTile ? static_cast<uint32_t>(rem) : kTile;
        const float* s0 = acc + sg.acc_idx + e0;
        const float* l0 = kComp ? acc_lo + sg.acc_idx + e0 : nullptr;
        // the sum side is always 128-byte aligned; the output (and base) may not be
        uintptr_t amask = reinterpret_cast<uintptr_t>(sg.out) + e0 * sizeof(Tout);
        if constexpr (kApply) amask |= reinterpret_cast<uintptr_t>(sg.base) + e0 * sizeof(Tout);
        if ((amask & 15u) == 0) {
            if (cnt == kTile) {
                // every load of the tile first: a store (asm volatile, memory clobber) would
                // otherwise hold the next vector's loads back, leaving one in flight per thread
                float hi[kUnroll][8], lo[kUnroll][8] = {};
                float b[kUnroll][8];
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const uint32_t v = threadIdx.x + u * kBlock;
                    ld8f(s0 + v * kVec, hi[u]);
                    if constexpr (kComp) ld8f(l0 + v * kVec, lo[u]);
                    if constexpr (kApply) LoadBase<Tout>::vec(sg.base, e0 + v * kVec, b[u]);
                }
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const uint32_t v = threadIdx.x + u * kBlock;
                    float q[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        q[i] = kApply ? quotient<kComp>(hi[u][i], lo[u][i], sg.div)
                                      : quotient_out<kComp, Tout>(hi[u][i], lo[u][i], sg.div);
                    if constexpr (kApply) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) q[i] = __fmaf_rn(lr, q[i], b[u][i]);
                    }
                    store8_global<Tout>(sg.out, e0 + v * kVec, q);
                }
            } else {
                const uint32_t nv = cnt / kVec;
                for (uint32_t v = threadIdx.x; v < nv; v += kBlock)
                    fin_vec<Tout, kApply, kComp>(sg, e0 + v * kVec, s0 + v * kVec,
                                                 kComp ? l0 + v * kVec : nullptr, lr);
                const uint32_t tail = cnt - nv * kVec;
                if (threadIdx.x < tail) {
                    const uint32_t e = nv * kVec + threadIdx.x;
                    fin_one<Tout, kApply, kComp>(sg, e0 + e, s0 + e, kComp ? l0 + e : nullptr, lr);
                }
            }
        } else {
            for (uint32_t e = threadIdx.x; e < cnt; e += kBlock)
                fin_one<Tout, kApply, kComp>(sg, e0 + e, s0 + e, kComp ? l0 + e : nullptr, lr);
        }
    }
}

// ----------------------------------------------------------------- host side
template <typename Tout, bool kApply, bool kComp>
cudaError_t finalize_t(uint32_t grid, const FinArgs& a, float lr, cudaStream_t stream) {
    // many keys per grid stride: search the segment table instead of walking it
    const bool search = a.nseg > 1 && static_cast<uint64_t>(a.ntiles) < static_cast<uint64_t>(a.nseg) * grid;
    // a plain launch (no programmatic dependency: the kernel reads the sum from its
    // first instruction); the status is this launch's own
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kBlock);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = nullptr;
    cfg.numAttrs = 0;
    return search ? cudaLaunchKernelEx(&cfg, finalize_kernel<Tout, kApply, kComp, true>, a, lr)
                  : cudaLaunchKernelEx(&cfg, finalize_kernel<Tout, kApply, kComp, false>, a, lr);
}

template <bool kComp>
cudaError_t finalize_pick(uint32_t grid, int dtype_out, bool apply, const FinArgs& a, float lr,
                          cudaStream_t stream) {
    if (dtype_out == 0) {
        return apply ? finalize_t<float, true, kComp>(grid, a, lr, stream)
                     : finalize_t<float, false, kComp>(grid, a, lr, stream);
    }
    return apply ? finalize_t<uint16_t, true, kComp>(grid, a, lr, stream)
                 : finalize_t<uint16_t, false, kComp>(grid, a, lr, stream);
}

template <bool kComp>
cudaError_t prepare_finalize_shapes_t(LaunchShape* s) {
    const int c = kComp ? 1 : 0;
    cudaError_t r = cudaSuccess;
    auto keep = [&r](cudaError_t x) { if (r == cudaSuccess) r = x; };
    keep(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&s->fin_ctas_per_sm[c][0][0],
                                                       finalize_kernel<float, false, kComp, false>, kBlock, 0));
    keep(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&s->fin_ctas_per_sm[c][0][1],
                                                       finalize_kernel<uint16_t, false, kComp, false>, kBlock, 0));
    keep(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&s->fin_ctas_per_sm[c][1][0],
                                                       finalize_kernel<float, true, kComp, false>, kBlock, 0));
    keep(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&s->fin_ctas_per_sm[c][1][1],
                                                       finalize_kernel<uint16_t, true, kComp, false>, kBlock, 0));
    return r;
}

}  // namespace

Divisor make_divisor(double n) {
    Divisor d;
    d.hi = static_cast<float>(n);
    d.lo = static_cast<float>(n - static_cast<double>(d.hi));
    d.rcp = static_cast<float>(1.0 / static_cast<double>(d.hi));
    return d;
}

cudaError_t prepare_finalize_shapes(LaunchShape* s) {
    cudaError_t e = prepare_finalize_shapes_t<false>(s);
    if (e == cudaSuccess) e = prepare_finalize_shapes_t<true>(s);
    return e;
}

cudaError_t launch_finalize(const FinArgs& a, int dtype_out, bool apply, float server_lr, bool host_out,
                            const LaunchShape& s, cudaStream_t stream) {
    if (a.ntiles == 0 || a.nseg == 0) return cudaSuccess;
    if (a.segs == nullptr && a.nseg > kFinInlineSegs) return cudaErrorInvalidValue;
    const int c = a.acc_lo ? 1 : 0;
    const int occ = s.fin_ctas_per_sm[c][apply ? 1 : 0][dtype_out == 0 ? 0 : 1];
    const uint32_t grid = grid_for(a.ntiles, s.sms, host_out ? occ : std::min(occ, kFinCtasPerSm));
    return c ? finalize_pick<true>(grid, dtype_out, apply, a, server_lr, stream)
             : finalize_pick<false>(grid, dtype_out, apply, a, server_lr, stream);
}

}  // namespace fa
