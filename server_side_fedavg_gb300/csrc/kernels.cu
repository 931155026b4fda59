// Aggregation kernels for sm_103a (see kernels.cuh).
//
// Design (GB300: 152 SMs, HBM3e):
//  - persistent CTAs, grid = SMs x resident CTAs per SM, striding over 4096-element
//    tiles; a tile never crosses a segment (one key's run), so each CTA takes one
//    uniform branch per tile;
//  - 128-bit loads and stores, 8 elements per vector: one 16-byte load of bf16
//    input (or two of fp32) and two 16-byte loads / stores of the fp32 sum; a warp
//    touches 512 contiguous bytes of the sum per vector step;
//  - client input is read once: non-coherent loads that skip L1; the sum keeps the
//    default policy so small layouts (adapters) stay resident in the 129 MB L2
//    between clients;
//  - ragged tails (len % 8) and segments whose pointers are not 16-byte aligned
//    take a scalar path, one element per thread.
// Arithmetic: __fmul_rn / __fmaf_rn / __fdiv_rn so the compiler never fuses or
// reorders: the first contribution is a rounded product, every later one one
// fused multiply-add, in client order.
#include "kernels.cuh"

#include <cuda_bf16.h>

namespace fa {
namespace {

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ float4 ld_v4f(const float* p) {
    float4 r;
    asm volatile("ld.global.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ void st_v4f(float* p, float4 v) {
    asm volatile("st.global.v4.f32 [%0], {%1,%2,%3,%4};" ::"l"(p), "f"(v.x), "f"(v.y),
                 "f"(v.z), "f"(v.w)
                 : "memory");
}

__device__ __forceinline__ void st_v4u(void* p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// bf16 -> fp32 is exact: the bf16 bits are the top half of the fp32 bits.
__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

template <typename Tin>
struct Load8;

template <>
struct Load8<uint16_t> {   // bf16
    static __device__ __forceinline__ void vec(const uint16_t* p, float (&v)[8]) {
        uint4 r = ld_stream_v4(p);
        v[0] = bf16_lo(r.x); v[1] = bf16_hi(r.x);
        v[2] = bf16_lo(r.y); v[3] = bf16_hi(r.y);
        v[4] = bf16_lo(r.z); v[5] = bf16_hi(r.z);
        v[6] = bf16_lo(r.w); v[7] = bf16_hi(r.w);
    }
    static __device__ __forceinline__ float one(const uint16_t* p) {
        uint16_t u;
        asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(u) : "l"(p));
        return __uint_as_float(static_cast<uint32_t>(u) << 16);
    }
};

template <>
struct Load8<float> {
    static __device__ __forceinline__ void vec(const float* p, float (&v)[8]) {
        uint4 a = ld_stream_v4(p);
        uint4 b = ld_stream_v4(p + 4);
        v[0] = __uint_as_float(a.x); v[1] = __uint_as_float(a.y);
        v[2] = __uint_as_float(a.z); v[3] = __uint_as_float(a.w);
        v[4] = __uint_as_float(b.x); v[5] = __uint_as_float(b.y);
        v[6] = __uint_as_float(b.z); v[7] = __uint_as_float(b.w);
    }
    static __device__ __forceinline__ float one(const float* p) {
        float f;
        asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(f) : "l"(p));
        return f;
    }
};

// One vector of 8 elements: r = first ? w0*x0 : sum;  r = fma(wj, xj, r) for j >= 1
// (j >= 0 when not first).
template <typename Tin, int J>
__device__ __forceinline__ void acc_vec(const AccArgs& a, uint64_t xe, float* s, bool first) {
    float x[J][8];
#pragma unroll
    for (int j = 0; j < J; ++j)
        Load8<Tin>::vec(static_cast<const Tin*>(a.x[j]) + xe, x[j]);
    float r[8];
    if (first) {
#pragma unroll
        for (int e = 0; e < 8; ++e) r[e] = __fmul_rn(a.w[0], x[0][e]);
    } else {
        float4 lo = ld_v4f(s), hi = ld_v4f(s + 4);
        r[0] = lo.x; r[1] = lo.y; r[2] = lo.z; r[3] = lo.w;
        r[4] = hi.x; r[5] = hi.y; r[6] = hi.z; r[7] = hi.w;
#pragma unroll
        for (int e = 0; e < 8; ++e) r[e] = __fmaf_rn(a.w[0], x[0][e], r[e]);
    }
#pragma unroll
    for (int j = 1; j < J; ++j) {
#pragma unroll
        for (int e = 0; e < 8; ++e) r[e] = __fmaf_rn(a.w[j], x[j][e], r[e]);
    }
    st_v4f(s, make_float4(r[0], r[1], r[2], r[3]));
    st_v4f(s + 4, make_float4(r[4], r[5], r[6], r[7]));
}

template <typename Tin, int J>
__device__ __forceinline__ void acc_one(const AccArgs& a, uint64_t xe, float* s, bool first) {
    float r = first ? __fmul_rn(a.w[0], Load8<Tin>::one(static_cast<const Tin*>(a.x[0]) + xe))
                    : __fmaf_rn(a.w[0], Load8<Tin>::one(static_cast<const Tin*>(a.x[0]) + xe), *s);
#pragma unroll
    for (int j = 1; j < J; ++j)
        r = __fmaf_rn(a.w[j], Load8<Tin>::one(static_cast<const Tin*>(a.x[j]) + xe), r);
    *s = r;
}

template <typename Tin, int J>
__global__ void __launch_bounds__(kBlock) accumulate_kernel(const __grid_constant__ AccArgs a) {
    constexpr int kVecPerTile = kTile / kVec;                  // 512
    constexpr int kUnroll = kVecPerTile / kBlock;              // 2
    uint32_t si = 0;
    for (uint32_t t = blockIdx.x; t < a.ntiles; t += gridDim.x) {
        while (si + 1 < a.nseg && t >= a.seg[si + 1].tile0) ++si;
        const AccSeg& sg = a.seg[si];
        const uint64_t e0 = static_cast<uint64_t>(t - sg.tile0) * kTile;
        const uint64_t rem = sg.len - e0;
        const uint32_t cnt = rem < kTile ? static_cast<uint32_t>(rem) : kTile;
        const bool first = sg.first != 0;
        const uint64_t xe0 = sg.x_off + e0;
        float* s0 = a.acc + sg.acc_idx + e0;
        if ((a.vec_ok >> si) & 1ull) {
            if (cnt == kTile) {
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const uint32_t v = threadIdx.x + u * kBlock;
                    acc_vec<Tin, J>(a, xe0 + v * kVec, s0 + v * kVec, first);
                }
            } else {
                const uint32_t nv = cnt / kVec;
                for (uint32_t v = threadIdx.x; v < nv; v += kBlock)
                    acc_vec<Tin, J>(a, xe0 + v * kVec, s0 + v * kVec, first);
                const uint32_t tail = cnt - nv * kVec;
                if (threadIdx.x < tail) {
                    const uint32_t e = nv * kVec + threadIdx.x;
                    acc_one<Tin, J>(a, xe0 + e, s0 + e, first);
                }
            }
        } else {
            for (uint32_t e = threadIdx.x; e < cnt; e += kBlock)
                acc_one<Tin, J>(a, xe0 + e, s0 + e, first);
        }
    }
}

template <typename Tout>
struct Store;

template <>
struct Store<float> {
    static __device__ __forceinline__ void vec(void* out, uint64_t e, const float (&q)[8]) {
        float* p = static_cast<float*>(out) + e;
        st_v4f(p, make_float4(q[0], q[1], q[2], q[3]));
        st_v4f(p + 4, make_float4(q[4], q[5], q[6], q[7]));
    }
    static __device__ __forceinline__ void one(void* out, uint64_t e, float q) {
        static_cast<float*>(out)[e] = q;
    }
};

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(a))) |
           (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(b))) << 16);
}

template <>
struct Store<uint16_t> {
    static __device__ __forceinline__ void vec(void* out, uint64_t e, const float (&q)[8]) {
        uint4 v = make_uint4(pack_bf16(q[0], q[1]), pack_bf16(q[2], q[3]),
                             pack_bf16(q[4], q[5]), pack_bf16(q[6], q[7]));
        st_v4u(static_cast<uint16_t*>(out) + e, v);
    }
    static __device__ __forceinline__ void one(void* out, uint64_t e, float q) {
        static_cast<uint16_t*>(out)[e] = __bfloat16_as_ushort(__float2bfloat16_rn(q));
    }
};

template <typename Tout>
__global__ void __launch_bounds__(kBlock) finalize_kernel(const FinSeg* __restrict__ segs,
                                                          uint32_t nseg, uint32_t ntiles,
                                                          const float* __restrict__ acc) {
    constexpr int kVecPerTile = kTile / kVec;
    constexpr int kUnroll = kVecPerTile / kBlock;
    uint32_t si = 0;
    uint32_t next0 = nseg > 1 ? segs[1].tile0 : 0xFFFFFFFFu;
    for (uint32_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
        while (t >= next0) {
            ++si;
            next0 = si + 1 < nseg ? segs[si + 1].tile0 : 0xFFFFFFFFu;
        }
        const FinSeg sg = segs[si];
        const uint64_t e0 = static_cast<uint64_t>(t - sg.tile0) * kTile;
        const uint64_t rem = sg.len - e0;
        const uint32_t cnt = rem < kTile ? static_cast<uint32_t>(rem) : kTile;
        const float* s0 = acc + sg.acc_idx + e0;
        const float d = sg.divisor;
        const uintptr_t oaddr = reinterpret_cast<uintptr_t>(sg.out) + e0 * sizeof(Tout);
        const bool vec_ok = (oaddr & 15u) == 0;   // the sum side is always 128-byte aligned
        if (vec_ok) {
            const uint32_t nv = cnt / kVec;
            if (cnt == kTile) {
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const uint32_t v = threadIdx.x + u * kBlock;
                    float4 lo = ld_v4f(s0 + v * kVec), hi = ld_v4f(s0 + v * kVec + 4);
                    float q[8] = {__fdiv_rn(lo.x, d), __fdiv_rn(lo.y, d), __fdiv_rn(lo.z, d),
                                  __fdiv_rn(lo.w, d), __fdiv_rn(hi.x, d), __fdiv_rn(hi.y, d),
                                  __fdiv_rn(hi.z, d), __fdiv_rn(hi.w, d)};
                    Store<Tout>::vec(sg.out, e0 + v * kVec, q);
                }
            } else {
                for (uint32_t v = threadIdx.x; v < nv; v += kBlock) {
                    float4 lo = ld_v4f(s0 + v * kVec), hi = ld_v4f(s0 + v * kVec + 4);
                    float q[8] = {__fdiv_rn(lo.x, d), __fdiv_rn(lo.y, d), __fdiv_rn(lo.z, d),
                                  __fdiv_rn(lo.w, d), __fdiv_rn(hi.x, d), __fdiv_rn(hi.y, d),
                                  __fdiv_rn(hi.z, d), __fdiv_rn(hi.w, d)};
                    Store<Tout>::vec(sg.out, e0 + v * kVec, q);
                }
                const uint32_t tail = cnt - nv * kVec;
                if (threadIdx.x < tail) {
                    const uint32_t e = nv * kVec + threadIdx.x;
                    Store<Tout>::one(sg.out, e0 + e, __fdiv_rn(s0[e], d));
                }
            }
        } else {
            for (uint32_t e = threadIdx.x; e < cnt; e += kBlock)
                Store<Tout>::one(sg.out, e0 + e, __fdiv_rn(s0[e], d));
        }
    }
}

template <typename Tin, int J>
cudaError_t launch_acc_t(const AccArgs& a, int ctas_per_sm, int sms, cudaStream_t stream) {
    if (a.ntiles == 0) return cudaSuccess;
    uint32_t cap = static_cast<uint32_t>(sms > 0 ? sms : 1) *
                   static_cast<uint32_t>(ctas_per_sm > 0 ? ctas_per_sm : 1);
    uint32_t grid = a.ntiles < cap ? a.ntiles : cap;
    accumulate_kernel<Tin, J><<<grid, kBlock, 0, stream>>>(a);
    return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_acc_j(const AccArgs& a, const LaunchShape& s, int in, cudaStream_t stream) {
    switch (a.J) {
        case 1: return launch_acc_t<Tin, 1>(a, s.acc_ctas_per_sm[in][0], s.sms, stream);
        case 2: return launch_acc_t<Tin, 2>(a, s.acc_ctas_per_sm[in][1], s.sms, stream);
        case 4: return launch_acc_t<Tin, 4>(a, s.acc_ctas_per_sm[in][2], s.sms, stream);
        case 8: return launch_acc_t<Tin, 8>(a, s.acc_ctas_per_sm[in][3], s.sms, stream);
        case 16: return launch_acc_t<Tin, 16>(a, s.acc_ctas_per_sm[in][4], s.sms, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <typename Tin, int J>
cudaError_t occ_acc(int* n) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, accumulate_kernel<Tin, J>, kBlock, 0);
}

}  // namespace

cudaError_t query_launch_shape(LaunchShape* s) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&s->sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    cudaError_t r = cudaSuccess;
    auto keep = [&r](cudaError_t x) { if (r == cudaSuccess) r = x; };
    keep(occ_acc<float, 1>(&s->acc_ctas_per_sm[0][0]));
    keep(occ_acc<float, 2>(&s->acc_ctas_per_sm[0][1]));
    keep(occ_acc<float, 4>(&s->acc_ctas_per_sm[0][2]));
    keep(occ_acc<float, 8>(&s->acc_ctas_per_sm[0][3]));
    keep(occ_acc<float, 16>(&s->acc_ctas_per_sm[0][4]));
    keep(occ_acc<uint16_t, 1>(&s->acc_ctas_per_sm[1][0]));
    keep(occ_acc<uint16_t, 2>(&s->acc_ctas_per_sm[1][1]));
    keep(occ_acc<uint16_t, 4>(&s->acc_ctas_per_sm[1][2]));
    keep(occ_acc<uint16_t, 8>(&s->acc_ctas_per_sm[1][3]));
    keep(occ_acc<uint16_t, 16>(&s->acc_ctas_per_sm[1][4]));
    keep(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&s->fin_ctas_per_sm[0],
                                                       finalize_kernel<float>, kBlock, 0));
    keep(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&s->fin_ctas_per_sm[1],
                                                       finalize_kernel<uint16_t>, kBlock, 0));
    return r;
}

cudaError_t launch_accumulate(const AccArgs& a, int dtype_in, const LaunchShape& s,
                              cudaStream_t stream) {
    return dtype_in == 0 ? launch_acc_j<float>(a, s, 0, stream)
                         : launch_acc_j<uint16_t>(a, s, 1, stream);
}

cudaError_t launch_finalize(const FinSeg* segs, uint32_t nseg, uint32_t ntiles, int dtype_out,
                            const float* acc, const LaunchShape& s, cudaStream_t stream) {
    if (ntiles == 0 || nseg == 0) return cudaSuccess;
    int per = s.fin_ctas_per_sm[dtype_out == 0 ? 0 : 1];
    uint32_t cap = static_cast<uint32_t>(s.sms > 0 ? s.sms : 1) *
                   static_cast<uint32_t>(per > 0 ? per : 1);
    uint32_t grid = ntiles < cap ? ntiles : cap;
    if (dtype_out == 0)
        finalize_kernel<float><<<grid, kBlock, 0, stream>>>(segs, nseg, ntiles, acc);
    else
        finalize_kernel<uint16_t><<<grid, kBlock, 0, stream>>>(segs, nseg, ntiles, acc);
    return cudaGetLastError();
}

}  // namespace fa
