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

__device__ unsigned int g_device_error;

namespace {

constexpr uint32_t kMaxWaitSpins = 1u << 24;   // bound on every mbarrier wait

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

// ---------------------------------------------------------------------------
// Streaming accumulate (one client per launch) through a shared-memory pipeline
// fed by bulk copies (cp.async.bulk, the 1-D form of TMA):
//   thread 0 keeps S-1 tiles in flight: for each tile it arms the stage's
//   mbarrier with the byte count and issues one bulk load of the input tile and,
//   unless this is the first contribution, one of the sum tile;
//   all 256 threads wait on the stage's mbarrier, compute in shared memory, and
//   thread 0 writes the sum tile back with one bulk store;
//   a stage is refilled once the bulk store that drained it has read it.
// A tile's vector part (multiple of 8 elements) moves by bulk copies; its ragged
// tail and any segment whose pointers are not 16-byte aligned use direct loads.
// Every mbarrier wait is bounded; a timeout sets g_device_error (read by
// fa_sync), makes the CTA wait (bounded) for its own loads in flight, and return.
template <typename Tin>
struct BulkStages;
template <>
struct BulkStages<uint16_t> { static constexpr int kS = 3; };   // 3 x 48 KB = 144 KB: 1 CTA per SM
template <>
struct BulkStages<float> { static constexpr int kS = 3; };      // 3 x 64 KB = 192 KB: 1 CTA per SM

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    for (uint32_t it = 0; it < kMaxWaitSpins; ++it) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done) : "r"(bar), "r"(parity) : "memory");
        if (done) return true;
    }
    return false;
}

struct TileAt {
    uint32_t si;
    uint64_t e0;
    uint32_t cnt;
};

__device__ __forceinline__ TileAt tile_at(const AccArgs& a, uint32_t t, uint32_t& cursor) {
    while (cursor + 1 < a.nseg && t >= a.seg[cursor + 1].tile0) ++cursor;
    const AccSeg& sg = a.seg[cursor];
    TileAt r;
    r.si = cursor;
    r.e0 = static_cast<uint64_t>(t - sg.tile0) * kBulkTile;
    const uint64_t rem = sg.len - r.e0;
    r.cnt = rem < kBulkTile ? static_cast<uint32_t>(rem) : kBulkTile;
    return r;
}

template <typename Tin>
__global__ void __launch_bounds__(kBlock, 1) accumulate_bulk_kernel(const __grid_constant__ AccArgs a) {
    constexpr int S = BulkStages<Tin>::kS;
    constexpr uint32_t XB = kBulkTile * sizeof(Tin);
    constexpr uint32_t SB = kBulkTile * sizeof(float);
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* xs = smem;
    uint8_t* ss = smem + S * XB;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * (XB + SB));
    const uint32_t count =
        blockIdx.x < a.ntiles ? (a.ntiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&bars[s])) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const Tin* x0 = static_cast<const Tin*>(a.x[0]);
    const float w = a.w[0];
    uint32_t pcur = 0, ccur = 0;      // segment cursors of the producer and the consumers
    uint32_t issued = 0;

    auto issue = [&](uint32_t i) {    // thread 0 only
        const int s = static_cast<int>(i % S);
        const TileAt ta = tile_at(a, blockIdx.x + i * gridDim.x, pcur);
        const AccSeg& sg = a.seg[ta.si];
        const uint32_t bar = smem_addr(&bars[s]);
        const uint32_t n8 = ta.cnt / kVec;
        if (((a.vec_ok >> ta.si) & 1ull) && n8 > 0) {
            const uint32_t xb = n8 * kVec * sizeof(Tin);
            const uint32_t sb = sg.first ? 0u : n8 * kVec * sizeof(float);
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                         ::"r"(bar), "r"(xb + sb) : "memory");
            asm volatile(
                "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                ::"r"(smem_addr(xs + s * XB)), "l"(x0 + sg.x_off + ta.e0), "r"(xb), "r"(bar)
                : "memory");
            if (sb)
                asm volatile(
                    "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                    ::"r"(smem_addr(ss + s * SB)), "l"(a.acc + sg.acc_idx + ta.e0), "r"(sb), "r"(bar)
                    : "memory");
        } else {
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
        }
    };

    if (threadIdx.x == 0) {
        for (uint32_t i = 0; i < count && i < static_cast<uint32_t>(S); ++i) issue(i);
        issued = count < static_cast<uint32_t>(S) ? count : static_cast<uint32_t>(S);
    }
    uint32_t consumed = 0;
    bool ok = true;
    for (uint32_t i = 0; i < count; ++i) {
        const int s = static_cast<int>(i % S);
        ok = mbar_wait(smem_addr(&bars[s]), (i / S) & 1u);
        const TileAt ta = tile_at(a, blockIdx.x + i * gridDim.x, ccur);
        const AccSeg& sg = a.seg[ta.si];
        const bool first = sg.first != 0;
        const uint64_t xe0 = sg.x_off + ta.e0;
        float* g0 = a.acc + sg.acc_idx + ta.e0;
        const bool bulk = ((a.vec_ok >> ta.si) & 1ull) && ta.cnt >= static_cast<uint32_t>(kVec);
        const uint32_t n8 = bulk ? ta.cnt / kVec : 0;
        if (ok && bulk) {
            const Tin* xt = reinterpret_cast<const Tin*>(xs + s * XB);
            float* st = reinterpret_cast<float*>(ss + s * SB);
            for (uint32_t v = threadIdx.x; v < n8; v += kBlock) {
                float xv[8];
                if constexpr (sizeof(Tin) == 2) {
                    const uint4 q = reinterpret_cast<const uint4*>(xt)[v];
                    xv[0] = bf16_lo(q.x); xv[1] = bf16_hi(q.x);
                    xv[2] = bf16_lo(q.y); xv[3] = bf16_hi(q.y);
                    xv[4] = bf16_lo(q.z); xv[5] = bf16_hi(q.z);
                    xv[6] = bf16_lo(q.w); xv[7] = bf16_hi(q.w);
                } else {
                    const float4 p = reinterpret_cast<const float4*>(xt)[2 * v];
                    const float4 q = reinterpret_cast<const float4*>(xt)[2 * v + 1];
                    xv[0] = p.x; xv[1] = p.y; xv[2] = p.z; xv[3] = p.w;
                    xv[4] = q.x; xv[5] = q.y; xv[6] = q.z; xv[7] = q.w;
                }
                float4* sv = reinterpret_cast<float4*>(st) + 2 * v;
                float4 lo, hi;
                if (first) {
                    lo = make_float4(__fmul_rn(w, xv[0]), __fmul_rn(w, xv[1]), __fmul_rn(w, xv[2]),
                                     __fmul_rn(w, xv[3]));
                    hi = make_float4(__fmul_rn(w, xv[4]), __fmul_rn(w, xv[5]), __fmul_rn(w, xv[6]),
                                     __fmul_rn(w, xv[7]));
                } else {
                    lo = sv[0];
                    hi = sv[1];
                    lo.x = __fmaf_rn(w, xv[0], lo.x); lo.y = __fmaf_rn(w, xv[1], lo.y);
                    lo.z = __fmaf_rn(w, xv[2], lo.z); lo.w = __fmaf_rn(w, xv[3], lo.w);
                    hi.x = __fmaf_rn(w, xv[4], hi.x); hi.y = __fmaf_rn(w, xv[5], hi.y);
                    hi.z = __fmaf_rn(w, xv[6], hi.z); hi.w = __fmaf_rn(w, xv[7], hi.w);
                }
                sv[0] = lo;
                sv[1] = hi;
            }
            const uint32_t tail = ta.cnt - n8 * kVec;
            if (threadIdx.x < tail) {
                const uint32_t e = n8 * kVec + threadIdx.x;
                acc_one<Tin, 1>(a, xe0 + e, g0 + e, first);
            }
        } else if (ok) {
            for (uint32_t e = threadIdx.x; e < ta.cnt; e += kBlock) acc_one<Tin, 1>(a, xe0 + e, g0 + e, first);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        if (!__syncthreads_and(ok)) break;
        consumed = i + 1;
        if (threadIdx.x == 0) {
            if (n8 > 0)
                asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                             ::"l"(g0), "r"(smem_addr(ss + s * SB)), "r"(n8 * kVec * 4u) : "memory");
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            // refill the stage drained one iteration ago once its store has read it
            if (i >= 1 && i - 1 + S < count) {
                asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
                issue(i - 1 + S);
                issued = i + S;
            }
        }
    }
    if (threadIdx.x == 0) {
        if (consumed < count) {
            atomicOr(&g_device_error, kErrWaitTimeout);
            for (uint32_t j = consumed; j < issued; ++j)
                mbar_wait(smem_addr(&bars[j % S]), (j / S) & 1u);
        }
        asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    }
    __syncthreads();
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

// Base values of delta rounds (dtype_out), 8 at a time or one.
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

// q = sum / N (IEEE division); delta rounds then add server_lr * q to the base
// with one rounding (fma).
template <typename Tout, bool kApply>
__device__ __forceinline__ void fin_vec(const FinSeg& sg, uint64_t e, const float* s, float d,
                                        float lr) {
    const float4 lo = ld_v4f(s), hi = ld_v4f(s + 4);
    float q[8] = {__fdiv_rn(lo.x, d), __fdiv_rn(lo.y, d), __fdiv_rn(lo.z, d), __fdiv_rn(lo.w, d),
                  __fdiv_rn(hi.x, d), __fdiv_rn(hi.y, d), __fdiv_rn(hi.z, d), __fdiv_rn(hi.w, d)};
    if constexpr (kApply) {
        float b[8];
        LoadBase<Tout>::vec(sg.base, e, b);
#pragma unroll
        for (int i = 0; i < 8; ++i) q[i] = __fmaf_rn(lr, q[i], b[i]);
    }
    Store<Tout>::vec(sg.out, e, q);
}

template <typename Tout, bool kApply>
__device__ __forceinline__ void fin_one(const FinSeg& sg, uint64_t e, const float* s, float d,
                                        float lr) {
    float q = __fdiv_rn(*s, d);
    if constexpr (kApply) q = __fmaf_rn(lr, q, LoadBase<Tout>::one(sg.base, e));
    Store<Tout>::one(sg.out, e, q);
}

template <typename Tout, bool kApply>
__global__ void __launch_bounds__(kBlock) finalize_kernel(const FinSeg* __restrict__ segs,
                                                          uint32_t nseg, uint32_t ntiles,
                                                          const float* __restrict__ acc,
                                                          float lr) {
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
        // the sum side is always 128-byte aligned; the output (and base) may not be
        uintptr_t amask = reinterpret_cast<uintptr_t>(sg.out) + e0 * sizeof(Tout);
        if constexpr (kApply) amask |= reinterpret_cast<uintptr_t>(sg.base) + e0 * sizeof(Tout);
        if ((amask & 15u) == 0) {
            if (cnt == kTile) {
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const uint32_t v = threadIdx.x + u * kBlock;
                    fin_vec<Tout, kApply>(sg, e0 + v * kVec, s0 + v * kVec, d, lr);
                }
            } else {
                const uint32_t nv = cnt / kVec;
                for (uint32_t v = threadIdx.x; v < nv; v += kBlock)
                    fin_vec<Tout, kApply>(sg, e0 + v * kVec, s0 + v * kVec, d, lr);
                const uint32_t tail = cnt - nv * kVec;
                if (threadIdx.x < tail) {
                    const uint32_t e = nv * kVec + threadIdx.x;
                    fin_one<Tout, kApply>(sg, e0 + e, s0 + e, d, lr);
                }
            }
        } else {
            for (uint32_t e = threadIdx.x; e < cnt; e += kBlock)
                fin_one<Tout, kApply>(sg, e0 + e, s0 + e, d, lr);
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
constexpr size_t bulk_smem_bytes() {
    return static_cast<size_t>(BulkStages<Tin>::kS) * kBulkTile * (sizeof(Tin) + sizeof(float)) +
           static_cast<size_t>(BulkStages<Tin>::kS) * sizeof(uint64_t);
}

// Number the tiles of every segment for a kernel whose tile is `tile` elements.
bool number_tiles(AccArgs* a, uint64_t tile) {
    uint64_t t = 0;
    for (uint32_t i = 0; i < a->nseg; ++i) {
        a->seg[i].tile0 = static_cast<uint32_t>(t);
        t += (a->seg[i].len + tile - 1) / tile;
        if (t > 0xFFFFFFFFull) return false;
    }
    a->ntiles = static_cast<uint32_t>(t);
    return true;
}

template <typename Tin>
cudaError_t launch_bulk(const AccArgs& a, int ctas_per_sm, int sms, cudaStream_t stream) {
    if (a.ntiles == 0) return cudaSuccess;
    uint32_t cap = static_cast<uint32_t>(sms > 0 ? sms : 1) *
                   static_cast<uint32_t>(ctas_per_sm > 0 ? ctas_per_sm : 1);
    uint32_t grid = a.ntiles < cap ? a.ntiles : cap;
    accumulate_bulk_kernel<Tin><<<grid, kBlock, bulk_smem_bytes<Tin>(), stream>>>(a);
    return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_acc_j(const AccArgs& a, const LaunchShape& s, int in, cudaStream_t stream) {
    switch (a.J) {
        case 1: return launch_bulk<Tin>(a, s.bulk_ctas_per_sm[in], s.sms, stream);
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
    keep(cudaFuncSetAttribute(accumulate_bulk_kernel<float>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(bulk_smem_bytes<float>())));
    keep(cudaFuncSetAttribute(accumulate_bulk_kernel<uint16_t>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(bulk_smem_bytes<uint16_t>())));
    keep(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&s->bulk_ctas_per_sm[0], accumulate_bulk_kernel<float>,
                                                       kBlock, bulk_smem_bytes<float>()));
    keep(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&s->bulk_ctas_per_sm[1], accumulate_bulk_kernel<uint16_t>,
                                                       kBlock, bulk_smem_bytes<uint16_t>()));
    keep(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&s->fin_ctas_per_sm[0][0],
                                                       finalize_kernel<float, false>, kBlock, 0));
    keep(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&s->fin_ctas_per_sm[0][1],
                                                       finalize_kernel<uint16_t, false>, kBlock, 0));
    keep(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&s->fin_ctas_per_sm[1][0],
                                                       finalize_kernel<float, true>, kBlock, 0));
    keep(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&s->fin_ctas_per_sm[1][1],
                                                       finalize_kernel<uint16_t, true>, kBlock, 0));
    return r;
}

cudaError_t take_device_error(unsigned int* code) {
    unsigned int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(code, g_device_error, sizeof(unsigned int));
    if (e == cudaSuccess && *code != 0) e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero);
    return e;
}

cudaError_t launch_accumulate(const AccArgs& args, int dtype_in, const LaunchShape& s,
                              cudaStream_t stream) {
    AccArgs a = args;
    if (a.nseg == 0 || a.nseg > static_cast<uint32_t>(kMaxSegs)) return cudaErrorInvalidValue;
    if (!number_tiles(&a, a.J == 1 ? kBulkTile : kTile)) return cudaErrorInvalidValue;
    return dtype_in == 0 ? launch_acc_j<float>(a, s, 0, stream)
                         : launch_acc_j<uint16_t>(a, s, 1, stream);
}

cudaError_t launch_finalize(const FinSeg* segs, uint32_t nseg, uint32_t ntiles, int dtype_out,
                            const float* acc, bool apply, float server_lr, const LaunchShape& s,
                            cudaStream_t stream) {
    if (ntiles == 0 || nseg == 0) return cudaSuccess;
    int per = s.fin_ctas_per_sm[apply ? 1 : 0][dtype_out == 0 ? 0 : 1];
    uint32_t cap = static_cast<uint32_t>(s.sms > 0 ? s.sms : 1) *
                   static_cast<uint32_t>(per > 0 ? per : 1);
    uint32_t grid = ntiles < cap ? ntiles : cap;
    if (dtype_out == 0) {
        if (apply) finalize_kernel<float, true><<<grid, kBlock, 0, stream>>>(segs, nseg, ntiles, acc, server_lr);
        else finalize_kernel<float, false><<<grid, kBlock, 0, stream>>>(segs, nseg, ntiles, acc, server_lr);
    } else {
        if (apply) finalize_kernel<uint16_t, true><<<grid, kBlock, 0, stream>>>(segs, nseg, ntiles, acc, server_lr);
        else finalize_kernel<uint16_t, false><<<grid, kBlock, 0, stream>>>(segs, nseg, ntiles, acc, server_lr);
    }
    return cudaGetLastError();
}

}  // namespace fa
