// Device helpers shared by the aggregation kernels (internal to the library).
//
// Every kernel is a bandwidth-bound streaming pass on GB300 (152 SMs, HBM3e): loads and
// stores are 128-bit, pipelined kernels move tiles with bulk copies (cp.async.bulk, the
// 1-D form of TMA) into shared memory under mbarriers, and ragged tails (< 8 elements)
// or segments whose pointers are not 16-byte aligned use per-element accesses.
// Arithmetic: __fmul_rn / __fmaf_rn / __fdiv_rn so the compiler never contracts or
// reorders: the first contribution is a rounded product, every later one one fused
// multiply-add, in client order -- so every path yields the same bits.  Compensated
// mode (kComp) replaces each of these by the Dot2 step (see kernels.cuh), again in
// client order on every path.
// Every mbarrier wait is bounded; a timeout sets a bit in the caller's device error
// word (read by fa_sync), makes the CTA wait (bounded) for its own loads in flight,
// and return.
//
// Everything here has internal linkage: each kernel file compiles its own copy.
#pragma once

#include "kernels.cuh"
#include "tiles.hpp"

#include <cuda_bf16.h>

#include <algorithm>

namespace fa {

namespace {

constexpr uint32_t kMaxWaitSpins = 1u << 24;   // bound on every mbarrier wait
constexpr int kStages = 3;

// ----------------------------------------------------------------- memory helpers
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

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(a))) |
           (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(b))) << 16);
}

// One element of dtype Tin from global memory, read-only path.
template <typename Tin>
__device__ __forceinline__ float load_one(const Tin* p);

template <>
__device__ __forceinline__ float load_one<uint16_t>(const uint16_t* p) {
    uint16_t u;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(u) : "l"(p));
    return __uint_as_float(static_cast<uint32_t>(u) << 16);
}

template <>
__device__ __forceinline__ float load_one<float>(const float* p) {
    float f;
    asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(f) : "l"(p));
    return f;
}

// Eight elements of dtype Tin from a 16-byte aligned shared-memory vector slot.
template <typename Tin>
__device__ __forceinline__ void smem_vec8(const uint8_t* base, uint32_t v, float (&x)[8]) {
    if constexpr (sizeof(Tin) == 2) {
        const uint4 q = reinterpret_cast<const uint4*>(base)[v];
        x[0] = bf16_lo(q.x); x[1] = bf16_hi(q.x);
        x[2] = bf16_lo(q.y); x[3] = bf16_hi(q.y);
        x[4] = bf16_lo(q.z); x[5] = bf16_hi(q.z);
        x[6] = bf16_lo(q.w); x[7] = bf16_hi(q.w);
    } else {
        const float4 p = reinterpret_cast<const float4*>(base)[2 * v];
        const float4 q = reinterpret_cast<const float4*>(base)[2 * v + 1];
        x[0] = p.x; x[1] = p.y; x[2] = p.z; x[3] = p.w;
        x[4] = q.x; x[5] = q.y; x[6] = q.z; x[7] = q.w;
    }
}

// Eight fp32 values from / to a 32-byte shared-memory slot.
__device__ __forceinline__ void smem_ld8f(const uint8_t* base, uint32_t v, float (&r)[8]) {
    const float4 lo = reinterpret_cast<const float4*>(base)[2 * v];
    const float4 hi = reinterpret_cast<const float4*>(base)[2 * v + 1];
    r[0] = lo.x; r[1] = lo.y; r[2] = lo.z; r[3] = lo.w;
    r[4] = hi.x; r[5] = hi.y; r[6] = hi.z; r[7] = hi.w;
}

__device__ __forceinline__ void smem_st8f(uint8_t* base, uint32_t v, const float (&r)[8]) {
    reinterpret_cast<float4*>(base)[2 * v] = make_float4(r[0], r[1], r[2], r[3]);
    reinterpret_cast<float4*>(base)[2 * v + 1] = make_float4(r[4], r[5], r[6], r[7]);
}

// Store eight results of dtype Tout (RNE for bf16) to shared memory vector slot v.
template <typename Tout>
__device__ __forceinline__ void smem_store8(uint8_t* base, uint32_t v, const float (&q)[8]) {
    if constexpr (sizeof(Tout) == 2) {
        reinterpret_cast<uint4*>(base)[v] = make_uint4(pack_bf16(q[0], q[1]), pack_bf16(q[2], q[3]),
                                                       pack_bf16(q[4], q[5]), pack_bf16(q[6], q[7]));
    } else {
        smem_st8f(base, v, q);
    }
}

template <typename Tout>
__device__ __forceinline__ void store_one(void* out, uint64_t e, float q) {
    if constexpr (sizeof(Tout) == 2)
        static_cast<uint16_t*>(out)[e] = __bfloat16_as_ushort(__float2bfloat16_rn(q));
    else
        static_cast<float*>(out)[e] = q;
}

// Eight results of dtype Tout (RNE for bf16) to a 16-byte aligned global address.
template <typename Tout>
__device__ __forceinline__ void store8_global(void* out, uint64_t e, const float (&q)[8]) {
    if constexpr (sizeof(Tout) == 2) {
        st_v4u(static_cast<uint16_t*>(out) + e,
               make_uint4(pack_bf16(q[0], q[1]), pack_bf16(q[2], q[3]), pack_bf16(q[4], q[5]),
                          pack_bf16(q[6], q[7])));
    } else {
        float* p = static_cast<float*>(out) + e;
        st_v4f(p, make_float4(q[0], q[1], q[2], q[3]));
        st_v4f(p + 4, make_float4(q[4], q[5], q[6], q[7]));
    }
}

// ----------------------------------------------------------------- arithmetic
// The first contribution to an element and every later one.  Plain mode: a rounded
// product, then one fused multiply-add per client.  Compensated mode: the Dot2 step of
// Ogita, Rump and Oishi -- the product split exactly into its rounded value ph and its
// error pl (fma), ph added to hi by Knuth's TwoSum (sum s and exact error e), and the
// two errors summed into lo.
template <bool kComp>
__device__ __forceinline__ void contrib_first(float w, float x, float& hi, float& lo) {
    hi = __fmul_rn(w, x);
    if constexpr (kComp) lo = __fmaf_rn(w, x, -hi);
}

template <bool kComp>
__device__ __forceinline__ void contrib_add(float w, float x, float& hi, float& lo) {
    if constexpr (kComp) {
        const float ph = __fmul_rn(w, x);
        const float pl = __fmaf_rn(w, x, -ph);
        const float s = __fadd_rn(hi, ph);
        const float bv = __fsub_rn(s, hi);
        const float e = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bv)), __fsub_rn(ph, bv));
        lo = __fadd_rn(lo, __fadd_rn(e, pl));
        hi = s;
    } else {
        hi = __fmaf_rn(w, x, hi);
    }
}

// q = (s + s_lo) / N with N = d.hi + d.lo.  When N is exact in fp32 (d.lo == 0) and there
// is no lo part, this is one IEEE division.  Otherwise q1 = s / d.hi is corrected by the
// remainder: r = s - q1 * d.hi is exact (fma), s_lo joins it, q1 * d.lo leaves it, and
// q = q1 + r / d.hi.  A non-finite q1 (inf or NaN sums) is returned as it is.
template <bool kComp>
__device__ __forceinline__ float quotient(float s, float s_lo, const Divisor& d) {
    if (!kComp && d.lo == 0.0f) return __fdiv_rn(s, d.hi);
    const float q1 = __fdiv_rn(s, d.hi);
    if (!isfinite(q1)) return q1;
    float r = __fmaf_rn(-q1, d.hi, s);
    if constexpr (kComp) r = __fadd_rn(r, s_lo);
    r = __fmaf_rn(-q1, d.lo, r);
    return __fadd_rn(q1, __fmul_rn(r, d.rcp));
}

// The value to store for an output of dtype Tout.  Compensated mode with a bf16 output:
// the quotient q above plus the exact error e of its last rounding (Fast2Sum, since the
// correction is smaller than q1), and where q's bits below bf16 precision are exactly a
// tie (low 16 bits 0x8000) q is moved one fp32 ulp toward q + e -- so the RNE cast rounds
// the quotient's full value, not its fp32 rounding, to bf16 (no double rounding).  The
// fp32 output and the default mode store q itself.
template <bool kComp, typename Tout>
__device__ __forceinline__ float quotient_out(float s, float s_lo, const Divisor& d) {
    if constexpr (kComp && sizeof(Tout) == 2) {
        const float q1 = __fdiv_rn(s, d.hi);
        if (!isfinite(q1)) return q1;
        float r = __fmaf_rn(-q1, d.hi, s);
        r = __fadd_rn(r, s_lo);
        r = __fmaf_rn(-q1, d.lo, r);
        const float c = __fmul_rn(r, d.rcp);
        const float q = __fadd_rn(q1, c);
        const float e = __fadd_rn(__fsub_rn(q1, q), c);
        uint32_t u = __float_as_uint(q);
        if ((u & 0xFFFFu) == 0x8000u && e != 0.0f) u = ((e > 0.0f) == (q > 0.0f)) ? u + 1u : u - 1u;
        return __uint_as_float(u);
    } else {
        return quotient<kComp>(s, s_lo, d);
    }
}

// ----------------------------------------------------------------- pipeline helpers
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

__device__ __forceinline__ void mbar_init(uint64_t* bars, int n) {
    for (int s = 0; s < n; ++s)
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&bars[s])) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void bulk_load(void* dst_smem, const void* src, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_addr(dst_smem)), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void bulk_store(void* dst, const void* src_smem, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                 ::"l"(dst), "r"(smem_addr(src_smem)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

struct TileAt {
    uint32_t si;
    uint64_t e0;
    uint32_t cnt;
};

// Tile t (numbered across segments by tile0) with `tile` elements per tile; the cursor
// only moves forward because each CTA visits its tiles in increasing order.
template <typename Seg>
__device__ __forceinline__ TileAt tile_at(const Seg* segs, uint32_t nseg, uint32_t t,
                                          uint32_t tile, uint32_t& cursor) {
    while (cursor + 1 < nseg && t >= segs[cursor + 1].tile0) ++cursor;
    const Seg& sg = segs[cursor];
    TileAt r;
    r.si = cursor;
    r.e0 = static_cast<uint64_t>(t - sg.tile0) * tile;
    const uint64_t rem = sg.len - r.e0;
    r.cnt = rem < tile ? static_cast<uint32_t>(rem) : tile;
    return r;
}

// The bounded end of a pipelined kernel: after an early exit (a wait gave up) the
// elected thread flags the error and waits for the loads it still has in flight;
// in every case it waits for its bulk stores before the CTA leaves.
__device__ __forceinline__ void pipeline_drain(uint64_t* bars, uint32_t consumed,
                                               uint32_t issued, uint32_t count,
                                               unsigned int* err) {
    if (consumed < count) {
        atomicOr(err, kErrWaitTimeout);
        for (uint32_t j = consumed; j < issued; ++j)
            mbar_wait(smem_addr(&bars[j % kStages]), (j / kStages) & 1u);
    }
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ----------------------------------------------------------------- plain global loads
// Coherent loads (no read-only path): the form for host memory the device reads in
// place, and for the running sum.
__device__ __forceinline__ uint4 ld_plain_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

template <typename Tin>
__device__ __forceinline__ float load_plain(const Tin* p);

template <>
__device__ __forceinline__ float load_plain<uint16_t>(const uint16_t* p) {
    uint16_t u;
    asm volatile("ld.global.u16 %0, [%1];" : "=h"(u) : "l"(p));
    return __uint_as_float(static_cast<uint32_t>(u) << 16);
}

template <>
__device__ __forceinline__ float load_plain<float>(const float* p) {
    float f;
    asm volatile("ld.global.f32 %0, [%1];" : "=f"(f) : "l"(p));
    return f;
}

// Eight elements of dtype Tin from a 16-byte aligned global address.
template <typename Tin>
__device__ __forceinline__ void plain_vec8(const Tin* p, float (&x)[8]) {
    if constexpr (sizeof(Tin) == 2) {
        const uint4 q = ld_plain_v4(p);
        x[0] = bf16_lo(q.x); x[1] = bf16_hi(q.x);
        x[2] = bf16_lo(q.y); x[3] = bf16_hi(q.y);
        x[4] = bf16_lo(q.z); x[5] = bf16_hi(q.z);
        x[6] = bf16_lo(q.w); x[7] = bf16_hi(q.w);
    } else {
        const uint4 a = ld_plain_v4(p);
        const uint4 b = ld_plain_v4(p + 4);
        x[0] = __uint_as_float(a.x); x[1] = __uint_as_float(a.y);
        x[2] = __uint_as_float(a.z); x[3] = __uint_as_float(a.w);
        x[4] = __uint_as_float(b.x); x[5] = __uint_as_float(b.y);
        x[6] = __uint_as_float(b.z); x[7] = __uint_as_float(b.w);
    }
}

__device__ __forceinline__ void ld8f(const float* p, float (&r)[8]) {
    const float4 lo = ld_v4f(p), hi = ld_v4f(p + 4);
    r[0] = lo.x; r[1] = lo.y; r[2] = lo.z; r[3] = lo.w;
    r[4] = hi.x; r[5] = hi.y; r[6] = hi.z; r[7] = hi.w;
}

__device__ __forceinline__ void st8f(float* p, const float (&r)[8]) {
    st_v4f(p, make_float4(r[0], r[1], r[2], r[3]));
    st_v4f(p + 4, make_float4(r[4], r[5], r[6], r[7]));
}

// ----------------------------------------------------------------- warp-specialised reduces
// The J-client and subset reduce kernels: warps 0-7 compute, one lane of warp 8 moves
// data; one CTA per SM with kStages stages of at most kReduceStageBytes each.
constexpr int kReduceWarps = kBlock / 32;               // compute warps
constexpr int kReduceThreads = kBlock + 32;             // + one producer warp
constexpr size_t kReduceSmemBytes =
    static_cast<size_t>(kStages) * kReduceStageBytes + 2 * kStages * sizeof(uint64_t);

// ----------------------------------------------------------------- launch helpers (host)
// Launch as a programmatic dependent of the previous kernel on the stream: its launch
// and prologue overlap that kernel's tail (the kernel itself waits, with
// griddepcontrol.wait, before reading or writing global memory).
template <typename Arg>
cudaError_t launch_dependent(void (*kern)(Arg), uint32_t grid, uint32_t block, size_t smem,
                             cudaStream_t stream, const Arg& arg) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, arg);
}

}  // namespace

}  // namespace fa
