// Aggregation kernels for sm_103a (see kernels.cuh).
//
// GB300: 152 SMs, HBM3e.  Every kernel is a bandwidth-bound streaming pass:
//  - accumulate_bulk_kernel (one client per launch, the streaming hot path) and
//    reduce_bulk_kernel (J resident clients per launch) move their tiles with bulk
//    copies (cp.async.bulk, the 1-D form of TMA) through a three-stage shared-memory
//    pipeline: one elected thread arms a stage's mbarrier with the byte count and
//    issues the loads, all threads compute in shared memory, the elected thread
//    writes the result tile back with one bulk store, and a stage is refilled once
//    that store has read it.  Persistent grids, one or two CTAs per SM, keep about
//    150-200 KB of copies in flight per SM -- a timed sweep of tile sizes, stage
//    counts and direct-load variants on GB300 chose these shapes;
//  - accumulate_direct_kernel reads its input in place with plain loads: the form for
//    pinned host memory read over the NVLink-C2C link, where the link sets the pace;
//  - finalize_kernel reads the sum with 128-bit loads and writes 128-bit stores;
//  - ragged tails (< 8 elements) and segments whose pointers are not 16-byte
//    aligned use direct per-element loads and stores.
// Arithmetic: __fmul_rn / __fmaf_rn / __fdiv_rn so the compiler never contracts or
// reorders: the first contribution is a rounded product, every later one one fused
// multiply-add, in client order -- so every path yields the same bits.  Compensated
// mode (kComp) replaces each of these by the Dot2 step (see kernels.cuh), again in
// client order on every path.
// Every mbarrier wait is bounded; a timeout sets a bit in the caller's device error
// word (read by fa_sync), makes the CTA wait (bounded) for its own loads in flight,
// and return.
#include "kernels.cuh"

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

// ----------------------------------------------------------------- streaming accumulate
// One element through global memory (ragged tails, unaligned segments).
template <typename Tin, bool kComp>
__device__ __forceinline__ void acc_one(const Tin* x, float w, float* s, float* sl, bool first) {
    const float xv = load_one<Tin>(x);
    float hi, lo = 0.0f;
    if (first) {
        contrib_first<kComp>(w, xv, hi, lo);
    } else {
        hi = *s;
        if constexpr (kComp) lo = *sl;
        contrib_add<kComp>(w, xv, hi, lo);
    }
    *s = hi;
    if constexpr (kComp) *sl = lo;
}

template <bool kComp>
__host__ __device__ constexpr uint32_t bulk_tile() {
    return static_cast<uint32_t>(kComp ? kBulkTileComp : kBulkTile);
}

template <typename Tin, bool kComp>
constexpr size_t bulk_smem_bytes() {
    return static_cast<size_t>(kStages) * bulk_tile<kComp>() *
               (sizeof(Tin) + sizeof(float) * (kComp ? 2 : 1)) +
           static_cast<size_t>(kStages) * sizeof(uint64_t);
}

// Stage = input tile (T x Tin) + sum tile (T x fp32) [+ lo tile (T x fp32), compensated
// mode]: 48 KB for bf16 and 64 KB for fp32 input (T = 8192), 60 / 72 KB compensated
// (T = 6144); one CTA per SM.
template <typename Tin, bool kComp>
__global__ void __launch_bounds__(kBlock, 1) accumulate_bulk_kernel(const __grid_constant__ AccArgs a) {
    constexpr uint32_t T = bulk_tile<kComp>();
    constexpr uint32_t XB = T * sizeof(Tin);
    constexpr uint32_t SB = T * sizeof(float);
    constexpr uint32_t NS = kComp ? 2u : 1u;    // sum tiles per stage
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* xs = smem;
    uint8_t* ss = smem + kStages * XB;           // hi tiles, then (kComp) lo tiles
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * (XB + NS * SB));
    const uint32_t count =
        blockIdx.x < a.ntiles ? (a.ntiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    if (threadIdx.x == 0) mbar_init(bars, kStages);
    __syncthreads();
    // launched as a programmatic dependent: set-up above overlaps the previous kernel's
    // tail; nothing in global memory is touched before that kernel has completed
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const float w = a.w[0];
    uint32_t pcur = 0, ccur = 0;      // segment cursors of the producer and the consumers
    uint32_t issued = 0;

    auto issue = [&](uint32_t i) {    // thread 0 only
        const int s = static_cast<int>(i % kStages);
        const TileAt ta = tile_at(a.seg, a.nseg, blockIdx.x + i * gridDim.x, T, pcur);
        const AccSeg& sg = a.seg[ta.si];
        const uint32_t bar = smem_addr(&bars[s]);
        const uint32_t n8 = ta.cnt / kVec;
        if (((a.vec_ok >> ta.si) & 1ull) && n8 > 0) {
            const uint32_t xb = n8 * kVec * sizeof(Tin);
            const uint32_t sb = sg.first ? 0u : n8 * kVec * sizeof(float);
            mbar_expect(bar, xb + NS * sb);
            bulk_load(xs + s * XB, static_cast<const Tin*>(sg.x) + sg.x_off + ta.e0, xb, bar);
            if (sb) {
                bulk_load(ss + s * SB, a.acc + sg.acc_idx + ta.e0, sb, bar);
                if constexpr (kComp)
                    bulk_load(ss + (kStages + s) * SB, a.acc_lo + sg.acc_idx + ta.e0, sb, bar);
            }
        } else {
            mbar_arrive(bar);
        }
    };

    if (threadIdx.x == 0) {
        for (uint32_t i = 0; i < count && i < static_cast<uint32_t>(kStages); ++i) issue(i);
        issued = count < static_cast<uint32_t>(kStages) ? count : static_cast<uint32_t>(kStages);
    }
    uint32_t consumed = 0;
    for (uint32_t i = 0; i < count; ++i) {
        const int s = static_cast<int>(i % kStages);
        const bool expire = i == 0 && (a.debug & kDebugFirstWaitExpires) != 0;
        const bool ok = !expire && mbar_wait(smem_addr(&bars[s]), (i / kStages) & 1u);
        const TileAt ta = tile_at(a.seg, a.nseg, blockIdx.x + i * gridDim.x, T, ccur);
        const AccSeg& sg = a.seg[ta.si];
        const bool first = sg.first != 0;
        const Tin* xg = static_cast<const Tin*>(sg.x) + sg.x_off + ta.e0;   // tile in global memory
        float* g0 = a.acc + sg.acc_idx + ta.e0;
        float* l0 = kComp ? a.acc_lo + sg.acc_idx + ta.e0 : nullptr;
        const bool bulk = ((a.vec_ok >> ta.si) & 1ull) && ta.cnt >= static_cast<uint32_t>(kVec);
        const uint32_t n8 = bulk ? ta.cnt / kVec : 0;
        if (ok && bulk) {
            const uint8_t* xt = xs + s * XB;
            uint8_t* st = ss + s * SB;
            uint8_t* lt = ss + (kStages + s) * SB;
            for (uint32_t v = threadIdx.x; v < n8; v += kBlock) {
                float xv[8], hi[8], lo[8];
                smem_vec8<Tin>(xt, v, xv);
                if (first) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) contrib_first<kComp>(w, xv[e], hi[e], lo[e]);
                } else {
                    smem_ld8f(st, v, hi);
                    if constexpr (kComp) smem_ld8f(lt, v, lo);
#pragma unroll
                    for (int e = 0; e < 8; ++e) contrib_add<kComp>(w, xv[e], hi[e], lo[e]);
                }
                smem_st8f(st, v, hi);
                if constexpr (kComp) smem_st8f(lt, v, lo);
            }
            const uint32_t tail = ta.cnt - n8 * kVec;
            if (threadIdx.x < tail) {
                const uint32_t e = n8 * kVec + threadIdx.x;
                acc_one<Tin, kComp>(xg + e, w, g0 + e, kComp ? l0 + e : nullptr, first);
            }
        } else if (ok) {
            for (uint32_t e = threadIdx.x; e < ta.cnt; e += kBlock)
                acc_one<Tin, kComp>(xg + e, w, g0 + e, kComp ? l0 + e : nullptr, first);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        if (!__syncthreads_and(ok)) break;
        consumed = i + 1;
        if (threadIdx.x == 0) {
            if (n8 > 0) {
                bulk_store(g0, ss + s * SB, n8 * kVec * 4u);
                if constexpr (kComp) bulk_store(l0, ss + (kStages + s) * SB, n8 * kVec * 4u);
            }
            bulk_commit();
            // refill the stage drained one iteration ago once its store has read it
            if (i >= 1 && i - 1 + kStages < count) {
                asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
                issue(i - 1 + kStages);
                issued = i + kStages;
            }
        }
    }
    if (threadIdx.x == 0) pipeline_drain(bars, consumed, issued, count, a.err);
    __syncthreads();
}

// ----------------------------------------------------------------- direct accumulate
// Input read in place with plain coherent loads (no bulk copies, no read-only path),
// the form for pinned host memory the device reads over the NVLink-C2C link: the
// link moves about 0.2 TB/s against 6.7 TB/s of HBM, so the sum's read-modify-write
// in HBM is not the limit and no shared-memory staging is needed.  Tiles of
// kDirectTile elements, one 8-element vector per thread; many CTAs per SM keep enough
// loads in flight to cover the link's latency.
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

template <typename Tin, bool kComp>
__global__ void __launch_bounds__(kBlock) accumulate_direct_kernel(const __grid_constant__ AccArgs a) {
    static_assert(kDirectTile == kBlock * kVec, "one vector per thread per tile");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const float w = a.w[0];
    uint32_t cur = 0;
    for (uint32_t t = blockIdx.x; t < a.ntiles; t += gridDim.x) {
        const TileAt ta = tile_at(a.seg, a.nseg, t, kDirectTile, cur);
        const AccSeg& sg = a.seg[ta.si];
        const bool first = sg.first != 0;
        const Tin* xt = static_cast<const Tin*>(sg.x) + sg.x_off + ta.e0;
        float* g = a.acc + sg.acc_idx + ta.e0;
        float* gl = kComp ? a.acc_lo + sg.acc_idx + ta.e0 : nullptr;
        const uint32_t n8 = ((a.vec_ok >> ta.si) & 1ull) ? ta.cnt / kVec : 0u;
        if (threadIdx.x < n8) {
            float xv[8], hi[8], lo[8];
            plain_vec8<Tin>(xt + threadIdx.x * kVec, xv);
            float* gp = g + threadIdx.x * kVec;
            if (first) {
#pragma unroll
                for (int e = 0; e < 8; ++e) contrib_first<kComp>(w, xv[e], hi[e], lo[e]);
            } else {
                ld8f(gp, hi);
                if constexpr (kComp) ld8f(gl + threadIdx.x * kVec, lo);
#pragma unroll
                for (int e = 0; e < 8; ++e) contrib_add<kComp>(w, xv[e], hi[e], lo[e]);
            }
            st8f(gp, hi);
            if constexpr (kComp) st8f(gl + threadIdx.x * kVec, lo);
        }
        for (uint32_t e = n8 * kVec + threadIdx.x; e < ta.cnt; e += kBlock) {
            const float xv = load_plain<Tin>(xt + e);
            float hi, lo = 0.0f;
            if (first) {
                contrib_first<kComp>(w, xv, hi, lo);
            } else {
                hi = g[e];
                if constexpr (kComp) lo = gl[e];
                contrib_add<kComp>(w, xv, hi, lo);
            }
            g[e] = hi;
            if constexpr (kComp) gl[e] = lo;
        }
    }
}

// ----------------------------------------------------------------- J-client reduce
// Stage = J input tiles (T x Tin each) [+ sum tile (T x fp32), and in compensated mode a
// lo tile: sum mode, or final mode reading earlier contributions] [+ output tile
// (T x Tout): final mode]; T is chosen on the host so a stage fits kReduceStageBytes
// (one CTA per SM, three stages: about 200 KB of copies in flight).  Sum mode writes the
// running sum back; final mode divides by the segment's divisor and rounds to Tout.
// kJ > 0 fixes the client count at compile time so the per-client loop unrolls (J = 16
// and 8); kJ = 0 reads it from the arguments.
template <bool kFinal, bool kComp, typename Tin, typename Tout>
__host__ __device__ constexpr uint32_t reduce_elem_bytes(uint32_t J, bool has_sum) {
    return J * static_cast<uint32_t>(sizeof(Tin)) + (has_sum ? (kComp ? 8u : 4u) : 0u) +
           (kFinal ? static_cast<uint32_t>(sizeof(Tout)) : 0u);
}

template <typename Tin, typename Tout, bool kFinal, bool kComp>
__device__ __forceinline__ void red_one(const RedArgs& a, const RedSeg& sg, uint64_t e, uint32_t J) {
    // element e of the segment, through global memory
    const uint64_t xe = sg.x_off + e;
    float r, rl = 0.0f;
    uint32_t j0 = 0;
    if (sg.read_sum) {
        r = a.acc[sg.acc_idx + e];
        if constexpr (kComp) rl = a.acc_lo[sg.acc_idx + e];
    } else {
        contrib_first<kComp>(a.w[0], load_one<Tin>(static_cast<const Tin*>(a.x[0]) + xe), r, rl);
        j0 = 1;
    }
    for (uint32_t j = j0; j < J; ++j)
        contrib_add<kComp>(a.w[j], load_one<Tin>(static_cast<const Tin*>(a.x[j]) + xe), r, rl);
    if constexpr (kFinal) {
        store_one<Tout>(sg.out, e, quotient_out<kComp, Tout>(r, rl, sg.div));
    } else {
        a.acc[sg.acc_idx + e] = r;
        if constexpr (kComp) a.acc_lo[sg.acc_idx + e] = rl;
    }
}

// Warp-specialised: warps 0-7 compute, warp 8 (one lane) moves data.  Per stage two
// mbarriers: `full` (the producer arms it with the byte count of the stage's bulk loads)
// and `done` (each compute warp arrives once it has finished the stage).  The producer
// stores a stage's result tile when `done` completes and refills the stage once that
// store has read it; the compute warps never wait for producer work except data.
constexpr int kReduceWarps = kBlock / 32;               // compute warps
constexpr int kReduceThreads = kBlock + 32;             // + one producer warp

template <typename Tin, typename Tout, bool kFinal, int kJ, bool kComp>
__global__ void __launch_bounds__(kReduceThreads, 1) reduce_bulk_kernel(const __grid_constant__ RedArgs a) {
    const uint32_t T = a.tile;
    const uint32_t J = kJ > 0 ? static_cast<uint32_t>(kJ) : a.J;
    const uint32_t XB = T * sizeof(Tin);
    const uint32_t SB = a.has_sum ? T * static_cast<uint32_t>(sizeof(float)) : 0u;
    const uint32_t NS = kComp ? 2u : 1u;                  // sum tiles (hi [, lo])
    const uint32_t stage = T * reduce_elem_bytes<kFinal, kComp, Tin, Tout>(J, a.has_sum != 0);
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * stage);
    uint64_t* done = full + kStages;
    const uint32_t count =
        blockIdx.x < a.ntiles ? (a.ntiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&full[s])) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(&done[s])),
                         "r"(kReduceWarps) : "memory");
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    asm volatile("griddepcontrol.wait;" ::: "memory");   // see accumulate_bulk_kernel

    if (threadIdx.x >= static_cast<unsigned>(kBlock)) {
        // ------------------------------------------------------------ producer
        if (threadIdx.x != static_cast<unsigned>(kBlock)) return;
        uint32_t cur = 0, scur = 0;     // segment cursors for loads and for stores
        bool ok = true;
        auto store = [&](uint32_t i) {  // result tile of tile i, stage i % kStages
            const uint32_t s = i % kStages;
            const TileAt ta = tile_at(a.seg, a.nseg, blockIdx.x + i * gridDim.x, T, scur);
            const RedSeg& sg = a.seg[ta.si];
            const uint32_t n8 = (((a.vec_ok >> ta.si) & 1ull) && ta.cnt >= static_cast<uint32_t>(kVec))
                                    ? ta.cnt / kVec : 0u;
            if (n8 == 0) return;
            uint8_t* st = smem + s * stage;
            if constexpr (kFinal) {
                bulk_store(static_cast<Tout*>(sg.out) + ta.e0, st + J * XB + NS * SB,
                           n8 * kVec * sizeof(Tout));
            } else {
                bulk_store(a.acc + sg.acc_idx + ta.e0, st + J * XB, n8 * kVec * 4u);
                if constexpr (kComp)
                    bulk_store(a.acc_lo + sg.acc_idx + ta.e0, st + J * XB + SB, n8 * kVec * 4u);
            }
        };
        uint32_t stored = 0;
        for (uint32_t j = 0; j < count && ok; ++j) {
            const uint32_t s = j % kStages;
            if (j >= static_cast<uint32_t>(kStages)) {
                // stage s holds tile j - kStages: wait for the compute warps, store it,
                // and wait until the store has read the stage before refilling it
                ok = mbar_wait(smem_addr(&done[s]), ((j / kStages) - 1) & 1u);
                if (!ok) break;
                store(j - kStages);
                bulk_commit();
                stored = j - kStages + 1;
                asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
            }
            const TileAt ta = tile_at(a.seg, a.nseg, blockIdx.x + j * gridDim.x, T, cur);
            const RedSeg& sg = a.seg[ta.si];
            const uint32_t bar = smem_addr(&full[s]);
            const uint32_t n8 = ta.cnt / kVec;
            if (((a.vec_ok >> ta.si) & 1ull) && n8 > 0) {
                const uint32_t xb = n8 * kVec * sizeof(Tin);
                const uint32_t sb = sg.read_sum ? n8 * kVec * 4u : 0u;
                mbar_expect(bar, J * xb + NS * sb);
                uint8_t* st = smem + s * stage;
#pragma unroll
                for (uint32_t jj = 0; jj < (kJ > 0 ? static_cast<uint32_t>(kJ) : static_cast<uint32_t>(kMaxBatch)); ++jj) {
                    if (kJ == 0 && jj >= J) break;
                    bulk_load(st + jj * XB, static_cast<const Tin*>(a.x[jj]) + sg.x_off + ta.e0, xb, bar);
                }
                if (sb) {
                    bulk_load(st + J * XB, a.acc + sg.acc_idx + ta.e0, sb, bar);
                    if constexpr (kComp) bulk_load(st + J * XB + SB, a.acc_lo + sg.acc_idx + ta.e0, sb, bar);
                }
            } else {
                mbar_arrive(bar);
            }
        }
        // the last stages: wait for the compute warps and store
        for (uint32_t i = stored; i < count && ok; ++i) {
            ok = mbar_wait(smem_addr(&done[i % kStages]), (i / kStages) & 1u);
            if (ok) {
                store(i);
                bulk_commit();
            }
        }
        if (!ok) {
            // a wait gave up: flag it, and let every load issued so far land before
            // the CTA's shared memory can be released
            atomicOr(a.err, kErrWaitTimeout);
            const uint32_t last = count < stored + kStages ? count : stored + kStages;
            for (uint32_t i = stored; i < last; ++i)
                mbar_wait(smem_addr(&full[i % kStages]), (i / kStages) & 1u);
        }
        asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
        return;
    }

    // ---------------------------------------------------------------- compute warps
    uint32_t ccur = 0;
    const uint32_t lane = threadIdx.x & 31u;
    for (uint32_t i = 0; i < count; ++i) {
        const uint32_t s = i % kStages;
        if (!mbar_wait(smem_addr(&full[s]), (i / kStages) & 1u)) {
            atomicOr(a.err, kErrWaitTimeout);
            break;
        }
        const TileAt ta = tile_at(a.seg, a.nseg, blockIdx.x + i * gridDim.x, T, ccur);
        const RedSeg& sg = a.seg[ta.si];
        const bool bulk = ((a.vec_ok >> ta.si) & 1ull) && ta.cnt >= static_cast<uint32_t>(kVec);
        const uint32_t n8 = bulk ? ta.cnt / kVec : 0;
        uint8_t* st = smem + s * stage;
        uint8_t* sum = st + J * XB;                           // hi tile, then (kComp) lo tile
        uint8_t* res = st + J * XB + NS * SB;                 // final mode output tile
        if (bulk) {
            for (uint32_t v = threadIdx.x; v < n8; v += kBlock) {
                float r[8], rl[8];
                {
                    float xv[8];
                    smem_vec8<Tin>(st, v, xv);
                    if (sg.read_sum) {          // client 0 joins the earlier contributions
                        smem_ld8f(sum, v, r);
                        if constexpr (kComp) smem_ld8f(sum + SB, v, rl);
#pragma unroll
                        for (int e = 0; e < 8; ++e) contrib_add<kComp>(a.w[0], xv[e], r[e], rl[e]);
                    } else {                    // client 0 starts the sum
#pragma unroll
                        for (int e = 0; e < 8; ++e) contrib_first<kComp>(a.w[0], xv[e], r[e], rl[e]);
                    }
                }
#pragma unroll
                for (uint32_t j = 1; j < (kJ > 0 ? static_cast<uint32_t>(kJ) : static_cast<uint32_t>(kMaxBatch)); ++j) {
                    if (kJ == 0 && j >= J) break;
                    float xv[8];
                    smem_vec8<Tin>(st + j * XB, v, xv);
                    const float wj = a.w[j];
#pragma unroll
                    for (int e = 0; e < 8; ++e) contrib_add<kComp>(wj, xv[e], r[e], rl[e]);
                }
                if constexpr (kFinal) {
                    const Divisor d = sg.div;
#pragma unroll
                    for (int e = 0; e < 8; ++e) r[e] = quotient_out<kComp, Tout>(r[e], rl[e], d);
                    smem_store8<Tout>(res, v, r);
                } else {
                    smem_st8f(sum, v, r);
                    if constexpr (kComp) smem_st8f(sum + SB, v, rl);
                }
            }
            const uint32_t tail = ta.cnt - n8 * kVec;
            if (threadIdx.x < tail) red_one<Tin, Tout, kFinal, kComp>(a, sg, ta.e0 + n8 * kVec + threadIdx.x, J);
        } else {
            for (uint32_t e = threadIdx.x; e < ta.cnt; e += kBlock)
                red_one<Tin, Tout, kFinal, kComp>(a, sg, ta.e0 + e, J);
        }
        // shared-memory results become visible to the bulk store (async proxy); the
        // warp's lane 0 then reports the stage done
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&done[s]));
    }
}

constexpr size_t kReduceSmemBytes =
    static_cast<size_t>(kStages) * kReduceStageBytes + 2 * kStages * sizeof(uint64_t);

// ----------------------------------------------------------------- subset reduce
// A round of client key subsets straight to the output: one segment per key, each with
// its own reporters (GathSeg / GathSrc tables in device memory) applied in table order --
// the final mode of reduce_bulk_kernel with per-segment inputs and weights, warp-
// specialised the same way (warps 0-7 compute, one producer lane issues a stage's bulk
// loads and stores its output tile).  Stage = jmax input tiles + one output tile; a
// segment with fewer reporters leaves part of the stage unused.  A plain launch: its
// tables are uploaded on the stream just before it.
template <typename Tin, typename Tout, bool kComp>
__device__ __forceinline__ void gath_one(const GathArgs& a, const GathSeg& sg, uint64_t e) {
    const GathSrc* src = a.src + sg.src0;
    float r, rl = 0.0f;
    contrib_first<kComp>(src[0].w, load_one<Tin>(static_cast<const Tin*>(src[0].x) + e), r, rl);
    for (uint32_t j = 1; j < sg.J; ++j)
        contrib_add<kComp>(src[j].w, load_one<Tin>(static_cast<const Tin*>(src[j].x) + e), r, rl);
    store_one<Tout>(sg.out, e, quotient_out<kComp, Tout>(r, rl, sg.div));
}

// The segment holding tile t: a binary search over tile0 (the tables live in global
// memory, so a walk from segment 0 would be a long chain of dependent loads).
__device__ __forceinline__ uint32_t gath_seg_of(const GathSeg* segs, uint32_t nseg, uint32_t t) {
    uint32_t lo = 0, hi = nseg;              // the answer is in [lo, hi)
    while (hi - lo > 1) {
        const uint32_t mid = (lo + hi) / 2;
        if (segs[mid].tile0 <= t) lo = mid; else hi = mid;
    }
    return lo;
}

template <typename Tin, typename Tout, bool kComp>
__global__ void __launch_bounds__(kReduceThreads, 1) reduce_gather_kernel(const __grid_constant__ GathArgs a) {
    const uint32_t T = a.tile;
    const uint32_t XB = T * sizeof(Tin);
    const uint32_t stage = T * (a.jmax * static_cast<uint32_t>(sizeof(Tin)) + static_cast<uint32_t>(sizeof(Tout)));
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * stage);
    uint64_t* done = full + kStages;
    // each CTA takes a contiguous run of tiles, so its walk through the segment table
    // moves by at most one entry per tile
    const uint32_t q = a.ntiles / gridDim.x, rmd = a.ntiles % gridDim.x;
    const uint32_t count = q + (blockIdx.x < rmd ? 1u : 0u);
    const uint32_t first = blockIdx.x * q + (blockIdx.x < rmd ? blockIdx.x : rmd);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&full[s])) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(&done[s])),
                         "r"(kReduceWarps) : "memory");
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const uint32_t seg0 = count ? gath_seg_of(a.segs, a.nseg, first) : 0u;

    if (threadIdx.x >= static_cast<unsigned>(kBlock)) {
        // ------------------------------------------------------------ producer
        if (threadIdx.x != static_cast<unsigned>(kBlock)) return;
        uint32_t cur = seg0, scur = seg0;
        bool ok = true;
        auto store = [&](uint32_t i) {
            const TileAt ta = tile_at(a.segs, a.nseg, first + i, T, scur);
            const GathSeg sg = a.segs[ta.si];
            const uint32_t n8 = (sg.vec_ok && ta.cnt >= static_cast<uint32_t>(kVec)) ? ta.cnt / kVec : 0u;
            if (n8 == 0) return;
            bulk_store(static_cast<Tout*>(sg.out) + ta.e0, smem + (i % kStages) * stage + a.jmax * XB,
                       n8 * kVec * sizeof(Tout));
        };
        uint32_t stored = 0;
        for (uint32_t j = 0; j < count && ok; ++j) {
            const uint32_t s = j % kStages;
            if (j >= static_cast<uint32_t>(kStages)) {
                ok = mbar_wait(smem_addr(&done[s]), ((j / kStages) - 1) & 1u);
                if (!ok) break;
                store(j - kStages);
                bulk_commit();
                stored = j - kStages + 1;
                asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
            }
            const TileAt ta = tile_at(a.segs, a.nseg, first + j, T, cur);
            const GathSeg sg = a.segs[ta.si];
            const uint32_t bar = smem_addr(&full[s]);
            const uint32_t n8 = ta.cnt / kVec;
            if (sg.vec_ok && n8 > 0) {
                // every reporter's pointer first (independent loads), then the copies
                const GathSrc* src = a.src + sg.src0;
                const void* xp[kMaxBatch];
#pragma unroll
                for (int jj = 0; jj < kMaxBatch; ++jj)
                    xp[jj] = jj < static_cast<int>(sg.J) ? src[jj].x : nullptr;
                const uint32_t xb = n8 * kVec * sizeof(Tin);
                mbar_expect(bar, sg.J * xb);
                uint8_t* st = smem + s * stage;
#pragma unroll
                for (int jj = 0; jj < kMaxBatch; ++jj) {
                    if (jj >= static_cast<int>(sg.J)) break;
                    bulk_load(st + jj * XB, static_cast<const Tin*>(xp[jj]) + ta.e0, xb, bar);
                }
            } else {
                mbar_arrive(bar);
            }
        }
        for (uint32_t i = stored; i < count && ok; ++i) {
            ok = mbar_wait(smem_addr(&done[i % kStages]), (i / kStages) & 1u);
            if (ok) {
                store(i);
                bulk_commit();
            }
        }
        if (!ok) {
            atomicOr(a.err, kErrWaitTimeout);
            const uint32_t last = count < stored + kStages ? count : stored + kStages;
            for (uint32_t i = stored; i < last; ++i)
                mbar_wait(smem_addr(&full[i % kStages]), (i / kStages) & 1u);
        }
        asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
        return;
    }

    // ---------------------------------------------------------------- compute warps
    uint32_t ccur = seg0;
    const uint32_t lane = threadIdx.x & 31u;
    for (uint32_t i = 0; i < count; ++i) {
        const uint32_t s = i % kStages;
        if (!mbar_wait(smem_addr(&full[s]), (i / kStages) & 1u)) {
            atomicOr(a.err, kErrWaitTimeout);
            break;
        }
        const TileAt ta = tile_at(a.segs, a.nseg, first + i, T, ccur);
        const GathSeg sg = a.segs[ta.si];
        const bool bulk = sg.vec_ok && ta.cnt >= static_cast<uint32_t>(kVec);
        const uint32_t n8 = bulk ? ta.cnt / kVec : 0;
        uint8_t* st = smem + s * stage;
        uint8_t* res = st + a.jmax * XB;
        if (bulk) {
            const GathSrc* src = a.src + sg.src0;
            float wv[kMaxBatch];
#pragma unroll
            for (int j = 0; j < kMaxBatch; ++j) wv[j] = j < static_cast<int>(sg.J) ? src[j].w : 0.0f;
            for (uint32_t v = threadIdx.x; v < n8; v += kBlock) {
                float r[8], rl[8];
                {
                    float xv[8];
                    smem_vec8<Tin>(st, v, xv);
#pragma unroll
                    for (int e = 0; e < 8; ++e) contrib_first<kComp>(wv[0], xv[e], r[e], rl[e]);
                }
#pragma unroll
                for (int j = 1; j < kMaxBatch; ++j) {
                    if (j >= static_cast<int>(sg.J)) break;
                    float xv[8];
                    smem_vec8<Tin>(st + j * XB, v, xv);
#pragma unroll
                    for (int e = 0; e < 8; ++e) contrib_add<kComp>(wv[j], xv[e], r[e], rl[e]);
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) r[e] = quotient_out<kComp, Tout>(r[e], rl[e], sg.div);
                smem_store8<Tout>(res, v, r);
            }
            const uint32_t tail = ta.cnt - n8 * kVec;
            if (threadIdx.x < tail) gath_one<Tin, Tout, kComp>(a, sg, ta.e0 + n8 * kVec + threadIdx.x);
        } else {
            for (uint32_t e = threadIdx.x; e < ta.cnt; e += kBlock)
                gath_one<Tin, Tout, kComp>(a, sg, ta.e0 + e);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&done[s]));
    }
}

// ----------------------------------------------------------------- finalize
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

template <typename Tout>
__device__ __forceinline__ void global_store8(void* out, uint64_t e, const float (&q)[8]) {
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
    global_store8<Tout>(sg.out, e, q);
}

template <typename Tout, bool kApply, bool kComp>
__device__ __forceinline__ void fin_one(const FinSeg& sg, uint64_t e, const float* s,
                                        const float* sl, float lr) {
    float q = kApply ? quotient<kComp>(*s, kComp ? *sl : 0.0f, sg.div)
                     : quotient_out<kComp, Tout>(*s, kComp ? *sl : 0.0f, sg.div);
    if constexpr (kApply) q = __fmaf_rn(lr, q, LoadBase<Tout>::one(sg.base, e));
    store_one<Tout>(sg.out, e, q);
}

template <typename Tout, bool kApply, bool kComp>
__global__ void __launch_bounds__(kBlock) finalize_kernel(const FinSeg* __restrict__ segs,
                                                          uint32_t nseg, uint32_t ntiles,
                                                          const float* __restrict__ acc,
                                                          const float* __restrict__ acc_lo,
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
                    global_store8<Tout>(sg.out, e0 + v * kVec, q);
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

template <typename Seg>
bool number_tiles(Seg* segs, uint32_t nseg, uint64_t tile, uint32_t* ntiles) {
    uint64_t t = 0;
    for (uint32_t i = 0; i < nseg; ++i) {
        segs[i].tile0 = static_cast<uint32_t>(t);
        t += (segs[i].len + tile - 1) / tile;
        if (t > 0xFFFFFFFFull) return false;
    }
    *ntiles = static_cast<uint32_t>(t);
    return true;
}

uint32_t grid_for(uint32_t ntiles, int sms, int per_sm) {
    uint32_t cap = static_cast<uint32_t>(sms > 0 ? sms : 1) *
                   static_cast<uint32_t>(per_sm > 0 ? per_sm : 1);
    return ntiles < cap ? ntiles : cap;
}

// Elements per reduce tile: the largest multiple of 256 whose stage fits the budget.
uint32_t reduce_tile(uint32_t elem_bytes) {
    uint32_t t = kReduceStageBytes / elem_bytes / 256 * 256;
    return t < 256 ? 256 : t;
}

template <typename Tin, typename Tout, bool kFinal, bool kComp>
cudaError_t launch_reduce_t(RedArgs a, int per_sm, int sms, cudaStream_t stream) {
    // note: occupancy (per_sm) is the same for every J specialisation
    a.has_sum = kFinal ? 0u : 1u;
    for (uint32_t i = 0; i < a.nseg; ++i) a.has_sum |= a.seg[i].read_sum;
    const uint32_t eb = reduce_elem_bytes<kFinal, kComp, Tin, Tout>(a.J, a.has_sum != 0);
    a.tile = reduce_tile(eb);
    if (!number_tiles(a.seg, a.nseg, a.tile, &a.ntiles)) return cudaErrorInvalidValue;
    if (a.ntiles == 0) return cudaSuccess;
    const size_t smem = static_cast<size_t>(kStages) * a.tile * eb + 2 * kStages * sizeof(uint64_t);
    const uint32_t grid = grid_for(a.ntiles, sms, per_sm);
    if (a.J == 16)
        return launch_dependent(reduce_bulk_kernel<Tin, Tout, kFinal, 16, kComp>, grid, kReduceThreads, smem, stream, a);
    if (a.J == 8)
        return launch_dependent(reduce_bulk_kernel<Tin, Tout, kFinal, 8, kComp>, grid, kReduceThreads, smem, stream, a);
    return launch_dependent(reduce_bulk_kernel<Tin, Tout, kFinal, 0, kComp>, grid, kReduceThreads, smem, stream, a);
}

template <typename Tin, bool kComp>
cudaError_t launch_stream_t(AccArgs a, int per_sm, int sms, cudaStream_t stream) {
    if (!number_tiles(a.seg, a.nseg, bulk_tile<kComp>(), &a.ntiles)) return cudaErrorInvalidValue;
    if (a.ntiles == 0) return cudaSuccess;
    return launch_dependent(accumulate_bulk_kernel<Tin, kComp>, grid_for(a.ntiles, sms, per_sm), kBlock,
                            bulk_smem_bytes<Tin, kComp>(), stream, a);
}

template <typename Tin, bool kComp>
cudaError_t launch_direct_t(AccArgs a, int per_sm, int sms, cudaStream_t stream) {
    if (!number_tiles(a.seg, a.nseg, kDirectTile, &a.ntiles)) return cudaErrorInvalidValue;
    if (a.ntiles == 0) return cudaSuccess;
    return launch_dependent(accumulate_direct_kernel<Tin, kComp>, grid_for(a.ntiles, sms, per_sm), kBlock,
                            0, stream, a);
}

RedArgs to_reduce_args(const AccArgs& a) {
    RedArgs r;
    for (int j = 0; j < kMaxBatch; ++j) {
        r.x[j] = a.x[j];
        r.w[j] = a.w[j];
    }
    r.acc = a.acc;
    r.acc_lo = a.acc_lo;
    r.err = a.err;
    r.J = a.J;
    r.nseg = a.nseg;
    r.ntiles = 0;
    r.tile = 0;
    r.has_sum = 1;
    r.pad = 0;
    r.vec_ok = a.vec_ok;
    for (uint32_t i = 0; i < a.nseg; ++i) {
        RedSeg& s = r.seg[i];
        s.x_off = a.seg[i].x_off;
        s.acc_idx = a.seg[i].acc_idx;
        s.len = a.seg[i].len;
        s.out = nullptr;
        s.div = Divisor{1.0f, 0.0f, 1.0f};
        s.read_sum = a.seg[i].first ? 0u : 1u;
        s.tile0 = 0;
    }
    return r;
}

template <typename Tin, typename Tout, bool kFinal, int kJ, bool kComp>
cudaError_t prepare_reduce_j(int* occ) {
    cudaError_t e = cudaFuncSetAttribute(reduce_bulk_kernel<Tin, Tout, kFinal, kJ, kComp>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kReduceSmemBytes));
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, reduce_bulk_kernel<Tin, Tout, kFinal, kJ, kComp>,
                                                         kReduceThreads, kReduceSmemBytes);
}

template <typename Tin, typename Tout, bool kFinal, bool kComp>
cudaError_t prepare_reduce(int* occ) {
    int o16 = 0, o8 = 0;
    cudaError_t e = prepare_reduce_j<Tin, Tout, kFinal, 16, kComp>(&o16);
    if (e == cudaSuccess) e = prepare_reduce_j<Tin, Tout, kFinal, 8, kComp>(&o8);
    if (e == cudaSuccess) e = prepare_reduce_j<Tin, Tout, kFinal, 0, kComp>(occ);
    if (e == cudaSuccess) *occ = std::min(*occ, std::min(o16, o8));
    return e;
}

template <typename Tin, bool kComp>
cudaError_t prepare_stream(int* occ) {
    cudaError_t e = cudaFuncSetAttribute(accumulate_bulk_kernel<Tin, kComp>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(bulk_smem_bytes<Tin, kComp>()));
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, accumulate_bulk_kernel<Tin, kComp>, kBlock,
                                                         bulk_smem_bytes<Tin, kComp>());
}

template <typename Tin, typename Tout, bool kComp>
cudaError_t prepare_gather(int* occ) {
    cudaError_t e = cudaFuncSetAttribute(reduce_gather_kernel<Tin, Tout, kComp>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kReduceSmemBytes));
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, reduce_gather_kernel<Tin, Tout, kComp>,
                                                         kReduceThreads, kReduceSmemBytes);
}

template <typename Tin, typename Tout, bool kComp>
cudaError_t launch_gather_t(const GathArgs& a, int per_sm, int sms, cudaStream_t stream) {
    const size_t smem = static_cast<size_t>(kStages) * a.tile *
                            (a.jmax * sizeof(Tin) + sizeof(Tout)) + 2 * kStages * sizeof(uint64_t);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid_for(a.ntiles, sms, per_sm));
    cfg.blockDim = dim3(kReduceThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = nullptr;
    cfg.numAttrs = 0;
    return cudaLaunchKernelEx(&cfg, reduce_gather_kernel<Tin, Tout, kComp>, a);
}

template <bool kComp>
cudaError_t gather_pick(const GathArgs& a, int din, int dout, const LaunchShape& s, cudaStream_t stream) {
    const int c = kComp ? 1 : 0;
    const int per = s.gather_ctas_per_sm[c][din][dout];
    if (din == 0)
        return dout == 0 ? launch_gather_t<float, float, kComp>(a, per, s.sms, stream)
                         : launch_gather_t<float, uint16_t, kComp>(a, per, s.sms, stream);
    return dout == 0 ? launch_gather_t<uint16_t, float, kComp>(a, per, s.sms, stream)
                     : launch_gather_t<uint16_t, uint16_t, kComp>(a, per, s.sms, stream);
}

template <bool kComp>
cudaError_t prepare_all(LaunchShape* s) {
    const int c = kComp ? 1 : 0;
    cudaError_t r = cudaSuccess;
    auto keep = [&r](cudaError_t x) { if (r == cudaSuccess) r = x; };
    keep(prepare_gather<float, float, kComp>(&s->gather_ctas_per_sm[c][0][0]));
    keep(prepare_gather<float, uint16_t, kComp>(&s->gather_ctas_per_sm[c][0][1]));
    keep(prepare_gather<uint16_t, float, kComp>(&s->gather_ctas_per_sm[c][1][0]));
    keep(prepare_gather<uint16_t, uint16_t, kComp>(&s->gather_ctas_per_sm[c][1][1]));
    keep(prepare_stream<float, kComp>(&s->bulk_ctas_per_sm[c][0]));
    keep(prepare_stream<uint16_t, kComp>(&s->bulk_ctas_per_sm[c][1]));
    keep(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&s->direct_ctas_per_sm[c][0],
                                                       accumulate_direct_kernel<float, kComp>, kBlock, 0));
    keep(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&s->direct_ctas_per_sm[c][1],
                                                       accumulate_direct_kernel<uint16_t, kComp>, kBlock, 0));
    keep(prepare_reduce<float, float, false, kComp>(&s->reduce_ctas_per_sm[c][0][0]));
    keep(prepare_reduce<float, float, true, kComp>(&s->reduce_ctas_per_sm[c][0][1]));
    keep(prepare_reduce<float, uint16_t, true, kComp>(&s->reduce_ctas_per_sm[c][0][2]));
    keep(prepare_reduce<uint16_t, float, false, kComp>(&s->reduce_ctas_per_sm[c][1][0]));
    keep(prepare_reduce<uint16_t, float, true, kComp>(&s->reduce_ctas_per_sm[c][1][1]));
    keep(prepare_reduce<uint16_t, uint16_t, true, kComp>(&s->reduce_ctas_per_sm[c][1][2]));
    keep(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&s->fin_ctas_per_sm[c][0][0],
                                                       finalize_kernel<float, false, kComp>, kBlock, 0));
    keep(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&s->fin_ctas_per_sm[c][0][1],
                                                       finalize_kernel<uint16_t, false, kComp>, kBlock, 0));
    keep(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&s->fin_ctas_per_sm[c][1][0],
                                                       finalize_kernel<float, true, kComp>, kBlock, 0));
    keep(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&s->fin_ctas_per_sm[c][1][1],
                                                       finalize_kernel<uint16_t, true, kComp>, kBlock, 0));
    return r;
}

template <bool kComp>
cudaError_t accumulate_t(const AccArgs& a, int in, const LaunchShape& s, cudaStream_t stream) {
    const int c = kComp ? 1 : 0;
    if (a.J == 1) {
        return in == 0 ? launch_stream_t<float, kComp>(a, s.bulk_ctas_per_sm[c][0], s.sms, stream)
                       : launch_stream_t<uint16_t, kComp>(a, s.bulk_ctas_per_sm[c][1], s.sms, stream);
    }
    const RedArgs r = to_reduce_args(a);
    return in == 0 ? launch_reduce_t<float, float, false, kComp>(r, s.reduce_ctas_per_sm[c][0][0], s.sms, stream)
                   : launch_reduce_t<uint16_t, float, false, kComp>(r, s.reduce_ctas_per_sm[c][1][0], s.sms, stream);
}

template <bool kComp>
cudaError_t reduce_final_t(const RedArgs& a, int in, int dtype_out, const LaunchShape& s,
                           cudaStream_t stream) {
    const int c = kComp ? 1 : 0;
    const int oi = dtype_out == 0 ? 1 : 2;
    if (in == 0) {
        return dtype_out == 0
                   ? launch_reduce_t<float, float, true, kComp>(a, s.reduce_ctas_per_sm[c][0][oi], s.sms, stream)
                   : launch_reduce_t<float, uint16_t, true, kComp>(a, s.reduce_ctas_per_sm[c][0][oi], s.sms, stream);
    }
    return dtype_out == 0
               ? launch_reduce_t<uint16_t, float, true, kComp>(a, s.reduce_ctas_per_sm[c][1][oi], s.sms, stream)
               : launch_reduce_t<uint16_t, uint16_t, true, kComp>(a, s.reduce_ctas_per_sm[c][1][oi], s.sms, stream);
}

template <typename Tout, bool kApply, bool kComp>
cudaError_t finalize_t(uint32_t grid, const FinSeg* segs, uint32_t nseg, uint32_t ntiles,
                       const float* acc, const float* acc_lo, float lr, cudaStream_t stream) {
    // a plain launch (no programmatic dependency: the kernel reads the sum from its
    // first instruction); the status is this launch's own
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kBlock);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = nullptr;
    cfg.numAttrs = 0;
    return cudaLaunchKernelEx(&cfg, finalize_kernel<Tout, kApply, kComp>, segs, nseg, ntiles, acc,
                              acc_lo, lr);
}

template <bool kComp>
cudaError_t finalize_pick(uint32_t grid, int dtype_out, bool apply, const FinSeg* segs,
                          uint32_t nseg, uint32_t ntiles, const float* acc, const float* acc_lo,
                          float lr, cudaStream_t stream) {
    if (dtype_out == 0) {
        return apply ? finalize_t<float, true, kComp>(grid, segs, nseg, ntiles, acc, acc_lo, lr, stream)
                     : finalize_t<float, false, kComp>(grid, segs, nseg, ntiles, acc, acc_lo, lr, stream);
    }
    return apply ? finalize_t<uint16_t, true, kComp>(grid, segs, nseg, ntiles, acc, acc_lo, lr, stream)
                 : finalize_t<uint16_t, false, kComp>(grid, segs, nseg, ntiles, acc, acc_lo, lr, stream);
}

}  // namespace

Divisor make_divisor(double n) {
    Divisor d;
    d.hi = static_cast<float>(n);
    d.lo = static_cast<float>(n - static_cast<double>(d.hi));
    d.rcp = static_cast<float>(1.0 / static_cast<double>(d.hi));
    return d;
}

cudaError_t query_launch_shape(LaunchShape* s) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&s->sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = prepare_all<false>(s);
    if (e == cudaSuccess) e = prepare_all<true>(s);
    return e;
}

cudaError_t launch_accumulate_direct(const AccArgs& a, int dtype_in, const LaunchShape& s,
                                     cudaStream_t stream) {
    if (a.nseg == 0 || a.nseg > static_cast<uint32_t>(kMaxSegs) || a.J != 1 || a.err == nullptr)
        return cudaErrorInvalidValue;
    const int c = a.acc_lo ? 1 : 0;
    if (c)
        return dtype_in == 0 ? launch_direct_t<float, true>(a, s.direct_ctas_per_sm[c][0], s.sms, stream)
                             : launch_direct_t<uint16_t, true>(a, s.direct_ctas_per_sm[c][1], s.sms, stream);
    return dtype_in == 0 ? launch_direct_t<float, false>(a, s.direct_ctas_per_sm[c][0], s.sms, stream)
                         : launch_direct_t<uint16_t, false>(a, s.direct_ctas_per_sm[c][1], s.sms, stream);
}

cudaError_t launch_accumulate(const AccArgs& a, int dtype_in, const LaunchShape& s,
                              cudaStream_t stream) {
    if (a.nseg == 0 || a.nseg > static_cast<uint32_t>(kMaxSegs) || a.err == nullptr)
        return cudaErrorInvalidValue;
    if (a.J == 0 || a.J > static_cast<uint32_t>(kMaxBatch)) return cudaErrorInvalidValue;
    const int in = dtype_in == 0 ? 0 : 1;
    return a.acc_lo ? accumulate_t<true>(a, in, s, stream) : accumulate_t<false>(a, in, s, stream);
}

cudaError_t launch_reduce_final(const RedArgs& a, int dtype_in, int dtype_out,
                                const LaunchShape& s, cudaStream_t stream) {
    if (a.nseg == 0 || a.nseg > static_cast<uint32_t>(kMaxSegs) || a.err == nullptr)
        return cudaErrorInvalidValue;
    if (a.J == 0 || a.J > static_cast<uint32_t>(kMaxBatch)) return cudaErrorInvalidValue;
    const int in = dtype_in == 0 ? 0 : 1;
    return a.acc_lo ? reduce_final_t<true>(a, in, dtype_out, s, stream)
                    : reduce_final_t<false>(a, in, dtype_out, s, stream);
}

uint32_t gather_tile(uint32_t jmax, int dtype_in, int dtype_out) {
    const uint32_t eb = jmax * (dtype_in == 0 ? 4u : 2u) + (dtype_out == 0 ? 4u : 2u);
    return reduce_tile(eb);
}

bool plan_gather_tiles(GathSeg* segs, uint32_t nseg, uint32_t tile, uint32_t* ntiles) {
    return number_tiles(segs, nseg, tile, ntiles);
}

cudaError_t launch_gather_final(const GathArgs& a, int dtype_in, int dtype_out, bool comp,
                                const LaunchShape& s, cudaStream_t stream) {
    if (a.nseg == 0 || a.ntiles == 0) return cudaSuccess;
    if (a.err == nullptr || a.segs == nullptr || a.src == nullptr || a.jmax == 0 ||
        a.jmax > static_cast<uint32_t>(kMaxBatch) || a.tile != gather_tile(a.jmax, dtype_in, dtype_out))
        return cudaErrorInvalidValue;
    const int din = dtype_in == 0 ? 0 : 1, dout = dtype_out == 0 ? 0 : 1;
    return comp ? gather_pick<true>(a, din, dout, s, stream) : gather_pick<false>(a, din, dout, s, stream);
}

cudaError_t launch_finalize(const FinSeg* segs, uint32_t nseg, uint32_t ntiles, int dtype_out,
                            const float* acc, const float* acc_lo, bool apply, float server_lr,
                            bool host_out, const LaunchShape& s, cudaStream_t stream) {
    if (ntiles == 0 || nseg == 0) return cudaSuccess;
    const int c = acc_lo ? 1 : 0;
    const int occ = s.fin_ctas_per_sm[c][apply ? 1 : 0][dtype_out == 0 ? 0 : 1];
    const uint32_t grid = grid_for(ntiles, s.sms, host_out ? occ : std::min(occ, kFinCtasPerSm));
    return c ? finalize_pick<true>(grid, dtype_out, apply, segs, nseg, ntiles, acc, acc_lo, server_lr, stream)
             : finalize_pick<false>(grid, dtype_out, apply, segs, nseg, ntiles, acc, acc_lo, server_lr, stream);
}

}  // namespace fa
