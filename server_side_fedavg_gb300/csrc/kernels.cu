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
// multiply-add, in client order -- so every path yields the same bits.
// Every mbarrier wait is bounded; a timeout sets g_device_error (read by fa_sync),
// makes the CTA wait (bounded) for its own loads in flight, and return.
#include "kernels.cuh"

#include <cuda_bf16.h>

#include <algorithm>

namespace fa {

__device__ unsigned int g_device_error;

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

// Store eight results of dtype Tout (RNE for bf16) to shared memory vector slot v.
template <typename Tout>
__device__ __forceinline__ void smem_store8(uint8_t* base, uint32_t v, const float (&q)[8]) {
    if constexpr (sizeof(Tout) == 2) {
        reinterpret_cast<uint4*>(base)[v] = make_uint4(pack_bf16(q[0], q[1]), pack_bf16(q[2], q[3]),
                                                       pack_bf16(q[4], q[5]), pack_bf16(q[6], q[7]));
    } else {
        reinterpret_cast<float4*>(base)[2 * v] = make_float4(q[0], q[1], q[2], q[3]);
        reinterpret_cast<float4*>(base)[2 * v + 1] = make_float4(q[4], q[5], q[6], q[7]);
    }
}

template <typename Tout>
__device__ __forceinline__ void store_one(void* out, uint64_t e, float q) {
    if constexpr (sizeof(Tout) == 2)
        static_cast<uint16_t*>(out)[e] = __bfloat16_as_ushort(__float2bfloat16_rn(q));
    else
        static_cast<float*>(out)[e] = q;
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
                                               uint32_t issued, uint32_t count) {
    if (consumed < count) {
        atomicOr(&g_device_error, kErrWaitTimeout);
        for (uint32_t j = consumed; j < issued; ++j)
            mbar_wait(smem_addr(&bars[j % kStages]), (j / kStages) & 1u);
    }
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ----------------------------------------------------------------- streaming accumulate
// One element through global memory (ragged tails, unaligned segments).
template <typename Tin>
__device__ __forceinline__ void acc_one(const Tin* x, float w, float* s, bool first) {
    const float xv = load_one<Tin>(x);
    *s = first ? __fmul_rn(w, xv) : __fmaf_rn(w, xv, *s);
}

template <typename Tin>
constexpr size_t bulk_smem_bytes() {
    return static_cast<size_t>(kStages) * kBulkTile * (sizeof(Tin) + sizeof(float)) +
           static_cast<size_t>(kStages) * sizeof(uint64_t);
}

// Stage = input tile (kBulkTile x Tin) + sum tile (kBulkTile x fp32): 48 KB for bf16,
// 64 KB for fp32 input; one CTA per SM.
template <typename Tin>
__global__ void __launch_bounds__(kBlock, 1) accumulate_bulk_kernel(const __grid_constant__ AccArgs a) {
    constexpr uint32_t XB = kBulkTile * sizeof(Tin);
    constexpr uint32_t SB = kBulkTile * sizeof(float);
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* xs = smem;
    uint8_t* ss = smem + kStages * XB;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * (XB + SB));
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
        const TileAt ta = tile_at(a.seg, a.nseg, blockIdx.x + i * gridDim.x, kBulkTile, pcur);
        const AccSeg& sg = a.seg[ta.si];
        const uint32_t bar = smem_addr(&bars[s]);
        const uint32_t n8 = ta.cnt / kVec;
        if (((a.vec_ok >> ta.si) & 1ull) && n8 > 0) {
            const uint32_t xb = n8 * kVec * sizeof(Tin);
            const uint32_t sb = sg.first ? 0u : n8 * kVec * sizeof(float);
            mbar_expect(bar, xb + sb);
            bulk_load(xs + s * XB, static_cast<const Tin*>(sg.x) + sg.x_off + ta.e0, xb, bar);
            if (sb) bulk_load(ss + s * SB, a.acc + sg.acc_idx + ta.e0, sb, bar);
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
        const bool ok = mbar_wait(smem_addr(&bars[s]), (i / kStages) & 1u);
        const TileAt ta = tile_at(a.seg, a.nseg, blockIdx.x + i * gridDim.x, kBulkTile, ccur);
        const AccSeg& sg = a.seg[ta.si];
        const bool first = sg.first != 0;
        const Tin* xg = static_cast<const Tin*>(sg.x) + sg.x_off + ta.e0;   // tile in global memory
        float* g0 = a.acc + sg.acc_idx + ta.e0;
        const bool bulk = ((a.vec_ok >> ta.si) & 1ull) && ta.cnt >= static_cast<uint32_t>(kVec);
        const uint32_t n8 = bulk ? ta.cnt / kVec : 0;
        if (ok && bulk) {
            const uint8_t* xt = xs + s * XB;
            float4* st = reinterpret_cast<float4*>(ss + s * SB);
            for (uint32_t v = threadIdx.x; v < n8; v += kBlock) {
                float xv[8];
                smem_vec8<Tin>(xt, v, xv);
                float4 lo, hi;
                if (first) {
                    lo = make_float4(__fmul_rn(w, xv[0]), __fmul_rn(w, xv[1]), __fmul_rn(w, xv[2]),
                                     __fmul_rn(w, xv[3]));
                    hi = make_float4(__fmul_rn(w, xv[4]), __fmul_rn(w, xv[5]), __fmul_rn(w, xv[6]),
                                     __fmul_rn(w, xv[7]));
                } else {
                    lo = st[2 * v];
                    hi = st[2 * v + 1];
                    lo.x = __fmaf_rn(w, xv[0], lo.x); lo.y = __fmaf_rn(w, xv[1], lo.y);
                    lo.z = __fmaf_rn(w, xv[2], lo.z); lo.w = __fmaf_rn(w, xv[3], lo.w);
                    hi.x = __fmaf_rn(w, xv[4], hi.x); hi.y = __fmaf_rn(w, xv[5], hi.y);
                    hi.z = __fmaf_rn(w, xv[6], hi.z); hi.w = __fmaf_rn(w, xv[7], hi.w);
                }
                st[2 * v] = lo;
                st[2 * v + 1] = hi;
            }
            const uint32_t tail = ta.cnt - n8 * kVec;
            if (threadIdx.x < tail) {
                const uint32_t e = n8 * kVec + threadIdx.x;
                acc_one<Tin>(xg + e, w, g0 + e, first);
            }
        } else if (ok) {
            for (uint32_t e = threadIdx.x; e < ta.cnt; e += kBlock)
                acc_one<Tin>(xg + e, w, g0 + e, first);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        if (!__syncthreads_and(ok)) break;
        consumed = i + 1;
        if (threadIdx.x == 0) {
            if (n8 > 0) bulk_store(g0, ss + s * SB, n8 * kVec * 4u);
            bulk_commit();
            // refill the stage drained one iteration ago once its store has read it
            if (i >= 1 && i - 1 + kStages < count) {
                asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
                issue(i - 1 + kStages);
                issued = i + kStages;
            }
        }
    }
    if (threadIdx.x == 0) pipeline_drain(bars, consumed, issued, count);
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

template <typename Tin>
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
        const uint32_t n8 = ((a.vec_ok >> ta.si) & 1ull) ? ta.cnt / kVec : 0u;
        if (threadIdx.x < n8) {
            float xv[8];
            plain_vec8<Tin>(xt + threadIdx.x * kVec, xv);
            float* gp = g + threadIdx.x * kVec;
            float4 lo, hi;
            if (first) {
                lo = make_float4(__fmul_rn(w, xv[0]), __fmul_rn(w, xv[1]), __fmul_rn(w, xv[2]),
                                 __fmul_rn(w, xv[3]));
                hi = make_float4(__fmul_rn(w, xv[4]), __fmul_rn(w, xv[5]), __fmul_rn(w, xv[6]),
                                 __fmul_rn(w, xv[7]));
            } else {
                lo = ld_v4f(gp);
                hi = ld_v4f(gp + 4);
                lo.x = __fmaf_rn(w, xv[0], lo.x); lo.y = __fmaf_rn(w, xv[1], lo.y);
                lo.z = __fmaf_rn(w, xv[2], lo.z); lo.w = __fmaf_rn(w, xv[3], lo.w);
                hi.x = __fmaf_rn(w, xv[4], hi.x); hi.y = __fmaf_rn(w, xv[5], hi.y);
                hi.z = __fmaf_rn(w, xv[6], hi.z); hi.w = __fmaf_rn(w, xv[7], hi.w);
            }
            st_v4f(gp, lo);
            st_v4f(gp + 4, hi);
        }
        for (uint32_t e = n8 * kVec + threadIdx.x; e < ta.cnt; e += kBlock) {
            const float xv = load_plain<Tin>(xt + e);
            g[e] = first ? __fmul_rn(w, xv) : __fmaf_rn(w, xv, g[e]);
        }
    }
}

// ----------------------------------------------------------------- J-client reduce
// Stage = J input tiles (T x Tin each) [+ sum tile (T x fp32): sum mode, or final mode
// reading earlier contributions] [+ output tile (T x Tout): final mode]; T is chosen on
// the host so a stage fits kReduceStageBytes (one CTA per SM, three stages: about
// 200 KB of copies in flight).  Sum mode writes the running sum back; final mode
// divides by the segment's divisor and rounds to Tout.  kJ > 0 fixes the client count
// at compile time so the per-client loop unrolls (J = 16 and 8); kJ = 0 reads it from
// the arguments.
template <bool kFinal, typename Tin, typename Tout>
__host__ __device__ constexpr uint32_t reduce_elem_bytes(uint32_t J, bool has_sum) {
    return J * static_cast<uint32_t>(sizeof(Tin)) + (has_sum ? 4u : 0u) +
           (kFinal ? static_cast<uint32_t>(sizeof(Tout)) : 0u);
}

template <typename Tin, typename Tout, bool kFinal>
__device__ __forceinline__ void red_one(const RedArgs& a, const RedSeg& sg, uint64_t e, uint32_t J) {
    // element e of the segment, through global memory
    const uint64_t xe = sg.x_off + e;
    float r;
    uint32_t j0 = 0;
    if (sg.read_sum) {
        r = a.acc[sg.acc_idx + e];
    } else {
        r = __fmul_rn(a.w[0], load_one<Tin>(static_cast<const Tin*>(a.x[0]) + xe));
        j0 = 1;
    }
    for (uint32_t j = j0; j < J; ++j)
        r = __fmaf_rn(a.w[j], load_one<Tin>(static_cast<const Tin*>(a.x[j]) + xe), r);
    if constexpr (kFinal)
        store_one<Tout>(sg.out, e, __fdiv_rn(r, sg.divisor));
    else
        a.acc[sg.acc_idx + e] = r;
}

// Warp-specialised: warps 0-7 compute, warp 8 (one lane) moves data.  Per stage two
// mbarriers: `full` (the producer arms it with the byte count of the stage's bulk loads)
// and `done` (each compute warp arrives once it has finished the stage).  The producer
// stores a stage's result tile when `done` completes and refills the stage once that
// store has read it; the compute warps never wait for producer work except data.
constexpr int kReduceWarps = kBlock / 32;               // compute warps
constexpr int kReduceThreads = kBlock + 32;             // + one producer warp

template <typename Tin, typename Tout, bool kFinal, int kJ>
__global__ void __launch_bounds__(kReduceThreads, 1) reduce_bulk_kernel(const __grid_constant__ RedArgs a) {
    const uint32_t T = a.tile;
    const uint32_t J = kJ > 0 ? static_cast<uint32_t>(kJ) : a.J;
    const uint32_t XB = T * sizeof(Tin);
    const uint32_t SB = a.has_sum ? T * static_cast<uint32_t>(sizeof(float)) : 0u;
    const uint32_t stage = T * reduce_elem_bytes<kFinal, Tin, Tout>(J, a.has_sum != 0);
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
            if constexpr (kFinal)
                bulk_store(static_cast<Tout*>(sg.out) + ta.e0, st + J * XB + SB, n8 * kVec * sizeof(Tout));
            else
                bulk_store(a.acc + sg.acc_idx + ta.e0, st + J * XB, n8 * kVec * 4u);
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
                mbar_expect(bar, J * xb + sb);
                uint8_t* st = smem + s * stage;
#pragma unroll
                for (uint32_t jj = 0; jj < (kJ > 0 ? static_cast<uint32_t>(kJ) : static_cast<uint32_t>(kMaxBatch)); ++jj) {
                    if (kJ == 0 && jj >= J) break;
                    bulk_load(st + jj * XB, static_cast<const Tin*>(a.x[jj]) + sg.x_off + ta.e0, xb, bar);
                }
                if (sb) bulk_load(st + J * XB, a.acc + sg.acc_idx + ta.e0, sb, bar);
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
            atomicOr(&g_device_error, kErrWaitTimeout);
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
            atomicOr(&g_device_error, kErrWaitTimeout);
            break;
        }
        const TileAt ta = tile_at(a.seg, a.nseg, blockIdx.x + i * gridDim.x, T, ccur);
        const RedSeg& sg = a.seg[ta.si];
        const bool bulk = ((a.vec_ok >> ta.si) & 1ull) && ta.cnt >= static_cast<uint32_t>(kVec);
        const uint32_t n8 = bulk ? ta.cnt / kVec : 0;
        uint8_t* st = smem + s * stage;
        float4* sum = reinterpret_cast<float4*>(st + J * XB);
        uint8_t* res = st + J * XB + SB;                      // final mode output tile
        if (bulk) {
            for (uint32_t v = threadIdx.x; v < n8; v += kBlock) {
                float r[8];
                {
                    float xv[8];
                    smem_vec8<Tin>(st, v, xv);
                    if (sg.read_sum) {          // client 0 joins the earlier contributions
                        const float4 lo = sum[2 * v], hi = sum[2 * v + 1];
                        r[0] = lo.x; r[1] = lo.y; r[2] = lo.z; r[3] = lo.w;
                        r[4] = hi.x; r[5] = hi.y; r[6] = hi.z; r[7] = hi.w;
#pragma unroll
                        for (int e = 0; e < 8; ++e) r[e] = __fmaf_rn(a.w[0], xv[e], r[e]);
                    } else {                    // client 0 starts the sum
#pragma unroll
                        for (int e = 0; e < 8; ++e) r[e] = __fmul_rn(a.w[0], xv[e]);
                    }
                }
#pragma unroll
                for (uint32_t j = 1; j < (kJ > 0 ? static_cast<uint32_t>(kJ) : static_cast<uint32_t>(kMaxBatch)); ++j) {
                    if (kJ == 0 && j >= J) break;
                    float xv[8];
                    smem_vec8<Tin>(st + j * XB, v, xv);
                    const float wj = a.w[j];
#pragma unroll
                    for (int e = 0; e < 8; ++e) r[e] = __fmaf_rn(wj, xv[e], r[e]);
                }
                if constexpr (kFinal) {
                    const float d = sg.divisor;
#pragma unroll
                    for (int e = 0; e < 8; ++e) r[e] = __fdiv_rn(r[e], d);
                    smem_store8<Tout>(res, v, r);
                } else {
                    sum[2 * v] = make_float4(r[0], r[1], r[2], r[3]);
                    sum[2 * v + 1] = make_float4(r[4], r[5], r[6], r[7]);
                }
            }
            const uint32_t tail = ta.cnt - n8 * kVec;
            if (threadIdx.x < tail) red_one<Tin, Tout, kFinal>(a, sg, ta.e0 + n8 * kVec + threadIdx.x, J);
        } else {
            for (uint32_t e = threadIdx.x; e < ta.cnt; e += kBlock)
                red_one<Tin, Tout, kFinal>(a, sg, ta.e0 + e, J);
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
    global_store8<Tout>(sg.out, e, q);
}

template <typename Tout, bool kApply>
__device__ __forceinline__ void fin_one(const FinSeg& sg, uint64_t e, const float* s, float d,
                                        float lr) {
    float q = __fdiv_rn(*s, d);
    if constexpr (kApply) q = __fmaf_rn(lr, q, LoadBase<Tout>::one(sg.base, e));
    store_one<Tout>(sg.out, e, q);
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
                // every load of the tile first: a store (asm volatile, memory clobber) would
                // otherwise hold the next vector's loads back, leaving one in flight per thread
                float4 lo[kUnroll], hi[kUnroll];
                float b[kUnroll][8];
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const uint32_t v = threadIdx.x + u * kBlock;
                    lo[u] = ld_v4f(s0 + v * kVec);
                    hi[u] = ld_v4f(s0 + v * kVec + 4);
                    if constexpr (kApply) LoadBase<Tout>::vec(sg.base, e0 + v * kVec, b[u]);
                }
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const uint32_t v = threadIdx.x + u * kBlock;
                    float q[8] = {__fdiv_rn(lo[u].x, d), __fdiv_rn(lo[u].y, d), __fdiv_rn(lo[u].z, d),
                                  __fdiv_rn(lo[u].w, d), __fdiv_rn(hi[u].x, d), __fdiv_rn(hi[u].y, d),
                                  __fdiv_rn(hi[u].z, d), __fdiv_rn(hi[u].w, d)};
                    if constexpr (kApply) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) q[i] = __fmaf_rn(lr, q[i], b[u][i]);
                    }
                    global_store8<Tout>(sg.out, e0 + v * kVec, q);
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

template <typename Tin, typename Tout, bool kFinal>
cudaError_t launch_reduce_t(RedArgs a, int per_sm, int sms, cudaStream_t stream) {
    // note: occupancy (per_sm) is the same for every J specialisation
    a.has_sum = kFinal ? 0u : 1u;
    for (uint32_t i = 0; i < a.nseg; ++i) a.has_sum |= a.seg[i].read_sum;
    const uint32_t eb = reduce_elem_bytes<kFinal, Tin, Tout>(a.J, a.has_sum != 0);
    a.tile = reduce_tile(eb);
    if (!number_tiles(a.seg, a.nseg, a.tile, &a.ntiles)) return cudaErrorInvalidValue;
    if (a.ntiles == 0) return cudaSuccess;
    const size_t smem = static_cast<size_t>(kStages) * a.tile * eb + 2 * kStages * sizeof(uint64_t);
    const uint32_t grid = grid_for(a.ntiles, sms, per_sm);
    if (a.J == 16)
        return launch_dependent(reduce_bulk_kernel<Tin, Tout, kFinal, 16>, grid, kReduceThreads, smem, stream, a);
    if (a.J == 8)
        return launch_dependent(reduce_bulk_kernel<Tin, Tout, kFinal, 8>, grid, kReduceThreads, smem, stream, a);
    return launch_dependent(reduce_bulk_kernel<Tin, Tout, kFinal, 0>, grid, kReduceThreads, smem, stream, a);
}

template <typename Tin>
cudaError_t launch_stream_t(AccArgs a, int per_sm, int sms, cudaStream_t stream) {
    if (!number_tiles(a.seg, a.nseg, kBulkTile, &a.ntiles)) return cudaErrorInvalidValue;
    if (a.ntiles == 0) return cudaSuccess;
    return launch_dependent(accumulate_bulk_kernel<Tin>, grid_for(a.ntiles, sms, per_sm), kBlock,
                            bulk_smem_bytes<Tin>(), stream, a);
}

template <typename Tin>
cudaError_t launch_direct_t(AccArgs a, int per_sm, int sms, cudaStream_t stream) {
    if (!number_tiles(a.seg, a.nseg, kDirectTile, &a.ntiles)) return cudaErrorInvalidValue;
    if (a.ntiles == 0) return cudaSuccess;
    return launch_dependent(accumulate_direct_kernel<Tin>, grid_for(a.ntiles, sms, per_sm), kBlock,
                            0, stream, a);
}

RedArgs to_reduce_args(const AccArgs& a) {
    RedArgs r;
    for (int j = 0; j < kMaxBatch; ++j) {
        r.x[j] = a.x[j];
        r.w[j] = a.w[j];
    }
    r.acc = a.acc;
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
        s.divisor = 1.0f;
        s.read_sum = a.seg[i].first ? 0u : 1u;
        s.tile0 = 0;
        s.pad = 0;
    }
    return r;
}

template <typename Tin, typename Tout, bool kFinal, int kJ>
cudaError_t prepare_reduce_j(int* occ) {
    cudaError_t e = cudaFuncSetAttribute(reduce_bulk_kernel<Tin, Tout, kFinal, kJ>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kReduceSmemBytes));
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, reduce_bulk_kernel<Tin, Tout, kFinal, kJ>,
                                                         kReduceThreads, kReduceSmemBytes);
}

template <typename Tin, typename Tout, bool kFinal>
cudaError_t prepare_reduce(int* occ) {
    int o16 = 0, o8 = 0;
    cudaError_t e = prepare_reduce_j<Tin, Tout, kFinal, 16>(&o16);
    if (e == cudaSuccess) e = prepare_reduce_j<Tin, Tout, kFinal, 8>(&o8);
    if (e == cudaSuccess) e = prepare_reduce_j<Tin, Tout, kFinal, 0>(occ);
    if (e == cudaSuccess) *occ = std::min(*occ, std::min(o16, o8));
    return e;
}

template <typename Tin>
cudaError_t prepare_stream(int* occ) {
    cudaError_t e = cudaFuncSetAttribute(accumulate_bulk_kernel<Tin>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(bulk_smem_bytes<Tin>()));
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, accumulate_bulk_kernel<Tin>, kBlock,
                                                         bulk_smem_bytes<Tin>());
}

}  // namespace

cudaError_t take_device_error_async(unsigned int* host, cudaStream_t stream) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(host, g_device_error, sizeof(unsigned int), 0,
                                              cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    void* word = nullptr;
    e = cudaGetSymbolAddress(&word, g_device_error);
    if (e != cudaSuccess) return e;
    return cudaMemsetAsync(word, 0, sizeof(unsigned int), stream);
}

cudaError_t query_launch_shape(LaunchShape* s) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&s->sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    cudaError_t r = cudaSuccess;
    auto keep = [&r](cudaError_t x) { if (r == cudaSuccess) r = x; };
    keep(prepare_stream<float>(&s->bulk_ctas_per_sm[0]));
    keep(prepare_stream<uint16_t>(&s->bulk_ctas_per_sm[1]));
    keep(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&s->direct_ctas_per_sm[0],
                                                       accumulate_direct_kernel<float>, kBlock, 0));
    keep(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&s->direct_ctas_per_sm[1],
                                                       accumulate_direct_kernel<uint16_t>, kBlock, 0));
    keep(prepare_reduce<float, float, false>(&s->reduce_ctas_per_sm[0][0]));
    keep(prepare_reduce<float, float, true>(&s->reduce_ctas_per_sm[0][1]));
    keep(prepare_reduce<float, uint16_t, true>(&s->reduce_ctas_per_sm[0][2]));
    keep(prepare_reduce<uint16_t, float, false>(&s->reduce_ctas_per_sm[1][0]));
    keep(prepare_reduce<uint16_t, float, true>(&s->reduce_ctas_per_sm[1][1]));
    keep(prepare_reduce<uint16_t, uint16_t, true>(&s->reduce_ctas_per_sm[1][2]));
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

cudaError_t launch_accumulate_direct(const AccArgs& a, int dtype_in, const LaunchShape& s,
                                     cudaStream_t stream) {
    if (a.nseg == 0 || a.nseg > static_cast<uint32_t>(kMaxSegs) || a.J != 1) return cudaErrorInvalidValue;
    return dtype_in == 0 ? launch_direct_t<float>(a, s.direct_ctas_per_sm[0], s.sms, stream)
                         : launch_direct_t<uint16_t>(a, s.direct_ctas_per_sm[1], s.sms, stream);
}

cudaError_t launch_accumulate(const AccArgs& a, int dtype_in, const LaunchShape& s,
                              cudaStream_t stream) {
    if (a.nseg == 0 || a.nseg > static_cast<uint32_t>(kMaxSegs)) return cudaErrorInvalidValue;
    if (a.J == 0 || a.J > static_cast<uint32_t>(kMaxBatch)) return cudaErrorInvalidValue;
    const int in = dtype_in == 0 ? 0 : 1;
    if (a.J == 1) {
        return in == 0 ? launch_stream_t<float>(a, s.bulk_ctas_per_sm[0], s.sms, stream)
                       : launch_stream_t<uint16_t>(a, s.bulk_ctas_per_sm[1], s.sms, stream);
    }
    const RedArgs r = to_reduce_args(a);
    return in == 0 ? launch_reduce_t<float, float, false>(r, s.reduce_ctas_per_sm[0][0], s.sms, stream)
                   : launch_reduce_t<uint16_t, float, false>(r, s.reduce_ctas_per_sm[1][0], s.sms, stream);
}

cudaError_t launch_reduce_final(const RedArgs& a, int dtype_in, int dtype_out,
                                const LaunchShape& s, cudaStream_t stream) {
    if (a.nseg == 0 || a.nseg > static_cast<uint32_t>(kMaxSegs)) return cudaErrorInvalidValue;
    if (a.J == 0 || a.J > static_cast<uint32_t>(kMaxBatch)) return cudaErrorInvalidValue;
    const int in = dtype_in == 0 ? 0 : 1;
    const int oi = dtype_out == 0 ? 1 : 2;
    if (in == 0) {
        return dtype_out == 0
                   ? launch_reduce_t<float, float, true>(a, s.reduce_ctas_per_sm[0][oi], s.sms, stream)
                   : launch_reduce_t<float, uint16_t, true>(a, s.reduce_ctas_per_sm[0][oi], s.sms, stream);
    }
    return dtype_out == 0
               ? launch_reduce_t<uint16_t, float, true>(a, s.reduce_ctas_per_sm[1][oi], s.sms, stream)
               : launch_reduce_t<uint16_t, uint16_t, true>(a, s.reduce_ctas_per_sm[1][oi], s.sms, stream);
}

cudaError_t launch_finalize(const FinSeg* segs, uint32_t nseg, uint32_t ntiles, int dtype_out,
                            const float* acc, bool apply, float server_lr, bool host_out,
                            const LaunchShape& s, cudaStream_t stream) {
    if (ntiles == 0 || nseg == 0) return cudaSuccess;
    const int occ = s.fin_ctas_per_sm[apply ? 1 : 0][dtype_out == 0 ? 0 : 1];
    const uint32_t grid = grid_for(ntiles, s.sms, host_out ? occ : std::min(occ, kFinCtasPerSm));
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
