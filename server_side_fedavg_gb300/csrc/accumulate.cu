// Streaming accumulate kernels: one client per launch, the running fp32 sum updated in
// place (see kernels.cuh for the operation and device.cuh for the shared conventions).
//  - accumulate_bulk_kernel (the streaming hot path) moves its tiles with bulk copies
//    through a three-stage shared-memory pipeline: one elected thread arms a stage's
//    mbarrier with the byte count and issues the loads, all threads compute in shared
//    memory, the elected thread writes the sum tile back with one bulk store, and a
//    stage is refilled once that store has read it.  A persistent grid of one CTA per
//    SM keeps about 150 KB of copies in flight per SM -- a timed sweep of tile sizes,
//    stage counts and direct-load variants on GB300 chose this shape;
//  - accumulate_direct_kernel reads its input in place with plain loads: the form for
//    pinned host memory read over the NVLink-C2C link, where the link sets the pace.
#include "device.cuh"

namespace fa {

namespace {

constexpr int kFinalThreads = 1024;   // threads of a final-form streaming CTA (see bulk_threads)

// ----------------------------------------------------------------- the last quotient
// Whether a segment's divisor admits quotient8's division-free path: N_p exact in fp32 (no
// lo part) and within [2^-20, 2^60].
__device__ __forceinline__ bool fast_divisor(const Divisor& d) {
    return d.lo == 0.0f && d.hi >= 0x1p-20f && d.hi <= 0x1p60f && d.rcp > 0.0f;
}

// The quotients of one 8-element vector of a final contribution: the bits of quotient_out.
// When the divisor admits it and every sum has 2^-60 <= |s| < 2^61 -- one test for the
// vector, so the common path has no branch per element -- they take no division:
// Markstein's correction of a reciprocal (P. Markstein, "Computation of elementary
// functions on the IBM RISC System/6000 processor", IBM J. Res. Develop. 34(1), 1990).
// With y = d.rcp = RN(1/d) (rounded once, on the host), q = RN(s*y) is within two ulps of
// s/d; one step q <- RN(q + RN(s - q*d)*y), its remainder from an fma, leaves q within an
// ulp; the remainder of such a q is exact, so a second step gives s/d + (s/d - q)(d*y - 1)
// before its one rounding, nearer to s/d than s/d is to any rounding midpoint (a quotient of
// two floats with 24-bit significands lies at least ulp/2^25 from one, and |d*y - 1| <
// 2^-24): the result is RN(s/d).  Nothing underflows or overflows in those ranges.  Any
// other vector (zeros, subnormals, infinities, NaN, larger sums), divisor or the
// compensated mode takes quotient_out.
template <bool kComp, typename Tout>
__device__ __forceinline__ void quotient8(float (&hi)[8], const float (&lo)[8], const Divisor& d, bool fast) {
    if constexpr (!kComp) {
        bool in = fast;
#pragma unroll
        for (int e = 0; e < 8; ++e) in &= ((__float_as_uint(hi[e]) >> 23) & 0xFFu) - 67u < 121u;
        if (in) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                float q = __fmul_rn(hi[e], d.rcp);
                q = __fmaf_rn(__fmaf_rn(-q, d.hi, hi[e]), d.rcp, q);
                hi[e] = __fmaf_rn(__fmaf_rn(-q, d.hi, hi[e]), d.rcp, q);
            }
            return;
        }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) hi[e] = quotient_out<kComp, Tout>(hi[e], lo[e], d);
}

// ----------------------------------------------------------------- streaming accumulate
// One element through global memory (ragged tails, unaligned segments).
// kFinal: the element's last contribution -- the quotient is written to out[0] (dtype
// Tout) instead of the sum.
template <typename Tin, bool kComp, bool kFinal, typename Tout>
__device__ __forceinline__ void acc_one(const Tin* x, float w, float* s, float* sl, bool first,
                                        void* out, const Divisor& d) {
    const float xv = load_one<Tin>(x);
    float hi, lo = 0.0f;
    if (first) {
        contrib_first<kComp>(w, xv, hi, lo);
    } else {
        hi = *s;
        if constexpr (kComp) lo = *sl;
        contrib_add<kComp>(w, xv, hi, lo);
    }
    if constexpr (kFinal) {
        store_one<Tout>(out, 0, quotient_out<kComp, Tout>(hi, lo, d));
    } else {
        *s = hi;
        if constexpr (kComp) *sl = lo;
    }
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
// (T = 6144); one CTA per SM.  kFinal (the elements' last contribution): the quotient
// is rounded to Tout into the sum tile's space and stored to the segment's output; the
// sum is not written back.
// Threads of a streaming-accumulate CTA: the plain form moves data and does one fma per
// element (8 warps keep the copies going); the final form also divides every element, a
// chain of dependent instructions that needs more warps to hide.
template <bool kFinal>
__host__ __device__ constexpr int bulk_threads() { return kFinal ? kFinalThreads : kBlock; }

template <typename Tin, bool kComp, bool kFinal, typename Tout>
__global__ void __launch_bounds__(bulk_threads<kFinal>(), 1) accumulate_bulk_kernel(const __grid_constant__ AccArgs a) {
    constexpr uint32_t NT = bulk_threads<kFinal>();
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
        [[maybe_unused]] const bool fast = kFinal && fast_divisor(sg.div);
        if (ok && bulk) {
            uint8_t* xt = xs + s * XB;
            uint8_t* st = ss + s * SB;
            uint8_t* lt = ss + (kStages + s) * SB;
            for (uint32_t v = threadIdx.x; v < n8; v += NT) {
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
                if constexpr (kFinal) {
                    // the results take this thread's own vector slot: of the sum tile for
                    // fp32 out, of the input tile for bf16 out (bf16 in: the same 16 bytes)
                    quotient8<kComp, Tout>(hi, lo, sg.div, fast);
                    smem_store8<Tout>(sizeof(Tout) == 4 ? st : xt, v, hi);
                } else {
                    smem_st8f(st, v, hi);
                    if constexpr (kComp) smem_st8f(lt, v, lo);
                }
            }
            const uint32_t tail = ta.cnt - n8 * kVec;
            if (threadIdx.x < tail) {
                const uint32_t e = n8 * kVec + threadIdx.x;
                acc_one<Tin, kComp, kFinal, Tout>(xg + e, w, g0 + e, kComp ? l0 + e : nullptr, first,
                                                  kFinal ? static_cast<Tout*>(sg.out) + ta.e0 + e : nullptr,
                                                  sg.div);
            }
        } else if (ok) {
            for (uint32_t e = threadIdx.x; e < ta.cnt; e += NT)
                acc_one<Tin, kComp, kFinal, Tout>(xg + e, w, g0 + e, kComp ? l0 + e : nullptr, first,
                                                  kFinal ? static_cast<Tout*>(sg.out) + ta.e0 + e : nullptr,
                                                  sg.div);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        if (!__syncthreads_and(ok)) break;
        consumed = i + 1;
        if (threadIdx.x == 0) {
            if (n8 > 0) {
                if constexpr (kFinal) {
                    static_assert(sizeof(Tout) == 4 || sizeof(Tin) == 2, "bf16 results need bf16 input slots");
                    bulk_store(static_cast<Tout*>(sg.out) + ta.e0, sizeof(Tout) == 4 ? ss + s * SB : xs + s * XB,
                               n8 * kVec * static_cast<uint32_t>(sizeof(Tout)));
                } else {
                    bulk_store(g0, ss + s * SB, n8 * kVec * 4u);
                    if constexpr (kComp) bulk_store(l0, ss + (kStages + s) * SB, n8 * kVec * 4u);
                }
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
// kFinal: the elements' last contribution; the quotient (dtype Tout) goes to the
// segment's output and the sum is not stored.
template <typename Tin, bool kComp, bool kFinal, typename Tout>
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
            if constexpr (kFinal) {
#pragma unroll
                for (int e = 0; e < 8; ++e) hi[e] = quotient_out<kComp, Tout>(hi[e], lo[e], sg.div);
                store8_global<Tout>(sg.out, ta.e0 + threadIdx.x * kVec, hi);
            } else {
                st8f(gp, hi);
                if constexpr (kComp) st8f(gl + threadIdx.x * kVec, lo);
            }
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
            if constexpr (kFinal) {
                store_one<Tout>(sg.out, ta.e0 + e, quotient_out<kComp, Tout>(hi, lo, sg.div));
            } else {
                g[e] = hi;
                if constexpr (kComp) gl[e] = lo;
            }
        }
    }
}

// ----------------------------------------------------------------- host side
template <typename Tin, bool kComp, bool kFinal = false, typename Tout = float>
cudaError_t launch_stream_t(AccArgs a, int per_sm, int sms, cudaStream_t stream) {
    if (!number_tiles(a.seg, a.nseg, bulk_tile<kComp>(), &a.ntiles)) return cudaErrorInvalidValue;
    if (a.ntiles == 0) return cudaSuccess;
    return launch_dependent(accumulate_bulk_kernel<Tin, kComp, kFinal, Tout>, grid_for(a.ntiles, sms, per_sm),
                            bulk_threads<kFinal>(), bulk_smem_bytes<Tin, kComp>(), stream, a);
}

template <typename Tin, bool kComp, bool kFinal = false, typename Tout = float>
cudaError_t launch_direct_t(AccArgs a, int per_sm, int sms, cudaStream_t stream) {
    if (!number_tiles(a.seg, a.nseg, kDirectTile, &a.ntiles)) return cudaErrorInvalidValue;
    if (a.ntiles == 0) return cudaSuccess;
    return launch_dependent(accumulate_direct_kernel<Tin, kComp, kFinal, Tout>, grid_for(a.ntiles, sms, per_sm),
                            kBlock, 0, stream, a);
}

template <typename Tin, bool kComp, bool kFinal, typename Tout>
cudaError_t prepare_stream_one(int* occ) {
    cudaError_t e = cudaFuncSetAttribute(accumulate_bulk_kernel<Tin, kComp, kFinal, Tout>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(bulk_smem_bytes<Tin, kComp>()));
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, accumulate_bulk_kernel<Tin, kComp, kFinal, Tout>,
                                                         bulk_threads<kFinal>(), bulk_smem_bytes<Tin, kComp>());
}

// The streaming kernel and its final variants (the same shared memory): the occupancy of
// all of them.  Final variants exist for the dtype pairs whose result fits the stage in
// place (see fused_final_bulk).
template <typename Tin, bool kComp>
cudaError_t prepare_stream(int* occ) {
    int o1 = 0, o2 = 0;
    cudaError_t e = prepare_stream_one<Tin, kComp, false, float>(occ);
    if (e == cudaSuccess) e = prepare_stream_one<Tin, kComp, true, float>(&o1);
    o2 = o1;
    if constexpr (sizeof(Tin) == 2) {
        if (e == cudaSuccess) e = prepare_stream_one<Tin, kComp, true, uint16_t>(&o2);
    }
    if (e == cudaSuccess) *occ = std::min(*occ, std::min(o1, o2));
    return e;
}

// The direct kernel's CTAs per SM (its final variants launch the same grid: a CTA that
// does not fit waits for a slot, which the grid-stride loop allows).
template <typename Tin, bool kComp>
cudaError_t direct_occupancy(int* occ) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, accumulate_direct_kernel<Tin, kComp, false, float>,
                                                         kBlock, 0);
}

template <bool kComp>
cudaError_t prepare_accumulate_shapes(LaunchShape* s) {
    const int c = kComp ? 1 : 0;
    cudaError_t r = cudaSuccess;
    auto keep = [&r](cudaError_t x) { if (r == cudaSuccess) r = x; };
    keep(prepare_stream<float, kComp>(&s->bulk_ctas_per_sm[c][0]));
    keep(prepare_stream<uint16_t, kComp>(&s->bulk_ctas_per_sm[c][1]));
    keep(direct_occupancy<float, kComp>(&s->direct_ctas_per_sm[c][0]));
    keep(direct_occupancy<uint16_t, kComp>(&s->direct_ctas_per_sm[c][1]));
    return r;
}

template <bool kComp>
cudaError_t accumulate_t(const AccArgs& a, int in, const LaunchShape& s, cudaStream_t stream) {
    const int c = kComp ? 1 : 0;
    return in == 0 ? launch_stream_t<float, kComp>(a, s.bulk_ctas_per_sm[c][0], s.sms, stream)
                   : launch_stream_t<uint16_t, kComp>(a, s.bulk_ctas_per_sm[c][1], s.sms, stream);
}

// The bulk kernel writes a tile's results into its own shared-memory vector slots before
// storing them: in the sum tile (fp32 out: 32 B per 8 elements, as the sum) or in the
// input tile (bf16 in and out: 16 B, as the input).  fp32 in with bf16 out fits neither
// slot for slot, so it runs the direct kernel (plain loads from device memory).
bool fused_final_bulk(int din, int dout) { return dout == 0 || din == 1; }

template <bool kComp>
cudaError_t final_t(const AccArgs& a, int in, int out, bool direct, const LaunchShape& s,
                    cudaStream_t stream) {
    const int c = kComp ? 1 : 0;
    if (direct || !fused_final_bulk(in, out)) {
        const int per = s.direct_ctas_per_sm[c][in];
        if (in == 0)
            return out == 0 ? launch_direct_t<float, kComp, true, float>(a, per, s.sms, stream)
                            : launch_direct_t<float, kComp, true, uint16_t>(a, per, s.sms, stream);
        return out == 0 ? launch_direct_t<uint16_t, kComp, true, float>(a, per, s.sms, stream)
                        : launch_direct_t<uint16_t, kComp, true, uint16_t>(a, per, s.sms, stream);
    }
    const int per = s.bulk_ctas_per_sm[c][in];
    if (in == 0) return launch_stream_t<float, kComp, true, float>(a, per, s.sms, stream);
    return out == 0 ? launch_stream_t<uint16_t, kComp, true, float>(a, per, s.sms, stream)
                    : launch_stream_t<uint16_t, kComp, true, uint16_t>(a, per, s.sms, stream);
}

}  // namespace

cudaError_t query_launch_shape(LaunchShape* s) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&s->sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = prepare_accumulate_shapes<false>(s);
    if (e == cudaSuccess) e = prepare_accumulate_shapes<true>(s);
    if (e == cudaSuccess) e = prepare_reduce_shapes(s);
    if (e == cudaSuccess) e = prepare_gather_shapes(s);
    if (e == cudaSuccess) e = prepare_finalize_shapes(s);
    return e;
}

cudaError_t launch_accumulate_final(const AccArgs& a, int dtype_in, int dtype_out, bool direct,
                                    const LaunchShape& s, cudaStream_t stream) {
    if (a.nseg == 0 || a.nseg > static_cast<uint32_t>(kMaxSegs) || a.J != 1 || a.err == nullptr)
        return cudaErrorInvalidValue;
    const int in = dtype_in == 0 ? 0 : 1, out = dtype_out == 0 ? 0 : 1;
    return a.acc_lo ? final_t<true>(a, in, out, direct, s, stream) : final_t<false>(a, in, out, direct, s, stream);
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
    if (a.J > 1) return launch_reduce_sum(a, dtype_in, s, stream);   // J resident clients
    const int in = dtype_in == 0 ? 0 : 1;
    return a.acc_lo ? accumulate_t<true>(a, in, s, stream) : accumulate_t<false>(a, in, s, stream);
}

}  // namespace fa
