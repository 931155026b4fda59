// Subset reduce kernel (fa_reduce_subsets; see kernels.cuh for the operation and
// device.cuh for the shared conventions): a round of client key subsets, each key with
// its own reporters, reduced straight to the output in one persistent launch -- a
// warp-specialised bulk-copy pipeline with one CTA per SM, its tiles split among the
// CTAs by bytes on the host (gather_plan.cpp).
#include "device.cuh"

namespace fa {

namespace {

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

template <typename Tin, typename Tout, bool kComp>
__global__ void __launch_bounds__(kReduceThreads, 1) reduce_gather_kernel(const __grid_constant__ GathArgs a) {
    const uint32_t T = a.tile;
    const uint32_t XB = T * sizeof(Tin);
    const uint32_t stage = T * (a.jmax * static_cast<uint32_t>(sizeof(Tin)) + static_cast<uint32_t>(sizeof(Tout)));
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * stage);
    uint64_t* done = full + kStages;
    // each CTA takes a contiguous run of tiles (balanced by bytes on the host) and starts
    // at the segment the host found for its first tile, so its walk through the segment
    // table moves by at most one entry per tile
    const uint32_t first = a.cta[2 * blockIdx.x];
    const uint32_t seg0 = a.cta[2 * blockIdx.x + 1];
    const uint32_t count = a.cta[2 * blockIdx.x + 2] - first;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&full[s])) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(&done[s])),
                         "r"(kReduceWarps) : "memory");
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

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

// ----------------------------------------------------------------- host side
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
cudaError_t launch_gather_t(const GathArgs& a, cudaStream_t stream) {
    const size_t smem = static_cast<size_t>(kStages) * a.tile *
                            (a.jmax * sizeof(Tin) + sizeof(Tout)) + 2 * kStages * sizeof(uint64_t);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.grid);
    cfg.blockDim = dim3(kReduceThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = nullptr;
    cfg.numAttrs = 0;
    return cudaLaunchKernelEx(&cfg, reduce_gather_kernel<Tin, Tout, kComp>, a);
}

template <bool kComp>
cudaError_t gather_pick(const GathArgs& a, int din, int dout, cudaStream_t stream) {
    if (din == 0)
        return dout == 0 ? launch_gather_t<float, float, kComp>(a, stream)
                         : launch_gather_t<float, uint16_t, kComp>(a, stream);
    return dout == 0 ? launch_gather_t<uint16_t, float, kComp>(a, stream)
                     : launch_gather_t<uint16_t, uint16_t, kComp>(a, stream);
}

template <bool kComp>
cudaError_t prepare_gather_shapes_t(LaunchShape* s) {
    const int c = kComp ? 1 : 0;
    cudaError_t r = cudaSuccess;
    auto keep = [&r](cudaError_t x) { if (r == cudaSuccess) r = x; };
    keep(prepare_gather<float, float, kComp>(&s->gather_ctas_per_sm[c][0][0]));
    keep(prepare_gather<float, uint16_t, kComp>(&s->gather_ctas_per_sm[c][0][1]));
    keep(prepare_gather<uint16_t, float, kComp>(&s->gather_ctas_per_sm[c][1][0]));
    keep(prepare_gather<uint16_t, uint16_t, kComp>(&s->gather_ctas_per_sm[c][1][1]));
    return r;
}

}  // namespace

cudaError_t prepare_gather_shapes(LaunchShape* s) {
    cudaError_t e = prepare_gather_shapes_t<false>(s);
    if (e == cudaSuccess) e = prepare_gather_shapes_t<true>(s);
    return e;
}

cudaError_t launch_gather_final(const GathArgs& a, int dtype_in, int dtype_out, bool comp,
                                const LaunchShape& s, cudaStream_t stream) {
    if (a.nseg == 0 || a.ntiles == 0) return cudaSuccess;
    if (a.err == nullptr || a.segs == nullptr || a.src == nullptr || a.cta == nullptr ||
        a.jmax == 0 || a.jmax > static_cast<uint32_t>(kMaxBatch) ||
        a.tile != gather_tile(a.jmax, dtype_in, dtype_out) ||
        a.grid != gather_grid(a.ntiles, dtype_in, dtype_out, comp, s))
        return cudaErrorInvalidValue;
    const int din = dtype_in == 0 ? 0 : 1, dout = dtype_out == 0 ? 0 : 1;
    return comp ? gather_pick<true>(a, din, dout, stream) : gather_pick<false>(a, din, dout, stream);
}

}  // namespace fa
