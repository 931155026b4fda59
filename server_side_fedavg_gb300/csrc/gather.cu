// Subset reduce kernel (fa_reduce_subsets; see kernels.cuh for the operation and
// device.cuh for the shared conventions): a round of client key subsets, each key with
// its own reporters, reduced straight to the output in one persistent launch -- a
// warp-specialised bulk-copy pipeline with one CTA per SM, its tiles handed out in
// chunks of about equal bytes planned on the host (gather_plan.cpp).
#include "device.cuh"
#include "gather.cuh"

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

// Stage metadata: the tile held by an input stage or an output buffer and its segment,
// or kNoTile once the CTA has no more work.  Written before the barrier that hands the
// stage or buffer over, read after waiting on it.
constexpr uint32_t kNoTile = 0xFFFFFFFFu;
constexpr int kGatherThreads = kBlock + 64;   // 8 compute warps, a loader and a storer warp

__host__ __device__ constexpr size_t gather_smem_bytes(uint32_t tile, uint32_t jmax, uint32_t s_in,
                                                       uint32_t s_out) {
    return static_cast<size_t>(tile) * (kGatherStages * jmax * s_in + kGatherOutBufs * s_out) +
           (2 * kGatherStages + 2 * kGatherOutBufs) * sizeof(uint64_t) +
           (kGatherStages + kGatherOutBufs) * sizeof(uint2);
}

// Tile t of segment si (t lies in that segment).
__device__ __forceinline__ TileAt gath_tile(const GathSeg* segs, uint32_t si, uint32_t t, uint32_t T) {
    const GathSeg& sg = segs[si];
    TileAt r;
    r.si = si;
    r.e0 = static_cast<uint64_t>(t - sg.tile0) * T;
    const uint64_t rem = sg.len - r.e0;
    r.cnt = rem < T ? static_cast<uint32_t>(rem) : T;
    return r;
}

// Three roles per CTA, each waiting only on the barrier of the buffer it needs next:
//  - the loader (one lane of warp 8) fills input stage s (jmax reporter tiles) with bulk
//    loads once the compute warps have released it (empty[s]), arming full[s] with the
//    byte count;
//  - the compute warps (0-7) wait for full[s] and for output buffer o to be free
//    (ofree[o]: its previous tile's store has read it), reduce the tile from stage s into
//    buffer o, release the stage (empty[s]) and hand the buffer on (ofull[o]);
//  - the storer (one lane of warp 9) writes buffer o to the output with one bulk store
//    and frees it once the store has read it.
// Stores therefore never delay the next loads.  Work is handed out in chunks: contiguous
// runs of tiles of about equal bytes planned on the host (cta: nchunk + 1 (first tile,
// segment) pairs).  CTA b starts with chunk b and then takes chunk
// grid + atomicAdd(counter, 1) until none is left, so CTAs that run faster (or start
// earlier) take more of the round and all finish together; the loader asks for the next
// chunk as soon as it starts one, so the atomic's latency is hidden behind that chunk.
template <typename Tin, typename Tout, bool kComp>
__global__ void __launch_bounds__(kGatherThreads, 1) reduce_gather_kernel(const __grid_constant__ GathArgs a) {
    const uint32_t T = a.tile;
    const uint32_t XB = T * sizeof(Tin);          // one reporter's input tile
    const uint32_t IB = a.jmax * XB;              // one input stage
    const uint32_t OB = T * sizeof(Tout);         // one output buffer
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* ins = smem;
    uint8_t* outs = smem + kGatherStages * IB;
    uint64_t* full = reinterpret_cast<uint64_t*>(outs + kGatherOutBufs * OB);
    uint64_t* empty = full + kGatherStages;
    uint64_t* ofull = empty + kGatherStages;
    uint64_t* ofree = ofull + kGatherOutBufs;
    uint2* meta = reinterpret_cast<uint2*>(ofree + kGatherOutBufs);
    uint2* ometa = meta + kGatherStages;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kGatherStages; ++s) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&full[s])) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(&empty[s])),
                         "r"(kReduceWarps) : "memory");
        }
        for (int o = 0; o < kGatherOutBufs; ++o) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(&ofull[o])),
                         "r"(kReduceWarps) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&ofree[o])) : "memory");
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const uint32_t warp = threadIdx.x / 32u, lane = threadIdx.x & 31u;

    if (warp == static_cast<uint32_t>(kReduceWarps)) {
        // ------------------------------------------------------------ loader
        if (lane != 0) return;
        uint32_t chunk = blockIdx.x;           // < nchunk: the host plans nchunk >= grid
        uint32_t t = a.cta[2 * chunk], cur = a.cta[2 * chunk + 1], tend = a.cta[2 * chunk + 2];
        uint32_t next = a.grid < a.nchunk ? a.grid + atomicAdd(a.counter, 1u) : a.nchunk;
        // the current segment, kept in registers while its tiles are issued
        uint32_t have = 0xFFFFFFFFu, nt0 = 0, J = 0, vec = 0;
        uint32_t t0 = 0;
        uint64_t len = 0;
        const void* xp[kMaxBatch];
        bool ok = true;
        uint32_t issued = 0;                   // tiles published to the stages
        for (;; ++issued) {
            while (t == tend && next < a.nchunk) {   // this chunk is done: take the next one
                chunk = next;
                t = a.cta[2 * chunk];
                cur = a.cta[2 * chunk + 1];
                tend = a.cta[2 * chunk + 2];
                next = a.grid + atomicAdd(a.counter, 1u);
            }
            const uint32_t s = issued % kGatherStages;
            if (issued >= static_cast<uint32_t>(kGatherStages)) {
                ok = mbar_wait(smem_addr(&empty[s]), ((issued / kGatherStages) - 1) & 1u);
                if (!ok) break;
            }
            const uint32_t bar = smem_addr(&full[s]);
            if (t == tend) {                   // no work left: tell the compute warps
                meta[s] = make_uint2(kNoTile, 0u);
                mbar_arrive(bar);
                break;
            }
            if (cur != have) nt0 = cur + 1 < a.nseg ? a.segs[cur + 1].tile0 : 0xFFFFFFFFu;
            while (t >= nt0) {
                ++cur;
                nt0 = cur + 1 < a.nseg ? a.segs[cur + 1].tile0 : 0xFFFFFFFFu;
            }
            if (cur != have) {
                const GathSeg& sg = a.segs[cur];
                J = sg.J;
                vec = sg.vec_ok;
                t0 = sg.tile0;
                len = sg.len;
                const GathSrc* src = a.src + sg.src0;
#pragma unroll
                for (int jj = 0; jj < kMaxBatch; ++jj)
                    xp[jj] = jj < static_cast<int>(J) ? src[jj].x : nullptr;
                have = cur;
            }
            meta[s] = make_uint2(t, cur);
            const uint64_t e0 = static_cast<uint64_t>(t - t0) * T;
            const uint64_t rem = len - e0;
            const uint32_t n8 = (rem < T ? static_cast<uint32_t>(rem) : T) / kVec;
            ++t;
            if (vec && n8 > 0) {
                const uint32_t xb = n8 * kVec * sizeof(Tin);
                mbar_expect(bar, J * xb);
                uint8_t* st = ins + s * IB;
#pragma unroll
                for (int jj = 0; jj < kMaxBatch; ++jj) {
                    if (jj >= static_cast<int>(J)) break;
                    bulk_load(st + jj * XB, static_cast<const Tin*>(xp[jj]) + e0, xb, bar);
                }
            } else {
                mbar_arrive(bar);
            }
        }
        if (!ok) {
            // a wait gave up: flag it, and wait (bounded) for the loads still in flight
            atomicOr(a.err, kErrWaitTimeout);
            for (uint32_t i = issued >= static_cast<uint32_t>(kGatherStages) ? issued - kGatherStages : 0u;
                 i < issued; ++i)
                mbar_wait(smem_addr(&full[i % kGatherStages]), (i / kGatherStages) & 1u);
        }
        return;
    }

    if (warp == static_cast<uint32_t>(kReduceWarps) + 1u) {
        // ------------------------------------------------------------ storer
        if (lane != 0) return;
        bool ok = true;
        for (uint32_t i = 0;; ++i) {
            const uint32_t o = i % kGatherOutBufs;
            ok = mbar_wait(smem_addr(&ofull[o]), (i / kGatherOutBufs) & 1u);
            if (!ok) break;
            const uint2 m = ometa[o];
            if (m.x == kNoTile) break;
            const TileAt ta = gath_tile(a.segs, m.y, m.x, T);
            const GathSeg& sg = a.segs[m.y];
            const uint32_t n8 = (sg.vec_ok && ta.cnt >= static_cast<uint32_t>(kVec)) ? ta.cnt / kVec : 0u;
            if (n8 > 0) {
                bulk_store(static_cast<Tout*>(sg.out) + ta.e0, outs + o * OB, n8 * kVec * sizeof(Tout));
                bulk_commit();
                asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
            }
            mbar_arrive(smem_addr(&ofree[o]));
        }
        if (!ok) atomicOr(a.err, kErrWaitTimeout);
        asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
        return;
    }

    // ---------------------------------------------------------------- compute warps
    for (uint32_t i = 0;; ++i) {
        const uint32_t s = i % kGatherStages, o = i % kGatherOutBufs;
        if (!mbar_wait(smem_addr(&full[s]), (i / kGatherStages) & 1u)) {
            atomicOr(a.err, kErrWaitTimeout);
            break;
        }
        const uint2 m = meta[s];
        if (i >= static_cast<uint32_t>(kGatherOutBufs) &&
            !mbar_wait(smem_addr(&ofree[o]), ((i / kGatherOutBufs) - 1) & 1u)) {
            atomicOr(a.err, kErrWaitTimeout);
            break;
        }
        if (m.x == kNoTile) {                  // no more tiles: tell the storer
            if (threadIdx.x == 0) ometa[o] = m;
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&ofull[o]));
            break;
        }
        const TileAt ta = gath_tile(a.segs, m.y, m.x, T);
        const GathSeg sg = a.segs[m.y];
        const bool bulk = sg.vec_ok && ta.cnt >= static_cast<uint32_t>(kVec);
        const uint32_t n8 = bulk ? ta.cnt / kVec : 0;
        const uint8_t* st = ins + s * IB;
        uint8_t* res = outs + o * OB;
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
        if (threadIdx.x == 0) ometa[o] = m;
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(smem_addr(&empty[s]));
            mbar_arrive(smem_addr(&ofull[o]));
        }
    }
}

// ----------------------------------------------------------------- host side
template <typename Tin, typename Tout, bool kComp>
cudaError_t prepare_gather(int* occ) {
    // the largest stage set any tile size picks (gather_tile keeps every one within it)
    const size_t smem = kGatherSmemBudget + gather_smem_bytes(0, 0, 0, 0);
    cudaError_t e = cudaFuncSetAttribute(reduce_gather_kernel<Tin, Tout, kComp>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, reduce_gather_kernel<Tin, Tout, kComp>,
                                                         kGatherThreads, smem);
}

template <typename Tin, typename Tout, bool kComp>
cudaError_t launch_gather_t(const GathArgs& a, cudaStream_t stream) {
    const size_t smem = gather_smem_bytes(a.tile, a.jmax, sizeof(Tin), sizeof(Tout));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.grid);
    cfg.blockDim = dim3(kGatherThreads);
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
        a.counter == nullptr || a.jmax == 0 || a.jmax > static_cast<uint32_t>(kMaxBatch) ||
        a.tile != gather_tile(a.jmax, dtype_in, dtype_out) ||
        a.grid != gather_grid(a.ntiles, dtype_in, dtype_out, comp, s) || a.grid == 0 ||
        a.nchunk < a.grid || a.nchunk > a.ntiles)
        return cudaErrorInvalidValue;
    const int din = dtype_in == 0 ? 0 : 1, dout = dtype_out == 0 ? 0 : 1;
    return comp ? gather_pick<true>(a, din, dout, stream) : gather_pick<false>(a, din, dout, stream);
}

}  // namespace fa
