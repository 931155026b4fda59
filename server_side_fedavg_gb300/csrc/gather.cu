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
// its own reporters applied in table order -- the final mode of reduce_bulk_kernel with
// per-segment inputs and weights.  The tables are either in device memory (GathArgs,
// uploaded on the stream just before a plain launch) or, for a small round, in the
// launch's own parameters (GathInline, a programmatic dependent launch with no upload).

// A segment as the kernel uses it, from either form of the tables.
struct SegV {
    uint64_t len;
    void* out;
    Divisor div;
    uint32_t J;
    uint32_t src0;
    uint32_t tile0;
    uint32_t vec_ok;
    uint32_t tile;      // elements per tile (gather_tile_for(J, s_in); set by the loader)
};

// Tables in device memory.
struct DevTables {
    const GathArgs* a;
    __device__ __forceinline__ uint32_t nseg() const { return a->nseg; }
    __device__ __forceinline__ uint32_t tile0(uint32_t i) const { return a->segs[i].tile0; }
    __device__ __forceinline__ SegV seg(uint32_t i) const {
        const GathSeg& g = a->segs[i];
        return SegV{g.len, g.out, g.div, g.J, g.src0, g.tile0, g.vec_ok, 0u};
    }
    __device__ __forceinline__ const void* x(const SegV& s, uint32_t j, uint32_t) const {
        return a->src[s.src0 + j].x;
    }
    __device__ __forceinline__ float w(const SegV& s, uint32_t j) const { return a->src[s.src0 + j].w; }
};

// Tables in the launch's parameters (read through the constant cache; every access is
// uniform across a warp).
struct ParTables {
    const GathInline* p;
    __device__ __forceinline__ const GathSegP& g(uint32_t i) const {
        return reinterpret_cast<const GathSegP*>(p->blob)[i];
    }
    __device__ __forceinline__ const GathSrcP& r(uint32_t k) const {
        return reinterpret_cast<const GathSrcP*>(p->blob + p->src_off)[k];
    }
    __device__ __forceinline__ uint32_t nseg() const { return p->nseg; }
    __device__ __forceinline__ uint32_t tile0(uint32_t i) const { return g(i).tile0; }
    __device__ __forceinline__ SegV seg(uint32_t i) const {
        const GathSegP& s = g(i);
        return SegV{s.len, s.out, s.div, s.J, s.src0, s.tile0, s.vec_ok, 0u};
    }
    __device__ __forceinline__ const void* x(const SegV& s, uint32_t j, uint32_t s_in) const {
        const GathSrcP& q = r(s.src0 + j);
        const char* base = reinterpret_cast<const char* const*>(p->blob + p->base_off)[q.client];
        return base + static_cast<uint64_t>(q.off) * s_in;
    }
    __device__ __forceinline__ float w(const SegV& s, uint32_t j) const {
        return reinterpret_cast<const float*>(p->blob + p->w_off)[r(s.src0 + j).client];
    }
};

// One element through global memory (ragged tails, unaligned segments).
template <typename Tin, typename Tout, bool kComp, typename Tab>
__device__ __forceinline__ void gath_one(const Tab& tb, const SegV& sg, uint64_t e) {
    float r, rl = 0.0f;
    contrib_first<kComp>(tb.w(sg, 0), load_one<Tin>(static_cast<const Tin*>(tb.x(sg, 0, sizeof(Tin))) + e),
                         r, rl);
    for (uint32_t j = 1; j < sg.J; ++j)
        contrib_add<kComp>(tb.w(sg, j), load_one<Tin>(static_cast<const Tin*>(tb.x(sg, j, sizeof(Tin))) + e),
                           r, rl);
    store_one<Tout>(sg.out, e, quotient_out<kComp, Tout>(r, rl, sg.div));
}

// What the compute warps need about a tile, written to shared memory by the loader
// (which already holds the tile's segment and reporters in registers) before it hands
// the stage over, so that the compute warps read no table per tile: t = kNoTile marks
// the end of the CTA's work.
struct TileMeta {
    uint64_t e0;               // first element of the tile in its key
    void* out;                 // the key's output (element 0)
    Divisor div;               // N_p
    uint32_t cnt;              // elements in the tile
    uint32_t J;                // reporters
    uint32_t vec;              // 1: bulk copies (aligned and at least kVec elements)
    uint32_t t;                // tile index, or kNoTile
    uint32_t si;               // segment
    uint32_t xb;               // bytes of one reporter's tile in the stage
    uint32_t pad[3];
    float w[kMaxBatch];        // the reporters' weights, in order
};
static_assert(sizeof(TileMeta) % 16 == 0, "meta slots stay 16-byte aligned");
constexpr uint32_t kNoTile = 0xFFFFFFFFu;
// 16 compute warps, then a loader warp.  A tile's reduction is a chain of dependent
// shared-memory loads and fmas per element (one reporter after another), so the compute
// warps hide latency by numbers.
constexpr int kGatherWarps = 16;
constexpr int kGatherCompute = kGatherWarps * 32;
constexpr int kGatherThreads = kGatherCompute + 32;
constexpr uint32_t kMaxInlineSegs = kGathInlineBlob / sizeof(GathSegP);

// Shared memory of a CTA: the input stages, the barriers (full / empty per stage), the
// tile metadata (per stage) and, for inline tables, each segment's first tile
// (nseg_cached entries).
__host__ __device__ constexpr size_t gather_smem_bytes(uint32_t nseg_cached) {
    return static_cast<size_t>(kGatherStages) * kGatherStageBytes + 2 * kGatherStages * sizeof(uint64_t) +
           kGatherStages * sizeof(TileMeta) + nseg_cached * sizeof(uint32_t);
}

__device__ __forceinline__ TileAt tile_in(const SegV& sg, uint32_t si, uint32_t t) {
    TileAt r;
    r.si = si;
    r.e0 = static_cast<uint64_t>(t - sg.tile0) * sg.tile;
    const uint64_t rem = sg.len - r.e0;
    r.cnt = rem < sg.tile ? static_cast<uint32_t>(rem) : sg.tile;
    return r;
}

// Two roles per CTA:
//  - the loader (one lane of warp 16) fills input stage s (jmax reporter tiles) with bulk
//    loads once the compute warps have released it (empty[s]), arming full[s] with the
//    byte count and writing the tile's metadata;
//  - the compute warps (0-15) wait for full[s], reduce the tile from stage s, write the
//    results straight from registers with 16-byte stores (coalesced across each warp)
//    and release the stage.
// Work is handed out dynamically, so that CTAs that run faster (or start earlier) take
// more of the round and all finish together: CTA b starts with unit b and then takes
// unit grid + atomicAdd(counter, 1) until none is left; the loader keeps two such
// requests in flight, so their latency is hidden behind the units before them.  A unit
// is a chunk of about equal bytes planned on the host (device tables: nchunk + 1 (first
// tile, segment) pairs) or unit_tiles consecutive tiles, whose first segment the loader
// finds by a binary search over the segments' first tiles, copied to shared memory at
// the start (inline tables).  Either way a CTA reads a segment's table entries once per
// unit or key boundary, not per tile.
template <typename Tin, typename Tout, bool kComp, bool kInline, typename Tab>
__device__ __forceinline__ void gather_body(const Tab& tb, uint32_t grid, uint32_t nunit, uint32_t ntiles,
                                            uint32_t unit_tiles, const uint32_t* cta, uint32_t* counter,
                                            uint32_t* done, unsigned int* err) {
    constexpr uint32_t IB = kGatherStageBytes;    // one input stage
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* ins = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kGatherStages * IB);
    uint64_t* empty = full + kGatherStages;
    TileMeta* meta = reinterpret_cast<TileMeta*>(empty + kGatherStages);
    const uint32_t* t0s = reinterpret_cast<const uint32_t*>(meta + kGatherStages);
    const uint32_t warp = threadIdx.x / 32u, lane = threadIdx.x & 31u;
    const uint32_t nseg = tb.nseg();

    if (warp == static_cast<uint32_t>(kGatherWarps)) {
        // ------------------------------------------------------------ loader
        if (lane != 0) return;
        uint32_t unit = blockIdx.x;            // < nunit: the host plans nunit >= grid
        uint32_t q0 = grid < nunit ? grid + atomicAdd(counter, 1u) : nunit;
        uint32_t q1 = grid < nunit ? grid + atomicAdd(counter, 1u) : nunit;
        uint32_t t, tend, cur;
        if constexpr (kInline) {
            t = unit < nunit ? unit * unit_tiles : ntiles;
            tend = t + unit_tiles < ntiles ? t + unit_tiles : ntiles;
            cur = 0;
        } else {
            t = cta[2 * unit];
            cur = cta[2 * unit + 1];
            tend = cta[2 * unit + 2];
        }
        // the current segment, kept in registers while its tiles are issued
        uint32_t have = 0xFFFFFFFFu, nt0 = 0;
        SegV sg{};
        const void* xp[kMaxBatch];
        float wv[kMaxBatch];
        bool ok = true;
        uint32_t issued = 0;                   // tiles published to the stages
        for (;; ++issued) {
            while (t == tend && q0 < nunit) {        // this unit is done: take the next one
                unit = q0;
                q0 = q1;
                q1 = grid + atomicAdd(counter, 1u);
                if constexpr (kInline) {
                    t = unit * unit_tiles;
                    tend = t + unit_tiles < ntiles ? t + unit_tiles : ntiles;
                } else {
                    t = cta[2 * unit];
                    cur = cta[2 * unit + 1];
                    tend = cta[2 * unit + 2];
                }
            }
            const uint32_t s = issued % kGatherStages;
            if (issued >= static_cast<uint32_t>(kGatherStages)) {
                ok = mbar_wait(smem_addr(&empty[s]), ((issued / kGatherStages) - 1) & 1u);
                if (!ok) break;
            }
            const uint32_t bar = smem_addr(&full[s]);
            TileMeta& m = meta[s];
            if (t == tend) {                   // no work left: tell the compute warps
                m.t = kNoTile;
                mbar_arrive(bar);
                break;
            }
            if constexpr (kInline) {
                if (t >= nt0) {
                    // the last segment whose first tile is at or before t, in [cur, nseg):
                    // this CTA's tiles only increase
                    uint32_t lo = cur, hi = nseg;
                    while (hi - lo > 1) {
                        const uint32_t mid = (lo + hi) / 2;
                        if (t0s[mid] <= t) lo = mid; else hi = mid;
                    }
                    cur = lo;
                    nt0 = cur + 1 < nseg ? t0s[cur + 1] : 0xFFFFFFFFu;
                }
            } else {
                if (cur != have) nt0 = cur + 1 < nseg ? tb.tile0(cur + 1) : 0xFFFFFFFFu;
                while (t >= nt0) {
                    ++cur;
                    nt0 = cur + 1 < nseg ? tb.tile0(cur + 1) : 0xFFFFFFFFu;
                }
            }
            if (cur != have) {
                sg = tb.seg(cur);
                sg.tile = gather_tile_for(sg.J, sizeof(Tin));
#pragma unroll
                for (int jj = 0; jj < kMaxBatch; ++jj) {
                    const bool in = jj < static_cast<int>(sg.J);
                    xp[jj] = in ? tb.x(sg, jj, sizeof(Tin)) : nullptr;
                    wv[jj] = in ? tb.w(sg, jj) : 0.0f;
                }
                have = cur;
            }
            const TileAt ta = tile_in(sg, cur, t);
            const uint32_t XB = sg.tile * sizeof(Tin);    // one reporter's tile in the stage
            const uint32_t n8 = ta.cnt / kVec;
            const bool bulk = sg.vec_ok && n8 > 0;
            m.e0 = ta.e0;
            m.out = sg.out;
            m.div = sg.div;
            m.cnt = ta.cnt;
            m.J = sg.J;
            m.vec = bulk ? 1u : 0u;
            m.t = t;
            m.si = cur;
            m.xb = XB;
#pragma unroll
            for (int jj = 0; jj < kMaxBatch; ++jj) m.w[jj] = wv[jj];
            ++t;
            if (bulk) {
                const uint32_t xb = n8 * kVec * sizeof(Tin);
                mbar_expect(bar, sg.J * xb);
                uint8_t* st = ins + s * IB;
#pragma unroll
                for (int jj = 0; jj < kMaxBatch; ++jj) {
                    if (jj >= static_cast<int>(sg.J)) break;
                    bulk_load(st + jj * XB, static_cast<const Tin*>(xp[jj]) + ta.e0, xb, bar);
                }
            } else {
                mbar_arrive(bar);
            }
        }
        if (!ok) {
            // a wait gave up: flag it, and wait (bounded) for the loads still in flight
            atomicOr(err, kErrWaitTimeout);
            for (uint32_t i = issued >= static_cast<uint32_t>(kGatherStages) ? issued - kGatherStages : 0u;
                 i < issued; ++i)
                mbar_wait(smem_addr(&full[i % kGatherStages]), (i / kGatherStages) & 1u);
        }
        if (done != nullptr) {
            // this CTA takes no more units; the last CTA to get here leaves the counter and
            // this word at 0 for the next launch (the fence orders each CTA's last hand-out
            // before its count, so the last one sees every hand-out done)
            __threadfence();
            if (atomicAdd(done, 1u) == grid - 1u) {
                atomicExch(counter, 0u);
                atomicExch(done, 0u);
            }
        }
        return;
    }

    // ---------------------------------------------------------------- compute warps
    for (uint32_t i = 0;; ++i) {
        const uint32_t s = i % kGatherStages;
        if (!mbar_wait(smem_addr(&full[s]), (i / kGatherStages) & 1u)) {
            atomicOr(err, kErrWaitTimeout);
            break;
        }
        const TileMeta& m = meta[s];
        if (m.t == kNoTile) break;
        const uint32_t J = m.J, cnt = m.cnt, XB = m.xb;
        const uint64_t e0 = m.e0;
        const uint8_t* st = ins + s * IB;
        if (m.vec) {
            const uint32_t n8 = cnt / kVec;
            const Divisor div = m.div;
            void* out = m.out;
            float wv[kMaxBatch];
#pragma unroll
            for (int j = 0; j < kMaxBatch; ++j) wv[j] = m.w[j];
            for (uint32_t v = threadIdx.x; v < n8; v += kGatherCompute) {
                float r[8], rl[8];
                {
                    float xv[8];
                    smem_vec8<Tin>(st, v, xv);
#pragma unroll
                    for (int e = 0; e < 8; ++e) contrib_first<kComp>(wv[0], xv[e], r[e], rl[e]);
                }
#pragma unroll
                for (int j = 1; j < kMaxBatch; ++j) {
                    if (j >= static_cast<int>(J)) break;
                    float xv[8];
                    smem_vec8<Tin>(st + j * XB, v, xv);
#pragma unroll
                    for (int e = 0; e < 8; ++e) contrib_add<kComp>(wv[j], xv[e], r[e], rl[e]);
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) r[e] = quotient_out<kComp, Tout>(r[e], rl[e], div);
                store8_global<Tout>(out, e0 + static_cast<uint64_t>(v) * kVec, r);
            }
            const uint32_t tail = cnt - n8 * kVec;
            if (threadIdx.x < tail) {
                const SegV sg = tb.seg(m.si);
                gath_one<Tin, Tout, kComp>(tb, sg, e0 + n8 * kVec + threadIdx.x);
            }
        } else {
            const SegV sg = tb.seg(m.si);
            for (uint32_t e = threadIdx.x; e < cnt; e += kGatherCompute)
                gath_one<Tin, Tout, kComp>(tb, sg, e0 + e);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&empty[s]));
    }
}

// The barriers of one CTA and, for inline tables, the segments' first tiles in shared
// memory (nseg_cached entries read through tb).
template <typename Tab>
__device__ __forceinline__ void gather_setup(const Tab& tb, uint32_t nseg_cached) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(kGatherStages) * kGatherStageBytes);
    uint64_t* empty = full + kGatherStages;
    uint32_t* t0s = reinterpret_cast<uint32_t*>(reinterpret_cast<TileMeta*>(empty + kGatherStages) +
                                                kGatherStages);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kGatherStages; ++s) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&full[s])) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(&empty[s])),
                         "r"(kGatherWarps) : "memory");
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    for (uint32_t i = threadIdx.x; i < nseg_cached; i += blockDim.x) t0s[i] = tb.tile0(i);
    __syncthreads();
}

// Tables in device memory: a plain launch after their upload; units are the planned chunks.
template <typename Tin, typename Tout, bool kComp>
__global__ void __launch_bounds__(kGatherThreads, 1) reduce_gather_kernel(const __grid_constant__ GathArgs a) {
    const DevTables tb{&a};
    gather_setup(tb, 0u);
    gather_body<Tin, Tout, kComp, false>(tb, a.grid, a.nchunk, a.ntiles, 0u, a.cta, a.counter, nullptr, a.err);
}

// Tables in the parameters: a programmatic dependent launch (its set-up overlaps the
// previous kernel's tail; nothing in global memory is touched before that kernel has
// completed); units of unit_tiles tiles are counted in p.counter[0], and the launch leaves
// both counter words at 0 (so a captured launch replays as it ran).
template <typename Tin, typename Tout, bool kComp>
__global__ void __launch_bounds__(kGatherThreads, 1) reduce_gather_inline_kernel(
    const __grid_constant__ GathInline p) {
    const ParTables tb{&p};
    gather_setup(tb, p.nseg);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    gather_body<Tin, Tout, kComp, true>(tb, p.grid, (p.ntiles + p.unit_tiles - 1) / p.unit_tiles, p.ntiles,
                                        p.unit_tiles, nullptr, p.counter, p.counter + 1, p.err);
}

// ----------------------------------------------------------------- host side
template <typename Tin, typename Tout, bool kComp>
cudaError_t prepare_gather(int* occ) {
    const size_t smem = gather_smem_bytes(kMaxInlineSegs);
    cudaError_t e = cudaFuncSetAttribute(reduce_gather_kernel<Tin, Tout, kComp>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(reduce_gather_inline_kernel<Tin, Tout, kComp>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    int occ_inline = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ_inline, reduce_gather_inline_kernel<Tin, Tout, kComp>,
                                                      kGatherThreads, smem);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, reduce_gather_kernel<Tin, Tout, kComp>,
                                                      kGatherThreads, smem);
    if (e == cudaSuccess) *occ = std::min(*occ, occ_inline);
    return e;
}

template <typename Tin, typename Tout, bool kComp>
cudaError_t launch_gather_t(const GathArgs& a, cudaStream_t stream) {
    const size_t smem = gather_smem_bytes(0u);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.grid);
    cfg.blockDim = dim3(kGatherThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = nullptr;
    cfg.numAttrs = 0;
    return cudaLaunchKernelEx(&cfg, reduce_gather_kernel<Tin, Tout, kComp>, a);
}

template <typename Tin, typename Tout, bool kComp>
cudaError_t launch_inline_t(const GathInline& p, cudaStream_t stream) {
    return launch_dependent(reduce_gather_inline_kernel<Tin, Tout, kComp>, p.grid, kGatherThreads,
                            gather_smem_bytes(p.nseg), stream, p);
}

template <bool kComp>
cudaError_t inline_pick(const GathInline& p, int din, int dout, cudaStream_t stream) {
    if (din == 0)
        return dout == 0 ? launch_inline_t<float, float, kComp>(p, stream)
                         : launch_inline_t<float, uint16_t, kComp>(p, stream);
    return dout == 0 ? launch_inline_t<uint16_t, float, kComp>(p, stream)
                     : launch_inline_t<uint16_t, uint16_t, kComp>(p, stream);
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
        a.grid != gather_grid(a.ntiles, dtype_in, dtype_out, comp, s) || a.grid == 0 ||
        a.nchunk < a.grid || a.nchunk > a.ntiles)
        return cudaErrorInvalidValue;
    const int din = dtype_in == 0 ? 0 : 1, dout = dtype_out == 0 ? 0 : 1;
    return comp ? gather_pick<true>(a, din, dout, stream) : gather_pick<false>(a, din, dout, stream);
}

cudaError_t launch_gather_inline(const GathInline& p, int dtype_in, int dtype_out, bool comp,
                                 const LaunchShape& s, cudaStream_t stream) {
    if (p.nseg == 0 || p.ntiles == 0) return cudaSuccess;
    uint32_t so = 0, bo = 0, wo = 0;
    if (p.err == nullptr || p.counter == nullptr || p.jmax == 0 || p.nseg > kMaxInlineSegs ||
        p.unit_tiles == 0 ||
        p.jmax > static_cast<uint32_t>(kMaxBatch) ||
        p.grid != gather_grid(p.ntiles, dtype_in, dtype_out, comp, s) || p.grid == 0 ||
        !gather_inline_layout(p.nseg, p.nsrc, p.nclient, &so, &bo, &wo) || so != p.src_off ||
        bo != p.base_off || wo != p.w_off)
        return cudaErrorInvalidValue;
    const int din = dtype_in == 0 ? 0 : 1, dout = dtype_out == 0 ? 0 : 1;
    return comp ? inline_pick<true>(p, din, dout, stream) : inline_pick<false>(p, din, dout, stream);
}

}  // namespace fa
