// Reduce kernels over resident client updates (see kernels.cuh for the operations and
// device.cuh for the shared conventions): reduce_bulk_kernel takes J <= 16 clients per
// launch over common segments, either writing the running sum (batched accumulate) or
// dividing and rounding straight to the output (a whole resident round).  It is a
// warp-specialised bulk-copy pipeline with one persistent CTA per SM.
#include "device.cuh"

namespace fa {

namespace {

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


// ----------------------------------------------------------------- host side
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

template <bool kComp>
cudaError_t prepare_reduce_shapes_t(LaunchShape* s) {
    const int c = kComp ? 1 : 0;
    cudaError_t r = cudaSuccess;
    auto keep = [&r](cudaError_t x) { if (r == cudaSuccess) r = x; };
    keep(prepare_reduce<float, float, false, kComp>(&s->reduce_ctas_per_sm[c][0][0]));
    keep(prepare_reduce<float, float, true, kComp>(&s->reduce_ctas_per_sm[c][0][1]));
    keep(prepare_reduce<float, uint16_t, true, kComp>(&s->reduce_ctas_per_sm[c][0][2]));
    keep(prepare_reduce<uint16_t, float, false, kComp>(&s->reduce_ctas_per_sm[c][1][0]));
    keep(prepare_reduce<uint16_t, float, true, kComp>(&s->reduce_ctas_per_sm[c][1][1]));
    keep(prepare_reduce<uint16_t, uint16_t, true, kComp>(&s->reduce_ctas_per_sm[c][1][2]));
    return r;
}

template <bool kComp>
cudaError_t reduce_sum_t(const AccArgs& a, int in, const LaunchShape& s, cudaStream_t stream) {
    const int c = kComp ? 1 : 0;
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

}  // namespace

cudaError_t prepare_reduce_shapes(LaunchShape* s) {
    cudaError_t e = prepare_reduce_shapes_t<false>(s);
    if (e == cudaSuccess) e = prepare_reduce_shapes_t<true>(s);
    return e;
}

cudaError_t launch_reduce_sum(const AccArgs& a, int dtype_in, const LaunchShape& s,
                              cudaStream_t stream) {
    if (a.nseg == 0 || a.nseg > static_cast<uint32_t>(kMaxSegs) || a.err == nullptr)
        return cudaErrorInvalidValue;
    if (a.J < 2 || a.J > static_cast<uint32_t>(kMaxBatch)) return cudaErrorInvalidValue;
    const int in = dtype_in == 0 ? 0 : 1;
    return a.acc_lo ? reduce_sum_t<true>(a, in, s, stream) : reduce_sum_t<false>(a, in, s, stream);
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

}  // namespace fa
