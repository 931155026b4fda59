// Host planning of a subset-reduce launch (fa_reduce_subsets): tile size, tile numbering,
// grid size and the split of the tiles among the CTAs.  Plain C++: the CPU tests compile
// it without CUDA device code.
#include "gather.cuh"
#include "tiles.hpp"

namespace fa {

uint32_t gather_tile(uint32_t J, int dtype_in) { return gather_tile_for(J, dtype_in == 0 ? 4u : 2u); }

bool plan_gather_tiles(GathSeg* segs, uint32_t nseg, int dtype_in, uint32_t* ntiles) {
    uint64_t t = 0;
    for (uint32_t i = 0; i < nseg; ++i) {
        const uint64_t tile = gather_tile(segs[i].J, dtype_in);
        segs[i].tile0 = static_cast<uint32_t>(t);
        t += (segs[i].len + tile - 1) / tile;
        if (t > 0xFFFFFFFFull) return false;
    }
    *ntiles = static_cast<uint32_t>(t);
    return true;
}

uint32_t gather_grid(uint32_t ntiles, int dtype_in, int dtype_out, bool comp, const LaunchShape& s) {
    const int per = s.gather_ctas_per_sm[comp ? 1 : 0][dtype_in == 0 ? 0 : 1][dtype_out == 0 ? 0 : 1];
    return grid_for(ntiles, s.sms, per);
}

bool gather_inline_layout(uint32_t nseg, uint32_t nsrc, uint32_t nclient, uint32_t* src_off,
                          uint32_t* base_off, uint32_t* w_off) {
    const uint64_t so = static_cast<uint64_t>(nseg) * sizeof(GathSegP);
    const uint64_t bo = so + static_cast<uint64_t>(nsrc) * sizeof(GathSrcP);
    const uint64_t wo = bo + static_cast<uint64_t>(nclient) * sizeof(void*);
    const uint64_t end = wo + static_cast<uint64_t>(nclient) * sizeof(float);
    if (end > kGathInlineBlob || nsrc > 0xFFFFu) return false;
    *src_off = static_cast<uint32_t>(so);
    *base_off = static_cast<uint32_t>(bo);
    *w_off = static_cast<uint32_t>(wo);
    return true;
}

uint32_t gather_unit_tiles(uint32_t ntiles, uint32_t grid) {
    const uint64_t per = grid ? ntiles / (8ull * grid) : 1;
    return per < 1 ? 1u : static_cast<uint32_t>(per);
}

uint32_t gather_chunks(uint32_t ntiles, uint32_t grid) {
    uint32_t n = ntiles / 4;
    if (n > kMaxGatherChunks) n = kMaxGatherChunks;
    if (n < grid) n = grid;
    return n < ntiles ? n : ntiles;
}

void plan_gather_ctas(const GathSeg* segs, uint32_t nseg, uint32_t ntiles, int dtype_in,
                      int dtype_out, uint32_t grid, uint32_t* cta) {
    // exact integer arithmetic: boundary b (1..grid-1) is the first tile t whose preceding
    // bytes P(t) satisfy P(t) * grid >= total * b; tiles of one segment cost the same
    // except its last (ragged) one, so each boundary is found by one division
    using u128 = unsigned __int128;
    const uint64_t si = dtype_in == 0 ? 4u : 2u, so = dtype_out == 0 ? 4u : 2u;
    u128 total = 0;
    for (uint32_t i = 0; i < nseg; ++i) total += static_cast<u128>(segs[i].len) * (segs[i].J * si + so);
    cta[0] = 0;
    uint32_t b = 1;
    u128 before = 0;                                    // P(first tile of segment i)
    for (uint32_t i = 0; i < nseg && b < grid; ++i) {
        const GathSeg& g = segs[i];
        const uint32_t nt = (i + 1 < nseg ? segs[i + 1].tile0 : ntiles) - g.tile0;
        const u128 per = g.J * si + so;                 // bytes per element of this segment
        const u128 end = before + static_cast<u128>(g.len) * per;
        if (nt > 0) {
            const u128 c = static_cast<u128>(gather_tile(g.J, dtype_in)) * per;   // bytes of a full tile
            while (b < grid && end * grid > total * b) {
                const u128 want = total * b, have = before * grid;
                const u128 k = want > have ? (want - have + c * grid - 1) / (c * grid) : 0;
                cta[2 * b++] = k < nt ? g.tile0 + static_cast<uint32_t>(k) : g.tile0 + nt;
            }
        }
        before = end;
    }
    while (b < grid) cta[2 * b++] = ntiles;
    cta[2 * grid] = ntiles;
    // the segment of each CTA's first tile, as the kernel's forward walk defines it: the
    // last segment whose first tile is at or before it
    uint32_t si_ = 0;
    for (uint32_t q = 0; q <= grid; ++q) {
        while (si_ + 1 < nseg && segs[si_ + 1].tile0 <= cta[2 * q]) ++si_;
        cta[2 * q + 1] = si_;
    }
}

}  // namespace fa
