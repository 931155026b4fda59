// Test-only C entry point over the host planning of a subset-reduce launch (compiled
// with g++ on the CPU, no CUDA device code): lets the CPU suite check how the tiles of
// a round are numbered and split among the CTAs.
#include <cstdint>
#include <vector>

#include "gather.cuh"

extern "C" {

// Segments of lens[i] elements with J[i] reporters each, tiles of gather_tile(J[i], din)
// elements.  Writes each segment's tile size and first tile, the tile count and the
// grid + 1 (first tile, segment) pairs of the CTA split.  Returns 0, or -1 if the tiles
// do not fit 32 bits.
int32_t gp_plan(const uint64_t* lens, const uint32_t* J, uint32_t nseg, int din, int dout,
                uint32_t grid, uint32_t* tiles, uint32_t* ntiles, uint32_t* tile0, uint32_t* cta) {
    std::vector<fa::GathSeg> segs(nseg);
    for (uint32_t i = 0; i < nseg; ++i) {
        segs[i] = fa::GathSeg{};
        segs[i].len = lens[i];
        segs[i].J = J[i];
        tiles[i] = fa::gather_tile(J[i], din);
    }
    if (!fa::plan_gather_tiles(segs.data(), nseg, din, ntiles)) return -1;
    for (uint32_t i = 0; i < nseg; ++i) tile0[i] = segs[i].tile0;
    fa::plan_gather_ctas(segs.data(), nseg, *ntiles, din, dout, grid, cta);
    return 0;
}

uint32_t gp_chunks(uint32_t ntiles, uint32_t grid) { return fa::gather_chunks(ntiles, grid); }

}  // extern "C"
