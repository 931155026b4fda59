// Host-side tiling helpers of the kernel launchers (plain C++, no device code): tile
// numbering across segments, persistent grid sizes and the reduce kernels' tile size.
#pragma once

#include <cstdint>

#include "kernels.cuh"

namespace fa {

// Sets tile0 of every segment (tiles of `tile` elements, numbered across the segments in
// order); false if there would be more than 2^32 - 1 tiles.
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

inline uint32_t grid_for(uint32_t ntiles, int sms, int per_sm) {
    uint32_t cap = static_cast<uint32_t>(sms > 0 ? sms : 1) *
                   static_cast<uint32_t>(per_sm > 0 ? per_sm : 1);
    return ntiles < cap ? ntiles : cap;
}

// Elements per reduce tile: the largest multiple of 256 whose stage fits the budget.
inline uint32_t reduce_tile(uint32_t elem_bytes) {
    uint32_t t = kReduceStageBytes / elem_bytes / 256 * 256;
    return t < 256 ? 256 : t;
}

}  // namespace fa
