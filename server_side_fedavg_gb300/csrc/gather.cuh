// Subset reduce (fa_reduce_subsets): its launch interface and host planning.  Kept apart
// from kernels.cuh so that the other kernels' sources do not depend on it.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "kernels.cuh"

namespace fa {

// kGatherStages input stages of kGatherStageBytes each.  A tile of a key with J reporters
// holds gather_tile(J, dtype_in) elements: the most that J reporter tiles fit in one
// stage (a multiple of 256), so keys with fewer reporters take longer tiles and a round
// has as few tiles as its bytes allow.
constexpr int kGatherStages = 3;
constexpr int kGatherStageBytes = 73728;

// Elements per tile of a key with J reporters of s_in bytes each (host and device).
#ifdef __CUDACC__
__host__ __device__
#endif
constexpr uint32_t gather_tile_for(uint32_t J, uint32_t s_in) {
    return (kGatherStageBytes / ((J ? J : 1u) * s_in)) / 256u * 256u;
}

// Round-level reduce of client key subsets (fa_reduce_subsets): one segment per key to
// write, each with its own reporters.  Reporter j of segment s is src[s.src0 + j], in the
// order the contributions apply.
struct GathSeg {
    uint64_t len;       // elements of the key
    void* out;          // destination of element 0 (dtype_out)
    Divisor div;        // N_p
    uint32_t J;         // reporters (1..16)
    uint32_t src0;      // first reporter in the source table
    uint32_t tile0;     // first tile (set by launch_gather_final)
    uint32_t vec_ok;    // 1: the output and every reporter's input are 16-byte aligned
};

struct GathSrc {
    const void* x;      // the reporter's values of this key (dtype_in, device memory)
    float w;            // (float) n_k
    uint32_t pad;
};

struct GathArgs {
    const GathSeg* segs;         // device table, nseg entries sorted by tile0
    const GathSrc* src;          // device table
    const uint32_t* cta;         // device table, nchunk + 1 pairs (plan_gather_ctas): chunk c
                                 // is tiles [cta[2c], cta[2c + 2]), its first tile in
                                 // segment cta[2c + 1]
    uint32_t* counter;           // device word, 0 at launch: chunks taken after the first
    unsigned int* err;           // the caller's device error word
    uint32_t nseg;
    uint32_t ntiles;             // tiles over all segments (plan_gather_tiles)
    uint32_t jmax;               // largest J over the segments (1..16)
    uint32_t grid;               // CTAs (gather_grid)
    uint32_t nchunk;             // chunks of work (gather_chunks, >= grid)
};

// The same tables in compact form, carried in the launch's own parameters when a round is
// small enough (gather_inline_layout): no upload before the launch and no table reads
// from global memory in the kernel.  A reporter is a client (its base pointer and weight
// in the client tables) and the key's element offset in that client's buffer.
struct GathSegP {
    void* out;          // destination of element 0 (dtype_out)
    Divisor div;        // N_p
    uint32_t len;       // elements of the key (< 2^32)
    uint32_t tile0;     // first tile
    uint16_t src0;      // first reporter in the reporter table
    uint8_t J;          // reporters (1..16)
    uint8_t vec_ok;     // 1: the output and every reporter's input are 16-byte aligned
};
static_assert(sizeof(GathSegP) == 32, "compact segment");

struct GathSrcP {
    uint32_t off;       // element offset of the key in the client's buffer (< 2^32)
    uint32_t client;    // index into the client tables
};

constexpr uint32_t kGathInlineBlob = 32640;   // bytes of tables in the parameters

struct GathInline {
    unsigned int* err;          // the caller's device error word
    uint32_t* counter;          // two device words of the caller's context, 0 at launch: units
                                // handed out, CTAs done; the launch leaves both at 0
    uint32_t pad0;
    uint32_t nseg;
    uint32_t nsrc;
    uint32_t nclient;
    uint32_t ntiles;
    uint32_t pad;
    uint32_t jmax;
    uint32_t grid;              // CTAs (gather_grid)
    uint32_t src_off;           // byte offsets in blob: reporters, client bases, client weights
    uint32_t base_off;          //   (the segments start at 0)
    uint32_t w_off;
    uint32_t unit_tiles;        // tiles per unit of work (gather_unit_tiles)
    alignas(16) uint8_t blob[kGathInlineBlob];
};
static_assert(sizeof(GathInline) <= 32764, "kernel parameters are limited to 32764 bytes");

// Byte offsets of the reporter, client-base and client-weight tables in GathInline::blob
// for nseg segments, nsrc reporters and nclient clients; false if they do not fit.
bool gather_inline_layout(uint32_t nseg, uint32_t nsrc, uint32_t nclient, uint32_t* src_off,
                          uint32_t* base_off, uint32_t* w_off);

// Tiles per unit of work of an inline launch: consecutive tiles, so that a CTA reads a
// segment's entries from the tables once per unit (or key boundary), not once per tile,
// while about eight units per CTA keep the hand-out balanced.
uint32_t gather_unit_tiles(uint32_t ntiles, uint32_t grid);

// Launches the subset reduce with its tables in the parameters, as a programmatic
// dependent of the previous kernel on the stream.  The caller fills every field; units
// of unit_tiles consecutive tiles are handed out from counter[0].
cudaError_t launch_gather_inline(const GathInline& p, int dtype_in, int dtype_out, bool comp,
                                 const LaunchShape& s, cudaStream_t stream);

// Round-level subset reduce: out = RNE(sum over the segment's reporters, in order, / N_p)
// per segment, straight from the reporters' inputs (no running sum); comp: compensated
// arithmetic (Dot2), the same operation sequence as every other path.  The caller numbers
// the tiles of its host copy of the segment table with plan_gather_tiles, takes
// grid = gather_grid(...) and nchunk = gather_chunks(...), splits the tiles into chunks
// with plan_gather_ctas, uploads the three tables and a zero counter word, and launches
// with a.ntiles, a.grid and a.nchunk set.  Each CTA starts with chunk blockIdx.x and
// takes further chunks from the counter.
// Elements per tile of a key with J reporters (gather_tile_for).
uint32_t gather_tile(uint32_t J, int dtype_in);
// Sets tile0 of every segment (each segment's tiles of gather_tile(J, dtype_in)
// elements, numbered across the segments in order); false if there would be more than
// 2^32 - 1 tiles.
bool plan_gather_tiles(GathSeg* segs, uint32_t nseg, int dtype_in, uint32_t* ntiles);
// CTAs of a subset-reduce launch over ntiles tiles (a persistent grid, at most one
// resident wave).
uint32_t gather_grid(uint32_t ntiles, int dtype_in, int dtype_out, bool comp, const LaunchShape& s);
// Chunks of work of a subset-reduce launch: about four tiles each, at least one per CTA,
// at most kMaxGatherChunks.
constexpr uint32_t kMaxGatherChunks = 65536;
uint32_t gather_chunks(uint32_t ntiles, uint32_t grid);
// Splits tiles [0, ntiles) into `grid` contiguous runs (chunks) of about equal HBM bytes
// (a tile of segment s moves cnt * (J_s * s_in + s_out) bytes, cnt up to that segment's
// tile size), so that keys with more reporters do not weigh more per chunk.  Writes grid + 1 pairs to cta: cta[2b] is chunk
// b's first tile (0 for b = 0, ntiles for b = grid, and in between the first tile whose
// preceding bytes reach b / grid of the total), cta[2b + 1] the last segment whose first
// tile is at or before it.  Segments numbered by plan_gather_tiles.
void plan_gather_ctas(const GathSeg* segs, uint32_t nseg, uint32_t ntiles, int dtype_in,
                      int dtype_out, uint32_t grid, uint32_t* cta);
cudaError_t launch_gather_final(const GathArgs& a, int dtype_in, int dtype_out, bool comp,
                                const LaunchShape& s, cudaStream_t stream);

}  // namespace fa
