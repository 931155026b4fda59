// Device kernels of the aggregation path and their launch interface.
//
//   accumulate  sum[i] = n_k * x[i]                (first contribution to element i)
//               sum[i] = fma(n_k, x[i], sum[i])    (every later one)
//   reduce      J resident clients in one pass, the same operation sequence in client
//               order with the partial sum in registers; either writes the running sum
//               (batched accumulate) or, in final mode, divides and rounds straight to
//               the output (a whole round when every update is resident)
//   finalize    out[i] = RNE(sum[i] / N_p)   (IEEE division, then RNE to bf16 or a
//                                             plain fp32 store); delta rounds add
//                                             server_lr * that quotient to a base
//
// Compensated mode (acc_lo != nullptr): the running sum is a pair (hi, lo) of fp32
// arrays updated by the Dot2 scheme of Ogita, Rump and Oishi ("Accurate sum and dot
// product", SIAM J. Sci. Comput. 26(6), 2005): each product n_k * x is split exactly
// into a rounded part and its error (fma), the rounded part is added to hi with an
// error-free TwoSum (Knuth), and both error terms are summed into lo.  The result is
// as accurate as a sum kept in about twice fp32's precision; finalize divides hi + lo.
//
// All are HBM-bandwidth bound streaming passes (about 0.1 flop per byte): no tensor
// cores.  Layout: the fp32 running sum is padded per key to 32 elements, so each key
// starts 128-byte aligned; in compensated mode lo has the same layout.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace fa {

constexpr int kBlock = 256;           // threads per CTA
constexpr int kVec = 8;               // elements per vector (16 B of bf16, 2 x 16 B of fp32)
constexpr int kTile = 4096;           // elements per tile of the finalize kernel
constexpr int kBulkTile = 8192;       // elements per pipeline stage of the streaming kernel
constexpr int kBulkTileComp = 6144;   // the same in compensated mode (a stage also holds lo)
constexpr int kDirectTile = kBlock * kVec;   // elements per tile of the direct-load accumulate
// Finalize CTAs per SM: with a tile's loads issued together, 4 CTAs (about 64 KB of loads
// in flight per SM) gave the best rate in a sweep of 2..8 on GB300; more in flight was slower.
constexpr int kFinCtasPerSm = 4;
constexpr int kMaxSegs = 48;          // segments per accumulate / reduce launch
constexpr int kMaxBatch = 16;         // resident clients per launch
constexpr int kReduceStageBytes = 73728;   // shared-memory budget per stage of the reduce kernel

// Device-side error bits, OR-ed into the caller's error word (AccArgs::err, RedArgs::err).
constexpr unsigned int kErrWaitTimeout = 1u;   // a bounded mbarrier wait gave up

// AccArgs::debug bits (test aids; 0 in normal use).
constexpr uint32_t kDebugFirstWaitExpires = 1u;   // streaming kernel: each CTA's first data
                                                  // wait gives up as if its bound ran out

// A divisor N (fp64 on the host) as an unevaluated pair of floats, hi = (float)N and
// lo = (float)(N - hi), with rcp = (float)(1 / hi).  lo is 0 whenever N is exact in fp32
// (every integer up to 2^24); the division then is one IEEE division.
struct Divisor {
    float hi;
    float lo;
    float rcp;
};

struct AccSeg {
    const void* x;      // one-client launches: this segment's input chunk (segments of one
                        // launch may come from different chunks); J > 1 uses AccArgs::x
    uint64_t x_off;     // element offset into the input chunk(s)
    uint64_t acc_idx;   // element index into the running sum
    uint64_t len;       // elements (>= 1)
    uint32_t first;     // 1: the first client of the launch starts the sum here
    uint32_t tile0;     // first tile of this segment (set by launch_accumulate)
    void* out;          // final launches: destination of the segment's element 0 (dtype_out)
    Divisor div;        // final launches: N_p
    uint32_t pad;
};

struct AccArgs {
    const void* x[kMaxBatch];   // J input chunk bases (device), dtype_in
    float w[kMaxBatch];         // (float) n_k per input
    float* acc;                 // running sum (compensated mode: its hi part)
    float* acc_lo;              // compensated mode: the error part, same layout; else nullptr
    unsigned int* err;          // the caller's device error word (never nullptr)
    uint32_t J;                 // 1..16
    uint32_t nseg;
    uint32_t ntiles;            // set by launch_accumulate
    uint32_t debug;             // kDebug* bits
    uint64_t vec_ok;            // bit s: segment s is 16-byte aligned for x and sum
    AccSeg seg[kMaxSegs];
};

struct RedSeg {
    uint64_t x_off;     // element offset into every input
    uint64_t acc_idx;   // element index into the running sum
    uint64_t len;       // elements (>= 1)
    void* out;          // final mode: destination of element 0 (dtype_out)
    Divisor div;        // final mode: N_p
    uint32_t read_sum;  // 1: earlier contributions are in the running sum
    uint32_t tile0;     // first tile (set by the launcher)
};

struct RedArgs {
    const void* x[kMaxBatch];   // J input bases (device), dtype_in
    float w[kMaxBatch];
    float* acc;
    float* acc_lo;              // compensated mode, else nullptr
    unsigned int* err;          // the caller's device error word
    uint32_t J;                 // 1..16
    uint32_t nseg;
    uint32_t ntiles;            // set by the launcher
    uint32_t tile;              // elements per tile (set by the launcher)
    uint32_t has_sum;           // set by the launcher: a stage holds a sum tile
    uint32_t pad;
    uint64_t vec_ok;            // bit s: segment s is 16-byte aligned for every pointer
    RedSeg seg[kMaxSegs];
};

struct FinSeg {
    uint64_t acc_idx;   // start in the running sum
    uint64_t len;       // elements
    void* out;          // destination of element 0 (device), dtype_out
    const void* base;   // delta rounds: current global model (dtype_out), else unused
    Divisor div;        // N_p
    uint32_t tile0;     // first tile of this segment
};

// Segments a finalize launch carries in its own parameters (48 B each, inside the 32,764
// bytes a launch takes): no table upload before the launch, and a launch captured into a
// CUDA graph replays from its own copy of the table.
constexpr uint32_t kFinInlineSegs = 600;

struct FinArgs {
    const FinSeg* segs;   // the segment table in device memory, or nullptr: seg[0..nseg)
    const float* acc;     // running sum (compensated mode: its hi part)
    const float* acc_lo;  // compensated mode: the lo part, else nullptr
    uint32_t nseg;
    uint32_t ntiles;
    FinSeg seg[kFinInlineSegs];
};
static_assert(sizeof(FinArgs) <= 32764, "kernel parameters are limited to 32764 bytes");

struct LaunchShape {
    int sms = 0;
    int bulk_ctas_per_sm[2][2] = {};       // [compensated][dtype_in], streaming kernel
    int direct_ctas_per_sm[2][2] = {};     // [compensated][dtype_in], direct-load accumulate
    int reduce_ctas_per_sm[2][2][3] = {};  // [compensated][dtype_in][sum mode, final fp32 out,
                                           // final bf16 out] (same for every J)
    int fin_ctas_per_sm[2][2][2] = {};     // [compensated][apply][dtype_out]
    int gather_ctas_per_sm[2][2][2] = {};  // [compensated][dtype_in][dtype_out]
};

// The pair form of a divisor given in fp64.
Divisor make_divisor(double n);

// Fills the occupancy table for the current device (and sets the kernels'
// shared-memory limits).
cudaError_t query_launch_shape(LaunchShape* s);

// The parts of query_launch_shape that live with their kernels (reduce kernel, subset
// reduce kernel, finalize kernel).
cudaError_t prepare_reduce_shapes(LaunchShape* s);
cudaError_t prepare_gather_shapes(LaunchShape* s);   // gather.cuh has the rest of its interface
cudaError_t prepare_finalize_shapes(LaunchShape* s);

// launch_accumulate with J = 2..16 resident clients: the reduce kernel in sum mode.
cudaError_t launch_reduce_sum(const AccArgs& a, int dtype_in, const LaunchShape& s,
                              cudaStream_t stream);

// dtype codes: 0 = fp32, 1 = bf16.  The caller fills x, w, acc, acc_lo, err, J (1..16),
// nseg, vec_ok, debug and each segment's x (J = 1) / x_off / acc_idx / len / first; the
// launcher numbers the tiles for the kernel it picks (J = 1: streaming kernel, else the
// reduce kernel in sum mode).
// Returns cudaErrorInvalidValue if the arguments are out of range.
cudaError_t launch_accumulate(const AccArgs& a, int dtype_in, const LaunchShape& s,
                              cudaStream_t stream);

// The last contribution to its elements (fa_accumulate_final), a.J == 1: the same
// operations as launch_accumulate, then out = RNE((sum) / N_p) per segment (AccSeg::out,
// AccSeg::div) written straight from the kernel; the running sum is not stored.  vec_ok
// bit s also requires the segment's output to be 16-byte aligned.  direct: the input is
// read in place by plain loads (as launch_accumulate_direct).
cudaError_t launch_accumulate_final(const AccArgs& a, int dtype_in, int dtype_out, bool direct,
                                    const LaunchShape& s, cudaStream_t stream);

// One client (a.J == 1) with the input read in place by plain loads, no bulk copies:
// for inputs in host memory the device can address (pinned memory read over the
// NVLink-C2C link), where the link sets the pace.  Same arguments and the same
// per-element arithmetic as launch_accumulate, so the sums are bit-identical.
cudaError_t launch_accumulate_direct(const AccArgs& a, int dtype_in, const LaunchShape& s,
                                     cudaStream_t stream);

// Final-mode reduce: out = RNE((sum so far +) J weighted inputs, / divisor) per segment.
// The caller fills everything but tile / ntiles / tile0.
cudaError_t launch_reduce_final(const RedArgs& a, int dtype_in, int dtype_out,
                                const LaunchShape& s, cudaStream_t stream);

// a.segs: device array of a.nseg FinSeg sorted by tile0, or nullptr with the table in
// a.seg (a.nseg <= kFinInlineSegs).
//   apply == false: out = RNE(sum / N)
//   apply == true:  out = RNE(fma(server_lr, sum / N, base))   (delta rounds)
// acc_lo: compensated mode (sum = acc + acc_lo), else nullptr.
// host_out: some outputs are host memory written in place over the host link; the grid
// then runs at full occupancy (more stores in flight for the link) instead of
// kFinCtasPerSm, the HBM-bound optimum.
cudaError_t launch_finalize(const FinArgs& a, int dtype_out, bool apply, float server_lr, bool host_out,
                            const LaunchShape& s, cudaStream_t stream);

}  // namespace fa
