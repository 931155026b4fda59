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
// All are HBM-bandwidth bound streaming passes (about 0.1 flop per byte): no tensor
// cores.  Layout: the fp32 running sum is padded per key to 32 elements, so each key
// starts 128-byte aligned.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace fa {

constexpr int kBlock = 256;           // threads per CTA
constexpr int kVec = 8;               // elements per vector (16 B of bf16, 2 x 16 B of fp32)
constexpr int kTile = 4096;           // elements per tile of the finalize kernel
constexpr int kBulkTile = 8192;       // elements per pipeline stage of the streaming kernel
constexpr int kDirectTile = kBlock * kVec;   // elements per tile of the direct-load accumulate
// Finalize CTAs per SM: with a tile's loads issued together, 4 CTAs (about 64 KB of loads
// in flight per SM) gave the best rate in a sweep of 2..8 on GB300; more in flight was slower.
constexpr int kFinCtasPerSm = 4;
constexpr int kMaxSegs = 48;          // segments per accumulate / reduce launch
constexpr int kMaxBatch = 16;         // resident clients per launch
constexpr int kReduceStageBytes = 73728;   // shared-memory budget per stage of the reduce kernel

struct AccSeg {
    const void* x;      // one-client launches: this segment's input chunk (segments of one
                        // launch may come from different chunks); J > 1 uses AccArgs::x
    uint64_t x_off;     // element offset into the input chunk(s)
    uint64_t acc_idx;   // element index into the running sum
    uint64_t len;       // elements (>= 1)
    uint32_t first;     // 1: the first client of the launch starts the sum here
    uint32_t tile0;     // first tile of this segment (set by launch_accumulate)
};

struct AccArgs {
    const void* x[kMaxBatch];   // J input chunk bases (device), dtype_in
    float w[kMaxBatch];         // (float) n_k per input
    float* acc;
    uint32_t J;                 // 1..16
    uint32_t nseg;
    uint32_t ntiles;            // set by launch_accumulate
    uint64_t vec_ok;            // bit s: segment s is 16-byte aligned for x and sum
    AccSeg seg[kMaxSegs];
};

struct RedSeg {
    uint64_t x_off;     // element offset into every input
    uint64_t acc_idx;   // element index into the running sum
    uint64_t len;       // elements (>= 1)
    void* out;          // final mode: destination of element 0 (dtype_out)
    float divisor;      // final mode: (float) N_p
    uint32_t read_sum;  // 1: earlier contributions are in the running sum
    uint32_t tile0;     // first tile (set by the launcher)
    uint32_t pad;
};

struct RedArgs {
    const void* x[kMaxBatch];   // J input bases (device), dtype_in
    float w[kMaxBatch];
    float* acc;
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
    float divisor;      // (float) N_p
    uint32_t tile0;     // first tile of this segment
};

struct LaunchShape {
    int sms = 0;
    int bulk_ctas_per_sm[2] = {};       // [dtype_in], streaming kernel
    int direct_ctas_per_sm[2] = {};     // [dtype_in], direct-load accumulate
    int reduce_ctas_per_sm[2][3] = {};  // [dtype_in][sum mode, final fp32 out, final bf16 out]
                                        // (same for every specialisation of J)
    int fin_ctas_per_sm[2][2] = {};     // [apply][dtype_out]
};

// Device-side error bits (file-scope word shared by every launch on a device).
constexpr unsigned int kErrWaitTimeout = 1u;   // a bounded mbarrier wait gave up

// Queue on `stream` a copy of the current device's error word into *host (pinned) followed
// by clearing it; the caller waits for the stream before reading *host.
cudaError_t take_device_error_async(unsigned int* host, cudaStream_t stream);

// Fills the occupancy table for the current device (and sets the kernels'
// shared-memory limits).
cudaError_t query_launch_shape(LaunchShape* s);

// dtype codes: 0 = fp32, 1 = bf16.  The caller fills x, w, acc, J (1..16), nseg, vec_ok
// and each segment's x (J = 1) / x_off / acc_idx / len / first; the launcher numbers the
// tiles for the kernel it picks (J = 1: streaming kernel, else the reduce kernel in sum
// mode).
// Returns cudaErrorInvalidValue if the arguments are out of range.
cudaError_t launch_accumulate(const AccArgs& a, int dtype_in, const LaunchShape& s,
                              cudaStream_t stream);

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

// segs: device array of nseg FinSeg sorted by tile0.
//   apply == false: out = RNE(sum / N)
//   apply == true:  out = RNE(fma(server_lr, sum / N, base))   (delta rounds)
// host_out: some outputs are host memory written in place over the host link; the grid
// then runs at full occupancy (more stores in flight for the link) instead of
// kFinCtasPerSm, the HBM-bound optimum.
cudaError_t launch_finalize(const FinSeg* segs, uint32_t nseg, uint32_t ntiles, int dtype_out,
                            const float* acc, bool apply, float server_lr, bool host_out,
                            const LaunchShape& s, cudaStream_t stream);

}  // namespace fa
