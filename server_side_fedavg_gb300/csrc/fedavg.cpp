// Runtime and C ABI of the aggregation library (declared in include/fedavg.h).
//
// One context = one round's state on one GPU:
//  - the fp32 running sum in device memory (padded layout, see ledger.hpp);
//  - the host ledger (weights, reporter masks, element counts, per-key totals);
//  - host chunks the device can address (pinned memory mapped at the same pointer;
//    pageable memory where the device walks the host page tables) are read in place
//    by the direct-load accumulate kernel over the host link, straight into the sum;
//  - a staging ring for the other host chunks (and all of them under FA_STAGE_HOST):
//    R device slots fed by cudaMemcpyAsync on a copy stream, overlapped with the
//    kernels on the caller's stream, plus R pinned host slots used only for pageable
//    sources.  This is the chunked, memory-bounded ingest that "Building Federated
//    Multimodal AI Workflows with NVIDIA FLARE" motivates ("Moving and aggregating
//    large model updates efficiently": the Tensor Downloader's chunk size trades
//    per-request overhead against per-chunk memory);
//  - an event chain: after every launch an event is recorded on the stream used and
//    the next launch (on any stream) waits for it, so contributions land in call
//    order and streams never race on the running sum.
// Every host wait polls with a deadline (opts.timeout_ms) and returns
// FA_ERR_TIMEOUT instead of blocking forever.
#include <fedavg.h>

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <chrono>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <memory>
#include <mutex>
#include <string>
#include <thread>
#include <vector>

#include "gather.cuh"
#include "kernels.cuh"
#include "ledger.hpp"

namespace {

constexpr uint64_t kDefaultSlotBytes = 64ull << 20;
constexpr uint32_t kDefaultSlots = 4;
constexpr uint32_t kDefaultTimeoutMs = 60000;

// kManaged: cudaMallocManaged memory, read in place with plain loads only (its pages may be
// on the host: plain loads take the migration faults; bulk copies are kept off it)
enum class Mem { kDevice, kManaged, kPinned, kPageable };

}  // namespace

struct fa_ctx {
    std::mutex mu;
    fa::Ledger ledger;
    int device = 0;
    int din = 0, dout = 0;        // 0 fp32, 1 bf16
    uint32_t s_in = 4, s_out = 4;
    uint32_t flags = 0;
    uint32_t timeout_ms = kDefaultTimeoutMs;
    uint32_t slots = kDefaultSlots;
    uint64_t slot_bytes = kDefaultSlotBytes;
    float* acc = nullptr;         // fp32 running sum (compensated mode: its hi part)
    float* acc_lo = nullptr;      // compensated mode (FA_COMPENSATED): the error part
    fa::LaunchShape shape;

    cudaEvent_t chain = nullptr;  // recorded after the last queued operation
    bool chain_valid = false;
    unsigned long long chain_stream_id = 0;   // stream the chain event was last recorded on
    cudaEvent_t user_ev = nullptr;
    cudaEvent_t read_ev = nullptr;   // end of an in-place read of a pageable chunk
    bool pageable_in_place = false;  // the device reads pageable memory through the host page tables

    cudaStream_t copy_stream = nullptr;
    std::vector<void*> dev_slot, host_slot;
    std::vector<cudaEvent_t> ev_copied, ev_free;
    std::vector<uint8_t> slot_used;
    uint32_t next_slot = 0;

    std::unique_ptr<fa::FinArgs> fin_args;   // a finalize launch's parameters (its table
                                             // inline up to kFinInlineSegs ranges)
    fa::FinSeg* fin_dev = nullptr;           // larger tables: uploaded from fin_host
    fa::FinSeg* fin_host = nullptr;
    size_t fin_cap = 0;           // entries of both (n_keys; more once final contributions split keys)
    cudaEvent_t fin_ev = nullptr;
    bool fin_pending = false;

    // fa_reduce_subsets: segment and source tables, pinned host copy and device copy
    uint8_t* gath_host = nullptr;
    uint8_t* gath_dev = nullptr;
    size_t gath_cap = 0;
    cudaEvent_t gath_ev = nullptr;
    bool gath_pending = false;
    // ... or, for a small round, its tables in the launch's parameters
    std::unique_ptr<fa::GathInline> gath_inline;
    uint32_t* gath_counter = nullptr;   // an inline subset reduce's two counter words (0 between
                                        // launches: each launch leaves them so)
    void* out_stage = nullptr;

    unsigned int* err_dev = nullptr;     // this context's device error word (kernels OR bits in)
    cudaStream_t err_stream = nullptr;   // private non-blocking stream for reading it
    cudaEvent_t err_ev = nullptr;
    unsigned int* err_host = nullptr;    // pinned copy of the device error word

    bool broken = false;          // a CUDA call failed after the ledger was updated
    bool reduced = false;         // this round was written by fa_reduce_resident
    fa_stats stats{};
    std::string err;
    std::vector<fa::Piece> pieces;
    std::vector<fa::FinItem> items;
};

namespace {

// An NVTX range over one library call (visible to Nsight tools, free otherwise).
class Range {
public:
    explicit Range(const char* name) { nvtxRangePushA(name); }
    ~Range() { nvtxRangePop(); }
};

// Switches to the context's device for the duration of a call.
class DeviceGuard {
public:
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev_) == cudaSuccess && prev_ != dev) {
            if (cudaSetDevice(dev) == cudaSuccess) restore_ = true;
        }
    }
    ~DeviceGuard() {
        if (restore_) cudaSetDevice(prev_);
    }

private:
    int prev_ = 0;
    bool restore_ = false;
};

// With FA_LOG set in the environment (to anything but "0"), every failure a call reports is
// also written to stderr.
void log_failure(fa_status s, const std::string& what) {
    static const bool on = [] {
        const char* v = std::getenv("FA_LOG");
        return v != nullptr && v[0] != '\0' && std::strcmp(v, "0") != 0;
    }();
    if (on) std::fprintf(stderr, "[fedavg] %s: %s\n", fa_strerror(s), what.c_str());
}

fa_status fail(fa_ctx* c, fa_status s, const std::string& what) {
    c->err = what;
    log_failure(s, what);
    return s;
}

fa_status cuda_fail(fa_ctx* c, cudaError_t e, const char* where) {
    c->err = std::string(where) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
    const fa_status s = e == cudaErrorMemoryAllocation ? FA_ERR_NOMEM : FA_ERR_CUDA;
    log_failure(s, c->err);
    return s;
}

#define FA_CUDA(ctx, call)                                   \
    do {                                                     \
        cudaError_t e_ = (call);                             \
        if (e_ != cudaSuccess) return cuda_fail(ctx, e_, #call); \
    } while (0)

// Poll an event until it completes or the deadline (timeout_ms) passes: yielding, then
// in 50 us sleeps -- or, with `spin`, yielding only (for short waits on the critical
// path, where a sleep's overshoot would leave the GPU idle).
fa_status wait_event(fa_ctx* c, cudaEvent_t ev, const char* what, bool spin = false) {
    auto t0 = std::chrono::steady_clock::now();
    uint32_t spins = 0;
    for (;;) {
        cudaError_t e = cudaEventQuery(ev);
        if (e == cudaSuccess) return FA_OK;
        if (e != cudaErrorNotReady) return cuda_fail(c, e, what);
        auto ms = std::chrono::duration_cast<std::chrono::milliseconds>(
                      std::chrono::steady_clock::now() - t0)
                      .count();
        if (ms > static_cast<long long>(c->timeout_ms)) {
            return fail(c, FA_ERR_TIMEOUT, std::string(what) + ": no completion within timeout_ms");
        }
        if (spin || ++spins < 64)
            std::this_thread::yield();
        else
            std::this_thread::sleep_for(std::chrono::microseconds(50));
    }
}

Mem classify(const void* p, int device, bool* other_device, bool* in_place = nullptr) {
    *other_device = false;
    if (in_place) *in_place = false;
    cudaPointerAttributes at;
    cudaError_t e = cudaPointerGetAttributes(&at, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return Mem::kPageable;
    }
    switch (at.type) {
        case cudaMemoryTypeDevice:
            *other_device = at.device != device;
            return Mem::kDevice;
        case cudaMemoryTypeManaged:
            return Mem::kManaged;
        case cudaMemoryTypeHost:
            // pinned memory the current device reads at the same address (unified
            // addressing): kernels may load it in place
            if (in_place) *in_place = at.devicePointer == p;
            return Mem::kPinned;
        default:
            return Mem::kPageable;
    }
}

// Whether `s` is capturing into a CUDA graph.  A captured call issues only work a graph
// replays as it ran -- kernels whose tables ride in their parameters, copies between fixed
// buffers -- and refuses (FA_ERR_STATE) what needs the host while the round runs: staged
// chunks, pageable memory, table uploads, allocations.  Captured work is ordered by the
// stream it is replayed on, not by the context's chain of calls.
bool capturing(cudaStream_t s) {
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    return cudaStreamIsCapturing(s, &st) == cudaSuccess && st != cudaStreamCaptureStatusNone;
}

// Make `s` wait for everything queued on the context so far.  Work on the same
// stream as the last record is already ordered after it (stream ids are unique
// for the life of the context, unlike handles), so the wait is only issued when
// the stream changes -- a cross-stream wait costs a full launch latency.
fa_status chain_in(fa_ctx* c, cudaStream_t s) {
    if (!c->chain_valid || capturing(s)) return FA_OK;
    unsigned long long id = 0;
    FA_CUDA(c, cudaStreamGetId(s, &id));
    if (id != c->chain_stream_id) FA_CUDA(c, cudaStreamWaitEvent(s, c->chain, 0));
    return FA_OK;
}

fa_status chain_out(fa_ctx* c, cudaStream_t s) {
    if (capturing(s)) {
        c->chain_valid = false;   // nothing of the capture has run: later calls need not wait
        return FA_OK;
    }
    FA_CUDA(c, cudaEventRecord(c->chain, s));
    FA_CUDA(c, cudaStreamGetId(s, &c->chain_stream_id));
    c->chain_valid = true;
    return FA_OK;
}

// Allocate the staging ring (device slots, events, copy stream) and, when a pageable
// source needs them, the pinned host slots.  All or nothing: after a failure nothing is
// kept, so a later call can try again.
fa_status ensure_ring(fa_ctx* c, bool need_host) {
    if (c->dev_slot.empty()) {
        std::vector<void*> dev(c->slots, nullptr);
        std::vector<cudaEvent_t> copied(c->slots, nullptr), freed(c->slots, nullptr);
        cudaStream_t cs = nullptr;
        cudaError_t e = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking);
        for (uint32_t i = 0; e == cudaSuccess && i < c->slots; ++i) {
            e = cudaMalloc(&dev[i], c->slot_bytes);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&copied[i], cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&freed[i], cudaEventDisableTiming);
        }
        if (e != cudaSuccess) {
            for (void* p : dev)
                if (p) cudaFree(p);
            for (auto ev : copied)
                if (ev) cudaEventDestroy(ev);
            for (auto ev : freed)
                if (ev) cudaEventDestroy(ev);
            if (cs) cudaStreamDestroy(cs);
            cudaGetLastError();
            return cuda_fail(c, e, "staging ring");
        }
        c->copy_stream = cs;
        c->dev_slot = dev;
        c->ev_copied = copied;
        c->ev_free = freed;
        c->host_slot.assign(c->slots, nullptr);
        c->slot_used.assign(c->slots, 0);
    }
    if (need_host && c->host_slot[0] == nullptr) {
        std::vector<void*> host(c->slots, nullptr);
        cudaError_t e = cudaSuccess;
        for (uint32_t i = 0; e == cudaSuccess && i < c->slots; ++i)
            e = cudaHostAlloc(&host[i], c->slot_bytes, cudaHostAllocDefault);
        if (e != cudaSuccess) {
            for (void* p : host)
                if (p) cudaFreeHost(p);
            cudaGetLastError();
            return cuda_fail(c, e, "pinned staging");
        }
        c->host_slot = host;
    }
    return FA_OK;
}

// Launch the accumulate kernel(s) for the pieces that fall in chunk elements
// [c0, c0 + n), reading inputs xs[0..J) whose element 0 is chunk element c0 -- or, for
// one client's several chunks (J = 1, fa_accumulate_keys), xs[i] is chunk i and each
// piece reads the chunk it was cut from.
// A final contribution (fa_accumulate_final) passes fin: each piece's N_p and the outputs
// (n_keys pointers, or one flat pointer with FA_FLAT_OUT); its launches then write the
// pieces' outputs instead of the sum.
struct FinalOut {
    const std::vector<double>* totals;
    void* const* outs;
};

fa_status launch_pieces(fa_ctx* c, const std::vector<fa::Piece>& pieces, uint64_t c0,
                        uint64_t n, const void* const* xs, const float* ws, uint32_t J,
                        cudaStream_t s, bool direct = false, const FinalOut* fin = nullptr) {
    // launches of up to 16 clients (one at a time for the direct kernel, which takes one);
    // after the first launch the sum is started everywhere
    uint32_t done = 0;
    while (done < J) {
        const uint32_t left = J - done;
        const uint32_t jb = direct ? 1u : (left < static_cast<uint32_t>(fa::kMaxBatch) ? left : fa::kMaxBatch);
        fa::AccArgs a;
        std::memset(&a, 0, sizeof a);
        for (uint32_t j = 0; j < jb; ++j) {
            a.x[j] = xs[done + j];
            a.w[j] = ws[done + j];
        }
        a.acc = c->acc;
        a.acc_lo = c->acc_lo;
        a.err = c->err_dev;
        a.debug = (c->flags & FA_TEST_WAIT_EXPIRES) ? fa::kDebugFirstWaitExpires : 0u;
        a.J = jb;
        auto flush = [&]() -> fa_status {
            if (a.nseg == 0) return FA_OK;
            FA_CUDA(c, fin ? fa::launch_accumulate_final(a, c->din, c->dout, direct, c->shape, s)
                           : direct ? fa::launch_accumulate_direct(a, c->din, c->shape, s)
                                    : fa::launch_accumulate(a, c->din, c->shape, s));
            c->stats.kernel_launches++;
            a.nseg = 0;
            a.vec_ok = 0;
            return FA_OK;
        };
        const bool flat = (c->flags & FA_FLAT_OUT) != 0;
        for (size_t pi = 0; pi < pieces.size(); ++pi) {
            const auto& p = pieces[pi];
            uint64_t b = std::max(p.chunk_off, c0);
            uint64_t e = std::min(p.chunk_off + p.len, c0 + n);
            if (b >= e) continue;
            if (fin && (*fin->totals)[pi] == 0.0) continue;   // N_p == 0: nothing to write
            if (a.nseg == static_cast<uint32_t>(fa::kMaxSegs)) {
                fa_status st = flush();
                if (st != FA_OK) return st;
            }
            fa::AccSeg& g = a.seg[a.nseg];
            // one client: each piece reads its own chunk (xs[p.chunk]); J > 1: xs[j]
            g.x = jb == 1 ? xs[done + p.chunk] : a.x[0];
            g.x_off = b - c0;
            g.acc_idx = p.acc_idx + (b - p.chunk_off);
            g.len = e - b;
            g.first = (p.first && done == 0) ? 1u : 0u;
            bool ok = (reinterpret_cast<uintptr_t>(c->acc + g.acc_idx) & 15u) == 0;
            if (fin) {
                // the output element of acc_idx: its key's output at the same offset in the key
                const uint64_t koff = g.acc_idx - c->ledger.acc_off(p.key);
                char* dst = static_cast<char*>(flat ? fin->outs[0] : fin->outs[p.key]);
                dst += (flat ? c->ledger.flat_off(p.key) + koff : koff) * c->s_out;
                g.out = dst;
                g.div = fa::make_divisor((*fin->totals)[pi]);
                ok = ok && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0;
            }
            for (uint32_t j = 0; j < jb && ok; ++j) {
                const void* base = jb == 1 ? g.x : a.x[j];
                uintptr_t xa = reinterpret_cast<uintptr_t>(base) + g.x_off * c->s_in;
                ok = (xa & 15u) == 0;
            }
            if (ok) a.vec_ok |= 1ull << a.nseg;
            a.nseg++;
        }
        fa_status st = flush();
        if (st != FA_OK) return st;
        done += jb;
    }
    return FA_OK;
}

// Pieces read in place -- from device memory (bulk or reduce kernel) or from host memory
// the device addresses (direct kernel, over the host link, one client per launch) --
// ordered after the context's earlier work.  ptrs/ws: J clients' chunks and weights, or
// for fa_accumulate_keys one client's several chunks (J = 1).  A pageable source is
// waited for before returning, so the caller may reuse it at once.
fa_status launch_in_place(fa_ctx* c, const void* const* ptrs, const float* ws, uint32_t J,
                          cudaStream_t s, bool host, bool pageable, const FinalOut* fin = nullptr) {
    fa_status r = chain_in(c, s);
    if (r == FA_OK) r = launch_pieces(c, c->pieces, 0, UINT64_MAX, ptrs, ws, J, s, host, fin);
    if (r == FA_OK && pageable) {
        cudaError_t ce = cudaEventRecord(c->read_ev, s);
        if (ce != cudaSuccess) r = cuda_fail(c, ce, "pageable read");
    }
    if (r == FA_OK) r = chain_out(c, s);
    if (r == FA_OK && pageable) r = wait_event(c, c->read_ev, "pageable chunk read", true);
    return r;
}

fa_status accumulate_impl(fa_ctx* c, uint32_t J, const uint32_t* ids, const double* weights,
                          int64_t key, uint64_t offset, const void* const* ptrs, uint64_t len,
                          cudaStream_t s, bool batch, void* const* final_outs = nullptr) {
    if (c->broken) return fail(c, FA_ERR_CUDA, "an earlier CUDA failure left this round inconsistent: call fa_reset");
    if (len > 0) {
        for (uint32_t j = 0; j < J; ++j)
            if (ptrs == nullptr || ptrs[j] == nullptr) return fail(c, FA_ERR_ARG, "chunk pointer is NULL");
    }
    // host chunks the device can address are read in place unless staging is asked for:
    // pinned memory mapped at the same pointer, and pageable memory where the device walks
    // the host page tables (then the call waits for the read, so the caller may reuse the
    // chunk on return as with staging)
    const bool stage = (c->flags & FA_STAGE_HOST) != 0;
    Mem kind = Mem::kDevice;
    bool all_device = true, all_in_place = true, any_pageable = false;
    uint32_t host_chunks = 0;
    if (len > 0) {
        for (uint32_t j = 0; j < J; ++j) {
            bool other = false, in_place = false;
            const Mem m = classify(ptrs[j], c->device, &other, &in_place);
            if (other) return fail(c, FA_ERR_ARG, "chunk is in another GPU's memory");
            all_device = all_device && m == Mem::kDevice;
            all_in_place = all_in_place &&
                           (m == Mem::kManaged ||
                            (!stage && ((m == Mem::kPinned && in_place) ||
                                        (m == Mem::kPageable && c->pageable_in_place))));
            any_pageable = any_pageable || m == Mem::kPageable;
            host_chunks += (m == Mem::kPinned || m == Mem::kPageable) ? 1u : 0u;
            kind = m;
        }
    }
    if (batch && len > 0 && !all_device && !all_in_place)
        return fail(c, FA_ERR_ARG,
                    "fa_accumulate_batch reads its chunks in place: all in this GPU's memory, or all "
                    "in managed memory or host memory the device addresses");
    const bool direct = !all_device && all_in_place;
    if (len > 0 && (any_pageable || (!all_device && !direct)) && capturing(s))
        return fail(c, FA_ERR_STATE,
                    "a captured call reads its chunks in place from this GPU's memory, managed memory or "
                    "pinned host memory (staged and pageable chunks need the host during the round)");
    if (final_outs && len > 0 && !all_device && !all_in_place)
        return fail(c, FA_ERR_ARG,
                    "fa_accumulate_final reads its chunk in place: this GPU's memory, managed memory, or "
                    "host memory the device addresses (not staged)");
    if (len > 0 && kind != Mem::kDevice && !direct) {
        // staging first: a failed allocation must not leave the round half-recorded
        fa_status rr = ensure_ring(c, kind == Mem::kPageable);
        if (rr != FA_OK) return rr;
    }
    std::string e;
    std::vector<double> totals;
    int32_t st = final_outs ? c->ledger.plan_accumulate_final(ids[0], weights[0], key, offset, len, &c->pieces,
                                                             &totals, &e)
                            : c->ledger.plan_accumulate(ids, weights, J, key, offset, len, &c->pieces, &e);
    if (st != fa::kOk) return fail(c, st, e);
    if (len == 0) return FA_OK;
    const FinalOut fo{&totals, final_outs};
    const FinalOut* fin = final_outs ? &fo : nullptr;

    std::vector<float> wv(J);
    for (uint32_t j = 0; j < J; ++j) wv[j] = static_cast<float>(weights[j]);
    const float* wp = wv.data();

    fa_status r = FA_OK;
    if (kind == Mem::kDevice) {
        r = chain_in(c, s);
        if (r == FA_OK) r = launch_pieces(c, c->pieces, 0, len, ptrs, wp, J, s, false, fin);
        if (r == FA_OK) r = chain_out(c, s);
    } else if (direct) {
        // host memory read by the kernel over the host link, ordered on `s` (a batch: one
        // direct launch per client, in batch order)
        r = launch_in_place(c, ptrs, wp, J, s, true, any_pageable, fin);
        if (r == FA_OK) c->stats.h2d_bytes += static_cast<uint64_t>(host_chunks) * len * c->s_in;
    } else {
        // host memory: through the staging ring, slot-sized pieces
        const uint64_t per = c->slot_bytes / c->s_in;
        const char* src0 = static_cast<const char*>(ptrs[0]);
        if (r == FA_OK && kind == Mem::kPinned) {
            // the copy must follow the caller's earlier work on `s`
            cudaError_t ce = cudaEventRecord(c->user_ev, s);
            if (ce == cudaSuccess) ce = cudaStreamWaitEvent(c->copy_stream, c->user_ev, 0);
            if (ce != cudaSuccess) r = cuda_fail(c, ce, "order copy after caller stream");
        }
        for (uint64_t c0 = 0; r == FA_OK && c0 < len; c0 += per) {
            const uint64_t n = std::min(per, len - c0);
            const uint32_t k = c->next_slot;
            c->next_slot = (k + 1) % c->slots;
            const void* src = src0 + c0 * c->s_in;
            if (kind == Mem::kPageable) {
                if (c->slot_used[k]) {
                    r = wait_event(c, c->ev_copied[k], "staging slot reuse");
                    if (r != FA_OK) break;
                }
                std::memcpy(c->host_slot[k], src, n * c->s_in);
                src = c->host_slot[k];
            }
            cudaError_t ce = cudaSuccess;
            if (c->slot_used[k]) ce = cudaStreamWaitEvent(c->copy_stream, c->ev_free[k], 0);
            if (ce == cudaSuccess)
                ce = cudaMemcpyAsync(c->dev_slot[k], src, n * c->s_in, cudaMemcpyHostToDevice,
                                     c->copy_stream);
            if (ce == cudaSuccess) ce = cudaEventRecord(c->ev_copied[k], c->copy_stream);
            if (ce == cudaSuccess) ce = cudaStreamWaitEvent(s, c->ev_copied[k], 0);
            if (ce != cudaSuccess) {
                r = cuda_fail(c, ce, "staging copy");
                break;
            }
            c->slot_used[k] = 1;
            c->stats.h2d_bytes += n * c->s_in;
            r = chain_in(c, s);
            const void* xs[1] = {c->dev_slot[k]};
            if (r == FA_OK) r = launch_pieces(c, c->pieces, c0, n, xs, wp, 1, s);
            if (r == FA_OK) r = chain_out(c, s);
            if (r == FA_OK) {
                ce = cudaEventRecord(c->ev_free[k], s);
                if (ce != cudaSuccess) r = cuda_fail(c, ce, "slot release");
            }
        }
    }
    if (r != FA_OK) {
        c->broken = true;
        return r;
    }
    c->stats.chunks++;
    c->stats.client_bytes += static_cast<uint64_t>(J) * len * c->s_in;
    return FA_OK;
}

void free_ctx(fa_ctx* c) {
    if (c->acc) cudaFree(c->acc);
    for (void* p : c->dev_slot)
        if (p) cudaFree(p);
    for (void* p : c->host_slot)
        if (p) cudaFreeHost(p);
    for (auto ev : c->ev_copied)
        if (ev) cudaEventDestroy(ev);
    for (auto ev : c->ev_free)
        if (ev) cudaEventDestroy(ev);
    if (c->copy_stream) cudaStreamDestroy(c->copy_stream);
    if (c->chain) cudaEventDestroy(c->chain);
    if (c->user_ev) cudaEventDestroy(c->user_ev);
    if (c->read_ev) cudaEventDestroy(c->read_ev);
    if (c->fin_ev) cudaEventDestroy(c->fin_ev);
    if (c->fin_dev) cudaFree(c->fin_dev);
    if (c->fin_host) cudaFreeHost(c->fin_host);
    if (c->gath_host) cudaFreeHost(c->gath_host);
    if (c->gath_dev) cudaFree(c->gath_dev);
    if (c->gath_ev) cudaEventDestroy(c->gath_ev);
    if (c->gath_counter) cudaFree(c->gath_counter);
    if (c->out_stage) cudaFree(c->out_stage);
    if (c->err_ev) cudaEventDestroy(c->err_ev);
    if (c->err_stream) cudaStreamDestroy(c->err_stream);
    if (c->err_host) cudaFreeHost(c->err_host);
    if (c->err_dev) cudaFree(c->err_dev);
    delete c;
}

fa_status sync_impl(fa_ctx* c) {
    if (c->chain_valid) {
        fa_status r = wait_event(c, c->chain, "fa_sync");
        if (r != FA_OK) return r;
    }
    for (size_t k = 0; k < c->ev_copied.size(); ++k) {
        if (!c->slot_used[k]) continue;
        fa_status r = wait_event(c, c->ev_copied[k], "fa_sync (copy)");
        if (r != FA_OK) return r;
    }
    // this context's device error word, read and cleared on a private stream and waited
    // for with the same bound (every kernel that could set it has completed by now)
    *c->err_host = 0;
    FA_CUDA(c, cudaMemcpyAsync(c->err_host, c->err_dev, sizeof(unsigned int), cudaMemcpyDeviceToHost,
                               c->err_stream));
    FA_CUDA(c, cudaMemsetAsync(c->err_dev, 0, sizeof(unsigned int), c->err_stream));
    FA_CUDA(c, cudaEventRecord(c->err_ev, c->err_stream));
    fa_status rw = wait_event(c, c->err_ev, "fa_sync (error word)");
    if (rw != FA_OK) return rw;
    const unsigned int code = *c->err_host;
    if (code != 0) {
        c->broken = true;
        return fail(c, FA_ERR_INTERNAL, "a device-side wait gave up (bounded mbarrier wait): results of this round are invalid");
    }
    return FA_OK;
}

}  // namespace

extern "C" {

const char* fa_strerror(fa_status s) {
    switch (s) {
        case FA_OK: return "ok";
        case FA_ERR_ARG: return "invalid argument";
        case FA_ERR_RANGE: return "offset or length out of range";
        case FA_ERR_DTYPE: return "unsupported dtype";
        case FA_ERR_WEIGHT: return "invalid or inconsistent client weight";
        case FA_ERR_INCOMPLETE: return "a client sent only part of a key";
        case FA_ERR_STATE: return "call not allowed in the current state";
        case FA_ERR_NOMEM: return "out of memory";
        case FA_ERR_CUDA: return "CUDA error";
        case FA_ERR_TIMEOUT: return "timed out waiting for the GPU";
        case FA_ERR_INTERNAL: return "internal error";
        default: return "unknown status";
    }
}

const char* fa_last_error(const fa_ctx* ctx) { return ctx ? ctx->err.c_str() : ""; }

fa_status fa_open(const fa_key* layout, uint32_t n_keys, fa_dtype dtype_in, fa_dtype dtype_out,
                  uint32_t max_clients, const fa_opts* opts, fa_ctx** out) {
    if (out == nullptr) return FA_ERR_ARG;
    *out = nullptr;
    if (layout == nullptr || n_keys == 0 || max_clients == 0) return FA_ERR_ARG;
    if ((dtype_in != FA_F32 && dtype_in != FA_BF16) || (dtype_out != FA_F32 && dtype_out != FA_BF16))
        return FA_ERR_DTYPE;
    fa_opts o{};
    if (opts) {
        if (opts->size < sizeof(uint32_t) * 2) return FA_ERR_ARG;
        std::memcpy(&o, opts, std::min<size_t>(opts->size, sizeof o));
    }
    fa_ctx* c = new (std::nothrow) fa_ctx;
    if (!c) return FA_ERR_NOMEM;
    c->din = dtype_in == FA_F32 ? 0 : 1;
    c->dout = dtype_out == FA_F32 ? 0 : 1;
    c->s_in = c->din == 0 ? 4 : 2;
    c->s_out = c->dout == 0 ? 4 : 2;
    c->flags = o.flags;
    if (o.timeout_ms) c->timeout_ms = o.timeout_ms;
    if (o.ring_slots) c->slots = o.ring_slots;
    if (o.slot_bytes) c->slot_bytes = (o.slot_bytes + 255) / 256 * 256;
    if (c->slots > 64) {
        delete c;
        return FA_ERR_ARG;
    }
    std::vector<uint64_t> numels(n_keys);
    for (uint32_t p = 0; p < n_keys; ++p) numels[p] = layout[p].numel;
    std::string e;
    if (c->ledger.init(numels.data(), n_keys, max_clients, &e) != fa::kOk) {
        delete c;
        return FA_ERR_ARG;
    }
    cudaError_t ce = cudaGetDevice(&c->device);
    if (ce == cudaSuccess) ce = fa::query_launch_shape(&c->shape);
    const bool comp = (c->flags & FA_COMPENSATED) != 0;
    if (ce == cudaSuccess)
        ce = cudaMalloc(&c->acc, c->ledger.padded_elems() * sizeof(float) * (comp ? 2 : 1));
    if (ce == cudaSuccess && comp) c->acc_lo = c->acc + c->ledger.padded_elems();
    if (ce == cudaSuccess) ce = cudaMalloc(&c->err_dev, 256);
    if (ce == cudaSuccess) ce = cudaMemset(c->err_dev, 0, 256);
    if (ce == cudaSuccess) ce = cudaEventCreateWithFlags(&c->chain, cudaEventDisableTiming);
    if (ce == cudaSuccess) ce = cudaEventCreateWithFlags(&c->user_ev, cudaEventDisableTiming);
    if (ce == cudaSuccess) ce = cudaEventCreateWithFlags(&c->read_ev, cudaEventDisableTiming);
    if (ce == cudaSuccess) {
        // pageable memory is read and written in place only where the device reaches it
        // through the host's own page tables (no migration of the caller's pages)
        int pma = 0, host_pt = 0;
        ce = cudaDeviceGetAttribute(&pma, cudaDevAttrPageableMemoryAccess, c->device);
        if (ce == cudaSuccess)
            ce = cudaDeviceGetAttribute(&host_pt, cudaDevAttrPageableMemoryAccessUsesHostPageTables, c->device);
        c->pageable_in_place = pma == 1 && host_pt == 1;
    }
    if (ce == cudaSuccess) ce = cudaEventCreateWithFlags(&c->fin_ev, cudaEventDisableTiming);
    if (ce == cudaSuccess) ce = cudaEventCreateWithFlags(&c->gath_ev, cudaEventDisableTiming);
    if (ce == cudaSuccess) ce = cudaMalloc(reinterpret_cast<void**>(&c->gath_counter), 2 * sizeof(uint32_t));
    if (ce == cudaSuccess) ce = cudaMemset(c->gath_counter, 0, 2 * sizeof(uint32_t));
    if (ce == cudaSuccess) c->fin_args.reset(new (std::nothrow) fa::FinArgs);
    if (ce == cudaSuccess && !c->fin_args) ce = cudaErrorMemoryAllocation;
    if (ce == cudaSuccess) ce = cudaMalloc(&c->fin_dev, sizeof(fa::FinSeg) * n_keys);
    if (ce == cudaSuccess) ce = cudaHostAlloc(&c->fin_host, sizeof(fa::FinSeg) * n_keys, cudaHostAllocDefault);
    if (ce == cudaSuccess) c->fin_cap = n_keys;
    if (ce == cudaSuccess) ce = cudaStreamCreateWithFlags(&c->err_stream, cudaStreamNonBlocking);
    if (ce == cudaSuccess) ce = cudaEventCreateWithFlags(&c->err_ev, cudaEventDisableTiming);
    if (ce == cudaSuccess)
        ce = cudaHostAlloc(reinterpret_cast<void**>(&c->err_host), sizeof(unsigned int), cudaHostAllocDefault);
    if (ce != cudaSuccess) {
        cudaGetLastError();
        free_ctx(c);
        return ce == cudaErrorMemoryAllocation ? FA_ERR_NOMEM : FA_ERR_CUDA;
    }
    *out = c;
    return FA_OK;
}

fa_status fa_accumulate(fa_ctx* ctx, uint32_t client_id, double weight_nk, int64_t key,
                        uint64_t offset_elems, const void* chunk_ptr, uint64_t len_elems,
                        void* stream) {
    Range range("fa_accumulate");
    if (!ctx) return FA_ERR_ARG;
    std::lock_guard<std::mutex> lk(ctx->mu);
    DeviceGuard dg(ctx->device);
    ctx->err.clear();
    const void* ptrs[1] = {chunk_ptr};
    return accumulate_impl(ctx, 1, &client_id, &weight_nk, key, offset_elems, ptrs, len_elems,
                           static_cast<cudaStream_t>(stream), false);
}

fa_status fa_accumulate_final(fa_ctx* ctx, uint32_t client_id, double weight_nk, int64_t key,
                              uint64_t offset_elems, const void* chunk_ptr, uint64_t len_elems,
                              void* const* out_ptrs, void* stream) {
    Range range("fa_accumulate_final");
    if (!ctx) return FA_ERR_ARG;
    std::lock_guard<std::mutex> lk(ctx->mu);
    DeviceGuard dg(ctx->device);
    fa_ctx* c = ctx;
    c->err.clear();
    if (out_ptrs == nullptr) return fail(c, FA_ERR_ARG, "out_ptrs is NULL");
    // the outputs this range writes: this GPU's memory, managed memory, or pinned host
    // memory the device addresses (written in place over the host link)
    const bool flat = (c->flags & FA_FLAT_OUT) != 0;
    uint64_t host_bytes = 0;
    if (len_elems > 0) {
        const uint32_t nk = c->ledger.n_keys();
        uint32_t p0 = 0, p1 = 0;   // keys [p0, p1] whose outputs are written
        if (key >= 0 && key < static_cast<int64_t>(nk)) {
            p0 = p1 = static_cast<uint32_t>(key);
        } else if (key == FA_KEY_FLAT && offset_elems < c->ledger.total_elems()) {
            uint32_t lo = 0, hi = nk;   // the last key starting at or before the offset
            while (hi - lo > 1) {
                const uint32_t mid = (lo + hi) / 2;
                if (c->ledger.flat_off(mid) <= offset_elems) lo = mid; else hi = mid;
            }
            p0 = p1 = lo;
            const uint64_t end = offset_elems + std::min(len_elems, c->ledger.total_elems() - offset_elems);
            while (p1 + 1 < nk && c->ledger.flat_off(p1 + 1) < end) ++p1;
        }   // else the range check below refuses the call
        for (uint32_t p = p0; p <= (flat ? p0 : p1); ++p) {
            void* dst = flat ? out_ptrs[0] : out_ptrs[p];
            bool other = false, in_place = false;
            const Mem m = dst ? classify(dst, c->device, &other, &in_place) : Mem::kPageable;
            if (dst == nullptr || other || !(m == Mem::kDevice || m == Mem::kManaged || (m == Mem::kPinned && in_place)))
                return fail(c, FA_ERR_ARG,
                            "fa_accumulate_final writes its outputs in place: this GPU's memory, managed "
                            "memory, or pinned host memory the device addresses");
            if (m == Mem::kPinned) host_bytes = len_elems * c->s_out;
        }
    }
    const void* ptrs[1] = {chunk_ptr};
    fa_status r = accumulate_impl(c, 1, &client_id, &weight_nk, key, offset_elems, ptrs, len_elems,
                                  static_cast<cudaStream_t>(stream), false, out_ptrs);
    if (r == FA_OK) c->stats.d2h_bytes += host_bytes;
    return r;
}

fa_status fa_accumulate_batch(fa_ctx* ctx, uint32_t n_clients, const uint32_t* client_ids,
                              const double* weights, int64_t key, uint64_t offset_elems,
                              const void* const* chunk_ptrs, uint64_t len_elems, void* stream) {
    Range range("fa_accumulate_batch");
    if (!ctx) return FA_ERR_ARG;
    std::lock_guard<std::mutex> lk(ctx->mu);
    DeviceGuard dg(ctx->device);
    ctx->err.clear();
    if (n_clients == 0 || client_ids == nullptr || weights == nullptr || chunk_ptrs == nullptr)
        return fail(ctx, FA_ERR_ARG, "empty batch");
    return accumulate_impl(ctx, n_clients, client_ids, weights, key, offset_elems, chunk_ptrs,
                           len_elems, static_cast<cudaStream_t>(stream), true);
}

fa_status fa_accumulate_keys(fa_ctx* ctx, uint32_t client_id, double weight_nk, uint32_t n_chunks,
                             const int64_t* keys, const uint64_t* offsets,
                             const void* const* chunk_ptrs, const uint64_t* lens, void* stream) {
    Range range("fa_accumulate_keys");
    if (!ctx) return FA_ERR_ARG;
    std::lock_guard<std::mutex> lk(ctx->mu);
    DeviceGuard dg(ctx->device);
    ctx->err.clear();
    fa_ctx* c = ctx;
    if (c->broken) return fail(c, FA_ERR_CUDA, "an earlier CUDA failure left this round inconsistent: call fa_reset");
    if (n_chunks > 0 && (keys == nullptr || offsets == nullptr || lens == nullptr || chunk_ptrs == nullptr))
        return fail(c, FA_ERR_ARG, "keys, offsets, chunk_ptrs or lens is NULL");
    // every chunk is read in place: all device memory, or all host memory the device
    // addresses
    bool any = false, all_device = true, all_host = true, pageable = false;
    uint64_t total = 0, host_total = 0;
    for (uint32_t i = 0; i < n_chunks; ++i) {
        if (lens[i] == 0) continue;
        if (chunk_ptrs[i] == nullptr) return fail(c, FA_ERR_ARG, "chunk pointer is NULL");
        bool other = false, in_place = false;
        const Mem m = classify(chunk_ptrs[i], c->device, &other, &in_place);
        if (other) return fail(c, FA_ERR_ARG, "chunk is in another GPU's memory");
        const bool host_ok = m == Mem::kManaged ||
                             ((c->flags & FA_STAGE_HOST) == 0 &&
                              ((m == Mem::kPinned && in_place) ||
                               (m == Mem::kPageable && c->pageable_in_place)));
        all_device = all_device && m == Mem::kDevice;
        all_host = all_host && host_ok;
        pageable = pageable || m == Mem::kPageable;
        any = true;
        total += lens[i];
        if (m == Mem::kPinned || m == Mem::kPageable) host_total += lens[i];
    }
    if (any && !all_device && !all_host)
        return fail(c, FA_ERR_ARG,
                    "fa_accumulate_keys reads its chunks in place: all in this GPU's memory, or all "
                    "in managed memory or host memory the device addresses; send others through "
                    "fa_accumulate");
    if (any && pageable && !all_device && capturing(static_cast<cudaStream_t>(stream)))
        return fail(c, FA_ERR_STATE, "a captured call reads no pageable chunk (its read needs the host)");
    std::string e;
    int32_t st = c->ledger.plan_accumulate_keys(client_id, weight_nk, n_chunks, keys, offsets, lens,
                                                &c->pieces, &e);
    if (st != fa::kOk) return fail(c, st, e);
    if (!any) return FA_OK;
    const float w = static_cast<float>(weight_nk);
    fa_status r = launch_in_place(c, chunk_ptrs, &w, 1, static_cast<cudaStream_t>(stream),
                                  !all_device, !all_device && pageable);
    if (r != FA_OK) {
        c->broken = true;
        return r;
    }
    for (uint32_t i = 0; i < n_chunks; ++i) c->stats.chunks += lens[i] > 0 ? 1 : 0;
    c->stats.client_bytes += total * c->s_in;
    c->stats.h2d_bytes += host_total * c->s_in;
    return FA_OK;
}

}  // extern "C"

namespace {

// A one-pass round (fa_reduce_subsets, or fa_reduce_resident with every client sending
// every key) with its tables in the launch's parameters, when they fit: no upload and no
// table reads from global memory.  The entries of the key of c->items[i] are
// [cnt[key], cnt[key + 1]) in the order they apply; entry e is client src_client[e] at
// element offset src_off[e] of that client's buffer.  Returns false (nothing done) if the
// round is too large for this form; otherwise launches, with *st the status.
bool launch_inline_round(fa_ctx* c, void* const* out_ptrs, uint32_t jmax, const std::vector<uint32_t>& cnt,
                         uint64_t n_entries, const uint32_t* src_client, const uint64_t* src_off,
                         uint32_t n_clients, const void* const* client_ptrs, const double* weights,
                         cudaStream_t s, fa_status* st) {
    const bool flat = (c->flags & FA_FLAT_OUT) != 0;
    const bool comp = c->acc_lo != nullptr;
    const uint32_t nseg = static_cast<uint32_t>(c->items.size());
    auto aligned = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
    uint32_t so = 0, bo = 0, wo = 0;
    // every key and client offset must fit 32 bits
    bool small = jmax <= static_cast<uint32_t>(fa::kMaxBatch) &&
                 fa::gather_inline_layout(nseg, static_cast<uint32_t>(std::min<uint64_t>(n_entries, 0xFFFFFFFFu)),
                                          n_clients, &so, &bo, &wo);
    for (uint32_t i = 0; small && i < nseg; ++i) small = c->items[i].numel <= 0xFFFFFFFFull;
    for (uint64_t e = 0; small && e < n_entries; ++e) small = src_off[e] <= 0xFFFFFFFFull;
    if (!small) return false;
    if (!c->gath_inline) c->gath_inline.reset(new fa::GathInline);
    fa::GathInline& gp = *c->gath_inline;
    gp.err = c->err_dev;
    gp.counter = c->gath_counter;
    gp.pad0 = 0;
    gp.nseg = nseg;
    gp.nsrc = static_cast<uint32_t>(n_entries);
    gp.nclient = n_clients;
    gp.jmax = jmax;
    gp.pad = 0;
    gp.src_off = so;
    gp.base_off = bo;
    gp.w_off = wo;
    auto* gs = reinterpret_cast<fa::GathSegP*>(gp.blob);
    auto* gr = reinterpret_cast<fa::GathSrcP*>(gp.blob + so);
    auto* gb = reinterpret_cast<const void**>(gp.blob + bo);
    auto* gw = reinterpret_cast<float*>(gp.blob + wo);
    uint64_t tiles = 0;
    for (uint32_t i = 0; i < nseg; ++i) {
        const fa::FinItem& it = c->items[i];
        fa::GathSegP& g = gs[i];
        char* dst = static_cast<char*>(flat ? out_ptrs[0] : out_ptrs[it.key]);
        g.out = flat ? dst + it.flat_off * c->s_out : dst;
        g.div = fa::make_divisor(it.total);
        g.len = static_cast<uint32_t>(it.numel);
        g.tile0 = static_cast<uint32_t>(tiles);
        g.src0 = static_cast<uint16_t>(cnt[it.key]);
        g.J = static_cast<uint8_t>(cnt[it.key + 1] - cnt[it.key]);
        bool ok = aligned(g.out);
        for (uint32_t q = 0; q < g.J && ok; ++q) {
            const uint64_t e = g.src0 + q;
            ok = aligned(static_cast<const char*>(client_ptrs[src_client[e]]) + src_off[e] * c->s_in);
        }
        g.vec_ok = ok ? 1u : 0u;
        const uint64_t tile = fa::gather_tile(g.J, c->din);
        tiles += (it.numel + tile - 1) / tile;
    }
    if (tiles > 0xFFFFFFFFull) {
        c->broken = true;
        *st = fail(c, FA_ERR_RANGE, "layout too large for one pass");
        return true;
    }
    gp.ntiles = static_cast<uint32_t>(tiles);
    for (uint64_t e = 0; e < n_entries; ++e)
        gr[e] = fa::GathSrcP{static_cast<uint32_t>(src_off[e]), src_client[e]};
    for (uint32_t j = 0; j < n_clients; ++j) {
        gb[j] = client_ptrs[j];
        gw[j] = static_cast<float>(weights[j]);
    }
    gp.grid = fa::gather_grid(gp.ntiles, c->din, c->dout, comp, c->shape);
    gp.unit_tiles = fa::gather_unit_tiles(gp.ntiles, gp.grid);
    cudaError_t ce = fa::launch_gather_inline(gp, c->din, c->dout, comp, c->shape, s);
    if (ce != cudaSuccess) {
        c->broken = true;
        *st = cuda_fail(c, ce, "one-pass round launch");
        return true;
    }
    if (gp.ntiles > 0) c->stats.kernel_launches++;
    *st = FA_OK;
    return true;
}

// Shared driver of fa_finalize and fa_finalize_apply (base_ptrs != NULL).
fa_status finalize_impl(fa_ctx* c, const void* const* base_ptrs, void* const* out_ptrs,
                        double server_lr, void* stream) {
    const bool apply = base_ptrs != nullptr;
    if (c->reduced)
        return fail(c, FA_ERR_STATE, "this round was reduced by fa_reduce_resident: its outputs are already written");
    if (c->broken) return fail(c, FA_ERR_CUDA, "an earlier CUDA failure left this round inconsistent: call fa_reset");
    if (out_ptrs == nullptr) return fail(c, FA_ERR_ARG, "out_ptrs is NULL");
    if (apply && c->ledger.has_final())
        return fail(c, FA_ERR_STATE,
                    "fa_finalize_apply: fa_accumulate_final wrote plain means this round; a delta round "
                    "sends its last client through fa_accumulate");
    const bool flat = (c->flags & FA_FLAT_OUT) != 0;
    std::string e;
    {
        int32_t st = c->ledger.plan_finalize(&c->items, &e);
        if (st != fa::kOk) return fail(c, st, e);
    }
    std::vector<Mem> kind(c->items.size());
    bool any_host = false;
    uint64_t written_in_place = 0;   // bytes the kernel stores straight into pinned host memory
    // a flat output (and base) is one buffer: classify it once, not once per key
    bool flat_done = false, flat_other = false, flat_in_place = false, flat_base_ok = false;
    Mem flat_kind = Mem::kDevice;
    for (size_t i = 0; i < c->items.size(); ++i) {
        const auto& it = c->items[i];
        void* dst = flat ? out_ptrs[0] : out_ptrs[it.key];
        if (dst == nullptr) return fail(c, FA_ERR_ARG, "output pointer is NULL for a key to be written");
        bool other = false, in_place = false;
        if (flat && flat_done) {
            kind[i] = flat_kind;
            other = flat_other;
            in_place = flat_in_place;
        } else {
            kind[i] = classify(dst, c->device, &other, &in_place);
        }
        if (other) return fail(c, FA_ERR_ARG, "output is in another GPU's memory");
        if (apply) {
            const void* b = flat ? base_ptrs[0] : base_ptrs[it.key];
            bool bo = false;
            const bool base_ok = flat && flat_done
                                     ? flat_base_ok
                                     : b != nullptr && classify(b, c->device, &bo) == Mem::kDevice && !bo;
            if (flat && !flat_done) flat_base_ok = base_ok;
            if (!base_ok)
                return fail(c, FA_ERR_ARG, "fa_finalize_apply: base values must be in this GPU's memory");
            if (kind[i] != Mem::kDevice)
                return fail(c, FA_ERR_ARG, "fa_finalize_apply: outputs must be in this GPU's memory");
        }
        if (flat && !flat_done) {
            flat_kind = kind[i];
            flat_other = other;
            flat_in_place = in_place;
            flat_done = true;
        }
        // pinned outputs the device addresses at the same pointer are written by the
        // finalize kernel itself, over the host link, unless staging is asked for.
        // Pageable outputs stay staged: an output buffer is often freshly allocated, and
        // the device's first touch of each of its pages is a fault serviced by the host
        // (a 7B aggregate took seconds in place against ~80 ms through the copy engine)
        if (kind[i] == Mem::kPinned && in_place && (c->flags & FA_STAGE_HOST) == 0) {
            kind[i] = Mem::kDevice;
            written_in_place += it.numel * c->s_out;
        }
        if (kind[i] == Mem::kManaged) kind[i] = Mem::kDevice;   // plain stores, no staging
        any_host = any_host || kind[i] != Mem::kDevice;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (capturing(s)) {
        bool pageable_out = false;
        for (size_t i = 0; i < c->items.size(); ++i) pageable_out = pageable_out || kind[i] == Mem::kPageable;
        if (c->items.size() > fa::kFinInlineSegs || pageable_out || (any_host && c->out_stage == nullptr))
            return fail(c, FA_ERR_STATE,
                        "a captured finalize writes at most 600 ranges, into this GPU's memory or pinned "
                        "host memory (a staged output needs its device buffer from an earlier finalize)");
    }
    if (any_host && c->out_stage == nullptr)
        FA_CUDA(c, cudaMalloc(&c->out_stage, c->ledger.total_elems() * c->s_out));
    // the table rides in the launch's parameters when it fits, else it is uploaded
    const bool inline_tab = c->items.size() <= fa::kFinInlineSegs;
    if (!inline_tab && c->fin_pending) {
        fa_status r = wait_event(c, c->fin_ev, "finalize table reuse");
        if (r != FA_OK) return r;
        c->fin_pending = false;
    }
    if (!inline_tab && c->items.size() > c->fin_cap) {
        // final contributions split some keys into several ranges to write
        const size_t cap = c->items.size() * 2;
        fa::FinSeg* dev = nullptr;
        fa::FinSeg* host = nullptr;
        cudaError_t ce = cudaMalloc(&dev, sizeof(fa::FinSeg) * cap);
        if (ce == cudaSuccess) ce = cudaHostAlloc(&host, sizeof(fa::FinSeg) * cap, cudaHostAllocDefault);
        if (ce != cudaSuccess) {
            if (dev) cudaFree(dev);
            cudaGetLastError();
            return fail(c, ce == cudaErrorMemoryAllocation ? FA_ERR_NOMEM : FA_ERR_CUDA, "finalize table");
        }
        cudaFree(c->fin_dev);
        cudaFreeHost(c->fin_host);
        c->fin_dev = dev;
        c->fin_host = host;
        c->fin_cap = cap;
    }
    uint32_t ntiles = 0;
    for (size_t i = 0; i < c->items.size(); ++i) {
        const auto& it = c->items[i];
        char* dst = static_cast<char*>(flat ? out_ptrs[0] : out_ptrs[it.key]);
        dst += (flat ? it.flat_off : it.koff) * c->s_out;
        if (kind[i] != Mem::kDevice)
            dst = static_cast<char*>(c->out_stage) + it.flat_off * c->s_out;
        fa::FinSeg& g = inline_tab ? c->fin_args->seg[i] : c->fin_host[i];
        g.acc_idx = it.acc_idx;
        g.len = it.numel;
        g.out = dst;
        g.base = nullptr;
        if (apply) {
            const char* b = static_cast<const char*>(flat ? base_ptrs[0] : base_ptrs[it.key]);
            g.base = b + (flat ? it.flat_off : it.koff) * c->s_out;
        }
        g.div = fa::make_divisor(it.total);
        g.tile0 = ntiles;
        uint64_t t = (it.numel + fa::kTile - 1) / fa::kTile;
        if (t > 0xFFFFFFFFull - ntiles) return fail(c, FA_ERR_RANGE, "layout too large for one finalize");
        ntiles += static_cast<uint32_t>(t);
    }
    // the round is closed from here on
    c->ledger.close();
    const uint32_t nseg = static_cast<uint32_t>(c->items.size());
    fa_status r = chain_in(c, s);
    if (r != FA_OK) return r;
    if (nseg > 0) {
        fa::FinArgs& fa_args = *c->fin_args;
        fa_args.segs = inline_tab ? nullptr : c->fin_dev;
        fa_args.acc = c->acc;
        fa_args.acc_lo = c->acc_lo;
        fa_args.nseg = nseg;
        fa_args.ntiles = ntiles;
        if (!inline_tab) {
            FA_CUDA(c, cudaMemcpyAsync(c->fin_dev, c->fin_host, sizeof(fa::FinSeg) * nseg,
                                       cudaMemcpyHostToDevice, s));
            FA_CUDA(c, cudaEventRecord(c->fin_ev, s));
            c->fin_pending = true;
        }
        FA_CUDA(c, fa::launch_finalize(fa_args, c->dout, apply, static_cast<float>(server_lr),
                                       written_in_place > 0, c->shape, s));
        c->stats.kernel_launches++;
        c->stats.d2h_bytes += written_in_place;
        // host outputs: copy the staged keys back, merging neighbours in the flat layout
        for (size_t i = 0; i < c->items.size();) {
            if (kind[i] == Mem::kDevice) {
                ++i;
                continue;
            }
            const auto& it = c->items[i];
            if (flat) {
                size_t j = i + 1;
                uint64_t end = it.flat_off + it.numel;
                while (j < c->items.size() && kind[j] != Mem::kDevice && c->items[j].flat_off == end) {
                    end += c->items[j].numel;
                    ++j;
                }
                char* dst = static_cast<char*>(out_ptrs[0]) + it.flat_off * c->s_out;
                const char* src = static_cast<const char*>(c->out_stage) + it.flat_off * c->s_out;
                uint64_t bytes = (end - it.flat_off) * c->s_out;
                FA_CUDA(c, cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToHost, s));
                c->stats.d2h_bytes += bytes;
                i = j;
            } else {
                const char* src = static_cast<const char*>(c->out_stage) + it.flat_off * c->s_out;
                uint64_t bytes = it.numel * c->s_out;
                FA_CUDA(c, cudaMemcpyAsync(static_cast<char*>(out_ptrs[it.key]) + it.koff * c->s_out, src,
                                           bytes, cudaMemcpyDeviceToHost, s));
                c->stats.d2h_bytes += bytes;
                ++i;
            }
        }
    }
    return chain_out(c, s);
}

}  // namespace

extern "C" {

fa_status fa_finalize(fa_ctx* ctx, void* const* out_ptrs, void* stream) {
    Range range("fa_finalize");
    if (!ctx) return FA_ERR_ARG;
    std::lock_guard<std::mutex> lk(ctx->mu);
    DeviceGuard dg(ctx->device);
    ctx->err.clear();
    return finalize_impl(ctx, nullptr, out_ptrs, 1.0, stream);
}

fa_status fa_finalize_apply(fa_ctx* ctx, const void* const* base_ptrs, void* const* out_ptrs,
                            double server_lr, void* stream) {
    Range range("fa_finalize_apply");
    if (!ctx) return FA_ERR_ARG;
    std::lock_guard<std::mutex> lk(ctx->mu);
    DeviceGuard dg(ctx->device);
    ctx->err.clear();
    if (base_ptrs == nullptr) return fail(ctx, FA_ERR_ARG, "base_ptrs is NULL");
    if (!std::isfinite(server_lr)) return fail(ctx, FA_ERR_ARG, "server_lr must be finite");
    return finalize_impl(ctx, base_ptrs, out_ptrs, server_lr, stream);
}

fa_status fa_reduce_resident(fa_ctx* ctx, uint32_t n_clients, const uint32_t* client_ids,
                             const double* weights, const void* const* flat_ptrs,
                             void* const* out_ptrs, void* stream) {
    Range range("fa_reduce_resident");
    if (!ctx) return FA_ERR_ARG;
    std::lock_guard<std::mutex> lk(ctx->mu);
    DeviceGuard dg(ctx->device);
    fa_ctx* c = ctx;
    c->err.clear();
    if (c->broken) return fail(c, FA_ERR_CUDA, "an earlier CUDA failure left this round inconsistent: call fa_reset");
    if (n_clients == 0 || client_ids == nullptr || weights == nullptr || flat_ptrs == nullptr ||
        out_ptrs == nullptr)
        return fail(c, FA_ERR_ARG, "empty client list or NULL argument");
    if (c->ledger.closed() || c->ledger.has_contributions())
        return fail(c, FA_ERR_STATE, "fa_reduce_resident needs a round with no contributions yet (fa_reset)");
    for (uint32_t j = 0; j < n_clients; ++j) {
        bool other = false;
        if (flat_ptrs[j] == nullptr || classify(flat_ptrs[j], c->device, &other) != Mem::kDevice || other)
            return fail(c, FA_ERR_ARG, "every client update must be in this GPU's memory");
    }
    const bool flat = (c->flags & FA_FLAT_OUT) != 0;
    const uint32_t nk = c->ledger.n_keys();
    double total = 0.0;
    for (uint32_t j = 0; j < n_clients; ++j) total += std::isfinite(weights[j]) ? weights[j] : 0.0;
    if (total > 0.0) {
        for (uint32_t p = 0; p < (flat ? 1u : nk); ++p) {
            bool other = false;
            if (out_ptrs[p] == nullptr || classify(out_ptrs[p], c->device, &other) != Mem::kDevice || other)
                return fail(c, FA_ERR_ARG, "fa_reduce_resident: outputs must be in this GPU's memory");
        }
    }
    // bookkeeping: every client sends every key (validates ids and weights first)
    std::string e;
    int32_t st = c->ledger.plan_accumulate(client_ids, weights, n_clients, -1, 0,
                                           c->ledger.total_elems(), &c->pieces, &e);
    if (st != fa::kOk) return fail(c, st, e);
    st = c->ledger.plan_finalize(&c->items, &e);
    if (st != fa::kOk) return fail(c, FA_ERR_INTERNAL, e);
    c->ledger.close();
    c->reduced = true;
    c->stats.chunks++;
    c->stats.client_bytes += static_cast<uint64_t>(n_clients) * c->ledger.total_elems() * c->s_in;
    if (c->items.empty()) return FA_OK;   // no weight anywhere: nothing is written

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    fa_status r = chain_in(c, s);
    if (r != FA_OK) return r;
    if (n_clients <= static_cast<uint32_t>(fa::kMaxBatch) && c->items.size() > static_cast<size_t>(fa::kMaxSegs)) {
        // more keys than one J-client reduce launch takes: if the layout is small enough, the
        // round as a one-pass round of every key from every client, its tables in the launch's
        // parameters -- one launch instead of one per 48 keys (the same operations in the same
        // order)
        const uint32_t nk = c->ledger.n_keys();
        std::vector<uint32_t> cnt(nk + 1);
        for (uint32_t p = 0; p <= nk; ++p) cnt[p] = p * n_clients;
        const uint64_t n_entries = static_cast<uint64_t>(nk) * n_clients;
        std::vector<uint32_t> src_client(n_entries);
        std::vector<uint64_t> src_off(n_entries);
        for (uint32_t p = 0; p < nk; ++p)
            for (uint32_t j = 0; j < n_clients; ++j) {
                src_client[cnt[p] + j] = j;
                src_off[cnt[p] + j] = c->ledger.flat_off(p);
            }
        fa_status st = FA_OK;
        if (launch_inline_round(c, out_ptrs, n_clients, cnt, n_entries, src_client.data(), src_off.data(),
                                n_clients, flat_ptrs, weights, s, &st))
            return st == FA_OK ? chain_out(c, s) : st;
    }
    const uint32_t K = n_clients;
    const uint32_t last = K - (K - 1) / fa::kMaxBatch * fa::kMaxBatch;   // 1..16 clients in the last pass
    const uint32_t head = K - last;                                       // earlier passes write the sum
    std::vector<float> w(K);
    for (uint32_t j = 0; j < K; ++j) w[j] = static_cast<float>(weights[j]);
    auto aligned = [&](const void* p, uint64_t off_bytes) {
        return ((reinterpret_cast<uintptr_t>(p) + off_bytes) & 15u) == 0;
    };
    for (uint32_t g = 0; g < head; g += fa::kMaxBatch) {
        fa::AccArgs a;
        std::memset(&a, 0, sizeof a);
        a.J = fa::kMaxBatch;
        for (uint32_t j = 0; j < a.J; ++j) {
            a.x[j] = flat_ptrs[g + j];
            a.w[j] = w[g + j];
        }
        a.acc = c->acc;
        a.acc_lo = c->acc_lo;
        a.err = c->err_dev;
        for (uint32_t p = 0; p < nk;) {
            a.nseg = 0;
            a.vec_ok = 0;
            for (; p < nk && a.nseg < static_cast<uint32_t>(fa::kMaxSegs); ++p) {
                fa::AccSeg& sg = a.seg[a.nseg];
                sg.x = a.x[0];
                sg.x_off = c->ledger.flat_off(p);
                sg.acc_idx = c->ledger.acc_off(p);
                sg.len = c->ledger.numel(p);
                sg.first = g == 0 ? 1u : 0u;
                bool ok = true;
                for (uint32_t j = 0; j < a.J; ++j) ok = ok && aligned(a.x[j], sg.x_off * c->s_in);
                if (ok) a.vec_ok |= 1ull << a.nseg;
                a.nseg++;
            }
            FA_CUDA(c, fa::launch_accumulate(a, c->din, c->shape, s));
            c->stats.kernel_launches++;
        }
    }
    fa::RedArgs ra;
    std::memset(&ra, 0, sizeof ra);
    ra.J = last;
    for (uint32_t j = 0; j < last; ++j) {
        ra.x[j] = flat_ptrs[head + j];
        ra.w[j] = w[head + j];
    }
    ra.acc = c->acc;
    ra.acc_lo = c->acc_lo;
    ra.err = c->err_dev;
    for (size_t i = 0; i < c->items.size();) {
        ra.nseg = 0;
        ra.vec_ok = 0;
        for (; i < c->items.size() && ra.nseg < static_cast<uint32_t>(fa::kMaxSegs); ++i) {
            const fa::FinItem& it = c->items[i];
            fa::RedSeg& sg = ra.seg[ra.nseg];
            sg.x_off = it.flat_off;
            sg.acc_idx = it.acc_idx;
            sg.len = it.numel;
            char* dst = static_cast<char*>(flat ? out_ptrs[0] : out_ptrs[it.key]);
            if (flat) dst += it.flat_off * c->s_out;
            sg.out = dst;
            sg.div = fa::make_divisor(it.total);
            sg.read_sum = head > 0 ? 1u : 0u;
            bool ok = aligned(dst, 0);
            for (uint32_t j = 0; j < last; ++j) ok = ok && aligned(ra.x[j], sg.x_off * c->s_in);
            if (ok) ra.vec_ok |= 1ull << ra.nseg;
            ra.nseg++;
        }
        FA_CUDA(c, fa::launch_reduce_final(ra, c->din, c->dout, c->shape, s));
        c->stats.kernel_launches++;
    }
    return chain_out(c, s);
}

fa_status fa_reduce_subsets(fa_ctx* ctx, uint32_t n_clients, const uint32_t* client_ids,
                            const double* weights, const void* const* client_ptrs,
                            const uint32_t* n_keys, const int64_t* keys, void* const* out_ptrs,
                            void* stream) {
    Range range("fa_reduce_subsets");
    if (!ctx) return FA_ERR_ARG;
    std::lock_guard<std::mutex> lk(ctx->mu);
    DeviceGuard dg(ctx->device);
    fa_ctx* c = ctx;
    c->err.clear();
    if (c->broken) return fail(c, FA_ERR_CUDA, "an earlier CUDA failure left this round inconsistent: call fa_reset");
    if (n_clients == 0 || client_ids == nullptr || weights == nullptr || client_ptrs == nullptr ||
        n_keys == nullptr || out_ptrs == nullptr)
        return fail(c, FA_ERR_ARG, "empty client list or NULL argument");
    if (c->ledger.closed() || c->ledger.has_contributions())
        return fail(c, FA_ERR_STATE, "fa_reduce_subsets needs a round with no contributions yet (fa_reset)");
    const uint32_t nk = c->ledger.n_keys();
    {
        std::vector<uint8_t> seen(c->ledger.max_clients(), 0);
        for (uint32_t j = 0; j < n_clients; ++j) {
            if (client_ids[j] >= c->ledger.max_clients())
                return fail(c, FA_ERR_ARG, "client id >= max_clients");
            if (seen[client_ids[j]]++) return fail(c, FA_ERR_ARG, "a client id appears twice");
        }
    }
    uint64_t n_entries = 0;
    for (uint32_t j = 0; j < n_clients; ++j) n_entries += n_keys[j];
    if (n_entries > 0 && keys == nullptr) return fail(c, FA_ERR_ARG, "keys is NULL");
    for (uint64_t e = 0; e < n_entries; ++e)
        if (keys[e] < 0 || keys[e] >= static_cast<int64_t>(nk))
            return fail(c, FA_ERR_ARG, "fa_reduce_subsets takes whole keys: every entry names a key id");
    // every client buffer is read with bulk copies: this GPU's memory (cudaMalloc'd)
    for (uint32_t j = 0; j < n_clients; ++j) {
        if (n_keys[j] == 0) continue;
        bool other = false;
        if (client_ptrs[j] == nullptr || classify(client_ptrs[j], c->device, &other) != Mem::kDevice || other)
            return fail(c, FA_ERR_ARG, "every client buffer must be in this GPU's memory (cudaMalloc'd)");
    }
    // bookkeeping, client by client in call order; the round was empty, so a failure is
    // undone by resetting it (all or nothing)
    std::string e;
    uint64_t o = 0;
    for (uint32_t j = 0; j < n_clients; ++j) {
        const uint32_t n = n_keys[j];
        int32_t st = c->ledger.record_whole_keys(client_ids[j], weights[j], n, keys + o, &e);
        if (st != fa::kOk) {
            c->ledger.reset();
            return fail(c, st, "client index " + std::to_string(j) + ": " + e);
        }
        o += n;
    }
    int32_t st = c->ledger.plan_finalize(&c->items, &e);
    if (st != fa::kOk) {
        c->ledger.reset();
        return fail(c, FA_ERR_INTERNAL, e);
    }
    // outputs: this GPU's memory
    const bool flat = (c->flags & FA_FLAT_OUT) != 0;
    if (!c->items.empty()) {
        for (size_t i = 0; i < (flat ? 1 : c->items.size()); ++i) {
            void* dst = flat ? out_ptrs[0] : out_ptrs[c->items[i].key];
            bool other = false;
            if (dst == nullptr || classify(dst, c->device, &other) != Mem::kDevice || other) {
                c->ledger.reset();
                return fail(c, FA_ERR_ARG, "fa_reduce_subsets: outputs must be in this GPU's memory");
            }
        }
    }
    // reporters per key in call order (compressed rows), and each entry's element offset
    // within its client's packed buffer
    std::vector<uint32_t> cnt(nk + 1, 0);
    for (uint64_t i = 0; i < n_entries; ++i) cnt[static_cast<uint32_t>(keys[i]) + 1]++;
    uint32_t jmax = 0;
    for (uint32_t p = 0; p < nk; ++p) {
        jmax = std::max(jmax, cnt[p + 1]);
        cnt[p + 1] += cnt[p];
    }
    std::vector<uint32_t> fill(cnt.begin(), cnt.end() - 1);
    std::vector<const void*> src_x(n_entries);
    std::vector<float> src_w(n_entries);
    std::vector<uint32_t> src_client(n_entries);
    std::vector<uint64_t> src_off(n_entries);
    o = 0;
    for (uint32_t j = 0; j < n_clients; ++j) {
        uint64_t off = 0;
        for (uint32_t i = 0; i < n_keys[j]; ++i, ++o) {
            const uint32_t p = static_cast<uint32_t>(keys[o]);
            const uint32_t slot = fill[p]++;
            src_x[slot] = static_cast<const char*>(client_ptrs[j]) + off * c->s_in;
            src_w[slot] = static_cast<float>(weights[j]);
            src_client[slot] = j;
            src_off[slot] = off;
            off += c->ledger.numel(p);
        }
    }
    c->ledger.close();
    c->reduced = true;
    c->stats.chunks += n_entries;
    for (uint64_t i = 0; i < n_entries; ++i)
        c->stats.client_bytes += c->ledger.numel(static_cast<uint32_t>(keys[i])) * c->s_in;
    if (c->items.empty()) return FA_OK;   // nothing sent with weight: nothing is written

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    fa_status r = chain_in(c, s);
    if (r != FA_OK) return r;
    if (jmax > static_cast<uint32_t>(fa::kMaxBatch)) {
        // more reporters on a key than one pass takes: each client's keys through the
        // streaming kernel (in call order), then the finalize kernel -- the same bits
        c->reduced = false;
        o = 0;
        std::vector<fa::Piece> pieces;
        std::vector<const void*> ptrs;
        std::vector<uint8_t> started(nk, 0);
        for (uint32_t j = 0; j < n_clients; ++j) {
            pieces.clear();
            ptrs.clear();
            uint64_t off = 0;
            for (uint32_t i = 0; i < n_keys[j]; ++i, ++o) {
                const uint32_t p = static_cast<uint32_t>(keys[o]);
                ptrs.push_back(static_cast<const char*>(client_ptrs[j]) + off * c->s_in);
                pieces.push_back({p, i, 0, c->ledger.acc_off(p), c->ledger.numel(p), started[p] == 0});
                started[p] = 1;
                off += c->ledger.numel(p);
            }
            if (pieces.empty()) continue;
            const float w = static_cast<float>(weights[j]);
            r = launch_pieces(c, pieces, 0, UINT64_MAX, ptrs.data(), &w, 1, s);
            if (r != FA_OK) {
                c->broken = true;
                return r;
            }
        }
        r = chain_out(c, s);
        if (r == FA_OK) r = finalize_impl(c, nullptr, out_ptrs, 1.0, stream);
        c->reduced = true;
        if (r != FA_OK) c->broken = true;
        return r;
    }
    const uint32_t nseg = static_cast<uint32_t>(c->items.size());
    const bool comp = c->acc_lo != nullptr;
    {
        fa_status st = FA_OK;
        if (launch_inline_round(c, out_ptrs, jmax, cnt, n_entries, src_client.data(), src_off.data(),
                                n_clients, client_ptrs, weights, s, &st))
            return st == FA_OK ? chain_out(c, s) : st;
    }
    if (capturing(s)) {
        c->broken = true;   // the round is recorded but cannot be captured: fa_reset
        return fail(c, FA_ERR_STATE,
                    "a captured fa_reduce_subsets carries its tables in the launch's parameters: this round "
                    "is too large for that (call fa_reset)");
    }
    // segment table (one entry per key to write) and source table in device memory
    const size_t seg_bytes = (sizeof(fa::GathSeg) * nseg + 15) / 16 * 16;
    const size_t src_bytes = (sizeof(fa::GathSrc) * n_entries + 15) / 16 * 16;
    // + the largest chunk table and the counter word
    const size_t need = seg_bytes + src_bytes +
                        2 * sizeof(uint32_t) * (static_cast<size_t>(fa::kMaxGatherChunks) + 1) + 16;
    if (c->gath_pending) {
        r = wait_event(c, c->gath_ev, "subset table reuse");
        if (r != FA_OK) return r;
        c->gath_pending = false;
    }
    if (need > c->gath_cap) {
        if (c->gath_host) cudaFreeHost(c->gath_host);
        if (c->gath_dev) cudaFree(c->gath_dev);
        c->gath_host = nullptr;
        c->gath_dev = nullptr;
        c->gath_cap = 0;
        const size_t cap = std::max<size_t>(need, 64 << 10);
        FA_CUDA(c, cudaHostAlloc(reinterpret_cast<void**>(&c->gath_host), cap, cudaHostAllocDefault));
        FA_CUDA(c, cudaMalloc(reinterpret_cast<void**>(&c->gath_dev), cap));
        c->gath_cap = cap;
    }
    auto* segs = reinterpret_cast<fa::GathSeg*>(c->gath_host);
    auto* srcs = reinterpret_cast<fa::GathSrc*>(c->gath_host + seg_bytes);
    for (uint64_t i = 0; i < n_entries; ++i) srcs[i] = fa::GathSrc{src_x[i], src_w[i], 0u};
    for (uint32_t i = 0; i < nseg; ++i) {
        const fa::FinItem& it = c->items[i];
        char* dst = static_cast<char*>(flat ? out_ptrs[0] : out_ptrs[it.key]);
        if (flat) dst += it.flat_off * c->s_out;
        fa::GathSeg& g = segs[i];
        g.len = it.numel;
        g.out = dst;
        g.div = fa::make_divisor(it.total);
        g.src0 = cnt[it.key];
        g.J = cnt[it.key + 1] - cnt[it.key];
        g.tile0 = 0;
        bool ok = (reinterpret_cast<uintptr_t>(dst) & 15u) == 0;
        for (uint32_t q = 0; q < g.J && ok; ++q) ok = (reinterpret_cast<uintptr_t>(srcs[g.src0 + q].x) & 15u) == 0;
        g.vec_ok = ok ? 1u : 0u;
    }
    fa::GathArgs ga;
    ga.segs = reinterpret_cast<const fa::GathSeg*>(c->gath_dev);
    ga.src = reinterpret_cast<const fa::GathSrc*>(c->gath_dev + seg_bytes);
    ga.cta = reinterpret_cast<const uint32_t*>(c->gath_dev + seg_bytes + src_bytes);
    ga.err = c->err_dev;
    ga.nseg = nseg;
    ga.jmax = jmax;
    if (!fa::plan_gather_tiles(segs, nseg, c->din, &ga.ntiles)) {
        c->broken = true;
        return fail(c, FA_ERR_RANGE, "layout too large for one subset reduce");
    }
    ga.grid = fa::gather_grid(ga.ntiles, c->din, c->dout, comp, c->shape);
    ga.nchunk = fa::gather_chunks(ga.ntiles, ga.grid);
    auto* cta = reinterpret_cast<uint32_t*>(c->gath_host + seg_bytes + src_bytes);
    fa::plan_gather_ctas(segs, nseg, ga.ntiles, c->din, c->dout, ga.nchunk, cta);
    // the chunk counter starts at 0: the word right after the chunk table, uploaded with
    // the tables in one copy
    const size_t counter_off = seg_bytes + src_bytes + 2 * sizeof(uint32_t) * (ga.nchunk + 1);
    std::memset(c->gath_host + counter_off, 0, sizeof(uint32_t));
    ga.counter = reinterpret_cast<uint32_t*>(c->gath_dev + counter_off);
    const size_t used = counter_off + sizeof(uint32_t);
    FA_CUDA(c, cudaMemcpyAsync(c->gath_dev, c->gath_host, used, cudaMemcpyHostToDevice, s));
    FA_CUDA(c, cudaEventRecord(c->gath_ev, s));
    c->gath_pending = true;
    cudaError_t ce = fa::launch_gather_final(ga, c->din, c->dout, comp, c->shape, s);
    if (ce != cudaSuccess) {
        c->broken = true;
        return cuda_fail(c, ce, "subset reduce launch");
    }
    c->stats.kernel_launches++;
    return chain_out(c, s);
}

fa_status fa_reset(fa_ctx* ctx) {
    Range range("fa_reset");
    if (!ctx) return FA_ERR_ARG;
    std::lock_guard<std::mutex> lk(ctx->mu);
    DeviceGuard dg(ctx->device);
    ctx->err.clear();
    // a device-side wait that gave up (FA_ERR_INTERNAL) invalidates the round being
    // discarded, not the context: the word is cleared, the reset goes ahead and the
    // status is still returned
    fa_status r = sync_impl(ctx);
    if (r != FA_OK && r != FA_ERR_INTERNAL) return r;
    ctx->ledger.reset();
    ctx->broken = false;
    ctx->reduced = false;
    ctx->flags &= ~FA_TEST_WAIT_EXPIRES;   // the test aid covers the first round only
    return r;
}

fa_status fa_close(fa_ctx* ctx) {
    if (!ctx) return FA_OK;
    DeviceGuard dg(ctx->device);
    fa_status r;
    {
        // wait for callers still inside the context, then for its GPU work
        std::lock_guard<std::mutex> lk(ctx->mu);
        r = sync_impl(ctx);
    }
    // the mutex is released before the context (and the mutex) is freed
    free_ctx(ctx);
    return r;
}

fa_status fa_key_total(const fa_ctx* ctx, uint32_t key, double* sum_nk, uint32_t* n_clients) {
    if (!ctx) return FA_ERR_ARG;
    fa_ctx* c = const_cast<fa_ctx*>(ctx);
    std::lock_guard<std::mutex> lk(c->mu);
    return c->ledger.key_total(key, sum_nk, n_clients) == fa::kOk ? FA_OK : FA_ERR_ARG;
}

fa_status fa_sync(fa_ctx* ctx) {
    Range range("fa_sync");
    if (!ctx) return FA_ERR_ARG;
    std::lock_guard<std::mutex> lk(ctx->mu);
    DeviceGuard dg(ctx->device);
    ctx->err.clear();
    return sync_impl(ctx);
}

fa_status fa_get_stats(const fa_ctx* ctx, fa_stats* out) {
    if (!ctx || !out) return FA_ERR_ARG;
    fa_ctx* c = const_cast<fa_ctx*>(ctx);
    std::lock_guard<std::mutex> lk(c->mu);
    *out = c->stats;
    return FA_OK;
}

}  // extern "C"
