/*
 * fedavg.h -- server-side FedAvg aggregation on one GPU (C ABI).
 *
 * Computes, for every key p (one tensor of a model state dict),
 *
 *     global[p][i] = sum_{k in S_p} n_k * w_k[p][i]  /  N_p,     N_p = sum_{k in S_p} n_k
 *
 * where S_p is the set of clients that sent key p in this round and n_k is
 * client k's weight (its sample count).  Client updates arrive as chunks,
 * in any order, from host or device memory; a fp32 running sum lives in
 * device memory, so memory does not grow with the number of clients.
 *
 * Passages the operations follow:
 *  [Clara]  "Federated learning implemented by NVIDIA Clara" (epnc.co.kr):
 *           opening section -- the server aggregates the clients' models as a
 *           simple average or weighted by each client's contribution, and
 *           clients share only part of the weights; "Server-side workflow" --
 *           after all updates arrive the server runs a weighted aggregation,
 *           updates the global model and starts the next round.
 *  [FLARE]  "Building Federated Multimodal AI Workflows with NVIDIA FLARE":
 *           "Coordinating training across clients" -- the client update
 *           contract fixes which components each client may update and how
 *           component-level updates are combined; "Moving and aggregating
 *           large model updates efficiently" -- the two memory pressures
 *           (one update in flight; many updates held during aggregation), the
 *           Tensor Downloader's tunable chunk size, and aggregation offloaded
 *           so server memory does not grow with the client count;
 *           "Federating small adapters on a frozen VLM with FedUMM" -- only
 *           adapter updates are aggregated.
 *  [Part]   "Technical Summary: Adaptive Data Partitioning for Energy-
 *           Efficient Federated and Distributed Learning in Heterogeneous
 *           Systems", section 2, "The adaptive controller", Measurement --
 *           each participant reports its sample count n_i for the round.
 *  [NVFP4]  "Accelerating LLM training with NVFP4 on NVIDIA Blackwell",
 *           list of ingredients, stochastic-rounding item -- weights are
 *           rounded to nearest even; "Applying NVFP4 in Transformer layers"
 *           -- low-precision results fold into fp32 master weights.
 *
 * Conventions for every call:
 *  - No call aborts, traps or waits without bound.  Errors come back as a
 *    negative fa_status; fa_last_error() gives a one-line detail.
 *  - Calls on one context are serialised by a mutex inside the context.
 *  - Device work is issued on the caller's `stream` (a cudaStream_t passed as
 *    void*, NULL = the legacy default stream).  Work on one context is
 *    chained across streams with events, so contributions apply in call
 *    order and two streams never race on the running sum.
 *  - Sizes and offsets are in ELEMENTS of the input dtype.
 *  - CUDA graphs: a round whose calls are issued on a stream that is capturing
 *    (cudaStreamBeginCapture) is recorded into the graph and replays as it ran:
 *    the same kernels on the same buffers with the same weights, over whatever
 *    the client buffers hold at replay.  Captured calls issue only kernels whose
 *    tables ride in their own parameters (a finalize of at most 600 ranges, a
 *    one-pass round whose tables fit a launch) and copies between fixed
 *    buffers; a call that needs the host while the round runs -- a staged or
 *    pageable chunk, a pageable output, a staged output before the context's
 *    first finalize, a one-pass round too large for its parameters (that round
 *    is then to be reset) -- returns FA_ERR_STATE and issues nothing, so the
 *    capture goes on.  Call fa_reset
 *    (which waits for the context's work) before the capture, not inside it;
 *    the context's host bookkeeping is that of the captured round, so the
 *    context serves the graph: replays are ordered by the stream they are
 *    launched on, and fa_reset comes before any further direct call.
 */
#ifndef FEDAVG_H
#define FEDAVG_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t fa_status;

#define FA_OK              0
#define FA_ERR_ARG        -1   /* null/invalid argument, unknown key, client id >= max_clients */
#define FA_ERR_RANGE      -2   /* offset+len past the key (or the flat layout), or more elements
                                  than numel sent by one client for one key */
#define FA_ERR_DTYPE      -3   /* unsupported dtype combination */
#define FA_ERR_WEIGHT     -4   /* weight not finite, < 0, > 2^24, or unlike this client's earlier chunks */
#define FA_ERR_INCOMPLETE -5   /* finalize: some client sent only part of a key */
#define FA_ERR_STATE      -6   /* accumulate after finalize (call fa_reset first) */
#define FA_ERR_NOMEM      -7   /* device or pinned host allocation failed */
#define FA_ERR_CUDA       -8   /* a CUDA runtime call failed (detail in fa_last_error) */
#define FA_ERR_TIMEOUT    -9   /* a bounded host wait ran out (opts.timeout_ms) */
#define FA_ERR_INTERNAL  -10   /* broken invariant inside the library */

typedef enum { FA_F32 = 0, FA_BF16 = 1 } fa_dtype;

/* One entry of the layout: key id = index in the layout array.  `name` is
 * informational (may be NULL); `numel` >= 1. */
typedef struct {
    const char* name;
    uint64_t numel;
} fa_key;

typedef struct fa_ctx fa_ctx;   /* opaque; owned by the library */

/* Pass as `key` to address the flat layout: the keys concatenated in layout
 * order without padding.  A flat chunk may span several keys. */
#define FA_KEY_FLAT (-1)

/* fa_opts.flags */
#define FA_FLAT_OUT   1u   /* fa_finalize takes ONE output pointer to the flat layout */
#define FA_STAGE_HOST 2u   /* host chunks go through the staging ring, and pinned host
                              outputs through a device buffer and a copy (copy engine),
                              even where the device could address them in place */
#define FA_COMPENSATED 4u  /* compensated running sum: a pair (hi, lo) of fp32 arrays updated
                              by the Dot2 scheme (Ogita, Rump & Oishi, "Accurate sum and dot
                              product", SIAM J. Sci. Comput. 26(6), 2005: an error-free
                              product by fma, Knuth's error-free TwoSum, errors summed into
                              lo), as accurate as a sum held in about twice fp32's precision,
                              so that the aggregate stays within one output ulp of the exact
                              weighted mean even where the sum nearly cancels.  [NVFP4]:
                              low-precision updates fold into fp32 master values; this keeps
                              that fold exact to the output's rounding.  Costs twice the sum's
                              device memory and 8 more bytes of HBM traffic per later
                              client-element when streaming (18 instead of 10 for bf16);
                              resident and batched reduces keep the pair in registers.  Every
                              path (streamed, batched, resident, in place from host memory)
                              gives the same bits in this mode, as in the default one. */
#define FA_TEST_WAIT_EXPIRES 0x80000000u
                           /* test aid, never for production: in the streaming accumulate
                              kernel each CTA's first data wait gives up at once, as if its
                              bound ran out, so that a test can check how a device-side
                              timeout is reported (fa_sync returns FA_ERR_INTERNAL and the
                              round's results are invalid) without hanging or faulting the
                              GPU.  The CTA still waits (bounded) for its loads in flight.
                              Applies until the context's first fa_reset, so the round after
                              it runs normally. */

typedef struct {
    uint32_t size;        /* sizeof(fa_opts): lets the struct grow */
    uint32_t ring_slots;  /* device staging slots for host chunks that are staged, not read
                             in place (0 = default 4) */
    uint64_t slot_bytes;  /* bytes per staging slot (0 = default 64 MiB; rounded up to 256 B) --
                             the chunk-size knob of [FLARE]'s Tensor Downloader, here a
                             trade of pinned/device staging memory against per-copy overhead */
    uint32_t timeout_ms;  /* bound on every host-side wait (0 = default 60000) */
    uint32_t flags;       /* FA_FLAT_OUT | FA_STAGE_HOST | FA_COMPENSATED */
} fa_opts;

typedef struct {
    uint64_t kernel_launches;   /* kernels this context has launched since fa_open */
    uint64_t client_bytes;      /* bytes of client updates accumulated */
    uint64_t h2d_bytes;         /* bytes of client updates brought from host memory (staging
                                   copies and in-place reads) */
    uint64_t d2h_bytes;         /* bytes of aggregate fa_finalize sent to host memory (copies
                                   and in-place stores) */
    uint64_t chunks;            /* accepted chunks: one per fa_accumulate / fa_accumulate_batch
                                   call, n_chunks per fa_accumulate_keys call */
} fa_stats;

/* Create an aggregation context on the current CUDA device.
 *   layout[0..n_keys)  the state dict's keys (copied; caller keeps ownership)
 *   dtype_in           element type of client updates (FA_F32 or FA_BF16)
 *   dtype_out          element type of the aggregate (FA_F32 or FA_BF16); rounding to
 *                      nearest even per [NVFP4]
 *   max_clients        client ids are 0..max_clients-1 (>= 1)
 *   opts               NULL for defaults
 * Allocates the fp32 running sum (sum of numel rounded up to 32 per key, x 4 bytes)
 * in device memory, the staging ring lazily on the first host chunk that is staged.
 * Errors: FA_ERR_ARG, FA_ERR_DTYPE, FA_ERR_NOMEM, FA_ERR_CUDA.  *out is NULL on error. */
fa_status fa_open(const fa_key* layout, uint32_t n_keys, fa_dtype dtype_in, fa_dtype dtype_out,
                  uint32_t max_clients, const fa_opts* opts, fa_ctx** out);

/* Add one chunk of client `client_id`'s update, weighted by `weight_nk`
 * ([Part]: the client's sample count; [Clara]: weighted aggregation).
 *   key            a key id, or FA_KEY_FLAT
 *   offset_elems   first element of the chunk within the key (or the flat layout)
 *   chunk_ptr      len_elems contiguous values of dtype_in, in device memory, managed
 *                  memory, or host memory (pinned or pageable; detected per call).
 *                  Managed memory (cudaMallocManaged) is read in place with plain loads,
 *                  since its pages may be on the host; stream-ordered like device memory.
 *   stream         cudaStream_t (as void*) ordering the read of chunk_ptr
 * The first chunk of a client in a round fixes its weight: later chunks must pass the
 * same value (else FA_ERR_WEIGHT).  weight_nk must be finite, >= 0 and <= 2^24.  The
 * device multiplies by (float)weight_nk: exact for integers in that range (sample counts,
 * the intended use); another value is rounded to fp32 first (a relative change of at
 * most 2^-24).  The per-key total N_p is summed in fp64 from the weights as given and
 * divided as a pair of floats, so totals above 2^24 keep their precision.
 * A client that sends a key must send all of it before fa_finalize (chunks of one
 * client and key must not overlap; the library counts elements).
 * Ownership: device and pinned-host chunks are read in order on `stream`: the caller
 * must not overwrite them until the work this call queued on `stream` has completed.
 * Pageable-host chunks have been consumed when the call returns: the caller may reuse
 * them at once.
 * Host chunks the device can address are read in place by the accumulate kernel over
 * the host link, with no staging copy -- the server receives a client's update straight
 * into its running sum: pinned memory mapped at the same pointer (unified addressing),
 * and pageable memory where the device reads through the host's page tables
 * (cudaDevAttrPageableMemoryAccessUsesHostPageTables; the call then waits, bounded by
 * timeout_ms, for the read to finish).  Other pageable chunks are copied into pinned
 * staging; FA_STAGE_HOST sends every host chunk through the staging ring.  All paths
 * give the same bits.  If a pageable in-place read times out (FA_ERR_TIMEOUT) it may
 * still be in flight: keep the chunk until the work queued on `stream` has completed.
 * len_elems == 0 is a no-op.  Argument, range, weight and state errors change nothing.
 * A CUDA failure or timeout after the chunk was accepted (FA_ERR_CUDA, FA_ERR_TIMEOUT,
 * FA_ERR_NOMEM) leaves the round inconsistent: every later call returns FA_ERR_CUDA
 * until fa_reset.
 * Errors: FA_ERR_ARG, FA_ERR_RANGE, FA_ERR_WEIGHT, FA_ERR_STATE, FA_ERR_CUDA,
 * FA_ERR_TIMEOUT, FA_ERR_NOMEM. */
fa_status fa_accumulate(fa_ctx* ctx, uint32_t client_id, double weight_nk, int64_t key,
                        uint64_t offset_elems, const void* chunk_ptr, uint64_t len_elems,
                        void* stream);

/* K-resident form of fa_accumulate: n_clients updates of the SAME element range,
 * reduced in one pass over the running sum when they are in device memory.  Equivalent
 * to calling fa_accumulate for client_ids[0], client_ids[1], ... in that order,
 * and bit-identical to it.  Client ids within one call must be distinct.
 * [FLARE]: the second memory pressure -- many client updates held at once --
 * turned into one read of each update and one write of the sum.
 * The chunks are read in place: all in this GPU's memory, or all in managed memory or
 * host memory the device addresses (as for fa_accumulate; then one plain-load launch per
 * client, in order -- the host link bounds that case anyway -- and a pageable batch is
 * waited for).
 * Errors: as fa_accumulate; FA_ERR_ARG for other memory, a mix, or host chunks under
 * FA_STAGE_HOST. */
fa_status fa_accumulate_batch(fa_ctx* ctx, uint32_t n_clients, const uint32_t* client_ids,
                              const double* weights, int64_t key, uint64_t offset_elems,
                              const void* const* chunk_ptrs, uint64_t len_elems, void* stream);

/* Several chunks of ONE client in one call: chunk i covers elements
 * [offsets[i], offsets[i] + lens[i]) of key keys[i] (FA_KEY_FLAT: of the flat layout)
 * and is read from chunk_ptrs[i].  Equivalent to n_chunks calls of fa_accumulate with
 * the same client, weight and stream, in index order, and bit-identical to them; the
 * library packs the chunks into launches of up to 48 key segments, so a client that
 * sends many small tensors -- an adapter subset, [FLARE]'s FedUMM LoRA modules --
 * costs a few launches instead of one per tensor.  Validated as a whole: on an
 * argument, range, weight or state error nothing is recorded.
 *   keys, offsets, lens, chunk_ptrs   n_chunks entries each (caller-owned, read during
 *                  the call); chunks of one key must not overlap, as for fa_accumulate
 * The chunks are read in place: all in this GPU's memory, or all in managed memory or
 * host memory the device addresses (as for fa_accumulate: pinned memory mapped at the same
 * pointer, or pageable memory where the device walks the host page tables, in which case
 * the call waits for the reads).  Other memory, a mix, or host chunks under FA_STAGE_HOST give
 * FA_ERR_ARG: send those through fa_accumulate.  Ownership and stream ordering as for
 * fa_accumulate; n_chunks == 0 or all lens zero is a no-op.
 * Errors: FA_ERR_ARG, FA_ERR_RANGE, FA_ERR_WEIGHT, FA_ERR_STATE, FA_ERR_CUDA,
 * FA_ERR_TIMEOUT. */
fa_status fa_accumulate_keys(fa_ctx* ctx, uint32_t client_id, double weight_nk, uint32_t n_chunks,
                             const int64_t* keys, const uint64_t* offsets,
                             const void* const* chunk_ptrs, const uint64_t* lens, void* stream);

/* The LAST contribution to a range, fused with the finalize of that range ([Clara]
 * "Server-side workflow": once the last update of the round is in, the aggregate
 * replaces the global model; here it is written while that update is read).  As
 * fa_accumulate for this chunk, then for every element i of the range, key p,
 *     out[p][i] = round_to_dtype_out( (sum[p][i] + n_k * x[i]) / N_p )
 * with the same operations, in the same order, as fa_accumulate followed by fa_finalize
 * (bit-identical), written straight from the kernel: the running sum of the range is
 * not stored, so the last client costs s_in + 4 + s_out bytes per element instead of
 * s_in + 8 plus the finalize's 4 + s_out.
 *   key, offset_elems, chunk_ptr, len_elems, stream   as fa_accumulate; the chunk is read
 *                  in place: this GPU's memory, managed memory, or host memory the device
 *                  addresses (FA_ERR_ARG for a staged chunk: use fa_accumulate there)
 *   out_ptrs       as fa_finalize (n_keys pointers, or one flat pointer with
 *                  FA_FLAT_OUT); the range's outputs must be in this GPU's memory, managed
 *                  memory, or pinned host memory the device addresses (written in place)
 * N_p is the key's total over its senders so far, this client included.  Every OTHER
 * client that sent a key of the range must already have sent all of it
 * (FA_ERR_INCOMPLETE).  From this call on the key takes no new sender, and the range
 * takes no further contribution (FA_ERR_STATE); fa_finalize later writes the rest of the
 * layout and leaves this range as written.  A key none of whose senders has weight
 * (N_p == 0) is not written.  The outputs hold plain means, so a round with a final
 * contribution ends in fa_finalize, not fa_finalize_apply (FA_ERR_STATE there): a delta
 * round sends its last client through fa_accumulate.  Ownership and errors otherwise as
 * fa_accumulate.
 * Errors: FA_ERR_ARG, FA_ERR_RANGE, FA_ERR_WEIGHT, FA_ERR_INCOMPLETE, FA_ERR_STATE,
 * FA_ERR_CUDA, FA_ERR_TIMEOUT. */
fa_status fa_accumulate_final(fa_ctx* ctx, uint32_t client_id, double weight_nk, int64_t key,
                              uint64_t offset_elems, const void* chunk_ptr, uint64_t len_elems,
                              void* const* out_ptrs, void* stream);

/* Write the aggregate: for every key with N_p > 0,
 *     out[p][i] = round_to_dtype_out( sum[p][i] / N_p )      (RNE)
 * where the quotient is one IEEE fp32 division when N_p is exact in fp32 (every integer
 * total up to 2^24); otherwise N_p = hi + lo as two floats and the quotient sum / hi is
 * corrected by its exact remainder (fma) less the lo part.  With FA_COMPENSATED, sum is
 * the pair hi + lo and the quotient is corrected the same way.
 * Keys no client sent (or whose reporters all have weight 0) are NOT written, so the
 * caller's previous global values survive (the frozen-backbone / adapter case of [FLARE]).
 *   out_ptrs  n_keys pointers (one per key, numel elements of dtype_out each), or, with
 *             FA_FLAT_OUT, one pointer to the flat layout.  Device or host memory;
 *             pinned host memory the device addresses at the same pointer is written
 *             in place by the kernel (no device staging), other host memory through a
 *             device buffer and a copy on `stream`.
 * Returns FA_ERR_INCOMPLETE, writing nothing, if a client sent part of a key.
 * Non-destructive: calling it again gives the same result.  After it, fa_accumulate
 * returns FA_ERR_STATE until fa_reset.  Output is complete once the work queued on
 * `stream` has completed (host outputs included: their stores or copies are on `stream`).
 * Errors: FA_ERR_ARG, FA_ERR_INCOMPLETE, FA_ERR_CUDA, FA_ERR_NOMEM, FA_ERR_TIMEOUT. */
fa_status fa_finalize(fa_ctx* ctx, void* const* out_ptrs, void* stream);

/* Finalize a round of DELTA updates into the global model ([Clara] "Server-side workflow":
 * after aggregating, the server updates the existing global model as a whole):
 *     out[p][i] = round_to_dtype_out( base[p][i] + server_lr * sum[p][i] / N_p )
 * computed as q = sum / (float)N_p (IEEE division), fma((float)server_lr, q, base) (one
 * rounding), then the RNE cast.  server_lr = 1 is plain FedAvg on deltas; the pages fix no
 * other value.  base_ptrs / out_ptrs: n_keys pointers each (or one flat pointer with
 * FA_FLAT_OUT), dtype_out values in this GPU's memory (cudaMalloc'd: managed memory is
 * refused); out may equal base (in place).
 * Keys with N_p == 0 are not written (out keeps its contents; in place, the model is
 * unchanged).  Otherwise as fa_finalize (closes the round, non-destructive, may repeat).
 * Errors: as fa_finalize; FA_ERR_ARG for host memory or a non-finite server_lr;
 * FA_ERR_STATE, changing nothing, after an fa_accumulate_final this round (the ranges it
 * wrote hold plain means). */
fa_status fa_finalize_apply(fa_ctx* ctx, const void* const* base_ptrs, void* const* out_ptrs,
                            double server_lr, void* stream);

/* A whole round in one pass when every client's FULL update is resident in device
 * memory ([FLARE] "Moving and aggregating large model updates efficiently": the second
 * memory pressure is holding many clients' updates during aggregation -- once they are
 * all in HBM, the weighted mean is one read of each update and one write of the output,
 * K*s_in + s_out bytes per element instead of streaming's ~10 per client-element).
 *   client_ids[j], weights[j]  as fa_accumulate; contributions apply in this order
 *   flat_ptrs[j]  client j's update over the whole flat layout (total numel values of
 *                 dtype_in, in this GPU's memory, cudaMalloc'd: managed memory is refused)
 *   out_ptrs      as fa_finalize (n_keys pointers, or one with FA_FLAT_OUT), in this
 *                 GPU's memory
 * Every client counts as having sent every key.  The result is bit-identical to
 * fa_accumulate of each update (in the same order) followed by fa_finalize; up to 16
 * clients take one pass, more take ceil(K/16) passes (the earlier ones through the
 * running sum).  A layout of more than 48 keys, small enough for the per-key tables to
 * travel in a launch's parameters, takes one launch of the subset-reduce kernel.  Needs a round with no contributions yet; closes it (fa_key_total works,
 * fa_finalize then returns FA_ERR_STATE because the outputs are already written).
 * If all weights are 0 nothing is written.
 * Errors: FA_ERR_ARG, FA_ERR_WEIGHT, FA_ERR_STATE, FA_ERR_CUDA. */
fa_status fa_reduce_resident(fa_ctx* ctx, uint32_t n_clients, const uint32_t* client_ids,
                             const double* weights, const void* const* flat_ptrs,
                             void* const* out_ptrs, void* stream);

/* A whole round of key subsets resident in device memory, reduced in one pass: the
 * adapter round of [FLARE] "Federating small adapters on a frozen VLM with FedUMM" (each
 * client sends only its adapter modules, a subset of the keys) combined per component as
 * "Coordinating training across clients" has it.  Client j sends the n_keys[j] whole keys
 * keys[o_j .. o_j + n_keys[j]) (o_j = n_keys[0] + ... + n_keys[j-1]), packed back to back
 * in that order in one buffer client_ptrs[j] (dtype_in values, this GPU's memory,
 * cudaMalloc'd).  For every key p with N_p > 0
 *     out[p][i] = round_to_dtype_out( sum over the clients that sent p, in call order, of
 *                                     n_k * x_k[p][i], / N_p )
 * straight from the client buffers: (J_p * s_in + s_out) bytes per element of key p, J_p
 * its reporters, where streaming moves s_in + 8 per client-element plus the finalize.
 * Bit-identical to fa_accumulate_keys for each client in call order followed by
 * fa_finalize.  Up to 16 reporters per key take one pass; if some key has more, the call
 * runs that sequence itself (the same bits).  Keys nobody sent, or whose reporters all
 * have weight 0, are not written.  A client id may appear once; weights as fa_accumulate.
 * Needs a round with no contributions yet (fa_reset); closes it (fa_key_total works,
 * fa_finalize then returns FA_ERR_STATE).  All or nothing: after an argument, range,
 * weight or state error the round is left empty.
 *   out_ptrs  as fa_finalize (n_keys pointers, or one with FA_FLAT_OUT), this GPU's memory
 * Ownership: the client buffers are read in order on `stream`; keep them until the work
 * queued there has completed.
 * Errors: FA_ERR_ARG, FA_ERR_RANGE, FA_ERR_WEIGHT, FA_ERR_STATE, FA_ERR_CUDA, FA_ERR_NOMEM,
 * FA_ERR_TIMEOUT. */
fa_status fa_reduce_subsets(fa_ctx* ctx, uint32_t n_clients, const uint32_t* client_ids,
                            const double* weights, const void* const* client_ptrs,
                            const uint32_t* n_keys, const int64_t* keys, void* const* out_ptrs,
                            void* stream);

/* Start a new round ([Clara] "Server-side workflow": the loop repeats per round):
 * forget weights, per-key totals, reporter masks and element counts.  The running sum
 * is not cleared (the first contribution of the next round overwrites it).  Waits
 * (bounded) for the context's queued work first.  If a device-side wait of the round
 * being discarded gave up (see fa_sync), the reset still happens and FA_ERR_INTERNAL is
 * returned.  Errors: FA_ERR_TIMEOUT, FA_ERR_CUDA (nothing reset), FA_ERR_INTERNAL. */
fa_status fa_reset(fa_ctx* ctx);

/* Wait (bounded by opts.timeout_ms) for the context's queued work, then free it (context
 * lifetime; no counterpart in the pages).  NULL is accepted.
 * Errors: FA_ERR_TIMEOUT (the context is then still freed). */
fa_status fa_close(fa_ctx* ctx);

/* Per-key weight total N_p (fp64, summed in ascending client id) and the number of
 * clients that sent key p, from the host bookkeeping -- exact, no device access.  The
 * per-component totals of [FLARE]'s client update contract ("Coordinating training across
 * clients"), over the sample counts of [Part] section 2. */
fa_status fa_key_total(const fa_ctx* ctx, uint32_t key, double* sum_nk, uint32_t* n_clients);

/* Wait, bounded by opts.timeout_ms, until all work the context queued has completed
 * (no counterpart in the pages).  Returns FA_ERR_TIMEOUT (never hangs) or FA_ERR_CUDA if
 * that work failed.  Every mbarrier wait inside the kernels is bounded too; one that gave
 * up sets a bit in this context's own device error word (never another context's), and
 * fa_sync (also fa_reset and fa_close, which call it) then returns FA_ERR_INTERNAL: that
 * round's results are invalid, and later calls return FA_ERR_CUDA until fa_reset, which
 * clears the word. */
fa_status fa_sync(fa_ctx* ctx);

/* Counters since fa_open (host-side, exact): among them the client bytes received per
 * round, the quantity [FLARE]'s "Federating small adapters on a frozen VLM with FedUMM"
 * compares between full-model and adapter-only updates. */
fa_status fa_get_stats(const fa_ctx* ctx, fa_stats* out);

/* Options of fa_partition_plan (NULL = {1, 0, 0.5, 0.05}: the "time only" policy). */
typedef struct {
    double w_time;      /* w_t >= 0: weight of the per-sample time cost */
    double w_energy;    /* w_e >= 0: weight of the per-sample energy cost (w_t + w_e > 0) */
    double ema_alpha;   /* 0 < alpha <= 1: weight of the newest measurement in the moving average */
    double deadband;    /* >= 0: keep the allocation if no share would move by more than this
                           fraction of its current value */
} fa_partition_opts;

/* Next round's sample counts n_i (the FedAvg weights) from this round's measurements:
 * the adaptive controller of [Part] section 2, "The adaptive controller" -- per-sample
 * costs tau_i = t_i / n_i and eps_i = e_i / n_i, smoothed by an exponential moving
 * average; combined cost c_i = w_t * tau^_i / median(tau^) + w_e * eps^_i / median(eps^);
 * the fixed budget sum(n_i) split inversely proportional to c_i (every participant keeps
 * at least one sample, remainders by largest fraction, ties to the lower index) unless
 * no share would move by more than the deadband.  The page fixes neither alpha nor the
 * deadband (defaults 0.5 and 5 %).  A zero median falls back to the mean (all zero: that
 * cost is left out); a zero combined cost is floored at 1e-12 of the largest.
 *   m           participants
 *   time_s, energy_j, samples   this round's t_i >= 0, e_i >= 0, n_i >= 1
 *   ema_tau, ema_eps            in/out moving-average state (negative or NaN = no history)
 *   new_samples out: next round's n_i (sums to the same budget)
 * Host code only; needs no GPU.  Errors: FA_ERR_ARG, FA_ERR_RANGE (budget overflow). */
fa_status fa_partition_plan(uint32_t m, const double* time_s, const double* energy_j,
                            const uint64_t* samples, double* ema_tau, double* ema_eps,
                            const fa_partition_opts* opts, uint64_t* new_samples);

/* Largest tensor fa_aggregate_noalloc takes (elements): 2^22, i.e. a 16 MiB fp32 sum. */
#define FA_NOALLOC_MAX_ELEMS 4194304ull

/* Aggregate ONE tensor of n_clients resident updates without allocating anything.
 * The pages have no counterpart: this is for callers that cannot let a library call
 * cudaMalloc -- a process whose device memory belongs to another allocator (a
 * framework's caching pool, a server that reserves its memory at start-up) or that
 * forbids allocation on its request path.  It computes what fa_open + fa_accumulate
 * (client 0, 1, ... in order) + fa_finalize + fa_close compute for a one-key layout,
 * with the same accumulate and finalize kernels and the same bits, but keeps its device
 * state in fixed arrays inside the library's device image instead of allocated memory:
 * the fp32 running sum (FA_NOALLOC_MAX_ELEMS floats, 16 MiB), a one-entry finalize
 * table (written by a one-thread kernel on `stream`) and an error word of its own --
 * held on every GPU that loads the library until the process exits.
 *   weights[j]       n_j: finite, >= 0, <= 2^24
 *   client_ptrs[j]   numel values of dtype_in in this device's memory (cudaMalloc'd;
 *                    managed memory is refused)
 *   out              numel values of dtype_out in this device's memory (or managed memory,
 *                    written with plain stores); left untouched
 *                    if sum(weights) == 0
 *   stream           cudaStream_t (as void*) the work is queued on; the call does not wait
 * The first call on each device looks up the array's device address (set-up); make that
 * first call before any stream capture.  Every call uses the same array and it keeps the
 * previous call's contents: each call overwrites what it uses before reading it, and
 * calls that overlap on the GPU (different streams, or different host threads without
 * ordering) race on it.  Calls no cudaMalloc, cudaFree or other allocating routine.
 * The call does not wait, so a device-side wait that gave up (see fa_sync) cannot be
 * reported by it: fa_aggregate_noalloc_status reports it.  The status returned is that of
 * this call's own launches.
 * Errors: FA_ERR_RANGE if numel > FA_NOALLOC_MAX_ELEMS (nothing is launched),
 * FA_ERR_ARG, FA_ERR_WEIGHT, FA_ERR_DTYPE, FA_ERR_CUDA.  numel == 0 or n_clients == 0
 * is a no-op. */
fa_status fa_aggregate_noalloc(uint32_t n_clients, const double* weights,
                               const void* const* client_ptrs, uint64_t numel, fa_dtype dtype_in,
                               fa_dtype dtype_out, void* out, void* stream);

/* Whether the fa_aggregate_noalloc calls on the current device since the last check ran
 * clean (no counterpart in the pages).  Waits, bounded by timeout_ms (0 = 60000), for the
 * work queued on `stream` (the stream the calls used), then reads the no-allocation error
 * word of the current device and clears it.  Allocates nothing.  The word is shared by
 * every fa_aggregate_noalloc call on the device (never by contexts, which have their own),
 * so check after the calls whose results are to be trusted.
 * Returns FA_OK, FA_ERR_INTERNAL (a bounded device-side wait gave up in one of those
 * calls: their outputs are invalid), FA_ERR_TIMEOUT (the stream's work did not finish in
 * time; nothing was read) or FA_ERR_CUDA. */
fa_status fa_aggregate_noalloc_status(void* stream, uint32_t timeout_ms);

/* Static text for a status code (no counterpart in the pages). */
const char* fa_strerror(fa_status status);

/* Detail of the last error on this context ("" if none; no counterpart in the pages);
 * valid until the next call.
 * With FA_LOG set in the environment (any value but "0"), each failure a call reports is
 * also written to stderr as "[fedavg] <status text>: <detail>". */
const char* fa_last_error(const fa_ctx* ctx);

#ifdef __cplusplus
}
#endif

#endif /* FEDAVG_H */
