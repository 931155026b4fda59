// Host bookkeeping for one aggregation round: layout, client weights, which
// client sent which key (the reporter mask), element counts per (client, key),
// and which elements of the running sum already hold a contribution.
//
// The client update contract of "Building Federated Multimodal AI Workflows
// with NVIDIA FLARE" ("Coordinating training across clients") lets clients
// update different components; the per-key reporter set S_p and its own total
// N_p implement it.  Weights are sample counts ("Technical Summary: Adaptive
// Data Partitioning ...", section 2, "The adaptive controller").
//
// Pure C++ (no CUDA): the runtime turns the pieces planned here into kernel
// launches.
#pragma once

#include <cstdint>
#include <string>
#include <utility>
#include <vector>

namespace fa {

// Elements per key are padded to this multiple in the running sum so every
// key starts on a 128-byte boundary.
constexpr uint64_t kAccPad = 32;

enum Status : int32_t {
    kOk = 0,
    kErrArg = -1,
    kErrRange = -2,
    kErrDtype = -3,
    kErrWeight = -4,
    kErrIncomplete = -5,
    kErrState = -6,
    kErrNomem = -7,
    kErrCuda = -8,
    kErrTimeout = -9,
    kErrInternal = -10,
};

// One contiguous run of a chunk that lands in one key.
struct Piece {
    uint32_t key;
    uint32_t chunk;       // which chunk of the call (0 for a single-chunk call)
    uint64_t chunk_off;   // element offset within the chunk
    uint64_t acc_idx;     // element index in the padded running sum
    uint64_t len;         // elements
    bool first;           // no earlier contribution to these elements this round
};

// One range of a key to write at finalize: the whole key, or the part of it that no final
// contribution has written yet.
struct FinItem {
    uint32_t key;
    uint64_t acc_idx;     // start in the padded running sum
    uint64_t flat_off;    // start in the flat (unpadded) layout
    uint64_t numel;       // elements of the range
    double total;         // N_p
    uint32_t reporters;   // |S_p|
    uint64_t koff = 0;    // start of the range within the key
};

class Ledger {
public:
    // numels[0..n_keys) >= 1.  Returns kOk or kErrArg.
    int32_t init(const uint64_t* numels, uint32_t n_keys, uint32_t max_clients, std::string* err);

    // Validate and record J client chunks over one element range (J = 1 for a
    // plain accumulate).  On success fills `out` with the pieces (in key order;
    // a piece's `first` flag tells whether the first client of the batch
    // starts the running sum there).  On error nothing changes.
    int32_t plan_accumulate(const uint32_t* clients, const double* weights, uint32_t J,
                            int64_t key, uint64_t offset, uint64_t len,
                            std::vector<Piece>* out, std::string* err);

    // Validate and record n chunks of ONE client, chunk i covering [offsets[i], +lens[i])
    // of key keys[i] (or of the flat layout for -1), as n plain accumulates in that order
    // would -- counts sent earlier in the same call included.  All or nothing: on error
    // nothing changes.  Pieces come in chunk order, each tagged with its chunk index.
    int32_t plan_accumulate_keys(uint32_t client, double weight, uint32_t n, const int64_t* keys,
                                 const uint64_t* offsets, const uint64_t* lens,
                                 std::vector<Piece>* out, std::string* err);

    // Record n WHOLE keys sent by one client (a round-level subset reduce): every key id
    // in range, none sent by this client before (in this call or earlier), the weight
    // valid and consistent.  O(n); no pieces (the caller reduces the round in one pass,
    // so the first-contribution tracking is not needed; the round is closed right after).
    // All or nothing: on error nothing changes.
    int32_t record_whole_keys(uint32_t client, double weight, uint32_t n, const int64_t* keys,
                              std::string* err);

    // Validate and record ONE client's last contribution to a range (fa_accumulate_final):
    // as plan_accumulate with J = 1, and for every key the range touches, every OTHER
    // sender of that key has already sent all of it (else kErrIncomplete), so the key's
    // weight total is final.  On success `out` holds the pieces and `totals` each piece's
    // N_p (this client included); the keys touched are frozen (no new sender from now on)
    // and the range is marked written (no further contribution to it; plan_finalize
    // leaves it out).  All or nothing: on error nothing changes.
    int32_t plan_accumulate_final(uint32_t client, double weight, int64_t key, uint64_t offset,
                                  uint64_t len, std::vector<Piece>* out, std::vector<double>* totals,
                                  std::string* err);

    // Check completeness and list the ranges to write: every key with N_p > 0, less what
    // final contributions have already written.  Changes nothing.
    int32_t plan_finalize(std::vector<FinItem>* out, std::string* err) const;

    // Close the round: accumulation is refused until reset().
    void close() { closed_ = true; }

    void reset();

    int32_t key_total(uint32_t key, double* total, uint32_t* reporters) const;

    uint32_t n_keys() const { return static_cast<uint32_t>(numel_.size()); }
    uint32_t max_clients() const { return max_clients_; }
    uint64_t numel(uint32_t p) const { return numel_[p]; }
    uint64_t flat_off(uint32_t p) const { return flat_off_[p]; }
    uint64_t acc_off(uint32_t p) const { return acc_off_[p]; }
    uint64_t total_elems() const { return total_; }
    uint64_t padded_elems() const { return padded_; }
    bool closed() const { return closed_; }
    // True once any client has sent any element this round.
    bool has_contributions() const;
    // True once a final contribution (plan_accumulate_final) has written a range this round.
    bool has_final() const;

private:
    // One run of a chunk inside one key.
    struct Span {
        uint32_t p;
        uint64_t koff, n, coff;   // offset within the key, length, offset within the chunk
    };
    // Range-check a chunk and cut it at key boundaries (appends to *spans).
    int32_t chunk_spans(int64_t key, uint64_t offset, uint64_t len, std::vector<Span>* spans,
                        std::string* err) const;
    int32_t check_client(uint32_t c, double w, std::string* err) const;
    // Pieces of spans[from, to) in order (marks them started), tagged with chunk `chunk`.
    void emit_pieces(const std::vector<Span>& spans, size_t from, size_t to, uint32_t chunk,
                     std::vector<Piece>* out);

    // Split [a, b) of key p into runs that are fresh / already started, then
    // mark all of [a, b) started.
    void split_and_mark(uint32_t p, uint64_t a, uint64_t b,
                        std::vector<std::pair<uint64_t, bool>>* runs_end_first);
    // Spans that a contribution of client c may not make: a new sender of a frozen key, or
    // a range a final contribution has written.  kOk or kErrState (with *err).
    int32_t check_frozen(uint32_t c, const std::vector<Span>& spans, size_t from, size_t to,
                         std::string* err) const;

    std::vector<uint64_t> numel_, flat_off_, acc_off_;
    uint64_t total_ = 0, padded_ = 0;
    uint32_t max_clients_ = 0;
    std::vector<double> weight_;        // per client
    std::vector<uint8_t> has_weight_;   // per client
    std::vector<uint64_t> recv_;        // [client * n_keys + key]
    std::vector<std::vector<std::pair<uint64_t, uint64_t>>> started_;  // per key, sorted disjoint
    std::vector<std::vector<std::pair<uint64_t, uint64_t>>> written_;  // per key: ranges a final
                                                                       // contribution wrote
    std::vector<uint8_t> frozen_;       // per key: its senders are final
    bool closed_ = false;
};

}  // namespace fa
