// Test-only C entry points over the host ledger of the aggregation library
// (compiled with g++ on the CPU, no CUDA): lets the CPU suite check the
// bookkeeping -- validation, per-key totals, reporter masks, first-contribution
// tracking, flat-chunk splitting -- without a GPU.
#include <cstring>
#include <string>
#include <vector>

#include "ledger.hpp"

namespace {
struct Handle {
    fa::Ledger lg;
    std::string err;
    std::vector<fa::Piece> pieces;
    std::vector<fa::FinItem> items;
};
}  // namespace

extern "C" {

void* lg_new(const uint64_t* numels, uint32_t n_keys, uint32_t max_clients, int32_t* status) {
    auto* h = new Handle;
    *status = h->lg.init(numels, n_keys, max_clients, &h->err);
    if (*status != 0) {
        delete h;
        return nullptr;
    }
    return h;
}

void lg_free(void* p) { delete static_cast<Handle*>(p); }

const char* lg_error(void* p) { return static_cast<Handle*>(p)->err.c_str(); }

// pieces out: rows of (key, chunk_off, acc_idx, len, first)
int32_t lg_accumulate(void* p, const uint32_t* clients, const double* weights, uint32_t J,
                      int64_t key, uint64_t offset, uint64_t len, uint64_t* rows,
                      uint32_t max_rows, uint32_t* n_rows) {
    auto* h = static_cast<Handle*>(p);
    int32_t st = h->lg.plan_accumulate(clients, weights, J, key, offset, len, &h->pieces, &h->err);
    *n_rows = static_cast<uint32_t>(h->pieces.size());
    for (uint32_t i = 0; i < *n_rows && i < max_rows; ++i) {
        const auto& q = h->pieces[i];
        uint64_t* r = rows + 5 * i;
        r[0] = q.key;
        r[1] = q.chunk_off;
        r[2] = q.acc_idx;
        r[3] = q.len;
        r[4] = q.first ? 1 : 0;
    }
    return st;
}

// one client, n chunks; pieces out: rows of (chunk, key, chunk_off, acc_idx, len, first)
int32_t lg_accumulate_keys(void* p, uint32_t client, double weight, uint32_t n,
                           const int64_t* keys, const uint64_t* offsets, const uint64_t* lens,
                           uint64_t* rows, uint32_t max_rows, uint32_t* n_rows) {
    auto* h = static_cast<Handle*>(p);
    int32_t st = h->lg.plan_accumulate_keys(client, weight, n, keys, offsets, lens, &h->pieces,
                                            &h->err);
    *n_rows = static_cast<uint32_t>(h->pieces.size());
    for (uint32_t i = 0; i < *n_rows && i < max_rows; ++i) {
        const auto& q = h->pieces[i];
        uint64_t* r = rows + 6 * i;
        r[0] = q.chunk;
        r[1] = q.key;
        r[2] = q.chunk_off;
        r[3] = q.acc_idx;
        r[4] = q.len;
        r[5] = q.first ? 1 : 0;
    }
    return st;
}

int32_t lg_whole_keys(void* p, uint32_t client, double weight, uint32_t n, const int64_t* keys) {
    auto* h = static_cast<Handle*>(p);
    return h->lg.record_whole_keys(client, weight, n, keys, &h->err);
}

// items out: rows of (key, acc_idx, flat_off, numel, reporters) and totals
int32_t lg_finalize(void* p, uint64_t* rows, double* totals, uint32_t max_rows, uint32_t* n_rows) {
    auto* h = static_cast<Handle*>(p);
    int32_t st = h->lg.plan_finalize(&h->items, &h->err);
    if (st == 0) h->lg.close();
    *n_rows = static_cast<uint32_t>(h->items.size());
    for (uint32_t i = 0; i < *n_rows && i < max_rows; ++i) {
        const auto& q = h->items[i];
        uint64_t* r = rows + 5 * i;
        r[0] = q.key;
        r[1] = q.acc_idx;
        r[2] = q.flat_off;
        r[3] = q.numel;
        r[4] = q.reporters;
        totals[i] = q.total;
    }
    return st;
}

// one client's final contribution; pieces out as lg_accumulate, plus each piece's N_p
int32_t lg_accumulate_final(void* p, uint32_t client, double weight, int64_t key, uint64_t offset,
                            uint64_t len, uint64_t* rows, double* totals, uint32_t max_rows,
                            uint32_t* n_rows) {
    auto* h = static_cast<Handle*>(p);
    std::vector<double> tot;
    int32_t st = h->lg.plan_accumulate_final(client, weight, key, offset, len, &h->pieces, &tot, &h->err);
    *n_rows = static_cast<uint32_t>(h->pieces.size());
    for (uint32_t i = 0; i < *n_rows && i < max_rows; ++i) {
        const auto& q = h->pieces[i];
        uint64_t* r = rows + 5 * i;
        r[0] = q.key;
        r[1] = q.chunk_off;
        r[2] = q.acc_idx;
        r[3] = q.len;
        r[4] = q.first ? 1 : 0;
        totals[i] = tot[i];
    }
    return st;
}

// whether a final contribution has written a range this round
int32_t lg_has_final(void* p) { return static_cast<Handle*>(p)->lg.has_final() ? 1 : 0; }

// ranges to write (without closing the round): rows of (key, koff, acc_idx, flat_off, numel,
// reporters) and totals
int32_t lg_finalize_ranges(void* p, uint64_t* rows, double* totals, uint32_t max_rows, uint32_t* n_rows) {
    auto* h = static_cast<Handle*>(p);
    int32_t st = h->lg.plan_finalize(&h->items, &h->err);
    *n_rows = static_cast<uint32_t>(h->items.size());
    for (uint32_t i = 0; i < *n_rows && i < max_rows; ++i) {
        const auto& q = h->items[i];
        uint64_t* r = rows + 6 * i;
        r[0] = q.key;
        r[1] = q.koff;
        r[2] = q.acc_idx;
        r[3] = q.flat_off;
        r[4] = q.numel;
        r[5] = q.reporters;
        totals[i] = q.total;
    }
    return st;
}

void lg_reset(void* p) { static_cast<Handle*>(p)->lg.reset(); }

int32_t lg_key_total(void* p, uint32_t key, double* total, uint32_t* reporters) {
    return static_cast<Handle*>(p)->lg.key_total(key, total, reporters);
}

uint64_t lg_acc_off(void* p, uint32_t key) { return static_cast<Handle*>(p)->lg.acc_off(key); }
uint64_t lg_padded(void* p) { return static_cast<Handle*>(p)->lg.padded_elems(); }
}
