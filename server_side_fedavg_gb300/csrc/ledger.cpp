// Host bookkeeping for one aggregation round (see ledger.hpp).
#include "ledger.hpp"

#include <algorithm>
#include <cmath>
#include <cstdio>

namespace fa {

namespace {

std::string fmt(const char* f, unsigned long long a = 0, unsigned long long b = 0,
                unsigned long long c = 0, unsigned long long d = 0) {
    char buf[256];
    std::snprintf(buf, sizeof buf, f, a, b, c, d);
    return buf;
}

constexpr double kMaxWeight = 16777216.0;  // 2^24: integers up to here are exact in fp32

}  // namespace

int32_t Ledger::init(const uint64_t* numels, uint32_t n_keys, uint32_t max_clients,
                     std::string* err) {
    if (numels == nullptr || n_keys == 0) {
        *err = "layout is empty";
        return kErrArg;
    }
    if (max_clients == 0) {
        *err = "max_clients must be >= 1";
        return kErrArg;
    }
    numel_.assign(numels, numels + n_keys);
    flat_off_.resize(n_keys);
    acc_off_.resize(n_keys);
    uint64_t flat = 0, acc = 0;
    for (uint32_t p = 0; p < n_keys; ++p) {
        uint64_t n = numel_[p];
        if (n == 0) {
            *err = fmt("key %llu has numel 0", p);
            return kErrArg;
        }
        if (n > (UINT64_MAX >> 4) - acc) {
            *err = "layout too large";
            return kErrArg;
        }
        flat_off_[p] = flat;
        acc_off_[p] = acc;
        flat += n;
        acc += (n + kAccPad - 1) / kAccPad * kAccPad;
    }
    total_ = flat;
    padded_ = acc;
    max_clients_ = max_clients;
    weight_.assign(max_clients, 0.0);
    has_weight_.assign(max_clients, 0);
    recv_.assign(static_cast<size_t>(max_clients) * n_keys, 0);
    started_.assign(n_keys, {});
    written_.assign(n_keys, {});
    frozen_.assign(n_keys, 0);
    closed_ = false;
    return kOk;
}

bool Ledger::has_contributions() const {
    for (uint64_t v : recv_)
        if (v != 0) return true;
    return false;
}

bool Ledger::has_final() const {
    for (const auto& w : written_)
        if (!w.empty()) return true;
    return false;
}

void Ledger::reset() {
    std::fill(weight_.begin(), weight_.end(), 0.0);
    std::fill(has_weight_.begin(), has_weight_.end(), 0);
    std::fill(recv_.begin(), recv_.end(), 0);
    for (auto& s : started_) s.clear();
    for (auto& s : written_) s.clear();
    std::fill(frozen_.begin(), frozen_.end(), 0);
    closed_ = false;
}

int32_t Ledger::check_frozen(uint32_t c, const std::vector<Span>& spans, size_t from, size_t to,
                             std::string* err) const {
    const uint32_t nk = n_keys();
    for (size_t i = from; i < to; ++i) {
        const Span& s = spans[i];
        if (!frozen_[s.p]) continue;
        if (recv_[static_cast<size_t>(c) * nk + s.p] == 0) {
            *err = fmt("key %llu already has a final contribution: client %llu cannot start sending it",
                       s.p, c);
            return kErrState;
        }
        for (const auto& w : written_[s.p]) {
            if (w.first < s.koff + s.n && s.koff < w.second) {
                *err = fmt("elements [%llu, %llu) of key %llu were already written by a final contribution",
                           w.first, w.second, s.p);
                return kErrState;
            }
        }
    }
    return kOk;
}

void Ledger::split_and_mark(uint32_t p, uint64_t a, uint64_t b,
                            std::vector<std::pair<uint64_t, bool>>* runs) {
    // runs: (end, first) pairs covering [a, b) in order
    auto& iv = started_[p];
    uint64_t cur = a;
    for (const auto& s : iv) {
        if (s.second <= cur) continue;
        if (s.first >= b) break;
        if (s.first > cur) {
            runs->emplace_back(s.first, true);
            cur = s.first;
        }
        uint64_t e = std::min(s.second, b);
        runs->emplace_back(e, false);
        cur = e;
        if (cur >= b) break;
    }
    if (cur < b) runs->emplace_back(b, true);
    // insert [a, b) and merge overlapping or touching intervals
    std::vector<std::pair<uint64_t, uint64_t>> merged;
    merged.reserve(iv.size() + 1);
    uint64_t na = a, nb = b;
    bool placed = false;
    for (const auto& s : iv) {
        if (s.second < na) {
            merged.push_back(s);
        } else if (s.first > nb) {
            if (!placed) {
                merged.emplace_back(na, nb);
                placed = true;
            }
            merged.push_back(s);
        } else {
            na = std::min(na, s.first);
            nb = std::max(nb, s.second);
        }
    }
    if (!placed) merged.emplace_back(na, nb);
    iv.swap(merged);
}

int32_t Ledger::check_client(uint32_t c, double w, std::string* err) const {
    if (c >= max_clients_) {
        *err = fmt("client id %llu >= max_clients %llu", c, max_clients_);
        return kErrArg;
    }
    if (!std::isfinite(w) || w < 0.0 || w > kMaxWeight) {
        *err = fmt("client %llu: weight must be finite, >= 0 and <= 2^24", c);
        return kErrWeight;
    }
    if (has_weight_[c] && weight_[c] != w) {
        *err = fmt("client %llu: weight differs from its earlier chunks this round", c);
        return kErrWeight;
    }
    return kOk;
}

int32_t Ledger::chunk_spans(int64_t key, uint64_t offset, uint64_t len, std::vector<Span>* spans,
                            std::string* err) const {
    const uint32_t nk = n_keys();
    if (key != -1 && (key < 0 || key >= static_cast<int64_t>(nk))) {
        *err = fmt("key %llu out of range (n_keys %llu)", static_cast<unsigned long long>(key), nk);
        return kErrArg;
    }
    const uint64_t limit = key == -1 ? total_ : numel_[static_cast<uint32_t>(key)];
    if (offset > limit || len > limit - offset) {
        *err = fmt("chunk [%llu, +%llu) past the end (%llu elements)", offset, len, limit);
        return kErrRange;
    }
    if (len == 0) return kOk;
    if (key >= 0) {
        spans->push_back({static_cast<uint32_t>(key), offset, len, 0});
        return kOk;
    }
    auto it = std::upper_bound(flat_off_.begin(), flat_off_.end(), offset);
    uint32_t p = static_cast<uint32_t>(it - flat_off_.begin()) - 1;
    uint64_t pos = offset, end = offset + len;
    while (pos < end) {
        uint64_t kend = flat_off_[p] + numel_[p];
        uint64_t e = std::min(end, kend);
        spans->push_back({p, pos - flat_off_[p], e - pos, pos - offset});
        pos = e;
        ++p;
    }
    return kOk;
}

void Ledger::emit_pieces(const std::vector<Span>& spans, size_t from, size_t to, uint32_t chunk,
                         std::vector<Piece>* out) {
    std::vector<std::pair<uint64_t, bool>> runs;
    for (size_t i = from; i < to; ++i) {
        const Span& s = spans[i];
        runs.clear();
        split_and_mark(s.p, s.koff, s.koff + s.n, &runs);
        uint64_t a = s.koff;
        for (const auto& r : runs) {
            Piece pc;
            pc.key = s.p;
            pc.chunk = chunk;
            pc.chunk_off = s.coff + (a - s.koff);
            pc.acc_idx = acc_off_[s.p] + a;
            pc.len = r.first - a;
            pc.first = r.second;
            out->push_back(pc);
            a = r.first;
        }
    }
}

int32_t Ledger::plan_accumulate(const uint32_t* clients, const double* weights, uint32_t J,
                                int64_t key, uint64_t offset, uint64_t len,
                                std::vector<Piece>* out, std::string* err) {
    out->clear();
    if (closed_) {
        *err = "round already finalized: call fa_reset before accumulating again";
        return kErrState;
    }
    if (J == 0 || clients == nullptr || weights == nullptr) {
        *err = "no clients given";
        return kErrArg;
    }
    for (uint32_t j = 0; j < J; ++j) {
        const uint32_t c = clients[j];
        for (uint32_t i = 0; i < j; ++i) {
            if (clients[i] == c) {
                *err = fmt("client id %llu appears twice in one batch", c);
                return kErrArg;
            }
        }
        int32_t st = check_client(c, weights[j], err);
        if (st != kOk) return st;
    }
    std::vector<Span> spans;
    int32_t st = chunk_spans(key, offset, len, &spans, err);
    if (st != kOk || len == 0) return st;
    const uint32_t nk = n_keys();
    for (uint32_t j = 0; j < J; ++j) {
        uint32_t c = clients[j];
        for (const auto& s : spans) {
            uint64_t have = recv_[static_cast<size_t>(c) * nk + s.p];
            if (s.n > numel_[s.p] - have) {
                *err = fmt("client %llu would send more than numel (%llu) elements of key %llu",
                           c, numel_[s.p], s.p);
                return kErrRange;
            }
        }
        st = check_frozen(c, spans, 0, spans.size(), err);
        if (st != kOk) return st;
    }
    // commit
    for (uint32_t j = 0; j < J; ++j) {
        uint32_t c = clients[j];
        weight_[c] = weights[j];
        has_weight_[c] = 1;
        for (const auto& s : spans) recv_[static_cast<size_t>(c) * nk + s.p] += s.n;
    }
    emit_pieces(spans, 0, spans.size(), 0, out);
    return kOk;
}

int32_t Ledger::plan_accumulate_keys(uint32_t client, double weight, uint32_t n,
                                     const int64_t* keys, const uint64_t* offsets,
                                     const uint64_t* lens, std::vector<Piece>* out,
                                     std::string* err) {
    out->clear();
    if (closed_) {
        *err = "round already finalized: call fa_reset before accumulating again";
        return kErrState;
    }
    if (n > 0 && (keys == nullptr || offsets == nullptr || lens == nullptr)) {
        *err = "keys, offsets or lengths is NULL";
        return kErrArg;
    }
    int32_t st = check_client(client, weight, err);
    if (st != kOk) return st;
    // every chunk's spans, and the counts this call adds per key, checked before anything
    // is recorded
    std::vector<Span> spans;
    std::vector<size_t> first_span(n + 1, 0);
    const uint32_t nk = n_keys();
    for (uint32_t i = 0; i < n; ++i) {
        first_span[i] = spans.size();
        st = chunk_spans(keys[i], offsets[i], lens[i], &spans, err);
        if (st != kOk) {
            *err = fmt("chunk %llu: ", i) + *err;
            return st;
        }
    }
    first_span[n] = spans.size();
    std::vector<uint64_t> pending;   // per key touched, sorted by key
    std::vector<uint32_t> touched;
    for (const auto& s : spans) touched.push_back(s.p);
    std::sort(touched.begin(), touched.end());
    touched.erase(std::unique(touched.begin(), touched.end()), touched.end());
    pending.assign(touched.size(), 0);
    for (const auto& s : spans) {
        const size_t t = static_cast<size_t>(
            std::lower_bound(touched.begin(), touched.end(), s.p) - touched.begin());
        pending[t] += s.n;
        const uint64_t have = recv_[static_cast<size_t>(client) * nk + s.p];
        if (pending[t] > numel_[s.p] - have) {
            *err = fmt("client %llu would send more than numel (%llu) elements of key %llu",
                       client, numel_[s.p], s.p);
            return kErrRange;
        }
    }
    st = check_frozen(client, spans, 0, spans.size(), err);
    if (st != kOk) return st;
    // commit
    if (spans.empty()) return kOk;
    weight_[client] = weight;
    has_weight_[client] = 1;
    for (size_t t = 0; t < touched.size(); ++t)
        recv_[static_cast<size_t>(client) * nk + touched[t]] += pending[t];
    for (uint32_t i = 0; i < n; ++i) emit_pieces(spans, first_span[i], first_span[i + 1], i, out);
    return kOk;
}

int32_t Ledger::record_whole_keys(uint32_t client, double weight, uint32_t n, const int64_t* keys,
                                  std::string* err) {
    if (closed_) {
        *err = "round already finalized: call fa_reset before accumulating again";
        return kErrState;
    }
    if (n > 0 && keys == nullptr) {
        *err = "keys is NULL";
        return kErrArg;
    }
    int32_t st = check_client(client, weight, err);
    if (st != kOk) return st;
    const uint32_t nk = n_keys();
    uint64_t* row = recv_.data() + static_cast<size_t>(client) * nk;
    uint32_t i = 0;
    for (; i < n; ++i) {
        const int64_t k = keys[i];
        if (k < 0 || k >= static_cast<int64_t>(nk)) {
            *err = fmt("entry %llu: key %llu out of range (n_keys %llu)", i,
                       static_cast<unsigned long long>(k), nk);
            st = kErrArg;
            break;
        }
        if (row[k] != 0) {
            *err = fmt("client %llu would send more than numel (%llu) elements of key %llu",
                       client, numel_[static_cast<size_t>(k)], static_cast<unsigned long long>(k));
            st = kErrRange;
            break;
        }
        if (frozen_[static_cast<size_t>(k)]) {
            *err = fmt("key %llu already has a final contribution", static_cast<unsigned long long>(k));
            st = kErrState;
            break;
        }
        row[k] = numel_[static_cast<size_t>(k)];
    }
    if (st != kOk) {
        for (uint32_t j = 0; j < i; ++j) row[keys[j]] = 0;   // undo this call's marks
        return st;
    }
    if (n > 0) {
        weight_[client] = weight;
        has_weight_[client] = 1;
    }
    return kOk;
}

int32_t Ledger::plan_accumulate_final(uint32_t client, double weight, int64_t key, uint64_t offset,
                                      uint64_t len, std::vector<Piece>* out, std::vector<double>* totals,
                                      std::string* err) {
    out->clear();
    totals->clear();
    if (closed_) {
        *err = "round already finalized: call fa_reset before accumulating again";
        return kErrState;
    }
    int32_t st = check_client(client, weight, err);
    if (st != kOk) return st;
    std::vector<Span> spans;
    st = chunk_spans(key, offset, len, &spans, err);
    if (st != kOk || len == 0) return st;
    const uint32_t nk = n_keys();
    for (const auto& s : spans) {
        const uint64_t have = recv_[static_cast<size_t>(client) * nk + s.p];
        if (s.n > numel_[s.p] - have) {
            *err = fmt("client %llu would send more than numel (%llu) elements of key %llu",
                       client, numel_[s.p], s.p);
            return kErrRange;
        }
        for (uint32_t c = 0; c < max_clients_; ++c) {
            if (c == client) continue;
            const uint64_t h = recv_[static_cast<size_t>(c) * nk + s.p];
            if (h != 0 && h != numel_[s.p]) {
                *err = fmt("a final contribution to key %llu needs every other sender's whole key: "
                           "client %llu has sent %llu of %llu elements",
                           s.p, c, h, numel_[s.p]);
                return kErrIncomplete;
            }
        }
    }
    st = check_frozen(client, spans, 0, spans.size(), err);
    if (st != kOk) return st;
    // commit
    weight_[client] = weight;
    has_weight_[client] = 1;
    for (const auto& s : spans) recv_[static_cast<size_t>(client) * nk + s.p] += s.n;
    emit_pieces(spans, 0, spans.size(), 0, out);
    for (const auto& s : spans) {
        frozen_[s.p] = 1;
        // add [koff, koff + n) to the written ranges (disjoint from them, checked above)
        auto& w = written_[s.p];
        w.emplace_back(s.koff, s.koff + s.n);
        std::sort(w.begin(), w.end());
        std::vector<std::pair<uint64_t, uint64_t>> merged;
        for (const auto& r : w) {
            if (!merged.empty() && merged.back().second == r.first) merged.back().second = r.second;
            else merged.push_back(r);
        }
        w.swap(merged);
    }
    for (const Piece& pc : *out) {
        double total = 0.0;
        key_total(pc.key, &total, nullptr);
        totals->push_back(total);
    }
    return kOk;
}

int32_t Ledger::plan_finalize(std::vector<FinItem>* out, std::string* err) const {
    out->clear();
    const uint32_t nk = n_keys();
    for (uint32_t c = 0; c < max_clients_; ++c) {
        for (uint32_t p = 0; p < nk; ++p) {
            uint64_t have = recv_[static_cast<size_t>(c) * nk + p];
            if (have != 0 && have != numel_[p]) {
                *err = fmt("client %llu sent %llu of %llu elements of key %llu", c, have,
                           numel_[p], p);
                return kErrIncomplete;
            }
        }
    }
    for (uint32_t p = 0; p < nk; ++p) {
        double total = 0.0;
        uint32_t reporters = 0;
        key_total(p, &total, &reporters);
        if (reporters == 0 || total == 0.0) continue;
        // the key less the ranges final contributions wrote
        uint64_t a = 0;
        for (const auto& w : written_[p]) {
            if (w.first > a)
                out->push_back({p, acc_off_[p] + a, flat_off_[p] + a, w.first - a, total, reporters, a});
            a = w.second;
        }
        if (a < numel_[p])
            out->push_back({p, acc_off_[p] + a, flat_off_[p] + a, numel_[p] - a, total, reporters, a});
    }
    return kOk;
}

int32_t Ledger::key_total(uint32_t key, double* total, uint32_t* reporters) const {
    if (key >= n_keys()) return kErrArg;
    const uint32_t nk = n_keys();
    double t = 0.0;
    uint32_t r = 0;
    for (uint32_t c = 0; c < max_clients_; ++c) {
        if (recv_[static_cast<size_t>(c) * nk + key] != 0) {
            t += weight_[c];
            ++r;
        }
    }
    if (total) *total = t;
    if (reporters) *reporters = r;
    return kOk;
}

}  // namespace fa
