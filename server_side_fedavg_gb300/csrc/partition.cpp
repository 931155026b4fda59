// Next round's sample counts n_i -- the weights FedAvg uses -- from measured time and
// energy: the adaptive controller of "Technical Summary: Adaptive Data Partitioning
// for Energy-Efficient Federated and Distributed Learning in Heterogeneous Systems",
// section 2, "The adaptive controller":
//   Measurement   each participant i reports time t_i, energy e_i, sample count n_i;
//   Cost          per-sample tau_i = t_i / n_i and eps_i = e_i / n_i, smoothed by an
//                 exponential moving average;
//   Weighted split  c_i = w_t * tau^_i / median(tau^) + w_e * eps^_i / median(eps^);
//   Allocation    a fixed budget of samples split inversely proportional to c_i, kept
//                 as it is when the change would be negligible (a deadband).
// Host code only (no device work).  The page gives neither the EMA coefficient nor the
// deadband width: they are parameters (defaults 0.5 and 5 %).
#include <fedavg.h>

#include <algorithm>
#include <cmath>
#include <vector>

namespace {

double median(std::vector<double> v) {
    std::sort(v.begin(), v.end());
    const size_t m = v.size();
    return m % 2 ? v[m / 2] : 0.5 * (v[m / 2 - 1] + v[m / 2]);
}

// Normalise by the median; a zero median falls back to the mean, and an all-zero
// column to 1 for everyone (that cost then does not discriminate).
void normalise(const std::vector<double>& v, std::vector<double>* out) {
    double d = median(v);
    if (d == 0.0) {
        double s = 0.0;
        for (double x : v) s += x;
        d = s / static_cast<double>(v.size());
    }
    out->resize(v.size());
    for (size_t i = 0; i < v.size(); ++i) (*out)[i] = d == 0.0 ? 1.0 : v[i] / d;
}

}  // namespace

extern "C" fa_status fa_partition_plan(uint32_t m, const double* time_s, const double* energy_j,
                                       const uint64_t* samples, double* ema_tau, double* ema_eps,
                                       const fa_partition_opts* opts, uint64_t* new_samples) {
    if (m == 0 || time_s == nullptr || energy_j == nullptr || samples == nullptr ||
        ema_tau == nullptr || ema_eps == nullptr || new_samples == nullptr)
        return FA_ERR_ARG;
    fa_partition_opts o{1.0, 0.0, 0.5, 0.05};
    if (opts) o = *opts;
    if (!(o.w_time >= 0.0) || !(o.w_energy >= 0.0) || !(o.w_time + o.w_energy > 0.0) ||
        !(o.ema_alpha > 0.0 && o.ema_alpha <= 1.0) || !(o.deadband >= 0.0) ||
        !std::isfinite(o.w_time) || !std::isfinite(o.w_energy) || !std::isfinite(o.deadband))
        return FA_ERR_ARG;
    uint64_t budget = 0;
    for (uint32_t i = 0; i < m; ++i) {
        if (!(time_s[i] >= 0.0) || !(energy_j[i] >= 0.0) || !std::isfinite(time_s[i]) ||
            !std::isfinite(energy_j[i]) || samples[i] == 0)
            return FA_ERR_ARG;
        if (samples[i] > UINT64_MAX - budget) return FA_ERR_RANGE;
        budget += samples[i];
    }
    // per-sample costs, smoothed (a non-finite or negative state means no history)
    std::vector<double> tau(m), eps(m);
    for (uint32_t i = 0; i < m; ++i) {
        const double n = static_cast<double>(samples[i]);
        const double t = time_s[i] / n, e = energy_j[i] / n;
        const bool hist = std::isfinite(ema_tau[i]) && ema_tau[i] >= 0.0 &&
                          std::isfinite(ema_eps[i]) && ema_eps[i] >= 0.0;
        tau[i] = hist ? o.ema_alpha * t + (1.0 - o.ema_alpha) * ema_tau[i] : t;
        eps[i] = hist ? o.ema_alpha * e + (1.0 - o.ema_alpha) * ema_eps[i] : e;
    }
    std::vector<double> nt, ne;
    normalise(tau, &nt);
    normalise(eps, &ne);
    // combined cost and target shares (inverse cost); a zero cost is floored at 1e-12 of
    // the largest so that every share stays finite
    std::vector<double> c(m);
    double cmax = 0.0;
    for (uint32_t i = 0; i < m; ++i) {
        c[i] = o.w_time * nt[i] + o.w_energy * ne[i];
        cmax = std::max(cmax, c[i]);
    }
    double inv_sum = 0.0;
    std::vector<double> share(m);
    for (uint32_t i = 0; i < m; ++i) {
        const double ci = std::max(c[i], 1e-12 * cmax);
        share[i] = ci > 0.0 ? 1.0 / ci : 1.0;
        inv_sum += share[i];
    }
    for (uint32_t i = 0; i < m; ++i) share[i] /= inv_sum;
    for (uint32_t i = 0; i < m; ++i) {
        ema_tau[i] = tau[i];
        ema_eps[i] = eps[i];
    }
    // deadband: keep the allocation if no share moves by more than `deadband` (relative)
    const double B = static_cast<double>(budget);
    bool move = false;
    for (uint32_t i = 0; i < m; ++i) {
        const double cur = static_cast<double>(samples[i]) / B;
        if (std::fabs(share[i] - cur) > o.deadband * cur) move = true;
    }
    if (!move) {
        for (uint32_t i = 0; i < m; ++i) new_samples[i] = samples[i];
        return FA_OK;
    }
    // every participant keeps at least one sample; the rest by largest remainder
    const uint64_t rest = budget - m;
    std::vector<double> frac(m);
    uint64_t given = 0;
    for (uint32_t i = 0; i < m; ++i) {
        const double q = static_cast<double>(rest) * share[i];
        const uint64_t f = static_cast<uint64_t>(std::floor(q));
        new_samples[i] = 1 + f;
        given += f;
        frac[i] = q - std::floor(q);
    }
    std::vector<uint32_t> order(m);
    for (uint32_t i = 0; i < m; ++i) order[i] = i;
    std::stable_sort(order.begin(), order.end(),
                     [&](uint32_t a, uint32_t b) { return frac[a] > frac[b]; });
    for (uint64_t k = 0; given + k < rest && k < m; ++k) new_samples[order[k]] += 1;
    return FA_OK;
}
