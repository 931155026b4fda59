"""Oracle of the adaptive allocation controller -- TEST INFRASTRUCTURE ONLY.

Plain fp64 Python, in the order of the steps of "Technical Summary: Adaptive Data
Partitioning for Energy-Efficient Federated and Distributed Learning in
Heterogeneous Systems", section 2, "The adaptive controller":
  Measurement  t_i, e_i, n_i per participant;
  Cost         tau_i = t_i / n_i, eps_i = e_i / n_i, smoothed by an exponential
               moving average (coefficient alpha, not given on the page);
  Split        c_i = w_t tau^_i / median(tau^) + w_e eps^_i / median(eps^);
  Allocation   the fixed budget inversely proportional to c_i, unless the change
               is below a deadband (width not given on the page).
Readings where the page is silent (stated the same way in the library's header):
median of an even count = mean of the two middle values; a zero median falls back
to the mean, an all-zero column to 1; every participant keeps >= 1 sample, the rest
go by floor then largest remainder (ties to the lower index); a zero combined cost
is floored at 1e-12 of the largest.
Pinned by tests/test_partition.py (hand-worked allocations and the page's stated
properties)."""
from __future__ import annotations

import math


def _median(v):
    s = sorted(v)
    m = len(s)
    return s[m // 2] if m % 2 else 0.5 * (s[m // 2 - 1] + s[m // 2])


def _normalise(v):
    d = _median(v)
    if d == 0.0:
        d = sum(v) / len(v)
    return [1.0 if d == 0.0 else x / d for x in v]


def partition_plan(time_s, energy_j, samples, ema_tau=None, ema_eps=None, w_time=1.0,
                   w_energy=0.0, ema_alpha=0.5, deadband=0.05):
    m = len(samples)
    budget = sum(samples)
    tau, eps = [], []
    for i in range(m):
        t = time_s[i] / samples[i]
        e = energy_j[i] / samples[i]
        hist = (ema_tau is not None and ema_eps is not None and math.isfinite(ema_tau[i])
                and ema_tau[i] >= 0 and math.isfinite(ema_eps[i]) and ema_eps[i] >= 0)
        tau.append(ema_alpha * t + (1.0 - ema_alpha) * ema_tau[i] if hist else t)
        eps.append(ema_alpha * e + (1.0 - ema_alpha) * ema_eps[i] if hist else e)
    nt, ne = _normalise(tau), _normalise(eps)
    c = [w_time * nt[i] + w_energy * ne[i] for i in range(m)]
    cmax = max(c)
    inv = []
    for ci in c:
        ci = max(ci, 1e-12 * cmax)
        inv.append(1.0 / ci if ci > 0 else 1.0)
    total = sum(inv)
    share = [x / total for x in inv]
    move = any(abs(share[i] - samples[i] / budget) > deadband * (samples[i] / budget) for i in range(m))
    if not move:
        return list(samples), tau, eps
    rest = budget - m
    q = [rest * s for s in share]
    new = [1 + math.floor(x) for x in q]
    left = rest - sum(math.floor(x) for x in q)
    order = sorted(range(m), key=lambda i: (-(q[i] - math.floor(q[i])), i))
    for i in order[:left]:
        new[i] += 1
    return new, tau, eps
