/* FedAvg oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 statement of server-side weighted aggregation, used to
 * check the CUDA path.  Only the tests, the smoke check and the bench's CPU
 * baseline may load it; the product never does.  It shares no code with the
 * CUDA library.
 *
 * What it computes, per key p of a state dict (layout order):
 *   S_p = the clients that reported key p
 *   N_p = sum of n_k over S_p                       (fp64, ascending k)
 *   if S_p is empty or N_p == 0: key p is not written
 *   else for every element i:
 *       s = sum over k in S_p, ascending k, of n_k * x_k[p][i]   (fp64)
 *       y = s / N_p                                               (fp64)
 *       out[p][i] = y rounded to the output type, to nearest (ties to even)
 *
 * Sources (the pages never print the formula; this is the plain reading):
 *  - "Federated learning implemented by NVIDIA Clara" (epnc.co.kr), opening
 *    section: the server's aggregation may be the simple average of all
 *    clients or weighted by what each client contributed; clients share only
 *    part of the model weights.  "Server-side workflow": once every update
 *    is in, the server aggregates with a weighted aggregation algorithm.
 *  - "Technical Summary: Adaptive Data Partitioning for Energy-Efficient
 *    Federated and Distributed Learning in Heterogeneous Systems",
 *    section 2, "The adaptive controller", Measurement: each participant i
 *    reports its sample count n_i for the round -- the weights n_k here.
 *  - "Building Federated Multimodal AI Workflows with NVIDIA FLARE",
 *    "Coordinating training across clients": the client update contract says
 *    which components each client may update and how component-level updates
 *    are combined -- hence the per-key reporter set S_p and its own N_p.
 *  - "Accelerating LLM training with NVFP4 on NVIDIA Blackwell", list of
 *    ingredients, stochastic-rounding item: weights keep round-to-nearest-
 *    even -- hence RNE for the output cast.
 */
#include <stdint.h>
#include <string.h>
#include <math.h>

enum { FO_F32 = 0, FO_BF16 = 1, FO_F64 = 2 };

/* Decode input element i of a client tensor to fp64 (exact).  FO_F64 inputs are
 * already fp64: they let the oracle nest (a mean of means, for silos). */
static double fo_load(const void* x, int dtype, uint64_t i) {
    if (dtype == FO_F64) return ((const double*)x)[i];
    if (dtype == FO_F32) return (double)((const float*)x)[i];
    uint32_t u = (uint32_t)((const uint16_t*)x)[i] << 16; /* bf16 = top half of a binary32 */
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* Round a double to the nearest bfloat16, ties to even, from the IEEE-754
 * definition: bfloat16 has 8 significand bits (7 stored), exponent range
 * -126..127, subnormal quantum 2^-133, largest finite (2 - 2^-7) * 2^127.
 * Steps: find the bf16 quantum q at |y|, split |y|/q (exact, a power-of-two
 * scaling) into integer and fraction, pick the nearer neighbour (even on a
 * tie), and encode that exactly representable value. */
uint16_t fo_bf16_rne(double y) {
    uint16_t sign = signbit(y) ? 0x8000 : 0;
    if (isnan(y)) return (uint16_t)(sign | 0x7FC0);
    double a = fabs(y);
    if (isinf(a)) return (uint16_t)(sign | 0x7F80);
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);                  /* a = m * 2^e, m in [0.5, 1) => a in [2^(e-1), 2^e) */
    int E = e - 1;                 /* a in [2^E, 2^(E+1)) */
    if (E < -126) E = -126;        /* bf16 subnormal range shares the minimum normal quantum */
    double q = ldexp(1.0, E - 7);  /* spacing of bf16 values in this binade */
    double t = a / q;              /* exact: power-of-two scaling */
    double fl = floor(t);
    double frac = t - fl;          /* exact */
    double k;
    if (frac > 0.5) k = fl + 1.0;
    else if (frac < 0.5) k = fl;
    else k = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
    double r = k * q;              /* exact: k <= 256 */
    if (r >= 0x1p128) return (uint16_t)(sign | 0x7F80);   /* overflow to infinity */
    float rf = (float)r;           /* exact: r is a bf16 value */
    uint32_t u;
    memcpy(&u, &rf, 4);
    return (uint16_t)(sign | ((u >> 16) & 0x7FFF));
}

/* Round a double to the nearest binary32 (C conversion, round to nearest even). */
float fo_f32_rn(double y) { return (float)y; }

/* Aggregate one key.
 *   K        number of clients (client ids 0..K-1)
 *   n        n[k], the weight of client k (its sample count)
 *   reported reported[k] != 0 if client k reported this key
 *   x        x[k] points at client k's numel values (dtype_in); unused if
 *            !reported[k]
 *   out      numel values of dtype_out, written only if the key has N_p > 0
 *   N_out, cnt_out  (optional) the key's weight total and reporter count
 * Returns 1 if out was written, 0 if the key is left untouched. */
int fo_fedavg_key(uint32_t K, const double* n, const uint8_t* reported,
                  const void* const* x, int dtype_in, uint64_t numel,
                  int dtype_out, void* out, double* N_out, uint32_t* cnt_out) {
    double N = 0.0;
    uint32_t cnt = 0;
    for (uint32_t k = 0; k < K; ++k) {
        if (reported[k]) {
            N += n[k];
            cnt += 1;
        }
    }
    if (N_out) *N_out = N;
    if (cnt_out) *cnt_out = cnt;
    if (cnt == 0 || N == 0.0) return 0;
    for (uint64_t i = 0; i < numel; ++i) {
        double s = 0.0;
        for (uint32_t k = 0; k < K; ++k) {
            if (reported[k]) s += n[k] * fo_load(x[k], dtype_in, i);
        }
        double y = s / N;
        if (dtype_out == FO_F32) ((float*)out)[i] = fo_f32_rn(y);
        else ((uint16_t*)out)[i] = fo_bf16_rne(y);
    }
    return 1;
}

/* The same aggregate before the output cast: y[i] = s / N_p in fp64. */
int fo_fedavg_key_f64(uint32_t K, const double* n, const uint8_t* reported,
                      const void* const* x, int dtype_in, uint64_t numel, double* y) {
    double N = 0.0;
    uint32_t cnt = 0;
    for (uint32_t k = 0; k < K; ++k) {
        if (reported[k]) {
            N += n[k];
            cnt += 1;
        }
    }
    if (cnt == 0 || N == 0.0) return 0;
    for (uint64_t i = 0; i < numel; ++i) {
        double s = 0.0;
        for (uint32_t k = 0; k < K; ++k) {
            if (reported[k]) s += n[k] * fo_load(x[k], dtype_in, i);
        }
        y[i] = s / N;
    }
    return 1;
}

/* Vector forms of the two casts, for tests. */
void fo_bf16_rne_n(const double* y, uint64_t m, uint16_t* out) {
    for (uint64_t i = 0; i < m; ++i) out[i] = fo_bf16_rne(y[i]);
}
void fo_f32_rn_n(const double* y, uint64_t m, float* out) {
    for (uint64_t i = 0; i < m; ++i) out[i] = fo_f32_rn(y[i]);
}

/* Delta rounds: clients send updates relative to the current global model and
 * the server applies their weighted mean to it -- "Federated learning
 * implemented by NVIDIA Clara", "Server-side workflow": after aggregation the
 * server updates the existing global model as a whole and serves it in the
 * next round.  With server_lr = 1 this is plain FedAvg on deltas; other values
 * scale the mean update (a server step size; the pages fix none).
 *   base    numel values of dtype_out: the current global model for this key
 *   out[i] = round_out( base[i] + server_lr * (sum_k n_k * x_k[i]) / N_p )   (fp64)
 * Keys with no weight are left untouched, as in fo_fedavg_key. */
int fo_fedavg_apply_key(uint32_t K, const double* n, const uint8_t* reported,
                        const void* const* x, int dtype_in, uint64_t numel, const void* base,
                        double server_lr, int dtype_out, void* out, double* N_out,
                        uint32_t* cnt_out) {
    double N = 0.0;
    uint32_t cnt = 0;
    for (uint32_t k = 0; k < K; ++k) {
        if (reported[k]) {
            N += n[k];
            cnt += 1;
        }
    }
    if (N_out) *N_out = N;
    if (cnt_out) *cnt_out = cnt;
    if (cnt == 0 || N == 0.0) return 0;
    for (uint64_t i = 0; i < numel; ++i) {
        double s = 0.0;
        for (uint32_t k = 0; k < K; ++k) {
            if (reported[k]) s += n[k] * fo_load(x[k], dtype_in, i);
        }
        double y = fo_load(base, dtype_out, i) + server_lr * (s / N);
        if (dtype_out == FO_F32) ((float*)out)[i] = fo_f32_rn(y);
        else ((uint16_t*)out)[i] = fo_bf16_rne(y);
    }
    return 1;
}
