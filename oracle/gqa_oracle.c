/*
 * CPU oracle for grouped-query decode attention, in double precision.
 *
 * TEST INFRASTRUCTURE ONLY. Only the test suite, the package's smoke check and
 * the bench's CPU-baseline / reference arm may load this code. The GPU path
 * shares no code with it and never calls it.
 *
 * What it computes is the plain definition from "GQA analysis" (section
 * "Grouped broadcast"): query head h reads only KV head
 *     g(h) = floor(h / (H / G)),
 *     score[h] = softmax(Q[h] . K[g(h)]^T / sqrt(D)),
 *     O[h]     = score[h] . V[g(h)],
 * evaluated for each decode row on its own, as the per-head loop of the
 * section "Incremental decode" of the same page does. The scale is an
 * argument (1/sqrt(D) in every workload). For sq > 1 new tokens per sequence
 * the causal mask of "Same GQA, Different Execution Cost Across Backends"
 * (section 7, "mask handling") is taken bottom-right aligned: the new token s
 * sits at absolute position T_b - sq + s and sees keys t <= T_b - sq + s.
 *
 * Per row (b, s, h), with P = T_b - sq + s:
 *     x_t  = scale * sum_d q[b,s,h,d] * k[b,g,t,d]      t = 0..P
 *     mu   = max_t x_t
 *     Z    = sum_t exp(x_t - mu)
 *     out  = sum_t exp(x_t - mu) * v[b,g,t,:] / Z
 *     lse  = mu + log(Z)                                (natural log)
 * A row with no visible key (P < 0) gets out = 0 and lse = -inf.
 * K and V are read through g(h) directly; nothing is expanded. Inputs are
 * bf16 bit patterns, widened exactly to double; every sum runs in index order.
 *
 * Layouts (all C-contiguous): q [B, sq, H, D], k and v [B, G, Tmax, D],
 * seq_lens [B] (int32, host), out [B, sq, H, D] double, lse [B, sq, H] double.
 * Rows are numbered r = (b*sq + s)*H + h; only rows [row_begin, row_end) are
 * computed and written, so callers may split the work or sample single rows.
 *
 * Returns 0, or -1 for arguments outside the definition (H % G != 0, a length
 * outside [0, Tmax], non-positive sizes, a bad row range).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double bf16_bits_to_double(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int oracle_gqa_decode_f64(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                          const int32_t* seq_lens, double scale, int B, int sq, int H,
                          int G, int D, int Tmax, long row_begin, long row_end,
                          double* out, double* lse) {
    if (B <= 0 || sq <= 0 || H <= 0 || G <= 0 || D <= 0 || Tmax <= 0) return -1;
    if (H % G != 0) return -1;
    long nrows = (long)B * sq * H;
    if (row_begin < 0 || row_end > nrows || row_begin > row_end) return -1;
    for (int b = 0; b < B; ++b)
        if (seq_lens[b] < 0 || seq_lens[b] > Tmax) return -1;

    const int heads_per_group = H / G;
    double* x = (double*)malloc(sizeof(double) * (size_t)Tmax);
    if (!x) return -1;

    for (long r = row_begin; r < row_end; ++r) {
        const int h = (int)(r % H);
        const int s = (int)((r / H) % sq);
        const int b = (int)(r / ((long)H * sq));
        const int g = h / heads_per_group;
        const int T = seq_lens[b];
        const long last = (long)T - sq + s; /* last visible key index */

        const uint16_t* qrow = q + (((long)b * sq + s) * H + h) * D;
        const uint16_t* kbase = k + ((long)b * G + g) * (long)Tmax * D;
        const uint16_t* vbase = v + ((long)b * G + g) * (long)Tmax * D;
        double* orow = out + r * D;

        if (last < 0) {
            for (int d = 0; d < D; ++d) orow[d] = 0.0;
            lse[r] = -INFINITY;
            continue;
        }
        const long n = last + 1;

        double mu = -INFINITY;
        for (long t = 0; t < n; ++t) {
            double dot = 0.0;
            for (int d = 0; d < D; ++d)
                dot += bf16_bits_to_double(qrow[d]) * bf16_bits_to_double(kbase[t * D + d]);
            x[t] = scale * dot;
            if (x[t] > mu) mu = x[t];
        }

        double Z = 0.0;
        for (long t = 0; t < n; ++t) Z += exp(x[t] - mu);

        for (int d = 0; d < D; ++d) orow[d] = 0.0;
        for (long t = 0; t < n; ++t) {
            double w = exp(x[t] - mu);
            for (int d = 0; d < D; ++d) orow[d] += w * bf16_bits_to_double(vbase[t * D + d]);
        }
        for (int d = 0; d < D; ++d) orow[d] /= Z;
        lse[r] = mu + log(Z);
    }
    free(x);
    return 0;
}

/*
 * The same definition with K and V given as double values -- for caches whose
 * elements are not bf16 (the fp8 cache, dequantised by the caller as code *
 * block scale). q stays bf16 bits; k and v are [B, G, Tmax, D] double.
 */
int oracle_gqa_decode_kvf64(const uint16_t* q, const double* k, const double* v,
                            const int32_t* seq_lens, double scale, int B, int sq, int H, int G,
                            int D, int Tmax, long row_begin, long row_end, double* out,
                            double* lse) {
    if (B <= 0 || sq <= 0 || H <= 0 || G <= 0 || D <= 0 || Tmax <= 0) return -1;
    if (H % G != 0) return -1;
    long nrows = (long)B * sq * H;
    if (row_begin < 0 || row_end > nrows || row_begin > row_end) return -1;
    for (int b = 0; b < B; ++b)
        if (seq_lens[b] < 0 || seq_lens[b] > Tmax) return -1;

    const int heads_per_group = H / G;
    double* x = (double*)malloc(sizeof(double) * (size_t)Tmax);
    if (!x) return -1;

    for (long r = row_begin; r < row_end; ++r) {
        const int h = (int)(r % H);
        const int s = (int)((r / H) % sq);
        const int b = (int)(r / ((long)H * sq));
        const int g = h / heads_per_group;
        const int T = seq_lens[b];
        const long last = (long)T - sq + s; /* last visible key index */

        const uint16_t* qrow = q + (((long)b * sq + s) * H + h) * D;
        const double* kbase = k + ((long)b * G + g) * (long)Tmax * D;
        const double* vbase = v + ((long)b * G + g) * (long)Tmax * D;
        double* orow = out + r * D;

        if (last < 0) {
            for (int d = 0; d < D; ++d) orow[d] = 0.0;
            lse[r] = -INFINITY;
            continue;
        }
        const long n = last + 1;

        double mu = -INFINITY;
        for (long t = 0; t < n; ++t) {
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += bf16_bits_to_double(qrow[d]) * kbase[t * D + d];
            x[t] = scale * dot;
            if (x[t] > mu) mu = x[t];
        }

        double Z = 0.0;
        for (long t = 0; t < n; ++t) Z += exp(x[t] - mu);

        for (int d = 0; d < D; ++d) orow[d] = 0.0;
        for (long t = 0; t < n; ++t) {
            double w = exp(x[t] - mu);
            for (int d = 0; d < D; ++d) orow[d] += w * vbase[t * D + d];
        }
        for (int d = 0; d < D; ++d) orow[d] /= Z;
        lse[r] = mu + log(Z);
    }
    free(x);
    return 0;
}
