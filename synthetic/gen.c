/*
 * Seeded synthetic inputs for grouped-query decode attention.
 *
 * This module only draws numbers; it holds none of the attention arithmetic.
 * Both the CPU oracle's tests and the GPU path's tests/bench take their inputs
 * from here, so that the two sides see bit-identical bf16 tensors.
 *
 * Generator (counter-based, so any slice can be regenerated on its own):
 *   key(seed, stream)   = mix64(seed + stream * GAMMA)
 *   h(seed, stream, i)  = mix64(key + (i + 1) * GAMMA)
 * where GAMMA = 0x9E3779B97F4A7C15 and mix64 is the SplitMix64 output
 * finaliser (Steele, Lea & Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014; constants as in Vigna's splitmix64.c). h(.,.,i) is
 * exactly the i-th output of a SplitMix64 stream whose state starts at key.
 *
 * Normal draws use the Box-Muller transform on counter pairs (2p, 2p+1):
 *   u1 = ((h(2p) >> 11) + 1) * 2^-53   in (0, 1]
 *   u2 =  (h(2p+1) >> 11)    * 2^-53   in [0, 1)
 *   z_even = sqrt(-2 ln u1) cos(2 pi u2),  z_odd = sqrt(-2 ln u1) sin(2 pi u2)
 * computed in double, rounded to float (round-to-nearest), then to bfloat16
 * with round-to-nearest-even on the float's bits.
 *
 * Uniform integers in [lo, hi] (both inclusive) use the high 64 bits of the
 * 128-bit product h * (hi - lo + 1) (Lemire's multiply-shift, no rejection).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GAMMA 0x9E3779B97F4A7C15ULL

static uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static uint64_t stream_key(uint64_t seed, uint64_t stream) {
    return mix64(seed + stream * GAMMA);
}

static uint64_t ctr_hash(uint64_t key, uint64_t i) {
    return mix64(key + (i + 1) * GAMMA);
}

static uint16_t float_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return 0x7FC0; /* NaN */
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

static const double TWO_PI = 6.283185307179586476925286766559;
static const double TWO_M53 = 1.1102230246251565404236316680908203125e-16; /* 2^-53 */

static double normal_at(uint64_t key, uint64_t i) {
    uint64_t p = i >> 1;
    uint64_t h1 = ctr_hash(key, 2 * p);
    uint64_t h2 = ctr_hash(key, 2 * p + 1);
    double u1 = (double)((h1 >> 11) + 1) * TWO_M53;
    double u2 = (double)(h2 >> 11) * TWO_M53;
    double r = sqrt(-2.0 * log(u1));
    double a = TWO_PI * u2;
    return (i & 1) ? r * sin(a) : r * cos(a);
}

/* Writes the draws at counter indices [first, first + n) to out[0 .. n). A pair
 * (2p, 2p+1) that lies wholly inside the range shares one Box-Muller step;
 * the values are the same as normal_at() gives one by one. */
static void fill_normal_range(uint64_t key, uint64_t first, uint64_t n, uint16_t* out) {
    uint64_t j = 0;
    if (n && (first & 1)) {
        out[0] = float_to_bf16_rne((float)normal_at(key, first));
        j = 1;
    }
    for (; j + 1 < n; j += 2) {
        uint64_t i = first + j; /* even */
        uint64_t h1 = ctr_hash(key, i);
        uint64_t h2 = ctr_hash(key, i + 1);
        double u1 = (double)((h1 >> 11) + 1) * TWO_M53;
        double u2 = (double)(h2 >> 11) * TWO_M53;
        double r = sqrt(-2.0 * log(u1));
        double a = TWO_PI * u2;
        out[j] = float_to_bf16_rne((float)(r * cos(a)));
        out[j + 1] = float_to_bf16_rne((float)(r * sin(a)));
    }
    if (j < n) out[j] = float_to_bf16_rne((float)normal_at(key, first + j));
}

/* out[j] = bf16 bits of the normal draw at counter index first + j. */
void synth_normal_bf16(uint64_t seed, uint64_t stream, uint64_t first, uint64_t n,
                       uint16_t* out) {
    fill_normal_range(stream_key(seed, stream), first, n, out);
}

/* out[j] = uniform integer in [lo, hi] at counter index first + j. */
void synth_uniform_int(uint64_t seed, uint64_t stream, uint64_t first, uint64_t n,
                       int64_t lo, int64_t hi, int32_t* out) {
    uint64_t key = stream_key(seed, stream);
    uint64_t span = (uint64_t)(hi - lo) + 1u;
    for (uint64_t j = 0; j < n; ++j) {
        uint64_t h = ctr_hash(key, first + j);
        uint64_t r = (uint64_t)(((unsigned __int128)h * span) >> 64);
        out[j] = (int32_t)(lo + (int64_t)r);
    }
}

/*
 * Fills batches [b_begin, b_end) of a [B, G, Tmax, D] cache. Element
 * (b, g, t, d) with t < seq_lens[b] is the normal draw at counter index
 * ((b*G + g)*Tmax + t)*D + d; entries with t >= seq_lens[b] get tail_bits.
 * `out` points at element (0,0,0,0) of the full cache.
 */
void synth_fill_cache(uint64_t seed, uint64_t stream, int B, int G, int Tmax, int D,
                      const int32_t* seq_lens, uint16_t tail_bits, int b_begin, int b_end,
                      uint16_t* out) {
    (void)B;
    uint64_t key = stream_key(seed, stream);
    for (int b = b_begin; b < b_end; ++b) {
        int tb = seq_lens[b];
        if (tb < 0) tb = 0;
        if (tb > Tmax) tb = Tmax;
        for (int g = 0; g < G; ++g) {
            uint64_t base = ((uint64_t)b * G + g) * (uint64_t)Tmax * D;
            uint64_t nvalid = (uint64_t)tb * D;
            uint64_t ntot = (uint64_t)Tmax * D;
            fill_normal_range(key, base, nvalid, out + base);
            for (uint64_t j = nvalid; j < ntot; ++j) out[base + j] = tail_bits;
        }
    }
}
