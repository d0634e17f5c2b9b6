/*
 * synth.c -- seeded synthetic inputs shared by the oracle and the CUDA path.
 *
 * This module holds no attention arithmetic. It turns (seed, tensor tag, flat element
 * index) into a bf16 bit pattern, so that any element can be regenerated on its own
 * (the oracle's sampled rows and the GPU upload see identical bits).
 *
 *   word(i, j) = splitmix64(splitmix64(seed ^ (tag << 56)) ^ (2*i + j)),  j in {0, 1}
 *   u1 = (top 53 bits of word(i,0) + 0.5) * 2^-53          in (0, 1)
 *   u2 =  top 53 bits of word(i,1)        * 2^-53          in [0, 1)
 *   z  = sqrt(-2 ln u1) * cos(2 pi u2)                      Box-Muller, one normal per i
 *   x  = mult * z, rounded double -> fp32 (RNE) -> bf16 (RNE)
 *
 * SplitMix64 is the finaliser of Steele, Lea and Flood, "Fast splittable pseudorandom
 * number generators" (OOPSLA 2014), with its published constants. Box-Muller is the
 * textbook transform (Box and Muller, 1958).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static uint64_t splitmix64(uint64_t x) {
    x += 0x9E3779B97F4A7C15ull;
    x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
    x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
    return x ^ (x >> 31);
}

static uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

static const double kTwoPi = 6.283185307179586476925286766559;

/* One element: the normal deviate for flat index i, scaled and rounded to bf16 bits. */
uint16_t synth_normal_bf16_one(uint64_t seed, uint32_t tag, uint64_t i, double mult) {
    uint64_t key = splitmix64(seed ^ ((uint64_t)tag << 56));
    uint64_t w0 = splitmix64(key ^ (2 * i));
    uint64_t w1 = splitmix64(key ^ (2 * i + 1));
    double u1 = ((double)(w0 >> 11) + 0.5) * 0x1.0p-53;
    double u2 = (double)(w1 >> 11) * 0x1.0p-53;
    double z = sqrt(-2.0 * log(u1)) * cos(kTwoPi * u2);
    return f32_to_bf16_rne((float)(mult * z));
}

/* Fill out[0..count) with elements offset..offset+count-1 of tensor (seed, tag). */
void synth_normal_bf16(uint64_t seed, uint32_t tag, uint64_t offset, uint64_t count, double mult,
                       uint16_t* out) {
    long long n = (long long)count;
#pragma omp parallel for schedule(static)
    for (long long j = 0; j < n; ++j) out[j] = synth_normal_bf16_one(seed, tag, offset + (uint64_t)j, mult);
}

/* Raw SplitMix64 word, exported so a test can check the generator against its definition. */
uint64_t synth_splitmix64(uint64_t x) { return splitmix64(x); }
