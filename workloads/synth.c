/*
 * Seeded, counter-based synthetic input generator.
 *
 * This file holds no arithmetic of the KV-cache method.  It turns a key
 * (seed, tensor, layer, batch, head) and an element index into an i.i.d.
 * N(0,1) sample, optionally multiplies it by a per-position scale (heavy-hitter
 * keys), and stores it as fp32 or bf16.  Both the CUDA path and the CPU oracle
 * receive the arrays written here; neither regenerates them.
 *
 * Generator: SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014) applied to a counter, two 53-bit uniforms
 * per pair of elements, Box-Muller transform (Box & Muller, Ann. Math. Stat.
 * 1958) to two normals.  Element 2p takes the cosine branch, 2p+1 the sine
 * branch.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static inline uint64_t splitmix64(uint64_t x) {
    x += 0x9E3779B97F4A7C15ull;
    x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
    x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
    return x ^ (x >> 31);
}

/* Stream key for one (seed, tensor, layer, batch, head). */
static uint64_t stream_key(uint64_t seed, uint32_t tensor, uint32_t layer,
                           uint32_t batch, uint32_t head) {
    uint64_t k = splitmix64(seed);
    k = splitmix64(k ^ ((uint64_t)tensor << 48));
    k = splitmix64(k ^ ((uint64_t)layer << 32));
    k = splitmix64(k ^ ((uint64_t)batch << 16));
    k = splitmix64(k ^ (uint64_t)head);
    return k;
}

/* uniform in (0, 1]: 53 random bits, never 0 so log() is finite. */
static inline double u01(uint64_t r) {
    return ((double)(r >> 11) + 1.0) * (1.0 / 9007199254740992.0);
}

/* fp32 -> bf16 bit pattern, round to nearest even (inputs are finite). */
static inline uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/*
 * Fill rows [pos0, pos0 + npos) of the stream, each row `dim` elements
 * (element index = pos * dim + c).  Row r is multiplied by row_scale[r] when
 * row_scale is non-NULL.  out_bf16 != 0 writes uint16 bf16 patterns, else
 * float32.  The product is taken in float32 before any rounding to bf16.
 */
void synth_fill(uint64_t seed, uint32_t tensor, uint32_t layer, uint32_t batch,
                uint32_t head, int64_t pos0, int64_t npos, int32_t dim,
                const float* row_scale, int32_t out_bf16, void* out) {
    uint64_t key = stream_key(seed, tensor, layer, batch, head);
    uint64_t first = (uint64_t)pos0 * (uint64_t)dim;
    uint64_t count = (uint64_t)npos * (uint64_t)dim;
    for (uint64_t i = 0; i < count;) {
        uint64_t idx = first + i;
        uint64_t pair = idx >> 1;
        uint64_t r1 = splitmix64(key ^ splitmix64(2 * pair));
        uint64_t r2 = splitmix64(key ^ splitmix64(2 * pair + 1));
        double rad = sqrt(-2.0 * log(u01(r1)));
        double th = 6.283185307179586476925286766559 * u01(r2);
        double z2[2] = {rad * cos(th), rad * sin(th)};
        for (int j = (int)(idx & 1); j < 2 && i < count; ++j, ++i) {
            float s = row_scale ? row_scale[i / (uint64_t)dim] : 1.0f;
            float x = (float)z2[j] * s;
            if (out_bf16)
                ((uint16_t*)out)[i] = f32_to_bf16_rne(x);
            else
                ((float*)out)[i] = x;
        }
    }
}

/* n uniforms in (0, 1] from the stream, element index = first + i. */
void synth_uniform(uint64_t seed, uint32_t tensor, uint32_t layer,
                   uint32_t batch, uint32_t head, int64_t first, int64_t n,
                   double* out) {
    uint64_t key = stream_key(seed, tensor, layer, batch, head);
    for (int64_t i = 0; i < n; ++i)
        out[i] = u01(splitmix64(key ^ splitmix64((uint64_t)(first + i))));
}
