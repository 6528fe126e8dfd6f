/* Counter-based synthetic input generator, host side (plain C).
 *
 * Shared by the oracle tests and the GPU path as a pure input source; it holds
 * none of the MoE layer's arithmetic. synth_dev.cu implements the same
 * definition for the GPU; the two agree bit for bit because every step below is
 * integer arithmetic plus one IEEE fp32 multiply and one round-to-nearest-even
 * conversion to bf16.
 *
 * Definition (element i of tensor `tid` under `seed`):
 *   mix(z)   = splitmix64 finalizer: z ^= z>>30; z *= 0xBF58476D1CE4E5B9;
 *              z ^= z>>27; z *= 0x94D049BB133111EB; z ^= z>>31
 *   key      = mix((seed + 1) * 0x9E3779B97F4A7C15 + tid * 0xD1B54A32D192ED03)
 *   r        = mix(key + (i + 1) * 0x9E3779B97F4A7C15)
 *   NORMAL : n = 2*(r16_0 + r16_1 + r16_2 + r16_3) - 262140   (four 16-bit fields)
 *            -> Irwin-Hall sum of 4 uniforms, centred; unit variance after K
 *   UNIFORM: n = 2*(r >> 41) - (2^23 - 1)                       (odd, |n| < 2^23)
 *   value    = (float)n * K  (one fp32 multiply; K is an fp32 constant given by caller)
 *   bf16     = round-to-nearest-even of value's fp32 bits
 */
#include <stdint.h>
#include <string.h>

static uint64_t mix64(uint64_t z) {
    z ^= z >> 30; z *= 0xBF58476D1CE4E5B9ULL;
    z ^= z >> 27; z *= 0x94D049BB133111EBULL;
    z ^= z >> 31;
    return z;
}

static float draw(uint64_t key, uint64_t i, int dist, float K) {
    uint64_t r = mix64(key + (i + 1) * 0x9E3779B97F4A7C15ULL);
    int32_t n;
    if (dist == 0) {
        uint32_t s = (uint32_t)(r & 0xFFFF) + (uint32_t)((r >> 16) & 0xFFFF) +
                     (uint32_t)((r >> 32) & 0xFFFF) + (uint32_t)(r >> 48);
        n = 2 * (int32_t)s - 262140;
    } else {
        n = 2 * (int32_t)(r >> 41) - ((1 << 23) - 1);
    }
    volatile float prod = (float)n * K;   /* keep a single fp32 multiply */
    return prod;
}

static uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return 0x7FC0;
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

uint64_t synth_key(uint64_t seed, uint64_t tid) {
    return mix64((seed + 1) * 0x9E3779B97F4A7C15ULL + tid * 0xD1B54A32D192ED03ULL);
}

/* Elements [offset, offset + count) of the tensor, as fp32. */
void synth_fill_f32(uint64_t seed, uint64_t tid, uint64_t offset, uint64_t count,
                    int dist, float K, float* out) {
    uint64_t key = synth_key(seed, tid);
    for (uint64_t j = 0; j < count; ++j) out[j] = draw(key, offset + j, dist, K);
}

/* Same elements, rounded to bf16 (bit patterns). */
void synth_fill_bf16(uint64_t seed, uint64_t tid, uint64_t offset, uint64_t count,
                     int dist, float K, uint16_t* out) {
    uint64_t key = synth_key(seed, tid);
    for (uint64_t j = 0; j < count; ++j) out[j] = f32_to_bf16_rne(draw(key, offset + j, dist, K));
}
