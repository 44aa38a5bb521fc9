/* Host implementation of the synthetic input generator described in synth.h.
 * Build with -ffp-contract=off: the block scale is a binary64 multiply followed by a binary64 add,
 * each rounded, and must not be fused. */
#include "synth.h"
#include <math.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ull

uint64_t synth_mix(uint64_t z) {
    z ^= z >> 30; z *= 0xBF58476D1CE4E5B9ull;
    z ^= z >> 27; z *= 0x94D049BB133111EBull;
    z ^= z >> 31;
    return z;
}

uint64_t synth_key(uint64_t seed, uint64_t layer, uint64_t tensor, uint64_t expert) {
    uint64_t a = synth_mix(seed + GOLDEN);
    uint64_t b = synth_mix(a + layer * GOLDEN + tensor);
    return synth_mix(b ^ ((expert + 1) * 0xC2B2AE3D27D4EB4Full));
}

uint64_t synth_rand(uint64_t key, uint64_t i) { return synth_mix(key + (i + 1) * GOLDEN); }

double synth_uniform(uint64_t key, uint64_t i) {
    return (double)(synth_rand(key, i) >> 11) * 0x1p-53;
}

double synth_normal(uint64_t key, uint64_t i) {
    double u1 = synth_uniform(key, 2 * i), u2 = synth_uniform(key, 2 * i + 1);
    return sqrt(-2.0 * log(1.0 - u1)) * cos(6.283185307179586 * u2);
}

/* Round a binary64 value to the nearest binary16 (ties to even); returns the bit pattern. */
static uint16_t to_binary16(double x) {
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isnan(x)) return 0x7E00;
    if (a >= 65520.0) return sign | 0x7C00;
    if (a < 0x1p-14) return sign | (uint16_t)nearbyint(a * 0x1p24); /* subnormal quantum 2^-24 */
    int e;
    frexp(a, &e);                                   /* a in [2^(e-1), 2^e) */
    uint32_t m = (uint32_t)nearbyint(ldexp(a, 11 - e)); /* 11-bit significand, may round to 2048 */
    int be = e - 1 + 15;
    if (m == 2048) { m = 1024; be++; }
    if (be >= 31) return sign | 0x7C00;
    return (uint16_t)(sign | (be << 10) | (m - 1024));
}

static double binary16_value(uint16_t h) {
    int be = (h >> 10) & 31, m = h & 1023;
    double v = be ? ldexp(1024.0 + m, be - 25) : ldexp((double)m, -24);
    return (h & 0x8000) ? -v : v;
}

/* Round a binary64 value to the nearest bfloat16 (ties to even); returns the bit pattern. */
static uint16_t to_bfloat16(double x) {
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isnan(x)) return 0x7FC0;
    if (a < 0x1p-126) return sign | (uint16_t)nearbyint(a * 0x1p133); /* subnormal quantum 2^-133 */
    int e;
    frexp(a, &e);
    uint32_t m = (uint32_t)nearbyint(ldexp(a, 8 - e)); /* 8-bit significand */
    int be = e - 1 + 127;
    if (m == 256) { m = 128; be++; }
    if (be >= 255) return sign | 0x7F80;
    return (uint16_t)(sign | (be << 7) | (m - 128));
}

static const int kBlockBytes[5] = {0, 0, 10, 14, 17};

int synth_blocks(int fmt, uint64_t key, int64_t first, int64_t n, uint8_t* out) {
    if (fmt < 2 || fmt > 4) return -1;
    int bb = kBlockBytes[fmt];
    for (int64_t i = 0; i < n; i++) {
        uint64_t b = (uint64_t)(first + i);
        uint8_t* p = out + i * bb;
        double t = 0.045 * synth_uniform(key, 4 * b);
        double s = 0.005 + t;
        uint16_t s16 = to_binary16(s);
        uint8_t codes[16];
        uint64_t r1 = synth_rand(key, 4 * b + 1), r2 = synth_rand(key, 4 * b + 2);
        for (int k = 0; k < 8; k++) { codes[k] = (uint8_t)(r1 >> (8 * k)); codes[8 + k] = (uint8_t)(r2 >> (8 * k)); }
        if (fmt == 4) {
            double sv = binary16_value(s16);
            int e2;
            frexp(sv, &e2);
            int fl = e2 - 1;                              /* floor(log2 s) */
            int k = (sv * sv < ldexp(1.0, 2 * fl + 1)) ? fl : fl + 1;
            p[0] = (uint8_t)(127 + k);
            memcpy(p + 1, codes, 16);
        } else {
            p[0] = (uint8_t)(s16 & 0xFF);
            p[1] = (uint8_t)(s16 >> 8);
            memcpy(p + 2, codes, (size_t)bb - 2);
        }
    }
    return 0;
}

int64_t synth_matrix(int fmt, uint64_t key, int64_t N, int64_t K, uint8_t* out) {
    if (fmt < 2 || fmt > 4 || N < 0 || K < 0 || K % 32) return -1;
    int64_t nb = N * (K / 32), bytes = nb * kBlockBytes[fmt];
    int64_t padded = (bytes + 15) / 16 * 16;
    synth_blocks(fmt, key, 0, nb, out);
    memset(out + bytes, 0, (size_t)(padded - bytes));
    return padded;
}

void synth_normal_f32(uint64_t key, int64_t first, int64_t n, double scale, float* out) {
    for (int64_t i = 0; i < n; i++) out[i] = (float)(scale * synth_normal(key, (uint64_t)(first + i)));
}

void synth_normal_bf16(uint64_t key, int64_t first, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; i++) out[i] = to_bfloat16(synth_normal(key, (uint64_t)(first + i)));
}
