/* Seeded synthetic inputs from a counter-based generator on the SplitMix64 finaliser (Steele, Lea,
 * Flood, OOPSLA 2014):
 *   mix(z): z ^= z>>30; z *= 0xBF58476D1CE4E5B9; z ^= z>>27; z *= 0x94D049BB133111EB; z ^= z>>31
 *   key = mix(mix(mix(seed+G) + layer*G + tensor) ^ (expert+1)*0xC2B2AE3D27D4EB4F)
 *   rand(key,i) = mix(key + (i+1)*G), G = 0x9E3779B97F4A7C15;  U = (rand>>11) * 2^-53
 *   N(key,i) = sqrt(-2 ln(1-U(2i))) cos(2 pi U(2i+1))
 * Packed block b: scale s = RN_binary16(0.005 + 0.045*U(4b)) (unfused binary64 ops); FP2/FP3 store s
 * in bytes 0-1, FP4 stores the E8M0 byte 127 + round(log2 s) (decided by comparing s^2 with
 * 2^(2k+1)); the code bytes are those of rand(4b+1) then rand(4b+2).
 *
 * This module only draws inputs (packed blocks with uniform codes and uniform binary16 scales,
 * normal router weights and tokens). It holds none of the decode, GEMV, routing or quantization
 * arithmetic. The host implementation (synth.c) and the device twin (synth_dev.cu) are written
 * independently from the published SplitMix64 finaliser and must produce identical bytes. */
#ifndef SYNTH_H
#define SYNTH_H
#include <stdint.h>
#ifdef __cplusplus
extern "C" {
#endif

uint64_t synth_mix(uint64_t z);
uint64_t synth_key(uint64_t seed, uint64_t layer, uint64_t tensor, uint64_t expert);
uint64_t synth_rand(uint64_t key, uint64_t i);
double synth_uniform(uint64_t key, uint64_t i);
double synth_normal(uint64_t key, uint64_t i);

/* Packed blocks b = first .. first+n-1 of a matrix keyed by `key`, written contiguously.
 * fmt is 2, 3 or 4. Returns 0, or -1 for a bad format. */
int synth_blocks(int fmt, uint64_t key, int64_t first, int64_t n, uint8_t* out);
/* A whole N x K packed matrix, pad bytes up to the 16-byte storage size set to zero.
 * Returns the number of bytes written, or -1. */
int64_t synth_matrix(int fmt, uint64_t key, int64_t N, int64_t K, uint8_t* out);
/* n values RN_binary32(scale * N(key, first + i)). */
void synth_normal_f32(uint64_t key, int64_t first, int64_t n, double scale, float* out);
/* n values RN_bfloat16(N(key, first + i)), as raw bfloat16 bit patterns. */
void synth_normal_bf16(uint64_t key, int64_t first, int64_t n, uint16_t* out);

#ifdef __cplusplus
}
#endif
#endif
