/* CPU oracle for the low-bit MoE decode/verify path. TEST INFRASTRUCTURE ONLY: see oracle.h for who
 * may call it. binary64, naive loops, OpenMP only over independent output rows (deterministic).
 *
 * Block layouts (a reading: the pages give only the sizes, 32 weights per block, FP2 = 10 bytes,
 * FP3 = 3.50 and FP4 = 4.25 bits per weight, with one or two small scales; "DeepSeek V4 Flash hits
 * 32 tok/s on AMD Ryzen AI MAX+ 395", the ROCmFPX paragraph). Little-endian throughout.
 *   FP2 (10 B): bytes 0-1 binary16 scale d; code c_j = bits 2j..2j+1 of bytes 2-9; w = d(2c-3).
 *   FP3 (14 B): bytes 0-1 binary16 d; low bits l_j = bits 2j..2j+1 of bytes 2-9; high bit
 *               h_j = bit j of bytes 10-13; c = l + 4h; w = d(2c-7).
 *   FP4 (17 B): byte 0 E8M0 exponent e (255 invalid), scale 2^(e-127); code q_j = bits 4j..4j+3
 *               of bytes 1-16, E2M1: sign bit 3, magnitude {0,.5,1,1.5,2,3,4,6}[q & 7].
 * A matrix is row-major, K/32 blocks per row, stored in N*K/32*B bytes rounded up to 16. */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static const double kE2M1[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

int orc_block_bytes(int fmt) { return fmt == 2 ? 10 : fmt == 3 ? 14 : fmt == 4 ? 17 : 0; }

int64_t orc_matrix_bytes(int fmt, int64_t N, int64_t K) {
    int bb = orc_block_bytes(fmt);
    if (!bb || N < 0 || K < 0 || K % 32) return -1;
    int64_t bytes = N * (K / 32) * bb;
    return (bytes + 15) / 16 * 16;
}

int orc_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Sets the number of OpenMP threads later calls use (n >= 1); returns the previous number. */
int orc_set_threads(int n) {
    int prev = orc_threads();
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
    return prev;
}

/* Value of a binary16 bit pattern (exact in binary64). */
static double binary16_to_double(unsigned h) {
    unsigned ex = (h >> 10) & 31, man = h & 1023;
    double v;
    if (ex == 31) v = man ? NAN : INFINITY;
    else if (ex == 0) v = ldexp((double)man, -24);
    else v = ldexp((double)(1024 + man), (int)ex - 25);
    return (h & 0x8000) ? -v : v;
}

/* Nearest binary16 to x, ties to even significand; returns the bit pattern. */
static unsigned double_to_binary16(double x) {
    unsigned sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs(x);
    if (isnan(x)) return 0x7E00u;
    /* Largest finite binary16 is 65504 (significand 2047 * 2^5); halfway to 2^16 is 65520. */
    if (a >= 65520.0) return sign | 0x7C00u;
    if (a < ldexp(1.0, -14)) return sign | (unsigned)nearbyint(ldexp(a, 24));
    int e;
    frexp(a, &e);                        /* a in [2^(e-1), 2^e) */
    double sig = nearbyint(ldexp(a, 11 - e)); /* integer significand in [1024, 2048] */
    int ex = e - 1 + 15;
    if (sig == 2048.0) { sig = 1024.0; ex++; }
    if (ex >= 31) return sign | 0x7C00u;
    return sign | ((unsigned)ex << 10) | ((unsigned)sig - 1024u);
}

/* Nearest bfloat16 value to x (ties to even significand), returned as a binary64 value. */
static double round_to_bfloat16(double x) {
    if (x == 0.0 || isnan(x) || isinf(x)) return x;
    double a = fabs(x);
    double r;
    if (a < ldexp(1.0, -126)) {
        r = ldexp(nearbyint(ldexp(a, 133)), -133); /* subnormal quantum 2^-133 */
    } else {
        int e;
        frexp(a, &e);
        r = ldexp(nearbyint(ldexp(a, 8 - e)), e - 8); /* 8-bit significand */
        if (r >= ldexp(1.0, 128)) r = INFINITY; /* beyond the largest bfloat16, 255 * 2^120 */
    }
    return x < 0 ? -r : r;
}

int orc_decode_block(int fmt, const uint8_t* blk, double* w) {
    if (fmt == 2) {
        double d = binary16_to_double((unsigned)blk[0] | ((unsigned)blk[1] << 8));
        for (int j = 0; j < 32; j++) {
            int c = (blk[2 + j / 4] >> (2 * (j % 4))) & 3;
            w[j] = d * (2 * c - 3);
        }
        return ORC_OK;
    }
    if (fmt == 3) {
        double d = binary16_to_double((unsigned)blk[0] | ((unsigned)blk[1] << 8));
        for (int j = 0; j < 32; j++) {
            int lo = (blk[2 + j / 4] >> (2 * (j % 4))) & 3;
            int hi = (blk[10 + j / 8] >> (j % 8)) & 1;
            w[j] = d * (2 * (lo + 4 * hi) - 7);
        }
        return ORC_OK;
    }
    if (fmt == 4) {
        if (blk[0] == 255) return ORC_EDATA;
        double s = ldexp(1.0, (int)blk[0] - 127);
        for (int j = 0; j < 32; j++) {
            int qc = (blk[1 + j / 2] >> (4 * (j % 2))) & 15;
            double v = s * kE2M1[qc & 7];
            w[j] = (qc & 8) ? -v : v;
        }
        return ORC_OK;
    }
    return ORC_EINVAL;
}

int orc_dequantize(int fmt, const uint8_t* Wq, int64_t N, int64_t K, double* W) {
    int bb = orc_block_bytes(fmt);
    if (!bb || N < 0 || K < 0 || K % 32) return ORC_EINVAL;
    int64_t nb = K / 32;
    int status = ORC_OK;
    for (int64_t r = 0; r < N; r++)
        for (int64_t b = 0; b < nb; b++) {
            int st = orc_decode_block(fmt, Wq + (r * nb + b) * bb, W + r * K + b * 32);
            if (st) status = st;
        }
    return status;
}

/* Decodes row r of a packed matrix into row[K]. */
static int decode_row(int fmt, const uint8_t* Wq, int64_t K, int64_t r, double* row) {
    int bb = orc_block_bytes(fmt);
    int64_t nb = K / 32;
    int status = ORC_OK;
    for (int64_t b = 0; b < nb; b++) {
        int st = orc_decode_block(fmt, Wq + (r * nb + b) * bb, row + b * 32);
        if (st) status = st;
    }
    return status;
}

int orc_gemv(int fmt, const uint8_t* Wq, int64_t N, int64_t K, const double* x, int q, double* y,
             double* M) {
    if (!orc_block_bytes(fmt) || N < 0 || K < 0 || K % 32 || q < 1) return ORC_EINVAL;
    int status = ORC_OK;
#pragma omp parallel
    {
        double* row = (double*)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
#pragma omp for schedule(static)
        for (int64_t n = 0; n < N; n++) {
            int st = decode_row(fmt, Wq, K, n, row); /* each row decoded once, used by all q */
            if (st) {
#pragma omp critical
                status = st;
            }
            for (int t = 0; t < q; t++) {
                double acc = 0.0, mag = 0.0;
                for (int64_t k = 0; k < K; k++) {
                    double p = row[k] * x[(int64_t)t * K + k];
                    acc += p;
                    mag += fabs(p);
                }
                y[(int64_t)t * N + n] = acc;
                if (M) M[(int64_t)t * N + n] = mag;
            }
        }
        free(row);
    }
    return status;
}

/* FP2/FP3 code for value v with binary16 scale d (as double), Kmax = 3 or 7: sign from signbit,
 * magnitude index = number of midpoints 2d, 4d, ... strictly below |v| (ties to the smaller level). */
static int odd_level_code(double v, double d, int kmax) {
    double a = fabs(v);
    int i = 0;
    for (int m = 1; m <= kmax / 2; m++)
        if (a > 2.0 * m * d) i = m;
    int half = (kmax + 1) / 2; /* 2 for FP2, 4 for FP3 */
    return signbit(v) ? half - 1 - i : half + i;
}

/* E2M1 magnitude index for t >= 0: nearest grid value, ties to the even significand bit (the code's
 * lowest bit), saturating at 6. */
static int e2m1_index(double t) {
    if (t >= 6.0) return 7;
    int m = 0;
    while (m < 7 && kE2M1[m + 1] <= t) m++;
    if (m == 7) return 7;
    double mid = 0.5 * (kE2M1[m] + kE2M1[m + 1]);
    if (t < mid) return m;
    if (t > mid) return m + 1;
    return (m % 2 == 0) ? m : m + 1;
}

int orc_quantize(int fmt, const float* W, int64_t N, int64_t K, const float* scales, uint8_t* out) {
    int bb = orc_block_bytes(fmt);
    if (!bb || N < 0 || K < 0 || K % 32) return ORC_EINVAL;
    int64_t nb = K / 32;
    for (int64_t r = 0; r < N; r++) {
        for (int64_t b = 0; b < nb; b++) {
            const float* v = W + r * K + b * 32;
            uint8_t* p = out + (r * nb + b) * bb;
            double amax = 0.0;
            for (int j = 0; j < 32; j++) {
                if (!isfinite(v[j])) return ORC_ERANGE;
                if (fabs((double)v[j]) > amax) amax = fabs((double)v[j]);
            }
            if (fmt == 2 || fmt == 3) {
                int kmax = fmt == 2 ? 3 : 7;
                unsigned d16;
                if (scales) {
                    double s = (double)scales[r * nb + b];
                    if (!(s >= 0.0) || isinf(s)) return ORC_EINVAL;
                    d16 = double_to_binary16(s);
                } else {
                    d16 = double_to_binary16(amax / kmax);
                }
                if ((d16 & 0x7C00u) == 0x7C00u) return ORC_ERANGE;
                double d = binary16_to_double(d16);
                memset(p, 0, (size_t)bb);
                p[0] = (uint8_t)(d16 & 0xFF);
                p[1] = (uint8_t)(d16 >> 8);
                for (int j = 0; j < 32; j++) {
                    int c = odd_level_code((double)v[j], d, kmax);
                    p[2 + j / 4] |= (uint8_t)((c & 3) << (2 * (j % 4)));
                    if (fmt == 3) p[10 + j / 8] |= (uint8_t)(((c >> 2) & 1) << (j % 8));
                }
            } else {
                int e;
                if (scales) {
                    double s = (double)scales[r * nb + b];
                    int ex;
                    if (!(s > 0.0) || isinf(s) || frexp(s, &ex) != 0.5) return ORC_EINVAL;
                    e = ex - 1 + 127; /* s = 2^(ex-1) */
                    if (e < 0 || e > 254) return ORC_EINVAL;
                } else if (amax == 0.0) {
                    e = 0;
                } else {
                    int ex;
                    frexp(amax, &ex); /* floor(log2 amax) = ex - 1 */
                    e = ex - 1 - 2 + 127;
                    if (e < 0) e = 0;
                    if (e > 254) e = 254;
                }
                double scale = ldexp(1.0, e - 127);
                memset(p, 0, (size_t)bb);
                p[0] = (uint8_t)e;
                for (int j = 0; j < 32; j++) {
                    int m = e2m1_index(fabs((double)v[j]) / scale);
                    int qc = m | (signbit(v[j]) ? 8 : 0);
                    p[1 + j / 2] |= (uint8_t)(qc << (4 * (j % 2)));
                }
            }
        }
    }
    return ORC_OK;
}

/* One block under one candidate scale: its bytes (as orc_quantize writes them) and its weighted
 * squared error in binary64, summed in weight order. d16 / e: the binary16 scale or E8M0 exponent. */
static double weighted_block(int fmt, const float* v, const float* imp, unsigned d16, int e, uint8_t* p) {
    int bb = orc_block_bytes(fmt);
    memset(p, 0, (size_t)bb);
    double err = 0.0;
    if (fmt == 2 || fmt == 3) {
        int kmax = fmt == 2 ? 3 : 7;
        double d = binary16_to_double(d16);
        p[0] = (uint8_t)(d16 & 0xFF);
        p[1] = (uint8_t)(d16 >> 8);
        for (int j = 0; j < 32; j++) {
            int c = odd_level_code((double)v[j], d, kmax);
            p[2 + j / 4] |= (uint8_t)((c & 3) << (2 * (j % 4)));
            if (fmt == 3) p[10 + j / 8] |= (uint8_t)(((c >> 2) & 1) << (j % 8));
            double diff = (double)v[j] - d * (double)(2 * c - kmax);
            err += (imp ? (double)imp[j] : 1.0) * (diff * diff);
        }
    } else {
        double scale = ldexp(1.0, e - 127);
        p[0] = (uint8_t)e;
        for (int j = 0; j < 32; j++) {
            int m = e2m1_index(fabs((double)v[j]) / scale);
            int qc = m | (signbit(v[j]) ? 8 : 0);
            p[1 + j / 2] |= (uint8_t)(qc << (4 * (j % 2)));
            double w = (signbit(v[j]) ? -kE2M1[m] : kE2M1[m]) * scale;
            double diff = (double)v[j] - w;
            err += (imp ? (double)imp[j] : 1.0) * (diff * diff);
        }
    }
    return err;
}

int orc_quantize_weighted(int fmt, const float* W, int64_t N, int64_t K, const float* imp, uint8_t* out) {
    int bb = orc_block_bytes(fmt);
    if (!bb || N < 0 || K < 0 || K % 32) return ORC_EINVAL;
    if (imp)
        for (int64_t k = 0; k < K; k++)
            if (!isfinite(imp[k]) || imp[k] < 0.0f) return ORC_ERANGE;
    int64_t nb = K / 32;
    uint8_t cand[17];
    for (int64_t r = 0; r < N; r++) {
        for (int64_t b = 0; b < nb; b++) {
            const float* v = W + r * K + b * 32;
            const float* im = imp ? imp + b * 32 : NULL;
            uint8_t* p = out + (r * nb + b) * bb;
            double amax = 0.0;
            for (int j = 0; j < 32; j++) {
                if (!isfinite(v[j])) return ORC_ERANGE;
                if (fabs((double)v[j]) > amax) amax = fabs((double)v[j]);
            }
            double best = 0.0;
            int found = 0;
            if (fmt == 2 || fmt == 3) {
                int kmax = fmt == 2 ? 3 : 7;
                for (int j = 0; j < 16; j++) {
                    unsigned d16 = double_to_binary16(amax / kmax * ((double)(12 + j) / 20.0));
                    if ((d16 & 0x7C00u) == 0x7C00u) continue; /* overflows binary16 */
                    double err = weighted_block(fmt, v, im, d16, 0, cand);
                    if (!found || err < best) { best = err; found = 1; memcpy(p, cand, (size_t)bb); }
                }
            } else {
                int e0;
                if (amax == 0.0) {
                    e0 = 0;
                } else {
                    int ex;
                    frexp(amax, &ex);
                    e0 = ex - 1 - 2 + 127;
                    if (e0 < 0) e0 = 0;
                    if (e0 > 254) e0 = 254;
                }
                for (int j = -1; j <= 1; j++) {
                    int e = e0 + j < 0 ? 0 : (e0 + j > 254 ? 254 : e0 + j);
                    double err = weighted_block(fmt, v, im, 0, e, cand);
                    if (!found || err < best) { best = err; found = 1; memcpy(p, cand, (size_t)bb); }
                }
            }
            if (!found) return ORC_ERANGE;
        }
    }
    return ORC_OK;
}

int orc_topk(const double* v, int n, int k, int32_t* idx) {
    if (n < 1 || k < 1 || k > n) return ORC_EINVAL;
    char* taken = (char*)calloc((size_t)n, 1);
    for (int r = 0; r < k; r++) {
        int best = -1;
        for (int i = 0; i < n; i++) {
            if (taken[i]) continue;
            if (best < 0 || v[i] > v[best]) best = i; /* strict: equal values keep the lower index */
        }
        taken[best] = 1;
        idx[r] = best;
    }
    free(taken);
    return ORC_OK;
}

static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

int orc_route(const float* R, int E, int H, const double* x, int q, int k, double* logits,
              double* Ml, int32_t* idx, double* w, int32_t* uni, int32_t* n_uni) {
    if (E < 1 || H < 1 || q < 1 || k < 1 || k > E || !idx) return ORC_EINVAL;
    double* l = (double*)malloc(sizeof(double) * (size_t)E);
    char* used = (char*)calloc((size_t)E, 1);
    for (int t = 0; t < q; t++) {
        for (int e = 0; e < E; e++) {
            double acc = 0.0, mag = 0.0;
            for (int h = 0; h < H; h++) {
                double p = (double)R[(int64_t)e * H + h] * x[(int64_t)t * H + h];
                acc += p;
                mag += fabs(p);
            }
            l[e] = acc;
            if (logits) logits[(int64_t)t * E + e] = acc;
            if (Ml) Ml[(int64_t)t * E + e] = mag;
        }
        orc_topk(l, E, k, idx + (int64_t)t * k);
        double ssum = 0.0;
        for (int r = 0; r < k; r++) ssum += sigmoid(l[idx[(int64_t)t * k + r]]);
        for (int r = 0; r < k; r++) {
            if (w) w[(int64_t)t * k + r] = sigmoid(l[idx[(int64_t)t * k + r]]) / ssum;
            used[idx[(int64_t)t * k + r]] = 1;
        }
    }
    int n = 0;
    for (int e = 0; e < E; e++)
        if (used[e]) {
            if (uni) uni[n] = e;
            n++;
        }
    if (n_uni) *n_uni = n;
    free(l);
    free(used);
    return ORC_OK;
}

/* One expert applied to nt tokens (rows of X, stride H): g = G x, u = U x, h = silu(g) u, y = D h.
 * Also the first-order error magnitudes: Mg = sum |G x|, Mu = sum |U x| (the gate and up GEMVs' own
 * allowances), Mh = |silu'(g) u| Mg + |silu(g)| Mu + |h|, My_i = sum_j |D_ij| Mh_j: the gate and up
 * allowances carried through h, plus the down GEMV's own allowance sum_j |D_ij h_j| (the |h| term).
 * Writes Y[nt][H] and MY[nt][H]. */
static int expert_apply(int fg, int fd, const uint8_t* G, const uint8_t* U, const uint8_t* D, int H,
                        int I, const double* X, int nt, double* Y, double* MY) {
    double* g = (double*)calloc((size_t)nt * I, sizeof(double));
    double* u = (double*)calloc((size_t)nt * I, sizeof(double));
    double* mg = (double*)calloc((size_t)nt * I, sizeof(double));
    double* mu = (double*)calloc((size_t)nt * I, sizeof(double));
    int status = ORC_OK;
    if (orc_gemv(fg, G, I, H, X, nt, g, mg)) status = ORC_EDATA;
    if (orc_gemv(fg, U, I, H, X, nt, u, mu)) status = ORC_EDATA;
    double* hh = (double*)malloc(sizeof(double) * (size_t)nt * I);
    double* mh = (double*)malloc(sizeof(double) * (size_t)nt * I);
    for (int64_t i = 0; i < (int64_t)nt * I; i++) {
        double s = sigmoid(g[i]);
        double silu = g[i] * s, dsilu = s * (1.0 + g[i] * (1.0 - s));
        hh[i] = silu * u[i];
        mh[i] = fabs(dsilu * u[i]) * mg[i] + fabs(silu) * mu[i] + fabs(hh[i]);
    }
    /* y = D h; the magnitude uses |D| against Mh, so decode D directly rather than via orc_gemv. */
#pragma omp parallel
    {
        double* row = (double*)malloc(sizeof(double) * (size_t)I);
#pragma omp for schedule(static)
        for (int i = 0; i < H; i++) {
            if (decode_row(fd, D, I, i, row)) {
#pragma omp critical
                status = ORC_EDATA;
            }
            for (int t = 0; t < nt; t++) {
                double acc = 0.0, mag = 0.0;
                for (int j = 0; j < I; j++) {
                    acc += row[j] * hh[(int64_t)t * I + j];
                    mag += fabs(row[j]) * mh[(int64_t)t * I + j];
                }
                Y[(int64_t)t * H + i] = acc;
                MY[(int64_t)t * H + i] = mag;
            }
        }
        free(row);
    }
    free(g); free(u); free(mg); free(mu); free(hh); free(mh);
    return status;
}

/* The layer: route, run every selected expert once for all tokens that chose it and the shared
 * expert for all tokens, then combine out[t] = sum_r w[t][r] y_{e(t,r)}[t] + y_shared[t] (rank order,
 * shared last).
 * Tolerance magnitude M[t][i]: the largest first-order change of out[t][i] when every GEMV output of
 * the layer (logits, gate, up and down rows, routed and shared) is off by up to its own
 * 2e-3 * sum|w x| allowance, each with its worst sign:
 *   M = sum_r w_r My_r,i + sum_r s'_r Ml_r |y_r,i - ybar_i| / S + My_shared,i,
 * with s = sigmoid(logit), s' = s (1 - s), S = sum_r s_r, ybar_i = sum_r w_r y_r,i (a logit error
 * dl_r moves out by s'_r (y_r - ybar) dl_r / S, since dw_j/dl_r = s'_r (delta_jr - w_j) / S) and My the
 * expert's magnitude from expert_apply. */
int orc_moe_layer(int H, int I, int E, const float* R, const uint8_t* const* gate,
                  const uint8_t* const* up, const uint8_t* const* down, const uint8_t* sh_gate,
                  const uint8_t* sh_up, const uint8_t* sh_down, const double* x, int q, int k,
                  const int32_t* idx_force, double* y, double* M, int32_t* idx_out, double* w_out,
                  double* logits_out) {
    if (H < 32 || I < 32 || H % 32 || I % 32 || E < 1 || q < 1 || k < 1 || k > E) return ORC_EINVAL;
    int status = ORC_OK;
    double* logits = (double*)malloc(sizeof(double) * (size_t)q * E);
    double* ml = (double*)malloc(sizeof(double) * (size_t)q * E);
    int32_t* idx = (int32_t*)malloc(sizeof(int32_t) * (size_t)q * k);
    double* w = (double*)malloc(sizeof(double) * (size_t)q * k);
    double* mw = (double*)malloc(sizeof(double) * (size_t)q * k);
    orc_route(R, E, H, x, q, k, logits, ml, idx, w, NULL, NULL);
    if (idx_force) {
        memcpy(idx, idx_force, sizeof(int32_t) * (size_t)q * k);
        for (int t = 0; t < q; t++) {
            double ssum = 0.0;
            for (int r = 0; r < k; r++) {
                int e = idx[t * k + r];
                if (e < 0 || e >= E) { status = ORC_EINVAL; goto done; }
                ssum += sigmoid(logits[(int64_t)t * E + e]);
            }
            for (int r = 0; r < k; r++) w[t * k + r] = sigmoid(logits[(int64_t)t * E + idx[t * k + r]]) / ssum;
        }
    }
    for (int t = 0; t < q; t++) {
        /* mw[t][r] = s'_r Ml_r / S: the output's sensitivity to logit r's allowance, per unit of
         * |y_r - ybar| */
        double S = 0.0;
        for (int r = 0; r < k; r++) S += sigmoid(logits[(int64_t)t * E + idx[t * k + r]]);
        for (int r = 0; r < k; r++) {
            int e = idx[t * k + r];
            double s = sigmoid(logits[(int64_t)t * E + e]);
            mw[t * k + r] = s * (1.0 - s) * ml[(int64_t)t * E + e] / S;
        }
    }
    {
        /* per (token, rank) expert outputs */
        double* yr = (double*)calloc((size_t)q * k * H, sizeof(double));
        double* myr = (double*)calloc((size_t)q * k * H, sizeof(double));
        int32_t* toks = (int32_t*)malloc(sizeof(int32_t) * (size_t)q * k);
        int32_t* ranks = (int32_t*)malloc(sizeof(int32_t) * (size_t)q * k);
        double* X = (double*)malloc(sizeof(double) * (size_t)q * k * H);
        double* Y = (double*)malloc(sizeof(double) * (size_t)q * k * H);
        double* MY = (double*)malloc(sizeof(double) * (size_t)q * k * H);
        for (int e = 0; e < E; e++) {
            int nt = 0;
            for (int t = 0; t < q; t++)
                for (int r = 0; r < k; r++)
                    if (idx[t * k + r] == e) { toks[nt] = t; ranks[nt] = r; nt++; }
            if (!nt) continue;
            if (!gate[e] || !up[e] || !down[e]) { status = ORC_EINVAL; break; }
            for (int n = 0; n < nt; n++) memcpy(X + (int64_t)n * H, x + (int64_t)toks[n] * H, sizeof(double) * (size_t)H);
            if (expert_apply(2, 3, gate[e], up[e], down[e], H, I, X, nt, Y, MY)) status = ORC_EDATA;
            for (int n = 0; n < nt; n++) {
                int64_t o = ((int64_t)toks[n] * k + ranks[n]) * H;
                memcpy(yr + o, Y + (int64_t)n * H, sizeof(double) * (size_t)H);
                memcpy(myr + o, MY + (int64_t)n * H, sizeof(double) * (size_t)H);
            }
        }
        double* ys = (double*)malloc(sizeof(double) * (size_t)q * H);
        double* mys = (double*)malloc(sizeof(double) * (size_t)q * H);
        if (status == ORC_OK && expert_apply(4, 4, sh_gate, sh_up, sh_down, H, I, x, q, ys, mys)) status = ORC_EDATA;
        for (int t = 0; t < q; t++)
            for (int i = 0; i < H; i++) {
                double acc = 0.0, mag = 0.0;
                for (int r = 0; r < k; r++) {
                    int64_t o = ((int64_t)t * k + r) * H + i;
                    acc += w[t * k + r] * yr[o];
                    mag += w[t * k + r] * myr[o];
                }
                for (int r = 0; r < k; r++)  /* acc = ybar here */
                    mag += fabs(yr[((int64_t)t * k + r) * H + i] - acc) * mw[t * k + r];
                y[(int64_t)t * H + i] = acc + ys[(int64_t)t * H + i];
                if (M) M[(int64_t)t * H + i] = mag + mys[(int64_t)t * H + i];
            }
        free(yr); free(myr); free(toks); free(ranks); free(X); free(Y); free(MY); free(ys); free(mys);
    }
    if (idx_out) memcpy(idx_out, idx, sizeof(int32_t) * (size_t)q * k);
    if (w_out) memcpy(w_out, w, sizeof(double) * (size_t)q * k);
    if (logits_out) memcpy(logits_out, logits, sizeof(double) * (size_t)q * E);
done:
    free(logits); free(ml); free(idx); free(w); free(mw);
    return status;
}

int orc_rmsnorm_bf16(const float* r, int q, int H, double* u) {
    if (q < 1 || H < 1) return ORC_EINVAL;
    for (int t = 0; t < q; t++) {
        double ss = 0.0;
        for (int h = 0; h < H; h++) ss += (double)r[(int64_t)t * H + h] * r[(int64_t)t * H + h];
        double inv = 1.0 / sqrt(ss / H + 1e-6);
        for (int h = 0; h < H; h++) u[(int64_t)t * H + h] = round_to_bfloat16(r[(int64_t)t * H + h] * inv);
    }
    return ORC_OK;
}

typedef struct { int32_t key, pos; } keypos;

static int cmp_keypos(const void* a, const void* b) {
    const keypos* x = (const keypos*)a;
    const keypos* y = (const keypos*)b;
    if (x->key != y->key) return x->key < y->key ? -1 : 1;
    return x->pos < y->pos ? -1 : (x->pos > y->pos);
}

int orc_stable_argsort(const int32_t* keys, int n, int nkeys, int32_t* perm, int32_t* offsets) {
    if (n < 0 || nkeys < 1) return ORC_EINVAL;
    keypos* kp = (keypos*)malloc(sizeof(keypos) * (size_t)(n > 0 ? n : 1));
    for (int i = 0; i < n; i++) {
        if (keys[i] < 0 || keys[i] >= nkeys) { free(kp); return ORC_EINVAL; }
        kp[i].key = keys[i];
        kp[i].pos = i;
    }
    qsort(kp, (size_t)n, sizeof(keypos), cmp_keypos); /* (key, position) order is the stable order */
    for (int i = 0; i < n; i++) perm[i] = kp[i].pos;
    for (int e = 0; e <= nkeys; e++) {
        int c = 0;
        for (int i = 0; i < n; i++) c += keys[i] < e;
        offsets[e] = c;
    }
    free(kp);
    return ORC_OK;
}


/* ------------------------------------------------------------------ speculative verify / commit */

/* The target's choice at each verified position is its largest logit (plain scan, lowest index kept
 * on ties, NaN skipped); drafts are accepted while they equal those choices; the first mismatch (or
 * the position after the last draft) takes the target's choice. */
int orc_dspark_commit(const float* logits, int q, int V, const int32_t* drafts, int32_t* pred, int32_t* n_accept,
                      int32_t* committed) {
    if (!logits || q < 1 || V < 1 || (q > 1 && !drafts) || !pred || !n_accept || !committed) return ORC_EINVAL;
    int st = ORC_OK;
    for (int i = 0; i < q; i++) {
        int best = -1;
        for (int v = 0; v < V; v++) {
            const float x = logits[(size_t)i * V + v];
            if (x != x) continue;
            if (best < 0 || x > logits[(size_t)i * V + best]) best = v;
        }
        if (best < 0) { best = 0; st = ORC_ERANGE; }
        pred[i] = best;
    }
    int n = 0;
    while (n < q - 1 && drafts[n] == pred[n]) n++;
    *n_accept = n;
    for (int i = 0; i < q; i++) committed[i] = i < n ? drafts[i] : (i == n ? pred[n] : -1);
    return st;
}

/* Integer-dot activations: per (column, 32-entry block), the exponent e of the largest magnitude
 * (2^(e-1) <= a < 2^e, from frexp) and X = nearest integer to x * 2^(14-e), ties to even (nearbyint
 * in the default rounding mode). x * 2^(14-e) is exact in binary64 for every binary32 input. */
int orc_quantize_act16(const double* x, int q, int64_t K, int32_t* X, int32_t* e, double* xhat) {
    if (q < 1 || K < 0 || K % 32) return ORC_EINVAL;
    int64_t nb = K / 32;
    for (int t = 0; t < q; t++) {
        for (int64_t b = 0; b < nb; b++) {
            const double* v = x + (int64_t)t * K + b * 32;
            double a = 0.0;
            for (int j = 0; j < 32; j++) {
                if (!isfinite(v[j])) return ORC_ERANGE;
                if (fabs(v[j]) > a) a = fabs(v[j]);
            }
            int ex = 0;
            if (a > 0.0) frexp(a, &ex); /* a = f * 2^ex, 0.5 <= f < 1 */
            if (e) e[(int64_t)t * nb + b] = ex;
            for (int j = 0; j < 32; j++) {
                double r = a > 0.0 ? nearbyint(ldexp(v[j], 14 - ex)) : 0.0;
                int64_t i = (int64_t)t * K + b * 32 + j;
                if (X) X[i] = (int32_t)r;
                if (xhat) xhat[i] = ldexp(r, ex - 14);
            }
        }
    }
    return ORC_OK;
}
