/* CPU oracle for the low-bit MoE decode/verify path. TEST INFRASTRUCTURE ONLY.
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's CPU baseline may load or call this library.
 * The product path (the CUDA library and its Python binding) never does.
 *
 * Everything is binary64 with naive loops. The block layouts and the layer definition it follows are
 * written out in oracle.c next to the code that reads them; they fix what the pages leave open:
 *   - "DeepSeek V4 Flash hits 32 tok/s on AMD Ryzen AI MAX+ 395", the ROCmFPX paragraph (32-weight
 *     blocks, 10-byte FP2, 3.50 / 4.25 bits per weight FP3 / FP4, FP2 gate/up, FP3 down) and the
 *     decoding paragraph (q = 4 verification columns, each packed weight decoded once, top-4 routing,
 *     43 layers);
 *   - "Token Freedom via APU: AMD Ryzen AI MAX+ 395 Runs DeepSeek V4 Flash at 32 tok/s on a 284B
 *     Model", section "Lucebox's Optimization Trio" (256 routed + 1 shared expert, TOP-K and ARGSORT
 *     in the routing path, q = 4 weight reuse).
 * It shares no code, header, table or constant with the CUDA library.
 *
 * Parity status: bit compatibility with Lucebox's own ROCmFPX files is unpinned (the pages publish
 * no layout); every function here is pinned by tests/test_oracle_*.py against byte counts, hand-worked
 * blocks, closed forms and brute force.
 *
 * Return values: 0 on success, ORC_EINVAL for bad arguments, ORC_EDATA for an invalid block
 * (an FP4 scale byte of 255), ORC_ERANGE for a non-finite quantizer input or a scale overflow. */
#ifndef FPX_ORACLE_H
#define FPX_ORACLE_H
#include <stdint.h>

#define ORC_OK 0
#define ORC_EINVAL 1
#define ORC_ERANGE 3
#define ORC_EDATA 6

int orc_block_bytes(int fmt);
int64_t orc_matrix_bytes(int fmt, int64_t N, int64_t K);
int orc_threads(void);
int orc_set_threads(int n);

/* One block -> 32 binary64 values. */
int orc_decode_block(int fmt, const uint8_t* blk, double* w);
/* Packed N x K matrix -> W[N][K]. */
int orc_dequantize(int fmt, const uint8_t* Wq, int64_t N, int64_t K, double* W);
/* y[t][n] = sum_k W[n][k] x[t][k] and M[t][n] = sum_k |W[n][k] x[t][k]| (M may be NULL). */
int orc_gemv(int fmt, const uint8_t* Wq, int64_t N, int64_t K, const double* x, int q,
             double* y, double* M);
/* W[N][K] binary32 -> packed blocks; scales (NULL or [N*K/32]) are the scales to use. */
int orc_quantize(int fmt, const float* W, int64_t N, int64_t K, const float* scales, uint8_t* out);

/* Top-k of n values: descending, ties to the lower index. */
int orc_topk(const double* v, int n, int k, int32_t* idx);
/* Router: logits[t][e], Ml[t][e] = sum |R x|, top-k idx[t][r], normalised sigmoid weights w[t][r],
 * sorted union uni[0..n_uni-1]. Any output pointer may be NULL except idx. */
int orc_route(const float* R, int E, int H, const double* x, int q, int k, double* logits,
              double* Ml, int32_t* idx, double* w, int32_t* uni, int32_t* n_uni);

/* One MoE layer on q tokens (any q >= 1: decode verification columns or a prefill batch).
 * gate/up/down are arrays of E pointers to each routed expert's packed matrix (an entry may be NULL
 * if no token routes to it). If idx_force is non-NULL it replaces the oracle's own top-k (the
 * weights are still recomputed from the oracle's logits).
 * Outputs: y[t][H]; M[t][H] the first-order error magnitude used by the tolerance (see
 * oracle.c, orc_moe_layer); idx_out[t][k], w_out[t][k], logits_out[t][E] (each may be NULL). */
int orc_moe_layer(int H, int I, int E, const float* R, const uint8_t* const* gate,
                  const uint8_t* const* up, const uint8_t* const* down, const uint8_t* sh_gate,
                  const uint8_t* sh_up, const uint8_t* sh_down, const double* x, int q, int k,
                  const int32_t* idx_force, double* y, double* M, int32_t* idx_out, double* w_out,
                  double* logits_out);

/* Stack layer input: u[t][h] = RN_bfloat16(r / sqrt(mean(r^2) + 1e-6)), returned as the binary64
 * value of that bfloat16. */
int orc_rmsnorm_bf16(const float* r, int q, int H, double* u);

/* Stable argsort of n keys in [0, nkeys): perm lists the positions in key order, equal keys in
 * position order; offsets[e] = number of keys < e (nkeys + 1 entries). */
int orc_stable_argsort(const int32_t* keys, int n, int nkeys, int32_t* perm, int32_t* offsets);

/* Importance-weighted quantizer ([zh] page, section "ROCmFPX": quantization guided by an importance
 * matrix; the real matrix needs calibration data, so the importance here is any caller vector): for
 * each block, try the scales (amax / Kmax) * f, f = 0.60, 0.65, ..., 1.35 rounded to binary16
 * (FP2/FP3), or the E8M0 exponents e0 - 1, e0, e0 + 1 around the plain quantizer's e0 (FP4); under
 * each, the codes of orc_quantize; keep the one with the least sum over the block's 32 weights of
 * imp[col] * (w - w_hat)^2 (binary64, summed in weight order; the earliest candidate on equal sums).
 * imp [K] per column, NULL = all ones; a negative or non-finite importance or input is ORC_ERANGE. */
int orc_quantize_weighted(int fmt, const float* W, int64_t N, int64_t K, const float* imp, uint8_t* out);

/* Speculative verify/commit of one sequence ("DeepSeek V4 Flash hits 32 tok/s on AMD Ryzen AI MAX+
 * 395", paragraph 3, and the zh-TW page, section "DSpark", steps Propose / Verify / Commit): the
 * target scored q positions (the seed and q - 1 draft tokens) in one pass, logits [q][V]. pred[i] is
 * the target's choice at position i: the index of the largest logit, the lowest index among equal
 * maxima, NaN logits never chosen (all-NaN row: index 0 and ORC_ERANGE). Draft token d[j] (j = 0 ..
 * q - 2) proposes the token after position j; the accepted count n is the largest n <= q - 1 with
 * d[j] == pred[j] for every j < n. committed[0 .. n] = d[0 .. n-1] then pred[n] (the target's
 * correction at the first mismatch, or its next token after an all-accepted draft); entries past n
 * are -1. */
int orc_dspark_commit(const float* logits, int q, int V, const int32_t* drafts, int32_t* pred, int32_t* n_accept,
                      int32_t* committed);

/* Activations of the integer-dot GEMV ("DeepSeek V4 Flash hits 32 tok/s on AMD Ryzen AI MAX+ 395",
 * paragraph 3: codebooks expanded in registers feed integer dot products; the pages leave the
 * activation side open). For each column t and each run of 32 consecutive entries (a block): a = the
 * largest |x|; e = the integer with 2^(e-1) <= a < 2^e (e = 0 for an all-zero block); X = x * 2^(14-e)
 * rounded to the nearest integer, ties to even, so |X| <= 2^14. xhat = X * 2^(e-14) is the value the
 * integer dot products see; the variant's result is exactly W * xhat. X [q][K], e [q][K/32] and xhat
 * [q][K] may each be NULL; a non-finite x is ORC_ERANGE. */
int orc_quantize_act16(const double* x, int q, int64_t K, int32_t* X, int32_t* e, double* xhat);

#endif
