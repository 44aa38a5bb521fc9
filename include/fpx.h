/* fpx.h - C ABI of libfpx.so: block-quantized (FP2/FP3/FP4) GEMVs and the low-bit MoE
 * decode/verify step, hand-written CUDA for sm_103a (B300).
 *
 * Sources. The operations follow the public descriptions of the ROCmFPX formats and the DeepSeek V4
 * Flash decode path:
 *   [P-dsv4] "DeepSeek V4 Flash hits 32 tok/s on AMD Ryzen AI MAX+ 395" - paragraph 2 (the ROCmFPX
 *            family: 32-weight blocks of packed codes plus scales, FP2 10 bytes / 2.50 bits,
 *            FP3 3.50 bits, FP4 4.25 bits; FP2 routed gate/up, FP3 routed down, FP4 dense and
 *            sensitive projections) and paragraph 3 (memory-bound decode over 43 layers; each packed
 *            weight decoded once and applied to all four verification columns; TOP_K and ARGSORT
 *            kernels on the routing path; q = 4 verification in one fused pass).
 *   [P-apu]  "Token Freedom via APU: AMD Ryzen AI MAX+ 395 Runs DeepSeek V4 Flash at 32 tok/s on a
 *            284B Model" - section "Lucebox's Optimization Trio" (256 routed + 1 shared expert,
 *            6 active by default; q = 4 weight reuse; TOP-K / ARGSORT).
 *   [P-zh]   the zh-TW page, section "DSpark：在記憶體頻寬受限的 APU 上做 speculative decoding"
 *            (verify four positions, including the seed, in one graph pass).
 * The pages publish no API, byte layout or code; everything below that they leave open is a reading
 * made by this project and is stated where it is used.
 *
 * Block layouts (little-endian; 32 weights per block; a matrix W[N][K], K % 32 == 0, is row-major
 * with K/32 blocks per row and occupies fpx_matrix_bytes(), i.e. N*K/32*B rounded up to 16 bytes):
 *   FP2, 10 B: [0..1] binary16 scale d; [2..9] codes, c_j = bits 2j..2j+1; w_j = d*(2c_j - 3).
 *   FP3, 14 B: [0..1] binary16 d; [2..9] low bits l_j = bits 2j..2j+1; [10..13] high bit h_j = bit j;
 *              c = l + 4h; w_j = d*(2c_j - 7).
 *   FP4, 17 B: [0] E8M0 exponent e (scale 2^(e-127), 255 invalid); [1..16] E2M1 codes,
 *              q_j = bits 4j..4j+3 (sign bit 3, magnitude {0,.5,1,1.5,2,3,4,6}) - OCP MXFP4.
 *
 * Conventions for every call:
 *   - Pointers named in a signature are DEVICE pointers owned by the caller, unless a comment says
 *     host. Matrix and workspace pointers must be 16-byte aligned (FPX_EALIGN otherwise); vectors 4-,
 *     except where a call says otherwise (the activations of the tensor-core GEMVs 16-, of the
 *     router and decode-layer calls 8-byte, which their kernels read in 16- or 8-byte units).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream), never
 *     allocate and never synchronise; they are safe to capture in a CUDA graph. The return value
 *     reports argument errors and launch failures only.
 *   - Errors the device detects (an FP4 scale byte of 255, a non-finite quantizer input, an expert
 *     index out of range) set bit (1 << status) of a device status word: the `dev_status` argument
 *     (the caller zeroes it), or the first word of the workspace (zeroed by each layer or stack call
 *     when it starts). Read it after the stream completes (fpx_read_status).
 *   - Results are deterministic: no floating-point atomics, and every reduction has a fixed order
 *     for given inputs and shapes, so a repeated call gives the same bits. That order depends on
 *     neither q nor the other columns: column t of a q-column call (fpx_gemv_q, fpx_gemv_q_idot,
 *     moe_layer_decode, moe_layer_decode_tiered, moe_stack_verify) is bit-identical to a q = 1 call
 *     on column t alone. In the layer calls every expert matrix is streamed in pieces whose K ranges
 *     are fixed by the matrix shape (never by the expert union or the grid), added in piece order.
 */
#ifndef FPX_H
#define FPX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FPX_OK = 0,
    FPX_EINVAL = 1,   /* bad format, shape, q, k or dtype */
    FPX_EALIGN = 2,   /* a pointer is not aligned as required */
    FPX_ERANGE = 3,   /* non-finite quantizer input or scale overflow (device-detected) */
    FPX_ECUDA = 4,    /* a CUDA launch or attribute call failed */
    FPX_ETIMEOUT = 5, /* a bounded device-side wait gave up */
    FPX_EDATA = 6,    /* invalid block (FP4 scale 255) or routing index (device-detected) */
    FPX_ESPACE = 7    /* the workspace passed is smaller than the *_workspace_bytes query */
} fpx_status;

enum { FPX_FP2 = 2, FPX_FP3 = 3, FPX_FP4 = 4 };
enum { FPX_DTYPE_F32 = 0, FPX_DTYPE_BF16 = 1 };

const char* fpx_status_string(int status);

/* Bytes per 32-weight block: 10 / 14 / 17 for FP2 / FP3 / FP4, 0 for any other format. [P-dsv4] */
size_t fpx_block_bytes(int fmt);

/* Storage bytes of a packed N x K matrix (N*K/32 blocks, rounded up to 16), or -1 when K % 32 != 0,
 * N < 0 or the format is unknown. Stacked expert matrices use this value as their stride. */
int64_t fpx_matrix_bytes(int fmt, int64_t N, int64_t K);

/* Host call: copies the device status word *dev_status to *host_out after synchronising `stream`.
 * The only call that synchronises. */
int fpx_read_status(const int32_t* dev_status, int32_t* host_out, void* stream);

/* Quantize W[N][K] (binary32, row-major) into packed blocks at `out` (fpx_matrix_bytes bytes).
 * Per block: FP2/FP3 scale d = RN_binary16(amax/3 or amax/7) (or RN_binary16(block_scales[b])),
 * codes = nearest level, ties toward the smaller magnitude, sign = signbit; FP4 e = floor(log2 amax)
 * - 2 + 127 clamped to [0, 254] (or the exponent of block_scales[b], which must be a power of two),
 * codes = E2M1 round-to-nearest-even, saturating. block_scales (nullable) holds N*K/32 binary32
 * scales to use instead of the amax rule. A non-finite input or a binary16 overflow sets the
 * FPX_ERANGE bit (an unusable given scale the FPX_EINVAL bit) of *dev_status (nullable) and leaves
 * that block's bytes undefined. [P-dsv4] paragraph 2. */
int fpx_quantize(int fmt, const float* W, int64_t N, int64_t K, const float* block_scales,
                 uint8_t* out, int32_t* dev_status, void* stream);

/* Decode packed blocks into W[N][K] binary32 (every value is exact). An FP4 scale byte of 255 sets
 * the FPX_EDATA bit of *dev_status (nullable) and decodes that block as zeros. [P-dsv4] paragraph 2. */
int fpx_dequantize(int fmt, const uint8_t* Wq, int64_t N, int64_t K, float* W, int32_t* dev_status,
                   void* stream);

/* Importance-weighted quantizer (same block layouts and codes as fpx_quantize): for each block, tries
 * the scales (amax / Kmax) * f, f = 0.60, 0.65, ..., 1.35 rounded to binary16 (FP2/FP3; overflowing
 * ones skipped), or the E8M0 exponents e0 - 1, e0, e0 + 1 around fpx_quantize's e0 (FP4), and keeps
 * the one whose quantization has the least sum over the block's 32 weights of
 * importance[col] * (w - w_hat)^2 (binary64, summed in weight order, the earliest candidate on equal
 * sums). importance [K] per column (nullable: all ones); the plain scale is among the candidates, so
 * the weighted error never exceeds fpx_quantize's. A non-finite input or a negative or non-finite
 * importance sets FPX_ERANGE in *dev_status (that block's bytes are unspecified). [P-zh] section
 * "ROCmFPX" (quantization guided by an importance matrix; the real one needs calibration data). */
int fpx_quantize_weighted(int fmt, const float* W, int64_t N, int64_t K, const float* importance, uint8_t* out,
                          int32_t* dev_status, void* stream);

/* Rearranges `count` packed matrices (N x K, format fmt; matrix m at src + m * src_stride) between the
 * row-major layout and the box-tiled layout the MoE layer kernels read (matrix m at dst + m *
 * dst_stride; the same number of bytes). Box-tiled: each matrix is cut into tiles of R rows x B bytes
 * of each row (R x B = 256 x 80 for FP2, 256 x 112 for FP3, 64 x 272 for FP4); the tiles are stored
 * contiguously in (row block, column piece) order, each with its R rows at a pitch of B bytes, so the
 * byte at (row r, offset j within the row) is at ((r / R) * P + j / B) * R * B + (r % R) * B + j % B
 * with P = row bytes / B. inverse = 0 tiles a row-major src, 1 restores row-major from a tiled src.
 * Requires N % R == 0 and the row bytes (K / 32 * block bytes) a multiple of B; src, dst and the
 * strides 16-byte aligned; src != dst. The blocks themselves are unchanged: this is a layout for
 * streaming whole tiles with one bulk copy each, not part of the pages' format. */
int fpx_tile_matrices(int fmt, const uint8_t* src, int64_t N, int64_t K, int count, int64_t src_stride,
                      uint8_t* dst, int64_t dst_stride, int inverse, void* stream);

/* y[t][n] = sum_k W[n][k] * x[t][k] for t < q (1 <= q <= 4): the dense FPX GEMV of the verify step.
 * Every packed block is read from memory and decoded once per call, whatever q. x is [q][K]
 * contiguous, binary32 (x_dtype FPX_DTYPE_F32) or bfloat16 (FPX_DTYPE_BF16); y is [q][N] binary32.
 * Column t of the result is bit-identical to a q = 1 call on x[t]. An FP4 scale byte of 255 sets
 * the FPX_EDATA bit of *dev_status (nullable; that block counts as zeros). x must be 16-byte aligned
 * (FPX_EALIGN otherwise). [P-dsv4] paragraph 3, [P-apu]. */
int fpx_gemv_q(int fmt, const uint8_t* Wq, int64_t N, int64_t K, const void* x, int x_dtype, int q,
               float* y, int32_t* dev_status, void* stream);

/* Workspace bytes fpx_gemv_q_idot needs for K and q: (K/32 rounded up to a multiple of 32) * q * 68
 * (the activation table) + 16 (a row-block counter). 0 for invalid arguments. */
size_t fpx_gemv_idot_workspace_bytes(int64_t K, int q);

/* Integer-dot variant of fpx_gemv_q: the packed blocks are expanded with byte permutes into signed
 * bytes (FP2 2c - 3, FP3 2c - 7, FP4 twice the E2M1 value) and multiplied against integer activations
 * with 4-way byte dot products ([P-dsv4] paragraph 3: codebooks expanded in registers feed integer
 * dot products). The pages leave the activation side open; here, per column t and block b of 32
 * entries, a = max |x|, e with 2^(e-1) <= a < 2^e (0 for an all-zero block), X = RN_even(x 2^(14-e))
 * (|X| <= 2^14, sent as a signed high byte and an unsigned low byte), so every block dot product is an
 * exact integer and y[t][n] = sum_b d_nb 2^(e_tb - 14) sum_j v_j X_j, i.e. the plain GEMV of
 * x_hat = X 2^(e-14) up to binary32 rounding of the block terms and of their sums (|x_hat - x| <=
 * 2^(e-15)). Same arguments and layouts as fpx_gemv_q (x 4-byte aligned suffices), plus a caller workspace ws (16-byte aligned,
 * >= fpx_gemv_idot_workspace_bytes(K, q) bytes, else FPX_ESPACE; overwritten) that carries the activation table from the
 * first kernel to the second. Requires K % 256 == 0 (FP2 / FP3) or K % 512 == 0 (FP4), so rows are
 * whole 16-byte units, and K * q small enough for the table to sit in shared memory next to two weight
 * stages (FPX_EINVAL otherwise; about K * q <= 2^16). A non-finite x entry sets FPX_ERANGE (it counts
 * as 0); an FP4 scale byte of 255 sets FPX_EDATA (that block counts as zeros). Column t of the result
 * is bit-identical to a q = 1 call on x[t]; the sums run in a fixed order. */
int fpx_gemv_q_idot(int fmt, const uint8_t* Wq, int64_t N, int64_t K, const void* x, int x_dtype, int q,
                    float* y, void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/* Workspace bytes fpx_gemv_q_tiled needs for these shapes: P * q * N * 4 (the partial rows of P > 1
 * pieces, see below), else 16. 0 for invalid arguments. */
size_t fpx_gemv_tiled_workspace_bytes(int fmt, int64_t N, int64_t K, int q);

/* fpx_gemv_q on one box-tiled matrix (fpx_tile_matrices with count 1): y[t][n] = sum_k W[n][k] x[t][k]
 * for t < q (1 <= q <= 4), streamed the way the MoE layer kernels stream their experts (one bulk copy
 * per tile of R rows, decoded by the same tensor-core engine; exact products, binary32 sums). Requires
 * N % R == 0 (R = 256 for FP2 / FP3, 64 for FP4), K % 256 == 0 (FP2 / FP3) or K % 512 == 0 (FP4), and
 * the activation table (9 K bytes FP2 / FP3, 8 K FP4) beside a 140 KB ring within the shared memory
 * per block (K <= 9728 with 227 KB), FPX_EINVAL otherwise; Wt, x and ws 16-byte aligned, y 4-byte.
 * ws holds at least fpx_gemv_tiled_workspace_bytes(fmt, N, K, q) bytes (FPX_ESPACE otherwise) and is
 * overwritten. A row tile's K range is split into P = min(K / stage, ceil(592 / (N / R))) pieces of
 * consecutive stages (stage = 256 weights FP2 / FP3, 512 FP4), a function of N and K alone, whose sums
 * are added in piece order: column t of the result is bit-identical to a q = 1 call on x[t]. The sums
 * run in another order than fpx_gemv_q's, so the two agree within the GEMV tolerance, not bit for
 * bit. An FP4 scale byte of 255 sets FPX_EDATA in *dev_status (nullable; that block counts as zeros).
 * [P-dsv4] paragraph 3. */
int fpx_gemv_q_tiled(int fmt, const uint8_t* Wt, int64_t N, int64_t K, const void* x, int x_dtype, int q,
                     float* y, void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/* Router + top-k + normalise + union for q tokens (1 <= q <= 4): logits[t][e] = sum_h R[e][h] x[t][h]
 * (R binary32 [E][H], x bfloat16 [q][H]); idx[t][r], r < k, the k largest logits in descending order,
 * ties to the lower expert index; w[t][r] = sigmoid(l) / sum over the k selected sigmoids; uni the
 * sorted distinct experts of all tokens (n_uni of them, at most q*k; uni has q*k entries).
 * Limits: 1 <= k <= 8, k <= E <= 1024, H % 16 == 0, and (2q + 8) H bytes within the device's shared
 * memory per block (x and two router rows are staged there: H <= 14528 at q = 4 with 227 KB),
 * FPX_EINVAL otherwise; x 8-byte aligned (FPX_EALIGN otherwise). logits [q][E] is required: it is also the top-k input. [P-apu], [P-dsv4]
 * paragraph 3. */
int moe_route_topk(const float* R, int E, int H, const uint16_t* x, int q, int k, float* logits,
                   int32_t* idx, float* w, int32_t* uni, int32_t* n_uni, void* stream);

/* One MoE layer's weights (device pointers inside a host struct). Routed experts e = 0..E-1 are
 * stacked: expert e's gate matrix starts at gate + e*fpx_matrix_bytes(FP2, I, H); likewise up (FP2,
 * I x H) and down (FP3, H x I). The shared expert is FP4: sh_gate, sh_up [I][H], sh_down [H][I].
 * Every expert matrix is in the box-tiled layout of fpx_tile_matrices.
 * router is binary32 [E][H]. H and I are multiples of 512 and at most 4608 (the tensor-core
 * kernels hold a 144 KB ring of weight boxes and two activation tables of 8*H bytes in shared
 * memory). [P-dsv4] paragraph 2,
 * [P-apu]. */
typedef struct {
    int H, I, E;
    const float* router;
    const uint8_t* gate;
    const uint8_t* up;
    const uint8_t* down;
    const uint8_t* sh_gate;
    const uint8_t* sh_up;
    const uint8_t* sh_down;
} moe_layer;

/* Workspace bytes moe_layer_decode / moe_stack_verify need for these shapes (16-byte aligned). */
size_t moe_workspace_bytes(const moe_layer* layer, int q, int k);

/* One MoE decode/verify layer for q tokens (1 <= q <= 4, 1 <= k <= 8): route each token, run every
 * selected expert once for all q columns (g = G x, u = U x, h = silu(g) u in binary32, y = D h), the
 * shared expert for all tokens, and combine out[t] = sum_r w[t][r] y_{e(t,r)}[t] + y_shared[t]
 * (ranks in order, shared last). x is bfloat16 [q][H] (8-byte aligned), y binary32 [q][H]; idx_out (nullable) gets
 * idx[q][k], w_out (nullable) w[q][k], logits_out (nullable) logits[q][E]. `ws` must hold
 * moe_workspace_bytes(layer, q, k) bytes (ws_bytes); its first word is the status word. The layer
 * pointer is read on the host during the call only. [P-dsv4] paragraph 3, [P-zh], [P-apu]. */
int moe_layer_decode(const moe_layer* layer, const uint16_t* x, int q, int k, float* y,
                     int32_t* idx_out, float* w_out, float* logits_out, void* ws, size_t ws_bytes,
                     void* stream);

/* Two-tier expert residency for moe_layer_decode_tiered ([P-apu] section "Asymmetric Dual-GPU": the
 * popular experts live in the fast memory, the cold ones in the large pool, results merged on one
 * device; the Paiton page on DeepSeek V4.1 Flash, section "Keeping useful work on the GPU": the most
 * used experts on the GPU, the rest in host memory, streamed to the GPU for long prompts). The layer's gate / up / down arrays then hold n_slots expert slots in HBM (stacked as
 * in moe_layer, slot s at s * fpx_matrix_bytes), not E experts:
 *   slot_of     device int32 [E]: the HBM slot that holds expert e's three matrices, or -1 when e is
 *               cold (only in the cold tier);
 *   cold_gate, cold_up, cold_down: HOST pointers to pinned (page-locked) memory holding all E experts
 *               stacked exactly as moe_layer's arrays (box-tiled); read by the device over the host
 *               link, so they must stay pinned and unchanged during the call;
 *   stage_slot0, n_stage: the HBM slots [stage_slot0, stage_slot0 + n_stage) that receive the cold
 *               experts a call needs; n_stage >= min(q * k, E), stage_slot0 + n_stage <= n_slots,
 *               and no hot expert may sit in that range;
 *   cache       nullable device int32 [2 + 2 n_stage] (n_stage <= 1024 then): the staging slots keep
 *               their experts across calls (see moe_tiers_cache_reset). Layout: [0] a call counter,
 *               [1] the number of experts copied so far, [2 + i] the expert held by staging slot i
 *               (-1: none), [2 + n_stage + i] the counter value of slot i's last use. NULL: every
 *               call copies every cold expert of its union. */
typedef struct {
    const int32_t* slot_of;
    const uint8_t* cold_gate;
    const uint8_t* cold_up;
    const uint8_t* cold_down;
    int n_slots;
    int stage_slot0;
    int n_stage;
    int32_t* cache;
} moe_tiers;

/* moe_layer_decode on a two-tier layer: after routing, every cold expert of the union gets a staging
 * slot and the layer runs on the slots. Without a cache the i-th cold item (ascending expert order)
 * takes slot stage_slot0 + i and is copied from the host tier. With tiers->cache, a cold expert that a
 * staging slot already holds is used there without a copy; each other one is copied into the slot
 * whose last use is oldest among the slots this call has not taken (ties to the lower slot), and the
 * cache records it. Results (y, routing, logits) are bit-identical to moe_layer_decode on a layer
 * holding all E experts in HBM. A slot_of entry >= n_slots or inside the staging range sets FPX_EDATA
 * in the status word and that expert is treated as cold. Same workspace as moe_layer_decode. Returns
 * FPX_EINVAL if a cold pointer is not pinned host memory or (with a cache) n_stage > 1024; calls
 * sharing staging slots or a cache must be ordered on one stream. The pages' own design computes
 * cold experts on the CPU cores; here every expert runs on the GPU and only the weights move (the
 * Paiton page's streaming mode). The host link (about 51 GB/s measured) is the bound of a call that
 * copies: an expert's three matrices take about 0.18 ms, against about 0.07 ms for the whole layer
 * from HBM, which is why a cached expert is not copied again. */
int moe_layer_decode_tiered(const moe_layer* layer, const moe_tiers* tiers, const uint16_t* x, int q, int k,
                            float* y, int32_t* idx_out, float* w_out, float* logits_out, void* ws,
                            size_t ws_bytes, void* stream);

/* Empties tiers->cache (enqueued on stream): counter and copy count 0, no expert in any staging slot.
 * Call it before the first moe_layer_decode_tiered with that cache, and again whenever the cold tier's
 * contents, slot_of or the staging slots change outside these calls: the cache trusts that a slot
 * still holds the expert it recorded. FPX_EINVAL without a cache or with n_stage outside 1..1024.
 * Part of the two-tier residency ([P-apu] section "Asymmetric Dual-GPU"); the pages do not say how
 * streamed experts are kept, so the least-recently-used rule is this library's. */
int moe_tiers_cache_reset(const moe_tiers* tiers, void* stream);

/* moe_layer_decode for callers that cannot allocate device memory: a plugin or library running
 * inside a host framework that owns every device allocation (its own arena or allocator) and allows
 * no others, or a latency-critical loop that must never call cudaMalloc/cudaFree because they can
 * synchronise the device. The pages have no counterpart to this call; it exists for deployment only.
 * Same arguments and results as moe_layer_decode, except that the scratch is a 16 MiB array inside
 * libfpx.so (one per device, held until the process exits) instead of a caller workspace, and the
 * status word is copied to dev_status (nullable, device, 4-byte aligned) at the end of the call.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 *   - Shapes whose moe_workspace_bytes() exceeds 16 MiB fail with FPX_ESPACE (the decode shapes,
 *     H = 4096, I = 2048, E = 256, q <= 4, k <= 8, need at most 9.4 MB).
 *   - The first call on a device looks up the array's device address (cudaGetSymbolAddress) with
 *     that device current; make that first call before capturing a stream into a graph.
 *   - Every call on a device shares the one array, which keeps the previous call's contents: calls
 *     whose work overlaps on the GPU (different streams, or several host threads) race. Issue them
 *     in order on one stream. */
int moe_layer_decode_static_ws(const moe_layer* layer, const uint16_t* x, int q, int k, float* y,
                               int32_t* idx_out, float* w_out, float* logits_out, int32_t* dev_status,
                               void* stream);

/* The verify pass over a stack of n_layers layers (host array of structs, all with the same H, I,
 * E): state r binary32 [q][H] starts at r0; layer l takes u_l = RN_bfloat16(r_l / sqrt(mean(r_l^2)
 * + 1e-6)) and sets r_{l+1} = r_l + MoE_l(u_l). rL receives r_{n_layers}; r0 and rL may alias.
 * idx_out (nullable) gets idx[n_layers][q][k]; r_trace (nullable) gets r_l for l = 0..n_layers-1
 * ([n_layers][q][H]). Enqueues a copy and a small memset and then 5 kernels per layer (router,
 * gate/up, h + down tables, down, combine), each launched as a programmatic dependent launch so that
 * it overlaps the previous kernel's tail, and nothing else, so the whole pass can be captured as one
 * CUDA graph. events (nullable) is a host array of 5*n_layers + 1 cudaEvent_t: events[5l + j] is
 * recorded on `stream` just before kernel j of layer l and events[5*n_layers] after the last kernel,
 * so a caller can time each kernel (with events the kernels run without overlap).
 * The normalisation is this project's reading (the pages do not define the residual stream):
 * without it the synthetic state overflows binary32 within a few dozen layers.
 * [P-dsv4] paragraph 3 (43 layers; every token streams the active weights of all layers). */
int moe_stack_verify(const moe_layer* layers, int n_layers, const float* r0, int q, int k, float* rL,
                     int32_t* idx_out, float* r_trace, void* ws, size_t ws_bytes, void* const* events,
                     void* stream);

/* Workspace bytes moe_layer_prefill needs for T tokens and top-k (16-byte aligned; about
 * T*k*(10 I + 6 H) + T*(10 I + 8 H) + 6 E H bytes: 0.67 GB at T = 2048, k = 6, H = 4096, I = 2048,
 * E = 256).
 * 0 for invalid arguments. */
size_t moe_prefill_workspace_bytes(const moe_layer* layer, int T, int k);

/* Batched prefill of one MoE layer over T tokens (T >= 1, 1 <= k <= 8, k <= E <= 1024):
 *   - route every token by the rule of moe_route_topk (top-k by logit with ties to the lower expert
 *     index, sigmoid weights renormalised over the k selected) on binary32 logits summed on the
 *     tensor cores from exact products (the router split into three bfloat16 parts); the summation
 *     order differs from moe_route_topk's, so logits agree to binary32 rounding, not bit for bit;
 *   - stable argsort of the T*k pairs p = t*k + r by expert: perm[s] = p lists the pairs in expert
 *     order, p ascending within an expert; offsets[e] .. offsets[e+1] is expert e's range;
 *   - run each routed expert once over its pairs (grouped GEMMs on the tensor cores over the same
 *     box-tiled weights as moe_layer_decode: g = G x, u = U x, h = silu(g) u in binary32, y = D h)
 *     and the shared expert over all tokens;
 *   - out[t] = sum_r w[t][r] y_{e(t,r)}[t] (ranks in order) + y_shared[t].
 * x is bfloat16 [T][H], y binary32 [T][H]. Nullable outputs: idx_out [T][k], w_out [T][k],
 * logits_out [T][E], perm_out [T*k], offsets_out [E+1]. The GEMMs (tcgen05 tensor cores) take the
 * activations as binary16 rows scaled by a power of two per row (h likewise; exact), FP2 / FP3
 * weights d (2c - 3), d (2c - 7) rounded once to binary16 (relative error <= 2^-11) and FP4 weights
 * scaled per row by a power of two (exact for blocks within 2^14 of the row's largest block scale,
 * binary16 subnormals below that, zero below 2^-25 of it); the sums are binary32. ws
 * holds moe_prefill_workspace_bytes(layer, T, k) bytes (ws_bytes); its first word is the status
 * word. [P-dsv4] paragraph 3 (TOP_K, ARGSORT), [P-apu] section "Lucebox's Optimization Trio"; the
 * grouping of a batch by expert is this project's reading (the pages describe decode). */
int moe_layer_prefill(const moe_layer* layer, const uint16_t* x, int T, int k, float* y, int32_t* idx_out,
                      float* w_out, float* logits_out, int32_t* perm_out, int32_t* offsets_out, void* ws,
                      size_t ws_bytes, void* stream);

/* Test hook for the bounded device waits of the layer kernels (moe_layer_decode, _tiered, _static_ws,
 * moe_stack_verify) on the current device; not for production use. wait_ns (1 .. 500,000,000; the
 * default is 500,000,000) bounds each wait between a streaming kernel's producer and its consumers.
 * drop_stage >= 0 makes CTA 0 of the gate/up kernel withhold its drop_stage-th weight copy, as if
 * it were lost: its consumers wait wait_ns for it, give up, set FPX_ETIMEOUT in the status word and
 * return, every copy that was issued having landed first; the result of that call is undefined, and
 * later calls (with drop_stage = -1, the default) are unaffected. Host call, synchronous (it writes
 * two device variables); make it between calls, never while a layer call runs. FPX_EINVAL for
 * arguments out of range. The pages have no counterpart: this exists to test failure detection. */
int fpx_debug_ring_wait(uint64_t wait_ns, int drop_stage);

/* Speculative verify/commit for B sequences (B >= 0, 1 <= q <= 16, V >= 1): the target scored q
 * positions of each sequence (the seed and q - 1 draft tokens) in one pass; logits is binary32
 * [B][q][V], drafts int32 [B][q-1] (nullable when q == 1). Outputs: pred [B][q], the target's choice
 * at each position (the largest logit, lowest index among equal maxima, NaN never chosen; an all-NaN
 * row gives 0 and sets FPX_ERANGE in *dev_status, nullable); n_accept [B], the largest n <= q - 1
 * with drafts[b][j] == pred[b][j] for all j < n; committed [B][q] = the n accepted drafts, then
 * pred[b][n], then -1. Reads the logits once (HBM-bound). [P-dsv4] paragraph 3 (four positions
 * including the seed; correct proposals commit, the first error is corrected by the target),
 * [P-zh] section "DSpark" (Propose / Verify / Commit). */
int dspark_verify_commit(const float* logits, int B, int q, int V, const int32_t* drafts, int32_t* pred,
                         int32_t* n_accept, int32_t* committed, int32_t* dev_status, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* FPX_H */
