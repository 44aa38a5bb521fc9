// Batched prefill of one MoE layer over T tokens: routing, a stable argsort of the (token, rank) pairs
// by expert, grouped GEMMs over the box-tiled expert weights (gate/up, SiLU gating, down, for the
// routed experts and the shared one) and the weighted combine.
//
// "DeepSeek V4 Flash hits 32 tok/s on AMD Ryzen AI MAX+ 395", paragraph 3 (TOP_K and ARGSORT on the
// routing path; the same low-bit experts), and "Token Freedom via APU: ...", section "Lucebox's
// Optimization Trio" (256 routed + 1 shared expert, 6 active). The pages describe decode; a prefill
// that groups the tokens of a batch by expert and runs each expert once over its group is this
// project's reading of running the same layer on many tokens at once.
//
// Pipeline (one stream, no host synchronisation):
//   k_to_f16   x (bfloat16) -> binary16 rows scaled by a per-token power of two (exact), + shifts
//   k_rsplit / k_plogits_tc  logits[t][e] = sum_h R[e][h] x[t][h] on the tcgen05 tensor cores: the
//              binary32 router split into three exact bfloat16 parts, binary32 sums
//   k_ptopk    one warp per token: top-k by logit (ties to the lower index), sigmoid weights
//   k_phist / k_pscan / k_pscatter: stable counting sort of the T*k pairs p = t*k + r by expert:
//              perm[s] = p in expert order (p ascending within an expert), inv[p] = s, offsets[E+1]
//   k_pgather  the pairs' activation rows in expert order, each 16-group in the decode's pair order
//   k_tcunits  the tensor-core GEMM units (expert, pair tile of <= 128, 256-row block)
//   k_tcgemm   grouped GEMM on the tcgen05 tensor cores: out[s][m] = sum_k W_e[m][k] b_s[k]
//              (routed gate / up FP2, routed down FP3; the shared expert's FP4 gate / up / down over
//              every token after k_fp4_rowexp, k_perm4 and k_tcunits_dense)
//   k_ph       h = silu(g) u (binary32), then binary16 rows scaled by a per-row power of two
//   k_pcombine out[t] = sum_r w[t][r] y[inv[t*k+r]] (ranks in order) + y_shared[t]
//
// GEMM arithmetic. B is the activation row in binary16 times its power-of-two scale (exact). FP2 /
// FP3: the A operand is the weight d (2c - 3) or d (2c - 7) rounded once to binary16 (relative error
// at most 2^-11 per weight, a quarter of the 2e-3 bound). FP4: the E2M1 value times 2^(e - E_m + 1),
// E_m the row's largest block exponent; exact in binary16 for blocks within 2^14 of the row's largest
// scale, smaller ones rounded as binary16 subnormals and blocks more than 2^24 below it dropped (their
// share of the row is below 2^-24 of its largest block's). The row factor 2^(E_m - 128) is applied to
// the binary32 accumulator. The tensor core accumulates in binary32 across the whole K.
#include "fpx_mma.cuh"
#include "route.cuh"
#include "tc.cuh"

using namespace fpx;

namespace {

constexpr int kPMaxK = 8;

// ------------------------------------------------------------------ workspace

struct PWs {
    size_t status, logits, idx, w, counts, offsets, perm, inv, x16, shx;
    size_t g, u, gsh, ush, h16, shh, hsh16, shsh, yp, ysh, xg, gshift, tcu_gu, tcu_dn, ntc;
    size_t xs4, rexp, tcu_sgu, tcu_sdn, rsplit, total;
};

inline size_t up256(size_t v) { return (v + 255) & ~size_t(255); }

PWs pws_layout(int64_t T, int64_t E, int64_t H, int64_t I, int64_t k) {
    PWs w{};
    size_t o = 0;
    const int64_t P = T * k;
    w.status = o; o = up256(o + 16);
    w.logits = o; o = up256(o + 4 * T * E);
    w.idx = o; o = up256(o + 4 * P);
    w.w = o; o = up256(o + 4 * P);
    w.counts = o; o = up256(o + 4 * (E + 1));
    w.offsets = o; o = up256(o + 4 * (E + 1));
    w.perm = o; o = up256(o + 4 * P);
    w.inv = o; o = up256(o + 4 * P);
    w.x16 = o; o = up256(o + 2 * T * H);
    w.shx = o; o = up256(o + 4 * T);
    w.g = o; o = up256(o + 4 * P * I);
    w.u = o; o = up256(o + 4 * P * I);
    w.gsh = o; o = up256(o + 4 * T * I);
    w.ush = o; o = up256(o + 4 * T * I);
    w.h16 = o; o = up256(o + 2 * P * I);
    w.shh = o; o = up256(o + 4 * P);
    w.hsh16 = o; o = up256(o + 2 * T * I);
    w.shsh = o; o = up256(o + 4 * T);
    w.yp = o; o = up256(o + 4 * P * H);
    w.ysh = o; o = up256(o + 4 * T * H);
    w.xg = o; o = up256(o + 2 * P * H);                            // activations gathered per pair, K-permuted
    w.gshift = o; o = up256(o + 4 * P);
    w.tcu_gu = o; o = up256(o + 16 * (P / 128 + E) * (I / 256));  // tensor-core GEMM units
    w.tcu_dn = o; o = up256(o + 16 * (P / 128 + E) * (H / 256));
    w.ntc = o; o = up256(o + 16);
    w.xs4 = o; o = up256(o + 2 * T * H);                           // tokens in the FP4 decode's pair order
    w.rexp = o; o = up256(o + 4 * (2 * I + H));                    // FP4 row exponents: gate, up, down
    w.tcu_sgu = o; o = up256(o + 16 * ((T + 127) / 128) * (I / 256));  // shared expert's units
    w.tcu_sdn = o; o = up256(o + 16 * ((T + 127) / 128) * (H / 256));
    w.rsplit = o; o = up256(o + 2 * 3 * E * H);                    // router weights as three bfloat16 parts
    w.total = o;
    return w;
}

// ------------------------------------------------------------------ activations to binary16

// Row r of src (bfloat16 [R][L], or binary32 when F32) -> dst binary16 row scaled by 2^sh, with
// sh = column_shift(max |row|) (largest element in [2^14, 2^15)); shift[r] = sh. One CTA per row.
template <bool F32>
__global__ void __launch_bounds__(256) k_to_f16(const void* __restrict__ src, int L, __half* __restrict__ dst,
                                                int32_t* __restrict__ shift) {
    __shared__ float red[8];
    __shared__ int sh_s;
    const size_t r = blockIdx.x;
    float m = 0.f;
    for (int i = threadIdx.x; i < L; i += blockDim.x) {
        const float v = F32 ? reinterpret_cast<const float*>(src)[r * L + i]
                            : __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(src)[r * L + i] << 16);
        m = fmaxf(m, fabsf(v));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x / 32] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float mm = 0.f;
        for (int i = 0; i < 8; i++) mm = fmaxf(mm, red[i]);
        sh_s = column_shift(mm);
        shift[r] = sh_s;
    }
    __syncthreads();
    const float sc = exp2i(sh_s);
    for (int i = threadIdx.x; i < L; i += blockDim.x) {
        const float v = F32 ? reinterpret_cast<const float*>(src)[r * L + i]
                            : __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(src)[r * L + i] << 16);
        dst[r * L + i] = __float2half_rn(v * sc);
    }
}

// ------------------------------------------------------------------ routing

// One warp per token.
__global__ void __launch_bounds__(256) k_ptopk(const float* __restrict__ logits, int T, int E, int k, int32_t* idx,
                                               float* w) {
    const int t = blockIdx.x * 8 + threadIdx.x / 32;
    if (t >= T) return;
    warp_topk(logits + (size_t)t * E, E, k, idx + (size_t)t * k, w + (size_t)t * k);
}

__global__ void k_phist(const int32_t* __restrict__ idx, int P, int E, int32_t* counts, int32_t* status) {
    const int p = blockIdx.x * blockDim.x + threadIdx.x;
    if (p >= P) return;
    const int e = idx[p];
    if (e < 0 || e >= E) { flag(status, FPX_EDATA); return; }
    atomicAdd(counts + e, 1);
}

// One CTA of 1024 threads (E <= 1024): offsets = exclusive scan of counts.
__global__ void __launch_bounds__(1024) k_pscan(const int32_t* __restrict__ counts, int E, int32_t* offsets) {
    __shared__ int32_t a[1024];
    const int e = threadIdx.x;
    const int n = e < E ? counts[e] : 0;
    a[e] = n;
    __syncthreads();
    for (int o = 1; o < 1024; o <<= 1) {  // inclusive scan (Hillis-Steele)
        const int va = e >= o ? a[e - o] : 0;
        __syncthreads();
        a[e] += va;
        __syncthreads();
    }
    if (e < E) offsets[e] = a[e] - n;
    if (e == E - 1) offsets[E] = a[e];
}

// One CTA per expert: the pairs routed to it, in increasing pair index (stable).
__global__ void __launch_bounds__(256) k_pscatter(const int32_t* __restrict__ idx, int P, const int32_t* __restrict__ offsets,
                                                  int32_t* perm, int32_t* inv) {
    __shared__ int32_t wc[8];
    const int e = blockIdx.x, warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    int base = offsets[e];
    for (int p0 = 0; p0 < P; p0 += 256) {
        const int p = p0 + threadIdx.x;
        const bool m = p < P && idx[p] == e;
        const uint32_t bal = __ballot_sync(0xffffffffu, m);
        if (lane == 0) wc[warp] = __popc(bal);
        __syncthreads();
        int before = 0, tot = 0;
        for (int i = 0; i < 8; i++) {
            before += i < warp ? wc[i] : 0;
            tot += wc[i];
        }
        if (m) {
            const int s = base + before + __popc(bal & ((1u << lane) - 1u));
            perm[s] = p;
            inv[p] = s;
        }
        base += tot;
        __syncthreads();
    }
}

// ------------------------------------------------------------------ binary16 pair arithmetic

__device__ __forceinline__ uint32_t hfma2_u(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t hmul2_u(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// ------------------------------------------------------------------ tcgen05 grouped GEMM (routed)
//
// The routed experts' GEMMs on the fifth-generation tensor cores. A unit is (expert e, 256 weight
// rows, up to 128 of the expert's pairs): D[256 x n] = W_e[rows][K] * B[pairs][K]^T, accumulated in
// binary32 in tensor memory as two M = 128 halves. The decoded weights never touch shared memory: they
// are the MMA's A operand in tensor memory. The K loop runs in stages of 128 (two 64-wide slabs):
//   warp 0       streams the packed weight boxes (one 1-D bulk copy per 256 x 256 box) into a ring;
//   warp 1       streams the stage's B (2-D TMA tiles of 16 rows x 64, 128-byte swizzle, only the
//                unit's n rows rounded up to 16) into a shared-memory stage;
//   warps 4..19  a weight row and 64 of the stage's 128 K per thread (code groups 2 p, 2 p + 1 of both
//                slabs; tensor-memory lane quarter warp % 4): decode the codes in registers into
//                binary16 weights d (2c - 3) or d (2c - 7) (rounded once, as in the rest of the
//                prefill) and store them into the A stage with one tcgen05.st;
//   warps 2, 3   (one thread each, one per accumulator half: a single issuing thread cannot keep the
//                tensor core busy at n <= 64) issue 8 tcgen05.mma of 128 x n x 16 (A in tensor memory,
//                B in shared memory) and commit them to the stages' release barriers; after the last
//                stage, to the accumulator barrier;
//   warps 20..23 read the finished accumulator (tcgen05.ld), scale each column by 2^-shift of its B
//                row and store out[pair][row].
// Every handshake costs instructions in each of the 16 decoder warps; 128-wide stages halve them per
// weight, which matters because the decode is issue-bound.
// Tensor memory: columns 0..255 accumulators, 256..511 two A stages of 128 columns (two halves x 64;
// within a half, the 8 K steps of 16 sit in the order 0, 1, 4, 5, 2, 3, 6, 7 so that each decoder
// thread's 32 columns are contiguous). A unit of n <= 64 pairs uses one of two 128-column accumulator
// buffers (halves at +0 and +64), so its epilogue overlaps the next unit's MMAs; a larger unit uses
// both (halves at 0 and 128).
// The decode produces each 16-weight group in the order its binary16 pairs come out of the register
// decode (FP2 / FP3: pair p = weights p and p + 8; FP4: weights p + 4 (p / 4) and that + 4); the B rows
// are stored in the same order (k_pgather and k_ph<1> for FP2 / FP3, k_perm4 and k_ph<2> for FP4), so the
// products pair up as in the plain dot product.
constexpr int kTcN = 128;                                           // pairs per unit at most
constexpr int kTcSK = 128;                                          // K per stage
constexpr int kTcAStages = 2;                                       // A stages in tensor memory
constexpr int kTcDec = 16, kTcEpi = 4;                              // decoder and epilogue warps
constexpr int kTcIss = 2;                                           // MMA-issuing warps (one per half)
constexpr int kTcDec0 = 2 + kTcIss;                                 // first decoder warp
constexpr int kTcThreads = (kTcDec0 + kTcDec + kTcEpi) * 32;
constexpr int kTcBRows = 16;                                        // rows of one B tile load
constexpr int kTcBTile = kTcN * 128;                                // 128 rows x 64 binary16
constexpr int kTcBStage = 2 * kTcBTile;                             // a stage: two 64-wide tiles
// Ring slot of packed weights: FP2 / FP3 one 256 x 256 box (FP3's 28 KB), FP4 the four 64-row boxes
// of 256 rows x 512 K; slots in flight; B stages.
__host__ __device__ constexpr int tc_slot_bytes(int fmt) { return fmt == 4 ? 4 * stage_bytes(4) : stage_bytes(3); }
__host__ __device__ constexpr int tc_slot_k(int fmt) { return fmt == 4 ? 512 : 256; }
__host__ __device__ constexpr int tc_ring_slots(int fmt) { return fmt == 4 ? 2 : 3; }
__host__ __device__ constexpr int tc_bstages(int fmt) { return fmt == 4 ? 2 : 4; }
// (+ 1024 for aligning the base, + 64: the FP4 decode's last word load may run 20 bytes past a row)
__host__ __device__ constexpr int tc_smem(int fmt) {
    return tc_ring_slots(fmt) * tc_slot_bytes(fmt) + tc_bstages(fmt) * kTcBStage + 1024 + 64;
}
constexpr int kTcMaxRS = 3, kTcMaxBS = 4;
constexpr int kTcCols = 512;
constexpr uint32_t kTcACol = 256;                                   // first A-stage column
static_assert(tc_slot_bytes(2) % 1024 == 0 && tc_slot_bytes(4) % 1024 == 0 && kTcBTile % 1024 == 0, "1024-byte aligned stages");
static_assert(tc_smem(2) + kTcEpi * kTcN * 4 + 1024 <= 227 * 1024 && tc_smem(4) + kTcEpi * kTcN * 4 + 1024 <= 227 * 1024,
              "shared memory per CTA");
static_assert(kTcACol + 128 * kTcAStages <= kTcCols, "tensor-memory columns");

// Column block (8 columns) of K step kk (0..7, 16 K each) within a half's 64 A-stage columns. FP2 /
// FP3 (kk = slab kk / 4, code group kk % 4): thread p of a row owns blocks 4 p .. 4 p + 3 (groups 2 p,
// 2 p + 1 of both slabs). FP4: thread p owns the stage's 32-weight blocks 2 p, 2 p + 1, i.e. K steps
// 4 p .. 4 p + 3 in order.
template <int FMT>
__host__ __device__ constexpr uint32_t tc_kblock(int kk) {
    return FMT == 4 ? (uint32_t)kk : 4u * ((kk & 3) >> 1) + 2u * (kk >> 2) + (kk & 1);
}

struct TcArgs {
    CUtensorMap bmap;         // B: binary16 [rows][K], K-permuted, box 64 x 16, 128-byte swizzle
    const uint8_t* W;         // box-tiled matrix of expert 0
    int64_t mstride;          // bytes between experts' matrices
    int M, K;
    const int4* units;        // (expert, first B row, pairs, 256-row block)
    const int32_t* nunits;
    const int32_t* shift;     // power-of-two scale exponent of every B row
    const int32_t* rowexp;    // FP4: largest valid block exponent of every weight row (else unused)
    float* out;               // [B rows][M]
    int32_t* status;
};

// 16 weights of one decoded code group as binary16 pairs (pair p = weights p and p + 8) with the block
// scale folded in: a = 1024 + c 2^P (decode_fp2 / decode_fp3_box), then 2c - K0 exactly
// (2^(1-P) a - (2^(11-P) + K0)), then the product with d rounded once.
template <int K0, int P>
__device__ __forceinline__ uint32_t tc_level(uint32_t a, uint32_t d2) {
    return hmul2_u(hfma2_u(a, f16x2(P + 0 >= 1 ? 2.0 / double(1 << P) : 1.0), f16x2(-(double(1 << (11 - P)) + K0))), d2);
}

// One code group: its 8 pairs into o[8 G .. 8 G + 7].
template <int FMT, int G, int NO>
__device__ __forceinline__ void tc_group(const uint32_t (&a)[8], uint32_t d2, int odd, uint32_t (&o)[NO]) {
    if constexpr (FMT == 2) {
        o[8 * G + 0] = tc_level<3, pair_shift(2, 0)>(a[0], d2); o[8 * G + 1] = tc_level<3, pair_shift(2, 1)>(a[1], d2);
        o[8 * G + 2] = tc_level<3, pair_shift(2, 2)>(a[2], d2); o[8 * G + 3] = tc_level<3, pair_shift(2, 3)>(a[3], d2);
        o[8 * G + 4] = tc_level<3, pair_shift(2, 4)>(a[4], d2); o[8 * G + 5] = tc_level<3, pair_shift(2, 5)>(a[5], d2);
        o[8 * G + 6] = tc_level<3, pair_shift(2, 6)>(a[6], d2); o[8 * G + 7] = tc_level<3, pair_shift(2, 7)>(a[7], d2);
    } else if (!odd) {
        o[8 * G + 0] = tc_level<7, fp3_box_shift(0, 0)>(a[0], d2); o[8 * G + 1] = tc_level<7, fp3_box_shift(0, 1)>(a[1], d2);
        o[8 * G + 2] = tc_level<7, fp3_box_shift(0, 2)>(a[2], d2); o[8 * G + 3] = tc_level<7, fp3_box_shift(0, 3)>(a[3], d2);
        o[8 * G + 4] = tc_level<7, fp3_box_shift(0, 4)>(a[4], d2); o[8 * G + 5] = tc_level<7, fp3_box_shift(0, 5)>(a[5], d2);
        o[8 * G + 6] = tc_level<7, fp3_box_shift(0, 6)>(a[6], d2); o[8 * G + 7] = tc_level<7, fp3_box_shift(0, 7)>(a[7], d2);
    } else {
        o[8 * G + 0] = tc_level<7, fp3_box_shift(1, 0)>(a[0], d2); o[8 * G + 1] = tc_level<7, fp3_box_shift(1, 1)>(a[1], d2);
        o[8 * G + 2] = tc_level<7, fp3_box_shift(1, 2)>(a[2], d2); o[8 * G + 3] = tc_level<7, fp3_box_shift(1, 3)>(a[3], d2);
        o[8 * G + 4] = tc_level<7, fp3_box_shift(1, 4)>(a[4], d2); o[8 * G + 5] = tc_level<7, fp3_box_shift(1, 5)>(a[5], d2);
        o[8 * G + 6] = tc_level<7, fp3_box_shift(1, 6)>(a[6], d2); o[8 * G + 7] = tc_level<7, fp3_box_shift(1, 7)>(a[7], d2);
    }
}

// Slab C (0..3) of a box row, code groups 2 p and 2 p + 1: cw[i] = the row's code words of group 2 p + i
// (FP2: 4 words, word C is the slab's; FP3: 6 words, slab pair C / 2 at 3 (C / 2)); sc = the row's
// binary16 scales 4 p + 0..3 (scale 4 p + C = block 2 C + p, both groups' block).
template <int FMT, int C, int NW>
__device__ __forceinline__ void tc_half_slab(const uint32_t (&cw)[2][NW], const uint2& sc, uint32_t magic, uint32_t (&o)[16]) {
    const uint32_t sw = C < 2 ? sc.x : sc.y;
    const uint32_t d = (C & 1) ? (sw >> 16) : (sw & 0xFFFFu);
    const uint32_t d2 = d | (d << 16);
    uint32_t a[8], b[8];
    if constexpr (FMT == 2) {
        decode_fp2(cw[0][C], magic, a); tc_group<2, 0>(a, d2, 0, o);
        decode_fp2(cw[1][C], magic, a); tc_group<2, 1>(a, d2, 0, o);
    } else {
        constexpr int m = C >> 1, odd = C & 1;
        decode_fp3_box(cw[0][3 * m], cw[0][3 * m + 1], cw[0][3 * m + 2], magic, a, b); tc_group<3, 0>(odd ? b : a, d2, odd, o);
        decode_fp3_box(cw[1][3 * m], cw[1][3 * m + 1], cw[1][3 * m + 2], magic, a, b); tc_group<3, 1>(odd ? b : a, d2, odd, o);
    }
}

// Accumulator placement of a unit (identical sequence in the MMA thread and the epilogue): a unit of
// n16 <= 64 columns takes buffer `toggle` (flipping it), a larger one both buffers.
struct TcAcc {
    uint32_t toggle = 0, uses0 = 0, uses1 = 0, full0 = 0, full1 = 0;
    // buffers mask, primary buffer, column of half h = col0 + h * hstep
    __device__ void place(uint32_t n16, uint32_t& mask, uint32_t& prim, uint32_t& col0, uint32_t& hstep) {
        if (n16 <= 64) {
            prim = toggle; mask = 1u << toggle; col0 = toggle * 128u; hstep = 64u;
            toggle ^= 1u;
        } else {
            prim = 0; mask = 3u; col0 = 0; hstep = 128u;
        }
    }
    __device__ uint32_t uses(int b) const { return b ? uses1 : uses0; }
    __device__ uint32_t fulls(uint32_t b) const { return b ? full1 : full0; }
    __device__ void done(uint32_t mask, uint32_t prim) {
        uses0 += mask & 1u;
        uses1 += mask >> 1;
        full0 += prim == 0u;
        full1 += prim == 1u;
    }
};

template <int FMT>
__global__ void __launch_bounds__(kTcThreads, 1) k_tcgemm(const __grid_constant__ TcArgs A) {
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr int kTcRS = tc_ring_slots(FMT), kTcBStages = tc_bstages(FMT), kTcBox = tc_slot_bytes(FMT);
    __shared__ uint64_t bars[2 * kTcMaxRS + 2 * kTcAStages + 2 * kTcMaxBS + 5];
    __shared__ uint32_t taddr_s;
    __shared__ float efac[kTcEpi][kTcN];  // per epilogue warp: 2^-shift of the unit's B rows
    uint8_t* base = smem + ((1024u - (smem_u32(smem) & 1023u)) & 1023u);
    uint8_t* Bs = base;
    uint8_t* ring = base + kTcBStages * kTcBStage;
    uint64_t* ring_full = bars;                   // [kTcRS]
    uint64_t* ring_empty = ring_full + kTcRS;     // [kTcRS], kTcDec arrivals
    uint64_t* a_full = ring_empty + kTcRS;        // [kTcAStages], kTcDec arrivals
    uint64_t* a_free = a_full + kTcAStages;       // [kTcAStages], one tcgen05.commit
    uint64_t* b_full = a_free + kTcAStages;       // [kTcBStages]
    uint64_t* b_free = b_full + kTcBStages;       // [kTcBStages], one tcgen05.commit
    uint64_t* acc_full = b_free + kTcBStages;     // [2], one tcgen05.commit
    uint64_t* acc_free = acc_full + 2;            // [2], kTcEpi arrivals
    uint64_t* done = acc_free + 2;                // the MMA thread's last commit
    const int tid = threadIdx.x, warp = tid / 32, lane = tid & 31;
    if (tid == 0) {
        for (int i = 0; i < kTcRS; i++) { mbar_init(ring_full + i, 1); mbar_init(ring_empty + i, kTcDec); }
        for (int i = 0; i < kTcAStages; i++) { mbar_init(a_full + i, kTcDec); mbar_init(a_free + i, kTcIss); }
        for (int i = 0; i < kTcBStages; i++) { mbar_init(b_full + i, 1); mbar_init(b_free + i, kTcIss); }
        for (int i = 0; i < 2; i++) { mbar_init(acc_full + i, kTcIss); mbar_init(acc_free + i, kTcEpi); }
        mbar_init(done, kTcIss);
    }
    fence_barrier_init();
    __syncthreads();
    if (warp == 2) tmem_alloc(smem_u32(&taddr_s), kTcCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t taddr = taddr_s;
    const int nunits = __ldg(A.nunits), G = gridDim.x, c = blockIdx.x;
    const int nslab = A.K / 64, nstage = A.K / kTcSK;

    if (warp < 2) {
        // ---------------------------------------------------------------- loads (one thread each, in
        // warps of their own so that neither waits while the other sleeps): warp 0 the packed boxes,
        // warp 1 the B slabs, each as far ahead as its own ring allows
        if (warp == 0 && lane == 0) {
            uint32_t gb = 0;
            bool live = true;
            for (int u = c; u < nunits && live; u += G) {
                const int4 un = A.units[u];
                const int nkb = A.K / stage_k(FMT);  // boxes along K
                const uint8_t* wb = A.W + (int64_t)un.x * A.mstride + (int64_t)un.w * (256 / stage_rows(FMT)) * nkb * stage_bytes(FMT);
                for (int bx = 0; bx < A.K / tc_slot_k(FMT); bx++, gb++) {
                    const uint32_t sl = gb % kTcRS;
                    if (gb >= (uint32_t)kTcRS && !mbar_wait(ring_empty + sl, ((gb / kTcRS) + 1u) & 1u)) { live = false; break; }
                    mbar_expect_tx(ring_full + sl, FMT == 4 ? 4 * stage_bytes(4) : stage_bytes(FMT));
                    if constexpr (FMT == 4) {
                        // the unit's four 64-row boxes at this K
                        for (int i = 0; i < 4; i++)
                            bulk_load(ring + sl * kTcBox + i * stage_bytes(4), wb + ((int64_t)i * nkb + bx) * stage_bytes(4),
                                      stage_bytes(4), ring_full + sl);
                    } else {
                        bulk_load(ring + sl * kTcBox, wb + (int64_t)bx * stage_bytes(FMT), stage_bytes(FMT), ring_full + sl);
                    }
                }
            }
            if (!live) flag(A.status, FPX_ETIMEOUT);
            // no copy may land after the CTA exits
            for (uint32_t i = gb > (uint32_t)kTcRS ? gb - kTcRS : 0u; i < gb; i++) mbar_wait(ring_full + i % kTcRS, (i / kTcRS) & 1u);
        } else if (warp == 1 && lane == 0) {
            uint32_t gs = 0;
            bool live = true;
            for (int u = c; u < nunits && live; u += G) {
                const int4 un = A.units[u];
                const int nt = (un.z + kTcBRows - 1) / kTcBRows;
                for (int j = 0; j < nstage; j++, gs++) {
                    const uint32_t st = gs % kTcBStages;
                    if (gs >= (uint32_t)kTcBStages && !mbar_wait(b_free + st, ((gs / kTcBStages) + 1u) & 1u)) { live = false; break; }
                    mbar_expect_tx(b_full + st, (uint32_t)(2 * nt * kTcBRows * 128));
                    for (int t = 0; t < 2; t++)
                        for (int r = 0; r < nt; r++)
                            tma_load_2d(Bs + st * kTcBStage + t * kTcBTile + r * (kTcBRows * 128), &A.bmap, kTcSK * j + 64 * t,
                                        un.y + r * kTcBRows, b_full + st);
                }
            }
            if (!live) flag(A.status, FPX_ETIMEOUT);
            for (uint32_t i = gs > (uint32_t)kTcBStages ? gs - kTcBStages : 0u; i < gs; i++) mbar_wait(b_full + i % kTcBStages, (i / kTcBStages) & 1u);
        }
    } else if (warp < 2 + kTcIss) {
        // ---------------------------------------------------------------- MMA issue (one thread per half)
        if (lane == 0) {
            const uint32_t h = (uint32_t)(warp - 2);
            uint32_t gs = 0;
            TcAcc acc;
            bool live = true, pre_a = false, pre_b = false;  // pre_*: stage gs's barrier already seen complete
            for (int u = c; u < nunits && live; u += G) {
                const int4 un = A.units[u];
                const uint32_t n16 = (uint32_t)((un.z + 15) & ~15), idesc = f16_idesc(128, n16);
                uint32_t mask, prim, col0, hstep;
                acc.place(n16, mask, prim, col0, hstep);
                for (int b = 0; b < 2; b++)
                    if (((mask >> b) & 1u) && acc.uses(b) > 0 && !mbar_wait(acc_free + b, (acc.uses(b) - 1u) & 1u)) live = false;
                if (!live) break;
                tc_fence_after();
                const uint32_t dcol = taddr + col0 + h * hstep;
                for (int j = 0; j < nstage && live; j++, gs++) {
                    const uint32_t sa = gs % kTcAStages, sb = gs % kTcBStages;
                    if ((!pre_a && !mbar_wait(a_full + sa, (gs / kTcAStages) & 1u)) ||
                        (!pre_b && !mbar_wait(b_full + sb, (gs / kTcBStages) & 1u))) {
                        live = false;
                        break;
                    }
                    tc_fence_after();
                    // test the next stage's barriers now: the answers arrive while this stage's MMAs issue
                    // (a blocking wait here would cost its full latency on every slab)
                    const uint32_t gn = gs + 1u;
                    pre_a = mbar_test_wait(a_full + gn % kTcAStages, (gn / kTcAStages) & 1u);
                    pre_b = mbar_test_wait(b_full + gn % kTcBStages, (gn / kTcBStages) & 1u);
                    const uint32_t a0 = taddr + kTcACol + 128u * sa + 64u * h;
                    // B: tile kk / 4 (16 KB = 1024 in the descriptor's address field), + 2 per K step of 32 bytes
                    const uint64_t bd = sw128_desc(smem_u32(Bs + sb * kTcBStage));
#pragma unroll
                    for (int kk = 0; kk < 8; kk++)
                        tc_mma_f16_ta(dcol, a0 + 8u * tc_kblock<FMT>(kk), bd + 1024u * (kk >> 2) + 2u * (kk & 3), idesc, (j | kk) != 0);
                    tc_commit(smem_u32(a_free + sa));
                    tc_commit(smem_u32(b_free + sb));
                }
                if (!live) break;
                tc_commit(smem_u32(acc_full + prim));
                acc.done(mask, prim);
            }
            if (!live) flag(A.status, FPX_ETIMEOUT);
            tc_commit(smem_u32(done));
        }
    } else if (warp < kTcDec0 + kTcDec) {
        // ---------------------------------------------------------------- decode (16 warps): a weight
        // row per thread, code groups 2 p, 2 p + 1 of every slab
        const int dw = warp - kTcDec0, q = warp & 3, h = (dw >> 2) & 1, p = dw >> 3;
        const int row = h * 128 + 32 * q + lane;
        const uint32_t lane_base = taddr + ((uint32_t)(32 * q) << 16) + kTcACol + 64u * (uint32_t)h + 32u * (uint32_t)p;
        // the row's two chunks are read in an order that depends on the lane, halving bank conflicts
        const uint32_t rot = (uint32_t)(lane >> 2) & 1u;
        constexpr int NW = FMT == 2 ? 4 : 6;  // code words of a group
        uint32_t gs = 0, gb = 0;
        bool live = true;
        const uint32_t magic = kMagic;
        uint32_t bad = 0;
        if constexpr (FMT == 4) {
            // A row of the unit lies in 64-row box row / 64 of the slot, at byte (row % 64) * 272; a stage
            // (128 K) holds blocks 4 S .. 4 S + 3 of the box row, 17 bytes each; this thread decodes blocks
            // 4 S + 2 p and 4 S + 2 p + 1 (one scale byte, then 16 bytes of two E2M1 codes each)
            const uint32_t row_ofs = (uint32_t)(row >> 6) * stage_bytes(4) + (uint32_t)(row & 63) * 272u;
            for (int u = c; u < nunits && live; u += G) {
                const int erow = __ldg(A.rowexp + A.units[u].w * 256 + row);
                for (int bx = 0; bx < A.K / 512 && live; bx++, gb++) {
                    const uint32_t sl = gb % kTcRS;
                    if (!__any_sync(0xffffffffu, mbar_wait(ring_full + sl, (gb / kTcRS) & 1u))) { live = false; break; }
                    const uint32_t rbase = smem_u32(ring + sl * kTcBox) + row_ofs;
#pragma unroll
                    for (int S = 0; S < 4; S++, gs++) {
                        // both blocks' scale bytes and codes (the codes realigned to words)
                        uint32_t e[2], cw[2][4];
#pragma unroll
                        for (int j = 0; j < 2; j++) {
                            const uint32_t ob = rbase + 17u * (uint32_t)(4 * S + 2 * p + j);
                            e[j] = lds8<0>(ob);
                            const uint32_t cb = (ob + 1u) & ~3u, cs = 8u * ((ob + 1u) & 3u);
                            uint32_t x[5];
#pragma unroll
                            for (int i = 0; i < 5; i++) x[i] = lds32<0>(cb + 4u * (uint32_t)i);
#pragma unroll
                            for (int i = 0; i < 4; i++) cw[j][i] = __funnelshift_r(x[i], x[i + 1], cs);
                        }
                        if (S == 3) {
                            __syncwarp();
                            if (lane == 0) mbar_arrive(ring_empty + sl);
                        }
                        uint32_t o[32];
#pragma unroll
                        for (int j = 0; j < 2; j++) {
                            // 2^(e - erow + 15) in binary16 (normal, subnormal or zero): times the decoded
                            // E2M1 value * 2^-14 gives value * 2^(e - erow + 1), exact while normal
                            const int f = (int)e[j] - erow + 30;
                            uint32_t mb = f >= 1 ? (uint32_t)f << 10 : f >= -9 ? 1u << (f + 9) : 0u;
                            if (e[j] == 255u) { mb = 0u; bad = 1u; }
                            const uint32_t m2 = mb | (mb << 16);
                            uint32_t a[8];
                            decode_fp4(cw[j][0], cw[j][1], a);
#pragma unroll
                            for (int k = 0; k < 8; k++) o[16 * j + k] = hmul2_u(a[k], m2);
                            decode_fp4(cw[j][2], cw[j][3], a);
#pragma unroll
                            for (int k = 0; k < 8; k++) o[16 * j + 8 + k] = hmul2_u(a[k], m2);
                        }
                        const uint32_t st = gs % kTcAStages;
                        if (live && gs >= (uint32_t)kTcAStages)
                            live = __any_sync(0xffffffffu, mbar_wait(a_free + st, ((gs / kTcAStages) + 1u) & 1u));
                        if (!live) break;
                        tc_fence_after();
                        tmem_st32(lane_base + 128u * st, o);
                        tmem_st_wait();
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(a_full + st);
                    }
                }
            }
        } else {
        for (int u = c; u < nunits && live; u += G) {
            for (int bx = 0; bx < nslab / 4 && live; bx++, gb++) {
                const uint32_t sl = gb % kTcRS;
                if (!__any_sync(0xffffffffu, mbar_wait(ring_full + sl, (gb / kTcRS) & 1u))) { live = false; break; }
                const uint32_t box = smem_u32(ring + sl * kTcBox);
                uint32_t v[2][NW], cw[2][NW];
#pragma unroll
                for (int i = 0; i < 2; i++) {
                    const uint32_t g = 2u * (uint32_t)p + (((uint32_t)i + rot) & 1u);
                    if constexpr (FMT == 2) {
                        const uint4 x = lds128<0>(box + (uint32_t)row * 64u + 16u * g);
                        v[i][0] = x.x; v[i][1] = x.y; v[i][2] = x.z; v[i][3] = x.w;
                    } else {
                        const uint32_t cb = box + (uint32_t)row * 96u + 24u * g;
                        const uint2 x0 = lds64<0>(cb), x1 = lds64<8>(cb), x2 = lds64<16>(cb);
                        v[i][0] = x0.x; v[i][1] = x0.y; v[i][2] = x1.x; v[i][3] = x1.y; v[i][4] = x2.x; v[i][5] = x2.y;
                    }
                }
                // scales 4 p + C (C = 0..3) of the row: blocks 2 C + p
                const uint2 sc = lds64<0>(box + (uint32_t)(box_scale_offset(FMT) + row * 16 + 8 * p));
                __syncwarp();
                if (lane == 0) mbar_arrive(ring_empty + sl);
#pragma unroll
                for (int w = 0; w < NW; w++) {
                    cw[0][w] = rot ? v[1][w] : v[0][w];
                    cw[1][w] = rot ? v[0][w] : v[1][w];
                }
                // the box's two stages: slabs 0, 1 and 2, 3
#pragma unroll
                for (int S = 0; S < 2; S++, gs++) {
                    // decode first, then wait for the stage: the decode overlaps the MMAs that still
                    // read the stage, so it is not on the stage's round trip
                    uint32_t o[32];
                    uint32_t(&o0)[16] = *reinterpret_cast<uint32_t(*)[16]>(&o[0]);
                    uint32_t(&o1)[16] = *reinterpret_cast<uint32_t(*)[16]>(&o[16]);
                    if (S == 0) {
                        tc_half_slab<FMT, 0>(cw, sc, magic, o0);
                        tc_half_slab<FMT, 1>(cw, sc, magic, o1);
                    } else {
                        tc_half_slab<FMT, 2>(cw, sc, magic, o0);
                        tc_half_slab<FMT, 3>(cw, sc, magic, o1);
                    }
                    const uint32_t st = gs % kTcAStages;
                    if (live && gs >= (uint32_t)kTcAStages)
                        live = __any_sync(0xffffffffu, mbar_wait(a_free + st, ((gs / kTcAStages) + 1u) & 1u));
                    if (!live) break;
                    tc_fence_after();
                    tmem_st32(lane_base + 128u * st, o);
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(a_full + st);
                }
            }
        }
        }
        if (!live && lane == 0) flag(A.status, FPX_ETIMEOUT);
        if (__any_sync(0xffffffffu, bad != 0u) && lane == 0) flag(A.status, FPX_EDATA);
    } else {
        // ---------------------------------------------------------------- epilogue (4 warps)
        const int q = warp & 3;  // tensor-memory lane quarter of this warp
        float* fac = efac[warp - kTcDec0 - kTcDec];
        TcAcc acc;
        bool live = true;
        for (int u = c; u < nunits && live; u += G) {
            const int4 un = A.units[u];
            const int n = un.z, n16 = (n + 15) & ~15;
            // the unit's column factors 2^-shift, read before the accumulator is ready
            __syncwarp();
            for (int s = lane; s < n; s += 32) fac[s] = exp2i(-__ldg(A.shift + un.y + s));
            __syncwarp();
            uint32_t mask, prim, col0, hstep;
            acc.place((uint32_t)n16, mask, prim, col0, hstep);
            live = __any_sync(0xffffffffu, mbar_wait(acc_full + prim, acc.fulls(prim) & 1u));
            if (!live) break;
            tc_fence_after();
            for (int hh = 0; hh < 2; hh++) {
                const int m = un.w * 256 + hh * 128 + 32 * q + lane;
                float* orow = A.out + (size_t)un.y * A.M + m;
                // FP4: the decode scaled row m by 2^(128 - rowexp[m]); undo it with the column factor
                const float rf = FMT == 4 ? exp2i(__ldg(A.rowexp + m) - 128) : 1.0f;
                for (int c0 = 0; c0 < n16; c0 += 16) {
                    float v[16];
                    tmem_ld16(taddr + ((uint32_t)(32 * q) << 16) + col0 + hstep * (uint32_t)hh + (uint32_t)c0, v);
#pragma unroll
                    for (int j = 0; j < 16; j++) {
                        const int s = c0 + j;
                        if (s < n) orow[(size_t)s * A.M] = v[j] * (fac[s] * rf);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                for (int b = 0; b < 2; b++)
                    if ((mask >> b) & 1u) mbar_arrive(acc_free + b);
            acc.done(mask, prim);
        }
        if (!live && lane == 0) flag(A.status, FPX_ETIMEOUT);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 2) {
        mbar_wait(done, 0);  // every MMA of this CTA has completed
        tmem_dealloc(taddr, kTcCols);
    }
}

// B rows for the routed gate/up GEMMs: xg[s] = the binary16 activation row of pair perm[s]'s token,
// each 16-element group stored in the decode's pair order (element p, then p + 8), and its scale
// exponent gshift[s]. One warp per row.
__global__ void __launch_bounds__(256) k_pgather(const __half* __restrict__ x16, const int32_t* __restrict__ shx,
                                                 const int32_t* __restrict__ perm, int P, int k, int H, __half* __restrict__ xg,
                                                 int32_t* __restrict__ gshift) {
    const int s = blockIdx.x * 8 + threadIdx.x / 32, lane = threadIdx.x & 31;
    if (s >= P) return;
    const int tok = perm[s] / k;
    if (lane == 0) gshift[s] = shx[tok];
    const uint4* src = reinterpret_cast<const uint4*>(x16 + (size_t)tok * H);
    uint4* dst = reinterpret_cast<uint4*>(xg + (size_t)s * H);
    for (int gi = lane; gi < H / 16; gi += 32) {
        const uint4 a = src[2 * gi], b = src[2 * gi + 1];
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        uint32_t o[8];
#pragma unroll
        for (int p = 0; p < 8; p++) o[p] = __byte_perm(w[p >> 1], w[4 + (p >> 1)], (p & 1) ? 0x7632u : 0x5410u);
        dst[2 * gi] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[2 * gi + 1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

// The tensor-core GEMM units of the routed experts: for every expert with pairs, its pairs in tiles of
// up to 128 (in sorted order), times the M / 256 row blocks; the row blocks of a tile are consecutive,
// so CTAs working at the same time share B tiles in L2. One CTA of 1024 threads (E <= 1024).
__global__ void __launch_bounds__(1024) k_tcunits(const int32_t* __restrict__ offsets, int E, int MT, int4* units,
                                                  int32_t* nunits) {
    __shared__ int part[32];
    const int e = threadIdx.x, lane = e & 31, wid = e / 32;
    const int n = e < E ? offsets[e + 1] - offsets[e] : 0, nt = (n + kTcN - 1) / kTcN;
    int incl = nt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) part[wid] = incl;
    __syncthreads();
    int before = 0;
    for (int w = 0; w < wid; w++) before += part[w];
    const int base = before + incl - nt;
    for (int i = 0; i < nt; i++)
        for (int mt = 0; mt < MT; mt++) {
            const int s0 = offsets[e] + i * kTcN;
            units[(size_t)(base + i) * MT + mt] = make_int4(e, s0, min(kTcN, offsets[e + 1] - s0), mt);
        }
    if (e == 1023) {
        int tot = 0;
        for (int w = 0; w < 32; w++) tot += part[w];
        *nunits = tot * MT;
    }
}

// h = silu(g) u for rows [0, Pr) of (g, u) -> binary16 rows scaled by 2^sh(row) (exact shift), shift[row].
// Each 16-element group is stored in a tensor-core decode's pair order (element lo(p), then lo(p) + D
// at positions 2 p, 2 p + 1): PERM 1 the FP2 / FP3 order (lo(p) = p, D = 8), PERM 2 the FP4 order
// (lo(p) = p + 4 (p / 4), D = 4).
template <int PERM>
__global__ void __launch_bounds__(256) k_ph(const float* __restrict__ g, const float* __restrict__ u, int L,
                                            __half* __restrict__ h16, int32_t* __restrict__ shift) {
    __shared__ __align__(16) float h_s[4608];  // the row's h (L <= 4608), so g and u are read once
    __shared__ float red[8];
    __shared__ int sh_s;
    const size_t r = blockIdx.x;
    float m = 0.f;
    const float4* g4 = reinterpret_cast<const float4*>(g + r * L);
    const float4* u4 = reinterpret_cast<const float4*>(u + r * L);
    for (int i = threadIdx.x; i < L / 4; i += blockDim.x) {
        const float4 a = __ldcs(g4 + i), b = __ldcs(u4 + i);
        float4 h;
        h.x = (a.x / (1.0f + expf(-a.x))) * b.x;
        h.y = (a.y / (1.0f + expf(-a.y))) * b.y;
        h.z = (a.z / (1.0f + expf(-a.z))) * b.z;
        h.w = (a.w / (1.0f + expf(-a.w))) * b.w;
        m = fmaxf(m, fmaxf(fmaxf(fabsf(h.x), fabsf(h.y)), fmaxf(fabsf(h.z), fabsf(h.w))));
        reinterpret_cast<float4*>(h_s)[i] = h;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x / 32] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float mm = 0.f;
        for (int i = 0; i < 8; i++) mm = fmaxf(mm, red[i]);
        sh_s = column_shift(mm);
        shift[r] = sh_s;
    }
    __syncthreads();
    const float sc = exp2i(sh_s);
    for (int gi = threadIdx.x; gi < L / 16; gi += blockDim.x) {
        float v[16];
#pragma unroll
        for (int j = 0; j < 16; j++) v[j] = h_s[16 * gi + j] * sc;
        uint32_t o[8];
#pragma unroll
        for (int p = 0; p < 8; p++) {
            const int lo = PERM == 1 ? p : p + 4 * (p >> 2), hi = lo + (PERM == 1 ? 8 : 4);
            const __half2 hp = __halves2half2(__float2half_rn(v[lo]), __float2half_rn(v[hi]));
            o[p] = *reinterpret_cast<const uint32_t*>(&hp);
        }
        uint4* dst = reinterpret_cast<uint4*>(h16 + r * L + 16 * gi);
        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

// dst row r = src row r (binary16 [R][L]) with each 16-element group in the FP4 decode's pair order
// (elements p + 4 (p / 4) and p + 4 (p / 4) + 4 at positions 2 p, 2 p + 1). One thread per group.
__global__ void __launch_bounds__(256) k_perm4(const __half* __restrict__ src, int64_t ngroups, __half* __restrict__ dst) {
    const int64_t gi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (gi >= ngroups) return;
    const uint4 a = reinterpret_cast<const uint4*>(src)[2 * gi], b = reinterpret_cast<const uint4*>(src)[2 * gi + 1];
    // words: a = elements (0,1)(2,3)(4,5)(6,7), b = (8,9) .. (14,15); pair p of each 8: (k, k + 4)
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t o[8];
#pragma unroll
    for (int p = 0; p < 8; p++) {
        const int lo = p + 4 * (p >> 2), hi = lo + 4;
        const uint32_t wl = w[lo >> 1], wh = w[hi >> 1];
        o[p] = __byte_perm(wl, wh, ((lo & 1) ? 0x0032u : 0x0010u) | ((hi & 1) ? 0x7600u : 0x5400u));
    }
    reinterpret_cast<uint4*>(dst)[2 * gi] = make_uint4(o[0], o[1], o[2], o[3]);
    reinterpret_cast<uint4*>(dst)[2 * gi + 1] = make_uint4(o[4], o[5], o[6], o[7]);
}

// rowexp[m] = the largest block exponent e != 255 of row m of a box-tiled FP4 matrix [M][K] (0 when
// none): the tensor-core decode scales row m by 2^(128 - rowexp[m]) to keep it in binary16 range. One
// warp per row; blockIdx.y picks one of three matrices.
struct RowExpArgs {
    const uint8_t* W[3];
    int M[3], K[3];
    int32_t* out[3];
};
__global__ void __launch_bounds__(256) k_fp4_rowexp(const __grid_constant__ RowExpArgs A) {
    const int mi = blockIdx.y, row = blockIdx.x * 8 + threadIdx.x / 32, lane = threadIdx.x & 31;
    const int M = A.M[mi], K = A.K[mi];
    if (row >= M) return;
    const int nkb = K / 512;
    const uint8_t* rb = A.W[mi] + (int64_t)(row >> 6) * nkb * stage_bytes(4) + (row & 63) * 272;
    int e = 0;
    for (int b = lane; b < K / 32; b += 32) {
        const int v = __ldg(rb + (int64_t)(b >> 4) * stage_bytes(4) + 17 * (b & 15));
        if (v != 255) e = max(e, v);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) e = max(e, __shfl_xor_sync(0xffffffffu, e, o));
    if (lane == 0) A.out[mi][row] = e;
}

// Units of a dense GEMM over T rows of B (the shared expert): tiles of 128 rows, times MT 256-row
// blocks of the weights, row blocks of a tile consecutive.
__global__ void k_tcunits_dense(int T, int MT, int4* units, int32_t* nunits) {
    const int nt = (T + kTcN - 1) / kTcN;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < nt * MT; i += gridDim.x * blockDim.x) {
        const int t = i / MT, mt = i % MT;
        units[i] = make_int4(0, t * kTcN, min(kTcN, T - t * kTcN), mt);
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) *nunits = nt * MT;
}

// out[t][c] = sum_r w[t][r] * yp[inv[t*k + r]][c] (ranks in order) + ysh[t][c].
__global__ void __launch_bounds__(256) k_pcombine(const float* __restrict__ yp, const float* __restrict__ ysh,
                                                  const float* __restrict__ w, const int32_t* __restrict__ inv, int T,
                                                  int H, int k, float* __restrict__ out) {
    const size_t o = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (o >= (size_t)T * H) return;
    const int t = (int)(o / H), c = (int)(o % H);
    float v[kPMaxK];
#pragma unroll
    for (int r = 0; r < kPMaxK; r++) v[r] = r < k ? yp[(size_t)inv[(size_t)t * k + r] * H + c] : 0.f;
    float acc = 0.f;
#pragma unroll
    for (int r = 0; r < kPMaxK; r++)
        if (r < k) acc = r == 0 ? w[(size_t)t * k] * v[0] : fmaf(w[(size_t)t * k + r], v[r], acc);
    out[o] = acc + ysh[o];
}

// ------------------------------------------------------------------ router logits on tcgen05

// logits[t][e] = sum_h R[e][h] x[t][h] on the tensor cores: R (binary32) is split into three
// bfloat16 parts R = R1 + R2 + R3 (exact: 3 x 8 significant bits), every product of a part with the
// bfloat16 activation is exact in binary32, and the tensor core sums the three parts' products over h
// in binary32. The sum runs in the same order for every (t, e), so equal router rows give equal
// logits. CTA = 128 experts x 64 tokens: warp 0 streams 64-wide K slabs of the three parts and of x
// (2-D TMA tiles, 128-byte swizzle) into a 3-stage ring, warp 1 issues 3 x 4 MMAs of 128 x 64 x 16
// per slab (bfloat16 inputs, binary32 accumulator in tensor memory), warps 2..5 write the logits.
constexpr int kLgM = 128, kLgN = 64, kLgStages = 3, kLgThreads = 6 * 32;
constexpr int kLgA = kLgM * 128, kLgB = kLgN * 128;               // one part's tile, the token tile
constexpr int kLgStage = 3 * kLgA + kLgB;
constexpr int kLgSmem = kLgStages * kLgStage + 1024;
static_assert(kLgSmem <= 227 * 1024 && kLgStage % 1024 == 0, "logit GEMM shared memory");

// r[i] -> three bfloat16 parts (rows [p][E][H] of rs): r1 = RN(r), r2 = RN(r - r1), r3 = RN(r - r1 - r2)
__global__ void __launch_bounds__(256) k_rsplit(const float* __restrict__ r, int64_t n, __nv_bfloat16* __restrict__ rs) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const float v = r[i];
    const __nv_bfloat16 a = __float2bfloat16_rn(v);
    const float d1 = v - __bfloat162float(a);  // exact (Sterbenz / the low bits of v)
    const __nv_bfloat16 b = __float2bfloat16_rn(d1);
    const __nv_bfloat16 c = __float2bfloat16_rn(d1 - __bfloat162float(b));
    rs[i] = a;
    rs[n + i] = b;
    rs[2 * n + i] = c;
}

struct LgArgs {
    CUtensorMap amap;  // rs: bfloat16 [3 E][H], box 64 x 128
    CUtensorMap bmap;  // x: bfloat16 [T][H], box 64 x 64
    int T, E, H;
    float* logits;
    int32_t* status;
};

__global__ void __launch_bounds__(kLgThreads, 1) k_plogits_tc(const __grid_constant__ LgArgs A) {
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ uint64_t full[kLgStages], empty[kLgStages], done;
    __shared__ uint32_t taddr_s;
    uint8_t* base = smem + ((1024u - (smem_u32(smem) & 1023u)) & 1023u);
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    const int e0 = blockIdx.x * kLgM, t0 = blockIdx.y * kLgN, nslab = A.H / 64;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kLgStages; i++) { mbar_init(full + i, 1); mbar_init(empty + i, 1); }
        mbar_init(&done, 1);
    }
    fence_barrier_init();
    __syncthreads();
    if (warp == 1) tmem_alloc(smem_u32(&taddr_s), kLgN);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t taddr = taddr_s;
    if (warp == 0) {
        if (lane == 0) {
            bool live = true;
            for (int j = 0; j < nslab && live; j++) {
                const int st = j % kLgStages;
                if (j >= kLgStages && !mbar_wait(empty + st, ((j / kLgStages) + 1) & 1)) { live = false; break; }
                uint8_t* sb = base + st * kLgStage;
                mbar_expect_tx(full + st, kLgStage);
                for (int p = 0; p < 3; p++) tma_load_2d(sb + p * kLgA, &A.amap, 64 * j, p * A.E + e0, full + st);
                tma_load_2d(sb + 3 * kLgA, &A.bmap, 64 * j, t0, full + st);
            }
            if (!live) flag(A.status, FPX_ETIMEOUT);
            const int j0 = nslab > kLgStages ? nslab - kLgStages : 0;
            for (int j = j0; j < nslab; j++) mbar_wait(full + j % kLgStages, (j / kLgStages) & 1);  // no copy outlives the CTA
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // binary32 accumulator, bfloat16 A and B (bits 7-9 and 10-12 = 1), K-major, N / 8, M / 16
            const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kLgN >> 3) << 17) | ((uint32_t)(kLgM >> 4) << 24);
            bool live = true;
            for (int j = 0; j < nslab && live; j++) {
                const int st = j % kLgStages;
                if (!mbar_wait(full + st, (j / kLgStages) & 1)) { live = false; break; }
                tc_fence_after();
                const uint32_t sb = smem_u32(base + st * kLgStage);
                const uint64_t bd = sw128_desc(sb + 3 * kLgA);
#pragma unroll
                for (int kk = 0; kk < 4; kk++)
#pragma unroll
                    for (int p = 0; p < 3; p++)
                        tc_mma_f16(taddr, sw128_desc(sb + p * kLgA) + 2u * kk, bd + 2u * kk, idesc, (j | kk | p) != 0);
                tc_commit(smem_u32(empty + st));
            }
            if (!live) flag(A.status, FPX_ETIMEOUT);
            tc_commit(smem_u32(&done));
        }
    } else {
        // epilogue: warp w reads tensor-memory lanes 32 (w % 4) .. + 31 = experts e0 + 32 (w % 4) + lane
        const int q = warp & 3;
        const bool ok = __any_sync(0xffffffffu, mbar_wait(&done, 0));
        if (!ok) { if (lane == 0) flag(A.status, FPX_ETIMEOUT); }
        else {
            tc_fence_after();
            const int e = e0 + 32 * q + lane;
            for (int c0 = 0; c0 < kLgN; c0 += 16) {
                float v[16];
                tmem_ld16(taddr + ((uint32_t)(32 * q) << 16) + (uint32_t)c0, v);
#pragma unroll
                for (int i = 0; i < 16; i++) {
                    const int t = t0 + c0 + i;
                    if (t < A.T && e < A.E) A.logits[(size_t)t * A.E + e] = v[i];
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        mbar_wait(&done, 0);  // every MMA has completed
        tmem_dealloc(taddr, kLgN);
    }
}

// A 2-D tensor map over a bfloat16 [rows][K] matrix with box 64 x box_rows and the 128-byte swizzle;
// rows past the end read as zeros.
int make_bf16_map(CUtensorMap* m, const void* p, int64_t rows, int64_t K, int box_rows) {
    auto enc = tensor_map_encoder();
    if (!enc) return FPX_ECUDA;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(K * 2)};
    cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t es[2] = {1u, 1u};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(p), dims, strides, box, es,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FPX_OK : FPX_ECUDA;
}

// A 2-D tensor map over B (binary16 [rows][K]) for the tensor-core GEMM: boxes of 64 elements x 16
// rows with the 128-byte swizzle; rows past the end read as zeros.
int make_b_map(CUtensorMap* m, const __half* B, int64_t rows, int64_t K) {
    auto enc = tensor_map_encoder();
    if (!enc) return FPX_ECUDA;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(K * 2)};
    cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(kTcBRows)};
    cuuint32_t es[2] = {1u, 1u};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<__half*>(B), dims, strides, box, es,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FPX_OK : FPX_ECUDA;
}

template <int FMT>
int launch_tc(TcArgs& a, const __half* B, int64_t rows, cudaStream_t s) {
    int st = make_b_map(&a.bmap, B, rows, a.K);
    if (st) return st;
    if (cudaFuncSetAttribute(k_tcgemm<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, tc_smem(FMT)) != cudaSuccess) return FPX_ECUDA;
    k_tcgemm<FMT><<<device_info().sms, kTcThreads, tc_smem(FMT), s>>>(a);
    return cudaGetLastError() == cudaSuccess ? FPX_OK : FPX_ECUDA;
}

}  // namespace

extern "C" {

size_t moe_prefill_workspace_bytes(const moe_layer* L, int T, int k) {
    if (!L || T < 1 || k < 1 || k > kPMaxK || L->E < 1) return 0;
    return pws_layout(T, L->E, L->H, L->I, k).total;
}

int moe_layer_prefill(const moe_layer* L, const uint16_t* x, int T, int k, float* y, int32_t* idx_out, float* w_out,
                      float* logits_out, int32_t* perm_out, int32_t* offsets_out, void* ws, size_t ws_bytes,
                      void* stream) {
    if (!L || T < 1 || k < 1 || k > kPMaxK || L->E < k || L->E > kRouteMaxE) return FPX_EINVAL;
    const int H = L->H, I = L->I, E = L->E;
    if (H < 512 || I < 512 || H % 512 || I % 512 || I > 4608) return FPX_EINVAL;
    if ((int64_t)T * k > INT32_MAX / 2 || (int64_t)T * H > INT32_MAX) return FPX_EINVAL;
    if (!x || !y || !ws || !L->router || !L->gate || !L->up || !L->down || !L->sh_gate || !L->sh_up || !L->sh_down)
        return FPX_EINVAL;
    if (!aligned(ws, 16) || !aligned(x, 16) || !aligned(y, 16) || !aligned(L->gate, 16) || !aligned(L->up, 16) ||
        !aligned(L->down, 16) || !aligned(L->sh_gate, 16) || !aligned(L->sh_up, 16) || !aligned(L->sh_down, 16) ||
        !aligned(L->router, 16))
        return FPX_EALIGN;
    const PWs W = pws_layout(T, E, H, I, k);
    if (ws_bytes < W.total) return FPX_ESPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* b = static_cast<uint8_t*>(ws);
    int32_t* status = reinterpret_cast<int32_t*>(b + W.status);
    float* logits = reinterpret_cast<float*>(b + W.logits);
    int32_t* idx = reinterpret_cast<int32_t*>(b + W.idx);
    float* w = reinterpret_cast<float*>(b + W.w);
    int32_t* counts = reinterpret_cast<int32_t*>(b + W.counts);
    int32_t* offsets = reinterpret_cast<int32_t*>(b + W.offsets);
    int32_t* perm = reinterpret_cast<int32_t*>(b + W.perm);
    int32_t* inv = reinterpret_cast<int32_t*>(b + W.inv);
    __half* x16 = reinterpret_cast<__half*>(b + W.x16);
    int32_t* shx = reinterpret_cast<int32_t*>(b + W.shx);
    float* g = reinterpret_cast<float*>(b + W.g);
    float* u = reinterpret_cast<float*>(b + W.u);
    float* gsh = reinterpret_cast<float*>(b + W.gsh);
    float* ush = reinterpret_cast<float*>(b + W.ush);
    __half* h16 = reinterpret_cast<__half*>(b + W.h16);
    int32_t* shh = reinterpret_cast<int32_t*>(b + W.shh);
    __half* hsh16 = reinterpret_cast<__half*>(b + W.hsh16);
    int32_t* shsh = reinterpret_cast<int32_t*>(b + W.shsh);
    float* yp = reinterpret_cast<float*>(b + W.yp);
    float* ysh = reinterpret_cast<float*>(b + W.ysh);
    __half* xg = reinterpret_cast<__half*>(b + W.xg);
    int32_t* gshift = reinterpret_cast<int32_t*>(b + W.gshift);
    int4* tcu_gu = reinterpret_cast<int4*>(b + W.tcu_gu);
    int4* tcu_dn = reinterpret_cast<int4*>(b + W.tcu_dn);
    int32_t* ntc = reinterpret_cast<int32_t*>(b + W.ntc);
    __half* xs4 = reinterpret_cast<__half*>(b + W.xs4);
    int32_t* rexp = reinterpret_cast<int32_t*>(b + W.rexp);
    int4* tcu_sgu = reinterpret_cast<int4*>(b + W.tcu_sgu);
    int4* tcu_sdn = reinterpret_cast<int4*>(b + W.tcu_sdn);
    const int P = T * k;

    if (cudaMemsetAsync(status, 0, 16, s) != cudaSuccess || cudaMemsetAsync(counts, 0, 4 * (E + 1), s) != cudaSuccess)
        return FPX_ECUDA;
    k_to_f16<false><<<T, 256, 0, s>>>(x, H, x16, shx);
    {
        __nv_bfloat16* rs = reinterpret_cast<__nv_bfloat16*>(b + W.rsplit);
        const int64_t n = (int64_t)E * H;
        k_rsplit<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(L->router, n, rs);
        LgArgs la{};
        la.T = T; la.E = E; la.H = H; la.logits = logits; la.status = status;
        if (make_bf16_map(&la.amap, rs, 3 * (int64_t)E, H, kLgM) || make_bf16_map(&la.bmap, x, T, H, kLgN)) return FPX_ECUDA;
        if (cudaFuncSetAttribute(k_plogits_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, kLgSmem) != cudaSuccess) return FPX_ECUDA;
        k_plogits_tc<<<dim3((E + kLgM - 1) / kLgM, (T + kLgN - 1) / kLgN), kLgThreads, kLgSmem, s>>>(la);
    }
    k_ptopk<<<(T + 7) / 8, 256, 0, s>>>(logits, T, E, k, idx, w);
    k_phist<<<(P + 255) / 256, 256, 0, s>>>(idx, P, E, counts, status);
    k_pscan<<<1, 1024, 0, s>>>(counts, E, offsets);
    k_pscatter<<<E, 256, 0, s>>>(idx, P, offsets, perm, inv);
    if (cudaGetLastError() != cudaSuccess) return FPX_ECUDA;

    const int64_t mb2 = fpx_matrix_bytes(2, I, H), mb3 = fpx_matrix_bytes(3, H, I);
    // routed experts on the tcgen05 tensor cores: activations gathered per pair in expert order
    k_pgather<<<(P + 7) / 8, 256, 0, s>>>(x16, shx, perm, P, k, H, xg, gshift);
    k_tcunits<<<1, 1024, 0, s>>>(offsets, E, I / 256, tcu_gu, ntc);
    k_tcunits<<<1, 1024, 0, s>>>(offsets, E, H / 256, tcu_dn, ntc + 1);
    if (cudaGetLastError() != cudaSuccess) return FPX_ECUDA;
    TcArgs ta{};
    ta.status = status;
    ta.M = I; ta.K = H; ta.units = tcu_gu; ta.nunits = ntc; ta.shift = gshift; ta.mstride = mb2;
    ta.W = L->gate; ta.out = g;
    int st = launch_tc<2>(ta, xg, P, s);
    if (st) return st;
    ta.W = L->up; ta.out = u;
    if ((st = launch_tc<2>(ta, xg, P, s))) return st;
    // shared gate and up (FP4): every token, on the tensor cores as well; the rows' exponents, the
    // tokens in the FP4 decode's pair order and the dense units first
    RowExpArgs rea{};
    rea.W[0] = L->sh_gate; rea.W[1] = L->sh_up; rea.W[2] = L->sh_down;
    rea.M[0] = I; rea.M[1] = I; rea.M[2] = H;
    rea.K[0] = H; rea.K[1] = H; rea.K[2] = I;
    rea.out[0] = rexp; rea.out[1] = rexp + I; rea.out[2] = rexp + 2 * I;
    k_fp4_rowexp<<<dim3((unsigned)((std::max(H, I) + 7) / 8), 3), 256, 0, s>>>(rea);
    k_perm4<<<(unsigned)(((int64_t)T * H / 16 + 255) / 256), 256, 0, s>>>(x16, (int64_t)T * H / 16, xs4);
    k_tcunits_dense<<<1, 256, 0, s>>>(T, I / 256, tcu_sgu, ntc + 2);
    k_tcunits_dense<<<1, 256, 0, s>>>(T, H / 256, tcu_sdn, ntc + 3);
    if (cudaGetLastError() != cudaSuccess) return FPX_ECUDA;
    TcArgs sa{};
    sa.status = status;
    sa.M = I; sa.K = H; sa.units = tcu_sgu; sa.nunits = ntc + 2; sa.shift = shx; sa.mstride = 0;
    sa.W = L->sh_gate; sa.rowexp = rexp; sa.out = gsh;
    if ((st = launch_tc<4>(sa, xs4, T, s))) return st;
    sa.W = L->sh_up; sa.rowexp = rexp + I; sa.out = ush;
    if ((st = launch_tc<4>(sa, xs4, T, s))) return st;
    // h in binary16 with per-row scales (routed rows K-permuted for the tensor-core GEMM)
    k_ph<1><<<P, 256, 0, s>>>(g, u, I, h16, shh);
    k_ph<2><<<T, 256, 0, s>>>(gsh, ush, I, hsh16, shsh);
    if (cudaGetLastError() != cudaSuccess) return FPX_ECUDA;
    // routed down: h rows already in expert order
    TcArgs tda = ta;
    tda.M = H; tda.K = I; tda.units = tcu_dn; tda.nunits = ntc + 1; tda.shift = shh; tda.mstride = mb3;
    tda.W = L->down; tda.out = yp;
    if ((st = launch_tc<3>(tda, h16, P, s))) return st;
    TcArgs dsa = sa;
    dsa.M = H; dsa.K = I; dsa.units = tcu_sdn; dsa.nunits = ntc + 3; dsa.shift = shsh;
    dsa.W = L->sh_down; dsa.rowexp = rexp + 2 * I; dsa.out = ysh;
    if ((st = launch_tc<4>(dsa, hsh16, T, s))) return st;
    k_pcombine<<<(unsigned)(((size_t)T * H + 255) / 256), 256, 0, s>>>(yp, ysh, w, inv, T, H, k, y);
    if (idx_out && cudaMemcpyAsync(idx_out, idx, 4 * (size_t)P, cudaMemcpyDeviceToDevice, s) != cudaSuccess) return FPX_ECUDA;
    if (w_out && cudaMemcpyAsync(w_out, w, 4 * (size_t)P, cudaMemcpyDeviceToDevice, s) != cudaSuccess) return FPX_ECUDA;
    if (logits_out && cudaMemcpyAsync(logits_out, logits, 4 * (size_t)T * E, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
        return FPX_ECUDA;
    if (perm_out && cudaMemcpyAsync(perm_out, perm, 4 * (size_t)P, cudaMemcpyDeviceToDevice, s) != cudaSuccess) return FPX_ECUDA;
    if (offsets_out && cudaMemcpyAsync(offsets_out, offsets, 4 * (size_t)(E + 1), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
        return FPX_ECUDA;
    return cudaGetLastError() == cudaSuccess ? FPX_OK : FPX_ECUDA;
}

}  // extern "C"
