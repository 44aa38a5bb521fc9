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
//   k_px16     x (bfloat16) -> binary16 rows scaled by a per-token power of two (exact), + shifts
//   k_plogits  logits[t][e] = sum_h R[e][h] x[t][h], binary32, fixed order over h
//   k_ptopk    one warp per token: top-k by logit (ties to the lower index), sigmoid weights
//   k_phist / k_pscan / k_pscatter: stable counting sort of the T*k pairs p = t*k + r by expert:
//              perm[s] = p in expert order (p ascending within an expert), inv[p] = s, offsets[E+1],
//              and the list of 64-pair GEMM tiles (expert, first sorted position)
//   k_pgemm    grouped GEMM: out[s][m] = sum_k W_e[m][k] b_s[k] for the rows s of a tile
//   k_ph       h = silu(g) u (binary32), then binary16 rows scaled by a per-row power of two
//   k_pcombine out[t] = sum_r w[t][r] y[inv[t*k+r]] (ranks in order) + y_shared[t]
//
// GEMM arithmetic. B is the activation row in binary16 times its power-of-two scale (exact). FP2 /
// FP3: the A operand is the weight d (2c - 3) or d (2c - 7) rounded once to binary16 (relative error
// at most 2^-11 per weight, a quarter of the 2e-3 bound), so the MMAs accumulate across blocks. FP4:
// A is the E2M1 value times 2^-14 (exact) and each MMA pair covers one 32-weight block whose binary32
// partial is multiplied by the block scale 2^(e-127) (exact for every exponent).
#include "fpx_mma.cuh"
#include "route.cuh"
#include "tc.cuh"

using namespace fpx;

namespace {

constexpr int kPT = 64;              // pairs (or tokens) per GEMM tile: 8 MMA column tiles
constexpr int kGemmThreads = 256;    // 8 warps
constexpr int kPMaxK = 8;

// ------------------------------------------------------------------ workspace

struct PWs {
    size_t status, logits, idx, w, counts, offsets, perm, inv, units, nunits, x16, shx;
    size_t g, u, gsh, ush, h16, shh, hsh16, shsh, yp, ysh, xg, gshift, tcu_gu, tcu_dn, ntc, total;
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
    w.units = o; o = up256(o + 8 * (P / kPT + E));
    w.nunits = o; o = up256(o + 16);
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

// logits[t][e] = sum_h R[e][h] x[t][h] (binary32; the sum runs over h in order for every (t, e), so
// equal router rows give equal logits). Tile: 64 tokens x 64 experts, 16 x 16 threads of 4 x 4; the
// next 32-wide slice of h is loaded into registers while the current one is used.
__global__ void __launch_bounds__(256) k_plogits(const float* __restrict__ R, const uint16_t* __restrict__ x, int T,
                                                 int E, int H, float* __restrict__ logits) {
    __shared__ float xs[2][32][65];
    __shared__ float rs[2][32][65];
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    const int t0 = blockIdx.x * 64, e0 = blockIdx.y * 64;
    float acc[4][4] = {};
    float xv[8], rv[8];
    auto load = [&](int h0) {
#pragma unroll
        for (int v = 0; v < 8; v++) {
            const int i = threadIdx.x + 256 * v, rr = i / 32, kk = i % 32;
            const int t = t0 + rr, e = e0 + rr;
            xv[v] = t < T ? __uint_as_float((uint32_t)x[(size_t)t * H + h0 + kk] << 16) : 0.f;
            rv[v] = e < E ? R[(size_t)e * H + h0 + kk] : 0.f;
        }
    };
    load(0);
    for (int h0 = 0, buf = 0; h0 < H; h0 += 32, buf ^= 1) {
#pragma unroll
        for (int v = 0; v < 8; v++) {
            const int i = threadIdx.x + 256 * v, rr = i / 32, kk = i % 32;
            xs[buf][kk][rr] = xv[v];
            rs[buf][kk][rr] = rv[v];
        }
        __syncthreads();
        if (h0 + 32 < H) load(h0 + 32);
#pragma unroll 8
        for (int kk = 0; kk < 32; kk++) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; i++) { a[i] = xs[buf][kk][ty + 16 * i]; b[i] = rs[buf][kk][tx + 16 * i]; }
#pragma unroll
            for (int i = 0; i < 4; i++)
#pragma unroll
                for (int j = 0; j < 4; j++) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
    }
#pragma unroll
    for (int i = 0; i < 4; i++)
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const int t = t0 + ty + 16 * i, e = e0 + tx + 16 * j;
            if (t < T && e < E) logits[(size_t)t * E + e] = acc[i][j];
        }
}

// One warp per token.
__global__ void __launch_bounds__(256) k_ptopk(const float* __restrict__ logits, int T, int E, int k, int32_t* idx,
                                               float* w) {
    const int t = blockIdx.x * 8 + threadIdx.x / 32;
    if (t >= T) return;
    int32_t ii[kPMaxK];
    float ww[kPMaxK];
    warp_topk(logits + (size_t)t * E, E, k, ii, ww);
    if ((threadIdx.x & 31) < k) {
        const int r = threadIdx.x & 31;
        int32_t iv = ii[0];
        float wv = ww[0];
        for (int j = 1; j < kPMaxK; j++)
            if (j == r) { iv = ii[j]; wv = ww[j]; }
        idx[(size_t)t * k + r] = iv;
        w[(size_t)t * k + r] = wv;
    }
}

__global__ void k_phist(const int32_t* __restrict__ idx, int P, int E, int32_t* counts, int32_t* status) {
    const int p = blockIdx.x * blockDim.x + threadIdx.x;
    if (p >= P) return;
    const int e = idx[p];
    if (e < 0 || e >= E) { flag(status, FPX_EDATA); return; }
    atomicAdd(counts + e, 1);
}

// One CTA of 1024 threads (E <= 1024): offsets = exclusive scan of counts; tiles of kPT sorted
// positions per expert, listed in expert order as (expert, first position).
__global__ void __launch_bounds__(1024) k_pscan(const int32_t* __restrict__ counts, int E, int32_t* offsets,
                                                int2* units, int32_t* nunits) {
    __shared__ int32_t a[1024], b[1024];
    const int e = threadIdx.x;
    const int n = e < E ? counts[e] : 0, nt = (n + kPT - 1) / kPT;
    a[e] = n;
    b[e] = nt;
    __syncthreads();
    for (int o = 1; o < 1024; o <<= 1) {  // inclusive scans (Hillis-Steele)
        const int va = e >= o ? a[e - o] : 0, vb = e >= o ? b[e - o] : 0;
        __syncthreads();
        a[e] += va;
        b[e] += vb;
        __syncthreads();
    }
    const int off = a[e] - n, ub = b[e] - nt;
    if (e < E) {
        offsets[e] = off;
        for (int j = 0; j < nt; j++) units[ub + j] = make_int2(e, off + j * kPT);
    }
    if (e == E - 1) {
        offsets[E] = a[e];
        *nunits = b[e];
    }
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

// ------------------------------------------------------------------ grouped GEMM

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// binary16 pair (lo, hi) of exactly representable values, at compile time
constexpr uint32_t f16x2_pair(double lo, double hi) { return (uint32_t(f16_bits(hi)) << 16) | f16_bits(lo); }
// decode constants (see a_frag)
constexpr uint32_t kF2Mul0 = f16x2_pair(1.0, 0.25), kF2Add0 = f16x2_pair(-1027.0, -259.0);
constexpr uint32_t kF2Mul2 = f16x2_pair(0.0625, 0.015625), kF2Add2 = f16x2_pair(-67.0, -19.0);
constexpr uint32_t kF3Mul = f16x2_pair(1.0, 1.0), kF3Add = f16x2_pair(-1031.0, -1031.0);

__device__ __forceinline__ uint32_t hfma2_u(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

struct PGemmArgs {
    const uint8_t* W;         // box-tiled matrix of expert 0, or the shared matrix
    int64_t mstride;          // bytes between consecutive experts' matrices (0: shared)
    int M, K;                 // rows and columns of each matrix
    const __half* B;          // binary16 activation rows [*][K]
    const int32_t* rows;      // routed gate/up: perm (B row = perm[s] / row_div); else B row = s
    int row_div;
    const int32_t* shift;     // power-of-two scale of each B row
    const int2* units;        // routed: tiles (expert, first sorted position); NULL: shared
    const int32_t* nunits;
    const int32_t* offsets;   // routed: expert ranges
    int n_rows;               // shared: number of rows (tokens)
    float* out;               // [rows][M]
    int32_t* status;
};

template <int FMT>
struct PGeo {
    static constexpr int R = stage_rows(FMT);                 // weight rows per tile (box rows)
    static constexpr int SK = stage_k(FMT);                   // weights per row per stage
    static constexpr int WB = stage_bytes(FMT);               // weight box bytes
    static constexpr int BP = SK * 2 + 32;                    // B row pitch (bytes): conflict-free 64-bit loads
    static constexpr int BB = kPT * BP;                       // B tile bytes
    static constexpr int BUF = WB + BB;
    static constexpr int SMEM = 2 * BUF + 2 * kPT * 4;        // + B row indices and shifts
    static constexpr int NB = SK / 32;                        // blocks per stage
    static constexpr int RT = FMT == 4 ? 1 : 2;               // 16-row tiles per warp
    static constexpr int NT = FMT == 4 ? 4 : 8;               // 8-column tiles per warp
};

// FP3 code j of pair slot (odd, p): the 3-bit field of the box layout (see fp3_slot).
__device__ __forceinline__ uint32_t fp3_code(uint32_t W0, uint32_t W1, uint32_t W2, int f, int hh) {
    if (f < 0) return ((W0 >> (16 * hh)) & 1u) | (((W1 >> (16 * hh)) & 1u) << 1) | (((W2 >> (16 * hh)) & 1u) << 2);
    const uint32_t w = f < 16 ? W0 : f < 32 ? W1 : W2;
    return (w >> (16 * hh + (f & 15))) & 7u;
}

// A fragment registers of one row for block b, half ww: a0 = k-slots (2t, 2t + 1), a2 = (2t + 8, 2t + 9),
// holding codes 16 ww + 4t + {0, 1} and {2, 3} of the block (B is loaded with the same order). A code c
// placed at binary16 mantissa bit P reads 1024 + c 2^P; one HFMA2 maps it to 2c - 3 (FP2) or 2c - 7
// (FP3) with constants exact in binary16 (P >= 1 keeps them within 11 significant bits).
__device__ __forceinline__ uint32_t hmul2_u(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

template <int FMT>
__device__ __forceinline__ void a_frag(uint32_t wbox, int row, int b, int ww, int t, uint32_t& a0, uint32_t& a2) {
    if constexpr (FMT == 2) {
        const int C = b >> 1, hb = b & 1;
        uint32_t wd;
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(wd) : "r"(wbox + (uint32_t)(row * 64 + 4 * (4 * (2 * hb + ww) + C))));
        // byte t (codes 4t .. 4t + 3, 2 bits each) in both halves, shifted up by one: c0 at P = 1 (low),
        // c1 at P = 3 (high), c2 at P = 5 (low), c3 at P = 7 (high)
        const uint32_t v2 = __byte_perm(wd, 0u, (uint32_t)t | 0x40u | ((uint32_t)t << 8) | 0x4000u) << 1;
        a0 = hfma2_u((v2 & 0x00180006u) | kMagic, kF2Mul0, kF2Add0);
        a2 = hfma2_u((v2 & 0x01800060u) | kMagic, kF2Mul2, kF2Add2);
    } else if constexpr (FMT == 3) {
        const int C = b >> 1, hb = b & 1, m = C >> 1, odd = C & 1;
        const int tl = 2 * hb + ww;  // the layout thread whose group holds these codes
        const uint32_t base = wbox + (uint32_t)(row * 96 + 24 * tl + 12 * m);
        uint32_t W0, W1, W2;
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(W0) : "r"(base));
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(W1) : "r"(base + 4));
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(W2) : "r"(base + 8));
        const int hh = t >> 1, p0 = 4 * (t & 1);
        uint32_t c[4];
#pragma unroll
        for (int i = 0; i < 4; i++) c[i] = fp3_code(W0, W1, W2, fp3_slot(odd, p0 + i), hh);
        // P = 1: 1024 + 2c - 1031 = 2c - 7
        a0 = hfma2_u(((c[0] | (c[1] << 16)) << 1) | kMagic, kF3Mul, kF3Add);
        a2 = hfma2_u(((c[2] | (c[3] << 16)) << 1) | kMagic, kF3Mul, kF3Add);
    } else {
        const uint32_t o = wbox + (uint32_t)(row * 272 + 17 * b + 1 + 8 * ww + 2 * t);
        uint16_t lo, hi;
        asm volatile("ld.shared.u8 %0, [%1];" : "=h"(lo) : "r"(o));
        asm volatile("ld.shared.u8 %0, [%1];" : "=h"(hi) : "r"(o + 1));
        const uint32_t v = (uint32_t)lo | ((uint32_t)hi << 8);
        const uint32_t v2 = v | (v << 12), v3 = v2 >> 8;
        a0 = ((v2 & 0x00070007u) << 9) | ((v2 & 0x00080008u) << 12);
        a2 = ((v3 & 0x00070007u) << 9) | ((v3 & 0x00080008u) << 12);
    }
}

// FP2 / FP3: the binary16 scale of block b of a row, in both halves of a pair.
template <int FMT>
__device__ __forceinline__ uint32_t blk_scale2(uint32_t wbox, int row, int b) {
    const int C = b >> 1, hb = b & 1;
    uint16_t d;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(d) : "r"(wbox + (uint32_t)(box_scale_offset(FMT) + row * 16 + 2 * (4 * hb + C))));
    return (uint32_t)d | ((uint32_t)d << 16);
}

// Scale of block b of a row (binary32); FP4: 2^(e - 127) * 2^14 (undoing the decode's 2^-14), 0 and a
// flag for the invalid exponent 255.
template <int FMT>
__device__ __forceinline__ float blk_scale(uint32_t wbox, int row, int b, uint32_t& bad) {
    if constexpr (FMT == 4) {
        uint16_t e;
        asm volatile("ld.shared.u8 %0, [%1];" : "=h"(e) : "r"(wbox + (uint32_t)(row * 272 + 17 * b)));
        bad |= e == 255;
        return e == 255 ? 0.f : exp2i((int)e - 127 + 14);
    } else {
        const int C = b >> 1, hb = b & 1;
        uint16_t d;
        asm volatile("ld.shared.u16 %0, [%1];" : "=h"(d) : "r"(wbox + (uint32_t)(box_scale_offset(FMT) + row * 16 + 2 * (4 * hb + C))));
        return __half2float(__ushort_as_half(d));
    }
}

template <int FMT>
__global__ void __launch_bounds__(kGemmThreads, 2) k_pgemm(const __grid_constant__ PGemmArgs A) {
    using G = PGeo<FMT>;
    extern __shared__ __align__(128) uint8_t smem[];
    int32_t* brow_s = reinterpret_cast<int32_t*>(smem + 2 * G::BUF);
    int32_t* bsh_s = brow_s + kPT;
    const int u = blockIdx.y;
    int e = 0, s0, n;
    if (A.units) {
        if (u >= __ldg(A.nunits)) return;
        const int2 un = A.units[u];
        e = un.x;
        s0 = un.y;
        n = min(kPT, A.offsets[e + 1] - s0);
    } else {
        s0 = u * kPT;
        if (s0 >= A.n_rows) return;
        n = min(kPT, A.n_rows - s0);
    }
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    if (threadIdx.x < kPT) {
        const int s = s0 + threadIdx.x;
        const int br = threadIdx.x < n ? (A.rows ? A.rows[s] / A.row_div : s) : -1;
        brow_s[threadIdx.x] = br;
        bsh_s[threadIdx.x] = br >= 0 ? A.shift[br] : 0;
    }
    __syncthreads();
    const int rb = blockIdx.x;  // row block of R rows
    const int nks = A.K / G::SK;
    const uint8_t* wbase = A.W + (int64_t)e * A.mstride + (int64_t)rb * nks * G::WB;
    const uint32_t sbase = smem_u32(smem);

    auto issue = [&](int ks, int buf) {
        const uint32_t wdst = sbase + (uint32_t)(buf * G::BUF), bdst = wdst + G::WB;
        const uint8_t* wsrc = wbase + (int64_t)ks * G::WB;
        for (int c = threadIdx.x; c < G::WB / 16; c += kGemmThreads) cp_async16(wdst + 16 * c, wsrc + 16 * c, 16);
        constexpr int CPR = G::SK * 2 / 16;  // 16-byte chunks per B row
        for (int c = threadIdx.x; c < kPT * CPR; c += kGemmThreads) {
            const int r = c / CPR, j = c % CPR;
            const int br = brow_s[r];
            const __half* src = br >= 0 ? A.B + (size_t)br * A.K + (size_t)ks * G::SK + 8 * j : A.B;
            cp_async16(bdst + (uint32_t)(r * G::BP + 16 * j), src, br >= 0 ? 16u : 0u);
        }
        cp_async_commit();
    };

    float y[G::RT][G::NT][4];
#pragma unroll
    for (int i = 0; i < G::RT; i++)
#pragma unroll
        for (int j = 0; j < G::NT; j++) y[i][j][0] = y[i][j][1] = y[i][j][2] = y[i][j][3] = 0.f;
    uint32_t bad = 0;
    // warp layout: FP2 / FP3: rows 32w .. 32w + 31 (two tiles), all 64 columns; FP4: rows
    // 16 (w % 4) .. +15, columns 32 (w / 4) .. +31
    const int row0 = FMT == 4 ? 16 * (warp & 3) : 32 * warp;
    const int col0 = FMT == 4 ? 32 * (warp >> 2) : 0;

    issue(0, 0);
    for (int ks = 0; ks < nks; ks++) {
        if (ks + 1 < nks) {
            issue(ks + 1, (ks + 1) & 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const uint32_t wbox = sbase + (uint32_t)((ks & 1) * G::BUF), btile = wbox + G::WB;
#pragma unroll 1
        for (int b = 0; b < G::NB; b++) {
            uint32_t af[G::RT][2][4];  // [row tile][half][a0 a1 a2 a3]
            float d[G::RT][2];
#pragma unroll
            for (int i = 0; i < G::RT; i++) {
                const int r0 = row0 + 16 * i + g, r8 = r0 + 8;
#pragma unroll
                for (int ww = 0; ww < 2; ww++) {
                    a_frag<FMT>(wbox, r0, b, ww, t, af[i][ww][0], af[i][ww][2]);
                    a_frag<FMT>(wbox, r8, b, ww, t, af[i][ww][1], af[i][ww][3]);
                }
                if constexpr (FMT == 4) {
                    d[i][0] = blk_scale<FMT>(wbox, r0, b, bad);
                    d[i][1] = blk_scale<FMT>(wbox, r8, b, bad);
                } else {  // fold the block scale into the binary16 weights
                    const uint32_t d0 = blk_scale2<FMT>(wbox, r0, b), d8 = blk_scale2<FMT>(wbox, r8, b);
#pragma unroll
                    for (int ww = 0; ww < 2; ww++) {
                        af[i][ww][0] = hmul2_u(af[i][ww][0], d0);
                        af[i][ww][2] = hmul2_u(af[i][ww][2], d0);
                        af[i][ww][1] = hmul2_u(af[i][ww][1], d8);
                        af[i][ww][3] = hmul2_u(af[i][ww][3], d8);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < G::NT; j++) {
                const uint32_t ba = btile + (uint32_t)((col0 + 8 * j + g) * G::BP + 2 * (32 * b + 4 * t));
                uint32_t b00, b01, b10, b11;
                asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(b00), "=r"(b01) : "r"(ba));
                asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(b10), "=r"(b11) : "r"(ba + 32));
#pragma unroll
                for (int i = 0; i < G::RT; i++) {
                    if constexpr (FMT == 4) {
                        float p[4];
                        mma_first(p, af[i][0][0], af[i][0][1], af[i][0][2], af[i][0][3], b00, b01);
                        mma_acc(p, af[i][1][0], af[i][1][1], af[i][1][2], af[i][1][3], b10, b11);
                        y[i][j][0] = fmaf(d[i][0], p[0], y[i][j][0]);
                        y[i][j][1] = fmaf(d[i][0], p[1], y[i][j][1]);
                        y[i][j][2] = fmaf(d[i][1], p[2], y[i][j][2]);
                        y[i][j][3] = fmaf(d[i][1], p[3], y[i][j][3]);
                    } else {
                        mma_acc(y[i][j], af[i][0][0], af[i][0][1], af[i][0][2], af[i][0][3], b00, b01);
                        mma_acc(y[i][j], af[i][1][0], af[i][1][1], af[i][1][2], af[i][1][3], b10, b11);
                    }
                }
            }
        }
        __syncthreads();  // the buffer is refilled by the next issue
    }
    if (__any_sync(0xffffffffu, bad != 0u) && lane == 0) flag(A.status, FPX_EDATA);
    // epilogue: out[s][m] = y * 2^-shift(s)
#pragma unroll
    for (int j = 0; j < G::NT; j++) {
#pragma unroll
        for (int c = 0; c < 2; c++) {
            const int col = col0 + 8 * j + 2 * t + c;
            if (col >= n) continue;
            const float sc = exp2i(-bsh_s[col]);
            float* o = A.out + (size_t)(s0 + col) * A.M + (size_t)rb * G::R;
#pragma unroll
            for (int i = 0; i < G::RT; i++) {
                o[row0 + 16 * i + g] = y[i][j][c] * sc;
                o[row0 + 16 * i + g + 8] = y[i][j][2 + c] * sc;
            }
        }
    }
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
// decode (pair p = weights p and p + 8); the B rows are stored in the same order (kpermute16), so the
// products pair up as in the plain dot product.
constexpr int kTcN = 128;                                           // pairs per unit at most
constexpr int kTcSK = 128;                                          // K per stage
constexpr int kTcAStages = 2;                                       // A stages in tensor memory
constexpr int kTcBStages = 4;                                       // B stages in shared memory
constexpr int kTcRS = 3;                                            // packed boxes in flight
constexpr int kTcDec = 16, kTcEpi = 4;                              // decoder and epilogue warps
constexpr int kTcIss = 2;                                           // MMA-issuing warps (one per half)
constexpr int kTcDec0 = 2 + kTcIss;                                 // first decoder warp
constexpr int kTcThreads = (kTcDec0 + kTcDec + kTcEpi) * 32;
constexpr int kTcBRows = 16;                                        // rows of one B tile load
constexpr int kTcBTile = kTcN * 128;                                // 128 rows x 64 binary16
constexpr int kTcBStage = 2 * kTcBTile;                             // a stage: two 64-wide tiles
constexpr int kTcBox = stage_bytes(3);                              // ring slot (an FP2 box fits)
constexpr int kTcSmem = kTcRS * kTcBox + kTcBStages * kTcBStage + 1024;
constexpr int kTcCols = 512;
constexpr uint32_t kTcACol = 256;                                   // first A-stage column
static_assert(kTcBox % 1024 == 0 && kTcBTile % 1024 == 0, "1024-byte aligned stages");
static_assert(kTcSmem + kTcEpi * kTcN * 4 + 1024 <= 227 * 1024, "shared memory per CTA");
static_assert(kTcACol + 128 * kTcAStages <= kTcCols, "tensor-memory columns");

// Column block (8 columns) of K step kk (0..7 = slab kk / 4, code group kk % 4) within a half's 64
// A-stage columns: thread p of a row owns blocks 4 p .. 4 p + 3 (groups 2 p, 2 p + 1 of both slabs).
__host__ __device__ constexpr uint32_t tc_kblock(int kk) { return 4u * ((kk & 3) >> 1) + 2u * (kk >> 2) + (kk & 1); }

struct TcArgs {
    CUtensorMap bmap;         // B: binary16 [rows][K], K-permuted, box 64 x 16, 128-byte swizzle
    const uint8_t* W;         // box-tiled matrix of expert 0
    int64_t mstride;          // bytes between experts' matrices
    int M, K;
    const int4* units;        // (expert, first B row, pairs, 256-row block)
    const int32_t* nunits;
    const int32_t* shift;     // power-of-two scale exponent of every B row
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
    __shared__ uint64_t bars[2 * kTcRS + 2 * kTcAStages + 2 * kTcBStages + 5];
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
                const uint8_t* wb = A.W + (int64_t)un.x * A.mstride + (int64_t)un.w * (A.K / stage_k(FMT)) * stage_bytes(FMT);
                for (int bx = 0; bx < nslab / 4; bx++, gb++) {
                    const uint32_t sl = gb % kTcRS;
                    if (gb >= (uint32_t)kTcRS && !mbar_wait(ring_empty + sl, ((gb / kTcRS) + 1u) & 1u)) { live = false; break; }
                    mbar_expect_tx(ring_full + sl, stage_bytes(FMT));
                    bulk_load(ring + sl * kTcBox, wb + (int64_t)bx * stage_bytes(FMT), stage_bytes(FMT), ring_full + sl);
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
                        tc_mma_f16_ta(dcol, a0 + 8u * tc_kblock(kk), bd + 1024u * (kk >> 2) + 2u * (kk & 3), idesc, (j | kk) != 0);
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
                    const uint32_t st = gs % kTcAStages;
                    if (live && gs >= (uint32_t)kTcAStages)
                        live = __any_sync(0xffffffffu, mbar_wait(a_free + st, ((gs / kTcAStages) + 1u) & 1u));
                    if (!live) break;
                    tc_fence_after();
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
                    tmem_st32(lane_base + 128u * st, o);
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(a_full + st);
                }
            }
        }
        if (!live && lane == 0) flag(A.status, FPX_ETIMEOUT);
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
                for (int c0 = 0; c0 < n16; c0 += 16) {
                    float v[16];
                    tmem_ld16(taddr + ((uint32_t)(32 * q) << 16) + col0 + hstep * (uint32_t)hh + (uint32_t)c0, v);
#pragma unroll
                    for (int j = 0; j < 16; j++) {
                        const int s = c0 + j;
                        if (s < n) orow[(size_t)s * A.M] = v[j] * fac[s];
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
// PERM: each 16-element group stored in the tensor-core decode's pair order (element p, then p + 8).
template <bool PERM>
__global__ void __launch_bounds__(256) k_ph(const float* __restrict__ g, const float* __restrict__ u, int L,
                                            __half* __restrict__ h16, int32_t* __restrict__ shift) {
    __shared__ float red[8];
    __shared__ int sh_s;
    const size_t r = blockIdx.x;
    float m = 0.f;
    for (int i = threadIdx.x; i < L; i += blockDim.x) {
        const float a = g[r * L + i], b = u[r * L + i];
        m = fmaxf(m, fabsf((a / (1.0f + expf(-a))) * b));
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
    if (!PERM) {
        for (int i = threadIdx.x; i < L; i += blockDim.x) {
            const float a = g[r * L + i], b = u[r * L + i];
            h16[r * L + i] = __float2half_rn(((a / (1.0f + expf(-a))) * b) * sc);
        }
        return;
    }
    for (int gi = threadIdx.x; gi < L / 16; gi += blockDim.x) {
        float v[16];
#pragma unroll
        for (int j = 0; j < 16; j++) {
            const float a = g[r * L + 16 * gi + j], b = u[r * L + 16 * gi + j];
            v[j] = ((a / (1.0f + expf(-a))) * b) * sc;
        }
        uint32_t o[8];
#pragma unroll
        for (int p = 0; p < 8; p++) {
            const __half2 hp = __halves2half2(__float2half_rn(v[p]), __float2half_rn(v[p + 8]));
            o[p] = *reinterpret_cast<const uint32_t*>(&hp);
        }
        uint4* dst = reinterpret_cast<uint4*>(h16 + r * L + 16 * gi);
        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
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

template <int FMT>
cudaError_t launch_gemm(const PGemmArgs& a, int grid_units, cudaStream_t s) {
    using G = PGeo<FMT>;
    cudaError_t e = cudaFuncSetAttribute(k_pgemm<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM);
    if (e != cudaSuccess) return e;
    if (grid_units <= 0) return cudaSuccess;
    k_pgemm<FMT><<<dim3(a.M / G::R, grid_units), kGemmThreads, G::SMEM, s>>>(a);
    return cudaGetLastError();
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
    if (cudaFuncSetAttribute(k_tcgemm<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem) != cudaSuccess) return FPX_ECUDA;
    k_tcgemm<FMT><<<device_info().sms, kTcThreads, kTcSmem, s>>>(a);
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
    if (H < 512 || I < 512 || H % 512 || I % 512) return FPX_EINVAL;
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
    int2* units = reinterpret_cast<int2*>(b + W.units);
    int32_t* nunits = reinterpret_cast<int32_t*>(b + W.nunits);
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
    const int P = T * k;

    if (cudaMemsetAsync(status, 0, 16, s) != cudaSuccess || cudaMemsetAsync(counts, 0, 4 * (E + 1), s) != cudaSuccess)
        return FPX_ECUDA;
    k_to_f16<false><<<T, 256, 0, s>>>(x, H, x16, shx);
    k_plogits<<<dim3((T + 63) / 64, (E + 63) / 64), 256, 0, s>>>(L->router, x, T, E, H, logits);
    k_ptopk<<<(T + 7) / 8, 256, 0, s>>>(logits, T, E, k, idx, w);
    k_phist<<<(P + 255) / 256, 256, 0, s>>>(idx, P, E, counts, status);
    k_pscan<<<1, 1024, 0, s>>>(counts, E, offsets, units, nunits);
    k_pscatter<<<E, 256, 0, s>>>(idx, P, offsets, perm, inv);
    if (cudaGetLastError() != cudaSuccess) return FPX_ECUDA;

    const int tok_units = (T + kPT - 1) / kPT;
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
    // shared gate and up: every token
    PGemmArgs sa{};
    sa.status = status;
    sa.M = I; sa.K = H; sa.B = x16; sa.rows = nullptr; sa.row_div = 1; sa.units = nullptr; sa.nunits = nullptr;
    sa.offsets = nullptr; sa.mstride = 0; sa.n_rows = T; sa.shift = shx;
    sa.W = L->sh_gate; sa.out = gsh;
    if (launch_gemm<4>(sa, tok_units, s) != cudaSuccess) return FPX_ECUDA;
    sa.W = L->sh_up; sa.out = ush;
    if (launch_gemm<4>(sa, tok_units, s) != cudaSuccess) return FPX_ECUDA;
    // h in binary16 with per-row scales (routed rows K-permuted for the tensor-core GEMM)
    k_ph<true><<<P, 256, 0, s>>>(g, u, I, h16, shh);
    k_ph<false><<<T, 256, 0, s>>>(gsh, ush, I, hsh16, shsh);
    if (cudaGetLastError() != cudaSuccess) return FPX_ECUDA;
    // routed down: h rows already in expert order
    TcArgs tda = ta;
    tda.M = H; tda.K = I; tda.units = tcu_dn; tda.nunits = ntc + 1; tda.shift = shh; tda.mstride = mb3;
    tda.W = L->down; tda.out = yp;
    if ((st = launch_tc<3>(tda, h16, P, s))) return st;
    PGemmArgs dsa = sa;
    dsa.M = H; dsa.K = I; dsa.B = hsh16; dsa.shift = shsh; dsa.W = L->sh_down; dsa.out = ysh;
    if (launch_gemm<4>(dsa, tok_units, s) != cudaSuccess) return FPX_ECUDA;
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
