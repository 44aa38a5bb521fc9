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

using namespace fpx;

namespace {

constexpr int kPT = 64;              // pairs (or tokens) per GEMM tile: 8 MMA column tiles
constexpr int kGemmThreads = 256;    // 8 warps
constexpr int kPMaxK = 8;

// ------------------------------------------------------------------ workspace

struct PWs {
    size_t status, logits, idx, w, counts, offsets, perm, inv, units, nunits, x16, shx;
    size_t g, u, gsh, ush, h16, shh, hsh16, shsh, yp, ysh, total;
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

// h = silu(g) u for rows [0, Pr) of (g, u) -> binary16 rows scaled by 2^sh(row) (exact shift), shift[row].
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
    for (int i = threadIdx.x; i < L; i += blockDim.x) {
        const float a = g[r * L + i], b = u[r * L + i];
        h16[r * L + i] = __float2half_rn(((a / (1.0f + expf(-a))) * b) * sc);
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

    const int max_units = P / kPT + E, tok_units = (T + kPT - 1) / kPT;
    const int64_t mb2 = fpx_matrix_bytes(2, I, H), mb3 = fpx_matrix_bytes(3, H, I);
    PGemmArgs a{};
    a.status = status;
    // routed gate and up: rows of x gathered by token, in expert order
    a.M = I; a.K = H; a.B = x16; a.rows = perm; a.row_div = k; a.shift = shx;
    a.units = units; a.nunits = nunits; a.offsets = offsets; a.mstride = mb2;
    a.W = L->gate; a.out = g;
    if (launch_gemm<2>(a, max_units, s) != cudaSuccess) return FPX_ECUDA;
    a.W = L->up; a.out = u;
    if (launch_gemm<2>(a, max_units, s) != cudaSuccess) return FPX_ECUDA;
    // shared gate and up: every token
    PGemmArgs sa = a;
    sa.rows = nullptr; sa.row_div = 1; sa.units = nullptr; sa.nunits = nullptr; sa.offsets = nullptr; sa.mstride = 0;
    sa.n_rows = T; sa.shift = shx;
    sa.W = L->sh_gate; sa.out = gsh;
    if (launch_gemm<4>(sa, tok_units, s) != cudaSuccess) return FPX_ECUDA;
    sa.W = L->sh_up; sa.out = ush;
    if (launch_gemm<4>(sa, tok_units, s) != cudaSuccess) return FPX_ECUDA;
    // h in binary16 with per-row scales
    k_ph<<<P, 256, 0, s>>>(g, u, I, h16, shh);
    k_ph<<<T, 256, 0, s>>>(gsh, ush, I, hsh16, shsh);
    if (cudaGetLastError() != cudaSuccess) return FPX_ECUDA;
    // routed down: h rows already in expert order
    PGemmArgs da = a;
    da.M = H; da.K = I; da.B = h16; da.rows = nullptr; da.row_div = 1; da.shift = shh; da.mstride = mb3;
    da.W = L->down; da.out = yp;
    if (launch_gemm<3>(da, max_units, s) != cudaSuccess) return FPX_ECUDA;
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
