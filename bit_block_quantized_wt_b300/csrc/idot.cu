// Integer-dot variant of the dense FPX GEMV ("DeepSeek V4 Flash hits 32 tok/s on AMD Ryzen AI MAX+
// 395", paragraph 3: the ROCmFPX kernels read packed blocks, expand the codebooks with byte-permute
// instructions in registers and feed integer dot products).
//
// Activations (the pages leave this side open; this is the project's reading). For each column t and
// each block b of 32 entries: a = max |x|, e the integer with 2^(e-1) <= a < 2^e, X = RN_even(x 2^(14-e)),
// |X| <= 2^14, split X = 256 hi + lo with hi = X >> 8 (signed, -64..64) and lo = X & 255 (unsigned).
// A block's weights expand to signed bytes v (FP2 2c - 3, FP3 2c - 7, FP4 2 E2M1 = 0, +-1 .. +-12),
// so sum_j v_j X_j = 256 dp4a(v, hi) + dp4a(v, lo) is exact in int32 (|sum| < 2^23), and the block
// term is (float)sum * d * 2^(e-14) with d the block scale (FP4: 2^(E-128)). The result is the plain
// GEMV of x_hat = X 2^(e-14) up to binary32 rounding of the block terms and of their sums.
//
// Kernels:
//   k_xquant   - builds the activation table (hi / lo bytes in the order the weight expansion
//                produces them, plus 2^(e-14) per column block) in the caller's workspace.
//   k_gemv_idot - persistent CTAs over 64-row blocks (CTA c starts with block c, then takes the next
//                free one from a counter); a producer thread streams stages of 64 rows x
//                one slice of 32 blocks (2-D TMA boxes of 20 / 28 / 34 KB) into a ring; 8 consumer
//                warps take 8 rows each, lane l owns block l of the slice: it keeps that block's
//                activation bytes in registers, expands each row's block with byte permutes, runs the
//                dp4a chains and scales once per (row, block, column). The 32 lanes' terms are summed
//                with a transposing butterfly; the slices of a row block are added in slice order.
#include <algorithm>
#include <type_traits>

#include "fpx_mma.cuh"

namespace fpx {
namespace {

constexpr int kIdWarps = 8;                       // consumer warps
constexpr int kIdThreads = (kIdWarps + 1) * 32;   // + the producer warp
constexpr int kIdRows = 64;                       // rows per stage
constexpr int kIdRowsPerWarp = kIdRows / kIdWarps;
constexpr int kIdMaxStages = 6;

__host__ __device__ constexpr int slice_bytes(int fmt) { return 32 * block_bytes(fmt); }  // 320 / 448 / 544
__host__ __device__ constexpr int id_stage_bytes(int fmt) { return kIdRows * slice_bytes(fmt); }

// Activation table (workspace and shared memory): nbp = blocks padded to whole slices (entries past
// K are zero). Code area: chunk c = 4t + 2 part + half (part 0 = hi bytes, 1 = lo bytes; half 0 / 1 =
// expanded weight words 0-3 / 4-7) of block b is 16 bytes at (c * nbp + b) * 16, so the 32 lanes of a
// warp read one chunk of 32 consecutive blocks without bank conflicts. Then the scale area:
// float 2^(e-14) of (column t, block b) at index t * nbp + b.
__host__ __device__ constexpr size_t xtab_code_bytes(int nbp, int q) { return (size_t)nbp * q * 64; }
__host__ __device__ constexpr size_t xtab_bytes(int nbp, int q) { return (size_t)nbp * q * 68; }
// workspace: the table, then a 16-byte row-block counter (zeroed by k_xquant)
__host__ __device__ constexpr size_t idot_ws_bytes(int nbp, int q) { return xtab_bytes(nbp, q) + 16; }

// Position of code j of a block among the expanded weight words: (word, byte).
//   FP2 / FP3: the 16 codes of a code word h expand into words 4h .. 4h + 3 holding the codes
//   {0, 2, 4, 6}, {8, 10, 12, 14}, {1, 3, 5, 7}, {9, 11, 13, 15} (+ 16h), low byte first.
//   FP4: codes in order, four per word.
template <int FMT>
__device__ __forceinline__ void code_slot(int j, int& word, int& byte) {
    if constexpr (FMT == 4) {
        word = j >> 2;
        byte = j & 3;
    } else {
        const int h = j >> 4, r = j & 15;
        word = 4 * h + 2 * (r & 1) + (r >> 3);
        byte = (r & 7) >> 1;
    }
}

__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// One warp per (column t, block b): lane j quantizes entry 32 b + j.
template <int FMT>
__global__ void __launch_bounds__(256) k_xquant(const void* __restrict__ x, int x_bf16, int K, int q, int nbp,
                                                uint8_t* __restrict__ tab, int32_t* st) {
    grid_dep_trigger();  // the GEMV may start streaming weights; it waits for this grid before reading the table
    const int lane = threadIdx.x & 31;
    const int unit = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (unit >= q * nbp) return;
    const int t = unit / nbp, b = unit % nbp;
    const int k = b * 32 + lane;
    float v = 0.0f;
    if (k < K) {
        const int64_t i = (int64_t)t * K + k;
        v = x_bf16 ? bf16_bits_to_float(reinterpret_cast<const uint16_t*>(x)[i]) : reinterpret_cast<const float*>(x)[i];
    }
    if (!isfinite(v)) {
        flag(st, FPX_ERANGE);
        v = 0.0f;
    }
    const float a = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v))));
    int X = 0;
    float scale = 0.0f;
    if (a > 0.0f) {
        int e;
        frexpf(a, &e);                          // a = f 2^e, 0.5 <= f < 1
        X = __float2int_rn(scalbnf(v, 14 - e));  // exact scaling, then nearest-even
        scale = scalbnf(1.0f, e - 14);
    }
    int word, byte;
    code_slot<FMT>(lane, word, byte);
    const size_t off = (size_t)(word & 3) * 4 + byte;
    const int c_hi = 4 * t + (word >> 2), c_lo = 4 * t + 2 + (word >> 2);
    tab[((size_t)c_hi * nbp + b) * 16 + off] = (uint8_t)(X >> 8);
    tab[((size_t)c_lo * nbp + b) * 16 + off] = (uint8_t)(X & 255);
    if (lane == 0) reinterpret_cast<float*>(tab + xtab_code_bytes(nbp, q))[t * nbp + b] = scale;
    if (unit == 0 && lane == 0) *reinterpret_cast<uint32_t*>(tab + xtab_bytes(nbp, q)) = 0u;  // row-block counter
}

__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_su(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Signed-byte codebooks for the byte permutes (selector nibbles index bytes 0..7 of {a, b}).
constexpr uint32_t kLut2 = 0x0301FFFDu;                          // 2c - 3, c = 0..3
constexpr uint32_t kLut3a = 0xFFFDFBF9u, kLut3b = 0x07050301u;  // 2c - 7, c = 0..7
constexpr uint32_t kLut4p0 = 0x03020100u, kLut4p1 = 0x0C080604u;  // 2 E2M1, positive
constexpr uint32_t kLut4n0 = 0xFDFEFF00u, kLut4n1 = 0xF4F8FAFCu;  // 2 E2M1, negative

// 16 2-bit codes -> four words of signed bytes (order of code_slot).
__device__ __forceinline__ void expand_fp2(uint32_t c, uint32_t* w) {
    const uint32_t m = c & 0x33333333u, n = (c >> 2) & 0x33333333u;
    w[0] = __byte_perm(kLut2, 0u, m);
    w[1] = __byte_perm(kLut2, 0u, m >> 16);
    w[2] = __byte_perm(kLut2, 0u, n);
    w[3] = __byte_perm(kLut2, 0u, n >> 16);
}

// 16 codes from a low-bit word l and 16 high bits hb (bits 0..15) -> four words (order of code_slot).
// The high bits are spread to every second bit and placed at bit 2 of each selector nibble.
__device__ __forceinline__ void expand_fp3(uint32_t l, uint32_t hb_sel_word, uint32_t sel, uint32_t* w) {
    uint32_t s = __byte_perm(hb_sel_word, 0u, sel);  // bytes (h0..7, 0, h8..15, 0)
    s = (s | (s << 4)) & 0x0F0F0F0Fu;
    s = (s | (s << 2)) & 0x33333333u;
    s = (s | (s << 1)) & 0x55555555u;                 // high bit of code i at bit 2i
    const uint32_t se = (l & 0x33333333u) | ((s << 2) & 0x44444444u);
    const uint32_t so = ((l >> 2) & 0x33333333u) | (s & 0x44444444u);
    w[0] = __byte_perm(kLut3a, kLut3b, se);
    w[1] = __byte_perm(kLut3a, kLut3b, se >> 16);
    w[2] = __byte_perm(kLut3a, kLut3b, so);
    w[3] = __byte_perm(kLut3a, kLut3b, so >> 16);
}

// 8 E2M1 codes -> two words of signed bytes: the magnitude index picks from the positive and the
// negative table, the sign bit picks between the two results byte by byte.
__device__ __forceinline__ void expand_fp4(uint32_t cw, uint32_t* w) {
    const uint32_t sel = cw & 0x77777777u;
    const uint32_t pick = ((cw >> 1) & 0x44444444u) | 0x32103210u;  // nibble i: byte i of (pos, neg)
    w[0] = __byte_perm(__byte_perm(kLut4p0, kLut4p1, sel), __byte_perm(kLut4n0, kLut4n1, sel), pick);
    const uint32_t sel_hi = sel >> 16;
    w[1] = __byte_perm(__byte_perm(kLut4p0, kLut4p1, sel_hi), __byte_perm(kLut4n0, kLut4n1, sel_hi), pick >> 16);
}

// Decodes the block a lane owns in one staged row: `a` is the shared address of the 32-bit word that
// holds the block's first byte, `sh` the bit offset of that byte in it. Returns the block scale d
// (FP4: 2^(E-128), so that the weight is d times its signed byte) and the eight expanded words.
template <int FMT, int OFF>
__device__ __forceinline__ float decode_row(uint32_t a, uint32_t sh, uint32_t (&w)[8], uint32_t& bad) {
    if constexpr (FMT == 2) {
        const uint32_t a0 = lds32<OFF>(a), a1 = lds32<OFF + 4>(a), a2 = lds32<OFF + 8>(a);
        expand_fp2(__funnelshift_rc(a0, a1, sh + 16), w);
        expand_fp2(__funnelshift_rc(a1, a2, sh + 16), w + 4);
        return __half2float(__ushort_as_half((uint16_t)((a0 >> sh) & 0xFFFFu)));
    } else if constexpr (FMT == 3) {
        const uint32_t a0 = lds32<OFF>(a), a1 = lds32<OFF + 4>(a), a2 = lds32<OFF + 8>(a), a3 = lds32<OFF + 12>(a);
        const uint32_t hp = __funnelshift_rc(a2, a3, sh + 16);
        expand_fp3(__funnelshift_rc(a0, a1, sh + 16), hp, 0x4140u, w);
        expand_fp3(__funnelshift_rc(a1, a2, sh + 16), hp, 0x4342u, w + 4);
        return __half2float(__ushort_as_half((uint16_t)((a0 >> sh) & 0xFFFFu)));
    } else {
        const uint32_t a0 = lds32<OFF>(a), a1 = lds32<OFF + 4>(a), a2 = lds32<OFF + 8>(a), a3 = lds32<OFF + 12>(a),
                       a4 = lds32<OFF + 16>(a);
        expand_fp4(__funnelshift_rc(a0, a1, sh + 8), w);
        expand_fp4(__funnelshift_rc(a1, a2, sh + 8), w + 2);
        expand_fp4(__funnelshift_rc(a2, a3, sh + 8), w + 4);
        expand_fp4(__funnelshift_rc(a3, a4, sh + 8), w + 6);
        const uint32_t e = (a0 >> sh) & 0xFFu;
        if (e == 255u) {
            bad = 1u;
            return 0.0f;
        }
        // 2^(e-128): normal for e >= 2, else the subnormals 2^-127 / 2^-128
        return __uint_as_float(e >= 2u ? (e - 1u) << 23 : 0x00200000u << e);
    }
}

// Sum over the 32 lanes of V values per lane (V a power of two <= 32) with the xor butterfly 16, 8,
// .., 1. The first log2(V) levels also transpose: a lane keeps half of its values and sends the other
// half, so every lane ends with the total of value index lane >> (5 - log2 V). Each level adds the
// same pairs as the plain butterfly, so a value's total does not depend on V.
template <int V>
__device__ __forceinline__ float transpose_reduce(float (&v)[V], int lane) {
    constexpr int L = V == 1 ? 0 : V == 2 ? 1 : V == 4 ? 2 : V == 8 ? 3 : V == 16 ? 4 : 5;
#pragma unroll
    for (int lev = 0; lev < L; lev++) {
        const int m = 16 >> lev;
        const int half = V >> (lev + 1);
        const bool up = (lane & m) != 0;
#pragma unroll
        for (int i = 0; i < half; i++) {
            const float keep = up ? v[i + half] : v[i];
            const float send = up ? v[i] : v[i + half];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
        }
    }
    float r = v[0];
#pragma unroll
    for (int m = 16 >> L; m > 0; m >>= 1) r += __shfl_xor_sync(0xffffffffu, r, m);
    return r;
}

struct IdotArgs {
    CUtensorMap map;       // rows x row bytes, 32-bit elements, box = one slice x 64 rows
    int N, nsl, nbp, nrb, NS;
    uint32_t tab_bytes;
    const uint8_t* tab;    // activation table in the workspace
    uint32_t* counter;     // row blocks handed out past the first gridDim.x
    float* y;
    int32_t* st;
};

template <int FMT, int Q>
__global__ void __launch_bounds__(kIdThreads, 1) k_gemv_idot(const __grid_constant__ IdotArgs A) {
    constexpr int SLB = slice_bytes(FMT), SB = id_stage_bytes(FMT), BB = block_bytes(FMT);
    constexpr int QP = Q == 3 ? 4 : Q;             // columns in the reduction (Q = 3 adds a zero column)
    constexpr int V = kIdRowsPerWarp * QP;
    constexpr int L = V == 8 ? 3 : V == 16 ? 4 : 5;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* ring = smem + ((128u - (smem_u32(smem) & 127u)) & 127u);
    uint8_t* tab = ring + (size_t)A.NS * SB;
    uint64_t* full = reinterpret_cast<uint64_t*>(tab + A.tab_bytes);
    uint64_t* empty = full + A.NS;
    uint64_t* tbar = empty + A.NS;
    int* slot_rb = reinterpret_cast<int*>(tbar + 1);  // row block of the stage in each slot (-1: no more)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NS = A.NS, nsl = A.nsl;

    if (threadIdx.x < 2 * NS + 1) mbar_init(full + threadIdx.x, threadIdx.x < NS ? 1u : threadIdx.x < 2 * NS ? (uint32_t)kIdWarps : 1u);
    fence_barrier_init();
    __syncthreads();

    if (warp == kIdWarps) {
        if (lane != 0) return;
        // stages in order: the nsl slices of row block blockIdx.x (gridDim.x <= row blocks), then of
        // each block taken from the counter, then one end marker (a slot completed without data)
        uint32_t issued = 0;
        bool marker = false;
        int rb = (int)blockIdx.x, s = 0;
        auto issue = [&]() {
            const int slot = (int)(issued % NS);
            slot_rb[slot] = rb;
            mbar_expect_tx(full + slot, SB);
            tma_load_2d(ring + (size_t)slot * SB, &A.map, s * (SLB / 4), rb * kIdRows, full + slot);
            issued++;
            s++;
        };
        while (issued < (uint32_t)NS && s < nsl) issue();  // the weights do not depend on k_xquant
        grid_dep_wait();
        mbar_expect_tx(tbar, A.tab_bytes);
        bulk_load(tab, A.tab, A.tab_bytes, tbar);
        for (;;) {
            if (s == nsl) {
                rb = (int)gridDim.x + (int)atomicAdd(A.counter, 1u);
                s = 0;
            }
            if (issued >= (uint32_t)NS && !mbar_wait(empty + issued % NS, ((issued / NS) + 1u) & 1u)) {
                flag(A.st, FPX_ETIMEOUT);
                break;
            }
            if (rb >= A.nrb) {
                slot_rb[issued % NS] = -1;
                mbar_arrive(full + issued % NS);
                marker = true;
                break;
            }
            issue();
        }
        // nothing may land after the CTA exits: wait (bounded) for the table and the copies of the last
        // NS stages. With the end marker placed, its slot's previous copy was consumed (the marker
        // waited for that slot to be released) and the slot's barrier has moved one phase further, so
        // that stage is skipped.
        mbar_wait(tbar, 0u);
        uint32_t first = issued > (uint32_t)NS ? issued - NS : 0u;
        if (marker && issued >= (uint32_t)NS) first = issued - NS + 1;
        for (uint32_t n = first; n < issued; n++) mbar_wait(full + n % NS, (n / NS) & 1u);
        return;
    }

    // consumers
    if (!mbar_wait_warp(smem_u32(tbar), 0u)) {
        if (lane == 0) flag(A.st, FPX_ETIMEOUT);
        return;
    }
    const uint32_t lane_off = (uint32_t)(lane * BB) & ~3u, sh = ((uint32_t)(lane * BB) & 3u) * 8u;
    const uint32_t code_base = smem_u32(tab) + (uint32_t)lane * 16u;
    const float* cscale = reinterpret_cast<const float*>(tab + xtab_code_bytes(A.nbp, Q));
    uint32_t bad = 0;
    float yacc = 0.0f;
    int s = 0;
    for (uint32_t n = 0;; n++) {
        const int slot = (int)(n % NS);
        if (!mbar_wait_warp(smem_u32(full + slot), (n / NS) & 1u)) {
            if (lane == 0) flag(A.st, FPX_ETIMEOUT);
            break;
        }
        const int rbi = slot_rb[slot];
        if (rbi < 0) break;
        // activation bytes of block 32 s + lane: hi[t][8], lo[t][8] words, and the column scales
        uint32_t xh[Q][8], xl[Q][8];
        float cs[Q];
        const int b = s * 32 + lane;
#pragma unroll
        for (int t = 0; t < Q; t++) {
#pragma unroll
            for (int h = 0; h < 2; h++) {
                const uint32_t ah = code_base + (uint32_t)(((4 * t + h) * A.nbp + s * 32) * 16);
                const uint32_t al = code_base + (uint32_t)(((4 * t + 2 + h) * A.nbp + s * 32) * 16);
                const uint4 vh = lds128<0>(ah), vl = lds128<0>(al);
                xh[t][4 * h] = vh.x; xh[t][4 * h + 1] = vh.y; xh[t][4 * h + 2] = vh.z; xh[t][4 * h + 3] = vh.w;
                xl[t][4 * h] = vl.x; xl[t][4 * h + 1] = vl.y; xl[t][4 * h + 2] = vl.z; xl[t][4 * h + 3] = vl.w;
            }
            cs[t] = cscale[t * A.nbp + b];
        }
        const uint32_t rowa = smem_u32(ring + (size_t)slot * SB) + (uint32_t)(warp * kIdRowsPerWarp * SLB) + lane_off;
        float v[V];
        auto row = [&](auto rr_c) {
            constexpr int rr = decltype(rr_c)::value;
            uint32_t w[8];
            const float d = decode_row<FMT, rr * SLB>(rowa, sh, w, bad);
#pragma unroll
            for (int t = 0; t < QP; t++) {
                if (t < Q) {
                    // two independent chains (high and low activation bytes), joined once
                    int ah = 0, al = 0;
#pragma unroll
                    for (int i = 0; i < 8; i++) {
                        ah = dp4a_ss(w[i], xh[t][i], ah);
                        al = dp4a_su(w[i], xl[t][i], al);
                    }
                    v[rr * QP + t] = (__int2float_rn(ah * 256 + al) * d) * cs[t];
                } else {
                    v[rr * QP + t] = 0.0f;
                }
            }
        };
        row(std::integral_constant<int, 0>{});
        row(std::integral_constant<int, 1>{});
        row(std::integral_constant<int, 2>{});
        row(std::integral_constant<int, 3>{});
        row(std::integral_constant<int, 4>{});
        row(std::integral_constant<int, 5>{});
        row(std::integral_constant<int, 6>{});
        row(std::integral_constant<int, 7>{});
        __syncwarp();
        if (lane == 0) mbar_arrive(empty + slot);
        const float tot = transpose_reduce<V>(v, lane);
        yacc = s == 0 ? tot : yacc + tot;
        if (s == nsl - 1) {
            const int i = lane >> (5 - L);
            const int rr = i / QP, t = i % QP;
            const int r = rbi * kIdRows + warp * kIdRowsPerWarp + rr;
            if ((lane & ((1 << (5 - L)) - 1)) == 0 && t < Q && r < A.N) A.y[(size_t)t * A.N + r] = yacc;
            s = 0;
        } else {
            s++;
        }
    }
    if (__any_sync(0xffffffffu, bad != 0u) && lane == 0) flag(A.st, FPX_EDATA);
}

inline int make_slice_map(CUtensorMap* m, const void* base, int64_t row_bytes, int64_t rows, int slice_b) {
    auto enc = tensor_map_encoder();
    if (!enc) return FPX_ECUDA;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes / 4), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(slice_b / 4), static_cast<cuuint32_t>(kIdRows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FPX_OK : FPX_ECUDA;
}

constexpr size_t kIdBarBytes = 8 * (2 * kIdMaxStages + 1) + 4 * kIdMaxStages;  // barriers, slot row blocks

template <int FMT, int Q>
int launch_idot(const uint8_t* Wq, int64_t N, int64_t K, const void* x, int x_bf16, float* y, uint8_t* ws,
                int32_t* st, cudaStream_t s) {
    const DeviceInfo di = device_info();
    const int nblk = (int)(K / 32), nsl = (nblk + 31) / 32, nbp = nsl * 32;
    const size_t tabB = xtab_bytes(nbp, Q);
    const int64_t avail = (int64_t)di.smem_optin - 128 - (int64_t)kIdBarBytes - (int64_t)tabB;
    const int NS = (int)std::min<int64_t>(kIdMaxStages, avail > 0 ? avail / id_stage_bytes(FMT) : 0);
    if (NS < 2) return FPX_EINVAL;  // K * q too large for the activation table in shared memory
    IdotArgs A{};
    const int64_t row_bytes = (int64_t)nblk * block_bytes(FMT);
    int rc = make_slice_map(&A.map, Wq, row_bytes, N, slice_bytes(FMT));
    if (rc) return rc;
    A.N = (int)N; A.nsl = nsl; A.nbp = nbp; A.nrb = (int)((N + kIdRows - 1) / kIdRows); A.NS = NS;
    A.tab_bytes = (uint32_t)tabB; A.tab = ws; A.counter = reinterpret_cast<uint32_t*>(ws + tabB); A.y = y; A.st = st;
    const int units = Q * nbp;
    k_xquant<FMT><<<(units + 7) / 8, 256, 0, s>>>(x, x_bf16, (int)K, Q, nbp, ws, st);
    if (cudaGetLastError() != cudaSuccess) return FPX_ECUDA;
    const size_t smem = 128 + (size_t)NS * id_stage_bytes(FMT) + tabB + kIdBarBytes;
    if (cudaFuncSetAttribute(k_gemv_idot<FMT, Q>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) return FPX_ECUDA;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)std::min<int64_t>(A.nrb, di.sms));
    cfg.blockDim = dim3(kIdThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, k_gemv_idot<FMT, Q>, A) != cudaSuccess) return FPX_ECUDA;
    return launch_status();
}

template <int FMT>
int launch_idot_q(const uint8_t* Wq, int64_t N, int64_t K, const void* x, int x_bf16, int q, float* y, uint8_t* ws,
                  int32_t* st, cudaStream_t s) {
    switch (q) {
        case 1: return launch_idot<FMT, 1>(Wq, N, K, x, x_bf16, y, ws, st, s);
        case 2: return launch_idot<FMT, 2>(Wq, N, K, x, x_bf16, y, ws, st, s);
        case 3: return launch_idot<FMT, 3>(Wq, N, K, x, x_bf16, y, ws, st, s);
        case 4: return launch_idot<FMT, 4>(Wq, N, K, x, x_bf16, y, ws, st, s);
        default: return FPX_EINVAL;
    }
}

}  // namespace
}  // namespace fpx

using namespace fpx;

extern "C" {

size_t fpx_gemv_idot_workspace_bytes(int64_t K, int q) {
    if (K < 0 || K % 32 || q < 1 || q > 4 || K > INT32_MAX / 8) return 0;
    const int64_t nbp = (K / 32 + 31) / 32 * 32;
    return idot_ws_bytes((int)nbp, q);
}

int fpx_gemv_q_idot(int fmt, const uint8_t* Wq, int64_t N, int64_t K, const void* x, int x_dtype, int q, float* y,
                    void* ws, size_t ws_bytes, int32_t* dev_status, void* stream) {
    if (matrix_bytes(fmt, N, K) < 0 || q < 1 || q > 4 || (x_dtype != FPX_DTYPE_F32 && x_dtype != FPX_DTYPE_BF16))
        return FPX_EINVAL;
    if (N > INT32_MAX || K > INT32_MAX / 8 || !mma_shape_ok(fmt, K == 0 ? 64 * box_chunks(fmt) : K)) return FPX_EINVAL;
    if (N == 0) return FPX_OK;
    if (!Wq || !x || !y) return FPX_EINVAL;
    if (!aligned(Wq, 16) || !aligned(x, 4) || !aligned(y, 4)) return FPX_EALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0) return cudaMemsetAsync(y, 0, sizeof(float) * (size_t)q * N, s) == cudaSuccess ? FPX_OK : FPX_ECUDA;
    if (!ws) return FPX_EINVAL;
    if (ws_bytes < fpx_gemv_idot_workspace_bytes(K, q)) return FPX_ESPACE;
    if (!aligned(ws, 16)) return FPX_EALIGN;
    const int bf = x_dtype == FPX_DTYPE_BF16;
    uint8_t* w = static_cast<uint8_t*>(ws);
    if (fmt == 2) return launch_idot_q<2>(Wq, N, K, x, bf, q, y, w, dev_status, s);
    if (fmt == 3) return launch_idot_q<3>(Wq, N, K, x, bf, q, y, w, dev_status, s);
    return launch_idot_q<4>(Wq, N, K, x, bf, q, y, w, dev_status, s);
}

}  // extern "C"
