// Core entry points: sizes, status, dequantize, quantize, and the dense FPX GEMV.
//
// The GEMV runs on the tensor-core decode engine (fpx_mma.cuh) whenever a row is a whole number of
// TMA boxes (K % 256 == 0 for FP2/FP3, K % 512 == 0 for FP4) and the activation table fits in shared
// memory; other shapes use the CUDA-core kernel. The choice depends only on the format and K, never on
// q, so every column of a call is bit-identical to the same column computed alone.
#include "fpx_mma.cuh"

#include <cmath>

using namespace fpx;

namespace {

// ------------------------------------------------------------------ dequantize

template <int FMT>
__global__ void k_dequantize(const uint8_t* __restrict__ Wq, int64_t nblocks, float* __restrict__ W, int32_t* st) {
    for (int64_t b = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; b < nblocks; b += (int64_t)gridDim.x * blockDim.x) {
        float v[32];
        float s = decode_levels<FMT>(Wq + b * block_bytes(FMT), v, st);
        float4* o = reinterpret_cast<float4*>(W + b * 32);
#pragma unroll
        for (int j = 0; j < 8; j++) o[j] = make_float4(s * v[4 * j], s * v[4 * j + 1], s * v[4 * j + 2], s * v[4 * j + 3]);
    }
}

// ------------------------------------------------------------------ quantize

// FP2/FP3 code from |v| against the exact midpoints 2d, 4d, 6d (ties to the smaller magnitude).
template <int FMT>
__device__ __forceinline__ uint32_t odd_code(float v, float d) {
    float a = fabsf(v);
    uint32_t i = 0;
#pragma unroll
    for (int m = 1; m <= (FMT == 2 ? 1 : 3); m++) i += (a > 2.0f * m * d) ? 1u : 0u;
    const uint32_t half = FMT == 2 ? 2u : 4u;
    return signbit(v) ? half - 1u - i : half + i;
}

// E2M1 magnitude index of t >= 0 (exact binary64): nearest grid value, ties to the even index.
__device__ __forceinline__ uint32_t e2m1_round(double t) {
    // grid 0 .5 1 1.5 2 3 4 6; midpoints .25 .75 1.25 1.75 2.5 3.5 5
    const double mid[7] = {0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0};
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 7; i++) {
        // above the midpoint -> next level; exactly on it -> the even index of the pair
        if (t > mid[i] || (t == mid[i] && ((i + 1) & 1) == 0)) m = i + 1;
    }
    return m;
}

template <int FMT>
__global__ void k_quantize(const float* __restrict__ W, int64_t N, int64_t K, const float* __restrict__ scales,
                           uint8_t* __restrict__ out, int32_t* st) {
    const int64_t nb = K / 32, total = N * nb;
    for (int64_t b = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; b < total; b += (int64_t)gridDim.x * blockDim.x) {
        const float* v = W + (b / nb) * K + (b % nb) * 32;
        uint8_t* p = out + b * block_bytes(FMT);
        float amax = 0.0f;
        bool finite = true;
        float x[32];
#pragma unroll
        for (int j = 0; j < 32; j++) {
            x[j] = v[j];
            finite = finite && isfinite(x[j]);
            amax = fmaxf(amax, fabsf(x[j]));
        }
        if (!finite) { flag(st, FPX_ERANGE); continue; }
        if constexpr (FMT == 2 || FMT == 3) {
            double src = scales ? (double)scales[b] : (double)amax / (FMT == 2 ? 3.0 : 7.0);
            if (scales && !(src >= 0.0 && src <= 3.4e38)) { flag(st, FPX_EINVAL); continue; }
            __half h = __double2half(src);
            uint16_t hb = __half_as_ushort(h);
            if ((hb & 0x7C00u) == 0x7C00u) { flag(st, FPX_ERANGE); continue; }
            float d = __half2float(h);
            uint32_t lo[2] = {0u, 0u}, hi = 0u;
#pragma unroll
            for (int j = 0; j < 32; j++) {
                uint32_t c = odd_code<FMT>(x[j], d);
                lo[j >> 4] |= (c & 3u) << (2 * (j & 15));
                if (FMT == 3) hi |= ((c >> 2) & 1u) << j;
            }
            p[0] = hb & 0xFF; p[1] = hb >> 8;
#pragma unroll
            for (int i = 0; i < 4; i++) { p[2 + i] = (lo[0] >> (8 * i)) & 0xFF; p[6 + i] = (lo[1] >> (8 * i)) & 0xFF; }
            if (FMT == 3) {
#pragma unroll
                for (int i = 0; i < 4; i++) p[10 + i] = (hi >> (8 * i)) & 0xFF;
            }
        } else {
            int e;
            if (scales) {
                float s = scales[b];
                int ex;
                float m = frexpf(s, &ex);
                e = ex - 1 + 127;
                if (!(s > 0.0f) || !isfinite(s) || m != 0.5f || e < 0 || e > 254) { flag(st, FPX_EINVAL); continue; }
            } else if (amax == 0.0f) {
                e = 0;
            } else {
                int ex;
                frexpf(amax, &ex);  // floor(log2 amax) = ex - 1
                e = min(254, max(0, ex - 1 - 2 + 127));
            }
            const double inv = ldexp(1.0, 127 - e);
            p[0] = (uint8_t)e;
#pragma unroll
            for (int j = 0; j < 16; j++) {
                uint32_t q0 = e2m1_round(fabs((double)x[2 * j]) * inv) | (signbit(x[2 * j]) ? 8u : 0u);
                uint32_t q1 = e2m1_round(fabs((double)x[2 * j + 1]) * inv) | (signbit(x[2 * j + 1]) ? 8u : 0u);
                p[1 + j] = (uint8_t)(q0 | (q1 << 4));
            }
        }
    }
}

// Importance-weighted quantizer: per block, the candidate scales (amax / Kmax) * (12 + j) / 20,
// j = 0..15, rounded to binary16 (FP2/FP3), or the E8M0 exponents e0 - 1, e0, e0 + 1 (FP4); under each,
// the codes of k_quantize; the kept candidate has the least sum over the block of
// imp[col] * (w - w_hat)^2, evaluated in binary64 in weight order with explicitly rounded operations
// (no fused multiply-add), the earliest candidate on equal sums. The zh-TW page, section "ROCmFPX"
// (quantization guided by an importance matrix); the importance here is any caller vector.
template <int FMT>
__device__ __forceinline__ double block_werr(const float (&x)[32], const float* imp, float d, int e) {
    double err = 0.0;
#pragma unroll
    for (int j = 0; j < 32; j++) {
        double w;
        if constexpr (FMT == 4) {
            const double inv = ldexp(1.0, 127 - e), sc = ldexp(1.0, e - 127);
            const uint32_t m = e2m1_round(fabs((double)x[j]) * inv);
            const double g[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
            w = __dmul_rn(signbit(x[j]) ? -g[m] : g[m], sc);
        } else {
            const int kmax = FMT == 2 ? 3 : 7;
            const int c = (int)odd_code<FMT>(x[j], d);
            w = __dmul_rn((double)d, (double)(2 * c - kmax));
        }
        const double diff = __dsub_rn((double)x[j], w);
        err = __dadd_rn(err, __dmul_rn(imp ? (double)imp[j] : 1.0, __dmul_rn(diff, diff)));
    }
    return err;
}

template <int FMT>
__global__ void k_quantize_weighted(const float* __restrict__ W, int64_t N, int64_t K, const float* __restrict__ imp,
                                    uint8_t* __restrict__ out, int32_t* st) {
    const int64_t nb = K / 32, total = N * nb;
    for (int64_t b = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; b < total; b += (int64_t)gridDim.x * blockDim.x) {
        const float* v = W + (b / nb) * K + (b % nb) * 32;
        const float* im = imp ? imp + (b % nb) * 32 : nullptr;
        uint8_t* p = out + b * block_bytes(FMT);
        float x[32];
        float amax = 0.0f;
        bool finite = true;
#pragma unroll
        for (int j = 0; j < 32; j++) {
            x[j] = v[j];
            finite = finite && isfinite(x[j]) && (!im || (isfinite(im[j]) && im[j] >= 0.0f));
            amax = fmaxf(amax, fabsf(x[j]));
        }
        if (!finite) { flag(st, FPX_ERANGE); continue; }
        if constexpr (FMT == 2 || FMT == 3) {
            const double kmax = FMT == 2 ? 3.0 : 7.0;
            bool found = false;
            double best = 0.0;
            uint16_t bh = 0;
            for (int j = 0; j < 16; j++) {
                const __half h = __double2half(__dmul_rn(__ddiv_rn((double)amax, kmax), __ddiv_rn((double)(12 + j), 20.0)));
                const uint16_t hb = __half_as_ushort(h);
                if ((hb & 0x7C00u) == 0x7C00u) continue;
                const double err = block_werr<FMT>(x, im, __half2float(h), 0);
                if (!found || err < best) { best = err; bh = hb; found = true; }
            }
            if (!found) { flag(st, FPX_ERANGE); continue; }
            const float d = __half2float(__ushort_as_half(bh));
            uint32_t lo[2] = {0u, 0u}, hi = 0u;
#pragma unroll
            for (int j = 0; j < 32; j++) {
                const uint32_t c = odd_code<FMT>(x[j], d);
                lo[j >> 4] |= (c & 3u) << (2 * (j & 15));
                if (FMT == 3) hi |= ((c >> 2) & 1u) << j;
            }
            p[0] = bh & 0xFF; p[1] = bh >> 8;
#pragma unroll
            for (int i = 0; i < 4; i++) { p[2 + i] = (lo[0] >> (8 * i)) & 0xFF; p[6 + i] = (lo[1] >> (8 * i)) & 0xFF; }
            if (FMT == 3) {
#pragma unroll
                for (int i = 0; i < 4; i++) p[10 + i] = (hi >> (8 * i)) & 0xFF;
            }
        } else {
            int e0 = 0;
            if (amax != 0.0f) {
                int ex;
                frexpf(amax, &ex);  // floor(log2 amax) = ex - 1
                e0 = min(254, max(0, ex - 1 - 2 + 127));
            }
            bool found = false;
            double best = 0.0;
            int be = e0;
            for (int j = -1; j <= 1; j++) {
                const int e = min(254, max(0, e0 + j));
                const double err = block_werr<FMT>(x, im, 0.0f, e);
                if (!found || err < best) { best = err; be = e; found = true; }
            }
            const double inv = ldexp(1.0, 127 - be);
            p[0] = (uint8_t)be;
#pragma unroll
            for (int j = 0; j < 16; j++) {
                uint32_t q0 = e2m1_round(fabs((double)x[2 * j]) * inv) | (signbit(x[2 * j]) ? 8u : 0u);
                uint32_t q1 = e2m1_round(fabs((double)x[2 * j + 1]) * inv) | (signbit(x[2 * j + 1]) ? 8u : 0u);
                p[1 + j] = (uint8_t)(q0 | (q1 << 4));
            }
        }
    }
}

// ------------------------------------------------------------------ GEMV, CUDA-core path

constexpr int kGemvThreads = 256;

template <int FMT, int Q, bool XSMEM>
__global__ void __launch_bounds__(kGemvThreads) k_gemv_cc(const uint8_t* __restrict__ Wq, int N, int K, const void* x,
                                                          int x_bf16, float* __restrict__ y, int32_t* st) {
    extern __shared__ float xs[];
    const int xstride = padded_len(K);
    if (XSMEM) {
        for (int i = threadIdx.x; i < Q * K; i += blockDim.x) {
            int t = i / K, k = i % K;
            float v = x_bf16 ? bf16_bits_to_float(reinterpret_cast<const uint16_t*>(x)[i]) : reinterpret_cast<const float*>(x)[i];
            xs[t * xstride + padded_index(k)] = v;
        }
        __syncthreads();
    }
    const int lane = threadIdx.x & 31;
    const int warps = blockDim.x / 32;
    const int nblk = K / 32;
    const int64_t row_bytes = (int64_t)nblk * block_bytes(FMT);
    for (int r = blockIdx.x * warps + threadIdx.x / 32; r < N; r += gridDim.x * warps) {
        float acc[Q];
        if (XSMEM) row_dot<FMT, Q>(Wq + r * row_bytes, nblk, XShared{xs, xstride}, lane, acc, st);
        else row_dot<FMT, Q>(Wq + r * row_bytes, nblk, XGlobal{x, K, x_bf16}, lane, acc, st);
        if (lane < Q) {
            float o = acc[0];
#pragma unroll
            for (int t = 1; t < Q; t++) o = lane == t ? acc[t] : o;
            y[(int64_t)lane * N + r] = o;
        }
    }
}

template <int FMT, int Q>
int launch_gemv_cc_q(const uint8_t* Wq, int64_t N, int64_t K, const void* x, int x_bf16, float* y, int32_t* st,
                     cudaStream_t s) {
    DeviceInfo di = device_info();
    size_t smem = (size_t)Q * padded_len((int)K) * sizeof(float);
    int64_t grid64 = (N + 7) / 8;
    int grid = (int)(grid64 < di.sms * 4 ? grid64 : di.sms * 4);
    if (grid < 1) grid = 1;
    if ((int64_t)smem <= di.smem_optin) {
        if (cudaFuncSetAttribute(k_gemv_cc<FMT, Q, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem))
            return FPX_ECUDA;
        k_gemv_cc<FMT, Q, true><<<grid, kGemvThreads, smem, s>>>(Wq, (int)N, (int)K, x, x_bf16, y, st);
    } else {
        k_gemv_cc<FMT, Q, false><<<grid, kGemvThreads, 0, s>>>(Wq, (int)N, (int)K, x, x_bf16, y, st);
    }
    return launch_status();
}

// ------------------------------------------------------------------ GEMV, tensor-core path

// A CTA processes groups of kWarps / S row tiles; the S warps of a tile split its K range and their
// partial sums are added in split order. Each warp streams its (tile, split) boxes through its ring.
// A row tile is gemv_tile_rows(FMT) rows: 32 for FP2 / FP3 (two 16-row MMA tiles sharing the
// activations), 16 for FP4, so that one TMA copy moves 2.5 / 3.5 / 4.3 KB: the single producer thread
// pays a fixed cost per copy, and small boxes left it, not HBM, setting the rate.
__host__ __device__ constexpr int gemv_tile_rows(int fmt) { return fmt == 4 ? 16 : 32; }
static_assert(32 * box_bytes(3) <= kSlotBytes && 16 * box_bytes(4) <= kSlotBytes, "tile fits a ring slot");
// One producer warp per consumer warp (lane 0 issues that warp's copies): the per-copy cost is paid
// by the issuing thread, so several issuers multiply the rate at which boxes can start. Measured on a
// 194 MB FP2 matrix at q = 4: 1 issuer 1.46 TB/s, 2 issuers 2.21, 4 issuers 2.98, 8 issuers 3.07.
constexpr int kGemvProducers = 8;
constexpr int kGemvMmaThreads = (kWarps + kGemvProducers) * 32;
struct GemvArgs {
    CUtensorMap map;
    int N, K, S;
    const void* x;
    int x_bf16;
    float* y;
    int32_t* st;
    uint32_t magic;  // kMagic, kept out of immediates (see decode_fp2)
};

template <int FMT, int Q>
__global__ void __launch_bounds__(kGemvMmaThreads, 1) k_gemv_mma(const __grid_constant__ GemvArgs A) {
    constexpr int TR = gemv_tile_rows(FMT), NT = TR / 16;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int shift[4];
    __shared__ float red4[(kWarps + kGemvProducers) * 4];
    __shared__ float part[kWarps][TR][4];
    const int K = A.K, N = A.N, S = A.S, tpg = kWarps / S;
    const Smem Sm = carve(smem, btab_bytes(K), FMT == 3 ? 2 : 1);
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    init_rings(Sm);
    const int U = K / (64 * box_chunks(FMT)) / S;  // boxes per (tile, split)
    const int ntiles = (N + TR - 1) / TR, ngroups = (ntiles + tpg - 1) / tpg;
    const int my_groups = (int)blockIdx.x < ngroups ? (ngroups - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;

    // producers: consumer warp w = (tile in group) * S + split streams U boxes per group; producer p
    // serves warps p, p + kGemvProducers, ... (its i-th warp is w = p + kGemvProducers * i)
    constexpr int kPer = kWarps / kGemvProducers;
    uint32_t issued[kPer];
    const bool producer = warp >= kWarps && lane == 0;
    const int pw = warp - kWarps;
    auto try_issue = [&](int i) -> bool {
        const int w = pw + kGemvProducers * i;
        const uint32_t n = issued[i];
        if (n >= (uint32_t)(my_groups * U)) return false;
        const Ring R = warp_ring(Sm, w);
        if (!ring_free(R, n)) return false;
        const int grp = (int)blockIdx.x + (int)(n / U) * (int)gridDim.x, u = (int)(n % U);
        const int tile = grp * tpg + w / S, split = w % S;  // rows past N read as zeros
        const int slot = n % kStages;
        mbar_expect_tx(R.full + slot, TR * box_bytes(FMT));
        tma_load_2d(R.slots + (size_t)slot * kSlotBytes, &A.map, (split * U + u) * (box_bytes(FMT) / elem_bytes(FMT)),
                    tile * TR, R.full + slot);
        issued[i] = n + 1;
        return true;
    };
    if (producer) {
#pragma unroll
        for (int i = 0; i < kPer; i++) issued[i] = 0u;
        for (int j = 0; j < kStages; j++)
#pragma unroll
            for (int i = 0; i < kPer; i++) try_issue(i);
    }

    if (A.x_bf16)
        build_tables<FMT, false>(SrcBF16{reinterpret_cast<const uint16_t*>(A.x)}, K, Q, Sm.tab0, Sm.tab1, nullptr, Sm.oq, shift, red4);
    else
        build_tables<FMT, false>(SrcF32{reinterpret_cast<const float*>(A.x)}, K, Q, Sm.tab0, Sm.tab1, nullptr, Sm.oq, shift, red4);
    __syncthreads();

    if (warp >= kWarps) {
        if (producer) {
            uint64_t idle_since = 0;
            for (;;) {
                bool pending = false, progress = false;
#pragma unroll
                for (int i = 0; i < kPer; i++) {
                    if (issued[i] < (uint32_t)(my_groups * U)) pending = true;
                    progress |= try_issue(i);
                }
                if (!pending) break;
                if (progress) {
                    idle_since = 0;
                } else {
                    const uint64_t now = global_ns();
                    if (!idle_since) idle_since = now;
                    else if (now - idle_since > kWaitNs) { flag(A.st, FPX_ETIMEOUT); break; }
                    __nanosleep(100);
                }
            }
        }
        return;
    }

    const int split = warp % S;
    const Ring R = warp_ring(Sm, warp);
    const int a_idx = b_active_index(lane);
    const LaneOfs lofs = lane_ofs<FMT>(t);
    uint32_t consumed = 0, bad = 0;
    bool ok = true;
    for (int n = 0; n < my_groups; n++) {
        const int grp = (int)blockIdx.x + n * (int)gridDim.x;
        float y[NT][4];
#pragma unroll
        for (int i = 0; i < NT; i++) y[i][0] = y[i][1] = y[i][2] = y[i][3] = 0.f;
        for (int u = 0; u < U && ok; u++) {
            if (!ring_wait(R, consumed, A.st)) { ok = false; break; }
            const uint8_t* slot = R.slots + (consumed % kStages) * kSlotBytes;
            const int chunk0 = (split * U + u) * box_chunks(FMT);
            box_tiles<FMT, NT, box_chunks(FMT)>(smem_u32(slot) + g * box_bytes(FMT), lofs, lane_tab(Sm.tab0, Sm.zero, a_idx, chunk0),
                                               lane_tab(Sm.tab1, Sm.zero, a_idx, chunk0), lane_oq(Sm.oq, chunk0, t), A.magic, y, bad);
            ring_release(R, consumed);
            consumed++;
        }
#pragma unroll
        for (int n = 0; n < NT; n++) {
            pair_reduce(y[n]);
            if (t < 2) {
#pragma unroll
                for (int i = 0; i < 4; i++) part[warp][16 * n + g + 8 * (i >> 1)][2 * t + (i & 1)] = y[n][i];
            }
        }
        consumers_sync();
        for (int o = threadIdx.x; o < tpg * TR * Q; o += kWarps * 32) {
            const int tg = o / (TR * Q), row = (o / Q) % TR, tok = o % Q;
            float acc = part[tg * S][row][tok];
            for (int s = 1; s < S; s++) acc += part[tg * S + s][row][tok];
            const int rr = (grp * tpg + tg) * TR + row;
            if (rr < N) A.y[(size_t)tok * N + rr] = acc * exp2i((FMT == 4 ? 14 : 0) - shift[tok]);
        }
        consumers_sync();
    }
    report_bad(bad, A.st);
    if (!ok) ring_drain(R, consumed, (uint32_t)(my_groups * U));
}

template <int FMT>
bool gemv_mma_fits(int64_t K) {
    return mma_shape_ok(FMT, K) && smem_bytes(btab_bytes((int)K), FMT == 3 ? 2 : 1) <= (size_t)device_info().smem_optin;
}

template <int FMT, int Q>
int launch_gemv_mma_q(const uint8_t* Wq, int64_t N, int64_t K, const void* x, int x_bf16, float* y, int32_t* st,
                      cudaStream_t s) {
    DeviceInfo di = device_info();
    GemvArgs A{};
    const int64_t rb = K / 32 * block_bytes(FMT);
    int rc = make_row_map(&A.map, Wq, rb, N, rb, box_bytes(FMT), gemv_tile_rows(FMT), elem_bytes(FMT));
    if (rc) return rc;
    const int64_t ntiles = (N + gemv_tile_rows(FMT) - 1) / gemv_tile_rows(FMT);
    const int units = (int)(K / (64 * box_chunks(FMT)));
    int S = 1;
    while (S < kWarps && ntiles * S < (int64_t)di.sms * kWarps && units % (2 * S) == 0) S *= 2;
    A.N = (int)N; A.K = (int)K; A.S = S; A.x = x; A.x_bf16 = x_bf16; A.y = y; A.st = st;
    A.magic = kMagic;
    const int64_t ngroups = (ntiles + kWarps / S - 1) / (kWarps / S);
    const int grid = (int)(ngroups < di.sms ? ngroups : di.sms);
    const size_t smem = smem_bytes(btab_bytes((int)K), FMT == 3 ? 2 : 1);
    if (cudaFuncSetAttribute(k_gemv_mma<FMT, Q>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) return FPX_ECUDA;
    k_gemv_mma<FMT, Q><<<grid, kGemvMmaThreads, smem, s>>>(A);
    return launch_status();
}

template <int FMT>
int launch_gemv_mma(const uint8_t* Wq, int64_t N, int64_t K, const void* x, int x_bf16, int q, float* y, int32_t* st,
                    cudaStream_t s) {
    switch (q) {
        case 1: return launch_gemv_mma_q<FMT, 1>(Wq, N, K, x, x_bf16, y, st, s);
        case 2: return launch_gemv_mma_q<FMT, 2>(Wq, N, K, x, x_bf16, y, st, s);
        case 3: return launch_gemv_mma_q<FMT, 3>(Wq, N, K, x, x_bf16, y, st, s);
        case 4: return launch_gemv_mma_q<FMT, 4>(Wq, N, K, x, x_bf16, y, st, s);
        default: return FPX_EINVAL;
    }
}

template <int FMT>
int launch_gemv_cc(const uint8_t* Wq, int64_t N, int64_t K, const void* x, int x_bf16, int q, float* y, int32_t* st,
                   cudaStream_t s) {
    switch (q) {
        case 1: return launch_gemv_cc_q<FMT, 1>(Wq, N, K, x, x_bf16, y, st, s);
        case 2: return launch_gemv_cc_q<FMT, 2>(Wq, N, K, x, x_bf16, y, st, s);
        case 3: return launch_gemv_cc_q<FMT, 3>(Wq, N, K, x, x_bf16, y, st, s);
        case 4: return launch_gemv_cc_q<FMT, 4>(Wq, N, K, x, x_bf16, y, st, s);
        default: return FPX_EINVAL;
    }
}

}  // namespace

// ------------------------------------------------------------------ box-tiled matrices

// Box-tiled layout (the MoE layer kernels stream it with 1-D bulk copies): a matrix of N rows is cut
// into tiles of R = stage_rows(fmt) rows x B = box_bytes(fmt) bytes of each row (256 x 80 FP2, 256 x 112
// FP3, 64 x 272 FP4), stored contiguously in the order (row block, column piece): tile
// (r / R) * P + j / B for byte j of row r, P = row_bytes / B.
// FP4 tiles hold the rows' bytes at a pitch of B. FP2 / FP3 tiles hold a code area of R rows x 64 / 96
// bytes and then a scale area of R rows x 16 bytes, regrouped per row as described with
// box_code_bytes (fpx_mma.cuh): FP2 word 4t + C = code word t % 2 of block 2C + t / 2; FP3 bytes
// 24t .. 24t + 23 = the 3-bit codes of blocks 2C + t / 2, codes 16 (t % 2) .. +15, at the fields of
// fp3_slot; scale 4h + C = the scale of block 2C + h.
__global__ void k_tile(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int64_t units, int64_t row_units,
                       int R, int B16, int64_t src_stride, int64_t dst_stride, int inverse) {
    const uint8_t* sm = src + (int64_t)blockIdx.y * src_stride;
    uint8_t* dm = dst + (int64_t)blockIdx.y * dst_stride;
    const int64_t P = row_units / B16, tile_units = (int64_t)R * B16;
    for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < units; u += (int64_t)gridDim.x * blockDim.x) {
        // u: 16-byte unit of the tiled matrix -> its row-major unit
        const int64_t t = u / tile_units, o = u % tile_units;
        const int64_t r = (t / P) * R + o / B16, j = (t % P) * B16 + o % B16;
        const int64_t v = r * row_units + j;
        if (inverse) reinterpret_cast<uint4*>(dm)[v] = reinterpret_cast<const uint4*>(sm)[u];
        else reinterpret_cast<uint4*>(dm)[u] = reinterpret_cast<const uint4*>(sm)[v];
    }
}

// 3-bit code c of FP3 field (odd, p, half hh) in the three words W of a chunk pair.
__device__ __forceinline__ void fp3_put(uint32_t (&W)[3], int odd, int p, int hh, uint32_t c) {
    const int f = fp3_slot(odd, p);
    if (f < 0) {
        for (int i = 0; i < 3; i++) W[i] |= ((c >> i) & 1u) << (16 * hh);
    } else {
        W[f / 16] |= c << (16 * hh + f % 16);
    }
}
__device__ __forceinline__ uint32_t fp3_get(const uint32_t (&W)[3], int odd, int p, int hh) {
    const int f = fp3_slot(odd, p);
    if (f < 0) {
        uint32_t c = 0;
        for (int i = 0; i < 3; i++) c |= ((W[i] >> (16 * hh)) & 1u) << i;
        return c;
    }
    return (W[f / 16] >> (16 * hh + f % 16)) & 7u;
}

// FP2 / FP3: one thread per (row, column piece) regroups the B row-major bytes of the piece into the
// tile's code and scale areas (or back, inverse).
template <int FMT>
__global__ void k_tile_rows(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int64_t pieces, int64_t P,
                            int64_t row_bytes, int64_t src_stride, int64_t dst_stride, int inverse) {
    constexpr int B = box_bytes(FMT), BB = block_bytes(FMT), CB = box_code_bytes(FMT), R = 256;
    const uint8_t* sm = src + (int64_t)blockIdx.y * src_stride;
    uint8_t* dm = dst + (int64_t)blockIdx.y * dst_stride;
    for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < pieces; u += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = u / P, jt = u % P;
        const int64_t rm = r * row_bytes + jt * B;  // row-major offset of the piece
        const int64_t tb = ((r / R) * P + jt) * (int64_t)R * B;
        const int64_t co = tb + (r % R) * CB, so = tb + (int64_t)R * CB + (r % R) * 16;
        alignas(16) uint8_t x[B];
        alignas(16) uint8_t c[CB];
        alignas(16) uint8_t sc[16];
        if (!inverse) {
            for (int i = 0; i < B / 16; i++) reinterpret_cast<uint4*>(x)[i] = reinterpret_cast<const uint4*>(sm + rm)[i];
            for (int h = 0; h < 2; h++)
                for (int C = 0; C < 4; C++) {
                    sc[2 * (4 * h + C)] = x[BB * (2 * C + h)];
                    sc[2 * (4 * h + C) + 1] = x[BB * (2 * C + h) + 1];
                }
            if constexpr (FMT == 2) {
                for (int t = 0; t < 4; t++)
                    for (int C = 0; C < 4; C++)
                        for (int b = 0; b < 4; b++) c[4 * (4 * t + C) + b] = x[BB * (2 * C + t / 2) + 2 + 4 * (t % 2) + b];
            } else {
                for (int t = 0; t < 4; t++)
                    for (int m = 0; m < 2; m++) {
                        uint32_t W[3] = {0u, 0u, 0u};
                        for (int odd = 0; odd < 2; odd++) {
                            const uint8_t* blk = x + BB * (2 * (2 * m + odd) + t / 2);
                            for (int j = 0; j < 16; j++) {
                                const int k = 16 * (t % 2) + j;
                                const uint32_t l = (blk[2 + k / 4] >> (2 * (k % 4))) & 3u, hb = (blk[10 + k / 8] >> (k % 8)) & 1u;
                                fp3_put(W, odd, j % 8, j / 8, l + 4u * hb);
                            }
                        }
                        for (int i = 0; i < 3; i++)
                            for (int b = 0; b < 4; b++) c[24 * t + 12 * m + 4 * i + b] = (uint8_t)(W[i] >> (8 * b));
                    }
            }
            for (int i = 0; i < CB / 16; i++) reinterpret_cast<uint4*>(dm + co)[i] = reinterpret_cast<const uint4*>(c)[i];
            reinterpret_cast<uint4*>(dm + so)[0] = reinterpret_cast<const uint4*>(sc)[0];
        } else {
            for (int i = 0; i < CB / 16; i++) reinterpret_cast<uint4*>(c)[i] = reinterpret_cast<const uint4*>(sm + co)[i];
            reinterpret_cast<uint4*>(sc)[0] = reinterpret_cast<const uint4*>(sm + so)[0];
            for (int h = 0; h < 2; h++)
                for (int C = 0; C < 4; C++) {
                    x[BB * (2 * C + h)] = sc[2 * (4 * h + C)];
                    x[BB * (2 * C + h) + 1] = sc[2 * (4 * h + C) + 1];
                }
            if constexpr (FMT == 2) {
                for (int t = 0; t < 4; t++)
                    for (int C = 0; C < 4; C++)
                        for (int b = 0; b < 4; b++) x[BB * (2 * C + t / 2) + 2 + 4 * (t % 2) + b] = c[4 * (4 * t + C) + b];
            } else {
                for (int i = 0; i < 8; i++) {  // clear the code bytes (lo and hi planes) of the 8 blocks
                    for (int b = 2; b < BB; b++) x[BB * i + b] = 0;
                }
                for (int t = 0; t < 4; t++)
                    for (int m = 0; m < 2; m++) {
                        uint32_t W[3];
                        for (int i = 0; i < 3; i++) {
                            W[i] = 0u;
                            for (int b = 0; b < 4; b++) W[i] |= (uint32_t)c[24 * t + 12 * m + 4 * i + b] << (8 * b);
                        }
                        for (int odd = 0; odd < 2; odd++) {
                            uint8_t* blk = x + BB * (2 * (2 * m + odd) + t / 2);
                            for (int j = 0; j < 16; j++) {
                                const int k = 16 * (t % 2) + j;
                                const uint32_t cc = fp3_get(W, odd, j % 8, j / 8);
                                blk[2 + k / 4] |= (uint8_t)((cc & 3u) << (2 * (k % 4)));
                                blk[10 + k / 8] |= (uint8_t)((cc >> 2) << (k % 8));
                            }
                        }
                    }
            }
            for (int i = 0; i < B / 16; i++) reinterpret_cast<uint4*>(dm + rm)[i] = reinterpret_cast<const uint4*>(x)[i];
        }
    }
}

extern "C" {

const char* fpx_status_string(int status) {
    switch (status) {
        case FPX_OK: return "ok";
        case FPX_EINVAL: return "invalid argument";
        case FPX_EALIGN: return "misaligned pointer";
        case FPX_ERANGE: return "non-finite input or scale overflow";
        case FPX_ECUDA: return "CUDA error";
        case FPX_ETIMEOUT: return "device wait timed out";
        case FPX_EDATA: return "invalid block or routing index";
        case FPX_ESPACE: return "workspace too small";
        default: return "unknown status";
    }
}

size_t fpx_block_bytes(int fmt) { return (size_t)block_bytes(fmt); }

int64_t fpx_matrix_bytes(int fmt, int64_t N, int64_t K) { return matrix_bytes(fmt, N, K); }

int fpx_read_status(const int32_t* dev_status, int32_t* host_out, void* stream) {
    if (!dev_status || !host_out) return FPX_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(host_out, dev_status, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess) return FPX_ECUDA;
    return cudaStreamSynchronize(s) == cudaSuccess ? FPX_OK : FPX_ECUDA;
}

int fpx_dequantize(int fmt, const uint8_t* Wq, int64_t N, int64_t K, float* W, int32_t* dev_status, void* stream) {
    if (matrix_bytes(fmt, N, K) < 0) return FPX_EINVAL;
    if (N == 0 || K == 0) return FPX_OK;
    if (!Wq || !W) return FPX_EINVAL;
    if (!aligned(Wq, 16) || !aligned(W, 16)) return FPX_EALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int64_t nb = N * (K / 32);
    int grid = (int)((nb + 255) / 256 < 148 * 8 ? (nb + 255) / 256 : 148 * 8);
    if (fmt == 2) k_dequantize<2><<<grid, 256, 0, s>>>(Wq, nb, W, dev_status);
    else if (fmt == 3) k_dequantize<3><<<grid, 256, 0, s>>>(Wq, nb, W, dev_status);
    else k_dequantize<4><<<grid, 256, 0, s>>>(Wq, nb, W, dev_status);
    return launch_status();
}

int fpx_quantize(int fmt, const float* W, int64_t N, int64_t K, const float* block_scales, uint8_t* out,
                 int32_t* dev_status, void* stream) {
    if (matrix_bytes(fmt, N, K) < 0) return FPX_EINVAL;
    if (N == 0 || K == 0) return FPX_OK;
    if (!W || !out) return FPX_EINVAL;
    if (!aligned(out, 16) || !aligned(W, 16) || (block_scales && !aligned(block_scales, 4))) return FPX_EALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int64_t nb = N * (K / 32);
    int grid = (int)((nb + 127) / 128 < 148 * 8 ? (nb + 127) / 128 : 148 * 8);
    if (fmt == 2) k_quantize<2><<<grid, 128, 0, s>>>(W, N, K, block_scales, out, dev_status);
    else if (fmt == 3) k_quantize<3><<<grid, 128, 0, s>>>(W, N, K, block_scales, out, dev_status);
    else k_quantize<4><<<grid, 128, 0, s>>>(W, N, K, block_scales, out, dev_status);
    return launch_status();
}

int fpx_quantize_weighted(int fmt, const float* W, int64_t N, int64_t K, const float* importance, uint8_t* out,
                          int32_t* dev_status, void* stream) {
    if (matrix_bytes(fmt, N, K) < 0) return FPX_EINVAL;
    if (N == 0 || K == 0) return FPX_OK;
    if (!W || !out) return FPX_EINVAL;
    if (!aligned(out, 16) || !aligned(W, 16) || (importance && !aligned(importance, 4))) return FPX_EALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int64_t nb = N * (K / 32);
    int grid = (int)((nb + 127) / 128 < 148 * 8 ? (nb + 127) / 128 : 148 * 8);
    if (fmt == 2) k_quantize_weighted<2><<<grid, 128, 0, s>>>(W, N, K, importance, out, dev_status);
    else if (fmt == 3) k_quantize_weighted<3><<<grid, 128, 0, s>>>(W, N, K, importance, out, dev_status);
    else k_quantize_weighted<4><<<grid, 128, 0, s>>>(W, N, K, importance, out, dev_status);
    return launch_status();
}

int fpx_tile_matrices(int fmt, const uint8_t* src, int64_t N, int64_t K, int count, int64_t src_stride, uint8_t* dst,
                      int64_t dst_stride, int inverse, void* stream) {
    if (matrix_bytes(fmt, N, K) < 0 || count < 0 || (inverse != 0 && inverse != 1)) return FPX_EINVAL;
    const int R = stage_rows(fmt), B = box_bytes(fmt);
    const int64_t row_bytes = K / 32 * block_bytes(fmt);
    if (N % R || row_bytes % B || N > INT32_MAX) return FPX_EINVAL;
    if (count == 0 || N == 0 || K == 0) return FPX_OK;
    if (!src || !dst || src == dst) return FPX_EINVAL;
    const int64_t bytes = N * row_bytes;
    if (src_stride < bytes || dst_stride < bytes) return FPX_EINVAL;
    if (!aligned(src, 16) || !aligned(dst, 16) || src_stride % 16 || dst_stride % 16) return FPX_EALIGN;
    if (count > 65535) return FPX_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (fmt == 4) {
        const int64_t units = bytes / 16;
        const int64_t gx = (units + 255) / 256 < 148 * 4 ? (units + 255) / 256 : 148 * 4;
        k_tile<<<dim3((unsigned)gx, (unsigned)count), 256, 0, s>>>(src, dst, units, row_bytes / 16, R, B / 16, src_stride,
                                                                     dst_stride, inverse);
    } else {
        const int64_t pieces = N * (row_bytes / B);
        const int64_t gx = (pieces + 127) / 128 < 148 * 8 ? (pieces + 127) / 128 : 148 * 8;
        if (fmt == 2)
            k_tile_rows<2><<<dim3((unsigned)gx, (unsigned)count), 128, 0, s>>>(src, dst, pieces, row_bytes / B, row_bytes,
                                                                               src_stride, dst_stride, inverse);
        else
            k_tile_rows<3><<<dim3((unsigned)gx, (unsigned)count), 128, 0, s>>>(src, dst, pieces, row_bytes / B, row_bytes,
                                                                               src_stride, dst_stride, inverse);
    }
    return launch_status();
}

int fpx_gemv_q(int fmt, const uint8_t* Wq, int64_t N, int64_t K, const void* x, int x_dtype, int q, float* y,
               int32_t* dev_status, void* stream) {
    if (matrix_bytes(fmt, N, K) < 0 || q < 1 || q > 4 || (x_dtype != FPX_DTYPE_F32 && x_dtype != FPX_DTYPE_BF16))
        return FPX_EINVAL;
    if (N > INT32_MAX || K > INT32_MAX / 8) return FPX_EINVAL;
    if (N == 0) return FPX_OK;
    if (!Wq || !x || !y) return FPX_EINVAL;
    // the tensor-core path's table builder reads x in 16-byte units
    if (!aligned(Wq, 16) || !aligned(x, 16) || !aligned(y, 4)) return FPX_EALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0) return cudaMemsetAsync(y, 0, sizeof(float) * (size_t)q * N, s) == cudaSuccess ? FPX_OK : FPX_ECUDA;
    int bf = x_dtype == FPX_DTYPE_BF16;
    if (fmt == 2) return gemv_mma_fits<2>(K) ? launch_gemv_mma<2>(Wq, N, K, x, bf, q, y, dev_status, s)
                                             : launch_gemv_cc<2>(Wq, N, K, x, bf, q, y, dev_status, s);
    if (fmt == 3) return gemv_mma_fits<3>(K) ? launch_gemv_mma<3>(Wq, N, K, x, bf, q, y, dev_status, s)
                                             : launch_gemv_cc<3>(Wq, N, K, x, bf, q, y, dev_status, s);
    return gemv_mma_fits<4>(K) ? launch_gemv_mma<4>(Wq, N, K, x, bf, q, y, dev_status, s)
                               : launch_gemv_cc<4>(Wq, N, K, x, bf, q, y, dev_status, s);
}

}  // extern "C"
