// Dense FPX GEMV over box-tiled matrices (fpx_tile_matrices), on the streaming CTA of the MoE layer
// kernels: one producer thread streams whole boxes (one 1-D bulk copy each, evict-first in L2) into a
// ring, and kLWarps consumer warps load their share of a box, release the slot and decode it into
// binary16 tensor-core fragments while the next box's words load (fpx_mma.cuh). The computation is
// fpx_gemv_q's ("DeepSeek V4 Flash hits 32 tok/s on AMD Ryzen AI MAX+ 395", paragraph 3: every
// packed block read and decoded once for all q columns); the box layout is what lets a consumer fetch
// a row's code words for four chunks at once.
//
// Work: a task is one row block (256 rows FP2 / FP3, 64 rows FP4) over all of K, split into P pieces
// of consecutive stages; P is a function of N and K alone (enough units for every SM), so a column's
// result does not depend on q. The units (task, piece) are dealt to the CTAs in contiguous ranges of
// equal count. With P > 1 each piece writes its own rows of a partial buffer and k_tg_sum adds a
// row's pieces in piece order.
#include "fpx_mma.cuh"

using namespace fpx;

namespace {

constexpr int kTgUnits = 592;  // P aims at this many units: 4 per SM of a 148-SM GPU

__host__ __device__ constexpr int tg_ring_slots(int fmt) { return fmt == 3 ? 5 : 7; }
__host__ __device__ constexpr int tg_slot_bytes(int fmt) { return fmt == 3 ? stage_bytes(3) : stage_bytes(2); }
// tables: FP2 [FP2 table | offset quads], FP3 [box-layout FP3 table | offset quads], FP4 [FP4 table]
__host__ __device__ constexpr int tg_tab_bytes(int fmt, int K) { return fmt == 4 ? btab_bytes(K) : btab_bytes(K) + oq_bytes(K); }
inline size_t tg_smem(int fmt, int K) { return cta_smem_bytes(tg_ring_slots(fmt) * tg_slot_bytes(fmt), tg_tab_bytes(fmt, K)); }

inline int tg_pieces(int fmt, int64_t N, int64_t K) {
    const int64_t tasks = N / stage_rows(fmt), S = K / stage_k(fmt);
    const int64_t p = (kTgUnits + tasks - 1) / tasks;
    return (int)(p > S ? S : p);
}

struct TgArgs {
    const uint8_t* W;  // box-tiled [N][K]
    int N, K, P;
    const void* x;     // [q][K], bfloat16 or binary32
    int x_bf16;
    float* out;        // P == 1: y [q][N]; P > 1: partial rows [P][q][N]
    int32_t* status;
    uint32_t magic;    // kMagic, kept out of immediates (see decode_fp2)
};

template <int FMT, int Q>
__global__ void __launch_bounds__(kLThreads, 1) k_gemv_tiled(const __grid_constant__ TgArgs A) {
    constexpr int NS = tg_ring_slots(FMT), SB = tg_slot_bytes(FMT);
    using Ring = CtaRing<NS, SB>;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int shift[4];
    const int K = A.K, N = A.N, P = A.P, S = K / stage_k(FMT);
    const CtaSmem Sm = cta_carve(smem, Ring::kBytes);
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const Ring R = cta_init<NS, SB>(Sm);
    const uint32_t U = (uint32_t)(N / stage_rows(FMT)) * (uint32_t)P, G = gridDim.x;
    const uint32_t u0 = (uint32_t)((uint64_t)U * blockIdx.x / G), u1 = (uint32_t)((uint64_t)U * (blockIdx.x + 1) / G);
    const int64_t task_bytes = (int64_t)S * stage_bytes(FMT);

    if (warp == kLWarps) {  // producer: streams the range's boxes while the consumers build the tables
        if (lane == 0) {
            uint32_t issued = 0;
            bool live = true;
            const uint64_t pol = l2_evict_first();
            for (uint32_t u = u0; u < u1 && live; u++) {
                const uint32_t tk = u / (uint32_t)P;
                const int pc = (int)(u - tk * (uint32_t)P);
                const uint8_t* base = A.W + (int64_t)tk * task_bytes;
                for (int s = pc * S / P; s < (pc + 1) * S / P; s++, issued++) {
                    if (!R.acquire(issued)) { flag(A.status, FPX_ETIMEOUT); live = false; break; }
                    mbar_expect_tx(R.bar(issued), stage_bytes(FMT));
                    bulk_load_hint(R.slot(issued), base + (int64_t)s * stage_bytes(FMT), stage_bytes(FMT), R.bar(issued), pol);
                }
            }
            R.drain(issued);
        }
        return;
    }

    // activation tables (column shifts per token) from x, by the consumer warps
    uint2* tab = reinterpret_cast<uint2*>(Sm.tabs);
    float* oq = reinterpret_cast<float*>(Sm.tabs + btab_bytes(K));
    if (A.x_bf16)
        build_tables<FMT, false, true, true>(SrcBF16{reinterpret_cast<const uint16_t*>(A.x)}, K, Q, tab, nullptr, nullptr, oq, shift, Sm.red);
    else
        build_tables<FMT, false, true, true>(SrcF32{reinterpret_cast<const float*>(A.x)}, K, Q, tab, nullptr, nullptr, oq, shift, Sm.red);
    layer_sync();

    // Every consumer warp runs the same sequence of consumer barriers whether or not a wait timed
    // out, so a timeout never leaves a barrier short of arrivals.
    const int a_idx = b_active_index(lane);
    const uint32_t magic = A.magic;
    const LaneOfs L4 = lane_ofs<4>(t);
    const uint32_t tab_lane = lane_tab(tab, Sm.zero, a_idx, 0), tab_step = a_idx >= 0 ? 4u * 512u : 0u;
    const uint32_t oq_lane = lane_oq(oq, 0, t);
    uint32_t bad = 0;
    bool ok = true;
    typename Ring::Pos pos{0u, 0u};
    constexpr int kFp4Ch = 8 / kFp4Parts;  // FP4 chunks per warp
    for (uint32_t u = u0; u < u1; u++) {
        const uint32_t tk = u / (uint32_t)P;
        const int pc = (int)(u - tk * (uint32_t)P), s0 = pc * S / P, s1 = (pc + 1) * S / P;
        float y[kLTiles][4];
#pragma unroll
        for (int i = 0; i < kLTiles; i++) y[i][0] = y[i][1] = y[i][2] = y[i][3] = 0.f;
        if constexpr (FMT != 4) {
            frag_stages<FMT, kLTiles>(R, pos, s1 - s0, warp * 16 * kLTiles + g, t, tab_lane + (uint32_t)s0 * tab_step, tab_step,
                                      oq_lane + (uint32_t)s0 * 256u, magic, y, ok);
        } else {
            for (int s = s0; s < s1; s++) {  // warps (w % 4) own a 16-row tile, (w / 4) half of the chunks
                if (ok) ok = R.wait_at(pos);
                if (ok) {
                    const int ch0 = s * box_chunks(4) + kFp4Ch * (warp >> 2);
                    box_tiles<4, 1, kFp4Ch>(R.slot_at(pos) + ((warp & 3) * 16 + g) * box_bytes(4) + kFp4Ch * (warp >> 2) * chunk_bytes(4),
                                            L4, lane_tab(tab, Sm.zero, a_idx, ch0), 0u, 0u, magic,
                                            *reinterpret_cast<float(*)[1][4]>(&y[0]), bad);
                    R.release_at(pos);
                }
                R.next(pos);
            }
        }
#pragma unroll
        for (int i = 0; i < kLTiles; i++) pair_reduce(y[i]);
        if (FMT == 4) fp4_reduce(Sm.red, y[0]);
        if (ok && t < 2 && (FMT != 4 || warp < 4)) {
            const int rb = (int)tk * stage_rows(FMT) + (FMT == 4 ? 16 : 16 * kLTiles) * warp + g;
            float* o = A.out + (size_t)pc * Q * N;
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const int tok = 2 * t + (i & 1), rr = rb + 8 * (i >> 1);
                if (tok < Q) {
                    // undo the per-token activation scale (and the 2^-14 of the FP4 decode)
                    const float sc = exp2i((FMT == 4 ? 14 : 0) - shift[tok]);
                    o[(size_t)tok * N + rr] = y[0][i] * sc;
#pragma unroll
                    for (int ti = 1; ti < kLTiles; ti++)
                        if (FMT != 4) o[(size_t)tok * N + rr + 16 * ti] = y[ti][i] * sc;
                }
            }
        }
    }
    if (!ok && lane == 0) flag(A.status, FPX_ETIMEOUT);
    report_bad(bad, A.status);
}

// y[i] = the sum of the P partial rows i, in piece order.
__global__ void __launch_bounds__(256) k_tg_sum(const float* __restrict__ part, int P, int64_t n, float* __restrict__ y) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    float v = part[i];
    for (int p = 1; p < P; p++) v += part[(size_t)p * n + i];
    y[i] = v;
}

template <int FMT>
int launch_tiled(const uint8_t* W, int64_t N, int64_t K, const void* x, int x_bf16, int q, float* y, void* ws,
                 int32_t* st, cudaStream_t s) {
    const DeviceInfo di = device_info();
    const size_t smem = tg_smem(FMT, (int)K);
    if (smem > (size_t)di.smem_optin) return FPX_EINVAL;
    TgArgs A{};
    A.W = W;
    A.N = (int)N;
    A.K = (int)K;
    A.P = tg_pieces(FMT, N, K);
    A.x = x;
    A.x_bf16 = x_bf16;
    A.out = A.P > 1 ? static_cast<float*>(ws) : y;
    A.status = st;
    A.magic = kMagic;
    const int64_t units = N / stage_rows(FMT) * A.P;
    const int grid = (int)(units < di.sms ? units : di.sms);
    void (*kern)(TgArgs) = q == 1 ? k_gemv_tiled<FMT, 1> : q == 2 ? k_gemv_tiled<FMT, 2> : q == 3 ? k_gemv_tiled<FMT, 3>
                                                                                                  : k_gemv_tiled<FMT, 4>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) return FPX_ECUDA;
    kern<<<grid, kLThreads, smem, s>>>(A);
    if (A.P > 1) {
        const int64_t n = (int64_t)q * N;
        k_tg_sum<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(static_cast<const float*>(ws), A.P, n, y);
    }
    return launch_status();
}

}  // namespace

extern "C" {

size_t fpx_gemv_tiled_workspace_bytes(int fmt, int64_t N, int64_t K, int q) {
    if ((fmt != 2 && fmt != 3 && fmt != 4) || q < 1 || q > 4 || N < 1 || K < 1 || N % stage_rows(fmt) || K % stage_k(fmt))
        return 0;
    const int P = tg_pieces(fmt, N, K);
    return P > 1 ? (size_t)P * q * N * sizeof(float) : 16;
}

int fpx_gemv_q_tiled(int fmt, const uint8_t* Wt, int64_t N, int64_t K, const void* x, int x_dtype, int q, float* y,
                     void* ws, size_t ws_bytes, int32_t* dev_status, void* stream) {
    if ((fmt != 2 && fmt != 3 && fmt != 4) || q < 1 || q > 4 || (x_dtype != FPX_DTYPE_F32 && x_dtype != FPX_DTYPE_BF16))
        return FPX_EINVAL;
    if (N < 1 || K < 1 || N % stage_rows(fmt) || K % stage_k(fmt) || N > INT32_MAX / 4 || K > 65536) return FPX_EINVAL;
    if (!Wt || !x || !y || !ws) return FPX_EINVAL;
    if (!aligned(Wt, 16) || !aligned(x, 16) || !aligned(y, 4) || !aligned(ws, 16) || (dev_status && !aligned(dev_status, 4)))
        return FPX_EALIGN;
    if (ws_bytes < fpx_gemv_tiled_workspace_bytes(fmt, N, K, q)) return FPX_ESPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int bf = x_dtype == FPX_DTYPE_BF16;
    if (fmt == 2) return launch_tiled<2>(Wt, N, K, x, bf, q, y, ws, dev_status, s);
    if (fmt == 3) return launch_tiled<3>(Wt, N, K, x, bf, q, y, ws, dev_status, s);
    return launch_tiled<4>(Wt, N, K, x, bf, q, y, ws, dev_status, s);
}

}  // extern "C"
