// The MoE decode/verify step: router + top-k + union, gate/up + SiLU, down + weighted combine, and
// the stack driver. Follows "DeepSeek V4 Flash hits 32 tok/s on AMD Ryzen AI MAX+ 395", paragraph 3
// (q = 4 verification columns, each packed weight decoded once and applied to all of them, routing
// through TOP_K/ARGSORT kernels, 43 memory-bound layers) and "Token Freedom via APU ...", section
// "Lucebox's Optimization Trio" (256 routed experts plus one shared expert).
//
// Readings (the pages leave these open): sigmoid scores, top-k on the logit with ties to the lower
// expert index, weights normalised over the selected k; h = silu(g) * u kept in binary32; a token's
// output sums its selected experts in ascending expert order (starting from the first product, so no
// zero-weight term is ever added) and then the shared expert; the stack's layer input is the
// bfloat16 RMS normalisation (eps 1e-6, no gain) of a binary32 residual.
//
// Per layer three kernels: k_router (normalise + router GEMV), k_gate_up (top-k + union recomputed
// per CTA, then gate/up on the tensor cores), k_down (h = silu(g) u, down projection on the tensor
// cores; the last task to finish a 128-row output group combines it).
#include "fpx_mma.cuh"

using namespace fpx;

namespace {

constexpr int kThreads = 256;  // router and top-k kernels
constexpr int kMaxK = 8;
constexpr int kMaxQ = 4;
constexpr int kMaxE = 1024;

// ------------------------------------------------------------------ workspace

struct Ws {
    size_t status, logits, u, idx, w, uni, nuni, gu, yi, cnt, total;
};

inline size_t up16(size_t v) { return (v + 15) & ~size_t(15); }

inline Ws ws_layout(int H, int I, int E, int q, int k) {
    Ws w{};
    size_t o = 0;
    w.status = o; o += 16;
    w.logits = o; o = up16(o + sizeof(float) * q * E);
    w.u = o; o = up16(o + sizeof(uint16_t) * q * H);
    w.idx = o; o = up16(o + sizeof(int32_t) * q * k);
    w.w = o; o = up16(o + sizeof(float) * q * k);
    w.uni = o; o = up16(o + sizeof(int32_t) * q * k);
    w.nuni = o; o += 16;
    w.gu = o; o = up16(o + sizeof(float) * (size_t)2 * (q * k + 1) * q * I);
    w.yi = o; o = up16(o + sizeof(float) * (size_t)(q * k + 1) * q * H);
    w.cnt = o; o = up16(o + sizeof(int32_t) * (size_t)(H / 128));
    w.total = o;
    return w;
}

struct WsPtrs {
    int32_t* status;
    float* logits;
    uint16_t* u;
    int32_t* idx;
    float* w;
    int32_t* uni;
    int32_t* nuni;
    float* gu;  // g and u of every item: [2 * item + (0 | 1)][q][I]
    float* yi;  // per-item outputs [item][q][H]
    int32_t* cnt;
};

inline WsPtrs ws_ptrs(void* ws, const Ws& l) {
    char* b = static_cast<char*>(ws);
    return WsPtrs{reinterpret_cast<int32_t*>(b + l.status), reinterpret_cast<float*>(b + l.logits),
                  reinterpret_cast<uint16_t*>(b + l.u),     reinterpret_cast<int32_t*>(b + l.idx),
                  reinterpret_cast<float*>(b + l.w),        reinterpret_cast<int32_t*>(b + l.uni),
                  reinterpret_cast<int32_t*>(b + l.nuni),   reinterpret_cast<float*>(b + l.gu),
                  reinterpret_cast<float*>(b + l.yi),       reinterpret_cast<int32_t*>(b + l.cnt)};
}

// Everything the gate/up and down kernels need about one layer: tensor maps over the stacked
// matrices (rows of all experts), shapes and strides.
struct LayerMaps {
    CUtensorMap gate, up, down, sh_gate, sh_up, sh_down;  // 64-byte aligned members first
    int H, I, E;
};

int make_layer_maps(const moe_layer& L, LayerMaps* m) {
    m->H = L.H; m->I = L.I; m->E = L.E;
    const int64_t rb2 = (int64_t)(L.H / 32) * 10, rb4h = (int64_t)(L.H / 32) * 17;
    const int64_t rb3 = (int64_t)(L.I / 32) * 14, rb4i = (int64_t)(L.I / 32) * 17;
    int st = make_row_map(&m->gate, L.gate, rb2, (int64_t)L.E * L.I, rb2, box_bytes(2), stage_rows(2), 1);
    st = st ? st : make_row_map(&m->up, L.up, rb2, (int64_t)L.E * L.I, rb2, box_bytes(2), stage_rows(2), 1);
    st = st ? st : make_row_map(&m->down, L.down, rb3, (int64_t)L.E * L.H, rb3, box_bytes(3), stage_rows(3), 1);
    st = st ? st : make_row_map(&m->sh_gate, L.sh_gate, rb4h, L.I, rb4h, box_bytes(4), stage_rows(4), 2);
    st = st ? st : make_row_map(&m->sh_up, L.sh_up, rb4h, L.I, rb4h, box_bytes(4), stage_rows(4), 2);
    st = st ? st : make_row_map(&m->sh_down, L.sh_down, rb4i, L.H, rb4i, box_bytes(4), stage_rows(4), 2);
    return st;
}

// ------------------------------------------------------------------ block-wide helpers

// Deterministic block sum (fixed order: per-thread strided partial, warp butterfly, warps in order).
__device__ float block_sum(float v, float* red) {
    v = warp_sum(v);
    const int w = threadIdx.x / 32, nw = blockDim.x / 32;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[w] = v;
    __syncthreads();
    float s = 0.0f;
    for (int i = 0; i < nw; i++) s += red[i];
    return s;
}

__device__ float block_max(float v, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int w = threadIdx.x / 32, nw = blockDim.x / 32;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[w] = v;
    __syncthreads();
    float s = 0.0f;
    for (int i = 0; i < nw; i++) s = fmaxf(s, red[i]);
    return s;
}

// ------------------------------------------------------------------ K1: router logits

// Computes the layer input u (binary32 values of bfloat16) and logits[t][e] for this CTA's experts.
// MODE 0: input x is bfloat16. MODE 1: input is the residual r; u = RN_bf16(r / rms(r)), and CTA 0
// publishes u (for the gate/up kernel) and r (the trace). Each CTA handles 2 experts with 4 warps per
// expert, each warp a quarter of H; the quarter sums are added in order.
template <int MODE>
__global__ void __launch_bounds__(kThreads) k_router(const float* __restrict__ R, int E, int H, int q,
                                                     const uint16_t* __restrict__ xin, const float* __restrict__ rin,
                                                     float* __restrict__ logits, uint16_t* __restrict__ u_out,
                                                     float* __restrict__ r_trace, int32_t* status_to_clear) {
    extern __shared__ __align__(16) float sm[];
    float* u_s = sm;                      // [q][H]
    float* part = sm + (size_t)q * H;     // [8 warps][kMaxQ]
    float* red = part + 8 * kMaxQ;        // [8]
    if (status_to_clear && blockIdx.x == 0 && threadIdx.x == 0) *status_to_clear = 0;
    if (MODE == 0) {
        for (int i = threadIdx.x; i < q * H; i += blockDim.x) u_s[i] = bf16_bits_to_float(xin[i]);
    } else {
        // each thread loads its float4s of r for all tokens at once (H % 4 == 0), then reduces
        constexpr int V = 16;
        const int n4 = q * H / 4;
        const float4* r4 = reinterpret_cast<const float4*>(rin);
        float ss[kMaxQ] = {0.f, 0.f, 0.f, 0.f};
        for (int base = threadIdx.x; base < n4; base += V * blockDim.x) {
            float4 rv[V];
#pragma unroll
            for (int i = 0; i < V; i++) {
                const int idx = base + i * blockDim.x;
                rv[i] = idx < n4 ? r4[idx] : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int i = 0; i < V; i++) {
                const int idx = base + i * blockDim.x;
                if (idx < n4) {
                    const int t = idx * 4 / H;
                    float a = 0.f;
                    a = fmaf(rv[i].x, rv[i].x, a); a = fmaf(rv[i].y, rv[i].y, a);
                    a = fmaf(rv[i].z, rv[i].z, a); a = fmaf(rv[i].w, rv[i].w, a);
#pragma unroll
                    for (int tt = 0; tt < kMaxQ; tt++) ss[tt] += tt == t ? a : 0.f;
                }
            }
        }
        float inv[kMaxQ];
        for (int t = 0; t < kMaxQ; t++) inv[t] = 1.0f / sqrtf(block_sum(ss[t], red) / (float)H + 1e-6f);
        for (int base = threadIdx.x; base < n4; base += V * blockDim.x) {
            float4 rv[V];
#pragma unroll
            for (int i = 0; i < V; i++) {
                const int idx = base + i * blockDim.x;
                rv[i] = idx < n4 ? r4[idx] : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int i = 0; i < V; i++) {
                const int idx = base + i * blockDim.x;
                if (idx < n4) {
                    const int t = idx * 4 / H;
                    const float iv = inv[0] * (t == 0) + inv[1] * (t == 1) + inv[2] * (t == 2) + inv[3] * (t == 3);
                    const float vv[4] = {rv[i].x, rv[i].y, rv[i].z, rv[i].w};
                    uint16_t ub[4];
#pragma unroll
                    for (int j = 0; j < 4; j++) {
                        const __nv_bfloat16 b = __float2bfloat16_rn(vv[j] * iv);
                        u_s[(size_t)idx * 4 + j] = __bfloat162float(b);
                        ub[j] = __bfloat16_as_ushort(b);
                    }
                    if (blockIdx.x == 0) {
                        reinterpret_cast<uint2*>(u_out)[idx] = make_uint2(ub[0] | (uint32_t(ub[1]) << 16), ub[2] | (uint32_t(ub[3]) << 16));
                        if (r_trace) reinterpret_cast<float4*>(r_trace)[idx] = rv[i];
                    }
                }
            }
        }
    }
    __syncthreads();
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    const int e = blockIdx.x * 2 + warp / 4, slice = warp % 4;
    const int h0 = H * slice / 4, h1 = H * (slice + 1) / 4;  // H % 16 == 0: quarters are float4-aligned
    float acc[kMaxQ] = {0.f, 0.f, 0.f, 0.f};
    if (e < E) {
        const float4* row = reinterpret_cast<const float4*>(R + (size_t)e * H);
        // batches of 8 independent loads per lane, then the FMAs (same order as a plain loop)
        for (int base = h0 / 4 + lane; base < h1 / 4; base += 8 * 32) {
            float4 rv[8];
#pragma unroll
            for (int b = 0; b < 8; b++) rv[b] = base + 32 * b < h1 / 4 ? __ldg(row + base + 32 * b) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int b = 0; b < 8; b++) {
                const int h4 = base + 32 * b;
                if (h4 >= h1 / 4) break;
#pragma unroll
                for (int t = 0; t < kMaxQ; t++) {
                    if (t < q) {
                        const float4 uv = *reinterpret_cast<const float4*>(u_s + (size_t)t * H + 4 * h4);
                        acc[t] = fmaf(rv[b].x, uv.x, acc[t]);
                        acc[t] = fmaf(rv[b].y, uv.y, acc[t]);
                        acc[t] = fmaf(rv[b].z, uv.z, acc[t]);
                        acc[t] = fmaf(rv[b].w, uv.w, acc[t]);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int t = 0; t < kMaxQ; t++) acc[t] = warp_sum(acc[t]);
    if (lane == 0)
        for (int t = 0; t < q; t++) part[warp * kMaxQ + t] = acc[t];
    __syncthreads();
    if (threadIdx.x < 2 * q) {
        int el = threadIdx.x / q, t = threadIdx.x % q;
        int ee = blockIdx.x * 2 + el;
        if (ee < E) {
            float s = part[(el * 4) * kMaxQ + t];
            for (int sl = 1; sl < 4; sl++) s += part[(el * 4 + sl) * kMaxQ + t];
            logits[(size_t)t * E + ee] = s;
        }
    }
}

// ------------------------------------------------------------------ top-k + union

// Warp-level top-k of lg[0..E) (descending, ties to the lower index), with sigmoid weights
// normalised over the selected k. Each lane keeps its E / 32 logits in registers (NM >= E / 32 slots).
template <int NM>
__device__ void warp_topk_n(const float* lg, int E, int k, int32_t* idx, float* w) {
    const int lane = threadIdx.x & 31;
    float v[NM];
#pragma unroll
    for (int m = 0; m < NM; m++) v[m] = lane + 32 * m < E ? lg[lane + 32 * m] : 0.0f;
    uint32_t taken = 0;  // bit m: element lane + 32 m already selected
    float sig[kMaxK];
    for (int r = 0; r < k; r++) {
        float bv = 0.0f;
        int bi = -1;
#pragma unroll
        for (int m = 0; m < NM; m++) {
            const int e = lane + 32 * m;  // ascending: equal values keep the lower index
            if (e < E && !((taken >> m) & 1u) && (bi < 0 || v[m] > bv)) { bv = v[m]; bi = e; }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            bool better = oi >= 0 && (bi < 0 || ov > bv || (ov == bv && oi < bi));
            if (better) { bv = ov; bi = oi; }
        }
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        idx[r] = bi;
        sig[r] = 1.0f / (1.0f + expf(-bv));
    }
    float S = sig[0];
    for (int r = 1; r < k; r++) S += sig[r];
    for (int r = 0; r < k; r++) w[r] = sig[r] / S;
}

__device__ void warp_topk(const float* lg, int E, int k, int32_t* idx, float* w) {
    if (E <= 256) warp_topk_n<8>(lg, E, k, idx, w);
    else warp_topk_n<kMaxE / 32>(lg, E, k, idx, w);
}

// Shared-memory routing state.
struct Route {
    int32_t idx[kMaxQ * kMaxK];
    float w[kMaxQ * kMaxK];
    int32_t uni[kMaxQ * kMaxK];
    uint32_t mask[kMaxE / 32];
    int32_t n_uni;
};

// Sorted union of r.idx over q tokens. Whole CTA; warp 0 works: lane w owns mask word w (experts
// 32w .. 32w + 31), and a warp prefix sum of the popcounts places every lane's experts in order.
__device__ void build_union(Route& r, int q, int k, int E) {
    __syncthreads();
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        uint32_t mask = 0u;
        for (int i = 0; i < q * k; i++) {
            const int e = r.idx[i];
            if ((e >> 5) == lane) mask |= 1u << (e & 31);
        }
        int incl = __popc(mask);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int o = incl - __popc(mask);
        while (mask) {
            const int b = __ffs(mask) - 1;
            mask &= mask - 1;
            r.uni[o++] = lane * 32 + b;
        }
        if (lane == 31) r.n_uni = incl;
    }
    __syncthreads();
}

__global__ void k_topk(const float* __restrict__ logits, int E, int q, int k, int32_t* idx, float* w, int32_t* uni,
                       int32_t* n_uni) {
    __shared__ Route r;
    const int warp = threadIdx.x / 32;
    if (warp < q) warp_topk(logits + (size_t)warp * E, E, k, r.idx + warp * k, r.w + warp * k);
    __syncthreads();
    build_union(r, q, k, E);
    for (int i = threadIdx.x; i < q * k; i += blockDim.x) {
        idx[i] = r.idx[i];
        w[i] = r.w[i];
        uni[i] = i < r.n_uni ? r.uni[i] : -1;
    }
    if (threadIdx.x == 0) *n_uni = r.n_uni;
}

// ------------------------------------------------------------------ K2: gate/up

// Task = (output matrix, row block): the union's gate and up matrices (FP2, 256-row blocks of I,
// H/256 stages each), then the shared expert's gate and up (FP4, 128-row blocks, 2 * H/512 stages:
// the two 64-row halves alternate).
// Matrix m = 2 * item + (0 gate | 1 up), the shared expert being item n_uni. Each CTA owns a
// contiguous task range; its producer thread streams the range's boxes through the CTA ring and all
// eight consumer warps decode every box. Outputs g and u (binary32) go to ws.gu[m][token][row]; the
// down kernel forms h = silu(g) u while building its activation table.
struct GateUpArgs {
    LayerMaps m;
    int q, k;
    const uint16_t* x;  // layer input, bfloat16 [q][H]
    WsPtrs ws;
    int32_t* idx_out;
    float* w_out;
    float* logits_out;
    uint32_t magic;  // kMagic, kept out of immediates (see decode_fp2)
};

// Ring geometry of the two layer kernels: 7 slots of one FP2 box, 5 slots of one FP3 box.
using GuRing = CtaRing<7, stage_bytes(2)>;
using DnRing = CtaRing<5, stage_bytes(3)>;

struct GuTask {
    int mat;    // output matrix index
    int fp4;    // shared expert (FP4) task
    int row0;   // first output row
    int grow0;  // first row in the stacked tensor map
};

__device__ __forceinline__ int gu_tasks(int n_uni, int I) { return 2 * n_uni * (I / 256) + 2 * (I / 128); }

__device__ __forceinline__ GuTask gu_task(int t, const Route& r, int I) {
    const int rb2 = I / 256, n2 = 2 * r.n_uni * rb2;
    GuTask k;
    if (t < n2) {
        k.mat = t / rb2;
        k.fp4 = 0;
        k.row0 = (t % rb2) * 256;
        k.grow0 = r.uni[k.mat >> 1] * I + k.row0;
    } else {
        const int t4 = t - n2, rb4 = I / 128;
        k.mat = 2 * r.n_uni + t4 / rb4;
        k.fp4 = 1;
        k.row0 = (t4 % rb4) * 128;
        k.grow0 = k.row0;
    }
    return k;
}

__device__ __forceinline__ void gu_issue(const GateUpArgs& A, const GuTask& k, int s, uint8_t* slot, uint64_t* bar) {
    if (!k.fp4) {
        mbar_expect_tx(bar, stage_bytes(2));
        tma_load_2d(slot, (k.mat & 1) ? &A.m.up : &A.m.gate, s * box_bytes(2), k.grow0, bar);
    } else {
        mbar_expect_tx(bar, stage_bytes(4));
        tma_load_2d(slot, (k.mat & 1) ? &A.m.sh_up : &A.m.sh_gate, (s >> 1) * (box_bytes(4) / 2), k.grow0 + 64 * (s & 1), bar);
    }
}

// Producer-side walk over a CTA's (task, stage) sequence.
struct StageCursor {
    int task, stage;
    uint32_t issued;
};

// Stages of a task: FP2/FP3 tasks stream one box per stage_k columns, FP4 tasks two (row halves).
__device__ __forceinline__ int task_stages(int fp4, int fmt_other, int K) {
    return fp4 ? 2 * (K / stage_k(4)) : K / stage_k(fmt_other);
}

template <int Q>
__global__ void __launch_bounds__(kCtaThreads, 1) k_gate_up(const __grid_constant__ GateUpArgs A) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ Route r;
    __shared__ int shift[kMaxQ];
    __shared__ float red4[(kWarps + 1) * 4];
    const int H = A.m.H, I = A.m.I;
    const CtaSmem S = cta_carve(smem, btab_bytes(H));
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const GuRing R = cta_init<7, stage_bytes(2)>(S);

    // routing (every CTA), published by CTA 0
    if (warp < Q) warp_topk(A.ws.logits + (size_t)warp * A.m.E, A.m.E, A.k, r.idx + warp * A.k, r.w + warp * A.k);
    build_union(r, Q, A.k, A.m.E);
    if (blockIdx.x == 0) {
        for (int i = threadIdx.x; i < Q * A.k; i += blockDim.x) {
            A.ws.idx[i] = r.idx[i];
            A.ws.w[i] = r.w[i];
            A.ws.uni[i] = i < r.n_uni ? r.uni[i] : -1;
            if (A.idx_out) A.idx_out[i] = r.idx[i];
            if (A.w_out) A.w_out[i] = r.w[i];
        }
        if (A.logits_out)
            for (int i = threadIdx.x; i < Q * A.m.E; i += blockDim.x) A.logits_out[i] = A.ws.logits[i];
        if (threadIdx.x == 0) *A.ws.nuni = r.n_uni;
    }

    const int total = gu_tasks(r.n_uni, I);
    const int c0 = (int)((int64_t)total * blockIdx.x / gridDim.x), c1 = (int)((int64_t)total * (blockIdx.x + 1) / gridDim.x);
    const bool producer = threadIdx.x == kWarps * 32;
    StageCursor pc{c0, 0, 0u};
    auto issue_next = [&]() {
        const GuTask k = gu_task(pc.task, r, I);
        gu_issue(A, k, pc.stage, R.slot(pc.issued), R.full + pc.issued % 7);
        pc.issued++;
        if (++pc.stage == task_stages(k.fp4, 2, H)) { pc.stage = 0; pc.task++; }
    };
    // fill the ring before building the activation tables, so the first loads overlap it
    if (producer)
        while (pc.task < c1 && pc.issued < 7u) issue_next();

    // activation tables: x scaled per token, FP2 (pair-shifted, with block offsets) and FP4
    build_tables<2, 4>(SrcBF16{A.x}, H, Q, S.tab[0], S.tab[1], S.csum, shift, red4);
    __syncthreads();

    if (warp == kWarps) {
        if (producer) {
            while (pc.task < c1) {
                if (!R.acquire(pc.issued)) { flag(A.ws.status, FPX_ETIMEOUT); break; }
                issue_next();
            }
            R.drain(pc.issued);
        }
        return;
    }

    const int a_idx = b_active_index(lane);
    const uint32_t magic = A.magic;
    uint32_t n = 0, bad = 0;
    bool ok = true;
    for (int tk = c0; tk < c1; tk++) {
        const GuTask k = gu_task(tk, r, I);
        float y[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        const int ns = task_stages(k.fp4, 2, H);
        for (int s = 0; s < ns; s++, n++) {
            if (ok) ok = R.wait(n, A.ws.status);
            if (!ok) continue;  // the producer gives up too once this warp stops releasing
            const uint8_t* slot = R.slot(n);
            if (!k.fp4) {
                const int ch0 = s * box_chunks(2);
                box_tiles<2, 2, box_chunks(2)>(slot + (warp * 32 + g) * box_bytes(2), lane_tab(S.tab[0], S.zero, a_idx, ch0),
                                               lane_csum(S.csum, ch0, t), t, magic, y, bad);
            } else if ((s & 1) == (warp >> 2)) {
                const int ch0 = (s >> 1) * box_chunks(4);
                box_tiles<4, 1, box_chunks(4)>(slot + ((warp & 3) * 16 + g) * box_bytes(4),
                                               lane_tab(S.tab[1], S.zero, a_idx, ch0), nullptr, t, magic,
                                               *reinterpret_cast<float(*)[1][4]>(&y[0]), bad);
            }
            R.release(n);
        }
        if (!ok) continue;
        pair_reduce(y[0]);
        pair_reduce(y[1]);
        if (t < 2) {
            const int rb = k.row0 + (k.fp4 ? 64 * (warp >> 2) + 16 * (warp & 3) : 32 * warp) + g;
            float* out = A.ws.gu + (size_t)k.mat * Q * I;
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const int tok = 2 * t + (i & 1), rr = rb + 8 * (i >> 1);
                if (tok < Q) {
                    // undo the per-token activation scale (and the 2^-14 of the FP4 decode)
                    const float sc = exp2i((k.fp4 ? 14 : 0) - shift[tok]);
                    out[(size_t)tok * I + rr] = y[0][i] * sc;
                    if (!k.fp4) out[(size_t)tok * I + rr + 16] = y[1][i] * sc;
                }
            }
        }
    }
    report_bad(bad, A.ws.status);
}

// ------------------------------------------------------------------ K3: down + combine

// Task = (item, row block of H): the union's down matrices (FP3, 256-row blocks, I/256 stages each),
// then the shared expert's (FP4, 128-row blocks, 2 * I/512 stages: the two 64-row halves alternate). Each CTA owns a contiguous task range,
// which spans at most two items (the grid has at least kMinDownCtas CTAs); it builds their
// activation tables from h = silu(g) u at start. Every 128-row group of the output has a counter;
// after a task's rows are in ws.yi, the task adds one to each group it covers, and the CTA that
// brings a group's count to n_uni + 1 combines the group for every token: selected experts in
// ascending expert order, then the shared expert.
constexpr int kMinDownCtas = 2 * (kMaxQ * kMaxK + 1);

struct DownArgs {
    LayerMaps m;
    int q, k;
    WsPtrs ws;
    float* out;  // MODE 0: y [q][H]; MODE 1: residual r [q][H], updated in place
    uint32_t magic;
};

struct DnTask {
    int item, fp4, row0, grow0;
};

__device__ __forceinline__ int dn_tasks(int n_uni, int H) { return n_uni * (H / 256) + H / 128; }

__device__ __forceinline__ DnTask dn_task(int t, const Route& r, int H) {
    const int rb3 = H / 256, n3 = r.n_uni * rb3;
    DnTask k;
    if (t < n3) {
        k.item = t / rb3;
        k.fp4 = 0;
        k.row0 = (t % rb3) * 256;
        k.grow0 = r.uni[k.item] * H + k.row0;
    } else {
        k.item = r.n_uni;
        k.fp4 = 1;
        k.row0 = (t - n3) * 128;
        k.grow0 = k.row0;
    }
    return k;
}

__device__ __forceinline__ void dn_issue(const DownArgs& A, const DnTask& k, int s, uint8_t* slot, uint64_t* bar) {
    if (!k.fp4) {
        mbar_expect_tx(bar, stage_bytes(3));
        tma_load_2d(slot, &A.m.down, s * box_bytes(3), k.grow0, bar);
    } else {
        mbar_expect_tx(bar, stage_bytes(4));
        tma_load_2d(slot, &A.m.sh_down, (s >> 1) * (box_bytes(4) / 2), k.grow0 + 64 * (s & 1), bar);
    }
}

template <int Q, int MODE>
__global__ void __launch_bounds__(kCtaThreads, 1) k_down(const __grid_constant__ DownArgs A) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ Route r;
    __shared__ float wsel[kMaxQ * kMaxK + 1][kMaxQ];  // weight of token t for union item j, NaN if unselected
    __shared__ int shift[2][kMaxQ];
    __shared__ float red4[(kWarps + 1) * 4];
    __shared__ int last_grp[2];
    const int H = A.m.H, I = A.m.I;
    const CtaSmem S = cta_carve(smem, btab_bytes(I));
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const DnRing R = cta_init<5, stage_bytes(3)>(S);

    if (threadIdx.x == 0) r.n_uni = *A.ws.nuni;
    for (int i = threadIdx.x; i < Q * A.k; i += blockDim.x) { r.idx[i] = A.ws.idx[i]; r.w[i] = A.ws.w[i]; r.uni[i] = A.ws.uni[i]; }
    __syncthreads();
    for (int i = threadIdx.x; i < r.n_uni * Q; i += blockDim.x) {
        const int j = i / Q, tok = i % Q;
        float wv = __int_as_float(0x7fc00000);
        for (int rr = 0; rr < A.k; rr++)
            if (r.idx[tok * A.k + rr] == r.uni[j]) wv = r.w[tok * A.k + rr];
        wsel[j][tok] = wv;
    }

    const int total = dn_tasks(r.n_uni, H);
    const int c0 = (int)((int64_t)total * blockIdx.x / gridDim.x), c1 = (int)((int64_t)total * (blockIdx.x + 1) / gridDim.x);
    if (c0 >= c1) return;  // CTA-uniform: nothing to do
    const int item_lo = dn_task(c0, r, H).item, item_hi = dn_task(c1 - 1, r, H).item;
    if (item_hi - item_lo > 1) {  // too small a grid (the host launches at least kMinDownCtas CTAs)
        if (threadIdx.x == 0) flag(A.ws.status, FPX_EINVAL);
        return;
    }

    const bool producer = threadIdx.x == kWarps * 32;
    StageCursor pc{c0, 0, 0u};
    auto issue_next = [&]() {
        const DnTask k = dn_task(pc.task, r, H);
        dn_issue(A, k, pc.stage, R.slot(pc.issued), R.full + pc.issued % 5);
        pc.issued++;
        if (++pc.stage == task_stages(k.fp4, 3, I)) { pc.stage = 0; pc.task++; }
    };
    if (producer)
        while (pc.task < c1 && pc.issued < 5u) issue_next();

    // activation tables for the (at most two) items of this CTA's range: h = silu(g) u
    for (int sl = 0; sl <= item_hi - item_lo; sl++) {
        const int item = item_lo + sl;
        const SrcSilu src{A.ws.gu + (size_t)(2 * item) * Q * I, A.ws.gu + (size_t)(2 * item + 1) * Q * I};
        uint2* tab = sl ? S.tab[1] : S.tab[0];
        if (item == r.n_uni) build_tables<4, 0>(src, I, Q, tab, nullptr, nullptr, shift[sl], red4);
        else build_tables<3, 0>(src, I, Q, tab, nullptr, nullptr, shift[sl], red4);
        __syncthreads();
    }

    if (warp == kWarps) {
        if (producer) {
            while (pc.task < c1) {
                if (!R.acquire(pc.issued)) { flag(A.ws.status, FPX_ETIMEOUT); break; }
                issue_next();
            }
            R.drain(pc.issued);
        }
        return;
    }

    // Consumers. Every consumer warp runs the same sequence of consumers_sync() whether or not a wait
    // timed out, so a timeout never leaves a barrier short of arrivals.
    const int a_idx = b_active_index(lane);
    const uint32_t magic = A.magic;
    uint32_t n = 0, bad = 0;
    bool ok = true;
    for (int tk = c0; tk < c1; tk++) {
        const DnTask k = dn_task(tk, r, H);
        const int sl = k.item - item_lo;
        const uint2* tab = sl ? S.tab[1] : S.tab[0];
        float y[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        const int ns = task_stages(k.fp4, 3, I);
        for (int s = 0; s < ns; s++, n++) {
            if (ok) ok = R.wait(n, A.ws.status);
            if (!ok) continue;
            const uint8_t* slot = R.slot(n);
            if (!k.fp4) {
                const int ch0 = s * box_chunks(3);
                box_tiles<3, 2, box_chunks(3)>(slot + (warp * 32 + g) * box_bytes(3), lane_tab(tab, S.zero, a_idx, ch0), nullptr,
                                               t, magic, y, bad);
            } else if ((s & 1) == (warp >> 2)) {
                const int ch0 = (s >> 1) * box_chunks(4);
                box_tiles<4, 1, box_chunks(4)>(slot + ((warp & 3) * 16 + g) * box_bytes(4), lane_tab(tab, S.zero, a_idx, ch0),
                                               nullptr, t, magic, *reinterpret_cast<float(*)[1][4]>(&y[0]), bad);
            }
            R.release(n);
        }
        if (ok) {
            pair_reduce(y[0]);
            pair_reduce(y[1]);
            if (t < 2) {
                const int rb = k.row0 + (k.fp4 ? 64 * (warp >> 2) + 16 * (warp & 3) : 32 * warp) + g;
                float* out = A.ws.yi + (size_t)k.item * Q * H;
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    const int tok = 2 * t + (i & 1), rr = rb + 8 * (i >> 1);
                    if (tok < Q) {
                        const float sc = exp2i((k.fp4 ? 14 : 0) - shift[sl][tok]);
                        out[(size_t)tok * H + rr] = y[0][i] * sc;
                        if (!k.fp4) out[(size_t)tok * H + rr + 16] = y[1][i] * sc;
                    }
                }
            }
        }
        // count this task into its 128-row groups; the last contributor combines a group (one thread
        // publishes the CTA's writes: the barrier orders them before its fence and atomic)
        consumers_sync();
        if (threadIdx.x == 0) {
            __threadfence();
            const int g0 = k.row0 / 128, ng = k.fp4 ? 1 : 2;
            for (int j = 0; j < 2; j++) last_grp[j] = (j < ng && atomicAdd(A.ws.cnt + g0 + j, 1) == r.n_uni) ? g0 + j : -1;
            __threadfence();
        }
        consumers_sync();
        for (int j = 0; j < 2; j++) {
            const int gi = last_grp[j];
            if (gi < 0) continue;
            for (int o = threadIdx.x; o < 128 * Q; o += kWarps * 32) {
                const int rr = gi * 128 + o / Q, tok = o % Q;
                // loads in batches of 8 (independent, in flight together), then the fixed-order sum;
                // item n_uni is the shared expert, added last
                const float* col = A.ws.yi + (size_t)tok * H + rr;
                const size_t istride = (size_t)Q * H;
                float acc = 0.0f, ysh = 0.0f;
                bool first = true;
                for (int j0 = 0; j0 <= r.n_uni; j0 += 8) {
                    float yv[8];
#pragma unroll
                    for (int u = 0; u < 8; u++) yv[u] = j0 + u <= r.n_uni ? __ldcg(col + (size_t)(j0 + u) * istride) : 0.0f;
#pragma unroll
                    for (int u = 0; u < 8; u++) {
                        const int jj = j0 + u;
                        if (jj == r.n_uni) ysh = yv[u];
                        if (jj >= r.n_uni) continue;
                        const float wv = wsel[jj][tok];
                        if (wv != wv) continue;  // expert not selected by this token
                        acc = first ? wv * yv[u] : fmaf(wv, yv[u], acc);
                        first = false;
                    }
                }
                acc += ysh;
                const size_t oi = (size_t)tok * H + rr;
                if (MODE == 0) A.out[oi] = acc;
                else A.out[oi] = A.out[oi] + acc;
            }
            if (threadIdx.x == 0) A.ws.cnt[gi] = 0;  // ready for the next call
        }
        consumers_sync();  // last_grp is rewritten by the next task
    }
    report_bad(bad, A.ws.status);
}

// ------------------------------------------------------------------ launch plumbing

int check_layer(const moe_layer* L) {
    if (!L || L->H < 512 || L->I < 512 || L->H % 512 || L->I % 512 || L->E < 1 || L->E > kMaxE) return FPX_EINVAL;
    if (!L->router || !L->gate || !L->up || !L->down || !L->sh_gate || !L->sh_up || !L->sh_down) return FPX_EINVAL;
    if (!aligned(L->router, 16) || !aligned(L->gate, 16) || !aligned(L->up, 16) || !aligned(L->down, 16) ||
        !aligned(L->sh_gate, 16) || !aligned(L->sh_up, 16) || !aligned(L->sh_down, 16))
        return FPX_EALIGN;
    if (cta_smem_bytes(btab_bytes(L->H > L->I ? L->H : L->I)) + 2048 > 227 * 1024) return FPX_EINVAL;  // + static
    return FPX_OK;
}

struct Plan {
    int g_router, g_gate, g_down;
    size_t sm_router, sm_gate, sm_down;
};

Plan make_plan(const moe_layer& L, int q) {
    DeviceInfo di = device_info();
    Plan p{};
    p.g_router = (L.E + 1) / 2;
    p.sm_router = sizeof(float) * ((size_t)q * L.H + 8 * kMaxQ + 8);
    p.g_gate = di.sms;
    p.sm_gate = cta_smem_bytes(btab_bytes(L.H));
    p.g_down = di.sms > kMinDownCtas ? di.sms : kMinDownCtas;
    p.sm_down = cta_smem_bytes(btab_bytes(L.I));
    return p;
}

template <int Q, int MODE>
int launch_layer(const moe_layer& L, const Plan& p, int k, const uint16_t* x, const float* r, float* out,
                 int32_t* idx_out, float* w_out, float* logits_out, float* r_trace, WsPtrs ws, bool clear,
                 cudaEvent_t const* ev, cudaStream_t s) {
    GateUpArgs ga{};
    DownArgs da{};
    int st = make_layer_maps(L, &ga.m);
    if (st) return st;
    da.m = ga.m;
    ga.q = da.q = Q;
    ga.k = da.k = k;
    ga.x = MODE == 0 ? x : ws.u;
    ga.ws = da.ws = ws;
    ga.idx_out = idx_out;
    ga.w_out = w_out;
    ga.logits_out = logits_out;
    ga.magic = da.magic = kMagic;
    da.out = out;
    if (cudaFuncSetAttribute(k_router<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.sm_router) ||
        cudaFuncSetAttribute(k_gate_up<Q>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.sm_gate) ||
        cudaFuncSetAttribute(k_down<Q, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.sm_down))
        return FPX_ECUDA;
    if (ev) cudaEventRecord(ev[0], s);
    k_router<MODE><<<p.g_router, kThreads, p.sm_router, s>>>(L.router, L.E, L.H, Q, x, r, ws.logits, ws.u, r_trace,
                                                             clear ? ws.status : nullptr);
    if (ev) cudaEventRecord(ev[1], s);
    k_gate_up<Q><<<p.g_gate, kCtaThreads, p.sm_gate, s>>>(ga);
    if (ev) cudaEventRecord(ev[2], s);
    k_down<Q, MODE><<<p.g_down, kCtaThreads, p.sm_down, s>>>(da);
    return launch_status();
}

template <int MODE>
int dispatch_q(int q, const moe_layer& L, const Plan& p, int k, const uint16_t* x, const float* r, float* out,
               int32_t* idx_out, float* w_out, float* logits_out, float* r_trace, WsPtrs ws, bool clear,
               cudaEvent_t const* ev, cudaStream_t s) {
    switch (q) {
        case 1: return launch_layer<1, MODE>(L, p, k, x, r, out, idx_out, w_out, logits_out, r_trace, ws, clear, ev, s);
        case 2: return launch_layer<2, MODE>(L, p, k, x, r, out, idx_out, w_out, logits_out, r_trace, ws, clear, ev, s);
        case 3: return launch_layer<3, MODE>(L, p, k, x, r, out, idx_out, w_out, logits_out, r_trace, ws, clear, ev, s);
        case 4: return launch_layer<4, MODE>(L, p, k, x, r, out, idx_out, w_out, logits_out, r_trace, ws, clear, ev, s);
        default: return FPX_EINVAL;
    }
}

}  // namespace

extern "C" {

int moe_route_topk(const float* R, int E, int H, const uint16_t* x, int q, int k, float* logits, int32_t* idx, float* w,
                   int32_t* uni, int32_t* n_uni, void* stream) {
    if (E < 1 || E > kMaxE || H < 16 || H % 16 || q < 1 || q > kMaxQ || k < 1 || k > kMaxK || k > E) return FPX_EINVAL;
    if (!R || !x || !logits || !idx || !w || !uni || !n_uni) return FPX_EINVAL;
    if (!aligned(R, 16) || !aligned(x, 4) || !aligned(logits, 4)) return FPX_EALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    size_t sm = sizeof(float) * ((size_t)q * H + 8 * kMaxQ + 8);
    if (cudaFuncSetAttribute(k_router<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm)) return FPX_ECUDA;
    k_router<0><<<(E + 1) / 2, kThreads, sm, s>>>(R, E, H, q, x, nullptr, logits, nullptr, nullptr, nullptr);
    k_topk<<<1, 32 * kMaxQ, 0, s>>>(logits, E, q, k, idx, w, uni, n_uni);
    return launch_status();
}

size_t moe_workspace_bytes(const moe_layer* layer, int q, int k) {
    if (!layer || q < 1 || q > kMaxQ || k < 1 || k > kMaxK || layer->H < 16 || layer->I < 16) return 0;
    return ws_layout(layer->H, layer->I, layer->E, q, k).total;
}

int moe_layer_decode(const moe_layer* layer, const uint16_t* x, int q, int k, float* y, int32_t* idx_out, float* w_out,
                     float* logits_out, void* ws, size_t ws_bytes, void* stream) {
    int st = check_layer(layer);
    if (st) return st;
    if (q < 1 || q > kMaxQ || k < 1 || k > kMaxK || k > layer->E || !x || !y || !ws) return FPX_EINVAL;
    if (!aligned(ws, 16) || !aligned(x, 4) || !aligned(y, 4)) return FPX_EALIGN;
    Ws wl = ws_layout(layer->H, layer->I, layer->E, q, k);
    if (ws_bytes < wl.total) return FPX_ESPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    WsPtrs wp = ws_ptrs(ws, wl);
    // the row-tile counters must start at zero; the kernels leave them at zero
    if (cudaMemsetAsync(wp.cnt, 0, sizeof(int32_t) * (layer->H / 128), s) != cudaSuccess) return FPX_ECUDA;
    Plan p = make_plan(*layer, q);
    return dispatch_q<0>(q, *layer, p, k, x, nullptr, y, idx_out, w_out, logits_out, nullptr, wp, true, nullptr, s);
}

int moe_stack_verify(const moe_layer* layers, int n_layers, const float* r0, int q, int k, float* rL, int32_t* idx_out,
                     float* r_trace, void* ws, size_t ws_bytes, void* const* events, void* stream) {
    if (!layers || n_layers < 1 || !r0 || !rL || !ws || q < 1 || q > kMaxQ || k < 1 || k > kMaxK) return FPX_EINVAL;
    for (int l = 0; l < n_layers; l++) {
        int st = check_layer(&layers[l]);
        if (st) return st;
        if (layers[l].H != layers[0].H || layers[l].I != layers[0].I || layers[l].E != layers[0].E || k > layers[l].E)
            return FPX_EINVAL;
    }
    if (!aligned(ws, 16) || !aligned(r0, 16) || !aligned(rL, 16)) return FPX_EALIGN;
    Ws wl = ws_layout(layers[0].H, layers[0].I, layers[0].E, q, k);
    if (ws_bytes < wl.total) return FPX_ESPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    WsPtrs wp = ws_ptrs(ws, wl);
    const size_t state = sizeof(float) * (size_t)q * layers[0].H;
    if (r0 != rL && cudaMemcpyAsync(rL, r0, state, cudaMemcpyDeviceToDevice, s) != cudaSuccess) return FPX_ECUDA;
    if (cudaMemsetAsync(wp.cnt, 0, sizeof(int32_t) * (layers[0].H / 128), s) != cudaSuccess) return FPX_ECUDA;
    Plan p = make_plan(layers[0], q);
    for (int l = 0; l < n_layers; l++) {
        int32_t* io = idx_out ? idx_out + (size_t)l * q * k : nullptr;
        float* tr = r_trace ? r_trace + (size_t)l * q * layers[0].H : nullptr;
        cudaEvent_t const* ev = events ? reinterpret_cast<cudaEvent_t const*>(events) + 3 * l : nullptr;
        int st = dispatch_q<1>(q, layers[l], p, k, nullptr, rL, rL, io, nullptr, nullptr, tr, wp, l == 0, ev, s);
        if (st) return st;
    }
    if (events && cudaEventRecord(reinterpret_cast<cudaEvent_t const*>(events)[3 * n_layers], s) != cudaSuccess)
        return FPX_ECUDA;
    return FPX_OK;
}

}  // extern "C"

// ------------------------------------------------------------------ fixed-scratch variant
//
// Some callers cannot allocate device memory: code that runs inside a host framework which owns every
// device allocation (a fixed arena or its own allocator) and forbids others, and latency-critical
// loops where cudaMalloc/cudaFree are off limits because they can synchronise the device. For them,
// moe_layer_decode_static_ws runs the same layer with its scratch in the array below, which exists
// once per device for the life of the process.

#include <mutex>

namespace {

constexpr size_t kStaticWsBytes = size_t(8) << 20;  // 8 MiB: the decode shapes need at most 4.4 MB
__device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

// In host code `g_static_ws` only names the symbol; its device address differs per device and is
// looked up once per device (with that device current) and cached here.
constexpr int kMaxDevices = 64;
void* g_static_ws_addr[kMaxDevices] = {};
std::mutex g_static_ws_mu;

int static_ws_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FPX_ECUDA;
    if (dev < 0 || dev >= kMaxDevices) return FPX_EINVAL;
    std::lock_guard<std::mutex> lock(g_static_ws_mu);
    if (!g_static_ws_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || !p) return FPX_ECUDA;
        g_static_ws_addr[dev] = p;
    }
    *out = g_static_ws_addr[dev];
    return FPX_OK;
}

}  // namespace

extern "C" int moe_layer_decode_static_ws(const moe_layer* layer, const uint16_t* x, int q, int k, float* y,
                                          int32_t* idx_out, float* w_out, float* logits_out, int32_t* dev_status,
                                          void* stream) {
    if (!layer || q < 1 || q > kMaxQ || k < 1 || k > kMaxK) return FPX_EINVAL;
    const size_t need = moe_workspace_bytes(layer, q, k);
    if (need == 0) return FPX_EINVAL;
    if (need > kStaticWsBytes) return FPX_ESPACE;
    if (dev_status && !aligned(dev_status, 4)) return FPX_EALIGN;
    void* ws = nullptr;
    int st = static_ws_address(&ws);
    if (st) return st;
    st = moe_layer_decode(layer, x, q, k, y, idx_out, w_out, logits_out, ws, need, stream);
    if (st) return st;
    if (dev_status &&
        cudaMemcpyAsync(dev_status, ws, sizeof(int32_t), cudaMemcpyDeviceToDevice, static_cast<cudaStream_t>(stream)) !=
            cudaSuccess)
        return FPX_ECUDA;
    return FPX_OK;
}
