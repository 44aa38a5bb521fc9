// The MoE decode/verify step: router + top-k + union, gate/up + SiLU, down + weighted combine, and
// the stack driver. Follows "DeepSeek V4 Flash hits 32 tok/s on AMD Ryzen AI MAX+ 395", paragraph 3
// (q = 4 verification columns, each packed weight decoded once and applied to all of them, routing
// through TOP_K/ARGSORT kernels, 43 memory-bound layers) and "Token Freedom via APU ...", section
// "Lucebox's Optimization Trio" (256 routed experts plus one shared expert).
//
// Readings (the pages leave these open): sigmoid scores, top-k on the logit with ties to the lower
// expert index, weights normalised over the selected k; h = silu(g) * u kept in binary32; combine in
// rank order with the shared expert last; the stack's layer input is the bfloat16 RMS normalisation
// (eps 1e-6, no gain) of a binary32 residual.
#include "fpx_common.cuh"

using namespace fpx;

namespace {

constexpr int kThreads = 256;
constexpr int kMaxK = 8;
constexpr int kMaxQ = 4;
constexpr int kMaxE = 1024;

// ------------------------------------------------------------------ workspace

struct Ws {
    size_t status, logits, u, idx, w, uni, nuni, h, total;
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
    w.h = o; o = up16(o + sizeof(float) * (size_t)(q * k + 1) * q * I);
    w.total = o;
    return w;
}

struct LayerPtrs {
    int H, I, E;
    const float* router;
    const uint8_t *gate, *up, *down, *sh_gate, *sh_up, *sh_down;
    int64_t mb_gu, mb_d, row_gu2, row_gu4, row_d3, row_d4;  // matrix strides and row bytes
};

inline LayerPtrs layer_ptrs(const moe_layer& L) {
    LayerPtrs p{};
    p.H = L.H; p.I = L.I; p.E = L.E;
    p.router = L.router;
    p.gate = L.gate; p.up = L.up; p.down = L.down;
    p.sh_gate = L.sh_gate; p.sh_up = L.sh_up; p.sh_down = L.sh_down;
    p.mb_gu = matrix_bytes(2, L.I, L.H);
    p.mb_d = matrix_bytes(3, L.H, L.I);
    p.row_gu2 = (int64_t)(L.H / 32) * 10;
    p.row_gu4 = (int64_t)(L.H / 32) * 17;
    p.row_d3 = (int64_t)(L.I / 32) * 14;
    p.row_d4 = (int64_t)(L.I / 32) * 17;
    return p;
}

struct WsPtrs {
    int32_t* status;
    float* logits;
    uint16_t* u;
    int32_t* idx;
    float* w;
    int32_t* uni;
    int32_t* nuni;
    float* h;
};

inline WsPtrs ws_ptrs(void* ws, const Ws& l) {
    char* b = static_cast<char*>(ws);
    return WsPtrs{reinterpret_cast<int32_t*>(b + l.status), reinterpret_cast<float*>(b + l.logits),
                  reinterpret_cast<uint16_t*>(b + l.u),     reinterpret_cast<int32_t*>(b + l.idx),
                  reinterpret_cast<float*>(b + l.w),        reinterpret_cast<int32_t*>(b + l.uni),
                  reinterpret_cast<int32_t*>(b + l.nuni),   reinterpret_cast<float*>(b + l.h)};
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

// ------------------------------------------------------------------ K1: router logits

// Computes the layer input into u_s (binary32 values of bfloat16) and logits[t][e] for this CTA's
// experts. MODE 0: input x is bfloat16. MODE 1: input is the residual r; u = RN_bf16(r / rms(r)).
// Each CTA handles 2 experts with 4 warps per expert, each warp a quarter of H; the quarter sums are
// added in order.
template <int MODE>
__global__ void __launch_bounds__(kThreads) k_router(const float* __restrict__ R, int E, int H, int q,
                                                     const uint16_t* __restrict__ xin, const float* __restrict__ rin,
                                                     float* __restrict__ logits, uint16_t* __restrict__ u_out,
                                                     float* __restrict__ r_trace, int32_t* status_to_clear) {
    extern __shared__ float sm[];
    float* u_s = sm;                      // [q][H]
    float* part = sm + (size_t)q * H;     // [8 warps][q]
    float* red = part + 8 * kMaxQ;        // [8]
    if (status_to_clear && blockIdx.x == 0 && threadIdx.x == 0) *status_to_clear = 0;
    if (MODE == 0) {
        for (int i = threadIdx.x; i < q * H; i += blockDim.x) u_s[i] = bf16_bits_to_float(xin[i]);
    } else {
        for (int t = 0; t < q; t++) {
            float ss = 0.0f;
            for (int h = threadIdx.x; h < H; h += blockDim.x) {
                float v = rin[(size_t)t * H + h];
                ss = fmaf(v, v, ss);
            }
            ss = block_sum(ss, red);
            const float inv = 1.0f / sqrtf(ss / (float)H + 1e-6f);
            for (int h = threadIdx.x; h < H; h += blockDim.x) {
                float rv = rin[(size_t)t * H + h];
                __nv_bfloat16 b = __float2bfloat16_rn(rv * inv);
                u_s[(size_t)t * H + h] = __bfloat162float(b);
                if (blockIdx.x == 0) {
                    u_out[(size_t)t * H + h] = __bfloat16_as_ushort(b);
                    if (r_trace) r_trace[(size_t)t * H + h] = rv;
                }
            }
        }
    }
    __syncthreads();
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    const int e = blockIdx.x * 2 + warp / 4, slice = warp % 4;
    const int h0 = (int)((int64_t)H * slice / 4), h1 = (int)((int64_t)H * (slice + 1) / 4);
    float acc[kMaxQ] = {0.f, 0.f, 0.f, 0.f};
    if (e < E) {
        const float* row = R + (size_t)e * H;
        for (int h = h0 + lane; h < h1; h += 32) {
            float rv = __ldg(row + h);
#pragma unroll
            for (int t = 0; t < kMaxQ; t++)
                if (t < q) acc[t] = fmaf(rv, u_s[(size_t)t * H + h], acc[t]);
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
// normalised over the selected k. taken[] is scratch of E bytes (shared memory, zeroed here).
__device__ void warp_topk(const float* lg, int E, int k, uint8_t* taken, int32_t* idx, float* w) {
    const int lane = threadIdx.x & 31;
    for (int e = lane; e < E; e += 32) taken[e] = 0;
    __syncwarp();
    float sig[kMaxK];
    for (int r = 0; r < k; r++) {
        float bv = 0.0f;
        int bi = -1;
        for (int e = lane; e < E; e += 32) {
            if (taken[e]) continue;
            float v = lg[e];
            if (bi < 0 || v > bv) { bv = v; bi = e; }  // e ascending: equal values keep the lower index
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            bool better = oi >= 0 && (bi < 0 || ov > bv || (ov == bv && oi < bi));
            if (better) { bv = ov; bi = oi; }
        }
        if (lane == 0) taken[bi] = 1;
        __syncwarp();
        idx[r] = bi;
        sig[r] = 1.0f / (1.0f + expf(-bv));
    }
    float S = sig[0];
    for (int r = 1; r < k; r++) S += sig[r];
    for (int r = 0; r < k; r++) w[r] = sig[r] / S;
}

// Shared-memory routing state used by the gate/up and down kernels.
struct Route {
    int32_t idx[kMaxQ * kMaxK];
    float w[kMaxQ * kMaxK];
    int32_t uni[kMaxQ * kMaxK];
    int32_t slot[kMaxQ * kMaxK];  // position of idx[t][r] in uni
    uint32_t mask[kMaxE / 32];
    int32_t n_uni;
};

// Fills Route from the top-k results already in r.idx / r.w: sorted union and slots. Whole CTA.
__device__ void build_union(Route& r, int q, int k, int E) {
    for (int i = threadIdx.x; i < kMaxE / 32; i += blockDim.x) r.mask[i] = 0u;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int i = 0; i < q * k; i++) r.mask[r.idx[i] >> 5] |= 1u << (r.idx[i] & 31);
        int n = 0;
        for (int wd = 0; wd < (E + 31) / 32; wd++) {
            uint32_t m = r.mask[wd];
            while (m) {
                int b = __ffs(m) - 1;
                m &= m - 1;
                r.uni[n++] = wd * 32 + b;
            }
        }
        r.n_uni = n;
        for (int i = 0; i < q * k; i++) {
            int s = 0;
            while (r.uni[s] != r.idx[i]) s++;
            r.slot[i] = s;
        }
    }
    __syncthreads();
}

__global__ void k_topk(const float* __restrict__ logits, int E, int q, int k, int32_t* idx, float* w, int32_t* uni,
                       int32_t* n_uni) {
    __shared__ Route r;
    __shared__ uint8_t taken[kMaxQ][kMaxE];
    const int warp = threadIdx.x / 32;
    if (warp < q) warp_topk(logits + (size_t)warp * E, E, k, taken[warp], r.idx + warp * k, r.w + warp * k);
    __syncthreads();
    build_union(r, q, k, E);
    for (int i = threadIdx.x; i < q * k; i += blockDim.x) {
        idx[i] = r.idx[i];
        w[i] = r.w[i];
        uni[i] = i < r.n_uni ? r.uni[i] : -1;
    }
    if (threadIdx.x == 0) *n_uni = r.n_uni;
}

// ------------------------------------------------------------------ K2: gate/up + SiLU

// Every CTA recomputes the routing from the logits (cheap, deterministic) so no extra launch or
// grid-wide synchronisation is needed; CTA 0 publishes it. Then the (item, row) pairs, item = union
// slot or the shared expert (last), are split evenly over the grid; each warp computes one row of
// G and U for all q columns and writes h = silu(g) * u.
template <int Q>
__global__ void __launch_bounds__(kThreads) k_gate_up(LayerPtrs L, int k, const uint16_t* __restrict__ x,
                                                      WsPtrs ws, int32_t* idx_out, float* w_out, float* logits_out) {
    extern __shared__ float sm[];
    __shared__ Route r;
    __shared__ uint8_t taken[kMaxQ][kMaxE];
    const int H = L.H, I = L.I;
    const int xstride = padded_len(H);
    float* xs = sm;
    for (int i = threadIdx.x; i < Q * H; i += blockDim.x)
        xs[(i / H) * xstride + padded_index(i % H)] = bf16_bits_to_float(x[i]);
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    if (warp < Q) warp_topk(ws.logits + (size_t)warp * L.E, L.E, k, taken[warp], r.idx + warp * k, r.w + warp * k);
    __syncthreads();
    build_union(r, Q, k, L.E);
    if (blockIdx.x == 0) {
        for (int i = threadIdx.x; i < Q * k; i += blockDim.x) {
            ws.idx[i] = r.idx[i];
            ws.w[i] = r.w[i];
            ws.uni[i] = i < r.n_uni ? r.uni[i] : -1;
            if (idx_out) idx_out[i] = r.idx[i];
            if (w_out) w_out[i] = r.w[i];
        }
        if (logits_out)
            for (int i = threadIdx.x; i < Q * L.E; i += blockDim.x) logits_out[i] = ws.logits[i];
        if (threadIdx.x == 0) *ws.nuni = r.n_uni;
    }
    const int n_items = r.n_uni + 1;
    const int64_t total = (int64_t)n_items * I;
    const int64_t b0 = total * blockIdx.x / gridDim.x, b1 = total * (blockIdx.x + 1) / gridDim.x;
    for (int64_t p = b0 + warp; p < b1; p += kThreads / 32) {
        const int item = (int)(p / I), row = (int)(p % I);
        float g[Q], u[Q];
        if (item < r.n_uni) {
            const int64_t e = r.uni[item];
            const uint8_t* G = L.gate + e * L.mb_gu + row * L.row_gu2;
            const uint8_t* U = L.up + e * L.mb_gu + row * L.row_gu2;
            row_dot<2, Q>(G, H / 32, XShared{xs, xstride}, lane, g, ws.status);
            row_dot<2, Q>(U, H / 32, XShared{xs, xstride}, lane, u, ws.status);
        } else {
            row_dot<4, Q>(L.sh_gate + row * L.row_gu4, H / 32, XShared{xs, xstride}, lane, g, ws.status);
            row_dot<4, Q>(L.sh_up + row * L.row_gu4, H / 32, XShared{xs, xstride}, lane, u, ws.status);
        }
#pragma unroll
        for (int t = 0; t < Q; t++)
            if (lane == t) {
                float hv = (g[t] / (1.0f + expf(-g[t]))) * u[t];
                ws.h[((size_t)item * Q + t) * I + row] = hv;
            }
    }
}

// ------------------------------------------------------------------ K3: down + combine

// CTA c owns output rows [c*H/G, (c+1)*H/G). For each item it stages h_item in shared memory and
// computes y_item for its rows; then out[t] = sum_r w[t][r] * y_{slot(t,r)}[t] + y_shared[t] in rank
// order. MODE 0 writes out to y; MODE 1 adds it to the residual r in place.
template <int Q, int MODE>
__global__ void __launch_bounds__(kThreads) k_down(LayerPtrs L, int k, WsPtrs ws, float* __restrict__ out,
                                                   int rows_max) {
    extern __shared__ float sm[];
    __shared__ Route r;
    const int H = L.H, I = L.I;
    const int hstride = padded_len(I);
    float* hs = sm;                              // [Q][padded I]
    float* ytile = sm + (size_t)Q * hstride;     // [items][Q][rows_max]
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) r.n_uni = *ws.nuni;
    for (int i = threadIdx.x; i < Q * k; i += blockDim.x) { r.idx[i] = ws.idx[i]; r.w[i] = ws.w[i]; r.uni[i] = ws.uni[i]; }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int i = 0; i < Q * k; i++) {
            int s = 0;
            while (s < r.n_uni - 1 && r.uni[s] != r.idx[i]) s++;
            if (r.uni[s] != r.idx[i]) flag(ws.status, FPX_EDATA);
            r.slot[i] = s;
        }
    }
    const int row0 = (int)((int64_t)H * blockIdx.x / gridDim.x), row1 = (int)((int64_t)H * (blockIdx.x + 1) / gridDim.x);
    const int n_items = r.n_uni + 1;
    for (int item = 0; item < n_items; item++) {
        __syncthreads();
        const float* hsrc = ws.h + (size_t)item * Q * I;
        for (int i = threadIdx.x; i < Q * I; i += blockDim.x) hs[(i / I) * hstride + padded_index(i % I)] = hsrc[i];
        __syncthreads();
        const bool shared = item == r.n_uni;
        const int64_t e = shared ? 0 : r.uni[item];
        if (!shared && (e < 0 || e >= L.E)) { flag(ws.status, FPX_EDATA); continue; }
        for (int row = row0 + warp; row < row1; row += kThreads / 32) {
            float acc[Q];
            if (shared) row_dot<4, Q>(L.sh_down + row * L.row_d4, I / 32, XShared{hs, hstride}, lane, acc, ws.status);
            else row_dot<3, Q>(L.down + e * L.mb_d + row * L.row_d3, I / 32, XShared{hs, hstride}, lane, acc, ws.status);
#pragma unroll
            for (int t = 0; t < Q; t++)
                if (lane == t) ytile[((size_t)item * Q + t) * rows_max + (row - row0)] = acc[t];
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < Q * (row1 - row0); i += blockDim.x) {
        const int t = i / (row1 - row0), rl = i % (row1 - row0);
        float o = r.w[t * k] * ytile[((size_t)r.slot[t * k] * Q + t) * rows_max + rl];
        for (int rr = 1; rr < k; rr++) o = fmaf(r.w[t * k + rr], ytile[((size_t)r.slot[t * k + rr] * Q + t) * rows_max + rl], o);
        o += ytile[((size_t)r.n_uni * Q + t) * rows_max + rl];
        const size_t oi = (size_t)t * H + row0 + rl;
        if (MODE == 0) out[oi] = o;
        else out[oi] = out[oi] + o;
    }
}

// ------------------------------------------------------------------ launch plumbing

int check_layer(const moe_layer* L) {
    if (!L || L->H < 256 || L->I < 256 || L->H % 256 || L->I % 256 || L->E < 1 || L->E > kMaxE) return FPX_EINVAL;
    if (!L->router || !L->gate || !L->up || !L->down || !L->sh_gate || !L->sh_up || !L->sh_down) return FPX_EINVAL;
    if (!aligned(L->router, 16) || !aligned(L->gate, 16) || !aligned(L->up, 16) || !aligned(L->down, 16) ||
        !aligned(L->sh_gate, 16) || !aligned(L->sh_up, 16) || !aligned(L->sh_down, 16))
        return FPX_EALIGN;
    return FPX_OK;
}

struct Plan {
    int g_router, g_gate, g_down, rows_max;
    size_t sm_router, sm_gate, sm_down;
};

Plan make_plan(const moe_layer& L, int q, int k) {
    DeviceInfo di = device_info();
    Plan p{};
    p.g_router = (L.E + 1) / 2;
    p.sm_router = sizeof(float) * ((size_t)q * L.H + 8 * kMaxQ + 8);
    p.g_gate = di.sms * 2;
    p.sm_gate = sizeof(float) * (size_t)q * padded_len(L.H);
    p.g_down = di.sms;
    p.rows_max = (L.H + p.g_down - 1) / p.g_down + 1;
    p.sm_down = sizeof(float) * ((size_t)q * padded_len(L.I) + (size_t)(q * k + 1) * q * p.rows_max);
    return p;
}

template <int Q, int MODE>
int launch_layer(const moe_layer& L, const Plan& p, int k, const uint16_t* x, const float* r, float* out,
                 int32_t* idx_out, float* w_out, float* logits_out, float* r_trace, WsPtrs ws, bool clear,
                 cudaEvent_t const* ev, cudaStream_t s) {
    LayerPtrs lp = layer_ptrs(L);
    if (cudaFuncSetAttribute(k_router<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.sm_router) ||
        cudaFuncSetAttribute(k_gate_up<Q>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.sm_gate) ||
        cudaFuncSetAttribute(k_down<Q, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.sm_down))
        return FPX_ECUDA;
    if (ev) cudaEventRecord(ev[0], s);
    k_router<MODE><<<p.g_router, kThreads, p.sm_router, s>>>(L.router, L.E, L.H, Q, x, r, ws.logits, ws.u, r_trace,
                                                             clear ? ws.status : nullptr);
    const uint16_t* xin = MODE == 0 ? x : ws.u;
    if (ev) cudaEventRecord(ev[1], s);
    k_gate_up<Q><<<p.g_gate, kThreads, p.sm_gate, s>>>(lp, k, xin, ws, idx_out, w_out, logits_out);
    if (ev) cudaEventRecord(ev[2], s);
    k_down<Q, MODE><<<p.g_down, kThreads, p.sm_down, s>>>(lp, k, ws, out, p.rows_max);
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
    if (E < 1 || E > kMaxE || H < 8 || H % 8 || q < 1 || q > kMaxQ || k < 1 || k > kMaxK || k > E) return FPX_EINVAL;
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
    if (!layer || q < 1 || q > kMaxQ || k < 1 || k > kMaxK) return 0;
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
    Plan p = make_plan(*layer, q, k);
    return dispatch_q<0>(q, *layer, p, k, x, nullptr, y, idx_out, w_out, logits_out, nullptr, ws_ptrs(ws, wl), true,
                         nullptr, static_cast<cudaStream_t>(stream));
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
    if (!aligned(ws, 16) || !aligned(r0, 4) || !aligned(rL, 4)) return FPX_EALIGN;
    Ws wl = ws_layout(layers[0].H, layers[0].I, layers[0].E, q, k);
    if (ws_bytes < wl.total) return FPX_ESPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t state = sizeof(float) * (size_t)q * layers[0].H;
    if (r0 != rL && cudaMemcpyAsync(rL, r0, state, cudaMemcpyDeviceToDevice, s) != cudaSuccess) return FPX_ECUDA;
    Plan p = make_plan(layers[0], q, k);
    WsPtrs wp = ws_ptrs(ws, wl);
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

constexpr size_t kStaticWsBytes = size_t(4) << 20;  // 4 MiB: the decode shapes need about 1.1 MB
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
