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
// per CTA, then gate/up on the tensor cores, h = silu(g) u), k_down (down projection on the tensor
// cores; the last task to finish a 16-row output tile combines it).
#include "fpx_mma.cuh"

using namespace fpx;

namespace {

constexpr int kThreads = 256;  // router and top-k kernels
constexpr int kMaxK = 8;
constexpr int kMaxQ = 4;
constexpr int kMaxE = 1024;

// ------------------------------------------------------------------ workspace

struct Ws {
    size_t status, logits, u, idx, w, uni, nuni, h, yi, cnt, total;
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
    w.yi = o; o = up16(o + sizeof(float) * (size_t)(q * k + 1) * q * H);
    w.cnt = o; o = up16(o + sizeof(int32_t) * (size_t)(H / kTileRows));
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
    float* h;
    float* yi;
    int32_t* cnt;
};

inline WsPtrs ws_ptrs(void* ws, const Ws& l) {
    char* b = static_cast<char*>(ws);
    return WsPtrs{reinterpret_cast<int32_t*>(b + l.status), reinterpret_cast<float*>(b + l.logits),
                  reinterpret_cast<uint16_t*>(b + l.u),     reinterpret_cast<int32_t*>(b + l.idx),
                  reinterpret_cast<float*>(b + l.w),        reinterpret_cast<int32_t*>(b + l.uni),
                  reinterpret_cast<int32_t*>(b + l.nuni),   reinterpret_cast<float*>(b + l.h),
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
    int st = make_row_map(&m->gate, L.gate, rb2, (int64_t)L.E * L.I, rb2, box_bytes(2), kTileRows, 1);
    st = st ? st : make_row_map(&m->up, L.up, rb2, (int64_t)L.E * L.I, rb2, box_bytes(2), kTileRows, 1);
    st = st ? st : make_row_map(&m->down, L.down, rb3, (int64_t)L.E * L.H, rb3, box_bytes(3), kTileRows, 1);
    st = st ? st : make_row_map(&m->sh_gate, L.sh_gate, rb4h, L.I, rb4h, box_bytes(4), kTileRows, 2);
    st = st ? st : make_row_map(&m->sh_up, L.sh_up, rb4h, L.I, rb4h, box_bytes(4), kTileRows, 2);
    st = st ? st : make_row_map(&m->sh_down, L.sh_down, rb4i, L.H, rb4i, box_bytes(4), kTileRows, 2);
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
// normalised over the selected k. Each lane keeps its E / 32 logits in registers.
__device__ void warp_topk(const float* lg, int E, int k, int32_t* idx, float* w) {
    const int lane = threadIdx.x & 31;
    float v[kMaxE / 32];
#pragma unroll
    for (int m = 0; m < kMaxE / 32; m++) v[m] = lane + 32 * m < E ? lg[lane + 32 * m] : 0.0f;
    uint32_t taken = 0;  // bit m: element lane + 32 m already selected
    float sig[kMaxK];
    for (int r = 0; r < k; r++) {
        float bv = 0.0f;
        int bi = -1;
#pragma unroll
        for (int m = 0; m < kMaxE / 32; m++) {
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

// ------------------------------------------------------------------ K2: gate/up + SiLU

// Task = (item, 16-row tile of I); items are the union's experts in order, then the shared expert.
// A routed task streams H/256 units, each a G box and a U box (16 rows x 80 B of FP2); the shared
// task streams 2 * H/512 units, alternately G and U boxes of 16 rows x 272 B of FP4. Consumer warp w
// of a CTA takes the CTA's tasks w, w + 8, ...; the producer warp keeps every consumer's ring full.
struct GateUpArgs {
    LayerMaps m;
    int q, k;
    const uint16_t* x;  // layer input, bfloat16 [q][H]
    WsPtrs ws;
    int32_t* idx_out;
    float* w_out;
    float* logits_out;
};

__device__ __forceinline__ int gu_units(int shared_item, int H) { return shared_item ? 2 * (H / 512) : H / 256; }

// Issues unit `u` of task (item, tile) into slot.
__device__ __forceinline__ void gu_issue(const GateUpArgs& A, const Route& r, int item, int tile, int u, uint8_t* slot,
                                         uint64_t* bar) {
    const int row0 = tile * kTileRows;
    if (item < r.n_uni) {
        const int e = r.uni[item];
        mbar_expect_tx(bar, 2 * kTileRows * box_bytes(2));
        tma_load_2d(slot, &A.m.gate, u * box_bytes(2), e * A.m.I + row0, bar);
        tma_load_2d(slot + kTileRows * box_bytes(2), &A.m.up, u * box_bytes(2), e * A.m.I + row0, bar);
    } else {
        mbar_expect_tx(bar, kTileRows * box_bytes(4));
        tma_load_2d(slot, (u & 1) ? &A.m.sh_up : &A.m.sh_gate, (u >> 1) * (box_bytes(4) / 2), row0, bar);
    }
}

// Producer state for one consumer warp: next task ordinal, next unit in it, units issued.
struct Cursor {
    int pt, pu;
    uint32_t issued;
};

template <int Q>
__global__ void __launch_bounds__(kCtaThreads, 1) k_gate_up(const __grid_constant__ GateUpArgs A) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ Route r;
    __shared__ int shift[kMaxQ];
    __shared__ float red4[(kWarps + 1) * 4];
    const int H = A.m.H, I = A.m.I;
    const Smem S = carve(smem, btab_bytes(H), 2);
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    init_rings(S);

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

    // the CTA's task range; consumer warp w takes tasks c0 + w, c0 + w + kWarps, ...
    const int tiles = I / kTileRows, n_items = r.n_uni + 1;
    const int total = n_items * tiles;
    const int c0 = (int)((int64_t)total * blockIdx.x / gridDim.x), c1 = (int)((int64_t)total * (blockIdx.x + 1) / gridDim.x);
    auto tasks_of = [&](int w) { return c1 - c0 > w ? (c1 - c0 - w + kWarps - 1) / kWarps : 0; };

    // producer: fill every ring before building the activation tables, so the first loads overlap it
    Cursor cur[kWarps];
    const bool producer = warp == kWarps && lane == 0;
    auto try_issue = [&](int w) -> bool {
        Cursor& cw = cur[w];
        if (cw.pt >= tasks_of(w)) return false;
        const Ring R = warp_ring(S, w);
        if (!ring_free(R, cw.issued)) return false;
        const int task = c0 + w + cw.pt * kWarps, item = task / tiles, tile = task % tiles;
        const int slot = cw.issued % kStages;
        gu_issue(A, r, item, tile, cw.pu, R.slots + (size_t)slot * kSlotBytes, R.full + slot);
        cw.issued++;
        if (++cw.pu == gu_units(item == r.n_uni, H)) { cw.pu = 0; cw.pt++; }
        return true;
    };
    if (producer) {
#pragma unroll
        for (int w = 0; w < kWarps; w++) cur[w] = Cursor{0, 0, 0u};
        for (int i = 0; i < kStages; i++)
#pragma unroll
            for (int w = 0; w < kWarps; w++) try_issue(w);
    }

    // activation tables: x scaled per token, FP2 (pair-shifted, with block offsets) and FP4
    build_tables<2, 4, true>(A.x, H, Q, S.tab0, S.tab1, S.csum, shift, red4);
    __syncthreads();

    if (warp == kWarps) {
        if (producer) {
            uint64_t idle_since = 0;
            for (;;) {
                bool pending = false, progress = false;
#pragma unroll
                for (int w = 0; w < kWarps; w++) {
                    if (cur[w].pt < tasks_of(w)) pending = true;
                    progress |= try_issue(w);
                }
                if (!pending) break;
                if (progress) {
                    idle_since = 0;
                } else {
                    const uint64_t now = global_ns();
                    if (!idle_since) idle_since = now;
                    else if (now - idle_since > kWaitNs) { flag(A.ws.status, FPX_ETIMEOUT); break; }
                    __nanosleep(100);
                }
            }
        }
        return;
    }

    // consumers
    const Ring R = warp_ring(S, warp);
    const int my_n = tasks_of(warp);
    const int a_idx = b_active_index(lane);
    uint32_t consumed = 0, expected = 0;
    for (int n = 0; n < my_n; n++) {
        const int task = c0 + warp + n * kWarps;
        expected += gu_units((task / tiles) == r.n_uni, H);
    }
    bool ok = true;
    for (int n = 0; n < my_n && ok; n++) {
        const int task = c0 + warp + n * kWarps, item = task / tiles, tile = task % tiles;
        const bool sh = item == r.n_uni;
        float yg[4] = {0.f, 0.f, 0.f, 0.f}, yu[4] = {0.f, 0.f, 0.f, 0.f};
        const int units = gu_units(sh, H);
        for (int u = 0; u < units; u++) {
            if (!ring_wait(R, consumed, A.ws.status)) { ok = false; break; }
            const uint8_t* slot = R.slots + (consumed % kStages) * kSlotBytes;
            if (!sh) {
                box_mma2<2>(slot, slot + kTileRows * box_bytes(2), box_bytes(2), S.tab0, S.csum, u * box_chunks(2), a_idx, g, t,
                            yg, yu, A.ws.status);
            } else if (u & 1) {
                box_mma1<4>(slot, box_bytes(4), S.tab1, nullptr, (u >> 1) * box_chunks(4), a_idx, g, t, yu, A.ws.status);
            } else {
                box_mma1<4>(slot, box_bytes(4), S.tab1, nullptr, (u >> 1) * box_chunks(4), a_idx, g, t, yg, A.ws.status);
            }
            ring_release(R, consumed);
            consumed++;
        }
        if (!ok) break;
        pair_reduce(yg);
        pair_reduce(yu);
        if (t < 2) {
            const int row = tile * kTileRows + g;
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const int tok = 2 * t + (i & 1), rr = row + 8 * (i >> 1);
                if (tok < Q) {
                    // undo the per-token activation scale (and the 2^-14 of the FP4 decode)
                    const float sc = exp2i((sh ? 14 : 0) - shift[tok]);
                    const float gv = yg[i] * sc, uv = yu[i] * sc;
                    A.ws.h[((size_t)item * Q + tok) * I + rr] = (gv / (1.0f + expf(-gv))) * uv;
                }
            }
        }
    }
    if (!ok) ring_drain(R, consumed, expected);
}

// ------------------------------------------------------------------ K3: down + combine

// Task = (item, 16-row tile of H). A routed task streams I/256 FP3 units (16 rows x 112 B), the
// shared task I/512 FP4 units (16 rows x 272 B). Each CTA owns a contiguous item-major task range,
// which spans at most two items; it builds their activation tables from h at start. After a task
// writes its 16 x q outputs to ws.yi, the last task to finish that row tile (integer counter)
// combines the tile for every token: selected experts in ascending expert order, then the shared
// expert.
struct DownArgs {
    LayerMaps m;
    int q, k;
    WsPtrs ws;
    float* out;  // MODE 0: y [q][H]; MODE 1: residual r [q][H], updated in place
};

__device__ __forceinline__ int dn_units(int shared_item, int I) { return shared_item ? I / 512 : I / 256; }

__device__ __forceinline__ void dn_issue(const DownArgs& A, const Route& r, int item, int tile, int u, uint8_t* slot,
                                         uint64_t* bar) {
    const int row0 = tile * kTileRows;
    if (item < r.n_uni) {
        mbar_expect_tx(bar, kTileRows * box_bytes(3));
        tma_load_2d(slot, &A.m.down, u * box_bytes(3), r.uni[item] * A.m.H + row0, bar);
    } else {
        mbar_expect_tx(bar, kTileRows * box_bytes(4));
        tma_load_2d(slot, &A.m.sh_down, u * (box_bytes(4) / 2), row0, bar);
    }
}

template <int Q, int MODE>
__global__ void __launch_bounds__(kCtaThreads, 1) k_down(const __grid_constant__ DownArgs A) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ Route r;
    __shared__ float wsel[kMaxQ * kMaxK + 1][kMaxQ];  // weight of token t for union item j, NaN if unselected
    __shared__ int shift[2][kMaxQ];
    __shared__ float red4[(kWarps + 1) * 4];
    const int H = A.m.H, I = A.m.I;
    const Smem S = carve(smem, btab_bytes(I), 2);
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    init_rings(S);

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

    const int tiles = H / kTileRows, n_items = r.n_uni + 1;
    const int total = n_items * tiles;
    const int c0 = (int)((int64_t)total * blockIdx.x / gridDim.x), c1 = (int)((int64_t)total * (blockIdx.x + 1) / gridDim.x);
    const int item_lo = c0 / tiles;
    auto tasks_of = [&](int w) { return c1 - c0 > w ? (c1 - c0 - w + kWarps - 1) / kWarps : 0; };

    Cursor cur[kWarps];
    const bool producer = warp == kWarps && lane == 0;
    auto try_issue = [&](int w) -> bool {
        Cursor& cw = cur[w];
        if (cw.pt >= tasks_of(w)) return false;
        const Ring R = warp_ring(S, w);
        if (!ring_free(R, cw.issued)) return false;
        const int task = c0 + w + cw.pt * kWarps, item = task / tiles, tile = task % tiles;
        const int slot = cw.issued % kStages;
        dn_issue(A, r, item, tile, cw.pu, R.slots + (size_t)slot * kSlotBytes, R.full + slot);
        cw.issued++;
        if (++cw.pu == dn_units(item == r.n_uni, I)) { cw.pu = 0; cw.pt++; }
        return true;
    };
    if (producer) {
#pragma unroll
        for (int w = 0; w < kWarps; w++) cur[w] = Cursor{0, 0, 0u};
        for (int i = 0; i < kStages; i++)
#pragma unroll
            for (int w = 0; w < kWarps; w++) try_issue(w);
    }

    // activation tables for the (at most two) items of this CTA's range
    for (int s = 0; s < 2; s++) {
        const int item = item_lo + s;
        if (c1 <= c0 || item >= n_items || item * tiles >= c1) continue;
        const float* hsrc = A.ws.h + (size_t)item * Q * I;
        if (item == r.n_uni) build_tables<4, 0, false>(hsrc, I, Q, s ? S.tab1 : S.tab0, nullptr, nullptr, shift[s], red4);
        else build_tables<3, 0, false>(hsrc, I, Q, s ? S.tab1 : S.tab0, nullptr, nullptr, shift[s], red4);
        __syncthreads();
    }
    __syncthreads();

    if (warp == kWarps) {
        if (producer) {
            uint64_t idle_since = 0;
            for (;;) {
                bool pending = false, progress = false;
#pragma unroll
                for (int w = 0; w < kWarps; w++) {
                    if (cur[w].pt < tasks_of(w)) pending = true;
                    progress |= try_issue(w);
                }
                if (!pending) break;
                if (progress) {
                    idle_since = 0;
                } else {
                    const uint64_t now = global_ns();
                    if (!idle_since) idle_since = now;
                    else if (now - idle_since > kWaitNs) { flag(A.ws.status, FPX_ETIMEOUT); break; }
                    __nanosleep(100);
                }
            }
        }
        return;
    }

    const Ring R = warp_ring(S, warp);
    const int my_n = tasks_of(warp);
    const int a_idx = b_active_index(lane);
    uint32_t consumed = 0, expected = 0;
    for (int n = 0; n < my_n; n++) expected += dn_units(((c0 + warp + n * kWarps) / tiles) == r.n_uni, I);
    bool ok = true;
    for (int n = 0; n < my_n && ok; n++) {
        const int task = c0 + warp + n * kWarps, item = task / tiles, tile = task % tiles;
        const bool sh = item == r.n_uni;
        const int s = item - item_lo;
        const uint2* tab = s ? S.tab1 : S.tab0;
        float y[4] = {0.f, 0.f, 0.f, 0.f};
        const int units = dn_units(sh, I);
        for (int u = 0; u < units; u++) {
            if (!ring_wait(R, consumed, A.ws.status)) { ok = false; break; }
            const uint8_t* slot = R.slots + (consumed % kStages) * kSlotBytes;
            if (!sh) box_mma1<3>(slot, box_bytes(3), tab, nullptr, u * box_chunks(3), a_idx, g, t, y, A.ws.status);
            else box_mma1<4>(slot, box_bytes(4), tab, nullptr, u * box_chunks(4), a_idx, g, t, y, A.ws.status);
            ring_release(R, consumed);
            consumed++;
        }
        if (!ok) break;
        pair_reduce(y);
        if (t < 2) {
            const int row = tile * kTileRows + g;
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const int tok = 2 * t + (i & 1), rr = row + 8 * (i >> 1);
                if (tok < Q) A.ws.yi[((size_t)item * Q + tok) * H + rr] = y[i] * exp2i((sh ? 14 : 0) - shift[s][tok]);
            }
        }
        // the last task to finish this row tile combines it
        __threadfence();
        __syncwarp();
        int last = 0;
        if (lane == 0) last = atomicAdd(A.ws.cnt + tile, 1) == n_items - 1;
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
            __threadfence();
            for (int o = lane; o < kTileRows * Q; o += 32) {
                const int rr = tile * kTileRows + o / Q, tok = o % Q;
                float acc = 0.0f;
                bool first = true;
                for (int j = 0; j < r.n_uni; j++) {
                    const float wv = wsel[j][tok];
                    if (wv != wv) continue;  // expert not selected by this token
                    const float yv = __ldcg(A.ws.yi + ((size_t)j * Q + tok) * H + rr);
                    acc = first ? wv * yv : fmaf(wv, yv, acc);
                    first = false;
                }
                acc += __ldcg(A.ws.yi + ((size_t)r.n_uni * Q + tok) * H + rr);
                const size_t oi = (size_t)tok * H + rr;
                if (MODE == 0) A.out[oi] = acc;
                else A.out[oi] = A.out[oi] + acc;
            }
            if (lane == 0) A.ws.cnt[tile] = 0;  // ready for the next call
        }
    }
    if (!ok) ring_drain(R, consumed, expected);
}

// ------------------------------------------------------------------ launch plumbing

int check_layer(const moe_layer* L) {
    if (!L || L->H < 512 || L->I < 512 || L->H % 512 || L->I % 512 || L->E < 1 || L->E > kMaxE) return FPX_EINVAL;
    if (!L->router || !L->gate || !L->up || !L->down || !L->sh_gate || !L->sh_up || !L->sh_down) return FPX_EINVAL;
    if (!aligned(L->router, 16) || !aligned(L->gate, 16) || !aligned(L->up, 16) || !aligned(L->down, 16) ||
        !aligned(L->sh_gate, 16) || !aligned(L->sh_up, 16) || !aligned(L->sh_down, 16))
        return FPX_EALIGN;
    if (smem_bytes(btab_bytes(L->H > L->I ? L->H : L->I), 2) > 227 * 1024) return FPX_EINVAL;
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
    p.sm_gate = smem_bytes(btab_bytes(L.H), 2);
    p.g_down = di.sms;
    p.sm_down = smem_bytes(btab_bytes(L.I), 2);
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
    if (cudaMemsetAsync(wp.cnt, 0, sizeof(int32_t) * (layer->H / kTileRows), s) != cudaSuccess) return FPX_ECUDA;
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
    if (cudaMemsetAsync(wp.cnt, 0, sizeof(int32_t) * (layers[0].H / kTileRows), s) != cudaSuccess) return FPX_ECUDA;
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

constexpr size_t kStaticWsBytes = size_t(4) << 20;  // 4 MiB: the decode shapes need at most 3.3 MB
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
