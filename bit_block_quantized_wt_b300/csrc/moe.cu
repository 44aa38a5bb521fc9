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
// Per layer five kernels, each launched to overlap the previous one's tail: k_router (normalise,
// router GEMV, gate/up activation tables; its last CTA routes every token), k_gate_up (gate/up on the
// tensor cores), k_hpack (h = silu(g) u and the down activation tables), k_down (down projection on
// the tensor cores) and k_combine (weighted sum per token).
#include "fpx_mma.cuh"
#include "route.cuh"

using namespace fpx;

namespace {

constexpr int kThreads = 256;  // router and top-k kernels
constexpr int kMaxK = 8;
constexpr int kMaxQ = 4;
constexpr int kMaxE = 1024;

// Fixed pieces. A task of S stages (one output matrix x one row block, streamed along K) is computed
// as pieces_of(S, D) pieces of consecutive stages, piece p covering stages [p S / P, (p + 1) S / P) with
// its own accumulators starting at zero; each piece writes its own partial buffer and the next kernel
// adds the pieces of a task in piece order. The split depends on the matrix shape alone, never on the
// expert union, the grid or the other tokens, so every column of a batched call is computed with the
// same roundings as a call on that column alone ("DeepSeek V4 Flash hits 32 tok/s on AMD Ryzen AI
// MAX+ 395", paragraph 3: each packed weight decoded once and applied to every verification column).
// Stages per piece: D_gu for the gate/up tasks, D_dn for the down tasks (coarser pieces cost fewer
// partial outputs; finer ones balance the CTAs better, which matters more for the shorter down tasks).
constexpr int kSppGu = 8, kSppDn = 4;
__host__ __device__ constexpr int pieces_of(int S, int D) { return (S + D - 1) / D; }
__host__ __device__ constexpr int piece_begin(int S, int D, int p) { return p * S / pieces_of(S, D); }
constexpr int kMaxPieces = pieces_of(4608 / 256, kSppDn < kSppGu ? kSppDn : kSppGu);  // H, I <= 4608

// Programmatic dependent launch: each layer kernel is launched so that it may start while the
// previous kernel's last CTAs still run; grid_dep_wait() blocks until that kernel has completed and
// its writes are visible. Work that does not read the previous kernel's output goes before it.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the next kernel launch early (it still waits for this one with grid_dep_wait()).
__device__ __forceinline__ void grid_dep_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------------------ workspace

struct Ws {
    size_t status, logits, u, idx, w, uni, uslot, nuni, stage, gu, yi, gt, dt, total;
    size_t gu_piece, yi_piece;  // floats between consecutive piece buffers
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
    w.uslot = o; o = up16(o + sizeof(int32_t) * q * k);
    w.nuni = o; o += 16;  // n_uni, then the router's arrival counter
    w.stage = o; o = up16(o + sizeof(int32_t) * (1 + 2 * q * k));  // two-tier copy list
    w.gu_piece = (size_t)2 * (q * k + 1) * q * I;
    w.yi_piece = (size_t)(q * k + 1) * q * H;
    w.gu = o; o = up16(o + sizeof(float) * pieces_of(H / stage_k(2), kSppGu) * w.gu_piece);  // FP2 tasks have the most pieces
    w.yi = o; o = up16(o + sizeof(float) * pieces_of(I / stage_k(3), kSppDn) * w.yi_piece);
    w.gt = o; o = up16(o + tset_bytes(H));
    w.dt = o; o = up16(o + (size_t)(q * k + 1) * dset_bytes(I));
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
    float* gu;  // g and u of every item: [piece][2 * item + (0 | 1)][q][I]
    float* yi;  // per-item outputs [piece][item][q][H]
    size_t gu_piece, yi_piece;
    uint8_t* gt;  // gate/up activation tables (table set for K = H), built by the router kernel
    uint8_t* dt;  // down activation tables, one table set for K = I per item, built by k_hpack
    int32_t* uslot;  // matrix slot of every union item (the expert id, or its slot in a two-tier layer)
    int32_t* stage;  // two-tier copy list: [count, expert[q k], slot[q k]]
};

inline WsPtrs ws_ptrs(void* ws, const Ws& l) {
    char* b = static_cast<char*>(ws);
    return WsPtrs{reinterpret_cast<int32_t*>(b + l.status), reinterpret_cast<float*>(b + l.logits),
                  reinterpret_cast<uint16_t*>(b + l.u),     reinterpret_cast<int32_t*>(b + l.idx),
                  reinterpret_cast<float*>(b + l.w),        reinterpret_cast<int32_t*>(b + l.uni),
                  reinterpret_cast<int32_t*>(b + l.nuni),   reinterpret_cast<float*>(b + l.gu),
                  reinterpret_cast<float*>(b + l.yi),       l.gu_piece,
                  l.yi_piece,                                reinterpret_cast<uint8_t*>(b + l.gt),
                  reinterpret_cast<uint8_t*>(b + l.dt),      reinterpret_cast<int32_t*>(b + l.uslot),
                  reinterpret_cast<int32_t*>(b + l.stage)};
}

// Everything the gate/up and down kernels need about one layer: the stacked box-tiled matrices
// (fpx_tile_matrices) and the shapes. A stage is one tile, streamed with one 1-D bulk copy.
struct LayerMaps {
    const uint8_t *gate, *up, *down, *sh_gate, *sh_up, *sh_down;
    int64_t mb2, mb3;  // bytes of one routed FP2 (I x H) and FP3 (H x I) matrix
    int H, I, E;
};

int make_layer_maps(const moe_layer& L, LayerMaps* m) {
    m->gate = L.gate; m->up = L.up; m->down = L.down;
    m->sh_gate = L.sh_gate; m->sh_up = L.sh_up; m->sh_down = L.sh_down;
    m->mb2 = matrix_bytes(2, L.I, L.H);
    m->mb3 = matrix_bytes(3, L.H, L.I);
    m->H = L.H; m->I = L.I; m->E = L.E;
    return FPX_OK;
}

// Byte offset of tile (row block of `row0`, column piece 0) of a box-tiled matrix with K columns.
__host__ __device__ constexpr int64_t tile_offset(int fmt, int row0, int K) {
    return (int64_t)(row0 / stage_rows(fmt)) * (K / stage_k(fmt)) * stage_bytes(fmt);
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

// ------------------------------------------------------------------ top-k + union

// Shared-memory routing state.
struct Route {
    int32_t idx[kMaxQ * kMaxK];
    float w[kMaxQ * kMaxK];
    int32_t uni[kMaxQ * kMaxK];
    int32_t slot[kMaxQ * kMaxK];  // where item j's matrices sit in the stacked arrays (see WsPtrs::uslot)
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

// ------------------------------------------------------------------ K1: router logits

// Computes the layer input u (bfloat16, in shared memory) and logits[t][e] for this CTA's 2 experts.
// MODE 0: input x is bfloat16. MODE 1: input is the residual r; u = RN_bf16(r / rms(r)) in one pass
// over r held in registers (q * ceil(H / 4096) <= kRouterV float4 groups per thread), and CTA 0
// publishes u (for the gate/up kernel) and r (the trace). 15 warps per expert, each a fifteenth of H;
// the slice sums are added in order; the last warp packs this CTA's slice of the gate/up activation
// tables meanwhile. With k > 0, the last CTA to finish routes every token (top-k,
// weights, union) and publishes the routing for the gate/up and down kernels.
constexpr int kRouterThreads = 1024;
constexpr int kRouterV = 8;  // q * ceil(H / 4096) <= 8: every q at H <= 4608 (the layer limit)

struct RouterArgs {
    const float* R;
    int E, H, q, k;  // k == 0: logits only
    const uint16_t* xin;
    const float* rin;
    float* logits;
    uint16_t* u_out;
    float* r_trace;
    int32_t* status_to_clear;
    WsPtrs ws;  // routing outputs and the arrival counter (k > 0)
    int32_t* idx_out;
    float* w_out;
    float* logits_out;
};

// Dynamic shared memory of the router: u [q][H] bfloat16, then two binary32 router rows.
inline size_t router_smem(int q, int H) { return sizeof(uint16_t) * (size_t)q * H + 2 * sizeof(float) * (size_t)H; }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// One warp packs this CTA's slice of the gate/up activation table set (4 token slots x H / 16 code
// groups; FP2, FP4 and block offsets) from u in shared memory. The slice has an even length, so the two
// groups of a block sit on lanes (2i, 2i + 1); absent tokens get zero entries.
__device__ __forceinline__ void pack_gate_up_slice(const uint16_t* u_s, const int* sh_s, uint8_t* gt, int H, int q) {
    const int lane = threadIdx.x & 31;
    const int ngr = 4 * H / 16, per = (((ngr + (int)gridDim.x - 1) / (int)gridDim.x) + 1) & ~1;
    const int gs = blockIdx.x * per;
    for (int gb = gs; gb < gs + per && gb < ngr; gb += 32) {
        const int gi = gb + lane;
        const bool valid = gi < ngr && gi < gs + per;
        const int tok = valid ? gi * 16 / H : 0, k0 = valid ? gi * 16 - tok * H : 0;
        float part = 0.f;
        if (valid) {
            float v[16];
#pragma unroll
            for (int j = 0; j < 16; j++) v[j] = tok < q ? __uint_as_float((uint32_t)u_s[(size_t)tok * H + k0 + j] << 16) : 0.f;
            part = pack_group<2>(gt, H, tok, k0, v, sh_s[tok]);
        }
        add_offsets<2>(gt, H, tok, k0, part, valid);
    }
}

template <int MODE>
__global__ void __launch_bounds__(kRouterThreads) k_router(const __grid_constant__ RouterArgs A) {
    const float* __restrict__ R = A.R;
    const int E = A.E, H = A.H, q = A.q;
    const uint16_t* __restrict__ xin = A.xin;
    const float* __restrict__ rin = A.rin;
    float* __restrict__ logits = A.logits;
    uint16_t* __restrict__ u_out = A.u_out;
    float* __restrict__ r_trace = A.r_trace;
    int32_t* status_to_clear = A.status_to_clear;
    extern __shared__ __align__(16) uint16_t u_s[];  // [q][H] bfloat16 bits, then this CTA's router rows
    __shared__ __align__(8) uint64_t rbar;
    __shared__ float red[kRouterThreads / 32][kMaxQ];
    __shared__ float redm[kRouterThreads / 32][kMaxQ];
    __shared__ float inv_s[kMaxQ];
    __shared__ int sh_s[kMaxQ];
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    // expert e = 2 * blockIdx + (warp >= kSlices): warps 0 .. kSlices - 1 and kSlices .. 2 kSlices - 1
    // each take a slice of the row's H / 4 float4 groups (the same slicing for both, so equal rows
    // give bit-equal logits); the last warp packs the gate/up tables meanwhile (k > 0). The router
    // weights do not depend on the previous kernel: one bulk copy stages this CTA's rows (adjacent in
    // R) in shared memory while the CTA waits.
    constexpr int kSlices = 15, kPackWarp = kRouterThreads / 32 - 1;
    const int e = blockIdx.x * 2 + (warp >= kSlices), sl = warp % kSlices;
    const bool dots = warp < 2 * kSlices;
    const int h4r = H / 4, g0 = h4r * sl / kSlices, g1 = dots ? h4r * (sl + 1) / kSlices : g0;
    float* w_s = reinterpret_cast<float*>(u_s + (size_t)q * H);  // q H * 2 bytes: a multiple of 32
    if (threadIdx.x == 0) {
        const uint32_t bytes = (uint32_t)(min(2, E - 2 * (int)blockIdx.x) * H) * 4u;
        mbar_init(&rbar, 1);
        fence_barrier_init();
        fence_proxy_async();
        mbar_expect_tx(&rbar, bytes);
        bulk_load_hint(w_s, R + (size_t)blockIdx.x * 2 * H, bytes, &rbar, l2_evict_first());
    }
    grid_dep_trigger();
    grid_dep_wait();  // r and the workspace come from the previous kernel
    if (status_to_clear && blockIdx.x == 0 && threadIdx.x == 0) *status_to_clear = 0;
    const int n4 = q * H / 4;  // groups of 4 consecutive elements (H % 16 == 0: never across tokens)
    // token of group idx (H / 4 groups per token), without a division
    auto tok_of = [h4r](int idx) { return (idx >= h4r) + (idx >= 2 * h4r) + (idx >= 3 * h4r); };
    // per-token maxima of |u| (the tables' column scales) and, MODE 1, sums of squares of r
    float ss[kMaxQ] = {0.f, 0.f, 0.f, 0.f}, mx[kMaxQ] = {0.f, 0.f, 0.f, 0.f};
    float4 rv[kRouterV];
    const int n_i = h4r > kRouterThreads ? 2 : 1;  // groups of a token per thread (H <= 8192)
    if (MODE == 0) {
        for (int i = threadIdx.x; i < n4; i += blockDim.x) {
            const uint2 pk = reinterpret_cast<const uint2*>(xin)[i];
            reinterpret_cast<uint2*>(u_s)[i] = pk;
            const float mm = fmaxf(fmaxf(fabsf(__uint_as_float(pk.x << 16)), fabsf(__uint_as_float(pk.x & 0xFFFF0000u))),
                                   fmaxf(fabsf(__uint_as_float(pk.y << 16)), fabsf(__uint_as_float(pk.y & 0xFFFF0000u))));
            const int t = tok_of(i);
#pragma unroll
            for (int tt = 0; tt < kMaxQ; tt++) mx[tt] = tt == t ? fmaxf(mx[tt], mm) : mx[tt];
        }
    } else {
        // thread x holds groups j = x + 1024 i (i < n_i) of every token, in slot t n_i + i: a token's
        // sum of squares runs through the same threads and the same reduction tree whatever q, so a
        // column normalises to the same bits alone or in a batch
        const float4* r4 = reinterpret_cast<const float4*>(rin);
#pragma unroll
        for (int sl = 0; sl < kRouterV; sl++) {
            const int t = n_i == 1 ? sl : sl >> 1, j = threadIdx.x + (sl - t * n_i) * kRouterThreads;
            rv[sl] = t < q && j < h4r ? r4[t * h4r + j] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int sl = 0; sl < kRouterV; sl++) {
            const int t = n_i == 1 ? sl : sl >> 1, j = threadIdx.x + (sl - t * n_i) * kRouterThreads;
            if (t < q && j < h4r) {
                float a = 0.f;
                a = fmaf(rv[sl].x, rv[sl].x, a); a = fmaf(rv[sl].y, rv[sl].y, a);
                a = fmaf(rv[sl].z, rv[sl].z, a); a = fmaf(rv[sl].w, rv[sl].w, a);
                const float mm = fmaxf(fmaxf(fabsf(rv[sl].x), fabsf(rv[sl].y)), fmaxf(fabsf(rv[sl].z), fabsf(rv[sl].w)));
#pragma unroll
                for (int tt = 0; tt < kMaxQ; tt++) {
                    ss[tt] += tt == t ? a : 0.f;
                    mx[tt] = tt == t ? fmaxf(mx[tt], mm) : mx[tt];
                }
            }
        }
    }
    // block reductions (fixed xor butterflies over lanes, then over warps)
#pragma unroll
    for (int tt = 0; tt < kMaxQ; tt++) {
        if (MODE == 1) ss[tt] = warp_sum(ss[tt]);
        mx[tt] = warp_max(mx[tt]);
    }
    if (lane == 0)
#pragma unroll
        for (int tt = 0; tt < kMaxQ; tt++) { red[warp][tt] = ss[tt]; redm[warp][tt] = mx[tt]; }
    __syncthreads();
    if (warp < kMaxQ) {  // warp tt reduces token tt's partials (the tokens in parallel)
        const int tt = warp;
        const float s = MODE == 1 ? warp_sum(red[lane][tt]) : 0.f, m = warp_max(redm[lane][tt]);
        if (lane == 0) {
            // max |u| = RN_bf16(max |r| * inv): rounding and scaling by inv > 0 are monotonic
            const float iv = MODE == 1 ? 1.0f / sqrtf(s / (float)H + 1e-6f) : 1.0f;
            const float mu = MODE == 1 ? __bfloat162float(__float2bfloat16_rn(m * iv)) : m;
            inv_s[tt] = iv;
            sh_s[tt] = column_shift(mu);
            if (A.k > 0 && blockIdx.x == 0) reinterpret_cast<int*>(A.ws.gt + tset_copy_bytes(H))[tt] = sh_s[tt];
        }
    }
    __syncthreads();
    if (MODE == 1) {
#pragma unroll
        for (int sl = 0; sl < kRouterV; sl++) {
            const int t = n_i == 1 ? sl : sl >> 1, j = threadIdx.x + (sl - t * n_i) * kRouterThreads, idx = t * h4r + j;
            if (t < q && j < h4r) {
                const float iv = inv_s[t];
                const __nv_bfloat162 lo = __floats2bfloat162_rn(rv[sl].x * iv, rv[sl].y * iv);
                const __nv_bfloat162 hi = __floats2bfloat162_rn(rv[sl].z * iv, rv[sl].w * iv);
                const uint2 pk = make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
                reinterpret_cast<uint2*>(u_s)[idx] = pk;
                if (blockIdx.x == 0) {
                    reinterpret_cast<uint2*>(u_out)[idx] = pk;
                    if (r_trace) reinterpret_cast<float4*>(r_trace)[idx] = rv[sl];
                }
            }
        }
        __syncthreads();
    }
    if (A.k > 0 && warp == kPackWarp) pack_gate_up_slice(u_s, sh_s, A.ws.gt, H, q);
    float acc[kMaxQ] = {0.f, 0.f, 0.f, 0.f};
    if (dots) {
        // the staged rows (a bounded wait; a lost copy leaves the logits at zero and flags a timeout)
        const bool ok = mbar_wait(&rbar, 0);
        if (!ok && lane == 0) flag(A.ws.status, FPX_ETIMEOUT);
        if (ok && e < E) {
            const float4* row = reinterpret_cast<const float4*>(w_s) + (size_t)(warp >= kSlices) * h4r;
            for (int h4 = g0 + lane; h4 < g1; h4 += 32) {  // ascending h4: the order of the sums
                const float4 wv = row[h4];
#pragma unroll
                for (int t = 0; t < kMaxQ; t++) {
                    if (t < q) {
                        const uint2 ub = reinterpret_cast<const uint2*>(u_s + (size_t)t * H)[h4];
                        acc[t] = fmaf(wv.x, __uint_as_float(ub.x << 16), acc[t]);
                        acc[t] = fmaf(wv.y, __uint_as_float(ub.x & 0xFFFF0000u), acc[t]);
                        acc[t] = fmaf(wv.z, __uint_as_float(ub.y << 16), acc[t]);
                        acc[t] = fmaf(wv.w, __uint_as_float(ub.y & 0xFFFF0000u), acc[t]);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int t = 0; t < kMaxQ; t++) acc[t] = warp_sum(acc[t]);
    if (lane == 0)
        for (int t = 0; t < q; t++) red[warp][t] = acc[t];
    __syncthreads();
    if (threadIdx.x < 2 * q) {
        const int el = threadIdx.x / q, t = threadIdx.x % q;
        const int ee = blockIdx.x * 2 + el;
        if (ee < E) {
            const int w0 = el * kSlices;
            float s = red[w0][t];
            for (int w = 1; w < kSlices; w++) s += red[w0 + w][t];
            logits[(size_t)t * E + ee] = s;
        }
    }
    if (A.k == 0) return;
    // The last CTA to finish routes every token. One thread counts the CTA in with an acquire-release
    // atomic: the barrier orders the CTA's logit stores before its release, and the last CTA's
    // acquire makes every CTA's logits visible to it (the barrier after it passes that on).
    __shared__ Route rt;
    __shared__ int last;
    __syncthreads();
    if (threadIdx.x == 0) {
        int old;
        asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(A.ws.nuni + 1) : "memory");
        last = old == (int)gridDim.x - 1;
    }
    __syncthreads();
    if (!last) return;  // CTA-uniform
    const int k = A.k;
    if (warp < q) warp_topk(logits + (size_t)warp * E, E, k, rt.idx + warp * k, rt.w + warp * k);
    build_union(rt, q, k, E);
    for (int i = threadIdx.x; i < q * k; i += blockDim.x) {
        A.ws.idx[i] = rt.idx[i];
        A.ws.w[i] = rt.w[i];
        A.ws.uni[i] = i < rt.n_uni ? rt.uni[i] : -1;
        A.ws.uslot[i] = i < rt.n_uni ? rt.uni[i] : -1;  // a two-tier call rewrites cold items (k_stage)
        if (A.idx_out) A.idx_out[i] = rt.idx[i];
        if (A.w_out) A.w_out[i] = rt.w[i];
    }
    if (A.logits_out)
        for (int i = threadIdx.x; i < q * E; i += blockDim.x) A.logits_out[i] = __ldcg(logits + i);
    if (threadIdx.x == 0) {
        A.ws.nuni[0] = rt.n_uni;
        A.ws.nuni[1] = 0;  // ready for the next call
    }
}

// ------------------------------------------------------------------ routing state

// Loads the routing the router kernel published (whole CTA; ends with __syncthreads()).
__device__ inline void load_route(Route& r, const WsPtrs& ws, int qk) {
    if (threadIdx.x == 0) r.n_uni = __ldcg(ws.nuni);
    for (int i = threadIdx.x; i < qk; i += blockDim.x) {
        r.idx[i] = __ldcg(ws.idx + i);
        r.w[i] = __ldcg(ws.w + i);
        r.uni[i] = __ldcg(ws.uni + i);
        r.slot[i] = __ldcg(ws.uslot + i);
    }
    __syncthreads();
}

// The units of a streaming kernel (one unit = one piece of one task): nA units of cost cA (the routed
// experts' tasks, in task order, pieces in order), then nB units of cost cB (the shared expert's). CTA b
// of G owns the units whose start cost c has floor(c G / total) == b: a contiguous range of about
// total / G, so every CTA streams about the same bytes whatever the union.
struct UnitList {
    // All products stay below 2^32 (checked on the host by fits): the partition needs only 32-bit
    // divisions.
    uint32_t nA, cA, nB, cB;
    __host__ __device__ __forceinline__ uint32_t units() const { return nA + nB; }
    __host__ __device__ __forceinline__ uint32_t total() const { return nA * cA + nB * cB; }
    // first unit of CTA b (b == G: units()): the smallest u with cost_before(u) * G >= total * b
    __host__ __device__ __forceinline__ uint32_t first(uint32_t b, uint32_t G) const {
        const uint32_t tgt = total() * b;
        if (tgt <= nA * cA * G) return (tgt + G * cA - 1) / (G * cA);
        return nA + (tgt - nA * cA * G + G * cB - 1) / (G * cB);
    }
    __host__ bool fits(uint32_t G) const { return (uint64_t)nA * cA + (uint64_t)nB * cB <= 0xFFFFFFFFull / (G + 1); }
};

// Relative time of a stage (in units of about 1 KB of a fast decode): bytes streamed for FP2 and FP3;
// FP4 boxes (17 KB) weighted for their slower decode, which the down kernel's FP3 stages outpace more.
constexpr uint32_t kCostFP2 = 20, kCostFP3 = 28, kCostFP4Gu = 23, kCostFP4Dn = 34;

__host__ __device__ constexpr uint32_t unit_cost(uint32_t c, int S, int D) {
    return (c * S + pieces_of(S, D) / 2) / pieces_of(S, D);
}

// Unit lists of the gate/up kernel (FP2 tasks: matrix x 256-row block, H/256 stages; FP4: matrix x
// 64-row block, H/512 stages) and of the down kernel (FP3: item x 256-row block, I/256 stages; FP4:
// 64-row block, I/512 stages).
__host__ __device__ inline UnitList gate_up_units(int n_uni, int H, int I) {
    const int sA = H / stage_k(2), sB = H / stage_k(4);
    return UnitList{2u * n_uni * (I / 256) * pieces_of(sA, kSppGu), unit_cost(kCostFP2, sA, kSppGu),
                    2u * (I / 64) * pieces_of(sB, kSppGu), unit_cost(kCostFP4Gu, sB, kSppGu)};
}
__host__ __device__ inline UnitList down_units(int n_uni, int H, int I) {
    const int sA = I / stage_k(3), sB = I / stage_k(4);
    return UnitList{(uint32_t)n_uni * (H / 256) * pieces_of(sA, kSppDn), unit_cost(kCostFP3, sA, kSppDn),
                    (uint32_t)(H / 64) * pieces_of(sB, kSppDn), unit_cost(kCostFP4Dn, sB, kSppDn)};
}

// ------------------------------------------------------------------ K2: gate/up

// Task = (output matrix, row block): the union's gate and up matrices (FP2, 256-row blocks of I,
// H/256 stages each), then the shared expert's gate and up (FP4, 64-row blocks, H/512 stages).
// Matrix m = 2 * item + (0 gate | 1 up), the shared expert being item n_uni. Each CTA owns a
// contiguous range of units (fixed pieces of tasks) of about equal cost (UnitList); its producer thread streams the
// range's boxes through the CTA ring and all consumer warps decode every box. Outputs g and u
// (binary32) go to ws.gu[piece][m][token][row]; k_hpack adds the pieces and forms h = silu(g) u.
struct GateUpArgs {
    LayerMaps m;
    int q, k;
    int G;  // grid size (the stage partition depends on it)
    const uint16_t* x;  // layer input, bfloat16 [q][H]
    WsPtrs ws;
    uint32_t magic;  // kMagic, kept out of immediates (see decode_fp2)
};

// Ring geometry of the two layer kernels: 7 slots of one FP2 box, 5 slots of one FP3 box (an FP4
// box, 17 KB, fits either). The down kernel holds four tables of I * 8 bytes; for I > 2048 it runs
// with a 2-slot ring so that they fit.
constexpr int kGuNS = 7;
using GuRing = CtaRing<kGuNS, stage_bytes(2)>;
template <int NS>
using DnRing = CtaRing<NS, stage_bytes(3)>;
static_assert(stage_bytes(4) <= stage_bytes(2), "FP4 box fits a slot");

// One unit of the gate/up kernel: a piece of a task, stages [s_beg, s_end) of the task.
struct GuTask {
    int mat;      // output matrix index
    int fp4;      // shared expert (FP4) task
    int row0;     // first output row
    int64_t off;  // byte offset of the task's first tile in its (stacked) matrix
    int piece, s_beg, s_end;
};

__device__ __forceinline__ GuTask gu_unit(uint32_t u, const Route& r, const LayerMaps& m) {
    const int I = m.I, rb2 = I / 256, sA = m.H / stage_k(2), pA = pieces_of(sA, kSppGu);
    const uint32_t nA = (uint32_t)(2 * r.n_uni * rb2 * pA);
    GuTask k;
    if (u < nA) {
        const int t = (int)u / pA;
        k.piece = (int)u - t * pA;
        k.mat = t / rb2;
        k.fp4 = 0;
        k.row0 = (t % rb2) * 256;
        k.off = r.slot[k.mat >> 1] * m.mb2 + tile_offset(2, k.row0, m.H);
        k.s_beg = piece_begin(sA, kSppGu, k.piece);
        k.s_end = piece_begin(sA, kSppGu, k.piece + 1);
    } else {
        const int sB = m.H / stage_k(4), pB = pieces_of(sB, kSppGu), rb4 = I / 64;
        const int t4 = (int)(u - nA) / pB;
        k.piece = (int)(u - nA) - t4 * pB;
        k.mat = 2 * r.n_uni + t4 / rb4;
        k.fp4 = 1;
        k.row0 = (t4 % rb4) * 64;
        k.off = tile_offset(4, k.row0, m.H);
        k.s_beg = piece_begin(sB, kSppGu, k.piece);
        k.s_end = piece_begin(sB, kSppGu, k.piece + 1);
    }
    return k;
}

__device__ __forceinline__ void gu_issue(const GateUpArgs& A, const GuTask& k, int s, uint8_t* slot, uint64_t* bar,
                                         uint64_t pol) {
    const int fmt = k.fp4 ? 4 : 2;
    const uint8_t* base = k.fp4 ? ((k.mat & 1) ? A.m.sh_up : A.m.sh_gate) : ((k.mat & 1) ? A.m.up : A.m.gate);
    mbar_expect_tx(bar, stage_bytes(fmt));
    bulk_load_hint(slot, base + k.off + (int64_t)s * stage_bytes(fmt), stage_bytes(fmt), bar, pol);
}

template <int Q>
__global__ void __launch_bounds__(kLThreads, 1) k_gate_up(const __grid_constant__ GateUpArgs A) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ Route r;
    __shared__ int shift[kMaxQ];
    const int H = A.m.H, I = A.m.I;
    const CtaSmem S = cta_carve(smem, GuRing::kBytes);
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const GuRing R = cta_init<kGuNS, stage_bytes(2)>(S);
    grid_dep_wait();     // routing and the activation tables come from the router kernel
    grid_dep_trigger();  // after the wait: the later kernels read the router's output before their own
    if (threadIdx.x == 0) {
        mbar_expect_tx(S.tbar, tset_copy_bytes(H));
        bulk_load(S.tabs, A.ws.gt, tset_copy_bytes(H), S.tbar);
    }
    load_route(r, A.ws, Q * A.k);

    const UnitList UL = gate_up_units(r.n_uni, H, I);
    const uint32_t G = A.G, u0 = UL.first(blockIdx.x, G), u1 = UL.first(blockIdx.x + 1, G);

    if (warp == kLWarps) {  // producer: streams the range's boxes while the consumers load the tables
        if (lane == 0) {
            uint32_t issued = 0;
            bool live = true;
            const uint64_t pol = l2_evict_first();
            // test hook: CTA 0 may withhold one copy (a lost message); its consumers' bounded waits
            // then run out and report FPX_ETIMEOUT
            const int32_t drop = blockIdx.x == 0 ? *reinterpret_cast<volatile int32_t*>(&g_ring_drop_stage) : -1;
            for (uint32_t u = u0; u < u1 && live; u++) {
                const GuTask k = gu_unit(u, r, A.m);
                for (int s = k.s_beg; s < k.s_end; s++, issued++) {
                    if (drop >= 0 && issued == (uint32_t)drop) { live = false; break; }
                    if (!R.acquire(issued)) { flag(A.ws.status, FPX_ETIMEOUT); live = false; break; }
                    gu_issue(A, k, s, R.slot(issued), R.bar(issued), pol);
                }
            }
            R.drain(issued);
        }
        return;
    }

    // activation tables (FP2 with block offsets, FP4), copied from the router kernel's table set
    if (threadIdx.x < kMaxQ) shift[threadIdx.x] = __ldcg(reinterpret_cast<const int*>(A.ws.gt + tset_copy_bytes(H)) + threadIdx.x);
    bool ok = __any_sync(0xffffffffu, mbar_wait(S.tbar, 0));
    if (!ok && lane == 0) flag(A.ws.status, FPX_ETIMEOUT);
    layer_sync();
    const uint2* tab2 = reinterpret_cast<const uint2*>(S.tabs);
    const uint2* tab4 = reinterpret_cast<const uint2*>(S.tabs + btab_bytes(H));
    const float* oq2 = reinterpret_cast<const float*>(S.tabs + 2 * btab_bytes(H));

    // Every consumer warp runs the same sequence of consumer barriers whether or not a wait timed
    // out, so a timeout never leaves a barrier short of arrivals.
    const int a_idx = b_active_index(lane);
    const uint32_t magic = A.magic;
    const LaneOfs L4 = lane_ofs<4>(t);
    const uint32_t tab2_lane = lane_tab(tab2, S.zero, a_idx, 0), tab2_step = a_idx >= 0 ? 4u * 512u : 0u;
    const uint32_t oq2_lane = lane_oq(oq2, 0, t);
    uint32_t bad = 0;
    typename decltype(R)::Pos pos{0u, 0u};
    constexpr int kFp4Ch = 8 / kFp4Parts;  // FP4 chunks per warp
    for (uint32_t u = u0; u < u1; u++) {
        const GuTask k = gu_unit(u, r, A.m);
        float y[kLTiles][4];
#pragma unroll
        for (int i = 0; i < kLTiles; i++) y[i][0] = y[i][1] = y[i][2] = y[i][3] = 0.f;
        if (!k.fp4) {
            const uint32_t s = (uint32_t)k.s_beg;
            frag_stages<2, kLTiles>(R, pos, k.s_end - k.s_beg, warp * 16 * kLTiles + g, t, tab2_lane + s * tab2_step, tab2_step,
                                    oq2_lane + s * 256u, magic, y, ok);
        } else {
            for (int s = k.s_beg; s < k.s_end; s++) {  // FP4 (shared expert) stages
                if (ok) ok = R.wait_at(pos);
                if (ok) {  // after a timeout the producer gives up too once this warp stops releasing
                    const int ch0 = s * box_chunks(4) + kFp4Ch * (warp >> 2);
                    box_tiles<4, 1, kFp4Ch>(R.slot_at(pos) + ((warp & 3) * 16 + g) * box_bytes(4) + kFp4Ch * (warp >> 2) * chunk_bytes(4),
                                            L4, lane_tab(tab4, S.zero, a_idx, ch0), 0u, 0u, magic,
                                            *reinterpret_cast<float(*)[1][4]>(&y[0]), bad);
                    R.release_at(pos);
                }
                R.next(pos);
            }
        }
#pragma unroll
        for (int i = 0; i < kLTiles; i++) pair_reduce(y[i]);
        if (k.fp4) fp4_reduce(S.red, y[0]);  // the same units run on every consumer warp
        if (ok && t < 2 && (!k.fp4 || warp < 4)) {
            const int rb = k.row0 + (k.fp4 ? 16 : 16 * kLTiles) * warp + g;
            float* out = A.ws.gu + (size_t)k.piece * A.ws.gu_piece + (size_t)k.mat * Q * I;
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const int tok = 2 * t + (i & 1), rr = rb + 8 * (i >> 1);
                if (tok < Q) {
                    // undo the per-token activation scale (and the 2^-14 of the FP4 decode)
                    const float sc = exp2i((k.fp4 ? 14 : 0) - shift[tok]);
                    out[(size_t)tok * I + rr] = y[0][i] * sc;
#pragma unroll
                    for (int ti = 1; ti < kLTiles; ti++)
                        if (!k.fp4) out[(size_t)tok * I + rr + 16 * ti] = y[ti][i] * sc;
                }
            }
        }
    }
    if (!ok && lane == 0) flag(A.ws.status, FPX_ETIMEOUT);
    report_bad(bad, A.ws.status);
}

// ------------------------------------------------------------------ K2b: h and the down tables

// One CTA per (union item or shared expert, token slot): h = silu(g) u over the item's I rows for the
// token (the pieces of g and u added in order first), its column shift, and that token's entries of
// the item's down activation table set (FP3 planes with block offsets; FP4 for the shared expert) in
// global memory. Token slots >= q get zero entries.
struct HpackArgs {
    int H, I, k;
    WsPtrs ws;
};

constexpr int kHpackThreads = 512;
constexpr int kHpackV = 3;  // float4 groups per thread, all loaded at once: I <= 3 * 4 * 512
static_assert(kHpackV * 4 * kHpackThreads >= 4608, "h buffer holds I <= 4608");

template <int Q>
__global__ void __launch_bounds__(kHpackThreads) k_hpack(const __grid_constant__ HpackArgs A) {
    __shared__ __align__(16) float h_s[kHpackV * 4 * kHpackThreads];  // [I]
    __shared__ float red[kHpackThreads / 32];
    __shared__ int sh_s;
    grid_dep_trigger();
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    const int I = A.I, j = blockIdx.x / 4, tok = blockIdx.x % 4;
    const int n_uni = __ldcg(A.ws.nuni);  // the router kernel's (completed before the gate/up kernel ran)
    if (j > n_uni) return;
    uint8_t* ts = A.ws.dt + (size_t)j * dset_bytes(I);
    float m = 0.f;
    if (tok < Q) {
        grid_dep_wait();  // g and u come from the gate/up kernel
        const float4* g = reinterpret_cast<const float4*>(A.ws.gu + ((size_t)(2 * j) * Q + tok) * I);
        const float4* u = reinterpret_cast<const float4*>(A.ws.gu + ((size_t)(2 * j + 1) * Q + tok) * I);
        const size_t pstride = A.ws.gu_piece / 4;
        // the fixed pieces of the item's gate and up tasks (routed: FP2, H/256 stages; shared: FP4,
        // H/512 stages), added in piece order
        const int np = pieces_of(j < n_uni ? A.H / stage_k(2) : A.H / stage_k(4), kSppGu);
        float4 ga[kHpackV], ua[kHpackV];
#pragma unroll
        for (int v = 0; v < kHpackV; v++) {
            const int e = threadIdx.x + v * kHpackThreads;
            const bool in = e < I / 4;
            float4 gp[kMaxPieces], up[kMaxPieces];
#pragma unroll
            for (int p = 0; p < kMaxPieces; p++) {
                gp[p] = in && p < np ? __ldcg(g + p * pstride + e) : make_float4(0.f, 0.f, 0.f, 0.f);
                up[p] = in && p < np ? __ldcg(u + p * pstride + e) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            ga[v] = gp[0]; ua[v] = up[0];
#pragma unroll
            for (int p = 1; p < kMaxPieces; p++) {
                if (p < np) {
                    ga[v].x += gp[p].x; ga[v].y += gp[p].y; ga[v].z += gp[p].z; ga[v].w += gp[p].w;
                    ua[v].x += up[p].x; ua[v].y += up[p].y; ua[v].z += up[p].z; ua[v].w += up[p].w;
                }
            }
        }
#pragma unroll
        for (int v = 0; v < kHpackV; v++) {
            const int e = threadIdx.x + v * kHpackThreads;
            if (e < I / 4) {
                const float a[4] = {ga[v].x, ga[v].y, ga[v].z, ga[v].w};
                const float b[4] = {ua[v].x, ua[v].y, ua[v].z, ua[v].w};
                float h[4];
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    h[i] = (a[i] / (1.0f + expf(-a[i]))) * b[i];
                    m = fmaxf(m, fabsf(h[i]));
                }
                reinterpret_cast<float4*>(h_s)[e] = make_float4(h[0], h[1], h[2], h[3]);
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) red[warp] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float mm = 0.f;
        for (int w = 0; w < kHpackThreads / 32; w++) mm = fmaxf(mm, red[w]);
        sh_s = column_shift(mm);
        reinterpret_cast<int*>(ts + dset_copy_bytes(I))[tok] = sh_s;
    }
    __syncthreads();
    // this token's I / 16 groups; the two groups of a block sit on lanes (2i, 2i + 1)
    const int ngr = I / 16;
    for (int gb = warp * 32; gb < ngr; gb += kHpackThreads) {
        const int gi = gb + lane;
        const bool valid = gi < ngr;
        const int k0 = valid ? gi * 16 : 0;
        float part = 0.f;
        if (valid) {
            float v[16];
#pragma unroll
            for (int q4 = 0; q4 < 4; q4++) {
                const float4 f = tok < Q ? reinterpret_cast<const float4*>(h_s + k0)[q4] : make_float4(0.f, 0.f, 0.f, 0.f);
                v[4 * q4] = f.x; v[4 * q4 + 1] = f.y; v[4 * q4 + 2] = f.z; v[4 * q4 + 3] = f.w;
            }
            part = j < n_uni ? pack_group<3>(ts, I, tok, k0, v, sh_s) : pack_group<4>(ts, I, tok, k0, v, sh_s);
        }
        if (j < n_uni) add_offsets<3>(ts, I, tok, k0, part, valid);  // CTA-uniform condition
    }
}

// ------------------------------------------------------------------ K3: down + combine

// Task = (item, row block of H): the union's down matrices (FP3, 256-row blocks, I/256 stages), then
// the shared expert's (FP4, 64-row blocks, I/512 stages). Each CTA owns a contiguous range of stages
// of units of about equal cost (UnitList), which spans at most two items; it copies their activation tables
// (built by k_hpack) at start. Outputs go to ws.yi[piece][item][token][row]; k_combine adds them up.
struct DownArgs {
    LayerMaps m;
    int q, k;
    int G;  // grid size (the stage partition depends on it)
    WsPtrs ws;
    float* out;  // MODE 0: y [q][H]; MODE 1: residual r [q][H], updated in place
    uint32_t magic;
};

// One unit of the down kernel: a piece of a task, stages [s_beg, s_end) of the task.
struct DnTask {
    int item, fp4, row0;
    int64_t off;  // byte offset of the task's first tile in its (stacked) matrix
    int piece, s_beg, s_end;
};

__device__ __forceinline__ DnTask dn_unit(uint32_t u, const Route& r, const LayerMaps& m) {
    const int H = m.H, rb3 = H / 256, sA = m.I / stage_k(3), pA = pieces_of(sA, kSppDn);
    const uint32_t nA = (uint32_t)(r.n_uni * rb3 * pA);
    DnTask k;
    if (u < nA) {
        const int t = (int)u / pA;
        k.piece = (int)u - t * pA;
        k.item = t / rb3;
        k.fp4 = 0;
        k.row0 = (t % rb3) * 256;
        k.off = r.slot[k.item] * m.mb3 + tile_offset(3, k.row0, m.I);
        k.s_beg = piece_begin(sA, kSppDn, k.piece);
        k.s_end = piece_begin(sA, kSppDn, k.piece + 1);
    } else {
        const int sB = m.I / stage_k(4), pB = pieces_of(sB, kSppDn);
        const int t4 = (int)(u - nA) / pB;
        k.piece = (int)(u - nA) - t4 * pB;
        k.item = r.n_uni;
        k.fp4 = 1;
        k.row0 = t4 * 64;
        k.off = tile_offset(4, k.row0, m.I);
        k.s_beg = piece_begin(sB, kSppDn, k.piece);
        k.s_end = piece_begin(sB, kSppDn, k.piece + 1);
    }
    return k;
}

__device__ __forceinline__ void dn_issue(const DownArgs& A, const DnTask& k, int s, uint8_t* slot, uint64_t* bar,
                                         uint64_t pol) {
    const int fmt = k.fp4 ? 4 : 3;
    mbar_expect_tx(bar, stage_bytes(fmt));
    bulk_load_hint(slot, (k.fp4 ? A.m.sh_down : A.m.down) + k.off + (int64_t)s * stage_bytes(fmt), stage_bytes(fmt), bar, pol);
}

template <int Q, int MODE, int NS>
__global__ void __launch_bounds__(kLThreads, 1) k_down(const __grid_constant__ DownArgs A) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ Route r;
    __shared__ int shift[2][kMaxQ];
    const int H = A.m.H, I = A.m.I;
    const CtaSmem S = cta_carve(smem, DnRing<NS>::kBytes);
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const DnRing<NS> R = cta_init<NS, stage_bytes(3)>(S);
    // the routing comes from the router kernel, which completed before the gate/up kernel passed its
    // own grid_dep_wait(); the weights do not depend on the kernels in between either, so the producer
    // starts streaming before grid_dep_wait()
    grid_dep_trigger();
    load_route(r, A.ws, Q * A.k);

    const UnitList UL = down_units(r.n_uni, H, I);
    const uint32_t G = A.G, u0 = UL.first(blockIdx.x, G), u1 = UL.first(blockIdx.x + 1, G);
    if (u0 >= u1) return;  // CTA-uniform: nothing to do
    const int item_lo = dn_unit(u0, r, A.m).item, item_hi = dn_unit(u1 - 1, r, A.m).item;
    if (item_hi - item_lo > 1) {  // cannot happen for the grids make_plan picks (each share < one item)
        if (threadIdx.x == 0) flag(A.ws.status, FPX_EINVAL);
        return;
    }

    if (warp == kLWarps) {  // producer: streams the range's boxes while the consumers load the tables
        if (lane == 0) {
            uint32_t issued = 0;
            bool live = true;
            const uint64_t pol = l2_evict_first();
            for (uint32_t u = u0; u < u1 && live; u++) {
                const DnTask k = dn_unit(u, r, A.m);
                for (int s = k.s_beg; s < k.s_end; s++, issued++) {
                    if (!R.acquire(issued)) { flag(A.ws.status, FPX_ETIMEOUT); live = false; break; }
                    dn_issue(A, k, s, R.slot(issued), R.bar(issued), pol);
                }
            }
            R.drain(issued);
        }
        return;
    }

    // activation tables of the (at most two) items of this CTA's range, built by k_hpack
    grid_dep_wait();
    const int nit = item_hi - item_lo + 1;
    if (threadIdx.x == 0) {
        mbar_expect_tx(S.tbar, nit * dset_copy_bytes(I));
        for (int sl = 0; sl < nit; sl++)
            bulk_load(S.tabs + (size_t)sl * dset_copy_bytes(I), A.ws.dt + (size_t)(item_lo + sl) * dset_bytes(I), dset_copy_bytes(I),
                      S.tbar);
    }
    if (threadIdx.x < 2 * kMaxQ) {
        const int sl = threadIdx.x / kMaxQ, tk = threadIdx.x % kMaxQ;
        shift[sl][tk] = sl < nit ? __ldcg(reinterpret_cast<const int*>(A.ws.dt + (size_t)(item_lo + sl) * dset_bytes(I) + dset_copy_bytes(I)) + tk) : 0;
    }
    bool ok = __any_sync(0xffffffffu, mbar_wait(S.tbar, 0));
    if (!ok && lane == 0) flag(A.ws.status, FPX_ETIMEOUT);
    layer_sync();

    // Every consumer warp runs the same sequence of consumer barriers whether or not a wait timed
    // out, so a timeout never leaves a barrier short of arrivals.
    const int a_idx = b_active_index(lane);
    const uint32_t magic = A.magic;
    const LaneOfs L4 = lane_ofs<4>(t);
    uint32_t bad = 0;
    typename decltype(R)::Pos pos{0u, 0u};
    constexpr int kFp4Ch = 8 / kFp4Parts;  // FP4 chunks per warp
    for (uint32_t u = u0; u < u1; u++) {
        const DnTask k = dn_unit(u, r, A.m);
        const int sl = k.item - item_lo;
        const uint8_t* ts = S.tabs + (size_t)sl * dset_copy_bytes(I);
        const uint2* tab = reinterpret_cast<const uint2*>(ts);
        const float* oq = reinterpret_cast<const float*>(ts + btab_bytes(I));
        float y[kLTiles][4];
#pragma unroll
        for (int i = 0; i < kLTiles; i++) y[i][0] = y[i][1] = y[i][2] = y[i][3] = 0.f;
        if (!k.fp4) {
            const uint32_t s = (uint32_t)k.s_beg, b_step = a_idx >= 0 ? 4u * 512u : 0u;
            frag_stages<3, kLTiles>(R, pos, k.s_end - k.s_beg, warp * 16 * kLTiles + g, t, lane_tab(tab, S.zero, a_idx, 0) + s * b_step,
                                    b_step, lane_oq(oq, 0, t) + s * 256u, magic, y, ok);
        } else {
            for (int s = k.s_beg; s < k.s_end; s++) {  // FP4 (shared expert) stages
                if (ok) ok = R.wait_at(pos);
                if (ok) {
                    const int ch0 = s * box_chunks(4) + kFp4Ch * (warp >> 2);
                    box_tiles<4, 1, kFp4Ch>(R.slot_at(pos) + ((warp & 3) * 16 + g) * box_bytes(4) + kFp4Ch * (warp >> 2) * chunk_bytes(4),
                                            L4, lane_tab(tab, S.zero, a_idx, ch0), 0u, 0u, magic,
                                            *reinterpret_cast<float(*)[1][4]>(&y[0]), bad);
                    R.release_at(pos);
                }
                R.next(pos);
            }
        }
#pragma unroll
        for (int i = 0; i < kLTiles; i++) pair_reduce(y[i]);
        if (k.fp4) fp4_reduce(S.red, y[0]);
        if (ok && t < 2 && (!k.fp4 || warp < 4)) {
            const int rb = k.row0 + (k.fp4 ? 16 : 16 * kLTiles) * warp + g;
            float* out = A.ws.yi + (size_t)k.piece * A.ws.yi_piece + (size_t)k.item * Q * H;
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const int tok = 2 * t + (i & 1), rr = rb + 8 * (i >> 1);
                if (tok < Q) {
                    const float sc = exp2i((k.fp4 ? 14 : 0) - shift[sl][tok]);
                    out[(size_t)tok * H + rr] = y[0][i] * sc;
#pragma unroll
                    for (int ti = 1; ti < kLTiles; ti++)
                        if (!k.fp4) out[(size_t)tok * H + rr + 16 * ti] = y[ti][i] * sc;
                }
            }
        }
    }
    if (!ok && lane == 0) flag(A.ws.status, FPX_ETIMEOUT);
    report_bad(bad, A.ws.status);
}

// ------------------------------------------------------------------ K4: combine

// out[t][h] (MODE 0) or r[t][h] += (MODE 1) sum over token t's selected experts, in ascending expert
// order, of w * y_e[t][h] (pieces added in order first), then the shared expert's y[t][h]. One thread per
// output; consecutive threads take consecutive rows. Only the token's k items and the shared one are
// loaded, all at once.
struct CombineArgs {
    int H, I, k;
    WsPtrs ws;
    float* out;  // MODE 0: y [q][H]; MODE 1: residual r [q][H], updated in place
};

constexpr int kCombineThreads = 256;
constexpr int kKernelsPerLayer = 5;  // router, gate/up, h + down tables, down, combine

template <int Q, int MODE>
__global__ void __launch_bounds__(kCombineThreads) k_combine(const __grid_constant__ CombineArgs A) {
    __shared__ Route r;
    __shared__ int sel[kMaxQ][kMaxK];     // union index of token t's selected experts, ascending
    __shared__ float selw[kMaxQ][kMaxK];  // their weights
    grid_dep_trigger();
    load_route(r, A.ws, Q * A.k);  // from the router kernel (completed two launches ago)
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    if (warp < Q) {  // warp t: the union items token t selected (each selected once), in union order
        const int tok = warp;
        float wv = 0.f;
        bool on = false;
        if (lane < r.n_uni)
            for (int rr = 0; rr < A.k; rr++)
                if (r.idx[tok * A.k + rr] == r.uni[lane]) { on = true; wv = r.w[tok * A.k + rr]; }
        const uint32_t m = __ballot_sync(0xffffffffu, on);
        if (on) {
            const int pos = __popc(m & ((1u << lane) - 1u));
            sel[tok][pos] = lane;
            selw[tok][pos] = wv;
        }
    }
    // the fixed pieces of the routed (FP3, I/256 stages) and shared (FP4, I/512 stages) down tasks
    const int H = A.H, np_r = pieces_of(A.I / stage_k(3), kSppDn), np_s = pieces_of(A.I / stage_k(4), kSppDn);
    __syncthreads();
    grid_dep_wait();  // the down kernel's outputs
    const int o = blockIdx.x * kCombineThreads + threadIdx.x;
    if (o >= Q * H) return;
    const int tok = o / H, rr = o % H, k = A.k;
    const float* col = A.ws.yi + (size_t)tok * H + rr;
    const size_t istride = (size_t)Q * H;
    float pv[kMaxK][kMaxPieces], ps[kMaxPieces];
#pragma unroll
    for (int i = 0; i < kMaxK; i++) {
        const size_t jo = (size_t)(i < k ? sel[tok][i] : 0) * istride;
#pragma unroll
        for (int p = 0; p < kMaxPieces; p++) pv[i][p] = i < k && p < np_r ? __ldcg(col + p * A.ws.yi_piece + jo) : 0.0f;
    }
#pragma unroll
    for (int p = 0; p < kMaxPieces; p++)
        ps[p] = p < np_s ? __ldcg(col + p * A.ws.yi_piece + (size_t)r.n_uni * istride) : 0.0f;
    // the fixed-order sum: pieces of an item in order, items in ascending expert order, shared last
    float acc = 0.0f;
#pragma unroll
    for (int i = 0; i < kMaxK; i++) {
        if (i < k) {
            float yv = pv[i][0];
#pragma unroll
            for (int p = 1; p < kMaxPieces; p++)
                if (p < np_r) yv += pv[i][p];
            acc = i == 0 ? selw[tok][i] * yv : fmaf(selw[tok][i], yv, acc);
        }
    }
    float ysh = ps[0];
#pragma unroll
    for (int p = 1; p < kMaxPieces; p++)
        if (p < np_s) ysh += ps[p];
    acc += ysh;
    if (MODE == 0) A.out[o] = acc;
    else A.out[o] = A.out[o] + acc;
}

// ------------------------------------------------------------------ launch plumbing

int check_layer(const moe_layer* L) {
    // H, I <= 4608: the fixed piece arrays (kMaxPieces), the router's registers and k_hpack's buffer
    if (!L || L->H < 512 || L->I < 512 || L->H % 512 || L->I % 512 || L->H > 4608 || L->I > 4608 || L->E < 1 ||
        L->E > kMaxE)
        return FPX_EINVAL;
    if (!L->router || !L->gate || !L->up || !L->down || !L->sh_gate || !L->sh_up || !L->sh_down) return FPX_EINVAL;
    if (!aligned(L->router, 16) || !aligned(L->gate, 16) || !aligned(L->up, 16) || !aligned(L->down, 16) ||
        !aligned(L->sh_gate, 16) || !aligned(L->sh_up, 16) || !aligned(L->sh_down, 16))
        return FPX_EALIGN;
    // shared memory (plus up to 2 KB of static): gate/up ring + one table set for K = H; down ring
    // (2 slots at least) + two table sets for K = I
    if (cta_smem_bytes(GuRing::kBytes, tset_copy_bytes(L->H)) + 2048 > 227 * 1024 ||
        cta_smem_bytes(DnRing<2>::kBytes, 2 * dset_copy_bytes(L->I)) + 2048 > 227 * 1024)
        return FPX_EINVAL;
    // the stage partitions' 32-bit arithmetic, for the largest union and grid
    const int nmax = kMaxQ * kMaxK < L->E ? kMaxQ * kMaxK : L->E;
    if (!gate_up_units(nmax, L->H, L->I).fits(1024) || !down_units(nmax, L->H, L->I).fits(1024)) return FPX_EINVAL;
    return FPX_OK;
}

struct Plan {
    int g_router, g_gate, g_down, g_comb, ns_down;  // g_gate, g_down: grids of the stage partitions
    size_t sm_router, sm_gate, sm_down;
};

Plan make_plan(const moe_layer& L, int q, int k) {
    DeviceInfo di = device_info();
    Plan p{};
    p.g_router = (L.E + 1) / 2;
    p.sm_router = router_smem(q, L.H);
    // one CTA per SM, but no more CTAs than the units of the smallest union (k experts), so that a
    // CTA's share stays below one routed item's units (the down kernel holds the tables of two items)
    auto grid_for = [&](const UnitList& U) { return (int)(U.units() < (uint32_t)di.sms ? U.units() : (uint32_t)di.sms); };
    p.g_gate = grid_for(gate_up_units(k, L.H, L.I));
    p.sm_gate = cta_smem_bytes(GuRing::kBytes, tset_copy_bytes(L.H));
    p.g_down = grid_for(down_units(k, L.H, L.I));
    p.ns_down = cta_smem_bytes(DnRing<5>::kBytes, 2 * dset_copy_bytes(L.I)) + 2048 <= 227 * 1024 ? 5 : 2;
    p.sm_down = cta_smem_bytes(p.ns_down == 5 ? DnRing<5>::kBytes : DnRing<2>::kBytes, 2 * dset_copy_bytes(L.I));
    p.g_comb = (q * L.H + kCombineThreads - 1) / kCombineThreads;
    return p;
}

// ------------------------------------------------------------------ two-tier residency
//
// A two-tier layer keeps the hot experts' matrices in HBM slots and the others (the cold tier) in
// pinned host memory ("Token Freedom via APU ...", section "Asymmetric Dual-GPU": popular experts in
// the fast memory, cold ones in the large pool; the Paiton page on DeepSeek V4.1 Flash, section
// "Keeping useful work on the GPU": cold experts streamed to the GPU when that pays). After routing,
// k_stage_plan gives every cold expert of the union a staging slot and lists the copies; k_stage
// copies their gate, up and down matrices from host memory into those slots (reads over the host
// link, 16 bytes per thread per load) and the union's slot list is rewritten; the gate/up and down
// kernels then stream every item from HBM as usual, and the combine still matches tokens to items by
// expert id, so the result is bit-identical to a layer whose experts are all in HBM.
//
// With a cache (moe_tiers.cache) the staging slots keep their experts across calls: a cold expert
// already in a slot is not copied again, and a missing one takes the least recently used slot that
// this call does not use. The host link moves about 51 GB/s against the HBM's 6.5 TB/s, so the copies
// dominate a call; not copying is what shortens it.

constexpr int kMaxStageCache = 1024;  // staging slots a cache can track

struct StageArgs {
    const int32_t* slot_of;               // [E]: HBM slot of expert e, or < 0 for the cold tier
    const uint8_t *cgate, *cup, *cdown;   // cold tier: all E experts, stacked (device view of host memory)
    uint8_t *gate, *up, *down;            // the layer's HBM slot arrays
    int64_t mb2, mb3;
    int E, n_slots, stage0, n_stage, qk;
    int32_t* cache;  // nullable: [clock, copies so far, expert of staging slot i (n_stage), last use of slot i (n_stage)]
    WsPtrs ws;
};

// One warp: the staging slot of every cold item of the union and the list of copies (ws.stage), in
// union order (ascending expert). Without a cache the i-th cold item takes staging slot i and is
// copied. With one: a slot that holds the expert is used as it is; otherwise the slot with the
// oldest last use among those this call has not taken (ties to the lower slot) receives it.
__global__ void __launch_bounds__(32) k_stage_plan(const __grid_constant__ StageArgs A) {
    grid_dep_trigger();  // the copy kernel waits for this grid before it reads the list
    grid_dep_wait();     // the union comes from the router kernel
    __shared__ int32_t cexp[kMaxStageCache], cuse[kMaxStageCache];
    __shared__ uint32_t taken[kMaxStageCache / 32];
    const int lane = threadIdx.x;
    const int n = min(__ldcg(A.ws.nuni), A.qk);
    const bool cached = A.cache != nullptr;
    const int ns = A.n_stage;
    const uint32_t clock = cached ? (uint32_t)__ldcg(A.cache) + 1u : 0u;
    // item `lane`: its expert and HBM slot (a slot outside the arrays or inside the staging range
    // cannot hold a hot expert: the expert is treated as cold and the status reports it)
    int e_l = -1, sl_l = -1;
    bool bad = false;
    if (lane < n) {
        e_l = __ldcg(A.ws.uni + lane);
        sl_l = e_l >= 0 && e_l < A.E ? A.slot_of[e_l] : -1;
        if (sl_l >= A.n_slots || (sl_l >= A.stage0 && sl_l < A.stage0 + ns)) {
            bad = true;
            sl_l = -1;
        }
    }
    if (cached) {
        for (int i = lane; i < ns; i += 32) {
            cexp[i] = __ldcg(A.cache + 2 + i);
            cuse[i] = __ldcg(A.cache + 2 + ns + i);
        }
        for (int i = lane; i < kMaxStageCache / 32; i += 32) taken[i] = 0u;
    }
    __syncwarp();
    int ncold = 0, ncopy = 0;
    for (int j = 0; j < n; j++) {
        const int e = __shfl_sync(0xffffffffu, e_l, j);
        int sl = __shfl_sync(0xffffffffu, sl_l, j);
        if (sl < 0 && e >= 0 && e < A.E) {
            int i = ncold;
            bool copy = true;
            if (cached) {
                int hit = -1;
                for (int b = 0; b < ns && hit < 0; b += 32) {
                    const uint32_t m = __ballot_sync(0xffffffffu, b + lane < ns && cexp[b + lane] == e);
                    if (m) hit = b + __ffs(m) - 1;
                }
                if (hit >= 0) {
                    i = hit;
                    copy = false;
                } else {  // oldest last use (as a distance back from this call's clock), lower slot on ties
                    uint64_t best = ~0ull;
                    for (int s2 = lane; s2 < ns; s2 += 32)
                        if (!((taken[s2 >> 5] >> (s2 & 31)) & 1u)) {
                            const uint64_t key = ((uint64_t)(0xFFFFFFFFu - (clock - (uint32_t)cuse[s2])) << 32) | (uint32_t)s2;
                            best = key < best ? key : best;
                        }
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        const uint64_t ob = __shfl_xor_sync(0xffffffffu, best, o);
                        best = ob < best ? ob : best;
                    }
                    i = (int)(best & 0xFFFFFFFFu);  // n_stage >= q k: a free slot always exists
                }
                if (lane == 0) {
                    cexp[i] = e;
                    cuse[i] = (int32_t)clock;
                    taken[i >> 5] |= 1u << (i & 31);
                }
                __syncwarp();
            }
            sl = A.stage0 + i;
            if (copy && lane == 0) {
                A.ws.stage[1 + ncopy] = e;
                A.ws.stage[1 + A.qk + ncopy] = sl;
            }
            ncopy += copy;
            ncold++;
        }
        if (lane == 0) A.ws.uslot[j] = sl;
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) flag(A.ws.status, FPX_EDATA);
    if (lane == 0) A.ws.stage[0] = ncopy;
    if (cached) {
        for (int i = lane; i < ns; i += 32) {
            A.cache[2 + i] = cexp[i];
            A.cache[2 + ns + i] = cuse[i];
        }
        if (lane == 0) {
            A.cache[0] = (int32_t)clock;
            A.cache[1] += ncopy;
        }
    }
}

constexpr int kStageThreads = 256;

// Copies the listed cold experts (gate, up and down matrices) from the host tier into their slots.
__global__ void __launch_bounds__(kStageThreads) k_stage(const __grid_constant__ StageArgs A) {
    grid_dep_trigger();  // the gate/up kernel waits for this grid before it reads the slots or weights
    grid_dep_wait();     // the list comes from k_stage_plan
    __shared__ int32_t src[kMaxQ * kMaxK], dst[kMaxQ * kMaxK];
    __shared__ int ncopy;
    if (threadIdx.x == 0) ncopy = min(__ldcg(A.ws.stage), A.qk);
    if (threadIdx.x < A.qk) {
        src[threadIdx.x] = __ldcg(A.ws.stage + 1 + threadIdx.x);
        dst[threadIdx.x] = __ldcg(A.ws.stage + 1 + A.qk + threadIdx.x);
    }
    __syncthreads();
    // copy the cold items: per item gate (mb2), up (mb2), down (mb3) bytes, in 16-byte units
    const int64_t u2 = A.mb2 / 16, u3 = A.mb3 / 16, per = 2 * u2 + u3;
    const int64_t total = per * ncopy;
    const int64_t stride = (int64_t)gridDim.x * kStageThreads;
    int64_t u = (int64_t)blockIdx.x * kStageThreads + threadIdx.x;
    auto addr = [&](int64_t v, const uint4*& from, uint4*& to) {
        const int it = (int)(v / per);
        int64_t r = v - (int64_t)it * per;
        const int64_t e = src[it], sl = dst[it];
        if (r < u2) {
            from = reinterpret_cast<const uint4*>(A.cgate + e * A.mb2) + r;
            to = reinterpret_cast<uint4*>(A.gate + sl * A.mb2) + r;
        } else if (r < 2 * u2) {
            r -= u2;
            from = reinterpret_cast<const uint4*>(A.cup + e * A.mb2) + r;
            to = reinterpret_cast<uint4*>(A.up + sl * A.mb2) + r;
        } else {
            r -= 2 * u2;
            from = reinterpret_cast<const uint4*>(A.cdown + e * A.mb3) + r;
            to = reinterpret_cast<uint4*>(A.down + sl * A.mb3) + r;
        }
    };
    // four loads in flight per thread before their stores
    for (; u + 3 * stride < total; u += 4 * stride) {
        const uint4 *f0, *f1, *f2, *f3;
        uint4 *t0, *t1, *t2, *t3;
        addr(u, f0, t0);
        addr(u + stride, f1, t1);
        addr(u + 2 * stride, f2, t2);
        addr(u + 3 * stride, f3, t3);
        const uint4 v0 = *f0, v1 = *f1, v2 = *f2, v3 = *f3;
        *t0 = v0;
        *t1 = v1;
        *t2 = v2;
        *t3 = v3;
    }
    for (; u < total; u += stride) {
        const uint4* f;
        uint4* t;
        addr(u, f, t);
        *t = *f;
    }
}

// Launches kern<<<grid, block, smem, s>>>(args), as a programmatic dependent launch when pdl is set
// (the kernel calls grid_dep_wait() before reading what the previous kernel wrote).
template <typename Args>
cudaError_t launch(void (*kern)(Args), int grid, int block, size_t smem, cudaStream_t s, bool pdl, const Args& args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args);
}

template <int Q, int MODE>
int launch_layer(const moe_layer& L, const Plan& p, int k, const uint16_t* x, const float* r, float* out,
                 int32_t* idx_out, float* w_out, float* logits_out, float* r_trace, WsPtrs ws, bool clear,
                 cudaEvent_t const* ev, bool pdl_first, cudaStream_t s, const StageArgs* tier = nullptr) {
    if (MODE == 1 && Q * ((L.H / 4 + kRouterThreads - 1) / kRouterThreads) > kRouterV) return FPX_EINVAL;  // router registers
    GateUpArgs ga{};
    DownArgs da{};
    int st = make_layer_maps(L, &ga.m);
    if (st) return st;
    da.m = ga.m;
    ga.q = da.q = Q;
    ga.k = da.k = k;
    ga.G = p.g_gate;
    da.G = p.g_down;
    ga.x = MODE == 0 ? x : ws.u;
    ga.ws = da.ws = ws;
    ga.magic = da.magic = kMagic;
    da.out = out;
    RouterArgs ra{};
    ra.R = L.router;
    ra.E = L.E; ra.H = L.H; ra.q = Q; ra.k = k;
    ra.xin = x; ra.rin = r;
    ra.logits = ws.logits; ra.u_out = ws.u; ra.r_trace = r_trace;
    ra.status_to_clear = clear ? ws.status : nullptr;
    ra.ws = ws;
    ra.idx_out = idx_out; ra.w_out = w_out; ra.logits_out = logits_out;
    auto kdown = p.ns_down == 5 ? k_down<Q, MODE, 5> : k_down<Q, MODE, 2>;
    HpackArgs ha{};
    ha.H = L.H; ha.I = L.I; ha.k = k; ha.ws = ws;
    if (cudaFuncSetAttribute(k_router<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.sm_router) ||
        cudaFuncSetAttribute(k_gate_up<Q>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.sm_gate) ||
        cudaFuncSetAttribute(kdown, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.sm_down))
        return FPX_ECUDA;
    CombineArgs ca{};
    ca.H = L.H; ca.I = L.I; ca.k = k; ca.ws = ws; ca.out = out;
    // timing events between the kernels would break the dependent-launch edges: no overlap then
    const bool pdl = ev == nullptr;
    cudaError_t e = cudaSuccess;
    if (ev) cudaEventRecord(ev[0], s);
    e = e ? e : launch(k_router<MODE>, p.g_router, kRouterThreads, p.sm_router, s, pdl && pdl_first, ra);
    if (tier) {
        StageArgs sa = *tier;
        sa.ws = ws;
        e = e ? e : launch(k_stage_plan, 1, 32, 0, s, pdl, sa);
        e = e ? e : launch(k_stage, 4 * device_info().sms, kStageThreads, 0, s, pdl, sa);
    }
    if (ev) cudaEventRecord(ev[1], s);
    e = e ? e : launch(k_gate_up<Q>, p.g_gate, kLThreads, p.sm_gate, s, pdl, ga);
    if (ev) cudaEventRecord(ev[2], s);
    e = e ? e : launch(k_hpack<Q>, 4 * (Q * k + 1), kHpackThreads, 0, s, pdl, ha);
    if (ev) cudaEventRecord(ev[3], s);
    e = e ? e : launch(kdown, p.g_down, kLThreads, p.sm_down, s, pdl, da);
    if (ev) cudaEventRecord(ev[4], s);
    e = e ? e : launch(k_combine<Q, MODE>, p.g_comb, kCombineThreads, 0, s, pdl, ca);
    return e == cudaSuccess ? launch_status() : FPX_ECUDA;
}

template <int MODE>
int dispatch_q(int q, const moe_layer& L, const Plan& p, int k, const uint16_t* x, const float* r, float* out,
               int32_t* idx_out, float* w_out, float* logits_out, float* r_trace, WsPtrs ws, bool clear,
               cudaEvent_t const* ev, bool pdl_first, cudaStream_t s, const StageArgs* tier = nullptr) {
    switch (q) {
        case 1: return launch_layer<1, MODE>(L, p, k, x, r, out, idx_out, w_out, logits_out, r_trace, ws, clear, ev, pdl_first, s, tier);
        case 2: return launch_layer<2, MODE>(L, p, k, x, r, out, idx_out, w_out, logits_out, r_trace, ws, clear, ev, pdl_first, s, tier);
        case 3: return launch_layer<3, MODE>(L, p, k, x, r, out, idx_out, w_out, logits_out, r_trace, ws, clear, ev, pdl_first, s, tier);
        case 4: return launch_layer<4, MODE>(L, p, k, x, r, out, idx_out, w_out, logits_out, r_trace, ws, clear, ev, pdl_first, s, tier);
        default: return FPX_EINVAL;
    }
}

}  // namespace

extern "C" {

int moe_route_topk(const float* R, int E, int H, const uint16_t* x, int q, int k, float* logits, int32_t* idx, float* w,
                   int32_t* uni, int32_t* n_uni, void* stream) {
    if (E < 1 || E > kMaxE || H < 16 || H % 16 || q < 1 || q > kMaxQ || k < 1 || k > kMaxK || k > E) return FPX_EINVAL;
    if (!R || !x || !logits || !idx || !w || !uni || !n_uni) return FPX_EINVAL;
    if (!aligned(R, 16) || !aligned(x, 8) || !aligned(logits, 4)) return FPX_EALIGN;  // x read in 8-byte units
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t sm = router_smem(q, H);
    if (sm > (size_t)device_info().smem_optin) return FPX_EINVAL;
    if (cudaFuncSetAttribute(k_router<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm)) return FPX_ECUDA;
    RouterArgs ra{};
    ra.R = R;
    ra.E = E; ra.H = H; ra.q = q; ra.k = 0;  // logits only; k_topk routes
    ra.xin = x; ra.logits = logits;
    k_router<0><<<(E + 1) / 2, kRouterThreads, sm, s>>>(ra);
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
    if (!aligned(ws, 16) || !aligned(x, 8) || !aligned(y, 4)) return FPX_EALIGN;  // the router reads x in 8-byte units
    Ws wl = ws_layout(layer->H, layer->I, layer->E, q, k);
    if (ws_bytes < wl.total) return FPX_ESPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    WsPtrs wp = ws_ptrs(ws, wl);
    // the router's arrival counter must start at zero; the router leaves it at zero
    if (cudaMemsetAsync(wp.nuni, 0, 16, s) != cudaSuccess) return FPX_ECUDA;
    Plan p = make_plan(*layer, q, k);
    return dispatch_q<0>(q, *layer, p, k, x, nullptr, y, idx_out, w_out, logits_out, nullptr, wp, true, nullptr, false, s);
}

int moe_layer_decode_tiered(const moe_layer* layer, const moe_tiers* tiers, const uint16_t* x, int q, int k, float* y,
                            int32_t* idx_out, float* w_out, float* logits_out, void* ws, size_t ws_bytes, void* stream) {
    int st = check_layer(layer);
    if (st) return st;
    if (!tiers || q < 1 || q > kMaxQ || k < 1 || k > kMaxK || k > layer->E || !x || !y || !ws) return FPX_EINVAL;
    if (!tiers->slot_of || !tiers->cold_gate || !tiers->cold_up || !tiers->cold_down) return FPX_EINVAL;
    const int need = q * k < layer->E ? q * k : layer->E;  // the largest union
    if (tiers->n_slots < 1 || tiers->stage_slot0 < 0 || tiers->n_stage < need ||
        (int64_t)tiers->stage_slot0 + tiers->n_stage > tiers->n_slots || (tiers->cache && tiers->n_stage > kMaxStageCache))
        return FPX_EINVAL;
    if (!aligned(ws, 16) || !aligned(x, 8) || !aligned(y, 4) || !aligned(tiers->slot_of, 4) || !aligned(tiers->cache, 4))
        return FPX_EALIGN;
    Ws wl = ws_layout(layer->H, layer->I, layer->E, q, k);
    if (ws_bytes < wl.total) return FPX_ESPACE;
    // the cold tier must be pinned host memory the device can read
    void* dv[3] = {nullptr, nullptr, nullptr};
    const uint8_t* hv[3] = {tiers->cold_gate, tiers->cold_up, tiers->cold_down};
    for (int i = 0; i < 3; i++) {
        if (cudaHostGetDevicePointer(&dv[i], const_cast<uint8_t*>(hv[i]), 0) != cudaSuccess || !dv[i]) {
            cudaGetLastError();  // not pinned: report it here, leave no error behind
            return FPX_EINVAL;
        }
        if (!aligned(dv[i], 16)) return FPX_EALIGN;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    WsPtrs wp = ws_ptrs(ws, wl);
    if (cudaMemsetAsync(wp.nuni, 0, 16, s) != cudaSuccess) return FPX_ECUDA;
    StageArgs sa{};
    sa.slot_of = tiers->slot_of;
    sa.cgate = static_cast<const uint8_t*>(dv[0]);
    sa.cup = static_cast<const uint8_t*>(dv[1]);
    sa.cdown = static_cast<const uint8_t*>(dv[2]);
    sa.gate = const_cast<uint8_t*>(layer->gate);
    sa.up = const_cast<uint8_t*>(layer->up);
    sa.down = const_cast<uint8_t*>(layer->down);
    sa.mb2 = matrix_bytes(2, layer->I, layer->H);
    sa.mb3 = matrix_bytes(3, layer->H, layer->I);
    sa.E = layer->E;
    sa.n_slots = tiers->n_slots;
    sa.stage0 = tiers->stage_slot0;
    sa.n_stage = tiers->n_stage;
    sa.qk = q * k;
    sa.cache = tiers->cache;
    Plan p = make_plan(*layer, q, k);
    return dispatch_q<0>(q, *layer, p, k, x, nullptr, y, idx_out, w_out, logits_out, nullptr, wp, true, nullptr, false, s,
                         &sa);
}

int moe_tiers_cache_reset(const moe_tiers* tiers, void* stream) {
    if (!tiers || !tiers->cache || tiers->n_stage < 1 || tiers->n_stage > kMaxStageCache) return FPX_EINVAL;
    if (!aligned(tiers->cache, 4)) return FPX_EALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t n = (size_t)tiers->n_stage;
    // clock and copy count 0, every slot empty (-1), last uses 0
    if (cudaMemsetAsync(tiers->cache, 0, sizeof(int32_t) * (2 + 2 * n), s) != cudaSuccess ||
        cudaMemsetAsync(tiers->cache + 2, 0xFF, sizeof(int32_t) * n, s) != cudaSuccess)
        return FPX_ECUDA;
    return FPX_OK;
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
    if (cudaMemsetAsync(wp.nuni, 0, 16, s) != cudaSuccess) return FPX_ECUDA;
    Plan p = make_plan(layers[0], q, k);
    for (int l = 0; l < n_layers; l++) {
        int32_t* io = idx_out ? idx_out + (size_t)l * q * k : nullptr;
        float* tr = r_trace ? r_trace + (size_t)l * q * layers[0].H : nullptr;
        cudaEvent_t const* ev = events ? reinterpret_cast<cudaEvent_t const*>(events) + kKernelsPerLayer * l : nullptr;
        int st = dispatch_q<1>(q, layers[l], p, k, nullptr, rL, rL, io, nullptr, nullptr, tr, wp, l == 0, ev, l > 0, s);
        if (st) return st;
    }
    if (events && cudaEventRecord(reinterpret_cast<cudaEvent_t const*>(events)[kKernelsPerLayer * n_layers], s) != cudaSuccess)
        return FPX_ECUDA;
    return FPX_OK;
}

int fpx_debug_ring_wait(uint64_t wait_ns, int drop_stage) {
    if (wait_ns == 0 || wait_ns > kWaitNs || drop_stage < -1) return FPX_EINVAL;
    const int32_t drop = drop_stage;
    if (cudaMemcpyToSymbol(g_ring_wait_ns, &wait_ns, sizeof(wait_ns)) != cudaSuccess ||
        cudaMemcpyToSymbol(g_ring_drop_stage, &drop, sizeof(drop)) != cudaSuccess)
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

constexpr size_t kStaticWsBytes = size_t(16) << 20;  // 16 MiB: the decode shapes need at most 13.7 MB
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
