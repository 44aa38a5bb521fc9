// Tensor-core decode engine: packed FPX rows staged by TMA, decoded in registers into binary16
// A fragments, multiplied on the tensor cores (mma.sync m16n8k16, binary32 accumulate) against the
// q <= 4 activation columns.
//
// Why tensor cores for a GEMV: at q = 4 the CUDA-core path needs 4 binary32 FMAs per weight, but an
// SM receives about 76 FP2 weights per clock from HBM and executes 128 FMAs per clock, so it is
// ALU-bound near 40% of the memory roofline. One m16n8k16 multiplies 16 rows x 16 weights against 8
// columns in one instruction, leaving the decode itself (about one ALU operation per weight) as the
// only per-weight cost.
//
// Fragment plan (one warp, lane = 4g + t). A "chunk" is 64 consecutive weights of a row = two blocks.
// Four MMAs cover a 16-row tile x one chunk. MMA output columns 0..3 are the q tokens against the
// chunk's first block, columns 4..7 the tokens against its second block, so every accumulator holds
// one (row, block, token) sum and the per-block scale is applied once per block in binary32. Thread
// t decodes block t/2, codes 16(t%2) .. 16(t%2)+15, of rows g and g+8: eight binary16 pairs, pair i
// feeding MMA i/2, k-slots (2t + 8(i%2), +1). The k-slot order inside a block is a permutation of the
// weights; the B table (activations) is laid out with the same permutation, so the dot product is
// unchanged.
//
// Exact decode. A pair of 2-bit codes is moved into the mantissa of a binary16 pair with one LOP3
// (mask | 0x6400, the binary16 1024), so the pair holds 1024 + c * 2^P exactly. The activation table
// holds B = 2 x * 2^-P, and the MMA starts from the per-block constant -sum B (1024 + 1.5 * 2^P) (the
// offset quads), so it sums (2c - 3) x directly. FP3 works the same way with 3-bit codes: one plane
// in the box layout of the layer kernels, a low and a high plane (each its own MMAs) in the row-major
// GEMV. FP4 maps E2M1 bits straight onto binary16 bits (value * 2^-14). Products are exact in
// binary32; only the tensor-core accumulation rounds.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "fpx_common.cuh"

namespace fpx {

constexpr int kWarps = 8;  // consumer warps of a dense-GEMV CTA (plus producer warps)

// Barrier among the kWarps consumer warps only (the producer warps do not take part).
__device__ __forceinline__ void consumers_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kWarps * 32) : "memory");
}

// The MoE layer's streaming CTAs (gate/up, down): kLWarps consumer warps plus one producer warp. Each
// consumer warp decodes kLTiles 16-row tiles of every FP2 / FP3 box (256 rows). A warp loads the
// activation fragments of a chunk once for all its tiles, so 16 warps of one tile (four per scheduler)
// measured slower than 8 warps of two (k_gate_up 36.8 against 35.2 us): the extra table loads cost
// more than the added latency hiding gained.
constexpr int kLWarps = 8;
constexpr int kLTiles = 256 / 16 / kLWarps;
constexpr int kLThreads = (kLWarps + 1) * 32;
constexpr int kFp4Parts = kLWarps / 4;  // FP4 boxes (64 rows = 4 tiles): warps split the 8 chunks
static_assert(kLTiles * 16 * kLWarps == 256 && 8 % kFp4Parts == 0, "layer CTA geometry");

// Barrier among the kLWarps consumer warps of a layer CTA.
__device__ __forceinline__ void layer_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kLWarps * 32) : "memory");
}

// ------------------------------------------------------------------ compile-time binary16 bits

// Bit pattern of a binary16 number that is exactly representable (a small integer times a power of
// two), computed at compile time.
__host__ __device__ constexpr uint16_t f16_bits(double v) {
    uint16_t sign = v < 0 ? 0x8000 : 0;
    double a = v < 0 ? -v : v;
    if (a == 0) return sign;
    int e = 0;
    while (a >= 2.0) { a /= 2.0; e++; }
    while (a < 1.0) { a *= 2.0; e--; }
    // normal numbers only (the constants used here are all >= 2^-14)
    return static_cast<uint16_t>(sign | ((e + 15) << 10) | static_cast<uint16_t>((a - 1.0) * 1024.0));
}
__host__ __device__ constexpr uint32_t f16x2(double v) { return (uint32_t(f16_bits(v)) << 16) | f16_bits(v); }

// ------------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking test of the phase with the given parity (never suspends the thread).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// try_wait that may suspend the thread for up to `ns` nanoseconds while the phase is incomplete (it
// resumes as soon as the phase completes): a waiting warp then stops taking issue slots from the
// warps that do work.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* b, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(b)), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity, giving up after limit_ns of wall time (or kSpinLimit
// polls; each poll may suspend the thread for up to kSleepNs). Returns false when it gives up.
constexpr uint32_t kSpinLimit = 1u << 24;
constexpr uint64_t kWaitNs = 500000000ull;  // 0.5 s
constexpr uint32_t kSleepNs = 20000;       // 20 us per poll
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, uint64_t limit_ns = kWaitNs) {
    if (mbar_try_wait(b, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 0; i < kSpinLimit; i++) {
        if (mbar_try_wait_sleep(b, parity, kSleepNs)) return true;
        if (global_ns() - t0 > limit_ns) return false;
    }
    return false;
}

// Test hooks of the streaming rings, one copy per translation unit (only the MoE layer file exposes a
// setter, fpx_debug_ring_wait): the wall-time limit of the waits between a ring's producer and its
// consumers (a stage's data, a free slot), and a stage index at which CTA 0's producer of the gate/up
// kernel stops issuing copies, as if that copy were lost (-1: none). Waits for copies already issued
// (the producer's drain, the activation tables) keep the fixed kWaitNs, so no copy can land in the
// shared memory of a CTA that has exited.
static __device__ uint64_t g_ring_wait_ns = kWaitNs;
static __device__ int32_t g_ring_drop_stage = -1;
__device__ __forceinline__ uint64_t ring_wait_ns() { return *reinterpret_cast<volatile uint64_t*>(&g_ring_wait_ns); }

// The same on 32-bit shared addresses, for the consumer hot loops: one poll inline, the bounded
// sleeping wait out of line (taken only when a stage has not landed yet).
__device__ __forceinline__ bool mbar_poll(uint32_t b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(b), "r"(parity)
        : "memory");
    return ok != 0;
}
// Whole warp; true when every lane saw the phase complete within the wait limits (ring_wait_ns()).
static __device__ __noinline__ bool mbar_wait_warp_slow(uint32_t b, uint32_t parity) {
    bool done = mbar_poll(b, parity);
    if (!done) {
        const uint64_t t0 = global_ns(), limit = ring_wait_ns();
        for (uint32_t i = 0; i < kSpinLimit && !done; i++) {
            uint32_t ok;
            asm volatile(
                "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                : "=r"(ok)
                : "r"(b), "r"(parity), "r"(kSleepNs)
                : "memory");
            done = ok != 0;
            if (!done && global_ns() - t0 > limit) break;
        }
    }
    return __all_sync(0xffffffffu, done);
}
__device__ __forceinline__ bool mbar_wait_warp(uint32_t b, uint32_t parity) {
    return __all_sync(0xffffffffu, mbar_poll(b, parity)) || mbar_wait_warp_slow(b, parity);
}
__device__ __forceinline__ void mbar_arrive_u32(uint32_t b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(b) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 2-D tiled TMA load of one box into shared memory, completing on mbarrier `bar`.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// Bulk (1-D) TMA copy of `bytes` (a multiple of 16) from global to shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// L2 policy for data read once per pass (the expert and router weights): evict first, so that a pass
// streaming more bytes than L2 holds does not push out what is reused (the kernels' code, the
// activation tables and partial outputs between kernels).
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// bulk_load with an L2 cache policy (l2_evict_first) for the source lines.
__device__ __forceinline__ void bulk_load_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// D = A * B + C, m16n8k16, binary16 inputs, binary32 accumulators.
__device__ __forceinline__ void mma_acc(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ------------------------------------------------------------------ decode into A pairs

// Exponent shift P of pair i (binary16 mantissa position of the code's low bit) for FP2 and FP3;
// FP4 pairs carry no shift (their values are scaled by 2^-14 instead).
__host__ __device__ constexpr int pair_shift(int fmt, int i) {
    return fmt == 4 ? 0 : (i == 0 || i == 1 || i == 5) ? 2 : (i == 2 || i == 6) ? 4 : (i == 3 || i == 7) ? 6 : 8;
}
// Code positions (within the thread's 16-code group) held by the low and high half of pair i.
__host__ __device__ constexpr int pair_lo(int fmt, int i) { return fmt == 4 ? 8 * (i / 4) + (i % 4) : i; }
__host__ __device__ constexpr int pair_hi(int fmt, int i) { return fmt == 4 ? 8 * (i / 4) + (i % 4) + 4 : i + 8; }

// FP3 field of pair p (0..7) of the even (odd = 0) or odd (odd = 1) chunk of a chunk pair: word w
// (0..2 within the pair's three words) * 16 + bit position x of the code's low bit inside each binary16
// half (x = 1, 4, 7: the code is already at mantissa bit x; x = 10, 13: after a shift right by 9, at
// x - 9). -1: the pair of spare bits, code bit i at bit 0 of the half in word i.
__host__ __device__ constexpr int fp3_slot(int odd, int p) {
    return odd == 0 ? (p < 5 ? 3 * p + 1 : 16 + 3 * (p - 5) + 1) : (p < 2 ? 16 + 10 + 3 * p : p < 7 ? 32 + 3 * (p - 2) + 1 : -1);
}
// Mantissa position P of the code's low bit in the decoded binary16 (1024 + c 2^P).
__host__ __device__ constexpr int fp3_box_shift(int odd, int p) {
    return fp3_slot(odd, p) < 0 ? 1 : (fp3_slot(odd, p) % 16 > 9 ? fp3_slot(odd, p) % 16 - 9 : fp3_slot(odd, p) % 16);
}

constexpr uint32_t kMagic = 0x64006400u;  // binary16 pair (1024, 1024)

// Eight A pairs from 16 FP2 codes (2 bits each, code k at bits 2k..2k+1 of w): pair i holds codes
// (i, i + 8) as the binary16 values 1024 + c * 2^P, one LOP3 each. The activations are stored as
// B = 2 x 2^-P, so the MMA sums sum (1024 + c 2^P) * 2 x 2^-P = 2 sum c x + 2048 sum x 2^-P; started
// from C = -sum x 2^-P (2048 + 3 2^P), a per-block constant of the activations, it yields
// sum (2c - 3) x directly.
// `magic` is kMagic, passed in a register: with both the mask and the magic as immediates the
// compiler splits each (w & mask) | magic into two logic operations.
__device__ __forceinline__ void decode_fp2(uint32_t w, uint32_t magic, uint32_t (&a)[8]) {
    const uint32_t s2 = w << 2, s8 = w >> 8;
    a[0] = (s2 & 0x000C000Cu) | magic;
    a[1] = (w & 0x000C000Cu) | magic;
    a[2] = (w & 0x00300030u) | magic;
    a[3] = (w & 0x00C000C0u) | magic;
    a[4] = (w & 0x03000300u) | magic;
    a[5] = (s8 & 0x000C000Cu) | magic;
    a[6] = (s8 & 0x00300030u) | magic;
    a[7] = (s8 & 0x00C000C0u) | magic;
}

// FP4: E2M1 nibble (s, e1, e0, m) -> binary16 bits (s << 15) | (e1 e0 m) << 9, i.e. the E2M1 value
// times 2^-14 (exponent field 0 gives the binary16 subnormals 0 and 2^-15 = 0.5 * 2^-14). Pair
// (k, k + 4) of a word of eight codes sits at bits 4k and 4k + 16.
template <int K>
__device__ __forceinline__ uint32_t fp4_pair(uint32_t w) {
    const uint32_t m = (K <= 2) ? (w << (9 - 4 * K)) : (w >> (4 * K - 9));
    const uint32_t s = (K <= 3) ? (w << (12 - 4 * K)) : (w >> (4 * K - 12));
    return (m & 0x0E000E00u) | (s & 0x80008000u);
}

// w0: codes 0..7, w1: codes 8..15 of the thread's group.
__device__ __forceinline__ void decode_fp4(uint32_t w0, uint32_t w1, uint32_t (&a)[8]) {
    a[0] = fp4_pair<0>(w0); a[1] = fp4_pair<1>(w0); a[2] = fp4_pair<2>(w0); a[3] = fp4_pair<3>(w0);
    a[4] = fp4_pair<0>(w1); a[5] = fp4_pair<1>(w1); a[6] = fp4_pair<2>(w1); a[7] = fp4_pair<3>(w1);
}

// ------------------------------------------------------------------ B table (activations)

// Layout: for chunk c (64 weights), active lane a (0..15), MMA j (0..3): a uint2 holding the B
// fragment registers {b0b1, b2b3} = pairs 2j and 2j+1 of that lane's k-slots. Lane (g, t) is active
// when its column (token g % 4, block g / 4) belongs to the block it decodes (t / 2), i.e.
// g / 4 == t / 2; then a = 8 (t / 2) + 2 (g % 4) + t % 2. Inactive lanes multiply zeros.
__host__ __device__ constexpr int btab_bytes(int K) { return (K / 64) * 16 * 4 * 8; }

__device__ __forceinline__ int b_active_index(int lane) {
    const int g = lane >> 2, t = lane & 3;
    return ((g >> 2) == (t >> 1)) ? 8 * (t >> 1) + 2 * (g & 3) + (t & 1) : -1;
}

// Column scale: x' = x * 2^(14 - floor(log2 max|x|)) puts a column's largest element in [2^14, 2^15).
// Every element within 2^28 of the largest is then a binary16 normal (a bfloat16 element within 2^31
// is exact), so the encoding adds at most 2^-11 |x| to an element, plus 2^(e - 40) for elements that
// fall into the binary16 subnormal range (max |x| in [2^(e-1), 2^e)). Returns the exponent shift (0 for
// an all-zero column), at most 110 so that 2^(shift + 3) stays a binary32 normal (a column whose largest
// element is below 2^-96 is scaled less; it is still exact down to 2^-24 of that scale).
__device__ __forceinline__ int column_shift(float amax) {
    if (!(amax > 0.0f) || !isfinite(amax)) return 0;
    int e;
    frexpf(amax, &e);  // amax in [2^(e-1), 2^e)
    return min(14 - (e - 1), 110);
}

// ------------------------------------------------------------------ activation tables, batched

// 2^e as binary32 (exact; bit construction in the normal range).
__device__ __forceinline__ float exp2i(int e) {
    return (e >= -126 && e <= 127) ? __int_as_float((e + 127) << 23) : ldexpf(1.0f, e);
}

// Activation sources for the table builder: load16 returns the 16 consecutive values (one code
// group) at element offset e0 (a multiple of 16) of a [q][K] column array; V is how many groups a
// thread loads before using them.
struct SrcBF16 {  // bfloat16 columns
    static constexpr int V = 4;
    const uint16_t* x;
    __device__ __forceinline__ void load16(size_t e0, float (&v)[16]) const {
        const uint4* p = reinterpret_cast<const uint4*>(x + e0);
        const uint4 a = p[0], b = p[1];
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 8; i++) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
};
struct SrcF32 {  // binary32 columns
    static constexpr int V = 2;
    const float* x;
    __device__ __forceinline__ void load16(size_t e0, float (&v)[16]) const {
        const float4* p = reinterpret_cast<const float4*>(x + e0);
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const float4 f = p[i];
            v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
        }
    }
};
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ float h2lo(uint32_t w) { return __half2float(__ushort_as_half((uint16_t)(w & 0xFFFFu))); }
__device__ __forceinline__ float h2hi(uint32_t w) { return __half2float(__ushort_as_half((uint16_t)(w >> 16))); }

// FP3 high-plane pair p carries its two bits at binary16 mantissa position Q(p).
__host__ __device__ constexpr int hi_shift(int p) { return p < 7 ? p + 3 : 9; }

// Table entries (32 bytes each) = the B registers of one active lane for one chunk, pairs 0..7 of a
// 16-activation code group. FP2/FP3 pair p holds codes (p, p + 8), FP4 pair p codes
// (8 (p/4) + p%4, +4). Scales: FP2 and the FP3 low plane 2^(sh + 1 - P(p)), the FP3 high plane
// 2^(sh + 3 - Q(p)), FP4 2^sh. `part` returns the group's share of the block offset that the MMA's
// initial accumulator removes: FP2 sum B (1024 + 1.5 2^P); FP3 sum [1024 B_lo + 1024 B_hi
// + 3.5 2^P B_lo] (from the binary16 values the MMA sees).
__device__ __forceinline__ void pack_fp2(const float (&v)[16], int sh, uint32_t (&w)[8], float& part) {
    part = 0.f;
#pragma unroll
    for (int p = 0; p < 8; p++) {
        const float sc = exp2i(sh + 1 - pair_shift(2, p));
        w[p] = pack_h2(v[p] * sc, v[p + 8] * sc);
        part = fmaf(h2lo(w[p]) + h2hi(w[p]), 1024.0f + 1.5f * float(1 << pair_shift(2, p)), part);
    }
}
__device__ __forceinline__ void pack_fp3(const float (&v)[16], int sh, uint32_t (&lo)[8], uint32_t (&hi)[8], float& part) {
    part = 0.f;
#pragma unroll
    for (int p = 0; p < 8; p++) {
        const float sl = exp2i(sh + 1 - pair_shift(3, p)), sh8 = exp2i(sh + 3 - hi_shift(p));
        lo[p] = pack_h2(v[p] * sl, v[p + 8] * sl);
        hi[p] = pack_h2(v[p] * sh8, v[p + 8] * sh8);
        const float bl = h2lo(lo[p]) + h2hi(lo[p]), bh = h2lo(hi[p]) + h2hi(hi[p]);
        part = fmaf(bl, 1024.0f + 3.5f * float(1 << pair_shift(3, p)), fmaf(bh, 1024.0f, part));
    }
}
// FP3 in the box layout (one plane, codes 0..7 at mantissa position P = fp3_box_shift(odd, p), odd =
// the parity of the group's chunk): B = 2^(sh + 1 - P); the MMA sees sum (1024 + c 2^P) B = 2 sum c x'
// + sum 1024 B, so the offset removed is sum B (1024 + 3.5 2^P), leaving sum (2c - 7) x'.
__device__ __forceinline__ void pack_fp3b(const float (&v)[16], int sh, int odd, uint32_t (&w)[8], float& part) {
    part = 0.f;
#pragma unroll
    for (int p = 0; p < 8; p++) {
        const int P = odd ? fp3_box_shift(1, p) : fp3_box_shift(0, p);
        const float sc = exp2i(sh + 1 - P);
        w[p] = pack_h2(v[p] * sc, v[p + 8] * sc);
        part = fmaf(h2lo(w[p]) + h2hi(w[p]), 1024.0f + 3.5f * float(1 << P), part);
    }
}
__device__ __forceinline__ void pack_fp4(const float (&v)[16], int sh, uint32_t (&w)[8]) {
    const float sc = exp2i(sh);
#pragma unroll
    for (int p = 0; p < 8; p++) w[p] = pack_h2(v[8 * (p / 4) + p % 4] * sc, v[8 * (p / 4) + p % 4 + 4] * sc);
}
__device__ __forceinline__ void store_entry(uint2* tab, size_t e, const uint32_t (&w)[8]) {
    uint4* d = reinterpret_cast<uint4*>(tab + e * 4);
    d[0] = make_uint4(w[0], w[1], w[2], w[3]);
    d[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

// Bytes of the FP2/FP3 offset quads: per block, two float4 {o(2h), o(2h+1), o(2h), o(2h+1)} (h = 0, 1)
// laid out as the MMA's initial accumulator of the lanes that decode the block.
__host__ __device__ constexpr int oq_bytes(int K) { return K; }

// Table sets for K weights, as built in global memory and copied as one block into shared memory,
// followed in global memory only by 16 bytes of column shifts. Gate/up: [FP2 table (8K) | FP4 table
// (8K) | offset quads (K)]. Down: [FP3 table (box layout, 8K) | offset quads (K)] for a routed expert,
// [FP4 table (8K)] for the shared expert.
__host__ __device__ constexpr int tset_copy_bytes(int K) { return 2 * btab_bytes(K) + oq_bytes(K); }
__host__ __device__ constexpr int tset_bytes(int K) { return tset_copy_bytes(K) + 16; }
__host__ __device__ constexpr int dset_copy_bytes(int K) { return btab_bytes(K) + oq_bytes(K); }
__host__ __device__ constexpr int dset_bytes(int K) { return dset_copy_bytes(K) + 16; }
// offset of the offset quads in a table set whose first table has format FA
__host__ __device__ constexpr int set_oq_offset(int FA, int K) { return FA == 2 ? 2 * btab_bytes(K) : btab_bytes(K); }

// Packs code group gi (16 consecutive activations v of token tok, starting at weight k0 of K) into a
// table set at `ts` (global memory): FA is the format of the first table (2: FP2 with FP4 second; 3:
// FP3 in the box layout; 4: FP4 only). Returns the group's share of its block offset (0 for FP4). Lanes
// holding the two groups of a block (gi even, gi + 1) add the shares with add_offsets().
template <int FA>
__device__ __forceinline__ float pack_group(uint8_t* ts, int K, int tok, int k0, const float (&v)[16], int sh) {
    const int c = k0 >> 6, half = (k0 >> 5) & 1, hw = (k0 >> 4) & 1;
    const size_t e = (size_t)c * 16 + 8 * half + 2 * tok + hw;
    uint2* ta = reinterpret_cast<uint2*>(ts);
    uint2* tb = reinterpret_cast<uint2*>(ts + btab_bytes(K));
    uint32_t w[8];
    float part = 0.f;
    if constexpr (FA == 2) {
        pack_fp2(v, sh, w, part);
        store_entry(ta, e, w);
        pack_fp4(v, sh, w);
        store_entry(tb, e, w);
    } else if constexpr (FA == 3) {
        (void)tb;
        pack_fp3b(v, sh, c & 1, w, part);
        store_entry(ta, e, w);
    } else {
        pack_fp4(v, sh, w);
        store_entry(ta, e, w);
    }
    return part;
}

// Whole warp, after pack_group on lane pairs (2i, 2i + 1) = the two groups of one block: writes the
// block's negated offset quad entries (valid lanes only).
template <int FA>
__device__ __forceinline__ void add_offsets(uint8_t* ts, int K, int tok, int k0, float part, bool valid) {
    const float nxt = __shfl_down_sync(0xffffffffu, part, 1);
    if (valid && ((k0 >> 4) & 1) == 0) {
        float* qd = reinterpret_cast<float*>(ts + set_oq_offset(FA, K)) + (size_t)((k0 >> 5) * 2 + (tok >> 1)) * 4 + (tok & 1);
        qd[0] = qd[2] = -(part + nxt);
    }
}

// Builds the activation tables for columns src[tok][k] (tok < q <= 4, K % 64 == 0) in format FMT:
// tab (FP2, FP3 low plane, or FP4), tab_hi (FP3 high plane) and, for FP2/FP3, the negated block
// offsets oq (the MMA's initial accumulator); WITH4 also builds the FP4 table tab4 from the same
// columns. BOX3: FP3 as the one box-layout table of the tiled boxes (pack_fp3b; tab_hi unused).
// shift[4] receives the column shifts. Each thread owns whole 16-weight code groups: it
// issues all of a pass's loads before using them and writes each table entry with two 16-byte
// stores. CONS: only the kWarps consumer warps (threads 0 .. 32 kWarps - 1) take part and
// synchronise on the consumer barrier, so the producer warp can issue loads meanwhile; otherwise the
// whole CTA.
template <int FMT, bool WITH4, bool CONS = false, bool BOX3 = false, class SRC>
__device__ void build_tables(const SRC src, int K, int q, uint2* tab, uint2* tab_hi, uint2* tab4, float* oq, int* shift,
                             float* red4) {
    constexpr int V = SRC::V;
    const int ngr = q * K / 16;
    const int tid = threadIdx.x, nt = CONS ? kWarps * 32 : blockDim.x;
    // pass 1: column maxima
    float m[4] = {0.f, 0.f, 0.f, 0.f};
    // loops start at the warp's first thread so every lane of a warp runs the same iterations (the
    // shuffles below need all 32 lanes); lanes past the end are predicated off
    const int lane = tid & 31;
    for (int base = tid - lane; base < ngr; base += V * nt) {
        float v[V][16];
#pragma unroll
        for (int it = 0; it < V; it++)
            if (base + lane + it * nt < ngr) src.load16((size_t)(base + lane + it * nt) * 16, v[it]);
#pragma unroll
        for (int it = 0; it < V; it++) {
            const int gi = base + lane + it * nt;
            if (gi < ngr) {
                const int tok = gi * 16 / K;
                float mm = 0.f;
#pragma unroll
                for (int j = 0; j < 16; j++) mm = fmaxf(mm, fabsf(v[it][j]));
#pragma unroll
                for (int t = 0; t < 4; t++) m[t] = t == tok ? fmaxf(m[t], mm) : m[t];
            }
        }
    }
#pragma unroll
    for (int t = 0; t < 4; t++) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m[t] = fmaxf(m[t], __shfl_xor_sync(0xffffffffu, m[t], o));
    }
    if ((tid & 31) == 0)
        for (int t = 0; t < 4; t++) red4[(tid >> 5) * 4 + t] = m[t];
    // entries of absent tokens stay zero
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    for (int i = tid; i < (K / 64) * 16; i += nt) {
        if (((i & 15) >> 1 & 3) >= q) {
            reinterpret_cast<uint4*>(tab + (size_t)i * 4)[0] = z;
            reinterpret_cast<uint4*>(tab + (size_t)i * 4)[1] = z;
            if (FMT == 3 && !BOX3) {
                reinterpret_cast<uint4*>(tab_hi + (size_t)i * 4)[0] = z;
                reinterpret_cast<uint4*>(tab_hi + (size_t)i * 4)[1] = z;
            }
            if (WITH4) {
                reinterpret_cast<uint4*>(tab4 + (size_t)i * 4)[0] = z;
                reinterpret_cast<uint4*>(tab4 + (size_t)i * 4)[1] = z;
            }
        }
    }
    if (FMT != 4)
        for (int i = tid; i < (K / 32) * 8; i += nt)
            if (2 * ((i >> 2) & 1) + (i & 1) >= q) oq[i] = 0.f;
    if (CONS) consumers_sync(); else __syncthreads();
    if (tid < 4) {
        float mm = 0.f;
        for (int w = 0; w < nt / 32; w++) mm = fmaxf(mm, red4[w * 4 + tid]);
        shift[tid] = column_shift(mm);
    }
    if (CONS) consumers_sync(); else __syncthreads();
    // pass 2: whole entries
    for (int base = tid - lane; base < ngr; base += V * nt) {
        float v[V][16];
#pragma unroll
        for (int it = 0; it < V; it++)
            if (base + lane + it * nt < ngr) src.load16((size_t)(base + lane + it * nt) * 16, v[it]);
#pragma unroll
        for (int it = 0; it < V; it++) {
            const int gi = base + lane + it * nt;
            float part = 0.f;
            if (gi < ngr) {
                const int tok = gi * 16 / K, k0 = gi * 16 - tok * K;
                const int c = k0 >> 6, half = (k0 >> 5) & 1, hw = (k0 >> 4) & 1;
                const size_t e = (size_t)c * 16 + 8 * half + 2 * tok + hw;
                const int sh = shift[tok];
                uint32_t w[8];
                if constexpr (FMT == 2) {
                    pack_fp2(v[it], sh, w, part);
                    store_entry(tab, e, w);
                } else if constexpr (FMT == 3 && BOX3) {
                    pack_fp3b(v[it], sh, c & 1, w, part);
                    store_entry(tab, e, w);
                } else if constexpr (FMT == 3) {
                    uint32_t wh[8];
                    pack_fp3(v[it], sh, w, wh, part);
                    store_entry(tab, e, w);
                    store_entry(tab_hi, e, wh);
                } else {
                    pack_fp4(v[it], sh, w);
                    store_entry(tab, e, w);
                }
                if (WITH4) {
                    pack_fp4(v[it], sh, w);
                    store_entry(tab4, e, w);
                }
            }
            if (FMT != 4) {
                // a 32-weight block is two consecutive groups (lanes 2i, 2i + 1): add them in order
                const float nxt = __shfl_down_sync(0xffffffffu, part, 1);
                if (gi < ngr && (gi & 1) == 0) {
                    const int tok = gi * 16 / K, blk = (gi * 16 - tok * K) / 32;
                    float* qd = oq + (size_t)(blk * 2 + (tok >> 1)) * 4 + (tok & 1);
                    qd[0] = qd[2] = -(part + nxt);
                }
            }
        }
    }
}

// ------------------------------------------------------------------ host: tensor maps

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;  // the driver entry point, looked up once
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// A 2-D map over `rows` rows of `row_bytes` bytes (row stride `stride` bytes), elements of 1 or 2
// bytes, box = box_bytes x box_rows. Out-of-range rows read as zeros.
inline int make_row_map(CUtensorMap* m, const void* base, int64_t row_bytes, int64_t rows, int64_t stride,
                        int box_bytes, int box_rows, int elem_bytes) {
    auto enc = tensor_map_encoder();
    if (!enc) return FPX_ECUDA;
    const CUtensorMapDataType dt = elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes / elem_bytes), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(stride)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_bytes / elem_bytes), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FPX_OK : FPX_ECUDA;
}

// Per-format staging geometry: a TMA box covers `box_bytes` of each row = `box_chunks` chunks of
// 64 weights (FP2 4 x 20 B, FP3 4 x 28 B, FP4 8 x 34 B; multiples of 16 bytes, at most 256
// elements). FP4 uses 2-byte elements so its 272-byte box stays within 256 elements.
__host__ __device__ constexpr int box_bytes(int fmt) { return fmt == 2 ? 80 : fmt == 3 ? 112 : 272; }
__host__ __device__ constexpr int box_chunks(int fmt) { return fmt == 4 ? 8 : 4; }
__host__ __device__ constexpr int chunk_bytes(int fmt) { return 2 * block_bytes(fmt); }
__host__ __device__ constexpr int elem_bytes(int fmt) { return fmt == 4 ? 2 : 1; }

// Rows decodable by the tensor-core path: whole boxes per row.
__host__ __device__ constexpr bool mma_shape_ok(int fmt, int64_t K) { return K > 0 && K % (64 * box_chunks(fmt)) == 0; }

// ------------------------------------------------------------------ chunk processing

// Shared-memory loads from a 32-bit shared address plus a compile-time byte offset, so the hot loop
// needs one base register per stream and no address arithmetic.
template <int OFF>
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1+%2];" : "=r"(v) : "r"(a), "n"(OFF));
    return v;
}
template <int OFF>
__device__ __forceinline__ uint32_t lds16(uint32_t a) {
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1+%2];" : "=h"(v) : "r"(a), "n"(OFF));
    return v;
}
template <int OFF>
__device__ __forceinline__ uint32_t lds8(uint32_t a) {
    uint16_t v;
    asm volatile("ld.shared.u8 %0, [%1+%2];" : "=h"(v) : "r"(a), "n"(OFF));
    return v;
}
template <int OFF>
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4+%5];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a), "n"(OFF));
    return v;
}

// Per-thread byte offsets inside a chunk, for thread t of its group of four (which decodes block
// t / 2, codes 16 (t % 2) .. 16 (t % 2) + 15):
//   FP2 chunk [d0 (2) | codes0 (8) | d1 (2) | codes1 (8)] = words 0..4: thread t reads words t and
//   t + 1 (so the 8 rows x 4 threads of a load touch 32 distinct banks at the 80-byte row pitch) and
//   takes its code bytes 2 + 4t .. (t < 2) or word t + 1 (t >= 2) with one PRMT; scale at 10 (t / 2).
//   FP3 chunk [d0 | lo0 (8) | hi0 (4) | d1 | lo1 | hi1]: low-plane word as FP2 (base 0 or 16), high
//   bits at 14 (t / 2) + 10 + 2hw, scale at 14 (t / 2).
//   FP4 chunk [e0 (1) | codes0 (16) | e1 | codes1]: 8 code bytes at 17 (t / 2) + 1 + 8hw, read as three
//   aligned words and a funnel shift; the alignment differs between even and odd chunks (chunks are
//   34 bytes); scale byte at 17 (t / 2).
struct LaneOfs {
    int w, w_odd;       // aligned code word offset (FP4: even / odd chunks)
    uint32_t sel, sh_odd;  // FP2/FP3: PRMT selector; FP4: funnel shifts (even / odd chunks)
    int s, h;           // scale and FP3 high-plane offsets
};

template <int FMT>
__device__ __forceinline__ LaneOfs lane_ofs(int t) {
    const int half = t >> 1, hw = t & 1;
    LaneOfs L{};
    if (FMT == 2) {
        L.w = 4 * t;
        L.sel = half ? 0x7654u : 0x5432u;
        L.s = 10 * half;
    } else if (FMT == 3) {
        L.w = half ? 16 + 4 * hw : 4 * hw;
        L.sel = half ? 0x3210u : 0x5432u;
        L.h = 14 * half + 10 + 2 * hw;
        L.s = 14 * half;
    } else {
        const int o = 17 * half + 1 + 8 * hw;
        L.w = o - (o & 3);
        L.sel = (uint32_t)(o & 3) * 8;
        L.w_odd = o - ((o + 2) & 3);
        L.sh_odd = (uint32_t)((o + 2) & 3) * 8;
        L.s = 17 * half;
    }
    return L;
}

// Per-stage base addresses of one thread: its row g of the first tile, plus the lane offsets.
struct RowAddr {
    uint32_t w, w_odd, s, h;
};
__device__ __forceinline__ RowAddr row_addr(uint32_t row, const LaneOfs& L) {
    return RowAddr{row + (uint32_t)L.w, row + (uint32_t)L.w_odd, row + (uint32_t)L.s, row + (uint32_t)L.h};
}

// FP3 as two exact binary16 planes: low-plane pair i = 1024 + l 2^P (as FP2), high-plane pair
// i = 1024 + h 2^Q(i). With B_lo = 2 x 2^-P and B_hi = 8 x 2^-Q the two MMAs sum 2 l x + 8 h x plus
// a per-block constant of the activations, removed by the initial accumulator: (2c - 7) x with
// c = l + 4h.
__device__ __forceinline__ void decode_fp3_planes(uint32_t lo, uint32_t hg, uint32_t magic, uint32_t (&al)[8],
                                                  uint32_t (&ah)[8]) {
    decode_fp2(lo, magic, al);
    const uint32_t sp = __byte_perm(hg, 0u, 0x4140);  // bit k -> k (k < 8), bit 8 + k -> 16 + k
    const uint32_t h3 = sp << 3, h2 = sp << 2;
    ah[0] = (h3 & 0x00080008u) | magic;
    ah[1] = (h3 & 0x00100010u) | magic;
    ah[2] = (h3 & 0x00200020u) | magic;
    ah[3] = (h3 & 0x00400040u) | magic;
    ah[4] = (h3 & 0x00800080u) | magic;
    ah[5] = (h3 & 0x01000100u) | magic;
    ah[6] = (h3 & 0x02000200u) | magic;
    ah[7] = (h2 & 0x02000200u) | magic;
}

// Decodes chunk C (compile-time) of the row at byte offset RO (compile-time) from the thread's base:
// A pairs (FP3: both planes) and the block scale in binary32.
template <int FMT, int RO, int C>
__device__ __forceinline__ float row_decode(const RowAddr& ra, const LaneOfs& L, uint32_t magic, uint32_t (&a)[8],
                                            uint32_t (&ah)[8], uint32_t& bad) {
    constexpr int CB = chunk_bytes(FMT);
    if constexpr (FMT == 2) {
        const uint32_t cw = __byte_perm(lds32<RO + C * CB>(ra.w), lds32<RO + C * CB + 4>(ra.w), L.sel);
        decode_fp2(cw, magic, a);
        return __half2float(__ushort_as_half((uint16_t)lds16<RO + C * CB>(ra.s)));
    } else if constexpr (FMT == 3) {
        const uint32_t lo = __byte_perm(lds32<RO + C * CB>(ra.w), lds32<RO + C * CB + 4>(ra.w), L.sel);
        decode_fp3_planes(lo, lds16<RO + C * CB>(ra.h), magic, a, ah);
        return __half2float(__ushort_as_half((uint16_t)lds16<RO + C * CB>(ra.s)));
    } else {
        const uint32_t base = (C & 1) ? ra.w_odd : ra.w;
        const uint32_t sh = (C & 1) ? L.sh_odd : L.sel;
        const uint32_t x0 = lds32<RO + C * CB>(base), x1 = lds32<RO + C * CB + 4>(base), x2 = lds32<RO + C * CB + 8>(base);
        decode_fp4(__funnelshift_r(x0, x1, sh), __funnelshift_r(x1, x2, sh), a);
        const uint32_t e = lds8<RO + C * CB>(ra.s);
        bad |= e == 255u;  // NaN scale: the block is invalid and counts as zeros
        // 2^(e-127): e in 1..254 is a normal binary32 power of two, e == 0 the subnormal 2^-127
        const float sc = e ? __uint_as_float(e << 23) : __uint_as_float(0x00400000u);
        return e == 255u ? 0.0f : sc;
    }
}

// D = A * B + C with C = {c.x, c.y, c.z, c.w} (m16n8k16, binary16 inputs, binary32 accumulators).
__device__ __forceinline__ void mma_c(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                      uint32_t b1, const float4& c) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c.x), "f"(c.y), "f"(c.z), "f"(c.w));
}

// Four MMAs over one plane of a 16-row tile x 64 weights: rows g (a0) and g + 8 (a8), B registers
// from the lane's 32-byte table entry (two 16-byte halves).
__device__ __forceinline__ void plane_mma(float (&acc)[4], const uint32_t (&a0)[8], const uint32_t (&a8)[8], const uint4& b0,
                                          const uint4& b1) {
    mma_acc(acc, a0[0], a8[0], a0[1], a8[1], b0.x, b0.y);
    mma_acc(acc, a0[2], a8[2], a0[3], a8[3], b0.z, b0.w);
    mma_acc(acc, a0[4], a8[4], a0[5], a8[5], b1.x, b1.y);
    mma_acc(acc, a0[6], a8[6], a0[7], a8[7], b1.z, b1.w);
}

// Zero area read by inactive lanes in place of table entries: one entry per chunk of a box.
constexpr int kZeroBytes = 8 * 64 * 8;  // box_chunks <= 8 chunks x 512 bytes

// Per-lane shared address of the table entry of chunk `chunk0` (512 bytes per chunk), or of the zero
// area for lanes whose B fragment is structurally zero.
__device__ __forceinline__ uint32_t lane_tab(const uint2* tab, const uint2* zero, int a_idx, int chunk0) {
    return a_idx >= 0 ? smem_u32(tab) + (uint32_t)chunk0 * 512u + (uint32_t)a_idx * 32u : smem_u32(zero);
}

// Per-lane shared address of the FP2/FP3 offset quad of chunk `chunk0` (64 bytes per chunk).
__device__ __forceinline__ uint32_t lane_oq(const float* oq, int chunk0, int t) {
    return smem_u32(oq) + (uint32_t)chunk0 * 64u + (uint32_t)(t >> 1) * 32u + (uint32_t)(t & 1) * 16u;
}

// NC chunks of a staged box (row pitch box_bytes(FMT)) for NT consecutive 16-row tiles sharing the
// activations. `row` is the shared address of the thread's row g of the first tile at the box's first
// chunk; b / bh / oq are the lane addresses of the table entries (FP3: low and high plane) and offset
// quads for that chunk. Fully unrolled so the decode of one chunk overlaps the MMAs of another.
template <int FMT, int NT, int NC, int C = 0>
__device__ __forceinline__ void box_tiles(uint32_t row, const LaneOfs& L, uint32_t b, uint32_t bh, uint32_t oq,
                                          uint32_t magic, float (&y)[NT][4], uint32_t& bad) {
    if constexpr (C < NC) {
        constexpr int P = box_bytes(FMT);
        const RowAddr ra = row_addr(row, L);
        const uint4 b0 = lds128<C * 512>(b), b1 = lds128<C * 512 + 16>(b);
        uint4 h0 = make_uint4(0u, 0u, 0u, 0u), h1 = h0;
        if constexpr (FMT == 3) { h0 = lds128<C * 512>(bh); h1 = lds128<C * 512 + 16>(bh); }
        float4 c4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if constexpr (FMT != 4) {
            const uint4 q = lds128<C * 64>(oq);
            c4 = make_float4(__uint_as_float(q.x), __uint_as_float(q.y), __uint_as_float(q.z), __uint_as_float(q.w));
        }
#pragma unroll
        for (int i = 0; i < NT; i++) {
            uint32_t a0[8], a8[8], g0[8], g8[8];
            const float d0 = i == 0 ? row_decode<FMT, 0, C>(ra, L, magic, a0, g0, bad) : row_decode<FMT, 16 * P, C>(ra, L, magic, a0, g0, bad);
            const float d8 = i == 0 ? row_decode<FMT, 8 * P, C>(ra, L, magic, a8, g8, bad) : row_decode<FMT, 24 * P, C>(ra, L, magic, a8, g8, bad);
            float acc[4];
            if constexpr (FMT == 3) {
                mma_c(acc, a0[0], a8[0], a0[1], a8[1], b0.x, b0.y, c4);
                mma_acc(acc, a0[2], a8[2], a0[3], a8[3], b0.z, b0.w);
                mma_acc(acc, a0[4], a8[4], a0[5], a8[5], b1.x, b1.y);
                mma_acc(acc, a0[6], a8[6], a0[7], a8[7], b1.z, b1.w);
                plane_mma(acc, g0, g8, h0, h1);
            } else {
                // two accumulator chains (alternate K steps) joined at the end: half the dependent
                // latency (measured: FP2 q = 4 GEMV 3.10 -> 3.18 TB/s; FP3's eight-MMA chain gained nothing)
                float acc2[4];
                mma_c(acc, a0[0], a8[0], a0[1], a8[1], b0.x, b0.y, c4);
                mma_c(acc2, a0[2], a8[2], a0[3], a8[3], b0.z, b0.w, make_float4(0.f, 0.f, 0.f, 0.f));
                mma_acc(acc, a0[4], a8[4], a0[5], a8[5], b1.x, b1.y);
                mma_acc(acc2, a0[6], a8[6], a0[7], a8[7], b1.z, b1.w);
                acc[0] += acc2[0]; acc[1] += acc2[1]; acc[2] += acc2[2]; acc[3] += acc2[3];
            }
            y[i][0] = fmaf(d0, acc[0], y[i][0]);
            y[i][1] = fmaf(d0, acc[1], y[i][1]);
            y[i][2] = fmaf(d8, acc[2], y[i][2]);
            y[i][3] = fmaf(d8, acc[3], y[i][3]);
        }
        box_tiles<FMT, NT, NC, C + 1>(row, L, b, bh, oq, magic, y, bad);
    }
}

// Whole warp: flags FPX_EDATA once if any lane decoded an FP4 block with the NaN scale.
__device__ __forceinline__ void report_bad(uint32_t bad, int32_t* st) {
    if (__any_sync(0xffffffffu, bad != 0u) && (threadIdx.x & 31) == 0) flag(st, FPX_EDATA);
}

// ------------------------------------------------------------------ per-warp TMA ring (dense GEMV)

constexpr int kStages = 4;           // TMA ring depth per warp
constexpr int kSlotBytes = 4352;     // one stage: 16 FP4 rows x 272 B, or an FP2 / FP3 box
constexpr int kRingBytes = kWarps * kStages * kSlotBytes;
constexpr int kTileRows = 16;

// Per-consumer-warp TMA ring: kStages slots of kSlotBytes. full[s] completes when the TMA data of the
// unit in slot s has landed; empty[s] when the consumer warp has finished reading it. The producer
// warp waits on empty before refilling a slot, the consumer on full before reading it.
struct Ring {
    uint8_t* slots;
    uint64_t* full;
    uint64_t* empty;
};

// Waits for the unit in slot (u % kStages), phase (u / kStages). On timeout flags FPX_ETIMEOUT and
// returns false.
__device__ __forceinline__ bool ring_wait(const Ring& R, uint32_t u, int32_t* st) {
    // every lane waits; the warp proceeds if any lane saw the phase complete, so all 32 lanes take
    // the same branch (the MMAs and warp syncs that follow need the whole warp)
    const bool done = __any_sync(0xffffffffu, mbar_wait(R.full + (u % kStages), (u / kStages) & 1u));
    if (!done && (threadIdx.x & 31) == 0) flag(st, FPX_ETIMEOUT);
    return done;
}

// The consumer warp is done with unit u: hand its slot back to the producer.
__device__ __forceinline__ void ring_release(const Ring& R, uint32_t u) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(R.empty + (u % kStages));
}

// Producer: may slot (n % kStages) receive the warp's n-th unit? (single poll)
__device__ __forceinline__ bool ring_free(const Ring& R, uint32_t n) {
    return n < (uint32_t)kStages || mbar_try_wait(R.empty + (n % kStages), ((n / kStages) + 1u) & 1u);
}

// After a timeout: wait (bounded) for the units this consumer still expects, so no copy lands after
// the CTA exits.
__device__ inline void ring_drain(const Ring& R, uint32_t consumed, uint32_t expected) {
    if ((threadIdx.x & 31) != 0) return;
    for (uint32_t u = consumed; u < expected && u < consumed + kStages; u++) mbar_wait(R.full + (u % kStages), (u / kStages) & 1u);
}

// Adds the partner thread's block-parity partial sums (lane ^ 2): afterwards lanes t and t ^ 2 hold
// the full sums of rows (g, g + 8) for tokens 2 (t % 2), 2 (t % 2) + 1.
__device__ __forceinline__ void pair_reduce(float (&y)[4]) {
#pragma unroll
    for (int i = 0; i < 4; i++) y[i] += __shfl_xor_sync(0xffffffffu, y[i], 2);
}

// Shared-memory carve-up of the per-warp-ring kernels.
struct Smem {
    uint8_t* ring;   // kRingBytes
    uint64_t* bars;  // full[kWarps * kStages], then empty[kWarps * kStages]
    uint2* zero;     // kZeroBytes of zeros
    uint2* tab0;     // activation tables (FP3: low plane)
    uint2* tab1;     // FP3 high plane
    float* oq;       // FP2/FP3 offset quads, K bytes
};

__device__ __forceinline__ Smem carve(uint8_t* raw, int tab_bytes, int ntabs) {
    // TMA destinations: align the ring to 128 bytes (the allocation has 128 bytes of slack)
    uint8_t* base = raw + ((128u - (smem_u32(raw) & 127u)) & 127u);
    Smem s;
    s.ring = base;
    s.bars = reinterpret_cast<uint64_t*>(base + kRingBytes);
    s.zero = reinterpret_cast<uint2*>(base + kRingBytes + 1024 + 16);  // odd 16-byte slot (see cta_carve)
    s.tab0 = reinterpret_cast<uint2*>(base + kRingBytes + 1024 + kZeroBytes + 32);
    s.tab1 = reinterpret_cast<uint2*>(base + kRingBytes + 1024 + kZeroBytes + 32 + tab_bytes);
    s.oq = reinterpret_cast<float*>(base + kRingBytes + 1024 + kZeroBytes + 32 + (size_t)ntabs * tab_bytes);
    return s;
}

__host__ __device__ constexpr size_t smem_bytes(int tab_bytes, int ntabs) {
    // ring, barriers, zero area, ntabs activation tables of tab_bytes = K * 8 bytes, offset quads of
    // K bytes = tab_bytes / 8, alignment slack
    return (size_t)kRingBytes + 1024 + kZeroBytes + 32 + (size_t)tab_bytes * ntabs + tab_bytes / 8 + 128;
}

__device__ __forceinline__ Ring warp_ring(const Smem& s, int warp) {
    Ring R;
    R.slots = s.ring + (size_t)warp * kStages * kSlotBytes;
    R.full = s.bars + warp * kStages;
    R.empty = s.bars + kWarps * kStages + warp * kStages;
    return R;
}

__device__ inline void init_rings(const Smem& s) {
    if (threadIdx.x < 2 * kWarps * kStages) mbar_init(s.bars + threadIdx.x, 1);
    for (int i = threadIdx.x; i < kZeroBytes / 16; i += blockDim.x) reinterpret_cast<uint4*>(s.zero)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_barrier_init();
    __syncthreads();
}

// ------------------------------------------------------------------ CTA-wide stages

// A TMA instruction occupies its issuing thread for a few hundred nanoseconds whatever the box size,
// so small per-warp boxes cannot keep up with HBM, and the issuing must stay off the consumers'
// path. The MoE kernels stage one large box per step for the whole CTA: FP2/FP3 boxes of 256 rows
// (20 and 28 KB), FP4 boxes of 64 rows (17 KB), in a ring of NS slots of SB bytes filled by one
// producer thread (warp kLWarps). All kLWarps consumer warps read every stage:
//   FP2/FP3 box: warp w decodes rows [16 kLTiles w, +16 kLTiles) (kLTiles 16-row tiles), all 4 chunks.
//   FP4 box: warp w decodes rows [16 (w % 4), +16), chunks 8 / kFp4Parts consecutive from
//   (8 / kFp4Parts) (w / 4); the kFp4Parts partial sums of a row (warps w % 4, w % 4 + 4, ...) are
//   added in warp order at the end of the task.
constexpr int kCtaRing = 143360;  // 7 x 20480 (FP2 boxes) = 5 x 28672 (FP3 boxes)

__host__ __device__ constexpr int stage_rows(int fmt) { return fmt == 4 ? 64 : 256; }
__host__ __device__ constexpr int stage_bytes(int fmt) { return box_bytes(fmt) * stage_rows(fmt); }
// weights of a row covered by one box
__host__ __device__ constexpr int stage_k(int fmt) { return 64 * box_chunks(fmt); }
static_assert(stage_rows(2) == 16 * kLTiles * kLWarps && stage_rows(4) == 64, "rows per warp");

template <int NS, int SB>
struct CtaRing {
    static_assert(NS * SB <= kCtaRing && SB % 128 == 0 && NS <= 8, "ring geometry");
    static constexpr int kBytes = NS * SB;
    uint8_t* slots;
    uint64_t* full;   // arrival count 1 (the producer's expect_tx) + the box's transaction bytes
    uint64_t* empty;  // arrival count kLWarps

    __device__ __forceinline__ uint8_t* slot(uint32_t n) const { return slots + (size_t)(n % NS) * SB; }
    __device__ __forceinline__ uint64_t* bar(uint32_t n) const { return full + (n % NS); }

    // Consumer warp: waits for stage n. The result is the same on all 32 lanes; on timeout lane 0
    // flags FPX_ETIMEOUT.
    __device__ __forceinline__ bool wait(uint32_t n, int32_t* st) const {
        const bool ok = __any_sync(0xffffffffu, mbar_wait(full + (n % NS), (n / NS) & 1u, ring_wait_ns()));
        if (!ok && (threadIdx.x & 31) == 0) flag(st, FPX_ETIMEOUT);
        return ok;
    }

    // Consumer warp: done with stage n.
    __device__ __forceinline__ void release(uint32_t n) const {
        __syncwarp();
        if ((threadIdx.x & 31) == 0) mbar_arrive(empty + (n % NS));
    }

    // Consumer position (slot index n % NS and phase (n / NS) & 1 of stage n), advanced
    // incrementally so the hot loops need no division.
    struct Pos {
        uint32_t idx, ph;
    };
    __device__ __forceinline__ void next(Pos& p) const {
        if (++p.idx == (uint32_t)NS) { p.idx = 0; p.ph ^= 1u; }
    }
    __device__ __forceinline__ uint32_t slot_at(const Pos& p) const { return smem_u32(slots) + p.idx * (uint32_t)SB; }
    // Whole consumer warp: waits (bounded) for the stage at p; false on a timeout.
    __device__ __forceinline__ bool wait_at(const Pos& p) const { return mbar_wait_warp(smem_u32(full) + p.idx * 8u, p.ph); }

    __device__ __forceinline__ void release_at(const Pos& p) const {
        __syncwarp();
        if ((threadIdx.x & 31) == 0) mbar_arrive_u32(smem_u32(empty) + p.idx * 8u);
    }

    // Producer: waits (bounded by ring_wait_ns()) until stage n's slot is free, i.e. every consumer
    // released n - NS.
    __device__ __forceinline__ bool acquire(uint32_t n) const {
        return n < (uint32_t)NS || mbar_try_wait(empty + (n % NS), ((n / NS) + 1u) & 1u) ||
               mbar_wait(empty + (n % NS), ((n / NS) + 1u) & 1u, ring_wait_ns());
    }

    // Producer, before exiting: waits (bounded) for the copies of the last stages it issued, so that
    // no copy lands after the CTA is gone even if the consumers gave up.
    __device__ void drain(uint32_t issued) const {
        for (uint32_t n = issued > (uint32_t)NS ? issued - NS : 0u; n < issued; n++)
            if (!mbar_wait(full + (n % NS), (n / NS) & 1u)) return;
    }
};

struct CtaSmem {
    uint8_t* ring;
    uint64_t* bars;  // 256 bytes: full[NS], empty[NS], then (at bars + 16) the tables' barrier
    uint2* zero;     // kZeroBytes of zeros
    float* red;      // kLWarps * 64 floats: cross-warp partial sums
    uint8_t* tabs;   // activation tables, copied from global memory
    uint64_t* tbar;
};

constexpr int kRedBytes = kLWarps * 64 * 4;

// ring (ring_bytes), barriers, zero area, reduction area, tables (tab_bytes), alignment slack
__host__ __device__ constexpr size_t cta_smem_bytes(int ring_bytes, int tab_bytes) {
    return (size_t)ring_bytes + 256 + kZeroBytes + 32 + kRedBytes + (size_t)tab_bytes + 128;
}

__device__ __forceinline__ CtaSmem cta_carve(uint8_t* raw, int ring_bytes) {
    uint8_t* base = raw + ((128u - (smem_u32(raw) & 127u)) & 127u);
    CtaSmem s;
    size_t o = ring_bytes;
    s.ring = base;
    s.bars = reinterpret_cast<uint64_t*>(base + o); o += 256;
    s.tbar = s.bars + 16;
    // the zero area starts 16 bytes past a 32-byte boundary, so the broadcast zero reads of inactive
    // lanes use other banks than the active lanes' table entries (32-byte aligned)
    s.zero = reinterpret_cast<uint2*>(base + o + 16); o += kZeroBytes + 32;
    s.red = reinterpret_cast<float*>(base + o); o += kRedBytes;
    s.tabs = base + o;  // 32-byte aligned (ring_bytes, the areas above are multiples of 32)
    return s;
}

template <int NS, int SB>
__device__ inline CtaRing<NS, SB> cta_init(const CtaSmem& s) {
    CtaRing<NS, SB> R{s.ring, s.bars, s.bars + NS};
    if (threadIdx.x < NS) mbar_init(R.full + threadIdx.x, 1);
    else if (threadIdx.x < 2 * NS) mbar_init(R.empty + (threadIdx.x - NS), kLWarps);
    else if (threadIdx.x == 2 * NS) mbar_init(s.tbar, 1);
    for (int i = threadIdx.x; i < kZeroBytes / 16; i += blockDim.x) reinterpret_cast<uint4*>(s.zero)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_barrier_init();
    __syncthreads();
    return R;
}

// ------------------------------------------------------------------ box-internal layout

// The layer kernels' FP2 and FP3 boxes are regrouped by the tiling transform (fpx_tile_matrices) so
// that one thread reads its code words for all four chunks of a row with one or three loads and the
// scales of a row with one load, and FP3 codes sit as contiguous 3-bit fields c = l + 4h (one MMA plane
// instead of a low and a high plane). Thread t of a row decodes, for chunk C = 0..3, block 2C + t/2,
// codes 16 (t % 2) + j (j = 0..15); pair p holds codes j = p (low binary16 half) and p + 8 (high half).
//   FP2 box: codes [256 rows x 64 B]: word 4t + C of a row = code word t % 2 of block 2C + t / 2 (the
//            row-major block's bytes 2 + 4 (t % 2) .. +3); scales [256 rows x 16 B].
//   FP3 box: codes [256 rows x 96 B]: bytes 24t .. 24t + 23 of a row = words W0..W5; chunk pair
//            (2m, 2m + 1) uses W3m..W3m+2 with the field positions of fp3_slot; scales as FP2.
//   Scales: binary16 4h + C of a row = the scale of block 2C + h.
// FP4 boxes keep the row-major bytes.
__host__ __device__ constexpr int box_code_bytes(int fmt) { return fmt == 2 ? 64 : 96; }  // per box row
__host__ __device__ constexpr int box_scale_offset(int fmt) { return 256 * box_code_bytes(fmt); }

// Sixteen A pairs (two chunks) from the three words of a chunk pair, one LOP3 per pair (plus four
// shifts): value 1024 + c 2^P with c the 3-bit code and P = fp3_box_shift.
__device__ __forceinline__ void decode_fp3_box(uint32_t W0, uint32_t W1, uint32_t W2, uint32_t magic, uint32_t (&a)[8],
                                               uint32_t (&b)[8]) {
    const uint32_t u0 = W0 >> 9, u1 = W1 >> 9, u2 = W2 >> 9;
    a[0] = (W0 & 0x000E000Eu) | magic;
    a[1] = (W0 & 0x00700070u) | magic;
    a[2] = (W0 & 0x03800380u) | magic;
    a[3] = (u0 & 0x000E000Eu) | magic;
    a[4] = (u0 & 0x00700070u) | magic;
    a[5] = (W1 & 0x000E000Eu) | magic;
    a[6] = (W1 & 0x00700070u) | magic;
    a[7] = (W1 & 0x03800380u) | magic;
    b[0] = (u1 & 0x000E000Eu) | magic;
    b[1] = (u1 & 0x00700070u) | magic;
    b[2] = (W2 & 0x000E000Eu) | magic;
    b[3] = (W2 & 0x00700070u) | magic;
    b[4] = (W2 & 0x03800380u) | magic;
    b[5] = (u2 & 0x000E000Eu) | magic;
    b[6] = (u2 & 0x00700070u) | magic;
    b[7] = (((W0 << 1) & 0x00020002u) | ((W1 << 2) & 0x00040004u)) | (((W2 << 3) & 0x00080008u) | magic);
}

template <int OFF>
__device__ __forceinline__ uint2 lds64(uint32_t a) {
    uint2 v;
    asm volatile("ld.shared.v2.b32 {%0,%1}, [%2+%3];" : "=r"(v.x), "=r"(v.y) : "r"(a), "n"(OFF));
    return v;
}

// Scale of chunk C from a thread's four binary16 scales (chunks 0..3).
template <int C>
__device__ __forceinline__ float scale_of(const uint2& s) {
    const uint32_t w = C < 2 ? s.x : s.y;
    const __half2 h = *reinterpret_cast<const __half2*>(&w);
    return (C & 1) ? __high2float(h) : __low2float(h);
}

// One consumer warp's share of a staged FP2/FP3 box (rows g and g + 8 of its two 16-row tiles): the
// code words and scales, loaded in one pass so the ring slot can be released before the MMAs run.
template <int FMT, int NT>
struct Frag;
template <int NT>
struct Frag<2, NT> {
    uint4 c[NT][2];  // [tile][row g / g + 8]: words of chunks 0..3
    uint2 s[NT][2];
};
template <int NT>
struct Frag<3, NT> {
    uint2 c[NT][2][3];  // words W0..W5
    uint2 s[NT][2];
};

// `row` = the warp's first row + g; t = lane % 4.
template <int FMT, int NT>
__device__ __forceinline__ void frag_load(Frag<FMT, NT>& f, uint32_t slot, int row, int t) {
    constexpr int CB = box_code_bytes(FMT);
    const uint32_t cb = slot + (uint32_t)(row * CB + (FMT == 2 ? 16 : 24) * t);
    const uint32_t sb = slot + (uint32_t)(box_scale_offset(FMT) + row * 16 + 8 * (t >> 1));
#pragma unroll
    for (int i = 0; i < NT; i++) {
#pragma unroll
        for (int h = 0; h < 2; h++) {
            const uint32_t r = (uint32_t)(16 * i + 8 * h);
            if constexpr (FMT == 2) {
                f.c[i][h] = lds128<0>(cb + r * CB);
            } else {
                f.c[i][h][0] = lds64<0>(cb + r * CB);
                f.c[i][h][1] = lds64<8>(cb + r * CB);
                f.c[i][h][2] = lds64<16>(cb + r * CB);
            }
            f.s[i][h] = lds64<0>(sb + r * 16);
        }
    }
}

template <int C>
__device__ __forceinline__ uint32_t word_of(const uint4& c) {
    return C == 0 ? c.x : C == 1 ? c.y : C == 2 ? c.z : c.w;
}

// MMAs of chunk C of both tiles: B registers from the lane's table entry b (32 bytes per chunk, 512
// bytes per chunk in the table) and the offset quad from oq (64 bytes per chunk).
__device__ __forceinline__ void chunk_mma(float (&acc)[4], const uint32_t (&a0)[8], const uint32_t (&a8)[8], const uint4& b0,
                                          const uint4& b1, const float4& c4) {
    // two accumulator chains (K steps 0, 2 and 1, 3) joined at the end: half the dependent MMA latency
    float acc2[4];
    mma_c(acc, a0[0], a8[0], a0[1], a8[1], b0.x, b0.y, c4);
    mma_c(acc2, a0[2], a8[2], a0[3], a8[3], b0.z, b0.w, make_float4(0.f, 0.f, 0.f, 0.f));
    mma_acc(acc, a0[4], a8[4], a0[5], a8[5], b1.x, b1.y);
    mma_acc(acc2, a0[6], a8[6], a0[7], a8[7], b1.z, b1.w);
    acc[0] += acc2[0]; acc[1] += acc2[1]; acc[2] += acc2[2]; acc[3] += acc2[3];
}

template <int C>
__device__ __forceinline__ float4 oq_quad(uint32_t oq) {
    const uint4 q = lds128<C * 64>(oq);
    return make_float4(__uint_as_float(q.x), __uint_as_float(q.y), __uint_as_float(q.z), __uint_as_float(q.w));
}

// Chunks C0 and C0 + 1 of a fragment, accumulated into y[tile][4] (rows g, g + 8 as in box_tiles).
template <int FMT, int C0, int NT>
__device__ __forceinline__ void frag_mma(const Frag<FMT, NT>& f, uint32_t b, uint32_t oq, uint32_t magic, float (&y)[NT][4]) {
    const uint4 b0 = lds128<C0 * 512>(b), b1 = lds128<C0 * 512 + 16>(b);
    const uint4 e0 = lds128<(C0 + 1) * 512>(b), e1 = lds128<(C0 + 1) * 512 + 16>(b);
    const float4 q0 = oq_quad<C0>(oq), q1 = oq_quad<C0 + 1>(oq);
#pragma unroll
    for (int i = 0; i < NT; i++) {
        uint32_t a0[8], a8[8], c0[8], c8[8];
        if constexpr (FMT == 2) {
            decode_fp2(word_of<C0>(f.c[i][0]), magic, a0);
            decode_fp2(word_of<C0>(f.c[i][1]), magic, a8);
            decode_fp2(word_of<C0 + 1>(f.c[i][0]), magic, c0);
            decode_fp2(word_of<C0 + 1>(f.c[i][1]), magic, c8);
        } else {
            constexpr int m = C0 / 2;
            const uint32_t x0[6] = {f.c[i][0][0].x, f.c[i][0][0].y, f.c[i][0][1].x, f.c[i][0][1].y, f.c[i][0][2].x, f.c[i][0][2].y};
            const uint32_t x8[6] = {f.c[i][1][0].x, f.c[i][1][0].y, f.c[i][1][1].x, f.c[i][1][1].y, f.c[i][1][2].x, f.c[i][1][2].y};
            decode_fp3_box(x0[3 * m], x0[3 * m + 1], x0[3 * m + 2], magic, a0, c0);
            decode_fp3_box(x8[3 * m], x8[3 * m + 1], x8[3 * m + 2], magic, a8, c8);
        }
        float acc[4], acd[4];
        chunk_mma(acc, a0, a8, b0, b1, q0);
        chunk_mma(acd, c0, c8, e0, e1, q1);
        const float d0 = scale_of<C0>(f.s[i][0]), d8 = scale_of<C0>(f.s[i][1]);
        const float f0 = scale_of<C0 + 1>(f.s[i][0]), f8 = scale_of<C0 + 1>(f.s[i][1]);
        y[i][0] = fmaf(f0, acd[0], fmaf(d0, acc[0], y[i][0]));
        y[i][1] = fmaf(f0, acd[1], fmaf(d0, acc[1], y[i][1]));
        y[i][2] = fmaf(f8, acd[2], fmaf(d8, acc[2], y[i][2]));
        y[i][3] = fmaf(f8, acd[3], fmaf(d8, acc[3], y[i][3]));
    }
}

// Runs stages s_first .. s_end - 1 of one FP2/FP3 task (ring positions p, p + 1, ...) through a
// double-buffered fragment: the next stage's words are loaded between the two halves of the current
// stage's MMAs, and a stage's slot is released as soon as its words are in registers. b / q: the
// lane's table entry and offset quad addresses for the task's stage s_first (advanced by b_step and
// 256 bytes per stage). On a timeout the warp stops waiting and releasing (so the producer gives up
// too) and ok turns false; the caller reports it.
template <int FMT, int NT, class RING>
__device__ __forceinline__ bool frag_step(const RING& R, const Frag<FMT, NT>& cur, Frag<FMT, NT>& nxt, typename RING::Pos& p,
                                          int& left, int row, int t, uint32_t& b, uint32_t b_step, uint32_t& q, uint32_t magic,
                                          float (&y)[NT][4], bool& ok) {
    if (ok) R.release_at(p);
    R.next(p);
    const bool more = --left > 0;
    frag_mma<FMT, 0, NT>(cur, b, q, magic, y);
    if (more && ok) {
        ok = R.wait_at(p);
        if (ok) frag_load<FMT, NT>(nxt, R.slot_at(p), row, t);
    }
    frag_mma<FMT, 2, NT>(cur, b, q, magic, y);
    b += b_step;
    q += 256u;
    return more;
}

template <int FMT, int NT, class RING>
__device__ __forceinline__ void frag_stages(const RING& R, typename RING::Pos& p, int count, int row, int t, uint32_t b,
                                            uint32_t b_step, uint32_t q, uint32_t magic, float (&y)[NT][4], bool& ok) {
    Frag<FMT, NT> fa, fb;
    if (ok) ok = R.wait_at(p);
    if (ok) frag_load<FMT, NT>(fa, R.slot_at(p), row, t);
    int left = count;
    while (frag_step<FMT, NT>(R, fa, fb, p, left, row, t, b, b_step, q, magic, y, ok) &&
           frag_step<FMT, NT>(R, fb, fa, p, left, row, t, b, b_step, q, magic, y, ok)) {
    }
}

// Adds the kFp4Parts FP4 partial sums of each row (warps w % 4, w % 4 + 4, ...) in warp order. Every
// consumer warp calls it with its pair-reduced y; afterwards warps 0..3 hold the sums. Contains two
// consumer barriers.
__device__ inline void fp4_reduce(float* red, float (&y)[4]) {
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    if (warp >= 4 && t < 2)
#pragma unroll
        for (int i = 0; i < 4; i++) red[(warp - 4) * 64 + (g + 8 * (i >> 1)) * 4 + 2 * t + (i & 1)] = y[i];
    layer_sync();
    if (warp < 4 && t < 2)
#pragma unroll
        for (int i = 0; i < 4; i++)
#pragma unroll
            for (int pp = 1; pp < kFp4Parts; pp++) y[i] += red[(warp + 4 * (pp - 1)) * 64 + (g + 8 * (i >> 1)) * 4 + 2 * t + (i & 1)];
    layer_sync();
}

}  // namespace fpx
