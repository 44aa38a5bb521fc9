// Batched speculative verify/commit over B sequences: the target scored q positions of each (the seed
// and q - 1 draft tokens) in one pass; drafts are accepted while they equal the target's own choice
// at the previous position, and the first mismatch (or the position after an all-accepted draft) takes
// the target's choice. "DeepSeek V4 Flash hits 32 tok/s on AMD Ryzen AI MAX+ 395", paragraph 3 (four
// positions including the seed verified in one pass; correct proposals commit, the first error is
// corrected by the target), and the zh-TW page, section "DSpark" (Propose / Verify / Commit).
//
// k_row_argmax: one CTA per (sequence, position): the largest logit of the row, lowest index among
// equal maxima, NaN never chosen (an all-NaN row gives index 0 and FPX_ERANGE). Reads the logits once
// with 16-byte loads when the rows allow it: HBM-bound.
// k_commit: one thread per sequence.
#include "fpx_common.cuh"

using namespace fpx;

namespace {

constexpr int kArgThreads = 512;

struct Best {
    float v;
    int i;  // -1: none yet
};

__device__ __forceinline__ Best better(Best a, Best b) {
    if (b.i < 0) return a;
    if (a.i < 0) return b;
    if (b.v > a.v || (b.v == a.v && b.i < a.i)) return b;
    return a;
}

__device__ __forceinline__ void take(Best& b, float x, int i) {  // visited in increasing index order
    if (x == x && (b.i < 0 || x > b.v)) { b.v = x; b.i = i; }
}

__global__ void __launch_bounds__(kArgThreads) k_row_argmax(const float* __restrict__ logits, int V, int32_t* pred,
                                                            int32_t* status) {
    __shared__ Best red[kArgThreads / 32];
    const size_t r = blockIdx.x;
    const float* row = logits + r * (size_t)V;
    Best b{0.f, -1};
    const bool vec = (V % 4) == 0 && ((reinterpret_cast<uintptr_t>(row) & 15) == 0);
    if (vec) {
        const float4* r4 = reinterpret_cast<const float4*>(row);
        const int n4 = V / 4;
        for (int i = threadIdx.x; i < n4; i += kArgThreads) {
            const float4 x = __ldcs(r4 + i);
            take(b, x.x, 4 * i); take(b, x.y, 4 * i + 1); take(b, x.z, 4 * i + 2); take(b, x.w, 4 * i + 3);
        }
    } else {
        for (int i = threadIdx.x; i < V; i += kArgThreads) take(b, __ldcs(row + i), i);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        Best o2{__shfl_xor_sync(0xffffffffu, b.v, o), __shfl_xor_sync(0xffffffffu, b.i, o)};
        b = better(b, o2);
    }
    if ((threadIdx.x & 31) == 0) red[threadIdx.x / 32] = b;
    __syncthreads();
    if (threadIdx.x == 0) {
        Best m = red[0];
        for (int w = 1; w < kArgThreads / 32; w++) m = better(m, red[w]);
        if (m.i < 0) {
            m.i = 0;
            if (status) flag(status, FPX_ERANGE);
        }
        pred[r] = m.i;
    }
}

__global__ void k_commit(const int32_t* __restrict__ pred, const int32_t* __restrict__ drafts, int B, int q,
                         int32_t* n_accept, int32_t* committed) {
    const int s = blockIdx.x * blockDim.x + threadIdx.x;
    if (s >= B) return;
    const int32_t* p = pred + (size_t)s * q;
    const int32_t* d = drafts + (size_t)s * (q - 1);
    int n = 0;
    while (n < q - 1 && d[n] == p[n]) n++;
    n_accept[s] = n;
    for (int i = 0; i < q; i++) committed[(size_t)s * q + i] = i < n ? d[i] : (i == n ? p[n] : -1);
}

}  // namespace

extern "C" int dspark_verify_commit(const float* logits, int B, int q, int V, const int32_t* drafts, int32_t* pred,
                                    int32_t* n_accept, int32_t* committed, int32_t* dev_status, void* stream) {
    if (B < 0 || q < 1 || q > 16 || V < 1 || (int64_t)B * q > INT32_MAX) return FPX_EINVAL;
    if (B == 0) return FPX_OK;
    if (!logits || !pred || !n_accept || !committed || (q > 1 && !drafts)) return FPX_EINVAL;
    if (!aligned(logits, 4) || !aligned(pred, 4) || !aligned(n_accept, 4) || !aligned(committed, 4) ||
        (drafts && !aligned(drafts, 4)))
        return FPX_EALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    k_row_argmax<<<(unsigned)(B * q), kArgThreads, 0, s>>>(logits, V, pred, dev_status);
    k_commit<<<(B + 127) / 128, 128, 0, s>>>(pred, drafts, B, q, n_accept, committed);
    return launch_status();
}
