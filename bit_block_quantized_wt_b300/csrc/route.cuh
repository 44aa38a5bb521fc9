// Warp-level top-k over one token's router logits, shared by the decode router and the prefill
// routing kernels: the TOP_K step of "DeepSeek V4 Flash hits 32 tok/s on AMD Ryzen AI MAX+ 395",
// paragraph 3, and "Token Freedom via APU: ...", section "Lucebox's Optimization Trio" (top-k by
// logit, sigmoid gate weights renormalised over the selected experts).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace fpx {

constexpr int kRouteMaxK = 8;      // experts per token
constexpr int kRouteMaxE = 1024;   // routed experts per layer

// Warp-level top-k of lg[0..E) (descending, ties to the lower index), with sigmoid weights
// normalised over the selected k: lane r < k writes idx[r] and w[r]. Each lane keeps its E / 32 logits
// in registers (NM >= E / 32 slots).
template <int NM>
__device__ void warp_topk_n(const float* lg, int E, int k, int32_t* idx, float* w) {
    const int lane = threadIdx.x & 31;
    float v[NM];
#pragma unroll
    for (int m = 0; m < NM; m++) v[m] = lane + 32 * m < E ? __ldcg(lg + lane + 32 * m) : 0.0f;
    uint32_t taken = 0;  // bit m: element lane + 32 m already selected
    // rounds unrolled up to the largest k, so that the selected values stay in registers
    float sig[kRouteMaxK];
    int sel[kRouteMaxK];
#pragma unroll
    for (int r = 0; r < kRouteMaxK; r++) {
        if (r < k) {
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
            sel[r] = bi;
            sig[r] = 1.0f / (1.0f + expf(-bv));
        }
    }
    float S = sig[0];
#pragma unroll
    for (int r = 1; r < kRouteMaxK; r++)
        if (r < k) S += sig[r];
    if (lane < k) {  // lane r writes rank r
#pragma unroll
        for (int r = 0; r < kRouteMaxK; r++)
            if (r == lane) { idx[r] = sel[r]; w[r] = sig[r] / S; }
    }
}

__device__ inline void warp_topk(const float* lg, int E, int k, int32_t* idx, float* w) {
    if (E <= 256) warp_topk_n<8>(lg, E, k, idx, w);
    else warp_topk_n<kRouteMaxE / 32>(lg, E, k, idx, w);
}

}  // namespace fpx
