// Shared device helpers of libfpx.so: block layouts, status word, reductions, launch helpers.
//
// Block layouts (a reading of the ROCmFPX paragraph of "DeepSeek V4 Flash hits 32 tok/s on AMD Ryzen
// AI MAX+ 395", which fixes only 32 weights per block and 10 B / 3.50 bpw / 4.25 bpw):
//   FP2 10 B: binary16 d | codes c_j at bits 2j..2j+1            w = d (2c - 3)
//   FP3 14 B: binary16 d | low bits l_j (bits 2j..) | high bits h_j (bit j)   c = l + 4h, w = d (2c - 7)
//   FP4 17 B: E8M0 e | E2M1 codes at bits 4j..4j+3              w = 2^(e-127) * e2m1(q)
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "../../include/fpx.h"

namespace fpx {

constexpr int kWarp = 32;

__host__ __device__ constexpr int block_bytes(int fmt) {
    return fmt == 2 ? 10 : fmt == 3 ? 14 : fmt == 4 ? 17 : 0;
}

inline int64_t matrix_bytes(int fmt, int64_t N, int64_t K) {
    int bb = block_bytes(fmt);
    if (!bb || N < 0 || K < 0 || K % 32) return -1;
    return (N * (K / 32) * bb + 15) / 16 * 16;
}

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Records status `code` as bit (1 << code) of the device status word (nullable).
__device__ __forceinline__ void flag(int32_t* st, int code) {
    if (st) atomicOr(st, 1 << code);
}

// Sum over the 32 lanes with a fixed xor butterfly; every lane ends with the same value.
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// E2M1 magnitude of a 3-bit index: {0, .5, 1, 1.5, 2, 3, 4, 6}.
__device__ __forceinline__ float e2m1_mag(int m) {
    // exponent field m >> 1 (bias 1), significand bit m & 1; field 0 is subnormal (0.5 * M)
    int E = m >> 1, M = m & 1;
    return E == 0 ? 0.5f * M : ldexpf(1.0f + 0.5f * M, E - 1);
}

// Decodes one block (CUDA-core path). Sets v[j] to the integer or E2M1 level of weight j and
// returns the block scale, so that w_j = scale * v[j] exactly. p is 2-byte aligned for FP2/FP3.
template <int FMT>
__device__ __forceinline__ float decode_levels(const uint8_t* __restrict__ p, float (&v)[32], int32_t* st) {
    if constexpr (FMT == 2 || FMT == 3) {
        const uint16_t* h = reinterpret_cast<const uint16_t*>(p);
        float d = __half2float(__ushort_as_half(__ldg(h)));
        uint32_t c0 = __ldg(h + 1) | (static_cast<uint32_t>(__ldg(h + 2)) << 16);
        uint32_t c1 = __ldg(h + 3) | (static_cast<uint32_t>(__ldg(h + 4)) << 16);
        if constexpr (FMT == 2) {
#pragma unroll
            for (int j = 0; j < 16; j++) {
                v[j] = static_cast<float>(2 * static_cast<int>((c0 >> (2 * j)) & 3u) - 3);
                v[16 + j] = static_cast<float>(2 * static_cast<int>((c1 >> (2 * j)) & 3u) - 3);
            }
        } else {
            uint32_t hb = __ldg(h + 5) | (static_cast<uint32_t>(__ldg(h + 6)) << 16);
#pragma unroll
            for (int j = 0; j < 32; j++) {
                uint32_t lo = ((j < 16 ? c0 : c1) >> (2 * (j & 15))) & 3u;
                uint32_t c = lo | (((hb >> j) & 1u) << 2);
                v[j] = static_cast<float>(2 * static_cast<int>(c) - 7);
            }
        }
        return d;
    } else {
        int e = __ldg(p);
        if (e == 255) {
            flag(st, FPX_EDATA);
#pragma unroll
            for (int j = 0; j < 32; j++) v[j] = 0.0f;
            return 0.0f;
        }
#pragma unroll
        for (int j = 0; j < 16; j++) {
            uint32_t byte = __ldg(p + 1 + j);
            uint32_t q0 = byte & 15u, q1 = byte >> 4;
            float m0 = e2m1_mag(q0 & 7), m1 = e2m1_mag(q1 & 7);
            v[2 * j] = (q0 & 8) ? -m0 : m0;
            v[2 * j + 1] = (q1 & 8) ? -m1 : m1;
        }
        return ldexpf(1.0f, e - 127);
    }
}

// Padded shared-memory layout for activations used by the CUDA-core path: element k of a column
// lives at (k / 32) * 33 + k % 32, so lanes reading the same position of consecutive blocks hit
// distinct banks.
__host__ __device__ constexpr int padded_len(int K) { return (K / 32) * 33; }
__device__ __forceinline__ int padded_index(int k) { return (k >> 5) * 33 + (k & 31); }

// Activation readers for row_dot: padded binary32 columns in shared memory, or the caller's [Q][K]
// array in global memory (binary32 or bfloat16) when the columns do not fit in shared memory.
struct XShared {
    const float* xs;
    int stride;
    __device__ __forceinline__ float operator()(int t, int b, int j) const { return xs[t * stride + b * 33 + j]; }
};
struct XGlobal {
    const void* x;
    int K;
    int bf16;
    __device__ __forceinline__ float operator()(int t, int b, int j) const {
        const int64_t i = (int64_t)t * K + b * 32 + j;
        return bf16 ? bf16_bits_to_float(__ldg(reinterpret_cast<const uint16_t*>(x) + i))
                    : __ldg(reinterpret_cast<const float*>(x) + i);
    }
};

// Dot products of one packed row (nblk blocks at `row`) with Q activation columns. One warp; lane l
// takes blocks l, l+32, ...; per block the level-times-activation products are chained in j order,
// scaled once, and the lanes are summed with a fixed butterfly. The order depends on neither Q, the
// other columns, nor where the activations are read from.
template <int FMT, int Q, class XR>
__device__ __forceinline__ void row_dot(const uint8_t* __restrict__ row, int nblk, const XR& xr, int lane,
                                        float (&acc)[Q], int32_t* st) {
#pragma unroll
    for (int t = 0; t < Q; t++) acc[t] = 0.0f;
    for (int b = lane; b < nblk; b += kWarp) {
        float v[32];
        float s = decode_levels<FMT>(row + static_cast<int64_t>(b) * block_bytes(FMT), v, st);
#pragma unroll
        for (int t = 0; t < Q; t++) {
            float part = 0.0f;
#pragma unroll
            for (int j = 0; j < 32; j++) part = fmaf(v[j], xr(t, b, j), part);
            acc[t] = fmaf(s, part, acc[t]);
        }
    }
#pragma unroll
    for (int t = 0; t < Q; t++) acc[t] = warp_sum(acc[t]);
}

struct DeviceInfo {
    int sms;
    int smem_optin;
};

inline DeviceInfo device_info() {
    int dev = 0;
    cudaGetDevice(&dev);
    DeviceInfo d{148, 227 * 1024};
    cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    return d;
}

inline int launch_status() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? FPX_OK : FPX_ECUDA;
}

}  // namespace fpx
