// Device twin of the synthetic input generator described in synth.h: packed blocks only.
// Written independently of synth.c from the same published definition; a GPU test checks that
// both produce identical bytes. Holds none of the decode/GEMV/routing/quantization arithmetic.
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

namespace {

constexpr uint64_t kG = 0x9E3779B97F4A7C15ull;
constexpr int kThreads = 256;

__host__ __device__ inline uint64_t mix(uint64_t z) {
    z ^= z >> 30; z *= 0xBF58476D1CE4E5B9ull;
    z ^= z >> 27; z *= 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

__host__ __device__ inline uint64_t make_key(uint64_t seed, uint64_t layer, uint64_t tensor, uint64_t expert) {
    uint64_t a = mix(seed + kG);
    uint64_t b = mix(a + layer * kG + tensor);
    return mix(b ^ ((expert + 1) * 0xC2B2AE3D27D4EB4Full));
}

__device__ inline uint64_t rnd(uint64_t key, uint64_t i) { return mix(key + (i + 1) * kG); }

__device__ inline int block_bytes(int fmt) { return fmt == 2 ? 10 : fmt == 3 ? 14 : 17; }

// Writes the bytes of block `b` into p (bb bytes).
__device__ void make_block(int fmt, uint64_t key, uint64_t b, uint8_t* p) {
    double u = (double)(rnd(key, 4 * b) >> 11) * 0x1p-53;
    double s = __dadd_rn(0.005, __dmul_rn(0.045, u));
    __half h = __double2half(s);
    uint16_t hb = __half_as_ushort(h);
    uint64_t r1 = rnd(key, 4 * b + 1), r2 = rnd(key, 4 * b + 2);
    int off;
    if (fmt == 4) {
        double sv = (double)__half2float(h);
        int e2;
        frexp(sv, &e2);
        int fl = e2 - 1;
        int k = (sv * sv < ldexp(1.0, 2 * fl + 1)) ? fl : fl + 1;
        p[0] = (uint8_t)(127 + k);
        off = 1;
    } else {
        p[0] = (uint8_t)(hb & 0xFF);
        p[1] = (uint8_t)(hb >> 8);
        off = 2;
    }
    int nc = block_bytes(fmt) - off;
    for (int k = 0; k < nc; k++) p[off + k] = (uint8_t)(k < 8 ? (r1 >> (8 * k)) : (r2 >> (8 * (k - 8))));
}

// grid.y enumerates matrices (experts); matrix m uses key(seed, layer, tensor, expert0 + m) and
// lives at out + m * stride. grid.x * kThreads blocks per launch chunk, looped.
__global__ void k_synth(int fmt, uint64_t seed, uint64_t layer, uint64_t tensor, uint64_t expert0,
                        int64_t nblocks, int64_t stride, uint8_t* out) {
    __shared__ __align__(16) uint8_t stage[kThreads * 17];
    const int bb = block_bytes(fmt);
    const uint64_t key = make_key(seed, layer, tensor, expert0 + blockIdx.y);
    uint8_t* dst = out + (int64_t)blockIdx.y * stride;
    for (int64_t base = (int64_t)blockIdx.x * kThreads; base < nblocks; base += (int64_t)gridDim.x * kThreads) {
        int64_t b = base + threadIdx.x;
        if (b < nblocks) make_block(fmt, key, (uint64_t)b, stage + threadIdx.x * bb);
        __syncthreads();
        int64_t nb = nblocks - base < kThreads ? nblocks - base : kThreads;
        int64_t bytes = nb * bb;
        uint8_t* d = dst + base * bb;
        if (nb == kThreads && ((reinterpret_cast<uintptr_t>(d) & 15) == 0)) {
            for (int64_t v = threadIdx.x; v < bytes / 16; v += kThreads)
                reinterpret_cast<uint4*>(d)[v] = reinterpret_cast<const uint4*>(stage)[v];
        } else {
            for (int64_t v = threadIdx.x; v < bytes; v += kThreads) d[v] = stage[v];
        }
        __syncthreads();
    }
    // zero the pad bytes up to the 16-byte storage size
    if (blockIdx.x == 0) {
        int64_t bytes = nblocks * bb, padded = (bytes + 15) / 16 * 16;
        for (int64_t v = bytes + threadIdx.x; v < padded; v += kThreads) dst[v] = 0;
    }
}

}  // namespace

extern "C" {

// Fills `count` consecutive N x K matrices (experts expert0 .. expert0+count-1) at out, each of
// storage size `stride` bytes (>= the padded matrix size). Returns 0 or a CUDA error code.
int synth_dev_matrices(int fmt, uint64_t seed, uint64_t layer, uint64_t tensor, uint64_t expert0,
                       int count, int64_t N, int64_t K, uint8_t* out, int64_t stride, cudaStream_t s) {
    if (fmt < 2 || fmt > 4 || N < 0 || K < 0 || K % 32 || count < 0 || count > 65535) return -1;
    int64_t nblocks = N * (K / 32);
    int bb = fmt == 2 ? 10 : fmt == 3 ? 14 : 17;
    if (stride < (nblocks * bb + 15) / 16 * 16) return -1;
    if (count == 0 || nblocks == 0) return 0;
    int64_t gx = (nblocks + kThreads - 1) / kThreads;
    if (gx > 4096) gx = 4096;
    k_synth<<<dim3((unsigned)gx, (unsigned)count), kThreads, 0, s>>>(fmt, seed, layer, tensor, expert0, nblocks, stride, out);
    return (int)cudaGetLastError();
}

uint64_t synth_dev_key(uint64_t seed, uint64_t layer, uint64_t tensor, uint64_t expert) {
    return make_key(seed, layer, tensor, expert);
}

}  // extern "C"
