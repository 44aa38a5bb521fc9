"""Helpers for the GPU parity tests: device tensors, synthetic layers built by the device generator,
and host copies of the experts the oracle needs."""
import numpy as np
import pytest
import torch

import bit_block_quantized_wt_b300 as fpx
import synth


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def status_word():
    return torch.zeros(4, dtype=torch.int32, device="cuda")


def read_status(st):
    return fpx.fpx_read_status(st)


class DeviceLayer:
    """One MoE layer generated on the device with the seeded generator (layer index `layer`), its expert
    matrices rearranged into the box-tiled layout the layer kernels read. `scratch` (optional) is a
    uint8 device tensor of at least E * max(matrix bytes) used for the row-major copies."""

    def __init__(self, H, I, E, seed=0, layer=0, scratch=None):
        self.H, self.I, self.E, self.seed, self.layer = H, I, E, seed, layer
        self.mb_gu = fpx.fpx_matrix_bytes(2, I, H)
        self.mb_d = fpx.fpx_matrix_bytes(3, H, I)
        self.mb_s = fpx.fpx_matrix_bytes(4, I, H)
        self.gate = torch.empty(E * self.mb_gu, dtype=torch.uint8, device="cuda")
        self.up = torch.empty(E * self.mb_gu, dtype=torch.uint8, device="cuda")
        self.down = torch.empty(E * self.mb_d, dtype=torch.uint8, device="cuda")
        self.sh = [torch.empty(self.mb_s, dtype=torch.uint8, device="cuda") for _ in range(3)]
        need = E * max(self.mb_gu, self.mb_d)
        tmp = scratch if scratch is not None and scratch.numel() >= need else torch.empty(need, dtype=torch.uint8, device="cuda")
        s = torch.cuda.current_stream().cuda_stream
        for dst, fmt, tensor, count, N, K, mb in ((self.gate, 2, synth.GATE, E, I, H, self.mb_gu),
                                                 (self.up, 2, synth.UP, E, I, H, self.mb_gu),
                                                 (self.down, 3, synth.DOWN, E, H, I, self.mb_d),
                                                 (self.sh[0], 4, synth.SH_GATE, 1, I, H, self.mb_s),
                                                 (self.sh[1], 4, synth.SH_UP, 1, I, H, self.mb_s),
                                                 (self.sh[2], 4, synth.SH_DOWN, 1, H, I, self.mb_s)):
            synth.device_matrices(fmt, seed, layer, tensor, 0, count, N, K, tmp.data_ptr(), mb, s)
            fpx.fpx_tile_matrices(fmt, tmp, N, K, count, mb, dst, mb, 0, s)
        self.R_host = synth.router(E, H, seed, layer)
        self.router = dev(self.R_host)
        self.c = fpx.moe_layer(H=H, I=I, E=E, router=self.router.data_ptr(), gate=self.gate.data_ptr(),
                               up=self.up.data_ptr(), down=self.down.data_ptr(), sh_gate=self.sh[0].data_ptr(),
                               sh_up=self.sh[1].data_ptr(), sh_down=self.sh[2].data_ptr())

    def host_experts(self, experts):
        """Host copies (from the host generator) of the listed routed experts and the shared expert,
        as the oracle's E-length pointer lists."""
        H, I, E, seed, layer = self.H, self.I, self.E, self.seed, self.layer
        g, u, d = [None] * E, [None] * E, [None] * E
        for e in sorted(set(int(v) for v in experts)):
            g[e] = synth.matrix(2, I, H, seed, layer, synth.GATE, e)
            u[e] = synth.matrix(2, I, H, seed, layer, synth.UP, e)
            d[e] = synth.matrix(3, H, I, seed, layer, synth.DOWN, e)
        sg = synth.matrix(4, I, H, seed, layer, synth.SH_GATE)
        su = synth.matrix(4, I, H, seed, layer, synth.SH_UP)
        sd = synth.matrix(4, H, I, seed, layer, synth.SH_DOWN)
        return g, u, d, sg, su, sd

    def oracle(self, x, k, idx_force=None):
        import oracle
        experts = idx_force.ravel() if idx_force is not None else range(self.E)
        g, u, d, sg, su, sd = self.host_experts(experts)
        return oracle.moe_layer(self.H, self.I, self.E, self.R_host, g, u, d, sg, su, sd, x, k, idx_force=idx_force)


def topk_of(logits_row, k):
    """Top-k of one row (descending, ties to the lower index) by a stable sort on the negated value."""
    order = np.argsort(-np.asarray(logits_row, np.float64), kind="stable")
    return order[:k]


def routing_gap_ok(logits, k, bound):
    """True when the k-th and (k+1)-th largest logits of every row differ by more than `bound`, so the
    top-k set is unique within that error."""
    s = -np.sort(-logits, axis=1)
    if s.shape[1] <= k:
        return np.ones(s.shape[0], bool)
    return (s[:, k - 1] - s[:, k]) > bound


def f32_to_bf16_bits(x):
    """Round-to-nearest-even binary32 -> bfloat16 bits (finite inputs)."""
    b = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def wide_bf16(q, K, seed, spike_log2, block_span):
    """Activations with a wide dynamic range, as (bfloat16 bits [q][K], binary32 values [q][K]): N(0, 1)
    entries whose 32-entry blocks are scaled by 2^j, j uniform in [-block_span, block_span]; 5% +0,
    5% -0, 5% bfloat16 subnormals of either sign; and one spike of magnitude 2^spike_log2 per column."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((q, K))
    x *= np.repeat(2.0 ** rng.integers(-block_span, block_span + 1, size=(q, K // 32)), 32, axis=1)
    m = rng.random((q, K))
    x[m < 0.05] = 0.0
    x[(m >= 0.05) & (m < 0.10)] = -0.0
    sub = (m >= 0.10) & (m < 0.15)
    x[sub] = rng.choice([-1.0, 1.0], sub.sum()) * rng.integers(1, 128, sub.sum()) * 2.0**-133
    for t in range(q):
        x[t, rng.integers(K)] = rng.choice([-1.0, 1.0]) * 2.0**spike_log2
    bits = f32_to_bf16_bits(x.astype(np.float32))
    return bits, synth.bf16_bits_to_f32(bits).reshape(q, K)


def zero_fp4_codes(Wq, N, K, frac, seed):
    """Copy of a packed FP4 matrix with a fraction `frac` of its codes set to +0 (code 0)."""
    W = np.array(Wq, np.uint8, copy=True)
    rng = np.random.default_rng(seed)
    blk = W[: N * (K // 32) * 17].reshape(-1, 17)
    codes = blk[:, 1:]
    lo = rng.random(codes.shape) < frac
    hi = rng.random(codes.shape) < frac
    codes[lo] &= 0xF0
    codes[hi] &= 0x0F
    blk[:, 1:] = codes
    return W
