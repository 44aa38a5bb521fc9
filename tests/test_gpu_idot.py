"""fpx_gemv_q_idot (integer-dot GEMV) against the oracle.

Two checks per output: against the oracle's integer-dot result (W applied to the activation grid
x_hat), within the binary32 rounding of the kernel's sums, (8 + slices) * 2^-24 * sum|w x_hat|; and
against the plain oracle GEMV within the tolerance of the verify step, 2e-3 * sum|w x|."""
import numpy as np
import pytest
import torch

import bit_block_quantized_wt_b300 as fpx
import oracle
import synth
from gpu_util import dev, host, need_gpu, read_status, status_word

pytestmark = pytest.mark.gpu
TOL = 2e-3


def idot(fmt, Wq_dev, N, K, x, q, expect_status=0):
    """x: numpy float32 [q][K] (binary32 path) or uint16 bfloat16 bits [q][K]."""
    xd = dev(x)
    dt = fpx.FPX_DTYPE_BF16 if x.dtype == np.uint16 else fpx.FPX_DTYPE_F32
    y = torch.full((q, N), float("nan"), device="cuda")
    wsb = fpx.fpx_gemv_idot_workspace_bytes(K, q)
    ws = torch.full((wsb,), 0xA5, dtype=torch.uint8, device="cuda")  # no reliance on a zeroed workspace
    st = status_word()
    fpx.fpx_gemv_q_idot(fmt, Wq_dev, N, K, xd, dt, q, y, ws, wsb, dev_status=st)
    assert read_status(st) == expect_status
    return host(y)


def rounding_tol(K, Mhat):
    nsl = (K // 32 + 31) // 32
    return (8 + nsl) * 2.0**-24 * Mhat + 1e-30


def check(fmt, Wq, N, K, xv, y):
    yi, Mi = oracle.gemv_idot(fmt, Wq, N, K, xv)
    err = np.abs(y.astype(np.float64) - yi)
    assert np.all(err <= rounding_tol(K, Mi)), float((err / np.maximum(Mi, 1e-300)).max())
    yo, M = oracle.gemv(fmt, Wq, N, K, xv)
    err = np.abs(y.astype(np.float64) - yo)
    assert np.all(err <= TOL * M), float((err / np.maximum(M, 1e-300)).max())


SHAPES = {2: [(1, 256), (77, 1280), (200, 1024), (64, 4096), (130, 8192)],
          3: [(1, 256), (77, 1280), (200, 1024), (64, 4096), (130, 8192)],
          4: [(1, 512), (77, 1536), (200, 1024), (64, 4096), (130, 8192)]}


@pytest.mark.parametrize("fmt", [2, 3, 4])
@pytest.mark.parametrize("i", range(5))
def test_idot_all_q(fmt, i):
    """Several row blocks, ragged last slice (K = 1280 / 1536) and ragged last row block; bfloat16
    activations; columns of a q = 4 call are bit-identical to q = 1..3 calls."""
    need_gpu()
    N, K = SHAPES[fmt][i]
    Wq = synth.matrix(fmt, N, K, seed=N + K + fmt)
    Wd = dev(Wq)
    bits, vals = synth.tokens_bf16(4, K, seed=N + 3)
    y4 = idot(fmt, Wd, N, K, bits, 4)
    check(fmt, Wq, N, K, vals.astype(np.float64), y4)
    for q in (1, 2, 3):
        yq = idot(fmt, Wd, N, K, bits[:q], q)
        assert np.array_equal(yq, y4[:q])
    for t in range(4):
        assert np.array_equal(idot(fmt, Wd, N, K, bits[t : t + 1], 1)[0], y4[t])
    assert np.array_equal(idot(fmt, Wd, N, K, bits, 4), y4)  # repeatable


@pytest.mark.parametrize("fmt", [2, 3, 4])
def test_idot_f32_wide_range(fmt):
    """binary32 activations whose magnitudes vary by 2^+-20 between blocks, zero blocks and exact
    half-step ties: the grid rounds, the oracle's grid result is matched within binary32 rounding."""
    need_gpu()
    N, K = 150, 2048
    Wq = synth.matrix(fmt, N, K, seed=9)
    rng = np.random.default_rng(fmt)
    x = (rng.standard_normal((3, K)) * np.exp2(rng.integers(-20, 20, (3, K // 32))).repeat(32, axis=1))
    x = x.astype(np.float32)
    x[1, 64:96] = 0.0
    x[2, 128:160] = 0.0
    x[2, 128] = 1.0
    x[2, 129:135] = np.ldexp(np.array([1, 3, 5, -1, -3, 7], np.float64), -14).astype(np.float32)  # ties
    y = idot(fmt, dev(Wq), N, K, x, 3)
    check(fmt, Wq, N, K, x.astype(np.float64), y)


def test_idot_config1_fp2_1024_fp32():
    """The single FP2 1024 x 1024 GEMV, q = 1, binary32 N(0,1) activation."""
    need_gpu()
    N = K = 1024
    Wq = synth.matrix(2, N, K, seed=0)
    x = synth.normal_f32(K, 1.0, seed=0)[None, :]
    y = idot(2, dev(Wq), N, K, x, 1)
    check(2, Wq, N, K, x.astype(np.float64), y)


@pytest.mark.parametrize("fmt", [2, 3, 4])
@pytest.mark.parametrize("N", [4096, 14336])
def test_idot_config2_full_size_sampled(fmt, N):
    """The dense sweep shapes at full size, q = 4; the oracle checks 192 sampled rows."""
    need_gpu()
    K = 4096
    Wq = synth.matrix(fmt, N, K, seed=1, tensor=synth.DENSE_W)
    Wd = dev(Wq)
    bits, vals = synth.tokens_bf16(4, K, seed=1)
    rb = K // 32 * fpx.fpx_block_bytes(fmt)
    rows = np.unique(np.concatenate([[0, N - 1], np.random.default_rng(fmt).integers(0, N, 190)]))
    sub = np.concatenate([Wq[r * rb : (r + 1) * rb] for r in rows])
    y4 = idot(fmt, Wd, N, K, bits, 4)
    check(fmt, sub, len(rows), K, vals.astype(np.float64), y4[:, rows])
    assert np.array_equal(idot(fmt, Wd, N, K, bits[2:3], 1)[0], y4[2])


def test_idot_flags():
    """An FP4 scale byte of 255 sets FPX_EDATA and its block counts as zeros; a NaN activation sets
    FPX_ERANGE and counts as 0."""
    need_gpu()
    N, K = 70, 1024
    Wq = synth.matrix(4, N, K, seed=4)
    bad = Wq.copy()
    bad[5 * (K // 32) * 17 + 3 * 17] = 255  # row 5, block 3
    bits, vals = synth.tokens_bf16(2, K, seed=4)
    y = idot(4, dev(bad), N, K, bits, 2, expect_status=1 << fpx.FPX_EDATA)
    zeroed = bad.copy()
    zeroed[5 * (K // 32) * 17 + 3 * 17 : 5 * (K // 32) * 17 + 4 * 17] = 0  # the block as zeros
    check(4, zeroed, N, K, vals.astype(np.float64), y)
    x = vals.copy()
    x[1, 300] = np.nan
    y = idot(4, dev(Wq), N, K, x, 2, expect_status=1 << fpx.FPX_ERANGE)
    x[1, 300] = 0.0
    check(4, Wq, N, K, x.astype(np.float64), y)
