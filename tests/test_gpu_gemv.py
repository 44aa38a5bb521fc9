"""fpx_gemv_q against the oracle: tolerance 2e-3 * sum|w x| per output, bit-exact closed forms and
bit-identical columns across q."""
import numpy as np
import pytest
import torch

import bit_block_quantized_wt_b300 as fpx
import oracle
import synth
from gpu_util import dev, host, need_gpu, read_status, status_word

pytestmark = pytest.mark.gpu
TOL = 2e-3


def gemv(fmt, Wq_dev, N, K, x, q):
    """x: numpy float32 [q][K] (binary32 path) or uint16 bfloat16 bits [q][K]."""
    xd = dev(x)
    dt = fpx.FPX_DTYPE_BF16 if x.dtype == np.uint16 else fpx.FPX_DTYPE_F32
    y = torch.full((q, N), float("nan"), device="cuda")
    st = status_word()
    fpx.fpx_gemv_q(fmt, Wq_dev, N, K, xd, dt, q, y, dev_status=st)
    assert read_status(st) == 0
    return host(y)


def check(y, yo, M):
    err = np.abs(y.astype(np.float64) - yo)
    assert np.all(err <= TOL * M), float((err / np.maximum(M, 1e-300)).max())


@pytest.mark.parametrize("fmt", [2, 3, 4])
@pytest.mark.parametrize("N,K", [(1, 32), (37, 256), (129, 96), (300, 1024), (64, 4096), (5, 14336)])
def test_gemv_small_all_q(fmt, N, K):
    need_gpu()
    Wq = synth.matrix(fmt, N, K, seed=N + K)
    Wd = dev(Wq)
    bits, vals = synth.tokens_bf16(4, K, seed=N)
    y4 = gemv(fmt, Wd, N, K, bits, 4)
    yo, M = oracle.gemv(fmt, Wq, N, K, vals.astype(np.float64))
    check(y4, yo, M)
    for q in (1, 2, 3):
        yq = gemv(fmt, Wd, N, K, bits[:q], q)
        assert np.array_equal(yq, y4[:q])  # bit-identical columns
    for t in range(4):
        y1 = gemv(fmt, Wd, N, K, bits[t : t + 1], 1)
        assert np.array_equal(y1[0], y4[t])


def test_gemv_config1_fp2_1024_fp32():
    """Single FP2 GEMV, q = 1: 1024 x 1024, fp32 N(0,1) activation."""
    need_gpu()
    N = K = 1024
    Wq = synth.matrix(2, N, K, seed=0)
    x = synth.normal_f32(K, 1.0, seed=0)[None, :]
    y = gemv(2, dev(Wq), N, K, x, 1)
    yo, M = oracle.gemv(2, Wq, N, K, x.astype(np.float64))
    check(y, yo, M)


@pytest.mark.parametrize("fmt", [2, 3, 4])
@pytest.mark.parametrize("N", [4096, 14336])
def test_gemv_config2_full_size_sampled(fmt, N):
    """Dense sweep shapes at full size; the oracle checks 192 sampled rows of every q column."""
    need_gpu()
    K = 4096
    Wq = synth.matrix(fmt, N, K, seed=1, tensor=synth.DENSE_W)
    Wd = dev(Wq)
    bits, vals = synth.tokens_bf16(4, K, seed=1)
    rb = K // 32 * fpx.fpx_block_bytes(fmt)
    rows = np.unique(np.concatenate([[0, N - 1], np.random.default_rng(fmt).integers(0, N, 190)]))
    sub = np.concatenate([Wq[r * rb : (r + 1) * rb] for r in rows])
    yo, M = oracle.gemv(fmt, sub, len(rows), K, vals.astype(np.float64))
    y4 = gemv(fmt, Wd, N, K, bits, 4)
    check(y4[:, rows], yo, M)
    y1 = gemv(fmt, Wd, N, K, bits[2:3], 1)
    assert np.array_equal(y1[0], y4[2])


@pytest.mark.parametrize("fmt", [2, 3, 4])
def test_gemv_unit_vector_gives_exact_column(fmt):
    need_gpu()
    N, K = 200, 512
    Wq = synth.matrix(fmt, N, K, seed=9)
    W = oracle.dequantize(fmt, Wq, N, K)
    Wd = dev(Wq)
    for j in (0, 1, 31, 32, 300, 511):
        x = np.zeros((1, K), np.float32)
        x[0, j] = 1.0
        y = gemv(fmt, Wd, N, K, x, 1)
        assert np.array_equal(y[0].astype(np.float64), W[:, j])


def test_gemv_edge_shapes_and_invalid_block():
    need_gpu()
    y = torch.full((2, 8), 5.0, device="cuda")
    x = torch.zeros(2, 32, device="cuda")
    W = torch.zeros(64, dtype=torch.uint8, device="cuda")
    fpx.fpx_gemv_q(2, W, 8, 0, x, fpx.FPX_DTYPE_F32, 2, y)  # K = 0: y = 0
    assert torch.all(y == 0)
    fpx.fpx_gemv_q(2, W, 0, 32, x, fpx.FPX_DTYPE_F32, 2, y)  # N = 0: nothing written
    Wq = synth.matrix(4, 4, 64, seed=2)
    Wq[17 * 2] = 255  # block 2 of row 1: FP4 scale byte 255
    st = status_word()
    out = torch.zeros(1, 4, device="cuda")
    fpx.fpx_gemv_q(4, dev(Wq), 4, 64, torch.ones(1, 64, device="cuda"), fpx.FPX_DTYPE_F32, 1, out, dev_status=st)
    assert read_status(st) == 1 << fpx.FPX_EDATA
