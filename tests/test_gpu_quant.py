"""fpx_quantize / fpx_dequantize against the oracle: codes and scales bit-exact."""
import numpy as np
import pytest
import torch

import bit_block_quantized_wt_b300 as fpx
import oracle
import synth
from gpu_util import dev, host, need_gpu, read_status, status_word

pytestmark = pytest.mark.gpu


def gpu_quantize(fmt, W, scales=None):
    N, K = W.shape
    out = torch.zeros(max(fpx.fpx_matrix_bytes(fmt, N, K), 16), dtype=torch.uint8, device="cuda")
    st = status_word()
    fpx.fpx_quantize(fmt, dev(W), N, K, out, block_scales=None if scales is None else dev(scales), dev_status=st)
    return host(out)[: fpx.fpx_matrix_bytes(fmt, N, K)], read_status(st)


def weights(N, K, seed):
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((N, K)) * rng.uniform(1e-3, 10, (N, 1))).astype(np.float32)
    W[0, :6] = [0.0, -0.0, 1e-40, -1e-40, 3.0, -3.0]
    W[1, :32] = 0.0
    W[2, :32] = np.float32(2.0**-140)  # tiny: FP4 exponent clamps to 0
    return W


@pytest.mark.parametrize("fmt", [2, 3, 4])
@pytest.mark.parametrize("N,K", [(3, 32), (17, 256), (256, 4096)])
def test_quantize_matches_oracle(fmt, N, K):
    need_gpu()
    W = weights(N, K, N * K + fmt)
    got, st = gpu_quantize(fmt, W)
    assert st == 0
    ost, ref = oracle.quantize(fmt, W)
    assert ost == 0
    assert np.array_equal(got, ref[: got.size])


@pytest.mark.parametrize("fmt", [2, 3, 4])
def test_quantize_round_trip_given_scales(fmt):
    need_gpu()
    N, K = 64, 1024
    Wq = synth.matrix(fmt, N, K, seed=21)
    Wf = torch.empty(N, K, device="cuda")
    fpx.fpx_dequantize(fmt, dev(Wq), N, K, Wf)
    Wh = host(Wf)
    assert np.array_equal(Wh.astype(np.float64), oracle.dequantize(fmt, Wq, N, K))
    b = Wq.reshape(N * K // 32, -1)
    if fmt == 4:
        sc = np.ldexp(1.0, b[:, 0].astype(np.int64) - 127).astype(np.float32)
    else:
        sc = (b[:, 0].astype(np.uint16) | (b[:, 1].astype(np.uint16) << 8)).view(np.float16).astype(np.float32)
    got, st = gpu_quantize(fmt, Wh, sc)
    assert st == 0 and np.array_equal(got, Wq)


def test_quantize_device_errors():
    need_gpu()
    W = np.ones((2, 64), np.float32)
    W[1, 5] = np.nan
    _, st = gpu_quantize(2, W)
    assert st == 1 << fpx.FPX_ERANGE
    W = np.ones((1, 32), np.float32) * 5e5  # 5e5 / 7 > 65520: the binary16 scale overflows
    _, st = gpu_quantize(3, W)
    assert st == 1 << fpx.FPX_ERANGE
    _, st = gpu_quantize(4, np.ones((1, 32), np.float32), np.full(1, 3.0, np.float32))
    assert st == 1 << fpx.FPX_EINVAL


def test_dequantize_invalid_fp4_block():
    need_gpu()
    Wq = synth.matrix(4, 2, 64, seed=3)
    Wq[17] = 255
    out = torch.zeros(2, 64, device="cuda")
    st = status_word()
    fpx.fpx_dequantize(4, dev(Wq), 2, 64, out, dev_status=st)
    assert read_status(st) == 1 << fpx.FPX_EDATA
    o = host(out)
    assert np.all(o[0, 32:] == 0)


def gpu_quantize_weighted(fmt, W, imp=None):
    N, K = W.shape
    out = torch.zeros(max(fpx.fpx_matrix_bytes(fmt, N, K), 16), dtype=torch.uint8, device="cuda")
    st = status_word()
    fpx.fpx_quantize_weighted(fmt, dev(W), N, K, out, importance=None if imp is None else dev(imp), dev_status=st)
    return host(out)[: fpx.fpx_matrix_bytes(fmt, N, K)], read_status(st)


@pytest.mark.parametrize("fmt", [2, 3, 4])
@pytest.mark.parametrize("N,K,with_imp", [(3, 32, True), (17, 256, False), (256, 4096, True)])
def test_quantize_weighted_matches_oracle(fmt, N, K, with_imp):
    """The importance-weighted quantizer: every candidate choice and code bit-exact against the oracle
    (the binary64 error sums are taken in the same order with the same roundings on both sides)."""
    need_gpu()
    W = weights(N, K, N * K + fmt + 7)
    imp = np.random.default_rng(N + K).uniform(0.0, 3.0, K).astype(np.float32) if with_imp else None
    if imp is not None:
        imp[:3] = [0.0, 1e-30, 100.0]
    got, st = gpu_quantize_weighted(fmt, W, imp)
    assert st == 0
    ost, ref = oracle.quantize_weighted(fmt, W, imp)
    assert ost == 0
    assert np.array_equal(got, ref[: got.size])


def test_quantize_weighted_flags_bad_importance():
    need_gpu()
    W = weights(4, 64, 1)
    imp = np.ones(64, np.float32)
    imp[40] = -1.0
    _, st = gpu_quantize_weighted(2, W, imp)
    assert st & (1 << fpx.FPX_ERANGE)
