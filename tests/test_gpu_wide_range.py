"""Activations with a wide dynamic range through the tensor-core paths (dense GEMV on row-major and
box-tiled matrices, decode layer, prefill): +-0, bfloat16 subnormals, 32-entry blocks scaled by up to 2^+-20 and one spike per column.

The tensor-core kernels take a column (or, in the prefill, a row) as binary16 scaled by one power of two
that puts its largest element in [2^14, 2^15). A bfloat16 element within 2^31 of the column's largest is
then exact, so only binary32 sums round; an element further down lands among the binary16 subnormals
and may move by up to 2^(e - 40) (largest element in [2^(e-1), 2^e)). That never matters when the
largest elements carry nonzero weights (FP2 and FP3 have no zero code, so Sum|w x| is at least the
spike times the block scale), nor when a column spans less than 2^28; those cases must meet the usual
2e-3 * Sum|w x|. For FP4 weights with many zero codes and a column spanning 2^60 the kernels meet
2e-3 * Sum|w x| + 2^(e - 40) * Sum|w|, which is checked as the stated bound of the encoding."""
import numpy as np
import pytest
import torch

import bit_block_quantized_wt_b300 as fpx
import oracle
import synth
from gpu_util import DeviceLayer, dev, host, need_gpu, read_status, status_word, wide_bf16, zero_fp4_codes

pytestmark = pytest.mark.gpu
TOL = 2e-3


def gemv(fmt, Wq, N, K, bits):
    q = bits.shape[0]
    y = torch.full((q, N), float("nan"), device="cuda")
    st = status_word()
    fpx.fpx_gemv_q(fmt, dev(Wq), N, K, dev(bits), fpx.FPX_DTYPE_BF16, q, y, dev_status=st)
    assert read_status(st) == 0
    return host(y)


@pytest.mark.parametrize("fmt", [2, 3])
@pytest.mark.parametrize("spike", [20, 60])
def test_gemv_wide_range_fp2_fp3(fmt, spike):
    need_gpu()
    N, K = 256, 2048
    Wq = synth.matrix(fmt, N, K, seed=40 + fmt)
    bits, vals = wide_bf16(4, K, seed=spike + fmt, spike_log2=spike, block_span=20)
    y = gemv(fmt, Wq, N, K, bits)
    yo, M = oracle.gemv(fmt, Wq, N, K, vals.astype(np.float64))
    err = np.abs(y.astype(np.float64) - yo)
    assert np.all(err <= TOL * M), float((err / M).max())
    for t in range(4):  # still bit-identical to a one-column call
        assert np.array_equal(gemv(fmt, Wq, N, K, bits[t : t + 1])[0], y[t])


def gemv_tiled(fmt, Wq, N, K, bits):
    """The same GEMV on the box-tiled copy of the matrix (fpx_gemv_q_tiled)."""
    q = bits.shape[0]
    src = dev(Wq)
    Wt = torch.empty_like(src)
    fpx.fpx_tile_matrices(fmt, src, N, K, 1, src.numel(), Wt, Wt.numel())
    y = torch.full((q, N), float("nan"), device="cuda")
    wb = fpx.fpx_gemv_tiled_workspace_bytes(fmt, N, K, q)
    ws = torch.empty(wb, dtype=torch.uint8, device="cuda")
    st = status_word()
    fpx.fpx_gemv_q_tiled(fmt, Wt, N, K, dev(bits), fpx.FPX_DTYPE_BF16, q, y, ws, wb, dev_status=st)
    assert read_status(st) == 0
    return host(y)


@pytest.mark.parametrize("fmt", [2, 3])
@pytest.mark.parametrize("spike", [20, 60])
def test_tiled_gemv_wide_range_fp2_fp3(fmt, spike):
    need_gpu()
    N, K = 512, 2048
    Wq = synth.matrix(fmt, N, K, seed=50 + fmt)
    bits, vals = wide_bf16(4, K, seed=spike + fmt + 7, spike_log2=spike, block_span=20)
    y = gemv_tiled(fmt, Wq, N, K, bits)
    yo, M = oracle.gemv(fmt, Wq, N, K, vals.astype(np.float64))
    err = np.abs(y.astype(np.float64) - yo)
    assert np.all(err <= TOL * M), float((err / M).max())
    for t in range(4):
        assert np.array_equal(gemv_tiled(fmt, Wq, N, K, bits[t : t + 1])[0], y[t])


def test_tiled_gemv_fp4_zero_codes_spanning_2_60_meets_the_encoding_bound():
    need_gpu()
    N, K = 256, 2048
    Wq = zero_fp4_codes(synth.matrix(4, N, K, seed=46), N, K, 0.5, seed=3)
    bits, vals = wide_bf16(4, K, seed=6, spike_log2=60, block_span=20)
    y = gemv_tiled(4, Wq, N, K, bits)
    yo, M = oracle.gemv(4, Wq, N, K, vals.astype(np.float64))
    absw = np.abs(oracle.dequantize(4, Wq, N, K)).sum(axis=1)
    _, e = np.frexp(np.abs(vals.astype(np.float64)).max(axis=1))
    bound = TOL * M + np.ldexp(1.0, e - 40)[:, None] * absw[None, :]
    err = np.abs(y.astype(np.float64) - yo)
    assert np.all(err <= bound), float((err / bound).max())


def test_gemv_fp4_zero_codes_within_binary16_range():
    """Half the FP4 codes zero and columns spanning less than 2^28: the usual tolerance."""
    need_gpu()
    N, K = 256, 2048
    Wq = zero_fp4_codes(synth.matrix(4, N, K, seed=44), N, K, 0.5, seed=1)
    bits, vals = wide_bf16(4, K, seed=3, spike_log2=12, block_span=6)
    y = gemv(4, Wq, N, K, bits)
    yo, M = oracle.gemv(4, Wq, N, K, vals.astype(np.float64))
    err = np.abs(y.astype(np.float64) - yo)
    assert np.all(err <= TOL * M), float((err / M).max())


def test_gemv_fp4_zero_codes_spanning_2_60_meets_the_encoding_bound():
    need_gpu()
    N, K = 256, 2048
    Wq = zero_fp4_codes(synth.matrix(4, N, K, seed=45), N, K, 0.5, seed=2)
    bits, vals = wide_bf16(4, K, seed=5, spike_log2=60, block_span=20)
    y = gemv(4, Wq, N, K, bits)
    yo, M = oracle.gemv(4, Wq, N, K, vals.astype(np.float64))
    absw = np.abs(oracle.dequantize(4, Wq, N, K)).sum(axis=1)
    _, e = np.frexp(np.abs(vals.astype(np.float64)).max(axis=1))  # max |x| in [2^(e-1), 2^e)
    bound = TOL * M + np.ldexp(1.0, e - 40)[:, None] * absw[None, :]
    err = np.abs(y.astype(np.float64) - yo)
    assert np.all(err <= bound), float((err / bound).max())


def test_layer_wide_range_tokens():
    """The decode layer on wide-range tokens (spikes 2^20 above the bulk): routing consistent with the
    logits, output within tolerance, and each column bit-identical to a one-token call."""
    need_gpu()
    q, k = 4, 4
    L = DeviceLayer(512, 512, 16, seed=31)
    bits, vals = wide_bf16(q, 512, seed=8, spike_log2=20, block_span=8)
    ws_b = fpx.moe_workspace_bytes(L.c, q, k)
    ws = torch.empty(ws_b, dtype=torch.uint8, device="cuda")

    def run(b):
        n = b.shape[0]
        y = torch.full((n, 512), float("nan"), device="cuda")
        idx = torch.empty(n, k, dtype=torch.int32, device="cuda")
        fpx.moe_layer_decode(L.c, dev(b), n, k, y, ws, ws_b, idx_out=idx)
        assert read_status(ws[:4].view(torch.int32)) == 0
        return host(y), host(idx)

    y, idx = run(bits)
    orc = L.oracle(vals.astype(np.float64), k, idx_force=idx)
    err = np.abs(y.astype(np.float64) - orc["y"])
    assert np.all(err <= TOL * orc["M"]), float((err / orc["M"]).max())
    for t in range(q):
        y1, i1 = run(bits[t : t + 1])
        assert np.array_equal(i1[0], idx[t]) and np.array_equal(y1[0], y[t])


def test_prefill_wide_range_tokens():
    need_gpu()
    T, k = 96, 4
    L = DeviceLayer(512, 512, 16, seed=33)
    bits, vals = wide_bf16(T, 512, seed=9, spike_log2=20, block_span=8)
    ws_b = fpx.moe_prefill_workspace_bytes(L.c, T, k)
    ws = torch.empty(ws_b, dtype=torch.uint8, device="cuda")
    y = torch.full((T, 512), float("nan"), device="cuda")
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    fpx.moe_layer_prefill(L.c, dev(bits), T, k, y, ws, ws_b, idx_out=idx)
    assert read_status(ws[:4].view(torch.int32)) == 0
    y, idx = host(y), host(idx)
    orc = L.oracle(vals.astype(np.float64), k, idx_force=idx)
    err = np.abs(y.astype(np.float64) - orc["y"])
    assert np.all(err <= TOL * orc["M"]), float((err / orc["M"]).max())
