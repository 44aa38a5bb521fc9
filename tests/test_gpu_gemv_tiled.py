"""fpx_gemv_q_tiled (the dense GEMV on a box-tiled matrix) against the oracle's GEMV of the same
packed blocks: within 2e-3 * sum|w x| per output, columns bit-identical across q, the split into K
pieces (small N) and the single piece (large N) both covered, an invalid FP4 scale reported, and at
the bench's full size (151552 x 4096 FP2) sampled rows checked against the oracle."""
import numpy as np
import pytest
import torch

import bit_block_quantized_wt_b300 as fpx
import oracle
import synth
from gpu_util import dev, host, need_gpu, read_status, status_word

pytestmark = pytest.mark.gpu
TOL = 2e-3
ROWS = {2: 256, 3: 256, 4: 64}


def tiled(fmt, Wq, N, K):
    """Device copy of the row-major packed matrix, box-tiled."""
    src = dev(Wq)
    dst = torch.empty_like(src)
    fpx.fpx_tile_matrices(fmt, src, N, K, 1, src.numel(), dst, dst.numel())
    return dst


def gemv_t(fmt, Wt, N, K, x, q):
    xd = dev(x)
    dt = fpx.FPX_DTYPE_BF16 if x.dtype == np.uint16 else fpx.FPX_DTYPE_F32
    y = torch.full((q, N), float("nan"), device="cuda")
    wb = fpx.fpx_gemv_tiled_workspace_bytes(fmt, N, K, q)
    assert wb > 0
    ws = torch.empty(wb, dtype=torch.uint8, device="cuda")
    st = status_word()
    fpx.fpx_gemv_q_tiled(fmt, Wt, N, K, xd, dt, q, y, ws, wb, dev_status=st)
    return host(y), read_status(st)


def check(y, yo, M):
    err = np.abs(y.astype(np.float64) - yo)
    assert np.all(err <= TOL * M), float((err / np.maximum(M, 1e-300)).max())


@pytest.mark.parametrize("fmt", [2, 3, 4])
@pytest.mark.parametrize("nb,K", [(1, 512), (3, 1024), (2, 4096), (12, 2048)])
def test_tiled_gemv_all_q(fmt, nb, K):
    """nb row tiles; small N splits every tile's K range into pieces (up to one stage each)."""
    need_gpu()
    N = nb * ROWS[fmt]
    Wq = synth.matrix(fmt, N, K, seed=N + K + fmt)
    Wt = tiled(fmt, Wq, N, K)
    bits, vals = synth.tokens_bf16(4, K, seed=N)
    y4, st = gemv_t(fmt, Wt, N, K, bits, 4)
    assert st == 0
    yo, M = oracle.gemv(fmt, Wq, N, K, vals.astype(np.float64))
    check(y4, yo, M)
    for q in (1, 2, 3):
        yq, _ = gemv_t(fmt, Wt, N, K, bits[:q], q)
        assert np.array_equal(yq, y4[:q])  # bit-identical columns
    for t in range(4):
        y1, _ = gemv_t(fmt, Wt, N, K, bits[t:t + 1], 1)
        assert np.array_equal(y1[0], y4[t])


def test_tiled_gemv_fp32_input_and_plain_gemv():
    """binary32 activations; the plain GEMV on the row-major matrix agrees within the tolerance."""
    need_gpu()
    N, K = 1024, 2048
    Wq = synth.matrix(2, N, K, seed=3)
    x = np.stack([synth.normal_f32(K, 1.0, seed=s) for s in range(3)])
    y, st = gemv_t(2, tiled(2, Wq, N, K), N, K, x, 3)
    assert st == 0
    yo, M = oracle.gemv(2, Wq, N, K, x.astype(np.float64))
    check(y, yo, M)
    yp = torch.empty(3, N, device="cuda")
    fpx.fpx_gemv_q(2, dev(Wq), N, K, dev(x), fpx.FPX_DTYPE_F32, 3, yp)
    assert np.all(np.abs(host(yp).astype(np.float64) - y) <= 2 * TOL * M)


def test_tiled_gemv_fp4_invalid_scale():
    need_gpu()
    N, K = 128, 512
    Wq = synth.matrix(4, N, K, seed=9).copy()
    Wq[17 * 5] = 255  # block 5 of row 0: its scale byte
    bits, vals = synth.tokens_bf16(2, K, seed=1)
    y, st = gemv_t(4, tiled(4, Wq, N, K), N, K, bits, 2)
    assert st == 1 << fpx.FPX_EDATA
    Wz = Wq.copy()
    Wz[17 * 5:17 * 6] = 0  # the invalid block counts as zeros: compare with an all-zero block there
    yo, M = oracle.gemv(4, Wz, N, K, vals.astype(np.float64))
    check(y, yo, M)


def test_tiled_gemv_full_size_sampled_rows():
    """151552 x 4096 FP2 (194 MB, one piece per row tile, the bench's shape), q = 4: 512 sampled rows
    (including the first and last tile's edges) against the oracle."""
    need_gpu()
    N, K = 151552, 4096
    Wq = synth.matrix(2, N, K, seed=11)
    Wt = tiled(2, Wq, N, K)
    bits, vals = synth.tokens_bf16(4, K, seed=5)
    y, st = gemv_t(2, Wt, N, K, bits, 4)
    assert st == 0
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([[0, 255, 256, N - 256, N - 1], rng.integers(0, N, 507)]))
    rb = K // 32 * 10
    sub = Wq.reshape(N, rb)[rows].reshape(-1)
    yo, M = oracle.gemv(2, sub, len(rows), K, vals.astype(np.float64))
    check(y[:, rows], yo, M)


def test_tiled_gemv_smallest_call():
    """One FP2 row tile over one piece of K (the argument errors are checked without a GPU)."""
    need_gpu()
    x = torch.zeros(4, 512, dtype=torch.bfloat16, device="cuda")
    y = torch.full((4, 256), float("nan"), device="cuda")
    W = torch.zeros(256 * 512 // 32 * 10, dtype=torch.uint8, device="cuda")
    wb = fpx.fpx_gemv_tiled_workspace_bytes(2, 256, 512, 4)
    ws = torch.zeros(wb, dtype=torch.uint8, device="cuda")
    fpx.fpx_gemv_q_tiled(2, W, 256, 512, x, fpx.FPX_DTYPE_BF16, 4, y, ws, wb)
    assert torch.all(y == 0)
