"""fpx_tile_matrices: the box-tiled layout of the MoE layer kernels, bit-exact against the layout
formula applied on the host to the host generator's row-major matrices, and the inverse restoring
row-major."""
import numpy as np
import pytest
import torch

import bit_block_quantized_wt_b300 as fpx
import synth
from gpu_util import host, need_gpu

pytestmark = pytest.mark.gpu

GEOM = {2: (256, 80), 3: (256, 112), 4: (64, 272)}  # rows x bytes of a tile


def host_tiled(rowmajor, N, K, fmt):
    """The layout formula of include/fpx.h applied with numpy: byte (r, j) goes to
    ((r // R) * P + j // B) * R * B + (r % R) * B + j % B."""
    R, B = GEOM[fmt]
    rb = K // 32 * fpx.fpx_block_bytes(fmt)
    P = rb // B
    a = np.frombuffer(rowmajor[: N * rb], np.uint8).reshape(N // R, R, P, B)
    return a.transpose(0, 2, 1, 3).reshape(-1)


@pytest.mark.parametrize("fmt,N,K", [(2, 512, 1024), (3, 768, 512), (4, 128, 2048), (2, 2048, 4096)])
def test_tile_matches_formula_and_inverts(fmt, N, K):
    need_gpu()
    mb = fpx.fpx_matrix_bytes(fmt, N, K)
    count = 3
    src = torch.empty(count * mb, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    synth.device_matrices(fmt, 5, 1, synth.GATE, 0, count, N, K, src.data_ptr(), mb, s)
    dst = torch.zeros(count * mb, dtype=torch.uint8, device="cuda")
    back = torch.zeros(count * mb, dtype=torch.uint8, device="cuda")
    fpx.fpx_tile_matrices(fmt, src, N, K, count, mb, dst, mb, 0, s)
    fpx.fpx_tile_matrices(fmt, dst, N, K, count, mb, back, mb, 1, s)
    d, b = host(dst), host(back)
    rb = K // 32 * fpx.fpx_block_bytes(fmt)
    for m in range(count):
        rm = synth.matrix(fmt, N, K, 5, 1, synth.GATE, m).tobytes()  # host generator, row-major
        assert np.array_equal(d[m * mb : m * mb + N * rb], host_tiled(rm, N, K, fmt))
        assert np.array_equal(b[m * mb : m * mb + N * rb], np.frombuffer(rm[: N * rb], np.uint8))


def test_tile_argument_errors():
    need_gpu()
    L = fpx.lib()
    t = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    p = t.data_ptr()
    mb = fpx.fpx_matrix_bytes(2, 256, 256)
    assert L.fpx_tile_matrices(2, p, 100, 256, 1, mb, p + (1 << 19), mb, 0, None) == fpx.FPX_EINVAL  # N % 256
    assert L.fpx_tile_matrices(2, p, 256, 256, 1, mb, p, mb, 0, None) == fpx.FPX_EINVAL  # in place
    assert L.fpx_tile_matrices(2, p + 8, 256, 256, 1, mb, p + (1 << 19), mb, 0, None) == fpx.FPX_EALIGN
    assert L.fpx_tile_matrices(2, p, 256, 256, 1, mb, p + (1 << 19), mb, 2, None) == fpx.FPX_EINVAL
