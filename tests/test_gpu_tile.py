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
CODE_BYTES = {2: 64, 3: 96}  # per tile row, FP2 / FP3 code area

# FP3 code fields of pair p for the even / odd chunk of a chunk pair: (word, bit of the code's low bit
# in each binary16 half); None = the spare bits (code bit i at bit 0 of word i)
FP3_FIELDS = [[(0, 1), (0, 4), (0, 7), (0, 10), (0, 13), (1, 1), (1, 4), (1, 7)],
              [(1, 10), (1, 13), (2, 1), (2, 4), (2, 7), (2, 10), (2, 13), None]]


def host_tiled(rowmajor, N, K, fmt):
    """The tiled layout of include/fpx.h built with numpy: tile (r // R) * P + j // B holds bytes j of rows
    r of one column piece; FP4 tiles are the rows' bytes, FP2 / FP3 tiles a regrouped code area and a
    scale area (scale 4h + C of a row = block 2C + h of the piece)."""
    R, B = GEOM[fmt]
    bb = fpx.fpx_block_bytes(fmt)
    rb = K // 32 * bb
    P = rb // B
    a = np.frombuffer(rowmajor[: N * rb], np.uint8).reshape(N // R, R, P, B).transpose(0, 2, 1, 3)
    if fmt == 4:
        return a.reshape(-1)
    blk = a.reshape(N // R, P, R, 8, bb)
    sc = blk[..., [0, 2, 4, 6, 1, 3, 5, 7], 0:2].reshape(N // R, P, R, 16)
    if fmt == 2:
        cd = np.empty((N // R, P, R, 16, 4), np.uint8)
        for t in range(4):
            for C in range(4):  # word 4t + C = code bytes 4 (t % 2) .. +3 of block 2C + t // 2
                cd[..., 4 * t + C, :] = blk[..., 2 * C + t // 2, 2 + 4 * (t % 2): 6 + 4 * (t % 2)]
    else:
        lo = np.unpackbits(blk[..., 2:10], axis=-1, bitorder="little").reshape(N // R, P, R, 8, 32, 2)
        hi = np.unpackbits(blk[..., 10:14], axis=-1, bitorder="little")  # bit k = code k
        c = (lo[..., 0] + 2 * lo[..., 1] + 4 * hi).astype(np.uint32)  # [.., block, code]
        W = np.zeros((N // R, P, R, 4, 2, 3), np.uint32)
        for t in range(4):
            for m in range(2):
                for odd in range(2):
                    for j in range(16):
                        v = c[..., 2 * (2 * m + odd) + t // 2, 16 * (t % 2) + j]
                        f, hh = FP3_FIELDS[odd][j % 8], j // 8
                        if f is None:
                            for i in range(3):
                                W[..., t, m, i] |= ((v >> i) & 1) << (16 * hh)
                        else:
                            W[..., t, m, f[0]] |= v << (16 * hh + f[1])
        cd = W.astype("<u4").view(np.uint8)
    cd = cd.reshape(N // R, P, R * CODE_BYTES[fmt])
    return np.concatenate([cd, sc.reshape(N // R, P, R * 16)], axis=-1).reshape(-1)


@pytest.mark.parametrize("fmt,N,K", [(2, 512, 1024), (3, 768, 512), (4, 128, 2048), (2, 2048, 4096), (3, 256, 4096)])
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
