"""The device twin of the input generator writes the same bytes as the host generator."""
import numpy as np
import pytest
import torch

import synth
from gpu_util import host, need_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fmt,N,K,count", [(2, 3, 96, 1), (3, 7, 256, 3), (4, 5, 64, 2), (2, 64, 4096, 2),
                                           (3, 129, 2048, 1), (4, 33, 4096, 1)])
def test_device_generator_matches_host(fmt, N, K, count):
    need_gpu()
    mb = synth.matrix_bytes(fmt, N, K)
    buf = torch.full((count * mb,), 0xEE, dtype=torch.uint8, device="cuda")
    synth.device_matrices(fmt, 5, 2, synth.GATE, 3, count, N, K, buf.data_ptr(), mb,
                          torch.cuda.current_stream().cuda_stream)
    got = host(buf).reshape(count, mb)
    for c in range(count):
        ref = synth.matrix(fmt, N, K, seed=5, layer=2, tensor=synth.GATE, expert=3 + c)
        assert np.array_equal(got[c], ref)
