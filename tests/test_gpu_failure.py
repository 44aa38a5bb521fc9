"""Failure detection of the layer kernels' bounded waits, without a GPU fault.

The waits between a streaming kernel's producer and its consumers give up after a time limit, flag
FPX_ETIMEOUT in the workspace status word and return. Here the failure is made on the host side: a test
hook (fpx_debug_ring_wait) shortens the limit to 2 ms and has CTA 0 of the gate/up kernel withhold one
weight copy, as if the copy were lost. The call must come back with FPX_ETIMEOUT set, every copy that
was issued having landed, and the next call, with the hook off, must give the normal result bit for bit
(the context is still usable)."""
import numpy as np
import pytest
import torch

import bit_block_quantized_wt_b300 as fpx
import synth
from gpu_util import DeviceLayer, dev, host, need_gpu, read_status

pytestmark = pytest.mark.gpu
DEFAULT_WAIT_NS = 500_000_000


def run(L, x, q, k, ws, ws_b):
    y = torch.full((q, L.H), float("nan"), device="cuda")
    idx = torch.full((q, k), -1, dtype=torch.int32, device="cuda")
    fpx.moe_layer_decode(L.c, x, q, k, y, ws, ws_b, idx_out=idx)
    return read_status(ws[:4].view(torch.int32)), host(y), host(idx)


@pytest.mark.parametrize("drop", [0, 1])
def test_lost_copy_times_out_and_the_next_call_is_normal(drop):
    need_gpu()
    q, k = 4, 2
    L = DeviceLayer(512, 512, 16, seed=21)
    x = dev(synth.tokens_bf16(q, 512, seed=4)[0])
    ws_b = fpx.moe_workspace_bytes(L.c, q, k)
    ws = torch.empty(ws_b, dtype=torch.uint8, device="cuda")
    st0, y0, i0 = run(L, x, q, k, ws, ws_b)
    assert st0 == 0
    try:
        fpx.fpx_debug_ring_wait(2_000_000, drop)
        st1, _, i1 = run(L, x, q, k, ws, ws_b)
    finally:
        fpx.fpx_debug_ring_wait(DEFAULT_WAIT_NS, -1)
    assert st1 & (1 << fpx.FPX_ETIMEOUT), st1
    assert np.array_equal(i1, i0)  # routing ran before the lost copy
    st2, y2, i2 = run(L, x, q, k, ws, ws_b)
    assert st2 == 0
    assert np.array_equal(y2, y0) and np.array_equal(i2, i0)

