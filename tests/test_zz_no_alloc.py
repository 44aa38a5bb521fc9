"""moe_layer_decode_static_ws: the layer for callers that cannot allocate device memory (a library inside
a framework that owns all device allocations, or a loop that must not call cudaMalloc/cudaFree because
they can synchronise the device). Its scratch is a fixed array inside libfpx.so, so this test compares it,
through the C ABI, with moe_layer_decode given a caller workspace, on two calls in a row: the second call
runs on the array the first one left behind. This file sorts last so a run that stops at the first failure
has already run every other test; it also passes alone in a fresh process (the first call on the device
does the array's one-time address lookup)."""
import numpy as np
import pytest
import torch

import bit_block_quantized_wt_b300 as fpx
import synth
from gpu_util import DeviceLayer, dev, host, need_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("k", [4, 6, 8])
def test_fixed_scratch_layer_matches_workspace_layer(k):
    """Up to the largest decode shape the array serves (q = 4, k = 8 at H = 4096, I = 2048, E = 256)."""
    need_gpu()
    H, I, E, q = 4096, 2048, 256, 4
    L = DeviceLayer(H, I, E, seed=3, layer=1)
    ws_b = fpx.moe_workspace_bytes(L.c, q, k)
    assert ws_b <= 16 << 20
    ws = torch.empty(ws_b, dtype=torch.uint8, device="cuda")
    for seed in (11, 12):
        x = dev(synth.tokens_bf16(q, H, seed=seed)[0])
        outs = []
        for fixed in (False, True):
            y = torch.full((q, H), float("nan"), device="cuda")
            idx = torch.full((q, k), -1, dtype=torch.int32, device="cuda")
            w = torch.full((q, k), float("nan"), device="cuda")
            lg = torch.full((q, E), float("nan"), device="cuda")
            if fixed:
                st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
                fpx.moe_layer_decode_static_ws(L.c, x, q, k, y, idx_out=idx, w_out=w, logits_out=lg, dev_status=st)
                assert int(host(st)[0]) == 0
            else:
                fpx.moe_layer_decode(L.c, x, q, k, y, ws, ws_b, idx_out=idx, w_out=w, logits_out=lg)
                assert fpx.fpx_read_status(ws[:4].view(torch.int32)) == 0
            outs.append([host(t) for t in (y, idx, w, lg)])
        (y0, i0, w0, l0), (y1, i1, w1, l1) = outs
        # same kernels on the same inputs: the results agree bit for bit, which is inside the 2e-3
        # tolerance the parity tests use
        assert np.all(np.isfinite(y1))
        assert np.array_equal(y1, y0) and np.array_equal(i1, i0)
        assert np.array_equal(w1, w0) and np.array_equal(l1, l0)


def test_fixed_scratch_rejects_shapes_beyond_its_size():
    need_gpu()
    big = fpx.moe_layer(H=8192, I=8192, E=256, router=1 << 20, gate=1 << 20, up=1 << 20, down=1 << 20,
                        sh_gate=1 << 20, sh_up=1 << 20, sh_down=1 << 20)
    assert fpx.moe_workspace_bytes(big, 4, 8) > 16 << 20
    st = fpx.lib().moe_layer_decode_static_ws(fpx.ctypes.byref(big), 1 << 20, 4, 8, 1 << 20, None, None, None, None,
                                              None)
    assert st == fpx.FPX_ESPACE
