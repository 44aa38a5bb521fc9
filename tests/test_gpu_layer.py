"""moe_layer_decode against the oracle: routing bit-exact, output within 2e-3 * M (the first-order
error magnitude). Each column of a q-token call is bit-identical to a q = 1 call on that column alone
(routing, weights and output): every packed weight is decoded once and applied to all columns, and
no rounding depends on the other columns or on the expert union."""
import numpy as np
import pytest
import torch

import bit_block_quantized_wt_b300 as fpx
import oracle
import synth
from gpu_util import DeviceLayer, dev, host, need_gpu, read_status, routing_gap_ok, topk_of

pytestmark = pytest.mark.gpu
TOL = 2e-3


def run_layer(L, bits, k):
    q = bits.shape[0]
    ws_b = fpx.moe_workspace_bytes(L.c, q, k)
    ws = torch.empty(ws_b, dtype=torch.uint8, device="cuda")
    y = torch.full((q, L.H), float("nan"), device="cuda")
    idx = torch.empty(q, k, dtype=torch.int32, device="cuda")
    w = torch.empty(q, k, device="cuda")
    lg = torch.empty(q, L.E, device="cuda")
    fpx.moe_layer_decode(L.c, dev(bits), q, k, y, ws, ws_b, idx_out=idx, w_out=w, logits_out=lg)
    st = read_status(ws[:4].view(torch.int32))
    assert st == 0
    return host(y), host(idx), host(w), host(lg)


def check_layer(L, bits, vals, k):
    y, idx, w, lg = run_layer(L, bits, k)
    q = bits.shape[0]
    for t in range(q):
        assert list(idx[t]) == list(topk_of(lg[t], k))
    orc = L.oracle(vals.astype(np.float64), k, idx_force=idx)
    assert np.all(np.abs(lg - orc["logits"]) <= 1e-4 + 1e-4 * np.abs(orc["logits"]))
    # where the oracle's own top-k (on its binary64 logits) is unique within the logit error, it must
    # agree; at every size (the oracle's router alone, without expanding every expert)
    own = oracle.route(L.R_host, vals.astype(np.float64), k)
    ok = routing_gap_ok(own["logits"], k, 1e-4)
    assert np.array_equal(own["idx"][ok], idx[ok])
    assert np.allclose(w, orc["w"], rtol=1e-5, atol=0)
    err = np.abs(y.astype(np.float64) - orc["y"])
    assert np.all(err <= TOL * orc["M"]), float((err / orc["M"]).max())
    return y, idx


@pytest.mark.parametrize("q", [1, 2, 3, 4])
@pytest.mark.parametrize("k", [1, 2, 4])
def test_layer_small(q, k):
    need_gpu()
    L = DeviceLayer(512, 512, 16, seed=q * 10 + k)
    bits, vals = synth.tokens_bf16(q, 512, seed=k)
    y, idx = check_layer(L, bits, vals, k)
    for t in range(q):  # each column alone: the same bits
        y1, i1 = check_layer(L, bits[t : t + 1], vals[t : t + 1], k)
        assert np.array_equal(i1[0], idx[t])
        assert np.array_equal(y1[0], y[t])


@pytest.mark.parametrize("k", [4, 6])
def test_layer_config3_full_size(k):
    """hidden 4096, 256 routed experts (FP2 gate/up [2048x4096], FP3 down), FP4 shared, q = 4."""
    need_gpu()
    L = DeviceLayer(4096, 2048, 256, seed=0, layer=0)
    bits, vals = synth.tokens_bf16(4, 4096, seed=0)
    y, idx = check_layer(L, bits, vals, k)
    for t in (0, 3):
        y1, i1 = check_layer(L, bits[t : t + 1], vals[t : t + 1], k)
        assert np.array_equal(i1[0], idx[t])
        assert np.array_equal(y1[0], y[t])
