"""moe_stack_verify against the oracle, layer by layer (teacher-forced on the GPU's residual), for the
q = 4 pass; the q = 1 pass of a column is bit-identical to that column of the q = 4 pass (final state,
every layer's residual and routing)."""
import numpy as np
import pytest
import torch

import bit_block_quantized_wt_b300 as fpx
import oracle
import synth
from gpu_util import DeviceLayer, dev, host, need_gpu, read_status, routing_gap_ok

pytestmark = pytest.mark.gpu
TOL = 2e-3


def run_stack(layers, r0, q, k):
    H = layers[0].H
    ws_b = fpx.moe_workspace_bytes(layers[0].c, q, k)
    ws = torch.empty(ws_b, dtype=torch.uint8, device="cuda")
    rL = torch.empty(q, H, device="cuda")
    idx = torch.empty(len(layers), q, k, dtype=torch.int32, device="cuda")
    tr = torch.empty(len(layers), q, H, device="cuda")
    fpx.moe_stack_verify([L.c for L in layers], dev(r0), q, k, rL, ws, ws_b, idx_out=idx, r_trace=tr)
    assert read_status(ws[:4].view(torch.int32)) == 0
    return host(rL), host(idx), host(tr)


def check_layer_step(L, r_in, r_out, idx, k):
    u = oracle.rmsnorm_bf16(r_in)
    orc = L.oracle(u, k, idx_force=idx)
    ref = r_in.astype(np.float64) + orc["y"]
    err = np.abs(r_out.astype(np.float64) - ref)
    bound = TOL * orc["M"] + 2.0**-22 * np.abs(ref)
    assert np.all(err <= bound), float((err / bound).max())
    own = oracle.route(L.R_host, u, k)
    ok = routing_gap_ok(own["logits"], k, 1e-4)
    assert np.array_equal(own["idx"][ok], idx[ok])


def check_pass(layers, r0, k, sample):
    rL, idx, tr = run_stack(layers, r0, r0.shape[0], k)
    assert np.array_equal(tr[0], r0)
    assert np.all(np.isfinite(rL))
    for l in sample:
        r_out = tr[l + 1] if l + 1 < len(layers) else rL
        check_layer_step(layers[l], tr[l], r_out, idx[l], k)
    return rL, idx, tr


def check_stack(layers, q, k, sample, columns):
    H = layers[0].H
    bits, vals = synth.tokens_bf16(q, H, seed=99)
    r0 = vals.astype(np.float32)
    rL, idx, tr = check_pass(layers, r0, k, sample)
    for t in columns:  # the q = 1 pass of column t: the same bits as column t of the batch
        rL1, idx1, tr1 = run_stack(layers, r0[t : t + 1], 1, k)
        assert np.array_equal(idx1[:, 0], idx[:, t])
        assert np.array_equal(tr1[:, 0], tr[:, t])
        assert np.array_equal(rL1[0], rL[t])


def test_stack_small():
    need_gpu()
    layers = [DeviceLayer(512, 512, 16, seed=7, layer=l) for l in range(5)]
    check_stack(layers, 4, 2, range(5), columns=range(4))


@pytest.mark.slow
def test_stack_config4_full_size():
    """43 config-3 layers (~99 GB of packed weights resident), q = 4 and q = 1, top-4; three layers
    checked against the oracle."""
    need_gpu()
    layers = [DeviceLayer(4096, 2048, 256, seed=0, layer=l) for l in range(43)]
    check_stack(layers, 4, 4, [0, 21, 42], columns=[0, 3])
