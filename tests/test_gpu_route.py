"""moe_route_topk: top-k bit-exact against the GPU's own binary32 logits, logits and weights within
tolerance of the oracle, union exact."""
import numpy as np
import pytest
import torch

import bit_block_quantized_wt_b300 as fpx
import oracle
import synth
from gpu_util import dev, host, need_gpu, topk_of

pytestmark = pytest.mark.gpu


def route(R, bits, k):
    E, H = R.shape
    q = bits.shape[0]
    lg = torch.empty(q, E, device="cuda")
    idx = torch.empty(q, k, dtype=torch.int32, device="cuda")
    w = torch.empty(q, k, device="cuda")
    uni = torch.empty(q * k, dtype=torch.int32, device="cuda")
    n = torch.empty(1, dtype=torch.int32, device="cuda")
    fpx.moe_route_topk(dev(R), E, H, dev(bits), q, k, lg, idx, w, uni, n)
    return host(lg), host(idx), host(w), host(uni), int(host(n)[0])


def check_route(R, bits, vals, k):
    lg, idx, w, uni, n = route(R, bits, k)
    ref = oracle.route(R, vals.astype(np.float64), k)
    assert np.all(np.abs(lg - ref["logits"]) <= 2e-3 * ref["Ml"])
    for t in range(bits.shape[0]):
        assert list(idx[t]) == list(topk_of(lg[t], k))
        s = 1 / (1 + np.exp(-lg[t][idx[t]].astype(np.float64)))
        assert np.allclose(w[t], s / s.sum(), rtol=2e-6, atol=0)
    assert n == len(set(idx.ravel().tolist()))
    assert list(uni[:n]) == sorted(set(idx.ravel().tolist()))
    return lg, idx


@pytest.mark.parametrize("E,H,q,k", [(8, 64, 1, 1), (8, 64, 4, 3), (16, 256, 3, 8), (64, 512, 4, 6), (1024, 256, 2, 8),
                                     (256, 4096, 4, 4), (256, 4096, 4, 6), (9, 128, 3, 4), (1023, 64, 4, 8)])
def test_route_matches_oracle(E, H, q, k):
    need_gpu()
    R = synth.router(E, H, seed=E + H)
    bits, vals = synth.tokens_bf16(q, H, seed=q)
    check_route(R, bits, vals, k)


def test_route_exact_ties_go_to_lower_index():
    """Duplicate router rows give bit-identical logits: the lower expert index must win."""
    need_gpu()
    E, H = 16, 128
    R = synth.router(E, H, seed=3)
    for a, b in [(2, 9), (5, 6), (11, 15), (0, 13)]:
        R[b] = R[a]
    bits, vals = synth.tokens_bf16(4, H, seed=3)
    lg, idx = check_route(R, bits, vals, 8)
    for t in range(4):
        for a, b in [(2, 9), (5, 6), (11, 15), (0, 13)]:
            assert lg[t, a] == lg[t, b]
            ia, ib = list(idx[t]).index(a) if a in idx[t] else 99, list(idx[t]).index(b) if b in idx[t] else 99
            if ib != 99:
                assert ia < ib
