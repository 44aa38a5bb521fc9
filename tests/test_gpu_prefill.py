"""moe_layer_prefill against the oracle: every token's top-k consistent with its logits, the logits
within 1e-4 of the oracle's, the argsort bit-exact against the oracle's stable argsort, and each
checked token's weights and output against the oracle's layer with the same routing (output within
2e-3 * M, the first-order error magnitude)."""
import numpy as np
import pytest
import torch

import bit_block_quantized_wt_b300 as fpx
import oracle
import synth
from gpu_util import DeviceLayer, dev, host, need_gpu, read_status, topk_of

pytestmark = pytest.mark.gpu
TOL = 2e-3


def run_prefill(L, bits, k):
    T = bits.shape[0]
    ws_b = fpx.moe_prefill_workspace_bytes(L.c, T, k)
    assert ws_b > 0
    ws = torch.empty(ws_b, dtype=torch.uint8, device="cuda")
    y = torch.full((T, L.H), float("nan"), device="cuda")
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, device="cuda")
    lg = torch.empty(T, L.E, device="cuda")
    perm = torch.empty(T * k, dtype=torch.int32, device="cuda")
    offs = torch.empty(L.E + 1, dtype=torch.int32, device="cuda")
    fpx.moe_layer_prefill(L.c, dev(bits), T, k, y, ws, ws_b, idx_out=idx, w_out=w, logits_out=lg, perm_out=perm,
                          offsets_out=offs)
    assert read_status(ws[:4].view(torch.int32)) == 0
    return host(y), host(idx), host(w), host(lg), host(perm), host(offs)


def check_prefill(L, bits, vals, k, sample):
    y, idx, w, lg, perm, offs = run_prefill(L, bits, k)
    T = bits.shape[0]
    assert np.all(np.isfinite(y))
    for t in range(T):
        assert list(idx[t]) == list(topk_of(lg[t], k))
    p_ref, o_ref = oracle.stable_argsort(idx.ravel(), L.E)
    assert np.array_equal(perm, p_ref) and np.array_equal(offs, o_ref)
    sample = np.asarray(sample)
    orc = L.oracle(vals[sample].astype(np.float64), k, idx_force=idx[sample])
    assert np.all(np.abs(lg[sample] - orc["logits"]) <= 1e-4 + 1e-4 * np.abs(orc["logits"]))
    assert np.allclose(w[sample], orc["w"], rtol=1e-5, atol=0)
    err = np.abs(y[sample].astype(np.float64) - orc["y"])
    assert np.all(err <= TOL * orc["M"]), float((err / orc["M"]).max())
    return y, idx


@pytest.mark.parametrize("T,k", [(100, 4), (64, 1), (1, 2), (130, 8)])
def test_prefill_small(T, k):
    """H = I = 512, 16 experts: every token checked; T not a multiple of the 64-pair tile, experts
    with several tiles and experts with none."""
    need_gpu()
    L = DeviceLayer(512, 512, 16, seed=T + k)
    bits, vals = synth.tokens_bf16(T, 512, seed=k)
    check_prefill(L, bits, vals, k, range(T))


def test_prefill_matches_decode_routing():
    """The prefill routes a token exactly as the decode layer does."""
    need_gpu()
    L = DeviceLayer(512, 512, 16, seed=5)
    bits, vals = synth.tokens_bf16(4, 512, seed=9)
    y, idx = check_prefill(L, bits, vals, 4, range(4))
    ws_b = fpx.moe_workspace_bytes(L.c, 4, 4)
    ws = torch.empty(ws_b, dtype=torch.uint8, device="cuda")
    yd = torch.empty(4, 512, device="cuda")
    idd = torch.empty(4, 4, dtype=torch.int32, device="cuda")
    fpx.moe_layer_decode(L.c, dev(bits), 4, 4, yd, ws, ws_b, idx_out=idd)
    assert np.array_equal(host(idd), idx)


def test_prefill_exact_ties_go_to_lower_index():
    """Duplicate router rows give equal logits: the lower expert index is selected first."""
    need_gpu()
    L = DeviceLayer(512, 512, 16, seed=3)
    R = L.R_host.copy()
    for a, b in [(2, 9), (5, 6), (0, 13)]:
        R[b] = R[a]
    L.R_host = R
    L.router.copy_(dev(R))
    bits, vals = synth.tokens_bf16(64, 512, seed=3)
    y, idx, w, lg, perm, offs = run_prefill(L, bits, 6)
    for t in range(64):
        for a, b in [(2, 9), (5, 6), (0, 13)]:
            assert lg[t, a] == lg[t, b]
            r = list(idx[t])
            if b in r:
                assert a in r and r.index(a) < r.index(b)


def test_prefill_full_size_config5():
    """2048 tokens, top-6, hidden 4096, 256 experts: routing and argsort for every token; the output of
    at least 64 tokens: for the 8 experts with the most pairs, the tokens at both ends of every 64-pair
    tile of the expert's group (the grouped GEMM's tile edges and the group's ragged tail), then the
    first and last token and seeded random ones."""
    need_gpu()
    L = DeviceLayer(4096, 2048, 256, seed=0, layer=0)
    bits, vals = synth.tokens_bf16(2048, 4096, seed=0)
    k = 6
    y, idx, w, lg, perm, offs = run_prefill(L, bits, k)
    for t in range(2048):
        assert list(idx[t]) == list(topk_of(lg[t], k))
    p_ref, o_ref = oracle.stable_argsort(idx.ravel(), L.E)
    assert np.array_equal(perm, p_ref) and np.array_equal(offs, o_ref)
    sizes = np.diff(offs)
    picked = {0, 2047}
    for e in np.argsort(-sizes, kind="stable")[:8]:
        n = int(sizes[e])
        for pos in sorted({p for t0 in range(0, n, 64) for p in (t0, min(t0 + 63, n - 1))}):
            picked.add(int(perm[offs[e] + pos]) // k)
    rng = np.random.default_rng(5)
    while len(picked) < 64:
        picked.add(int(rng.integers(2048)))
    sample = np.array(sorted(picked))
    orc = L.oracle(vals[sample].astype(np.float64), k, idx_force=idx[sample])
    assert np.all(np.abs(lg[sample] - orc["logits"]) <= 1e-4 + 1e-4 * np.abs(orc["logits"]))
    assert np.allclose(w[sample], orc["w"], rtol=1e-5, atol=0)
    err = np.abs(y[sample].astype(np.float64) - orc["y"])
    assert np.all(err <= TOL * orc["M"]), float((err / orc["M"]).max())
