"""Pins for the oracle's top-k, router, stable argsort, RMS normalisation and MoE layer (CPU only)."""
import itertools
import math

import numpy as np
import pytest

import oracle
import synth


def _dominant_subset(v, k):
    """Brute force over all C(n, k) subsets: the top-k set is the one whose every member beats every
    non-member under (value descending, index ascending). Exactly one subset qualifies."""
    n = len(v)
    beats = lambda a, b: v[a] > v[b] or (v[a] == v[b] and a < b)
    found = [S for S in itertools.combinations(range(n), k)
             if all(beats(a, b) for a in S for b in range(n) if b not in S)]
    assert len(found) == 1
    S = list(found[0])
    S.sort(key=lambda i: (-v[i], i))
    return S


@pytest.mark.parametrize("k", [1, 2, 3])
def test_topk_brute_force_with_ties(k):
    rng = np.random.default_rng(k)
    cases = [rng.standard_normal(8) for _ in range(40)]
    cases += [np.round(rng.standard_normal(8)) for _ in range(40)]  # many exact ties
    cases += [np.zeros(8), np.array([1, 1, 0, 0, 1, 1, 0, 0.0]), np.array([-0.0, 0.0] * 4)]
    for v in cases:
        assert list(oracle.topk(v, k)) == _dominant_subset(list(v), k)


def test_route_against_library_and_definition():
    E, H, q, k = 16, 96, 3, 4
    R = synth.router(E, H, seed=1)
    x = synth.tokens_bf16(q, H, seed=1)[1].astype(np.float64)
    r = oracle.route(R, x, k)
    ref = x @ R.astype(np.float64).T
    assert np.allclose(r["logits"], ref, rtol=0, atol=1e-14)
    assert np.allclose(r["Ml"], np.abs(x[:, None, :] * R[None, :, :].astype(np.float64)).sum(-1), rtol=1e-14)
    sig = lambda z: 1 / (1 + np.exp(-z))
    for t in range(q):
        assert list(r["idx"][t]) == _dominant_subset(list(r["logits"][t]), k)
        s = sig(r["logits"][t][r["idx"][t]])
        assert np.allclose(r["w"][t], s / s.sum(), rtol=1e-15)
        assert abs(r["w"][t].sum() - 1) < 1e-15
        assert all(np.diff(r["w"][t]) <= 0)  # descending logit -> descending weight
    assert list(r["uni"]) == sorted(set(r["idx"].ravel().tolist()))


def test_stable_argsort_against_library_and_counting_sort():
    rng = np.random.default_rng(0)
    for n, nk in [(0, 4), (1, 1), (50, 3), (12288, 256)]:
        keys = rng.integers(0, nk, n).astype(np.int32)
        perm, off = oracle.stable_argsort(keys, nk)
        assert np.array_equal(perm, np.argsort(keys, kind="stable"))
        # counting sort: positions bucketed by key in input order
        buckets = [[] for _ in range(nk)]
        for i, kk in enumerate(keys):
            buckets[kk].append(i)
        assert perm.tolist() == [i for b in buckets for i in b]
        assert np.array_equal(off, np.concatenate([[0], np.cumsum(np.bincount(keys, minlength=nk))]))


def test_rmsnorm_bf16_properties():
    rng = np.random.default_rng(2)
    r = (rng.standard_normal((3, 4096)) * np.array([[1e-3], [1.0], [50.0]])).astype(np.float32)
    u = oracle.rmsnorm_bf16(r)
    for t in range(3):
        v = r[t].astype(np.float64) / math.sqrt(np.mean(r[t].astype(np.float64) ** 2) + 1e-6)
        bits = u[t].astype(np.float32).view(np.uint32)
        assert np.all(bits & 0xFFFF == 0)  # every value is a bfloat16
        ulp = np.ldexp(1.0, np.frexp(np.abs(v))[1] - 8)
        assert np.all(np.abs(u[t] - v) <= ulp / 2)  # nearest
        tie = np.abs(u[t] - v) == ulp / 2
        assert np.all((bits[tie] >> 16) & 1 == 0)  # ties to even


# ---------------------------------------------------------------- layer invariants

H, I, E = 64, 32, 8


def _layer(seed=0, zero_routed_down=False):
    g = [synth.matrix(2, I, H, seed, 0, synth.GATE, e) for e in range(E)]
    u = [synth.matrix(2, I, H, seed, 0, synth.UP, e) for e in range(E)]
    d = [synth.matrix(3, H, I, seed, 0, synth.DOWN, e) for e in range(E)]
    if zero_routed_down:
        for m in d:
            m.reshape(-1, 14)[:, :2] = 0  # every binary16 scale 0
    sg = synth.matrix(4, I, H, seed, 0, synth.SH_GATE)
    su = synth.matrix(4, I, H, seed, 0, synth.SH_UP)
    sd = synth.matrix(4, H, I, seed, 0, synth.SH_DOWN)
    R = synth.router(E, H, seed)
    return R, g, u, d, sg, su, sd


def test_layer_tokens_are_independent():
    R, g, u, d, sg, su, sd = _layer(1)
    x = synth.tokens_bf16(4, H, seed=1)[1].astype(np.float64)
    full = oracle.moe_layer(H, I, E, R, g, u, d, sg, su, sd, x, 2)
    for t in range(4):
        one = oracle.moe_layer(H, I, E, R, g, u, d, sg, su, sd, x[t : t + 1], 2)
        assert np.array_equal(one["y"][0], full["y"][t])
        assert np.array_equal(one["M"][0], full["M"][t])
        assert np.array_equal(one["idx"][0], full["idx"][t])


def test_layer_expert_relabelling():
    """Permuting the expert ids (router rows and weights together) leaves the output unchanged and
    permutes the routing."""
    R, g, u, d, sg, su, sd = _layer(2)
    x = synth.tokens_bf16(3, H, seed=2)[1].astype(np.float64)
    a = oracle.moe_layer(H, I, E, R, g, u, d, sg, su, sd, x, 3)
    p = np.array([5, 2, 7, 0, 1, 6, 3, 4])  # new id of old expert e is p[e]
    inv = np.argsort(p)
    b = oracle.moe_layer(H, I, E, R[inv], [g[i] for i in inv], [u[i] for i in inv], [d[i] for i in inv],
                         sg, su, sd, x, 3)
    assert np.allclose(a["y"], b["y"], rtol=1e-13, atol=1e-15)
    assert np.array_equal(p[a["idx"]], b["idx"])


def test_layer_shared_only_when_routed_down_is_zero():
    R, g, u, d, sg, su, sd = _layer(3, zero_routed_down=True)
    x = synth.tokens_bf16(2, H, seed=3)[1].astype(np.float64)
    out = oracle.moe_layer(H, I, E, R, g, u, d, sg, su, sd, x, 2)
    # shared expert alone, from the GEMV oracle and the SiLU definition
    gg, _ = oracle.gemv(4, sg, I, H, x)
    uu, _ = oracle.gemv(4, su, I, H, x)
    h = gg / (1 + np.exp(-gg)) * uu
    y, _ = oracle.gemv(4, sd, H, I, h)
    assert np.allclose(out["y"], y, rtol=1e-13, atol=1e-15)


def test_layer_single_expert_weight_is_one():
    """k = 1: the normalised weight is exactly 1, so out = expert(x) + shared(x)."""
    R, g, u, d, sg, su, sd = _layer(4)
    x = synth.tokens_bf16(1, H, seed=4)[1].astype(np.float64)
    out = oracle.moe_layer(H, I, E, R, g, u, d, sg, su, sd, x, 1)
    assert out["w"][0, 0] == 1.0
    e = out["idx"][0, 0]

    def expert(fg, fd, G, U, D):
        gg, _ = oracle.gemv(fg, G, I, H, x)
        uu, _ = oracle.gemv(fg, U, I, H, x)
        y, _ = oracle.gemv(fd, D, H, I, gg / (1 + np.exp(-gg)) * uu)
        return y

    ref = expert(2, 3, g[e], u[e], d[e]) + expert(4, 4, sg, su, sd)
    assert np.allclose(out["y"], ref, rtol=1e-12, atol=1e-15)


def test_layer_combine_is_linear_in_routed_down():
    """Doubling every routed down-projection scale (exact in binary16) doubles the routed part."""
    R, g, u, d, sg, su, sd = _layer(5)
    x = synth.tokens_bf16(3, H, seed=5)[1].astype(np.float64)
    a = oracle.moe_layer(H, I, E, R, g, u, d, sg, su, sd, x, 2)
    d2 = []
    for m in d:
        m2 = m.copy()
        s = m2.reshape(-1, 14)[:, :2].copy().view(np.uint16).ravel()
        s2 = (s.view(np.float16).astype(np.float64) * 2).astype(np.float16).view(np.uint16)
        m2.reshape(-1, 14)[:, :2] = s2.view(np.uint8).reshape(-1, 2)
        d2.append(m2)
    _, _, _, dz, _, _, _ = _layer(5, zero_routed_down=True)
    b = oracle.moe_layer(H, I, E, R, g, u, d2, sg, su, sd, x, 2)
    z = oracle.moe_layer(H, I, E, R, g, u, dz, sg, su, sd, x, 2)  # shared part only
    assert np.allclose(b["y"] - z["y"], 2 * (a["y"] - z["y"]), rtol=1e-12, atol=1e-14)


def test_layer_forced_routing_and_magnitude():
    R, g, u, d, sg, su, sd = _layer(6)
    x = synth.tokens_bf16(2, H, seed=6)[1].astype(np.float64)
    a = oracle.moe_layer(H, I, E, R, g, u, d, sg, su, sd, x, 2)
    f = oracle.moe_layer(H, I, E, R, g, u, d, sg, su, sd, x, 2, idx_force=a["idx"])
    assert np.array_equal(a["y"], f["y"])
    assert np.all(a["M"] >= np.abs(a["y"]))
    swapped = a["idx"][:, ::-1].copy()
    s = oracle.moe_layer(H, I, E, R, g, u, d, sg, su, sd, x, 2, idx_force=swapped)
    assert np.allclose(s["y"], a["y"], rtol=1e-13, atol=1e-15)  # rank order does not change the sum
