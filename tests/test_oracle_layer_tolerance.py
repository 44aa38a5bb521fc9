"""Pins the oracle's layer tolerance magnitude M (orc_moe_layer) by brute force.

The tolerance model: every GEMV output of the layer (router logits, gate, up and down rows, routed and
shared) may be off by up to eps * sum_j |w_j x_j| of its own inputs, and the layer output may move by
whatever those errors cause to first order. For one output element the largest such move is
sum over error sources of |d out / d source| * allowance(source), each source taking its worst sign.
This test measures that sum by central differences, one source at a time, on a layer small enough to
enumerate every source, with a forward pass written here from the dequantized matrices (numpy, binary64),
and requires the oracle's M to equal it. A dropped term, a term counted twice, a wrong derivative or
a wrong sign inside an absolute value makes M differ from the brute-force sum somewhere.
"""
import numpy as np
import pytest

import oracle
import synth

EPS = 1e-6  # relative size of the finite-difference steps


def sigmoid(v):
    return 1.0 / (1.0 + np.exp(-v))


def silu(v):
    return v * sigmoid(v)


class TinyLayer:
    def __init__(self, H, I, E, seed):
        self.H, self.I, self.E = H, I, E
        self.R = synth.router(E, H, seed, 0)
        self.pk = {}
        self.W = {}
        for name, fmt, tensor, N, K in (("G", 2, synth.GATE, I, H), ("U", 2, synth.UP, I, H), ("D", 3, synth.DOWN, H, I)):
            self.pk[name] = [synth.matrix(fmt, N, K, seed, 0, tensor, e) for e in range(E)]
            self.W[name] = [oracle.dequantize(fmt, m, N, K) for m in self.pk[name]]
        for name, tensor, N, K in (("SG", synth.SH_GATE, I, H), ("SU", synth.SH_UP, I, H), ("SD", synth.SH_DOWN, H, I)):
            self.pk[name] = synth.matrix(4, N, K, seed, 0, tensor)
            self.W[name] = oracle.dequantize(4, self.pk[name], N, K)

    def oracle_layer(self, x, k):
        p = self.pk
        return oracle.moe_layer(self.H, self.I, self.E, self.R, p["G"], p["U"], p["D"], p["SG"], p["SU"], p["SD"], x, k)


def sources(L, x, idx):
    """Every error source of one token: (kind, slot, index, allowance). kind: 'l' logit of expert
    `index`; 'g', 'u' row `index` of the gate / up output of rank `slot` (slot k: shared); 'y' row `index`
    of the down output of rank `slot` (slot k: shared)."""
    R = L.R.astype(np.float64)
    out = [("l", 0, e, float(np.abs(R[e]) @ np.abs(x))) for e in range(L.E)]
    k = len(idx)
    mats = [(L.W["G"][e], L.W["U"][e], L.W["D"][e]) for e in idx] + [(L.W["SG"], L.W["SU"], L.W["SD"])]
    for slot, (G, U, D) in enumerate(mats):
        g, u = G @ x, U @ x
        h = silu(g) * u
        ag, au, ay = np.abs(G) @ np.abs(x), np.abs(U) @ np.abs(x), np.abs(D) @ np.abs(h)
        out += [("g", slot, i, ag[i]) for i in range(L.I)]
        out += [("u", slot, i, au[i]) for i in range(L.I)]
        out += [("y", slot, i, ay[i]) for i in range(L.H)]
    assert sum(1 for s in out if s[1] == k and s[0] != "l") == 2 * L.I + L.H
    return out


def forward(L, x, idx, src=None, delta=0.0):
    """The layer output of one token with the routing fixed to idx, one source shifted by delta."""
    R = L.R.astype(np.float64)
    kind, slot, i = (src[0], src[1], src[2]) if src else (None, -1, -1)
    logits = R @ x
    if kind == "l":
        logits[i] += delta
    s = sigmoid(logits[idx])
    w = s / s.sum()
    k = len(idx)
    out = np.zeros(L.H)
    mats = [(L.W["G"][e], L.W["U"][e], L.W["D"][e]) for e in idx] + [(L.W["SG"], L.W["SU"], L.W["SD"])]
    for sl, (G, U, D) in enumerate(mats):
        g, u = G @ x, U @ x
        if sl == slot and kind == "g":
            g[i] += delta
        if sl == slot and kind == "u":
            u[i] += delta
        y = D @ (silu(g) * u)
        if sl == slot and kind == "y":
            y[i] += delta
        out += y if sl == k else w[sl] * y
    return out


def brute_force_magnitude(L, x, idx):
    """sum over sources of |central difference of the output| / EPS."""
    T = np.zeros(L.H)
    for src in sources(L, x, idx):
        d = EPS * src[3]
        if d == 0.0:
            continue
        T += np.abs(forward(L, x, idx, src, d) - forward(L, x, idx, src, -d)) / (2.0 * EPS)
    return T


@pytest.mark.parametrize("k,seed", [(1, 3), (2, 5), (3, 7)])
def test_layer_magnitude_equals_brute_force_first_order_bound(k, seed):
    L = TinyLayer(64, 32, 8, seed)
    _, vals = synth.tokens_bf16(2, 64, seed=seed)
    x = vals.astype(np.float64)
    orc = L.oracle_layer(x, k)
    for t in range(2):
        idx = [int(e) for e in orc["idx"][t]]
        # the forward pass here reproduces the oracle's output (the same definition, written apart)
        y = forward(L, x[t], idx)
        assert np.allclose(y, orc["y"][t], rtol=1e-12, atol=1e-12 * np.abs(orc["M"][t]).max())
        T = brute_force_magnitude(L, x[t], idx)
        M = orc["M"][t]
        assert np.all(M > 0)
        # equal up to the finite-difference error (second order in EPS, relative)
        assert np.allclose(M, T, rtol=1e-5, atol=0), float(np.max(np.abs(M - T) / T))


def test_magnitude_has_the_down_projection_own_term():
    """A single-expert check by hand: with k = 1 the router weight is identically 1, so M is the
    routed expert's propagated bound plus the shared expert's. The down projection's own allowance
    sum_j |D_ij h_j| must be part of it: removing it from the brute force leaves M larger."""
    L = TinyLayer(64, 32, 8, 11)
    _, vals = synth.tokens_bf16(1, 64, seed=11)
    x = vals.astype(np.float64)[0]
    orc = L.oracle_layer(x[None, :], 1)
    idx = [int(orc["idx"][0][0])]
    T_no_own = np.zeros(L.H)
    for src in sources(L, x, idx):
        if src[0] == "y" or src[3] == 0.0:
            continue
        d = EPS * src[3]
        T_no_own += np.abs(forward(L, x, idx, src, d) - forward(L, x, idx, src, -d)) / (2.0 * EPS)
    G, U, D = L.W["G"][idx[0]], L.W["U"][idx[0]], L.W["D"][idx[0]]
    h = silu(G @ x) * (U @ x)
    hs = silu(L.W["SG"] @ x) * (L.W["SU"] @ x)
    own = np.abs(D) @ np.abs(h) + np.abs(L.W["SD"]) @ np.abs(hs)
    assert np.allclose(orc["M"][0], T_no_own + own, rtol=1e-5, atol=0)
