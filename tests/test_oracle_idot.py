"""Pins for the oracle's integer-dot activations and GEMV (CPU only): a hand-worked fixture, a brute
force of the exponent and of the rounding on exact rationals, the error bound of the grid, power-of-two
and sign symmetry, and the variant's GEMV against the plain GEMV within that bound."""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "act16.txt")


def parse_value(s):
    m, k = s.split("*2^")
    return float(np.ldexp(float(m), int(k)))


def read_cases():
    cases, cur = [], None
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *vals = line.split()
        if key == "case":
            cur = {"name": vals[0], "x": np.zeros(32), "X": np.zeros(32, np.int64)}
            cases.append(cur)
        elif key == "x":
            cur["x"][int(vals[0])] = parse_value(vals[1])
        elif key == "X":
            cur["X"][int(vals[0])] = int(vals[1])
        else:
            cur["e"] = int(vals[0])
    return cases


def to_bf16(x):
    """binary32 -> nearest bfloat16 (ties to even), as binary64 values."""
    b = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000
    return b.astype(np.uint32).view(np.float32).astype(np.float64)


def test_hand_worked_fixture():
    cases = read_cases()
    assert len(cases) == 6
    x = np.stack([c["x"] for c in cases])  # one column per case
    st, X, e, xhat = oracle.quantize_act16(x)
    assert st == 0
    for i, c in enumerate(cases):
        assert e[i, 0] == c["e"], c["name"]
        assert list(X[i]) == list(c["X"]), c["name"]
        assert np.array_equal(xhat[i], np.ldexp(c["X"].astype(np.float64), c["e"] - 14)), c["name"]


def brute(block):
    """Exponent by search and nearest integer (ties to even) on exact rationals."""
    vals = [Fraction(float(v)) for v in block]
    a = max(abs(v) for v in vals)
    if a == 0:
        return 0, [0] * 32
    e = -200
    while not a < Fraction(2) ** e:
        e += 1
    assert Fraction(2) ** (e - 1) <= a
    out = []
    for v in vals:
        s = v * Fraction(2) ** (14 - e)
        lo = s.numerator // s.denominator
        d = s - lo
        if d > Fraction(1, 2) or (d == Fraction(1, 2) and lo % 2 == 1):
            lo += 1
        out.append(lo)
    return e, out


def test_brute_force_blocks():
    rng = np.random.default_rng(5)
    blocks = []
    for i in range(60):
        scale = np.ldexp(1.0, int(rng.integers(-40, 40)))
        b = (rng.standard_normal(32) * scale).astype(np.float32)
        if i % 3 == 0:  # exact ties: odd multiples of half a grid step
            e = int(np.frexp(np.max(np.abs(b)))[1])
            b[5:9] = np.ldexp(np.array([1, 3, 5, -7], np.float64), e - 15).astype(np.float32)
        if i % 5 == 0:
            b[rng.integers(0, 32, 6)] = 0.0
        blocks.append(b)
    blocks.append(np.zeros(32, np.float32))
    x = np.stack(blocks).astype(np.float64)
    st, X, e, _ = oracle.quantize_act16(x)
    assert st == 0
    for i, b in enumerate(blocks):
        be, bX = brute(b)
        assert e[i, 0] == be and list(X[i]) == bX, i


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_grid_bounds(dtype):
    rng = np.random.default_rng(11)
    x = rng.standard_normal((4, 4096)) * np.exp(rng.uniform(-6, 6, (4, 128))).repeat(32, axis=1)
    x = x.astype(np.float32).astype(np.float64)
    if dtype == "bf16":
        x = to_bf16(x)
    st, X, e, xhat = oracle.quantize_act16(x)
    assert st == 0
    eb = np.repeat(e, 32, axis=1)
    assert np.all(np.abs(X) <= 1 << 14)
    assert np.all(np.abs(xhat - x) <= np.ldexp(1.0, eb - 15))
    bmax = np.abs(X).reshape(4, -1, 32).max(axis=2)
    assert np.all(bmax >= 1 << 13)  # the largest entry lands in [2^13, 2^14]
    if dtype == "bf16":  # 8 significant bits: exact down to 2^(e-7)
        big = np.abs(x) >= np.ldexp(1.0, eb - 7)
        assert np.array_equal(xhat[big], x[big])


def test_power_of_two_and_sign_symmetry():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((3, 256))
    x = x.astype(np.float32).astype(np.float64)
    _, X, e, xhat = oracle.quantize_act16(x)
    for k in (-30, -1, 1, 17):
        _, X2, e2, xhat2 = oracle.quantize_act16(np.ldexp(x, k))
        assert np.array_equal(X2, X) and np.array_equal(e2, e + k)
        assert np.array_equal(xhat2, np.ldexp(xhat, k))
    _, X3, e3, _ = oracle.quantize_act16(-x)
    assert np.array_equal(X3, -X) and np.array_equal(e3, e)


def test_errors():
    x = np.zeros((1, 64))
    x[0, 40] = np.nan
    assert oracle.quantize_act16(x)[0] == oracle.ERANGE
    assert oracle.quantize_act16(np.zeros((1, 48)))[0] == oracle.EINVAL


@pytest.mark.parametrize("fmt", [2, 3, 4])
def test_gemv_idot_within_grid_bound(fmt):
    N, K = 40, 512
    Wq = synth.matrix(fmt, N, K, seed=fmt + 70)
    rng = np.random.default_rng(fmt)
    x = (rng.standard_normal((4, K)) * np.exp(rng.uniform(-3, 3, (4, K)))).astype(np.float32).astype(np.float64)
    y, _ = oracle.gemv(fmt, Wq, N, K, x)
    yi, _ = oracle.gemv_idot(fmt, Wq, N, K, x)
    W = oracle.dequantize(fmt, Wq, N, K)
    _, _, e, _ = oracle.quantize_act16(x)
    step = np.ldexp(1.0, np.repeat(e, 32, axis=1) - 15)  # half a grid step per entry
    bound = np.abs(W) @ step.T  # [N][q]
    assert np.all(np.abs(yi - y) <= bound.T * (1 + 1e-12))
    assert np.max(np.abs(yi - y)) > 0  # the grid does round these inputs
    # inputs already on the grid (small integers, block max 3 or more) give the exact product
    xi = rng.integers(-3, 4, (4, K)).astype(np.float64)
    xi[:, ::32] = 3.0
    yi2, _ = oracle.gemv_idot(fmt, Wq, N, K, xi)
    y2, _ = oracle.gemv(fmt, Wq, N, K, xi)
    assert np.array_equal(yi2, y2)


def test_gemv_idot_special_cases():
    """All-zero activations give exact zeros; one nonzero entry per block lies on the grid (it is the
    block maximum, 8 significant bits at most) and gives the plain product exactly."""
    N, K = 9, 256
    Wq = synth.matrix(2, N, K, seed=3)
    yi, M = oracle.gemv_idot(2, Wq, N, K, np.zeros((2, K)))
    assert np.all(yi == 0.0) and np.all(M == 0.0)
    x = np.zeros((2, K))
    x[0, ::32] = [1.5, -0.375, 3.0, 0.75 * 2.0 ** -20, 2.0 ** 20, -7.0, 0.25, 96.0]
    x[1, 5::32] = -np.ldexp(1.0, np.arange(-4, 4))
    yi, _ = oracle.gemv_idot(2, Wq, N, K, x)
    y, _ = oracle.gemv(2, Wq, N, K, x)
    assert np.array_equal(yi, y)
