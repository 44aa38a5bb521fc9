"""Pins for the oracle's importance-weighted quantizer (CPU only). It must pick, per block, the
candidate scale whose quantization has the least importance-weighted squared error: checked by brute
force through the (separately pinned) fixed-scale quantizer and decoder, plus invariants (never worse
than the plain quantizer, invariant to scaling the importance by a power of two, None = all ones) and
the error statuses."""
import numpy as np
import pytest

import oracle


def blocks_of(fmt, packed, N, K):
    bb = oracle.block_bytes(fmt)
    return np.frombuffer(packed[: N * K // 32 * bb].tobytes(), np.uint8).reshape(N * K // 32, bb)


def werr(W, Wq_vals, imp):
    """Per-block sum of imp * (w - w_hat)^2 in weight order (Python binary64)."""
    N, K = W.shape
    out = []
    for r in range(N):
        for b in range(K // 32):
            e = 0.0
            for j in range(32):
                k = 32 * b + j
                d = float(W[r, k]) - float(Wq_vals[r, k])
                e += (1.0 if imp is None else float(imp[k])) * (d * d)
            out.append(e)
    return np.array(out)


def candidates(fmt, block):
    """The candidate scales of the definition: binary16 (amax / Kmax) f, f = 0.60 .. 1.35 (FP2/FP3);
    E8M0 exponents around the plain one (FP4), as the fixed-scale quantizer's scale values."""
    amax = float(np.max(np.abs(block.astype(np.float64))))
    if fmt in (2, 3):
        kmax = 3 if fmt == 2 else 7
        c = [np.float16(amax / kmax * ((12 + j) / 20.0)) for j in range(16)]
        return [np.float32(v) for v in c if np.isfinite(v)]
    e0 = 0 if amax == 0 else min(254, max(0, int(np.floor(np.log2(amax))) - 2 + 127))
    return [np.float32(2.0 ** (min(254, max(0, e0 + j)) - 127)) for j in (-1, 0, 1)]


@pytest.mark.parametrize("fmt", [2, 3, 4])
def test_brute_force_through_fixed_scales(fmt):
    rng = np.random.default_rng(fmt)
    N, K = 3, 96
    W = (rng.standard_normal((N, K)) * rng.uniform(0.01, 2.0, (N, 1))).astype(np.float32)
    imp = rng.uniform(0.0, 2.0, K).astype(np.float32)
    st, got = oracle.quantize_weighted(fmt, W, imp)
    assert st == 0
    gb = blocks_of(fmt, got, N, K)
    for r in range(N):
        for b in range(K // 32):
            blk = W[r : r + 1, 32 * b : 32 * b + 32]
            best, best_bytes = None, None
            for s in candidates(fmt, blk):
                st2, q = oracle.quantize(fmt, blk, scales=np.array([s], np.float32))
                assert st2 == 0
                vals = oracle.dequantize(fmt, q, 1, 32)
                e = werr(blk, vals, imp[32 * b : 32 * b + 32])[0]
                if best is None or e < best:
                    best, best_bytes = e, blocks_of(fmt, q, 1, 32)[0]
            assert np.array_equal(gb[r * (K // 32) + b], best_bytes), (r, b)


@pytest.mark.parametrize("fmt", [2, 3, 4])
def test_never_worse_than_plain_and_invariances(fmt):
    rng = np.random.default_rng(10 + fmt)
    N, K = 8, 128
    W = rng.standard_normal((N, K)).astype(np.float32) * 0.1
    imp = rng.uniform(0.0, 3.0, K).astype(np.float32)
    st, qw = oracle.quantize_weighted(fmt, W, imp)
    st0, qp = oracle.quantize(fmt, W)
    assert st == 0 and st0 == 0
    ew = werr(W, oracle.dequantize(fmt, qw, N, K), imp)
    ep = werr(W, oracle.dequantize(fmt, qp, N, K), imp)
    assert np.all(ew <= ep)
    assert np.sum(ew) < np.sum(ep)  # the search does find better scales on random data
    _, q4 = oracle.quantize_weighted(fmt, W, imp * 4)  # power-of-two scaling: every error scales exactly
    assert np.array_equal(q4, qw)
    _, qn = oracle.quantize_weighted(fmt, W, None)
    _, q1 = oracle.quantize_weighted(fmt, W, np.ones(K, np.float32))
    assert np.array_equal(qn, q1)


def test_single_weight_importance():
    """All importance on one weight: its own error is the least among the candidates."""
    rng = np.random.default_rng(7)
    W = rng.standard_normal((1, 32)).astype(np.float32)
    imp = np.zeros(32, np.float32); imp[5] = 1.0
    st, q = oracle.quantize_weighted(2, W, imp)
    assert st == 0
    v = oracle.dequantize(2, q, 1, 32)
    mine = abs(float(W[0, 5]) - float(v[0, 5]))
    for s in candidates(2, W):
        _, qq = oracle.quantize(2, W, scales=np.array([s], np.float32))
        assert mine <= abs(float(W[0, 5]) - float(oracle.dequantize(2, qq, 1, 32)[0, 5]))


def test_error_statuses():
    W = np.ones((1, 32), np.float32)
    imp = np.ones(32, np.float32)
    bad = imp.copy(); bad[3] = -1.0
    assert oracle.quantize_weighted(2, W, bad)[0] == oracle.ERANGE
    bad[3] = np.nan
    assert oracle.quantize_weighted(3, W, bad)[0] == oracle.ERANGE
    W2 = W.copy(); W2[0, 0] = np.inf
    assert oracle.quantize_weighted(4, W2, imp)[0] == oracle.ERANGE
