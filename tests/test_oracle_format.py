"""Pins for the oracle's block decode, GEMV and quantizer (CPU only).

Each test checks the oracle against something other than itself: the sizes the pages print, hand-worked
blocks, numpy's binary16 conversion, the OCP E2M1 bit-field definition, exactly rounded sums
(math.fsum) and brute force over the codebooks.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth
from conftest import load_blocks, load_kv

PAGES = load_kv("pages_numbers.txt")
HAND = load_blocks("hand_blocks.txt")


def test_block_sizes_match_pages():
    assert oracle.block_bytes(2) == PAGES["fp2_block_bytes"]
    for fmt, key in [(2, "fp2_bits_per_weight"), (3, "fp3_bits_per_weight"), (4, "fp4_bits_per_weight")]:
        assert oracle.block_bytes(fmt) * 8 / PAGES["weights_per_block"] == PAGES[key]


def test_matrix_bytes_and_padding():
    assert oracle.matrix_bytes(2, 1024, 1024) == 327680
    assert oracle.matrix_bytes(2, 2048, 4096) == 2621440
    assert oracle.matrix_bytes(3, 4096, 2048) == 3670016
    assert oracle.matrix_bytes(4, 2048, 4096) == 4456448
    assert oracle.matrix_bytes(2, 1, 32) == 16
    assert oracle.matrix_bytes(4, 3, 32) == 64
    assert oracle.matrix_bytes(2, 0, 32) == 0
    assert oracle.matrix_bytes(2, 4, 33) == -1
    assert oracle.matrix_bytes(5, 4, 32) == -1


def test_recipe_average_from_tensor_sizes():
    """The MoE recipe (FP2 gate/up, FP3 down, FP4 shared) recomputed from tensor sizes, beside the
    pages' whole-model figure 102.3 GB / 284B parameters (which also covers the non-MoE layers)."""
    H, I, E = 4096, 2048, 256
    routed = E * (2 * oracle.matrix_bytes(2, I, H) + oracle.matrix_bytes(3, H, I))
    p_routed = E * 3 * H * I
    shared = 2 * oracle.matrix_bytes(4, I, H) + oracle.matrix_bytes(4, H, I)
    router = E * H * 4
    avg_routed = routed * 8 / p_routed
    avg_shared = (routed + shared) * 8 / (p_routed + 3 * H * I)
    avg_router = (routed + shared + router) * 8 / (p_routed + 3 * H * I + E * H)
    pages = PAGES["model_bytes_gb"] * 1e9 * 8 / PAGES["model_params"]
    assert abs(pages - PAGES["average_bits_per_param"]) < 0.005
    assert avg_routed == pytest.approx(17 / 6, abs=1e-12)  # (2.5 + 2.5 + 3.5) / 3
    assert avg_shared == pytest.approx(2.8388, abs=1e-4)
    assert avg_router == pytest.approx(2.8436, abs=1e-4)
    assert abs(avg_router - pages) < 0.05


def test_pages_bookkeeping():
    assert PAGES["model_bytes_gb"] * 1e9 / 2**30 == pytest.approx(PAGES["model_gib"], abs=0.05)
    assert PAGES["model_params"] * 2 / 1e9 == PAGES["fp16_model_gb"]
    total = PAGES["model_bytes_gb"] + PAGES["draft_gb"] + PAGES["headroom_gb"]
    assert total == pytest.approx(PAGES["unified_memory_gb"], abs=1e-9)


@pytest.mark.parametrize("row", HAND, ids=lambda r: r["name"])
def test_hand_worked_blocks(row):
    blk = np.frombuffer(row["blk"], np.uint8)
    assert len(blk) == oracle.block_bytes(row["fmt"])
    ramp = np.arange(32, dtype=np.float64)
    y, M = oracle.gemv(row["fmt"], blk, 1, 32, ramp[None, :])
    assert y[0, 0] == float(Fraction(row["dot"]))
    assert M[0, 0] == float(Fraction(row["abs"]))
    y1, _ = oracle.gemv(row["fmt"], blk, 1, 32, np.ones((1, 32)))
    assert y1[0, 0] == float(Fraction(row["ones"]))


def test_hand_block_values_per_weight():
    d = 2.0**-5
    rows = {r["name"]: r for r in HAND}
    w2 = oracle.decode_block(2, np.frombuffer(rows["fp2_ramp"]["blk"], np.uint8))
    assert list(w2) == [d * (2 * (j % 4) - 3) for j in range(32)]
    w3 = oracle.decode_block(3, np.frombuffer(rows["fp3_ramp"]["blk"], np.uint8))
    assert list(w3) == [d * (2 * (j % 8) - 7) for j in range(32)]


def _ocp_e2m1(code):
    """E2M1 from its bit fields (OCP Microscaling Formats v1.0): sign bit 3, exponent bits 2..1 with
    bias 1, mantissa bit 0; exponent 0 is subnormal (0.5 * M)."""
    s, E, M = code >> 3, (code >> 1) & 3, code & 1
    mag = 0.5 * M if E == 0 else 2.0 ** (E - 1) * (1 + M / 2)
    return -mag if s else mag


@pytest.mark.parametrize("e", [0, 1, 100, 126, 127, 128, 200, 254])
def test_fp4_decode_matches_ocp_definition(e):
    blk = np.zeros(17, np.uint8)
    blk[0] = e
    for j in range(32):
        blk[1 + j // 2] |= (j % 16) << (4 * (j % 2))
    w = oracle.decode_block(4, blk)
    for j in range(32):
        ref = math.ldexp(_ocp_e2m1(j % 16), e - 127)
        assert w[j] == ref and math.copysign(1, w[j]) == math.copysign(1, ref)


def test_fp4_scale_255_is_invalid():
    blk = np.zeros(17, np.uint8)
    blk[0] = 255
    with pytest.raises(RuntimeError):
        oracle.decode_block(4, blk)


def test_binary16_scale_decode_all_patterns():
    """Every finite binary16 scale pattern: code 2 decodes to d and code 3 to 3d (numpy float16)."""
    bits = np.arange(65536, dtype=np.uint16)
    vals = bits.view(np.float16)
    fin = np.isfinite(vals)
    bits, vals = bits[fin], vals[fin].astype(np.float64)
    n = bits.size
    m = np.zeros((n, 10), np.uint8)
    m[:, 0] = bits & 0xFF
    m[:, 1] = bits >> 8
    m[:, 2:] = 0xAA  # codes 2
    W = oracle.dequantize(2, m.reshape(-1), n, 32)
    assert np.array_equal(W[:, 0], vals)
    m[:, 2:] = 0xFF  # codes 3
    W = oracle.dequantize(2, m.reshape(-1), n, 32)
    assert np.array_equal(W[:, 5], 3 * vals)


@pytest.mark.parametrize("fmt", [2, 3, 4])
def test_gemv_sum_is_exactly_rounded(fmt):
    """Products of decoded weights and bfloat16 activations are exact in binary64, so math.fsum gives
    the exactly rounded dot product; the oracle's naive sum stays within 1e-12 * sum|w x| of it."""
    N, K, q = 24, 512, 3
    Wq = synth.matrix(fmt, N, K, seed=7)
    x = synth.tokens_bf16(q, K, seed=7)[1].astype(np.float64)
    y, M = oracle.gemv(fmt, Wq, N, K, x)
    W = oracle.dequantize(fmt, Wq, N, K)
    for t in range(q):
        for n in range(N):
            exact = math.fsum(W[n] * x[t])
            assert abs(y[t, n] - exact) <= 1e-12 * M[t, n]
            assert M[t, n] == pytest.approx(math.fsum(np.abs(W[n] * x[t])), rel=1e-13)


@pytest.mark.parametrize("fmt", [2, 3, 4])
def test_gemv_closed_forms(fmt):
    N, K = 9, 96
    Wq = synth.matrix(fmt, N, K, seed=3)
    W = oracle.dequantize(fmt, Wq, N, K)
    for j in [0, 31, 32, 95]:
        e = np.zeros((1, K))
        e[0, j] = 1.0
        y, _ = oracle.gemv(fmt, Wq, N, K, e)
        assert np.array_equal(y[0], W[:, j])  # x = e_j gives column j exactly
    y, _ = oracle.gemv(fmt, Wq, N, K, np.ones((1, K)))
    assert np.allclose(y[0], W.sum(axis=1), rtol=0, atol=1e-15)
    # q columns are independent: a q=3 call equals three q=1 calls exactly
    x = synth.tokens_bf16(3, K, seed=4)[1].astype(np.float64)
    y3, M3 = oracle.gemv(fmt, Wq, N, K, x)
    for t in range(3):
        y1, M1 = oracle.gemv(fmt, Wq, N, K, x[t : t + 1])
        assert np.array_equal(y1[0], y3[t]) and np.array_equal(M1[0], M3[t])


# ---------------------------------------------------------------- quantizer

def _codebook(fmt, scale):
    if fmt == 2:
        return {c: scale * (2 * c - 3) for c in range(4)}
    if fmt == 3:
        return {c: scale * (2 * c - 7) for c in range(8)}
    return {c: math.ldexp(_ocp_e2m1(c), 0) * scale for c in range(16)}


@pytest.mark.parametrize("fmt", [2, 3, 4])
def test_quantize_round_trip_with_given_scales(fmt):
    N, K = 16, 256
    Wq = synth.matrix(fmt, N, K, seed=11)
    W = oracle.dequantize(fmt, Wq, N, K)
    blocks = Wq.reshape(N * K // 32, -1)
    if fmt == 4:
        scales = np.ldexp(1.0, blocks[:, 0].astype(np.int64) - 127)
    else:
        scales = (blocks[:, 0].astype(np.uint16) | (blocks[:, 1].astype(np.uint16) << 8)).view(np.float16)
    st, out = oracle.quantize(fmt, W.astype(np.float32), scales.astype(np.float32))
    assert st == 0
    assert np.array_equal(out[: Wq.size], Wq)


@pytest.mark.parametrize("fmt", [2, 3, 4])
def test_quantize_round_trip_without_scales(fmt):
    """Blocks holding a maximum-magnitude code reproduce their own scale and codes."""
    N, K = 64, 256
    Wq = synth.matrix(fmt, N, K, seed=12)
    W = oracle.dequantize(fmt, Wq, N, K)
    st, out = oracle.quantize(fmt, W.astype(np.float32))
    assert st == 0
    bb = oracle.block_bytes(fmt)
    Wb = W.reshape(-1, 32)
    top = {2: 3, 3: 7, 4: 4}[fmt]
    nmax = 0
    for b in range(Wb.shape[0]):
        scale = np.abs(oracle.decode_block(fmt, Wq[b * bb : (b + 1) * bb])).max()
        unit = _block_unit(fmt, Wq[b * bb : (b + 1) * bb])
        if np.abs(Wb[b]).max() >= top * unit and scale > 0:
            nmax += 1
            assert np.array_equal(out[b * bb : (b + 1) * bb], Wq[b * bb : (b + 1) * bb])
    assert nmax > Wb.shape[0] * 0.9


def _block_unit(fmt, blk):
    if fmt == 4:
        return math.ldexp(1.0, int(blk[0]) - 127)
    return float(np.array([int(blk[0]) | (int(blk[1]) << 8)], np.uint16).view(np.float16)[0])


@pytest.mark.parametrize("fmt", [2, 3, 4])
def test_quantize_is_nearest_level_by_brute_force(fmt):
    rng = np.random.default_rng(5)
    W = (rng.standard_normal((8, 128)) * 0.1).astype(np.float32)
    W[0, :8] = [0.0, -0.0, 1e-30, -1e-30, 0.1, -0.1, 0.3, -0.3]
    st, out = oracle.quantize(fmt, W)
    assert st == 0
    bb = oracle.block_bytes(fmt)
    for b in range(W.size // 32):
        blk = out[b * bb : (b + 1) * bb]
        vals = oracle.decode_block(fmt, blk)
        book = _codebook(fmt, _block_unit(fmt, blk))
        v = W.reshape(-1, 32)[b].astype(np.float64)
        amax = np.abs(v).max()
        if fmt == 4:
            e = (math.frexp(amax)[1] - 1) - 2 + 127 if amax > 0 else 0
            assert blk[0] == max(0, min(254, e))
        else:
            ref = np.float16(amax / (3 if fmt == 2 else 7))  # numpy: correctly rounded
            assert _block_unit(fmt, blk) == float(ref)
        for j in range(32):
            best = min(abs(c - v[j]) for c in book.values())
            assert abs(vals[j] - v[j]) == best
            assert math.copysign(1, vals[j]) == math.copysign(1, v[j]) or vals[j] != 0 and v[j] == 0


def test_quantize_ties():
    """Exact midpoints: FP2/FP3 go to the smaller magnitude, FP4 to the even E2M1 code."""
    d = 0.25
    W = np.zeros((1, 32), np.float32)
    W[0, :4] = [2 * d, -2 * d, 3 * d, 3 * d]  # amax = 3d -> scale d for FP2
    st, out = oracle.quantize(2, W)
    v = oracle.decode_block(2, out[:10])
    assert list(v[:4]) == [d, -d, 3 * d, 3 * d]
    W = np.zeros((1, 32), np.float32)
    W[0, :8] = [7 * d, 2 * d, 4 * d, 6 * d, -6 * d, 5 * d, 0.5 * d, -0.5 * d]
    st, out = oracle.quantize(3, W)
    v = oracle.decode_block(3, out[:14])
    assert list(v[:8]) == [7 * d, d, 3 * d, 5 * d, -5 * d, 5 * d, d, -d]
    # FP4, scale 1 (amax = 6): midpoints 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5
    W = np.zeros((1, 32), np.float32)
    W[0, :8] = [6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    st, out = oracle.quantize(4, W)
    assert out[0] == 127
    v = oracle.decode_block(4, out[:17])
    assert list(v[:8]) == [6.0, 0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]


def test_quantize_errors():
    W = np.zeros((1, 32), np.float32)
    W[0, 3] = np.nan
    assert oracle.quantize(2, W)[0] == oracle.ERANGE
    W[0, 3] = np.inf
    assert oracle.quantize(4, W)[0] == oracle.ERANGE
    W[0, 3] = 3e5  # 3e5 / 3 overflows binary16
    assert oracle.quantize(2, W)[0] == oracle.ERANGE
    W[0, 3] = 1.0
    assert oracle.quantize(4, W, np.full(1, 3.0, np.float32))[0] == oracle.EINVAL  # not a power of two
    assert oracle.quantize(2, W, np.full(1, -1.0, np.float32))[0] == oracle.EINVAL
