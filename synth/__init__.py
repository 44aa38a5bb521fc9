"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

Holds no decode, GEMV, routing or quantization arithmetic: it only draws packed blocks with uniform
codes and uniform binary16 scales, normal router weights and normal tokens, from the counter-based
generator described in ``synth.h``. The host library (``libsynth.so``) and its device twin
(``libsynth_dev.so``) produce identical packed bytes.
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_HOST = os.path.join(_HERE, "libsynth.so")
_DEV = os.path.join(_HERE, "libsynth_dev.so")

# tensor ids
GATE, UP, DOWN, SH_GATE, SH_UP, SH_DOWN, ROUTER, TOKENS, DENSE_W, DENSE_X = range(1, 11)
BLOCK_BYTES = {2: 10, 3: 14, 4: 17}


def _stale(out, src):
    return not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src)


def build(force=False, device=True):
    src = os.path.join(_HERE, "synth.c")
    if force or _stale(_HOST, src):
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                               "-o", _HOST, src, "-lm"])
    dsrc = os.path.join(_HERE, "synth_dev.cu")
    if device and (force or _stale(_DEV, dsrc)):
        subprocess.check_call(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo",
                               "-Xcompiler", "-fPIC", "-shared", "-o", _DEV, dsrc])


_h = None
_d = None


def host():
    global _h
    if _h is None:
        build(device=False)
        L = ctypes.CDLL(_HOST)
        U64, I, I64, P, D = ctypes.c_uint64, ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_double
        for name, res, args in [
            ("synth_mix", U64, [U64]), ("synth_key", U64, [U64, U64, U64, U64]),
            ("synth_rand", U64, [U64, U64]), ("synth_uniform", D, [U64, U64]),
            ("synth_normal", D, [U64, U64]), ("synth_blocks", I, [I, U64, I64, I64, P]),
            ("synth_matrix", I64, [I, U64, I64, I64, P]),
            ("synth_normal_f32", None, [U64, I64, I64, D, P]),
            ("synth_normal_bf16", None, [U64, I64, I64, P]),
        ]:
            f = getattr(L, name)
            f.restype, f.argtypes = res, args
        _h = L
    return _h


def device():
    global _d
    if _d is None:
        build()
        L = ctypes.CDLL(_DEV)
        U64, I, I64, P = ctypes.c_uint64, ctypes.c_int, ctypes.c_int64, ctypes.c_void_p
        L.synth_dev_matrices.restype = I
        L.synth_dev_matrices.argtypes = [I, U64, U64, U64, U64, I, I64, I64, P, I64, P]
        L.synth_dev_key.restype = U64
        L.synth_dev_key.argtypes = [U64, U64, U64, U64]
        _d = L
    return _d


def key(seed, layer, tensor, expert=0):
    return host().synth_key(seed, layer, tensor, expert)


def matrix_bytes(fmt, N, K):
    return (N * (K // 32) * BLOCK_BYTES[fmt] + 15) // 16 * 16


def matrix(fmt, N, K, seed=0, layer=0, tensor=DENSE_W, expert=0):
    """Packed N x K matrix (uint8, padded storage size)."""
    out = np.zeros(max(matrix_bytes(fmt, N, K), 16), np.uint8)
    n = host().synth_matrix(fmt, key(seed, layer, tensor, expert), N, K, out.ctypes.data)
    assert n >= 0
    return out[: matrix_bytes(fmt, N, K)]


def normal_f32(n, scale=1.0, seed=0, layer=0, tensor=DENSE_X, expert=0):
    out = np.zeros(n, np.float32)
    host().synth_normal_f32(key(seed, layer, tensor, expert), 0, n, scale, out.ctypes.data)
    return out


def normal_bf16_bits(n, seed=0, layer=0, tensor=TOKENS, expert=0):
    out = np.zeros(n, np.uint16)
    host().synth_normal_bf16(key(seed, layer, tensor, expert), 0, n, out.ctypes.data)
    return out


def bf16_bits_to_f32(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32)


def router(E, H, seed=0, layer=0):
    return normal_f32(E * H, 0.02, seed, layer, ROUTER).reshape(E, H)


def tokens_bf16(q, H, seed=0, layer=0):
    """(bits uint16 [q][H], values float32 [q][H])"""
    bits = normal_bf16_bits(q * H, seed, layer, TOKENS).reshape(q, H)
    return bits, bf16_bits_to_f32(bits).reshape(q, H)


def device_matrices(fmt, seed, layer, tensor, expert0, count, N, K, ptr, stride, stream=0):
    """Fills `count` packed matrices on the device at integer address `ptr`."""
    st = device().synth_dev_matrices(fmt, seed, layer, tensor, expert0, count, N, K, ptr, stride, stream)
    if st != 0:
        raise RuntimeError(f"synth_dev_matrices failed: {st}")
