"""CPU oracle for the low-bit MoE decode/verify path (binary64, naive loops).

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product path never does; it has no CPU fallback.

The C source (``oracle.c``) states the block layouts and the layer definition it follows. Every
function is pinned by ``tests/test_oracle_*.py``. Bit compatibility with Lucebox's own ROCmFPX files
is unpinned: the pages publish no layout.
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

EINVAL, ERANGE, EDATA = 1, 3, 6


def build(force=False):
    """Compiles liboracle.so next to its source (gcc, OpenMP)."""
    src = os.path.join(_HERE, "oracle.c")
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(src):
        return _LIB_PATH
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-Wall", "-fopenmp", "-fPIC", "-shared",
                           "-o", _LIB_PATH, src, "-lm"])
    return _LIB_PATH


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB_PATH)
        P, I, I64, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
        sig = {
            "orc_block_bytes": (I, [I]),
            "orc_matrix_bytes": (I64, [I, I64, I64]),
            "orc_threads": (I, []),
            "orc_set_threads": (I, [I]),
            "orc_decode_block": (I, [I, P, P]),
            "orc_dequantize": (I, [I, P, I64, I64, P]),
            "orc_gemv": (I, [I, P, I64, I64, P, I, P, P]),
            "orc_quantize": (I, [I, P, I64, I64, P, P]),
            "orc_topk": (I, [P, I, I, P]),
            "orc_route": (I, [P, I, I, P, I, I, P, P, P, P, P, P]),
            "orc_moe_layer": (I, [I, I, I, P, P, P, P, P, P, P, P, I, I, P, P, P, P, P, P]),
            "orc_rmsnorm_bf16": (I, [P, I, I, P]),
            "orc_stable_argsort": (I, [P, I, I, P, P]),
            "orc_dspark_commit": (I, [P, I, I, P, P, P, P]),
            "orc_quantize_weighted": (I, [I, P, I64, I64, P, P]),
            "orc_quantize_act16": (I, [P, I, I64, P, P, P]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype, f.argtypes = res, args
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(st, what):
    if st != 0:
        raise RuntimeError(f"oracle {what} failed with status {st}")


def block_bytes(fmt):
    return lib().orc_block_bytes(fmt)


def matrix_bytes(fmt, N, K):
    return lib().orc_matrix_bytes(fmt, N, K)


def threads():
    return lib().orc_threads()


def set_threads(n):
    """Sets the OpenMP thread count of later oracle calls; returns the previous count."""
    return lib().orc_set_threads(n)


def decode_block(fmt, blk):
    blk = np.ascontiguousarray(blk, dtype=np.uint8)
    out = np.zeros(32, np.float64)
    _check(lib().orc_decode_block(fmt, _p(blk), _p(out)), "decode_block")
    return out


def dequantize(fmt, Wq, N, K):
    Wq = np.ascontiguousarray(Wq, dtype=np.uint8)
    W = np.zeros((N, K), np.float64)
    _check(lib().orc_dequantize(fmt, _p(Wq), N, K, _p(W)), "dequantize")
    return W


def gemv(fmt, Wq, N, K, x):
    """x: [q][K] (any float dtype, converted exactly to binary64). Returns (y[q][N], M[q][N])."""
    Wq = np.ascontiguousarray(Wq, dtype=np.uint8)
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float64)
    q = x.shape[0]
    y = np.zeros((q, N), np.float64)
    M = np.zeros((q, N), np.float64)
    _check(lib().orc_gemv(fmt, _p(Wq), N, K, _p(x), q, _p(y), _p(M)), "gemv")
    return y, M


def quantize(fmt, W, scales=None):
    W = np.ascontiguousarray(W, dtype=np.float32)
    N, K = W.shape
    out = np.zeros(max(matrix_bytes(fmt, N, K), 1), np.uint8)
    sc = None if scales is None else np.ascontiguousarray(scales, dtype=np.float32)
    st = lib().orc_quantize(fmt, _p(W), N, K, _p(sc), _p(out))
    return st, out


def topk(v, k):
    v = np.ascontiguousarray(v, dtype=np.float64)
    idx = np.zeros(k, np.int32)
    _check(lib().orc_topk(_p(v), v.size, k, _p(idx)), "topk")
    return idx


def route(R, x, k):
    R = np.ascontiguousarray(R, dtype=np.float32)
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float64)
    E, H = R.shape
    q = x.shape[0]
    logits = np.zeros((q, E)); Ml = np.zeros((q, E))
    idx = np.zeros((q, k), np.int32); w = np.zeros((q, k))
    uni = np.zeros(q * k, np.int32); n = np.zeros(1, np.int32)
    _check(lib().orc_route(_p(R), E, H, _p(x), q, k, _p(logits), _p(Ml), _p(idx), _p(w), _p(uni), _p(n)), "route")
    return dict(logits=logits, Ml=Ml, idx=idx, w=w, uni=uni[: n[0]].copy())


def moe_layer(H, I, E, R, gate, up, down, sh_gate, sh_up, sh_down, x, k, idx_force=None):
    """gate/up/down: lists of E packed matrices (numpy uint8) or None. Returns a dict with y, M, idx,
    w, logits."""
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float64)
    q = x.shape[0]
    R = np.ascontiguousarray(R, dtype=np.float32)
    keep = []

    def ptrs(lst):
        arr = (ctypes.c_void_p * E)()
        for e in range(E):
            m = lst[e]
            if m is not None:
                m = np.ascontiguousarray(m, dtype=np.uint8)
                keep.append(m)
                arr[e] = m.ctypes.data
        keep.append(arr)
        return ctypes.cast(arr, ctypes.c_void_p)

    shs = [np.ascontiguousarray(a, dtype=np.uint8) for a in (sh_gate, sh_up, sh_down)]
    y = np.zeros((q, H)); M = np.zeros((q, H))
    idx = np.zeros((q, k), np.int32); w = np.zeros((q, k)); logits = np.zeros((q, E))
    f = None if idx_force is None else np.ascontiguousarray(idx_force, dtype=np.int32)
    st = lib().orc_moe_layer(H, I, E, _p(R), ptrs(gate), ptrs(up), ptrs(down), _p(shs[0]), _p(shs[1]),
                             _p(shs[2]), _p(x), q, k, _p(f), _p(y), _p(M), _p(idx), _p(w), _p(logits))
    _check(st, "moe_layer")
    return dict(y=y, M=M, idx=idx, w=w, logits=logits)


def rmsnorm_bf16(r):
    r = np.ascontiguousarray(np.atleast_2d(r), dtype=np.float32)
    q, H = r.shape
    u = np.zeros((q, H))
    _check(lib().orc_rmsnorm_bf16(_p(r), q, H, _p(u)), "rmsnorm_bf16")
    return u


def stable_argsort(keys, nkeys):
    keys = np.ascontiguousarray(keys, dtype=np.int32)
    perm = np.zeros(keys.size, np.int32)
    offsets = np.zeros(nkeys + 1, np.int32)
    _check(lib().orc_stable_argsort(_p(keys), keys.size, nkeys, _p(perm), _p(offsets)), "stable_argsort")
    return perm, offsets


def dspark_commit(logits, drafts):
    """logits float32 [q][V], drafts int [q-1] -> (pred [q], n_accept, committed [q], status)."""
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    q, V = logits.shape
    d = np.ascontiguousarray(drafts, dtype=np.int32).reshape(-1)
    pred = np.zeros(q, np.int32); n = np.zeros(1, np.int32); com = np.zeros(q, np.int32)
    st = lib().orc_dspark_commit(_p(logits), q, V, _p(d) if d.size else None, _p(pred), _p(n), _p(com))
    if st not in (0, ERANGE):
        _check(st, "dspark_commit")
    return pred, int(n[0]), com, st


def quantize_weighted(fmt, W, imp=None):
    """(status, packed bytes) of the importance-weighted quantizer; imp [K] or None (all ones)."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    N, K = W.shape
    out = np.zeros(max(matrix_bytes(fmt, N, K), 1), np.uint8)
    im = None if imp is None else np.ascontiguousarray(imp, dtype=np.float32)
    st = lib().orc_quantize_weighted(fmt, _p(W), N, K, _p(im), _p(out))
    return st, out


def quantize_act16(x):
    """Integer-dot activations of x [q][K] -> (status, X int32 [q][K], e int32 [q][K/32], xhat [q][K])."""
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float64)
    q, K = x.shape
    X = np.zeros((q, K), np.int32)
    e = np.zeros((q, max(K // 32, 1)), np.int32)
    xhat = np.zeros((q, K), np.float64)
    st = lib().orc_quantize_act16(_p(x), q, K, _p(X), _p(e), _p(xhat))
    return st, X, e[:, : K // 32], xhat


def gemv_idot(fmt, Wq, N, K, x):
    """The integer-dot GEMV: exactly W * xhat (the integer dot products are exact), as (y, M) of gemv."""
    st, _, _, xhat = quantize_act16(x)
    _check(st, "quantize_act16")
    return gemv(fmt, Wq, N, K, xhat)
