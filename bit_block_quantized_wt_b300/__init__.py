"""Python binding of libfpx.so: block-quantized FP2/FP3/FP4 GEMVs and the low-bit MoE decode/verify
step on sm_103a.

Argument marshalling only: every step of the path runs in the CUDA library. Tensors are torch CUDA
tensors (device memory); the stream defaults to torch's current stream. There is no CPU fallback: if
libfpx.so is missing or no GPU is present, calls raise.

Names and semantics mirror include/fpx.h. The operations follow the ROCmFPX and decode-path
paragraphs of "DeepSeek V4 Flash hits 32 tok/s on AMD Ryzen AI MAX+ 395" and the section
"Lucebox's Optimization Trio" of "Token Freedom via APU: AMD Ryzen AI MAX+ 395 Runs DeepSeek V4 Flash
at 32 tok/s on a 284B Model".
"""
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfpx.so")

FPX_OK, FPX_EINVAL, FPX_EALIGN, FPX_ERANGE, FPX_ECUDA, FPX_ETIMEOUT, FPX_EDATA, FPX_ESPACE = range(8)
FPX_FP2, FPX_FP3, FPX_FP4 = 2, 3, 4
FPX_DTYPE_F32, FPX_DTYPE_BF16 = 0, 1


class FpxError(RuntimeError):
    def __init__(self, status, what):
        super().__init__(f"{what}: status {status} ({status_string(status)})")
        self.status = status


class moe_layer(ctypes.Structure):
    """Mirror of the C struct: H, I, E and device pointers (router, stacked routed gate/up/down,
    shared gate/up/down)."""
    _fields_ = [("H", ctypes.c_int), ("I", ctypes.c_int), ("E", ctypes.c_int),
                ("router", ctypes.c_void_p), ("gate", ctypes.c_void_p), ("up", ctypes.c_void_p),
                ("down", ctypes.c_void_p), ("sh_gate", ctypes.c_void_p), ("sh_up", ctypes.c_void_p),
                ("sh_down", ctypes.c_void_p)]


class moe_tiers(ctypes.Structure):
    """Mirror of the C struct: device slot_of [E], host (pinned) cold-tier gate/up/down arrays, the
    number of HBM slots, the staging slot range and the optional device cache of staged experts."""
    _fields_ = [("slot_of", ctypes.c_void_p), ("cold_gate", ctypes.c_void_p), ("cold_up", ctypes.c_void_p),
                ("cold_down", ctypes.c_void_p), ("n_slots", ctypes.c_int), ("stage_slot0", ctypes.c_int),
                ("n_stage", ctypes.c_int), ("cache", ctypes.c_void_p)]


_lib = None

_SIGS = {
    "fpx_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "fpx_block_bytes": (ctypes.c_size_t, [ctypes.c_int]),
    "fpx_matrix_bytes": (ctypes.c_int64, [ctypes.c_int, ctypes.c_int64, ctypes.c_int64]),
    "fpx_read_status": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "fpx_quantize": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                    ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "fpx_dequantize": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                      ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "fpx_tile_matrices": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                         ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
                                         ctypes.c_int, ctypes.c_void_p]),
    "fpx_gemv_q": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                  ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                  ctypes.c_void_p, ctypes.c_void_p]),
    "fpx_gemv_idot_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int64, ctypes.c_int]),
    "fpx_gemv_q_idot": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                       ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                       ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p]),
    "fpx_gemv_tiled_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int]),
    "fpx_gemv_q_tiled": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                        ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p]),
    "moe_route_topk": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                      ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                      ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "moe_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(moe_layer), ctypes.c_int, ctypes.c_int]),
    "moe_layer_decode": (ctypes.c_int, [ctypes.POINTER(moe_layer), ctypes.c_void_p, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                        ctypes.c_void_p]),
    "moe_layer_decode_static_ws": (ctypes.c_int, [ctypes.POINTER(moe_layer), ctypes.c_void_p, ctypes.c_int,
                                                  ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                  ctypes.c_void_p]),
    "moe_layer_decode_tiered": (ctypes.c_int, [ctypes.POINTER(moe_layer), ctypes.POINTER(moe_tiers), ctypes.c_void_p,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                               ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                               ctypes.c_void_p]),
    "moe_tiers_cache_reset": (ctypes.c_int, [ctypes.POINTER(moe_tiers), ctypes.c_void_p]),
    "moe_stack_verify": (ctypes.c_int, [ctypes.POINTER(moe_layer), ctypes.c_int, ctypes.c_void_p,
                                        ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                        ctypes.c_void_p, ctypes.c_void_p]),
    "moe_prefill_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(moe_layer), ctypes.c_int, ctypes.c_int]),
    "moe_layer_prefill": (ctypes.c_int, [ctypes.POINTER(moe_layer), ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                         ctypes.c_void_p]),
    "dspark_verify_commit": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                            ctypes.c_void_p, ctypes.c_void_p]),
    "fpx_quantize_weighted": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                             ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "fpx_debug_ring_wait": (ctypes.c_int, [ctypes.c_uint64, ctypes.c_int]),
}

# Every symbol include/fpx.h declares (the export test checks them against the header).
EXPORTS = tuple(_SIGS)


def lib():
    """Loads libfpx.so (building it first if only the sources are present). Raises if it cannot."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            from . import build as _build
            _build.build()
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype, f.argtypes = res, args
        _lib = L
    return _lib


def status_string(status):
    return lib().fpx_status_string(status).decode()


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def _check(st, what):
    if st != FPX_OK:
        raise FpxError(st, what)


def fpx_block_bytes(fmt):
    return lib().fpx_block_bytes(fmt)


def fpx_matrix_bytes(fmt, N, K):
    return lib().fpx_matrix_bytes(fmt, N, K)


def fpx_read_status(dev_status, stream=None):
    out = ctypes.c_int32(0)
    _check(lib().fpx_read_status(_ptr(dev_status), ctypes.addressof(out), _stream(stream)), "fpx_read_status")
    return out.value


def fpx_quantize(fmt, W, N, K, out, block_scales=None, dev_status=None, stream=None):
    _check(lib().fpx_quantize(fmt, _ptr(W), N, K, _ptr(block_scales), _ptr(out), _ptr(dev_status),
                              _stream(stream)), "fpx_quantize")


def fpx_tile_matrices(fmt, src, N, K, count, src_stride, dst, dst_stride, inverse=0, stream=None):
    _check(lib().fpx_tile_matrices(fmt, _ptr(src), N, K, count, src_stride, _ptr(dst), dst_stride, inverse,
                                   _stream(stream)), "fpx_tile_matrices")


def fpx_dequantize(fmt, Wq, N, K, W, dev_status=None, stream=None):
    _check(lib().fpx_dequantize(fmt, _ptr(Wq), N, K, _ptr(W), _ptr(dev_status), _stream(stream)),
           "fpx_dequantize")


def fpx_gemv_q(fmt, Wq, N, K, x, x_dtype, q, y, dev_status=None, stream=None):
    _check(lib().fpx_gemv_q(fmt, _ptr(Wq), N, K, _ptr(x), x_dtype, q, _ptr(y), _ptr(dev_status),
                            _stream(stream)), "fpx_gemv_q")


def fpx_gemv_idot_workspace_bytes(K, q):
    return lib().fpx_gemv_idot_workspace_bytes(K, q)


def fpx_gemv_q_idot(fmt, Wq, N, K, x, x_dtype, q, y, ws, ws_bytes, dev_status=None, stream=None):
    """Integer-dot variant of fpx_gemv_q (see include/fpx.h)."""
    _check(lib().fpx_gemv_q_idot(fmt, _ptr(Wq), N, K, _ptr(x), x_dtype, q, _ptr(y), _ptr(ws), ws_bytes,
                                 _ptr(dev_status), _stream(stream)), "fpx_gemv_q_idot")


def fpx_gemv_tiled_workspace_bytes(fmt, N, K, q):
    return lib().fpx_gemv_tiled_workspace_bytes(fmt, N, K, q)


def fpx_gemv_q_tiled(fmt, Wt, N, K, x, x_dtype, q, y, ws, ws_bytes, dev_status=None, stream=None):
    """fpx_gemv_q on a box-tiled matrix (see include/fpx.h)."""
    _check(lib().fpx_gemv_q_tiled(fmt, _ptr(Wt), N, K, _ptr(x), x_dtype, q, _ptr(y), _ptr(ws), ws_bytes,
                                  _ptr(dev_status), _stream(stream)), "fpx_gemv_q_tiled")


def moe_route_topk(R, E, H, x, q, k, logits, idx, w, uni, n_uni, stream=None):
    _check(lib().moe_route_topk(_ptr(R), E, H, _ptr(x), q, k, _ptr(logits), _ptr(idx), _ptr(w),
                                _ptr(uni), _ptr(n_uni), _stream(stream)), "moe_route_topk")


def moe_workspace_bytes(layer, q, k):
    return lib().moe_workspace_bytes(ctypes.byref(layer), q, k)


def moe_layer_decode(layer, x, q, k, y, ws, ws_bytes, idx_out=None, w_out=None, logits_out=None,
                     stream=None):
    _check(lib().moe_layer_decode(ctypes.byref(layer), _ptr(x), q, k, _ptr(y), _ptr(idx_out),
                                  _ptr(w_out), _ptr(logits_out), _ptr(ws), ws_bytes, _stream(stream)),
           "moe_layer_decode")


def moe_layer_decode_tiered(layer, tiers, x, q, k, y, ws, ws_bytes, idx_out=None, w_out=None, logits_out=None,
                            stream=None):
    """moe_layer_decode on a two-tier layer (see include/fpx.h)."""
    _check(lib().moe_layer_decode_tiered(ctypes.byref(layer), ctypes.byref(tiers), _ptr(x), q, k, _ptr(y),
                                         _ptr(idx_out), _ptr(w_out), _ptr(logits_out), _ptr(ws), ws_bytes,
                                         _stream(stream)), "moe_layer_decode_tiered")


def moe_tiers_cache_reset(tiers, stream=None):
    """Empties the two-tier staging cache tiers.cache (see include/fpx.h)."""
    _check(lib().moe_tiers_cache_reset(ctypes.byref(tiers), _stream(stream)), "moe_tiers_cache_reset")


def moe_layer_decode_static_ws(layer, x, q, k, y, idx_out=None, w_out=None, logits_out=None,
                               dev_status=None, stream=None):
    """moe_layer_decode without a caller workspace, for callers that cannot allocate device memory
    (see include/fpx.h). The first call on a device must come before any stream capture; calls that
    overlap on the GPU share one scratch array and race."""
    _check(lib().moe_layer_decode_static_ws(ctypes.byref(layer), _ptr(x), q, k, _ptr(y), _ptr(idx_out),
                                            _ptr(w_out), _ptr(logits_out), _ptr(dev_status), _stream(stream)),
           "moe_layer_decode_static_ws")


def moe_stack_verify(layers, r0, q, k, rL, ws, ws_bytes, idx_out=None, r_trace=None, events=None,
                     stream=None):
    """events: optional list of 5*len(layers)+1 raw cudaEvent_t handles (ints), recorded before each
    kernel and after the last one."""
    arr = (moe_layer * len(layers))(*layers)
    ev = None
    if events is not None:
        ev = (ctypes.c_void_p * len(events))(*events)
    _check(lib().moe_stack_verify(arr, len(layers), _ptr(r0), q, k, _ptr(rL), _ptr(idx_out),
                                  _ptr(r_trace), _ptr(ws), ws_bytes, ev, _stream(stream)), "moe_stack_verify")


def moe_prefill_workspace_bytes(layer, T, k):
    return lib().moe_prefill_workspace_bytes(ctypes.byref(layer), T, k)


def moe_layer_prefill(layer, x, T, k, y, ws, ws_bytes, idx_out=None, w_out=None, logits_out=None, perm_out=None,
                      offsets_out=None, stream=None):
    """Batched prefill of one layer over T tokens (see include/fpx.h)."""
    _check(lib().moe_layer_prefill(ctypes.byref(layer), _ptr(x), T, k, _ptr(y), _ptr(idx_out), _ptr(w_out),
                                   _ptr(logits_out), _ptr(perm_out), _ptr(offsets_out), _ptr(ws), ws_bytes,
                                   _stream(stream)),
           "moe_layer_prefill")


def dspark_verify_commit(logits, B, q, V, drafts, pred, n_accept, committed, dev_status=None, stream=None):
    """Speculative verify/commit for B sequences (see include/fpx.h)."""
    _check(lib().dspark_verify_commit(_ptr(logits), B, q, V, _ptr(drafts), _ptr(pred), _ptr(n_accept),
                                      _ptr(committed), _ptr(dev_status), _stream(stream)), "dspark_verify_commit")


def fpx_quantize_weighted(fmt, W, N, K, out, importance=None, dev_status=None, stream=None):
    """Importance-weighted quantizer (see include/fpx.h)."""
    _check(lib().fpx_quantize_weighted(fmt, _ptr(W), N, K, _ptr(importance), _ptr(out), _ptr(dev_status),
                                       _stream(stream)), "fpx_quantize_weighted")


def fpx_debug_ring_wait(wait_ns, drop_stage=-1):
    """Test hook for the layer kernels' bounded waits (see include/fpx.h): the wait limit in
    nanoseconds and a weight copy for CTA 0 of the gate/up kernel to withhold (-1: none)."""
    _check(lib().fpx_debug_ring_wait(wait_ns, drop_stage), "fpx_debug_ring_wait")
