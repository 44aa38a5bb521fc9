"""The C ABI without a GPU: the library loads, exports every symbol include/fpx.h declares, and rejects
bad arguments before any CUDA call."""
import ctypes
import os
import re

import pytest

import bit_block_quantized_wt_b300 as fpx
from conftest import ROOT


def declared_functions():
    src = open(os.path.join(ROOT, "include", "fpx.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+char\s*\*|int64_t|size_t|int)\s+(\w+)\s*\(", src, flags=re.M)))


def test_library_exports_every_declared_symbol():
    names = declared_functions()
    assert len(names) >= 10
    L = fpx.lib()
    for n in names:
        assert hasattr(L, n), n
    assert sorted(fpx.EXPORTS) == names


def test_sizes_and_strings():
    assert [fpx.fpx_block_bytes(f) for f in (2, 3, 4, 5)] == [10, 14, 17, 0]
    assert fpx.fpx_matrix_bytes(2, 2048, 4096) == 2621440
    assert fpx.fpx_matrix_bytes(4, 3, 32) == 64
    assert fpx.fpx_matrix_bytes(3, 1, 33) == -1
    assert fpx.status_string(fpx.FPX_EDATA) == "invalid block or routing index"


FAKE = 1 << 20  # an aligned non-null address; these calls must fail before touching it


@pytest.mark.parametrize("args,expect", [
    ((5, FAKE, 8, 64, FAKE, 1, 1, FAKE), fpx.FPX_EINVAL),   # unknown format
    ((2, FAKE, 8, 60, FAKE, 1, 1, FAKE), fpx.FPX_EINVAL),   # K % 32 != 0
    ((2, FAKE, 8, 64, FAKE, 1, 0, FAKE), fpx.FPX_EINVAL),   # q = 0
    ((2, FAKE, 8, 64, FAKE, 1, 5, FAKE), fpx.FPX_EINVAL),   # q = 5
    ((2, FAKE, 8, 64, FAKE, 7, 1, FAKE), fpx.FPX_EINVAL),   # dtype
    ((2, None, 8, 64, FAKE, 1, 1, FAKE), fpx.FPX_EINVAL),   # null weights
    ((2, FAKE + 8, 8, 64, FAKE, 1, 1, FAKE), fpx.FPX_EALIGN),  # weights not 16-byte aligned
    ((2, FAKE, 8, 64, FAKE + 2, 1, 1, FAKE), fpx.FPX_EALIGN),  # x not 4-byte aligned
    ((2, FAKE, 8, 64, FAKE + 4, 1, 1, FAKE), fpx.FPX_EALIGN),  # x not 16-byte aligned (read in 16-byte units)
])
def test_gemv_argument_errors(args, expect):
    fmt, W, N, K, x, dt, q, y = args
    assert fpx.lib().fpx_gemv_q(fmt, W, N, K, x, dt, q, y, None, None) == expect


def _layer(**kw):
    d = dict(H=512, I=512, E=16, router=FAKE, gate=FAKE, up=FAKE, down=FAKE, sh_gate=FAKE, sh_up=FAKE,
             sh_down=FAKE)
    d.update(kw)
    return fpx.moe_layer(**d)


def test_layer_argument_errors():
    L = fpx.lib()
    ws = fpx.moe_workspace_bytes(_layer(), 4, 4)
    assert ws > 0 and ws % 16 == 0
    good = _layer()
    call = lambda lay, q=4, k=4, wsb=ws, wsp=FAKE: L.moe_layer_decode(ctypes.byref(lay), FAKE, q, k, FAKE, None, None,
                                                                     None, wsp, wsb, None)
    assert call(_layer(H=500)) == fpx.FPX_EINVAL
    assert call(_layer(I=100)) == fpx.FPX_EINVAL
    assert call(_layer(H=5120)) == fpx.FPX_EINVAL  # above the 4608 limit (and its tables too large)
    assert call(_layer(I=5632)) == fpx.FPX_EINVAL  # above the 4608 limit, although its tables would fit
    assert call(_layer(E=0)) == fpx.FPX_EINVAL
    assert call(_layer(down=None)) == fpx.FPX_EINVAL
    assert call(_layer(gate=FAKE + 4)) == fpx.FPX_EALIGN
    assert call(good, q=5) == fpx.FPX_EINVAL
    assert call(good, k=9) == fpx.FPX_EINVAL
    assert call(good, k=17) == fpx.FPX_EINVAL
    assert call(good, wsb=ws - 16) == fpx.FPX_ESPACE
    assert call(good, wsp=FAKE + 8) == fpx.FPX_EALIGN
    # the router reads x in 8-byte units
    assert L.moe_layer_decode(ctypes.byref(good), FAKE + 4, 4, 4, FAKE, None, None, None, FAKE, ws, None) == fpx.FPX_EALIGN
    arr = (fpx.moe_layer * 2)(good, _layer(I=1024))
    assert L.moe_stack_verify(arr, 2, FAKE, 4, 4, FAKE, None, None, FAKE, ws, None, None) == fpx.FPX_EINVAL
    assert L.moe_stack_verify(arr, 0, FAKE, 4, 4, FAKE, None, None, FAKE, ws, None, None) == fpx.FPX_EINVAL


def test_tiers_cache_argument_errors():
    L = fpx.lib()
    t = fpx.moe_tiers(slot_of=FAKE, cold_gate=FAKE, cold_up=FAKE, cold_down=FAKE, n_slots=32, stage_slot0=16,
                      n_stage=16, cache=None)
    assert L.moe_tiers_cache_reset(None, None) == fpx.FPX_EINVAL
    assert L.moe_tiers_cache_reset(ctypes.byref(t), None) == fpx.FPX_EINVAL  # no cache
    t.cache = FAKE
    t.n_stage = 0
    assert L.moe_tiers_cache_reset(ctypes.byref(t), None) == fpx.FPX_EINVAL
    t.n_stage = 1025  # a cache tracks at most 1024 staging slots
    assert L.moe_tiers_cache_reset(ctypes.byref(t), None) == fpx.FPX_EINVAL
    t.n_stage, t.cache = 16, FAKE + 2
    assert L.moe_tiers_cache_reset(ctypes.byref(t), None) == fpx.FPX_EALIGN
    lay = _layer()
    ws = fpx.moe_workspace_bytes(lay, 4, 4)
    call = lambda tt: L.moe_layer_decode_tiered(ctypes.byref(lay), ctypes.byref(tt), FAKE, 4, 4, FAKE, None, None,
                                                None, FAKE, ws, None)
    t.cache, t.n_slots, t.n_stage = FAKE, 1041, 1025
    assert call(t) == fpx.FPX_EINVAL  # too many staging slots for the cache
    t.n_slots, t.n_stage, t.cache = 32, 16, FAKE + 2
    assert call(t) == fpx.FPX_EALIGN


def test_tiled_gemv_argument_errors():
    L = fpx.lib()
    assert fpx.fpx_gemv_tiled_workspace_bytes(2, 256, 4096, 4) == 16 * 4 * 256 * 4  # 16 pieces of one stage
    assert fpx.fpx_gemv_tiled_workspace_bytes(2, 151552, 4096, 4) == 16            # 592 tiles: one piece
    assert fpx.fpx_gemv_tiled_workspace_bytes(2, 255, 4096, 4) == 0
    bf = fpx.FPX_DTYPE_BF16
    call = lambda fmt=2, W=FAKE, N=256, K=512, x=FAKE, q=4, ws=FAKE, wb=1 << 20: L.fpx_gemv_q_tiled(
        fmt, W, N, K, x, bf, q, FAKE, ws, wb, None, None)
    assert call(fmt=5) == fpx.FPX_EINVAL
    assert call(N=255) == fpx.FPX_EINVAL    # not whole row tiles
    assert call(fmt=4, N=96) == fpx.FPX_EINVAL
    assert call(K=384) == fpx.FPX_EINVAL    # not whole stages
    assert call(fmt=4, K=768) == fpx.FPX_EINVAL
    assert call(q=5) == fpx.FPX_EINVAL
    assert call(ws=None) == fpx.FPX_EINVAL
    assert call(W=FAKE + 8) == fpx.FPX_EALIGN
    assert call(x=FAKE + 8) == fpx.FPX_EALIGN
    assert call(wb=15) == fpx.FPX_ESPACE


def test_wait_hook_argument_errors():
    L = fpx.lib()
    assert L.fpx_debug_ring_wait(0, -1) == fpx.FPX_EINVAL             # no limit
    assert L.fpx_debug_ring_wait(500_000_001, -1) == fpx.FPX_EINVAL   # above the default 0.5 s
    assert L.fpx_debug_ring_wait(2_000_000, -2) == fpx.FPX_EINVAL     # stage index below -1


def test_route_and_quant_argument_errors():
    L = fpx.lib()
    assert L.moe_route_topk(FAKE, 8, 64, FAKE, 4, 9, FAKE, FAKE, FAKE, FAKE, FAKE, None) == fpx.FPX_EINVAL
    assert L.moe_route_topk(FAKE, 8, 64, FAKE, 4, 2, None, FAKE, FAKE, FAKE, FAKE, None) == fpx.FPX_EINVAL
    assert L.moe_route_topk(FAKE, 2000, 64, FAKE, 4, 2, FAKE, FAKE, FAKE, FAKE, FAKE, None) == fpx.FPX_EINVAL
    assert L.moe_route_topk(FAKE, 8, 64, FAKE + 4, 4, 2, FAKE, FAKE, FAKE, FAKE, FAKE, None) == fpx.FPX_EALIGN
    # x and two router rows staged in shared memory: (2 q + 8) H = 256 KB does not fit
    assert L.moe_route_topk(FAKE, 8, 16384, FAKE, 4, 2, FAKE, FAKE, FAKE, FAKE, FAKE, None) == fpx.FPX_EINVAL
    assert L.fpx_quantize(2, FAKE, 4, 48, None, FAKE, None, None) == fpx.FPX_EINVAL
    assert L.fpx_quantize(2, FAKE, 4, 64, None, FAKE + 1, None, None) == fpx.FPX_EALIGN
    assert L.fpx_dequantize(9, FAKE, 4, 64, FAKE, None, None) == fpx.FPX_EINVAL
    assert L.fpx_read_status(None, None, None) == fpx.FPX_EINVAL


def test_prefill_and_commit_argument_errors():
    L = fpx.lib()
    lay = _layer()
    assert fpx.moe_prefill_workspace_bytes(lay, 0, 4) == 0
    assert fpx.moe_prefill_workspace_bytes(lay, 16, 9) == 0
    ws = fpx.moe_prefill_workspace_bytes(lay, 16, 4)
    assert ws > 0 and ws % 16 == 0
    call = lambda lay, T=16, k=4, x=FAKE, wsb=ws: L.moe_layer_prefill(ctypes.byref(lay), x, T, k, FAKE, None, None, None,
                                                                      None, None, FAKE, wsb, None)
    assert call(lay, T=0) == fpx.FPX_EINVAL
    assert call(lay, k=9) == fpx.FPX_EINVAL
    assert call(_layer(H=500)) == fpx.FPX_EINVAL
    assert call(lay, x=FAKE + 2) == fpx.FPX_EALIGN
    assert call(lay, wsb=ws - 16) == fpx.FPX_ESPACE
    c = L.dspark_verify_commit
    assert c(FAKE, 4, 0, 10, FAKE, FAKE, FAKE, FAKE, None, None) == fpx.FPX_EINVAL   # q = 0
    assert c(FAKE, 4, 17, 10, FAKE, FAKE, FAKE, FAKE, None, None) == fpx.FPX_EINVAL  # q > 16
    assert c(FAKE, 4, 4, 0, FAKE, FAKE, FAKE, FAKE, None, None) == fpx.FPX_EINVAL    # V = 0
    assert c(FAKE, 4, 4, 10, None, FAKE, FAKE, FAKE, None, None) == fpx.FPX_EINVAL   # drafts needed
    assert c(FAKE + 2, 4, 4, 10, FAKE, FAKE, FAKE, FAKE, None, None) == fpx.FPX_EALIGN
    assert c(None, 0, 4, 10, None, None, None, None, None, None) == fpx.FPX_OK       # B = 0: nothing


def test_idot_argument_errors():
    L = fpx.lib()
    assert fpx.fpx_gemv_idot_workspace_bytes(4096, 4) == 128 * 4 * 68 + 16
    assert fpx.fpx_gemv_idot_workspace_bytes(1280, 1) == 64 * 68 + 16  # 40 blocks padded to 64
    assert fpx.fpx_gemv_idot_workspace_bytes(4096, 5) == 0
    assert fpx.fpx_gemv_idot_workspace_bytes(100, 1) == 0
    ws = fpx.fpx_gemv_idot_workspace_bytes(1024, 2)
    c = lambda fmt=2, W=FAKE, N=8, K=1024, x=FAKE, dt=1, q=2, wsp=FAKE, wsb=ws: L.fpx_gemv_q_idot(
        fmt, W, N, K, x, dt, q, FAKE, wsp, wsb, None, None)
    assert c(K=992) == fpx.FPX_EINVAL            # rows not whole 16-byte units (K % 256)
    assert c(fmt=4, K=768) == fpx.FPX_EINVAL     # FP4 needs K % 512
    assert c(q=5) == fpx.FPX_EINVAL
    assert c(dt=7) == fpx.FPX_EINVAL
    assert c(wsp=None) == fpx.FPX_EINVAL
    assert c(wsb=ws - 16) == fpx.FPX_ESPACE
    assert c(wsp=FAKE + 8) == fpx.FPX_EALIGN
    assert c(W=FAKE + 8) == fpx.FPX_EALIGN
    assert c(N=0) == fpx.FPX_OK                  # nothing to do


def test_tiered_argument_errors():
    L = fpx.lib()
    lay = _layer()
    ws = fpx.moe_workspace_bytes(lay, 4, 4)
    t = lambda **kw: fpx.moe_tiers(**dict(dict(slot_of=FAKE, cold_gate=FAKE, cold_up=FAKE, cold_down=FAKE,
                                                   n_slots=24, stage_slot0=8, n_stage=16), **kw))
    call = lambda tiers, q=4, k=4, wsb=ws: L.moe_layer_decode_tiered(ctypes.byref(lay), ctypes.byref(tiers), FAKE, q, k,
                                                                      FAKE, None, None, None, FAKE, wsb, None)
    assert L.moe_layer_decode_tiered(ctypes.byref(lay), None, FAKE, 4, 4, FAKE, None, None, None, FAKE, ws,
                                     None) == fpx.FPX_EINVAL
    assert call(t(slot_of=None)) == fpx.FPX_EINVAL
    assert call(t(cold_up=None)) == fpx.FPX_EINVAL
    assert call(t(n_stage=15)) == fpx.FPX_EINVAL       # fewer staging slots than the largest union (16)
    assert call(t(stage_slot0=9)) == fpx.FPX_EINVAL    # staging range past the slots
    assert call(t(stage_slot0=-1)) == fpx.FPX_EINVAL
    assert call(t(), q=5) == fpx.FPX_EINVAL
    assert call(t(slot_of=FAKE + 2)) == fpx.FPX_EALIGN
    assert call(t(), wsb=ws - 16) == fpx.FPX_ESPACE


def test_bench_traffic_needs_matching_sources(tmp_path, monkeypatch):
    """bench.py reports a recorded DRAM count only while the layer sources match the capture's digest."""
    import json
    import bench
    alg = 1_000_000
    got = bench.recorded_traffic("k_gate_up", alg)
    rec = json.load(open(os.path.join(bench.ROOT, "profiles", "traffic.json")))
    if rec["csrc"] == bench.csrc_digest():
        assert got == round(rec["kernels"]["k_gate_up"]["dram_per_algorithmic_byte"] * alg)
    else:
        assert got is None
    monkeypatch.setattr(bench, "csrc_digest", lambda: "0" * 16)  # sources changed since the capture
    assert bench.recorded_traffic("k_gate_up", alg) is None
    assert bench.recorded_traffic("no_such_kernel", alg) is None
