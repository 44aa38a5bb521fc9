#!/usr/bin/env python3
"""q=4 MoE verify throughput on the 43-layer synthetic stack; prints one JSON line.

A step is one q = 4 verify pass (top-4 routing) through 43 MoE layers of hidden 4096, 256 routed
experts (FP2 gate/up [2048 x 4096], FP3 down [4096 x 2048]) and an FP4 shared expert, all resident in
HBM (about 99 GB), on a batch of 4 synthetic tokens. The metric is packed-weight GB/s: the packed bytes
of every expert matrix the step touches (|union| * 8,912,896 + 13,369,344 per layer) divided by time.

--impl fpx (default) times the CUDA library; --impl reference times the CPU oracle on bounded samples
of the same workload. Under torchrun every rank runs an independent replica (no collective on the
data path); value is the whole job's bytes over the slowest rank's time.
"""
import argparse
import ctypes
import hashlib
import json
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

H, I, E, Q, K_TOP, LAYERS = 4096, 2048, 256, 4, 4, 43
METRIC = "q=4 MoE verify: packed-weight GB/s (frac of B300 HBM peak), layer-steps/s"
WORKLOAD = ("43-layer synthetic MoE stack, each layer hidden 4096, 256 routed experts (FP2 gate/up "
            "2048x4096, FP3 down 4096x2048), FP4 shared expert, fp32 router; q=4 verify pass, top-4")
N_BATCHES = 8


NK = 5  # kernels per layer: router, gate/up, h + down tables, down, combine

def layer_bytes(n_union):
    import bit_block_quantized_wt_b300 as fpx
    gu = fpx.fpx_matrix_bytes(2, I, H)
    d = fpx.fpx_matrix_bytes(3, H, I)
    s = fpx.fpx_matrix_bytes(4, I, H)
    return n_union * (2 * gu + d) + 3 * s


def gate_up_bytes(n_union):
    import bit_block_quantized_wt_b300 as fpx
    return n_union * 2 * fpx.fpx_matrix_bytes(2, I, H) + 2 * fpx.fpx_matrix_bytes(4, I, H)


def down_bytes(n_union):
    import bit_block_quantized_wt_b300 as fpx
    return n_union * fpx.fpx_matrix_bytes(3, H, I) + fpx.fpx_matrix_bytes(4, H, I)


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6400.0, "fallback"


def bf16_peak():
    """Measured dense bf16 tensor throughput (TFLOP/s) of the B300s: burst (a kernel timed on
    its own), or the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1800.0, "fallback"


PF_T, PF_K = 2048, 6  # the prefill workload: one layer, 2048 tokens, top-6


def prefill_measure(fpx, layer, warmup, reps=10):
    """moe_layer_prefill of one stack layer on 2048 synthetic tokens (bfloat16 N(0,1), seeded), timed
    with CUDA events over `reps` calls after `warmup` calls; FLOPs are the dense contraction's
    2 * (2 I H (T k + T) + H I (T k + T))."""
    import torch
    g = torch.Generator(device="cuda").manual_seed(5)
    x = torch.randn(PF_T, H, device="cuda", generator=g).to(torch.bfloat16)
    wsb = fpx.moe_prefill_workspace_bytes(layer, PF_T, PF_K)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    y = torch.empty(PF_T, H, device="cuda")
    for _ in range(warmup):
        fpx.moe_layer_prefill(layer, x, PF_T, PF_K, y, ws, wsb)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(reps):
        fpx.moe_layer_prefill(layer, x, PF_T, PF_K, y, ws, wsb)
    e1.record()
    e1.synchronize()
    ms = e0.elapsed_time(e1) / reps
    P = PF_T * PF_K
    flops = 2 * (2 * I * H * (P + PF_T) + H * I * (P + PF_T))
    peak, kind = bf16_peak()
    tf = flops / (ms / 1e3) / 1e12
    return {"workload": f"prefill of one layer (config above): {PF_T} tokens, top-{PF_K}, bfloat16 N(0,1) "
                        "synthetic tokens", "ms_per_layer": round(ms, 4), "tflops": round(tf, 1),
            "gflop_per_layer": round(flops / 1e9, 1), "peak_tflops": peak, "peak_kind": f"{kind} bf16 dense (burst)",
            "frac": round(tf / peak, 4), "tokens_per_s": round(PF_T / (ms / 1e3), 1), "reps": reps}


DS_B, DS_Q, DS_V = 128, 4, 131072  # verify/commit: sequences, positions, stand-in vocabulary size


def commit_measure(fpx, peak, reps=20):
    """dspark_verify_commit over 128 sequences x 4 positions x 131,072 binary32 logits (256 MB, larger
    than L2; synthetic N(0,1), drafts that match the target's choice half of the time), timed with
    CUDA events; HBM-bound: bytes are the logits read once."""
    import torch
    g = torch.Generator(device="cuda").manual_seed(7)
    lg = torch.randn(DS_B, DS_Q, DS_V, device="cuda", generator=g)
    best = lg.argmax(dim=2).to(torch.int32)
    flip = torch.rand(DS_B, DS_Q - 1, device="cuda", generator=g) < 0.5
    drafts = torch.where(flip, (best[:, : DS_Q - 1] + 1) % DS_V, best[:, : DS_Q - 1]).to(torch.int32).contiguous()
    pred = torch.empty(DS_B, DS_Q, dtype=torch.int32, device="cuda")
    n = torch.empty(DS_B, dtype=torch.int32, device="cuda")
    com = torch.empty(DS_B, DS_Q, dtype=torch.int32, device="cuda")
    for _ in range(3):
        fpx.dspark_verify_commit(lg, DS_B, DS_Q, DS_V, drafts, pred, n, com)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(reps):
        fpx.dspark_verify_commit(lg, DS_B, DS_Q, DS_V, drafts, pred, n, com)
    e1.record()
    e1.synchronize()
    ms = e0.elapsed_time(e1) / reps
    gbs = DS_B * DS_Q * DS_V * 4 / (ms / 1e3) / 1e9
    return {"workload": f"{DS_B} sequences x {DS_Q} verified positions x {DS_V} binary32 logits (synthetic)",
            "ms": round(ms, 4), "value": round(gbs, 1), "unit": "GB/s", "frac_of_hbm_peak": round(gbs / peak, 4),
            "mean_accepted": round(float(n.float().mean()), 3), "reps": reps}


def quantize_weighted_measure(fpx, reps=5):
    """fpx_quantize_weighted on one FP2 gate matrix shape (2048 x 4096 binary32 weights, N(0, 0.02)),
    importance U[0, 3) per column, CUDA events. Binary64-bound: 16 candidates x 32 weights x 5 binary64
    operations per block."""
    import torch
    g = torch.Generator(device="cuda").manual_seed(9)
    W = torch.randn(I, H, device="cuda", generator=g) * 0.02
    imp = torch.rand(H, device="cuda", generator=g) * 3
    out = torch.empty(fpx.fpx_matrix_bytes(2, I, H), dtype=torch.uint8, device="cuda")
    fpx.fpx_quantize_weighted(2, W, I, H, out, importance=imp)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(reps):
        fpx.fpx_quantize_weighted(2, W, I, H, out, importance=imp)
    e1.record()
    e1.synchronize()
    ms = e0.elapsed_time(e1) / reps
    blocks = I * H // 32
    return {"workload": f"FP2 {I}x{H} weights, per-column importance", "ms": round(ms, 4),
            "blocks_per_s": round(blocks / (ms / 1e3)), "fp64_ops_per_s": round(blocks * 16 * 32 * 5 / (ms / 1e3) / 1e12, 3),
            "fp64_unit": "Tops/s", "reps": reps}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def over_ranks(secs, nbytes, world, device="cuda"):
    """The whole job's time and work: the slowest rank's seconds and the sum of the bytes all ranks
    streamed (every rank streams its own replica). Collective on the default process group."""
    if world <= 1:
        return secs, float(nbytes)
    import torch
    t = torch.tensor([secs, float(nbytes)], dtype=torch.float64, device=device)
    tmax = t.clone()
    torch.distributed.all_reduce(tmax, op=torch.distributed.ReduceOp.MAX)
    tsum = t.clone()
    torch.distributed.all_reduce(tsum, op=torch.distributed.ReduceOp.SUM)
    return float(tmax[0]), float(tsum[1])


# ---------------------------------------------------------------------------- clocks (NVML)

class ClockSampler:
    """Samples SM clock and clock-event reasons through NVML (libnvidia-ml.so.1 via ctypes) every
    20 ms while running. Reading clocks changes nothing on the GPU."""
    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
               0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}
    NVML_CLOCK_SM = 1

    def __init__(self, cuda_index):
        self.samples, self.reasons, self.ok, self.err, self.max = [], 0, False, None, None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise RuntimeError("nvmlInit_v2 failed")
            h = ctypes.c_void_p()
            rc = -1
            try:
                import torch
                p = torch.cuda.get_device_properties(cuda_index)
                bus = f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0".encode()
                rc = nv.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(h))
            except Exception:  # noqa: BLE001 - fall back to the index
                rc = -1
            if rc != 0 and nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(cuda_index), ctypes.byref(h)) != 0:
                raise RuntimeError("no NVML handle")
            mx = ctypes.c_uint()
            nv.nvmlDeviceGetMaxClockInfo(h, self.NVML_CLOCK_SM, ctypes.byref(mx))
            self.nv, self.h, self.max, self.ok = nv, h, int(mx.value), True
            self.reason_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
        except Exception as e:  # noqa: BLE001 - reported in the JSON line
            self.err = f"{type(e).__name__}: {e}"[:200]
        self._stop = threading.Event()

    def _run(self):
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            if self.nv.nvmlDeviceGetClockInfo(self.h, self.NVML_CLOCK_SM, ctypes.byref(clk)) == 0:
                self.samples.append(int(clk.value))
            if self.reason_fn(self.h, ctypes.byref(rs)) == 0:
                self.reasons |= int(rs.value)
            time.sleep(0.02)

    def __enter__(self):
        if self.ok:
            self.t = threading.Thread(target=self._run, daemon=True)
            self.t.start()
        return self

    def __exit__(self, *a):
        if self.ok:
            self._stop.set()
            self.t.join()

    def summary(self):
        if not self.ok or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max, "reasons": [f"nvml unavailable ({self.err})"]}
        names = [n for b, n in self.REASONS.items() if self.reasons & b and n != "gpu_idle"]
        return {"sm_mhz": float(statistics.median(self.samples)), "sm_max_mhz": self.max, "reasons": names,
                "samples": len(self.samples)}


# ---------------------------------------------------------------------------- device stack

class Stack:
    def __init__(self, n_layers, seed=0):
        import torch
        import bit_block_quantized_wt_b300 as fpx
        import synth
        self.fpx, self.torch = fpx, torch
        mb_gu, mb_d, mb_s = fpx.fpx_matrix_bytes(2, I, H), fpx.fpx_matrix_bytes(3, H, I), fpx.fpx_matrix_bytes(4, I, H)
        s = torch.cuda.current_stream().cuda_stream
        self.bufs, self.layers = [], []
        # the kernels read box-tiled expert matrices: generate row-major into scratch, then tile
        tmp = torch.empty(E * max(mb_gu, mb_d), dtype=torch.uint8, device="cuda")
        for l in range(n_layers):
            g = torch.empty(E * mb_gu, dtype=torch.uint8, device="cuda")
            u = torch.empty(E * mb_gu, dtype=torch.uint8, device="cuda")
            d = torch.empty(E * mb_d, dtype=torch.uint8, device="cuda")
            sh = [torch.empty(mb_s, dtype=torch.uint8, device="cuda") for _ in range(3)]
            for dst, fmt, tensor, count, n, kk, mb in ((g, 2, synth.GATE, E, I, H, mb_gu), (u, 2, synth.UP, E, I, H, mb_gu),
                                                       (d, 3, synth.DOWN, E, H, I, mb_d),
                                                       (sh[0], 4, synth.SH_GATE, 1, I, H, mb_s),
                                                       (sh[1], 4, synth.SH_UP, 1, I, H, mb_s),
                                                       (sh[2], 4, synth.SH_DOWN, 1, H, I, mb_s)):
                synth.device_matrices(fmt, seed, l, tensor, 0, count, n, kk, tmp.data_ptr(), mb, s)
                fpx.fpx_tile_matrices(fmt, tmp, n, kk, count, mb, dst, mb, 0, s)
            R = torch.from_numpy(synth.router(E, H, seed, l)).cuda()
            self.bufs.append((g, u, d, sh, R))
            self.layers.append(fpx.moe_layer(H=H, I=I, E=E, router=R.data_ptr(), gate=g.data_ptr(), up=u.data_ptr(),
                                             down=d.data_ptr(), sh_gate=sh[0].data_ptr(), sh_up=sh[1].data_ptr(),
                                             sh_down=sh[2].data_ptr()))
        del tmp
        torch.cuda.synchronize()


def tokens_fp32(b, q):
    import synth
    return synth.tokens_bf16(q, H, seed=1000 + b)[1].astype(np.float32)


class Runner:
    """Holds the buffers of one verify-pass configuration and a captured CUDA graph of one pass."""

    def __init__(self, stack, q, k, graph=True):
        import torch
        fpx = stack.fpx
        self.stack, self.q, self.k, self.torch, self.fpx = stack, q, k, torch, fpx
        L = len(stack.layers)
        self.ws_b = fpx.moe_workspace_bytes(stack.layers[0], q, k)
        self.ws = torch.empty(self.ws_b, dtype=torch.uint8, device="cuda")
        self.rin = torch.empty(q, H, device="cuda")
        self.rL = torch.empty(q, H, device="cuda")
        self.idx = torch.empty(L, q, k, dtype=torch.int32, device="cuda")
        self.batches = torch.stack([torch.from_numpy(tokens_fp32(b, q)) for b in range(N_BATCHES)]).cuda()
        self.stream = torch.cuda.Stream()
        self.stream.wait_stream(torch.cuda.current_stream())
        self.graph = None
        if graph:
            with torch.cuda.stream(self.stream):
                self.rin.copy_(self.batches[0])
                self.call()  # warm the launch path (attributes) before capture
            self.stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=self.stream):
                self.call()
            self.graph = g
        torch.cuda.synchronize()

    def call(self, events=None):
        self.fpx.moe_stack_verify(self.stack.layers, self.rin, self.q, self.k, self.rL, self.ws, self.ws_b,
                                  idx_out=self.idx, events=events)

    def step(self, b):
        self.rin.copy_(self.batches[b % N_BATCHES], non_blocking=True)
        if self.graph is not None:
            self.graph.replay()
        else:
            self.call()

    def union_sizes(self):
        """Per batch, the number of distinct experts per layer (from the routing of a real pass)."""
        torch = self.torch
        out = []
        with torch.cuda.stream(self.stream):
            for b in range(N_BATCHES):
                self.rin.copy_(self.batches[b])
                self.call()
                self.stream.synchronize()
                idx = self.idx.cpu().numpy()
                out.append([len(set(idx[l].ravel().tolist())) for l in range(idx.shape[0])])
        status = self.fpx.fpx_read_status(self.ws[:4].view(torch.int32), self.stream)
        if status != 0:
            raise RuntimeError(f"device status {status}")
        return out


def timed(runner, steps, warmup, world):
    torch = runner.torch
    with torch.cuda.stream(runner.stream):
        for i in range(warmup):
            runner.step(i)
        runner.stream.synchronize()
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(runner.stream)
        for i in range(steps):
            runner.step(i)
        e1.record(runner.stream)
        e1.synchronize()
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
    return e0.elapsed_time(e1) / 1e3


def kernel_profile(runner, steps):
    """Per-kernel average durations (ms) from CUDA events recorded around every kernel, on the stream
    the kernels run on."""
    import ctypes as C
    torch = runner.torch
    L = len(runner.stack.layers)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(NK * L + 1)]
    with torch.cuda.stream(runner.stream):
        for e in evs:
            e.record(runner.stream)  # materialise the handles
        runner.stream.synchronize()
        handles = [e.cuda_event for e in evs]
        sums = np.zeros(NK)
        per_layer = np.zeros((NK, L))
        for i in range(steps):
            runner.rin.copy_(runner.batches[i % N_BATCHES])
            runner.call(events=handles)
            runner.stream.synchronize()
            for l in range(L):
                for j in range(NK):
                    dt = evs[NK * l + j].elapsed_time(evs[NK * l + j + 1])
                    sums[j] += dt
                    per_layer[j, l] += dt
    return sums / (steps * L), per_layer / steps


def e2e_pass(runner, steps, world):
    """The same metric through the public API with host buffers: each step copies the step's tokens
    from pinned host memory, runs the pass and reads the result (residual and routing) back."""
    torch = runner.torch
    host_in = [torch.from_numpy(tokens_fp32(b, runner.q)).pin_memory() for b in range(N_BATCHES)]
    host_r = torch.empty(runner.q, H).pin_memory()
    host_idx = torch.empty(runner.idx.shape, dtype=torch.int32).pin_memory()
    with torch.cuda.stream(runner.stream):
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(runner.stream)
        for i in range(steps):
            runner.rin.copy_(host_in[i % N_BATCHES], non_blocking=True)
            runner.graph.replay() if runner.graph is not None else runner.call()
            host_r.copy_(runner.rL, non_blocking=True)
            host_idx.copy_(runner.idx, non_blocking=True)
        e1.record(runner.stream)
        e1.synchronize()
        if world > 1:
            torch.distributed.barrier()
    h2d = host_in[0].numel() * 4
    d2h = host_r.numel() * 4 + host_idx.numel() * 4
    return e0.elapsed_time(e1) / 1e3, h2d, d2h


LAYER_SOURCES = ("fpx_common.cuh", "fpx_mma.cuh", "route.cuh", "moe.cu")  # what the MoE layer kernels are built from


def csrc_digest():
    """Digest of the layer kernels' sources and header: a recorded DRAM count is used only while it
    matches, i.e. while the profiled kernels are unchanged."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "bit_block_quantized_wt_b300", "csrc")
    for n in LAYER_SOURCES:
        h.update(open(os.path.join(d, n), "rb").read())
    h.update(open(os.path.join(ROOT, "include", "fpx.h"), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, alg_bytes):
    """DRAM bytes per launch from the committed ncu capture, if it was taken on the current sources: the
    captured launch's DRAM bytes per algorithmic byte (its union differs from the average one) times
    this run's algorithmic bytes per launch."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)
        if t.get("csrc") == csrc_digest() and kernel in t.get("kernels", {}):
            return round(t["kernels"][kernel]["dram_per_algorithmic_byte"] * alg_bytes)
    except Exception:
        pass
    return None


# ---------------------------------------------------------------------------- CPU oracle

def cpu_model():
    """The host CPU's model name (first 'model name' line of /proc/cpuinfo), or None."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return None


def oracle_layer_steps(stack_seed, r_trace, idx, budget_s, max_layers):
    """Times the oracle on whole layer-steps of the q=4 pass (teacher-forced on the GPU's residual):
    returns (seconds, packed bytes, layers)."""
    import oracle
    import synth
    spent, nbytes, done = 0.0, 0, 0
    for l in range(max_layers):
        uni = sorted(set(int(v) for v in idx[l].ravel()))
        g, u, d = [None] * E, [None] * E, [None] * E
        for e in uni:
            g[e] = synth.matrix(2, I, H, stack_seed, l, synth.GATE, e)
            u[e] = synth.matrix(2, I, H, stack_seed, l, synth.UP, e)
            d[e] = synth.matrix(3, H, I, stack_seed, l, synth.DOWN, e)
        sh = [synth.matrix(4, I, H, stack_seed, l, synth.SH_GATE), synth.matrix(4, I, H, stack_seed, l, synth.SH_UP),
              synth.matrix(4, H, I, stack_seed, l, synth.SH_DOWN)]
        R = synth.router(E, H, stack_seed, l)
        x = oracle.rmsnorm_bf16(r_trace[l])
        t0 = time.perf_counter()
        oracle.moe_layer(H, I, E, R, g, u, d, *sh, x, K_TOP)
        spent += time.perf_counter() - t0
        nbytes += layer_bytes(len(uni))
        done += 1
        if spent >= budget_s:
            break
    return spent, nbytes, done


ID_N, ID_K = 148 * 64 * 16, 4096  # integer-dot comparison: 151,552 rows (FP2 194 MB, larger than L2)


def idot_measure(fpx, peak, reps=10):
    """fpx_gemv_q_idot (byte-permute expansion + dp4a) against fpx_gemv_q (binary16 decode + tensor-core
    MMA) and fpx_gemv_q_tiled (the same decode on the box-tiled layout, streamed like the MoE layer's
    experts) on matrices of the same size, q = 4 and q = 1, CUDA events. Packed bytes are uniform
    (scales included; the values do not change the work, and a tiled matrix of uniform bytes is again
    uniform). Bytes per call: the packed matrix."""
    import torch
    g = torch.Generator(device="cuda").manual_seed(13)
    res = {}
    x = torch.randn(4, ID_K, device="cuda", generator=g).to(torch.bfloat16).contiguous()
    y = torch.empty(4, ID_N, device="cuda")
    wsb = fpx.fpx_gemv_idot_workspace_bytes(ID_K, 4)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    wtb = max(fpx.fpx_gemv_tiled_workspace_bytes(fmt, ID_N, ID_K, 4) for fmt in (2, 3, 4))
    wt = torch.empty(wtb, dtype=torch.uint8, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for fmt in (2, 3, 4):
        nb = fpx.fpx_matrix_bytes(fmt, ID_N, ID_K)
        Wq = torch.randint(0, 256, (nb,), dtype=torch.uint8, device="cuda", generator=g)
        for q in ((4, 1) if fmt == 2 else (4,)):
            for name, call in (("int_dot", lambda: fpx.fpx_gemv_q_idot(fmt, Wq, ID_N, ID_K, x, fpx.FPX_DTYPE_BF16, q,
                                                                        y, ws, wsb)),
                               ("tensor_core", lambda: fpx.fpx_gemv_q(fmt, Wq, ID_N, ID_K, x, fpx.FPX_DTYPE_BF16, q, y)),
                               ("tensor_core_tiled", lambda: fpx.fpx_gemv_q_tiled(fmt, Wq, ID_N, ID_K, x, fpx.FPX_DTYPE_BF16,
                                                                                  q, y, wt, wtb))):
                for _ in range(3):
                    call()
                torch.cuda.synchronize()
                e0.record()
                for _ in range(reps):
                    call()
                e1.record()
                e1.synchronize()
                ms = e0.elapsed_time(e1) / reps
                res[f"fp{fmt}_q{q}_{name}"] = {"ms": round(ms, 4), "GB/s": round(nb / (ms / 1e3) / 1e9, 1),
                                               "frac_of_hbm_peak": round(nb / (ms / 1e3) / 1e9 / peak, 4)}
        del Wq
    return {"workload": f"dense {ID_N}x{ID_K} packed matrices (FP2 {fpx.fpx_matrix_bytes(2, ID_N, ID_K) / 1e6:.0f} MB, "
                        "larger than L2), bfloat16 N(0,1) activations", "reps": reps, "results": res}


def tiered_measure(fpx, stack, reps=16):
    """moe_layer_decode_tiered on layer 0 with the 128 even-numbered experts in HBM slots and the other
    128 in pinned host memory, against moe_layer_decode on the all-HBM layer; q = 4, top-4, CUDA
    events. Without a cache (Q * K_TOP staging slots, 8 token batches rotating) every call copies the
    cold experts of its union (gate + up + down, counted from the routing). With the staging cache:
    16 slots on the same 8 rotating batches, and 64 slots on a new batch every call (no repeated
    tokens); their copies per call come from the cache's copy count."""
    import torch
    import synth
    g, u, d, sh, R = stack.bufs[0]
    mb_gu, mb_d = fpx.fpx_matrix_bytes(2, I, H), fpx.fpx_matrix_bytes(3, H, I)
    per_expert = 2 * mb_gu + mb_d
    hot = torch.arange(0, E, 2)
    n_hot = len(hot)
    cold = [full.cpu().pin_memory() for full in (g, u, d)]
    slot_of = torch.full((E,), -1, dtype=torch.int32)
    slot_of[hot] = torch.arange(n_hot, dtype=torch.int32)
    slot_of = slot_of.cuda()
    keep = []

    def tiered_layer(n_stage, cached):
        n_slots = n_hot + n_stage
        arrays = []
        for full, mb in ((g, mb_gu), (u, mb_gu), (d, mb_d)):
            a = torch.zeros(n_slots * mb, dtype=torch.uint8, device="cuda")
            a.view(n_slots, mb)[:n_hot] = full.view(E, mb)[hot.cuda()]
            arrays.append(a)
        cache = torch.zeros(2 + 2 * n_stage, dtype=torch.int32, device="cuda") if cached else None
        keep.append((arrays, cache))
        lay = fpx.moe_layer(H=H, I=I, E=E, router=R.data_ptr(), gate=arrays[0].data_ptr(), up=arrays[1].data_ptr(),
                            down=arrays[2].data_ptr(), sh_gate=sh[0].data_ptr(), sh_up=sh[1].data_ptr(),
                            sh_down=sh[2].data_ptr())
        tiers = fpx.moe_tiers(slot_of=slot_of.data_ptr(), cold_gate=cold[0].data_ptr(), cold_up=cold[1].data_ptr(),
                              cold_down=cold[2].data_ptr(), n_slots=n_slots, stage_slot0=n_hot, n_stage=n_stage,
                              cache=cache.data_ptr() if cached else None)
        if cached:
            fpx.moe_tiers_cache_reset(tiers)
        return lay, tiers, cache

    ws_b = fpx.moe_workspace_bytes(stack.layers[0], Q, K_TOP)
    ws = torch.empty(ws_b, dtype=torch.uint8, device="cuda")
    rot = [torch.from_numpy(synth.tokens_bf16(Q, H, seed=2000 + b)[0].view(np.int16)).cuda() for b in range(N_BATCHES)]
    fresh = [torch.from_numpy(synth.tokens_bf16(Q, H, seed=3000 + b)[0].view(np.int16)).cuda() for b in range(reps + 3)]
    y = torch.empty(Q, H, device="cuda")
    idx = torch.empty(Q, K_TOP, dtype=torch.int32, device="cuda")
    n_cold = []
    for b in range(N_BATCHES):
        fpx.moe_layer_decode(stack.layers[0], rot[b], Q, K_TOP, y, ws, ws_b, idx_out=idx)
        torch.cuda.synchronize()
        n_cold.append(sum(1 for e in set(idx.cpu().numpy().ravel().tolist()) if e % 2 == 1))
    modes = {"all_hbm": (None, rot), "two_tier": (tiered_layer(Q * K_TOP, False), rot),
             "two_tier_cache16": (tiered_layer(Q * K_TOP, True), rot), "two_tier_cache64_fresh": (tiered_layer(64, True), fresh)}
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    res, copies = {}, {}
    for name, (tl, xs) in modes.items():
        def run(b):
            if tl is None:
                fpx.moe_layer_decode(stack.layers[0], xs[b % len(xs)], Q, K_TOP, y, ws, ws_b, idx_out=idx)
            else:
                fpx.moe_layer_decode_tiered(tl[0], tl[1], xs[b % len(xs)], Q, K_TOP, y, ws, ws_b, idx_out=idx)
        for b in range(3):
            run(b)
        torch.cuda.synchronize()
        c0 = int(tl[2][1]) if tl is not None and tl[2] is not None else None
        e0.record()
        for b in range(3, 3 + reps):
            run(b)
        e1.record()
        e1.synchronize()
        res[name] = e0.elapsed_time(e1) / reps
        if c0 is not None:
            copies[name] = (int(tl[2][1]) - c0) / reps
    st = fpx.fpx_read_status(ws[:4].view(torch.int32))
    cold_rot = float(np.mean([n_cold[b % N_BATCHES] for b in range(3, 3 + reps)]))
    staged = cold_rot * per_expert
    extra = res["two_tier"] - res["all_hbm"]
    out = {"workload": f"layer 0 (H {H}, I {I}, {E} experts, q {Q}, top-{K_TOP}); even experts in HBM, odd in pinned "
                       "host memory", "hot_experts": n_hot, "status": st,
           "ms_per_layer_all_hbm": round(res["all_hbm"], 4), "ms_per_layer_two_tier": round(res["two_tier"], 4),
           "cold_experts_per_call": round(cold_rot, 2), "staged_MB_per_call": round(staged / 1e6, 2),
           "staged_GB_per_s": round(staged / (extra / 1e3) / 1e9, 1) if extra > 0 else None, "reps": reps}
    for name in ("two_tier_cache16", "two_tier_cache64_fresh"):
        out[name] = {"ms_per_layer": round(res[name], 4), "copied_experts_per_call": round(copies[name], 2),
                     "staged_MB_per_call": round(copies[name] * per_expert / 1e6, 2)}
    return out


def run_fpx(args):
    import torch
    world, rank, local = dist_env()
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    import bit_block_quantized_wt_b300 as fpx
    fpx.lib()
    peak, peak_kind = peaks()

    stack = Stack(args.layers)
    r4 = Runner(stack, Q, K_TOP, graph=not args.no_graph)
    unions = r4.union_sizes()
    bytes_per_batch = [sum(layer_bytes(n) for n in u) for u in unions]
    with ClockSampler(local) as clk:
        secs = timed(r4, args.steps, args.warmup, world)
    step_bytes = sum(bytes_per_batch[i % N_BATCHES] for i in range(args.steps))
    secs, total_bytes = over_ranks(secs, step_bytes, world)
    value = total_bytes / secs / 1e9
    ms_step = secs / args.steps * 1e3

    # per-kernel durations (events around every kernel of the pass, on its stream)
    prof_steps = max(3, min(20, args.steps))
    kavg, kper_layer = kernel_profile(r4, prof_steps)
    names = ["k_router", "k_gate_up", "k_hpack", "k_down", "k_combine"]
    mean_union = float(np.mean([np.mean(u) for u in unions]))
    # k_hpack reads the 2 K parts of g and u of every item and writes the down table sets (17 I bytes
    # each); k_combine reads the 2 K parts of every routed output, the shared output and r, and writes r
    alg = [stack.layers[0].E * H * 4, gate_up_bytes(mean_union),
           (mean_union + 1) * (4 * Q * I * 4 + 17 * I), down_bytes(mean_union),
           (2 * mean_union + 3) * Q * H * 4]
    dom = int(np.argmax(kavg))
    achieved = alg[dom] / (kavg[dom] / 1e3) / 1e9

    # q = 1 autoregressive pass
    r1 = Runner(stack, 1, K_TOP, graph=not args.no_graph)
    u1 = r1.union_sizes()
    b1 = [sum(layer_bytes(n) for n in u) for u in u1]
    s1 = max(10, args.steps // 2)
    secs1, bytes1 = over_ranks(timed(r1, s1, args.warmup, world), sum(b1[i % N_BATCHES] for i in range(s1)), world)

    e2e_steps = max(10, min(args.steps, 200))
    e2e_secs, h2d, d2h = e2e_pass(r4, e2e_steps, world)
    e2e_secs, e2e_bytes = over_ranks(e2e_secs, sum(bytes_per_batch[i % N_BATCHES] for i in range(e2e_steps)), world)

    if args.part == "stack":  # the stack pass alone (profiling runs)
        pf = dc = qw = idm = tm = None
    else:
        pf = prefill_measure(fpx, stack.layers[0], args.warmup)
        dc = commit_measure(fpx, peak)
        qw = quantize_weighted_measure(fpx)
        idm = idot_measure(fpx, peak)
        tm = tiered_measure(fpx, stack)

    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded generator; packed codes uniform, "
        "binary16 scales U[0.005,0.05], tokens N(0,1) bfloat16)",
        "config": {"workload": WORKLOAD, "layers": args.layers, "q": Q, "top_k": K_TOP,
                   "resident_weight_bytes": len(stack.layers) * layer_bytes(E) + len(stack.layers) * E * H * 4,
                   "l2": "inputs larger than L2: ~150 MB of distinct expert weights per step out of ~99 GB "
                         "resident, 8 token batches rotate", "graph": r4.graph is not None,
                   "parallelism": f"replicas x{world}"},
        "frac_of_hbm_peak": round(value / world / peak, 4),
        "layer_steps_per_s": round(args.layers * args.steps * world / secs, 1),
        "verified_tokens_per_s": round(Q * args.steps * world / secs, 1),
        "stack_passes_per_s": round(args.steps * world / secs, 2),
        "mean_union_experts": round(mean_union, 3),
        "q1": {"value": round(bytes1 / secs1 / 1e9, 2), "unit": "GB/s", "ms_per_step": round(secs1 / s1 * 1e3, 4),
               "layer_steps_per_s": round(args.layers * s1 * world / secs1, 1),
               "tokens_per_s": round(s1 * world / secs1, 1)},
        "kernels_ms": {n: round(float(v), 5) for n, v in zip(names, kavg)},
        # achieved GB/s of every layer kernel: its algorithmic bytes (above) over its event-timed duration
        "kernels_gbs": {n: round(a / (float(v) / 1e3) / 1e9, 1) for n, a, v in zip(names, alg, kavg)},
        "roofline": {"kernel": names[dom], "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": recorded_traffic(names[dom], alg[dom]), "algorithmic_bytes_per_launch": round(alg[dom]),
                     "avg_launch_ms": round(float(kavg[dom]), 5)},
        "e2e": {"value": round(e2e_bytes / e2e_secs / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "prefill": pf,
        "verify_commit": dc,
        "quantize_weighted": qw,
        "gemv_int_dot": idm,
        "two_tier": tm,
        "gpu_launches": args.steps * NK * args.layers,
        "clocks": clk.summary(),
    }
    if rank == 0 and world == 1 and not args.skip_cpu and args.part != "stack":
        import oracle
        with torch.cuda.stream(r4.stream):
            tr = torch.empty(args.layers, Q, H, device="cuda")
            r4.rin.copy_(r4.batches[0])
            fpx.moe_stack_verify(stack.layers, r4.rin, Q, K_TOP, r4.rL, r4.ws, r4.ws_b, idx_out=r4.idx, r_trace=tr)
            r4.stream.synchronize()
        trn, idn = tr.cpu().numpy(), r4.idx.cpu().numpy()
        cs, cb, cl = oracle_layer_steps(0, trn, idn, args.cpu_seconds, args.layers)
        cores = oracle.threads()
        prev = oracle.set_threads(1)  # the same layer-steps on one core, at least one, bounded in time
        cs1, cb1, cl1 = oracle_layer_steps(0, trn, idn, args.cpu_seconds / 2, args.layers)
        oracle.set_threads(prev)
        out["cpu_baseline"] = {"value": round(cb / cs / 1e9, 5), "unit": "GB/s", "cores": cores,
                               "kind": "oracle", "cpu_model": cpu_model(),
                               "sample": f"{cl} whole layer-steps (layers 0..{cl - 1}) of the q=4 "
                               f"verify pass on token batch 0, teacher-forced on the GPU residual; {cs:.1f} s",
                               "seconds": round(cs, 2), "bytes": cb,
                               "single_thread": {"value": round(cb1 / cs1 / 1e9, 5), "unit": "GB/s", "cores": 1,
                                                 "layer_steps": cl1, "seconds": round(cs1, 2)}}
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_reference(args):
    """The oracle as it stands on this host's cores: each step is a bounded sample of the workload
    (rows of the routed expert matrices one layer-step touches, applied to the q = 4 tokens)."""
    world, rank, local = dist_env()
    if rank != 0:
        return
    import oracle
    import synth
    budget = args.ref_seconds
    layer = 0
    R = synth.router(E, H, 0, layer)
    x = synth.tokens_bf16(Q, H, seed=1000)[1].astype(np.float64)
    route = oracle.route(R, x, K_TOP)
    uni = list(route["uni"])
    mats = []
    for e in uni:
        mats.append((2, synth.matrix(2, I, H, 0, layer, synth.GATE, e), I, H))
        mats.append((2, synth.matrix(2, I, H, 0, layer, synth.UP, e), I, H))
        mats.append((3, synth.matrix(3, H, I, 0, layer, synth.DOWN, e), H, I))
    hvec = synth.tokens_bf16(Q, I, seed=7)[1].astype(np.float64)

    def sample(rows):
        t0, nbytes = time.perf_counter(), 0
        for i, (fmt, m, N, Kd) in enumerate(mats):
            rb = Kd // 32 * oracle.block_bytes(fmt)
            r0 = (i * 97) % (N - rows + 1)
            oracle.gemv(fmt, m[r0 * rb:(r0 + rows) * rb], rows, Kd, x if Kd == H else hvec)
            nbytes += rows * rb
        return time.perf_counter() - t0, nbytes

    dt, _ = sample(16)
    per_row = dt / 16
    rows = int(max(4, min(I, budget / (args.steps + args.warmup) / per_row)))
    for _ in range(args.warmup):
        sample(rows)
    tot_t, tot_b = 0.0, 0
    for _ in range(args.steps):
        dt, nb = sample(rows)
        tot_t += dt
        tot_b += nb
    v = tot_b / tot_t / 1e9
    desc = (f"per step: {rows} rows of each of the {len(mats)} routed expert matrices (gate/up FP2, down FP3) "
            f"that one q=4 layer-step touches, applied to the 4 tokens")
    out = {"impl": "reference", "metric": METRIC, "value": round(v, 5), "unit": "GB/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tot_t / args.steps * 1e3, 3),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic", "config": {"workload": WORKLOAD, "layers": LAYERS, "q": Q, "top_k": K_TOP},
           "cpu_baseline": {"value": round(v, 5), "unit": "GB/s", "cores": oracle.threads(), "kind": "oracle",
                            "cpu_model": cpu_model(), "sample": desc},
           "e2e": {"value": round(v, 5), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["fpx", "reference"], default="fpx")
    p.add_argument("--layers", type=int, default=LAYERS)
    p.add_argument("--no-graph", action="store_true", help="launch the pass directly instead of a CUDA graph")
    p.add_argument("--skip-cpu", action="store_true", help="omit the CPU-oracle baseline")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--ref-seconds", type=float, default=90.0)
    p.add_argument("--part", choices=["all", "stack", "idot", "tiered", "prefill", "commit", "quantize"], default="all",
                   help="stack: only the stack passes (q = 4, q = 1, end to end; no CPU baseline); "
                        "idot: only the integer-dot / tensor-core GEMV comparison; tiered: only the two-tier "
                        "residency measurement on a one-layer stack; prefill: only the prefill of one layer "
                        "(--warmup calls, then --steps timed calls); commit: only the verify/commit rule; "
                        "quantize: only the importance-weighted quantizer (one JSON object each)")
    args = p.parse_args()
    if args.warmup < 3:
        p.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.part == "idot":
        import torch
        import bit_block_quantized_wt_b300 as fpx
        torch.cuda.set_device(0)
        fpx.lib()
        print(json.dumps(idot_measure(fpx, peaks()[0])), flush=True)
    elif args.part in ("tiered", "prefill", "commit", "quantize"):
        import torch
        import bit_block_quantized_wt_b300 as fpx
        torch.cuda.set_device(0)
        fpx.lib()
        if args.part == "tiered":
            res = tiered_measure(fpx, Stack(1))
        elif args.part == "prefill":
            res = prefill_measure(fpx, Stack(1).layers[0], args.warmup, reps=args.steps)
        elif args.part == "commit":
            res = commit_measure(fpx, peaks()[0], reps=args.steps)
        else:
            res = quantize_weighted_measure(fpx, reps=args.steps)
        print(json.dumps(res), flush=True)
    else:
        run_fpx(args)


if __name__ == "__main__":
    main()
