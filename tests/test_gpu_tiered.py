"""moe_layer_decode_tiered (two-tier expert residency) against moe_layer_decode on the same layer held
entirely in HBM: output, routing and logits bit-identical for any split of the experts into hot (HBM
slots) and cold (pinned host memory), and the staging slots hold exactly the cold experts of the
union afterwards. With a staging cache, the slots keep their experts across calls: the cache's slots,
last uses and copy count follow a host model of the least-recently-used policy call by call, a
repeated union copies nothing, and every slot the cache names holds that expert's matrices. The
all-HBM call is itself checked against the oracle (test_gpu_layer.py); one case here repeats that
check on the tiered output."""
import numpy as np
import pytest
import torch

import bit_block_quantized_wt_b300 as fpx
import synth
from gpu_util import DeviceLayer, dev, host, need_gpu, read_status

pytestmark = pytest.mark.gpu
TOL = 2e-3


class Tiered:
    """A two-tier copy of a DeviceLayer: the listed hot experts in HBM slots 0..n_hot-1, n_stage
    staging slots after them (filled with 0xA5), every expert in pinned host memory."""

    def __init__(self, L, hot, n_stage, bad_slot=None, cache=False):
        self.L, self.hot = L, list(hot)
        self.hot_eff = [e for e in self.hot if e != bad_slot]  # a bad slot makes its expert cold
        n_hot = len(self.hot)
        self.n_slots = n_hot + n_stage
        self.arrays = []
        for full, mb in ((L.gate, L.mb_gu), (L.up, L.mb_gu), (L.down, L.mb_d)):
            a = torch.full((self.n_slots * mb,), 0xA5, dtype=torch.uint8, device="cuda")
            for i, e in enumerate(self.hot):
                a[i * mb:(i + 1) * mb] = full[e * mb:(e + 1) * mb]
            self.arrays.append(a)
        self.cold = [full.cpu().pin_memory() for full in (L.gate, L.up, L.down)]
        slot_of = np.full(L.E, -1, np.int32)
        slot_of[self.hot] = np.arange(n_hot, dtype=np.int32)
        if bad_slot is not None:
            slot_of[bad_slot] = self.n_slots + 3  # outside the arrays: must be treated as cold
        self.slot_of = dev(slot_of)
        self.c = fpx.moe_layer(H=L.H, I=L.I, E=L.E, router=L.router.data_ptr(), gate=self.arrays[0].data_ptr(),
                               up=self.arrays[1].data_ptr(), down=self.arrays[2].data_ptr(),
                               sh_gate=L.sh[0].data_ptr(), sh_up=L.sh[1].data_ptr(), sh_down=L.sh[2].data_ptr())
        self.cache = torch.full((2 + 2 * n_stage,), 12345, dtype=torch.int32, device="cuda") if cache else None
        self.t = fpx.moe_tiers(slot_of=self.slot_of.data_ptr(), cold_gate=self.cold[0].data_ptr(),
                               cold_up=self.cold[1].data_ptr(), cold_down=self.cold[2].data_ptr(),
                               n_slots=self.n_slots, stage_slot0=n_hot, n_stage=n_stage,
                               cache=self.cache.data_ptr() if cache else None)
        if cache:
            fpx.moe_tiers_cache_reset(self.t)


def run(call, layer_c, bits, k, E, H):
    q = bits.shape[0]
    ws_b = fpx.moe_workspace_bytes(layer_c, q, k)
    ws = torch.empty(ws_b, dtype=torch.uint8, device="cuda")
    y = torch.full((q, H), float("nan"), device="cuda")
    idx = torch.empty(q, k, dtype=torch.int32, device="cuda")
    lg = torch.empty(q, E, device="cuda")
    call(ws, ws_b, y, idx, lg)
    return host(y), host(idx), host(lg), read_status(ws[:4].view(torch.int32))


def compare(L, T, bits, k, expect_status=0):
    q = bits.shape[0]
    xd = dev(bits)
    full = run(lambda ws, wb, y, idx, lg: fpx.moe_layer_decode(L.c, xd, q, k, y, ws, wb, idx_out=idx, logits_out=lg),
               L.c, bits, k, L.E, L.H)
    tier = run(lambda ws, wb, y, idx, lg: fpx.moe_layer_decode_tiered(T.c, T.t, xd, q, k, y, ws, wb, idx_out=idx,
                                                                      logits_out=lg),
               T.c, bits, k, L.E, L.H)
    assert full[3] == 0 and tier[3] == expect_status
    assert np.array_equal(full[1], tier[1])  # routing
    assert np.array_equal(full[2], tier[2])  # logits
    assert np.array_equal(full[0], tier[0])  # output, bit for bit
    uni = sorted(set(int(e) for e in full[1].ravel()))
    cold = [e for e in uni if e not in set(T.hot_eff)]
    stage0 = T.t.stage_slot0
    if T.cache is None:  # the i-th cold expert (ascending) sits in staging slot i
        where = {e: i for i, e in enumerate(cold)}
    else:  # every expert the cache names sits in its slot; the union's cold experts are among them
        held = host(T.cache)[2:2 + T.t.n_stage]
        where = {int(e): i for i, e in enumerate(held) if e >= 0}
        assert len(where) == int((held >= 0).sum())  # no expert in two slots
        assert set(cold) <= set(where)
    for e, i in where.items():
        for a, f, mb in zip(T.arrays, (L.gate, L.up, L.down), (L.mb_gu, L.mb_gu, L.mb_d)):
            s = stage0 + i
            assert torch.equal(a[s * mb:(s + 1) * mb], f[e * mb:(e + 1) * mb]), (e, s)
    return full, cold


@pytest.mark.parametrize("split", ["half", "all_cold", "all_hot", "one_hot"])
@pytest.mark.parametrize("q,k", [(1, 4), (4, 4), (3, 8)])
def test_tiered_small_bit_identical(split, q, k):
    need_gpu()
    E = 16
    L = DeviceLayer(512, 512, E, seed=q + k)
    rng = np.random.default_rng(q * 10 + k)
    hot = {"half": sorted(rng.choice(E, E // 2, replace=False)), "all_cold": [], "all_hot": list(range(E)),
           "one_hot": [int(rng.integers(E))]}[split]
    T = Tiered(L, hot, n_stage=min(q * k, E) + 1)
    bits, _ = synth.tokens_bf16(q, 512, seed=k + 1)
    _, cold = compare(L, T, bits, k)
    if split == "all_hot":
        assert cold == []


def test_tiered_repeated_calls_and_bad_slot():
    """Consecutive calls on different tokens reuse the staging slots; an out-of-range slot_of entry
    sets FPX_EDATA and that expert is staged like a cold one."""
    need_gpu()
    E = 16
    L = DeviceLayer(512, 1024, E, seed=5)
    T = Tiered(L, hot=[0, 3, 4, 9, 12], n_stage=16)
    for seed in range(3):
        bits, _ = synth.tokens_bf16(4, 512, seed=40 + seed)
        compare(L, T, bits, 4)
    bits, _ = synth.tokens_bf16(4, 512, seed=7)
    xd = dev(bits)
    ws_b = fpx.moe_workspace_bytes(L.c, 4, 4)
    ws = torch.empty(ws_b, dtype=torch.uint8, device="cuda")
    idx = torch.empty(4, 4, dtype=torch.int32, device="cuda")
    fpx.moe_layer_decode(L.c, xd, 4, 4, torch.empty(4, 512, device="cuda"), ws, ws_b, idx_out=idx)
    bad = int(host(idx).ravel()[0])  # an expert of the union: only union experts are looked up
    Tb = Tiered(L, hot=sorted({0, 3, 4, 9, 12, bad}), n_stage=16, bad_slot=bad)
    compare(L, Tb, bits, 4, expect_status=1 << fpx.FPX_EDATA)


def test_tiered_config3_against_oracle():
    """hidden 4096, 256 experts, q = 4, top-4, the 128 even-numbered experts hot: bit-identical to the
    all-HBM call, and within the tolerance of the oracle."""
    need_gpu()
    L = DeviceLayer(4096, 2048, 256, seed=0, layer=0)
    T = Tiered(L, hot=list(range(0, 256, 2)), n_stage=16)
    bits, vals = synth.tokens_bf16(4, 4096, seed=0)
    full, cold = compare(L, T, bits, 4)
    assert len(cold) > 0
    orc = L.oracle(vals.astype(np.float64), 4, idx_force=full[1])
    err = np.abs(full[0].astype(np.float64) - orc["y"])
    assert np.all(err <= TOL * orc["M"])


def test_tiered_rejects_pageable_cold_tier():
    need_gpu()
    L = DeviceLayer(512, 512, 16, seed=1)
    T = Tiered(L, hot=[1, 2], n_stage=8)
    pageable = np.zeros(L.gate.numel(), np.uint8)
    T.t.cold_gate = pageable.ctypes.data
    bits, _ = synth.tokens_bf16(2, 512, seed=2)
    ws_b = fpx.moe_workspace_bytes(T.c, 2, 4)
    ws = torch.empty(ws_b, dtype=torch.uint8, device="cuda")
    y = torch.empty(2, 512, device="cuda")
    with pytest.raises(fpx.FpxError) as e:
        fpx.moe_layer_decode_tiered(T.c, T.t, dev(bits), 2, 4, y, ws, ws_b)
    assert e.value.status == fpx.FPX_EINVAL


class LruModel:
    """Host model of the staging cache: a held expert is used in place; a missing one takes the slot
    whose last use is oldest among those not taken by this call, ties to the lower slot."""

    def __init__(self, n):
        self.exp, self.use, self.clock, self.copies = [-1] * n, [0] * n, 0, 0

    def call(self, cold):
        self.clock += 1
        taken = set()
        for e in cold:
            if e in self.exp:
                i = self.exp.index(e)
            else:
                free = [i for i in range(len(self.exp)) if i not in taken]
                i = min(free, key=lambda i: (-((self.clock - self.use[i]) % 2**32), i))
                self.copies += 1
            self.exp[i], self.use[i] = e, self.clock
            taken.add(i)

    def state(self):
        return [self.clock, self.copies] + self.exp + self.use


@pytest.mark.parametrize("n_stage,hot", [(16, [0, 3, 4, 9, 12]), (16, []), (24, [1, 2, 5, 6, 7, 8, 10, 11])])
def test_tiered_cache_follows_lru(n_stage, hot):
    """A sequence of calls (new tokens, then repeats): bit-identical to the all-HBM layer each time, the
    device cache equal to the host model after every call, and a repeated union copies nothing."""
    need_gpu()
    E, q, k = 16, 4, 4
    L = DeviceLayer(512, 1024, E, seed=11)
    T = Tiered(L, hot=hot, n_stage=n_stage, cache=True)
    assert list(host(T.cache)) == [0, 0] + [-1] * n_stage + [0] * n_stage
    model = LruModel(n_stage)
    seeds = [60, 61, 62, 61, 63, 60, 60, 64, 65, 62]
    for c, seed in enumerate(seeds):
        bits, _ = synth.tokens_bf16(q, 512, seed=seed)
        copied = int(host(T.cache)[1])
        _, cold = compare(L, T, bits, k)
        model.call(cold)
        assert list(host(T.cache)) == model.state(), seed
        if c > 0 and seeds[c - 1] == seed:  # the previous call's union again: nothing to copy
            assert int(host(T.cache)[1]) == copied
    assert model.copies > 0


def test_tiered_cache_reset_and_limits():
    need_gpu()
    L = DeviceLayer(512, 512, 16, seed=2)
    T = Tiered(L, hot=[1, 2], n_stage=8, cache=True)
    bits, _ = synth.tokens_bf16(2, 512, seed=3)
    compare(L, T, bits, 4)
    st = host(T.cache)
    assert st[0] == 1 and st[1] > 0
    fpx.moe_tiers_cache_reset(T.t)
    assert list(host(T.cache)) == [0, 0] + [-1] * 8 + [0] * 8
    T.t.n_stage = 2000  # a cache tracks at most 1024 staging slots
    with pytest.raises(fpx.FpxError) as e:
        fpx.moe_tiers_cache_reset(T.t)
    assert e.value.status == fpx.FPX_EINVAL
