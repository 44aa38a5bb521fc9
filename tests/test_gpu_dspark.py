"""dspark_verify_commit against the oracle's commit rule: the target's choices, the accepted count and
the committed tokens bit-exact for every sequence, over small and large vocabularies (vector and
scalar row paths), many exact ties, drafts built to accept 0..q-1 tokens, and NaN rows."""
import numpy as np
import pytest
import torch

import bit_block_quantized_wt_b300 as fpx
import oracle
from gpu_util import dev, host, need_gpu, read_status, status_word

pytestmark = pytest.mark.gpu


def make_case(B, q, V, seed, ties=False):
    rng = np.random.default_rng(seed)
    if ties:
        lg = rng.integers(0, 4, size=(B, q, V)).astype(np.float32)
    else:
        lg = rng.standard_normal((B, q, V)).astype(np.float32)
    # drafts: the first a_s follow the target's own choice (host argmax, lowest index on ties), the
    # next one differs, for a_s uniform in 0..q-1
    choice = np.array([[int(np.flatnonzero(r == r.max())[0]) for r in seq] for seq in lg])
    drafts = np.zeros((B, max(q - 1, 0)), np.int32)
    for s in range(B):
        a = rng.integers(0, q)
        for j in range(q - 1):
            drafts[s, j] = choice[s, j] if j < a else (choice[s, j] + 1 + rng.integers(0, max(V - 1, 1))) % V
    return lg, drafts


def run(lg, drafts):
    B, q, V = lg.shape
    pred = torch.empty(B, q, dtype=torch.int32, device="cuda")
    n = torch.empty(B, dtype=torch.int32, device="cuda")
    com = torch.empty(B, q, dtype=torch.int32, device="cuda")
    st = status_word()
    d = dev(drafts) if q > 1 else None
    fpx.dspark_verify_commit(dev(lg), B, q, V, d, pred, n, com, dev_status=st)
    return host(pred), host(n), host(com), read_status(st)


@pytest.mark.parametrize("B,q,V,ties", [(1, 1, 1, False), (33, 4, 7, True), (17, 3, 1000, True), (8, 4, 131072, False),
                                        (5, 2, 131071, False), (64, 4, 4096, True)])
def test_commit_matches_oracle(B, q, V, ties):
    need_gpu()
    lg, drafts = make_case(B, q, V, seed=B * 7 + q, ties=ties)
    pred, n, com, st = run(lg, drafts)
    assert st == 0
    for s in range(B):
        p, nn, c, ost = oracle.dspark_commit(lg[s], drafts[s] if q > 1 else [])
        assert ost == 0
        assert list(pred[s]) == list(p) and n[s] == nn and list(com[s]) == list(c), s


def test_commit_nan_rows():
    need_gpu()
    lg, drafts = make_case(4, 4, 300, seed=1)
    lg[1, 2, 17] = np.nan            # one NaN: never chosen
    lg[2, 0, :] = np.nan             # all NaN: index 0 and the range status
    pred, n, com, st = run(lg, drafts)
    assert st & (1 << fpx.FPX_ERANGE)
    for s in range(4):
        p, nn, c, _ = oracle.dspark_commit(lg[s], drafts[s])
        assert list(pred[s]) == list(p) and n[s] == nn and list(com[s]) == list(c)
