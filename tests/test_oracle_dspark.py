"""Pins for the oracle's speculative verify/commit rule (CPU only): the hand-worked fixture, a brute
force over every draft of tiny vocabularies, and the closed forms of the special cases."""
import itertools
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "dspark_commit.txt")


def read_cases():
    cases, cur = [], None
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *vals = line.split()
        if key == "case":
            cur = {"name": vals[0], "logits": []}
            cases.append(cur)
        elif key == "logits":
            cur["logits"].append([float(v) for v in vals])
        elif key == "n":
            cur["n"] = int(vals[0])
        else:
            cur[key] = [int(v) for v in vals]
    return cases


def test_hand_worked_fixture():
    cases = read_cases()
    assert len(cases) == 5
    for c in cases:
        pred, n, com, st = oracle.dspark_commit(np.array(c["logits"], np.float32), c["drafts"])
        assert st == 0, c["name"]
        assert list(pred) == c["pred"], c["name"]
        assert n == c["n"], c["name"]
        assert list(com) == c["committed"], c["name"]


def brute(logits, drafts):
    """Direct restatement: accept the longest prefix of drafts that the target would itself have chosen,
    by enumerating every prefix length."""
    pred = [int(min(np.flatnonzero(row == row.max()))) for row in logits]
    best = 0
    for n in range(len(drafts) + 1):
        if all(drafts[j] == pred[j] for j in range(n)):
            best = n
    return pred, best, list(drafts[:best]) + [pred[best]] + [-1] * (len(logits) - best - 1)


def test_brute_force_tiny_vocabularies():
    rng = np.random.default_rng(3)
    for V in (1, 2, 3):
        for q in (1, 2, 3, 4):
            for _ in range(10):
                lg = rng.integers(0, 3, size=(q, V)).astype(np.float32)  # many exact ties
                for d in itertools.product(range(V), repeat=q - 1):
                    pred, n, com, st = oracle.dspark_commit(lg, list(d))
                    p2, n2, c2 = brute(lg, d)
                    assert st == 0 and list(pred) == p2 and n == n2 and list(com) == c2


def test_special_cases():
    rng = np.random.default_rng(4)
    lg = rng.standard_normal((4, 50)).astype(np.float32)
    pred, _, _, _ = oracle.dspark_commit(lg, [0, 0, 0])
    assert list(pred) == list(np.argmax(lg, axis=1))  # no ties: numpy's argmax
    # drafts equal to the target's own choices: all accepted, the bonus token is the last choice
    _, n, com, _ = oracle.dspark_commit(lg, list(pred[:3]))
    assert n == 3 and list(com) == list(pred)
    # a wrong first draft: nothing accepted, the target's first choice committed
    _, n, com, _ = oracle.dspark_commit(lg, [(pred[0] + 1) % 50, pred[1], pred[2]])
    assert n == 0 and list(com) == [pred[0], -1, -1, -1]
    # NaN is never chosen; an all-NaN row reports the range status
    lg2 = lg.copy(); lg2[1, pred[1]] = np.nan
    p2, _, _, st = oracle.dspark_commit(lg2, [0, 0, 0])
    assert st == 0 and p2[1] != pred[1]
    lg2[2, :] = np.nan
    _, _, _, st = oracle.dspark_commit(lg2, [0, 0, 0])
    assert st == oracle.ERANGE
