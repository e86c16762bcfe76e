"""Pins for the oracle model of the host page allocator (oracle/allocator.py):
a hand-derived scenario (tests/golden/alloc_scenario.json) and invariants
that hold after every operation of random call sequences:
  - every page is free or held: free + used = num_pages;
  - a page's reference count equals the number of open sequences holding it;
  - a sequence holds ceil((committed + reserved) / 16) pages, no page twice;
  - a page held by two sequences is complete and committed in each;
  - a refused admission changes nothing."""
import json
import os

import numpy as np
import pytest

from alloc_driver import run_oracle
from conftest import GOLDEN
from oracle import allocator as OA


def _scenario():
    with open(os.path.join(GOLDEN, "alloc_scenario.json")) as f:
        return json.load(f)


def test_hand_derived_scenario():
    sc = _scenario()
    a = OA.Allocator(sc["num_pages"], sc["max_seqs"], sc["max_pages_per_seq"])
    for step in sc["steps"]:
        got = run_oracle(a, step)
        if "error" in step:
            assert got == step["error"], step
        elif "want" in step:
            assert got == step["want"], step
        else:
            assert got is None, step
        if "table" in step:
            seq = step["want"] if step["op"] == "fork" else step["seq"]
            assert a.block_table(seq, len(step["table"])) == step["table"], step
        if "info" in step:
            seq = step["want"] if step["op"] == "fork" else step["seq"]
            assert list(a.info(seq)) == step["info"], step


def _check_invariants(a):
    free, used, shared = a.stats()
    assert free + used == a.num_pages
    holders = [0] * a.num_pages
    for s, q in a.seqs.items():
        assert len(q["pages"]) == OA.pages_for(q["committed"] + q["reserved"])
        assert len(set(q["pages"])) == len(q["pages"])
        for p in q["pages"]:
            holders[p] += 1
    assert holders == a.refs
    for s, q in a.seqs.items():
        for k, p in enumerate(q["pages"]):
            if a.refs[p] >= 2:  # shared: a complete committed page of every holder
                assert (k + 1) * OA.PAGE <= q["committed"]
    assert shared == sum(1 for r in a.refs if r >= 2)


def random_ops(seed, n_ops=400, num_pages=40, max_seqs=6, max_pages=9):
    rng = np.random.default_rng(seed)
    ops = []
    for _ in range(n_ops):
        k = rng.choice(["open", "reserve", "reserve", "commit", "commit", "unreserve", "fork",
                        "release", "info", "stats", "batch", "reserve_many", "commit_many"])
        s = int(rng.integers(-1, max_seqs + 1))  # includes ids that are closed or out of range
        if k in ("reserve", "commit", "unreserve"):
            ops.append({"op": k, "seq": s, "n": int(rng.integers(-1, 40))})
        elif k in ("fork", "release", "info"):
            ops.append({"op": k, "seq": s})
        elif k in ("reserve_many", "commit_many"):
            ops.append({"op": k, "seqs": [int(x) for x in rng.permutation(max_seqs)[:3]],
                        "n": int(rng.integers(-1, 30))})
        elif k == "batch":
            ops.append({"op": k, "seqs": [int(x) for x in rng.integers(0, max_seqs, 3)],
                        "extra": int(rng.integers(0, 3)), "stride": max_pages})
        else:
            ops.append({"op": k})
    return (num_pages, max_seqs, max_pages), ops


@pytest.mark.parametrize("seed", range(10))
def test_invariants_under_random_calls(seed):
    sizes, ops = random_ops(seed)
    a = OA.Allocator(*sizes)
    for op in ops:
        before = json.dumps([a.refs, sorted((s, q["committed"], q["reserved"], q["pages"])
                                            for s, q in a.seqs.items())])
        got = run_oracle(a, op)
        if got in ("capacity", "arg") and op["op"] in ("reserve", "commit", "unreserve", "batch",
                                                       "reserve_many", "commit_many"):
            after = json.dumps([a.refs, sorted((s, q["committed"], q["reserved"], q["pages"])
                                               for s, q in a.seqs.items())])
            assert before == after, f"refused {op} changed the state"
        _check_invariants(a)


def test_lowest_free_pages_first_and_release_returns_them():
    a = OA.Allocator(8, 3, 8)
    s0, s1 = a.open(), a.open()
    a.reserve(s0, 40)   # 3 pages
    a.reserve(s1, 16)   # 1 page
    assert a.block_table(s0, 3) == [0, 1, 2] and a.block_table(s1, 1) == [3]
    a.release(s0)
    s2 = a.open()
    assert s2 == s0  # lowest closed id is reused
    a.reserve(s2, 64)
    assert a.block_table(s2, 4) == [0, 1, 2, 4]
