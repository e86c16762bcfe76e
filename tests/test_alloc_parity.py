"""The library's host page allocator (pkv_alloc_*, through the C ABI)
against the oracle model, on the CPU: the hand-derived scenario, and random
call sequences compared call by call (result or typed error) and state by
state (every open sequence's block table and counts, every page's
reference count, the statistics) -- exact equality throughout."""
import json
import os

import pytest

from alloc_driver import run_native, run_oracle
from conftest import GOLDEN
from oracle import allocator as OA
from test_oracle_allocator import random_ops


@pytest.fixture(scope="module")
def api():
    from paged_kv_decode_09_gb300 import api, build
    build.build()
    return api


def _state_native(a, sizes):
    num_pages, max_seqs, max_pages = sizes
    seqs = {}
    for s in range(max_seqs):
        try:
            info = a.info(s)
        except Exception:
            continue
        seqs[s] = (list(info), [int(x) for x in a.block_table(s, max_pages)])
    return seqs, [a.page_refs(p) for p in range(num_pages)], list(a.stats())


def _state_oracle(a, sizes):
    num_pages, max_seqs, max_pages = sizes
    seqs = {s: (list(a.info(s)), a.block_table(s, max_pages)) for s in sorted(a.seqs)}
    return seqs, list(a.refs), list(a.stats())


def test_scenario_native(api):
    with open(os.path.join(GOLDEN, "alloc_scenario.json")) as f:
        sc = json.load(f)
    a = api.PageAllocator(sc["num_pages"], sc["max_seqs"], sc["max_pages_per_seq"])
    for step in sc["steps"]:
        got = run_native(a, step)
        if "error" in step:
            assert got == step["error"], step
        elif "want" in step:
            assert got == step["want"], step
        if "table" in step:
            seq = step["want"] if step["op"] == "fork" else step["seq"]
            assert [int(x) for x in a.block_table(seq, len(step["table"]))] == step["table"], step


@pytest.mark.parametrize("seed", range(12))
def test_random_calls_match_oracle(api, seed):
    sizes, ops = random_ops(seed, n_ops=500)
    nat = api.PageAllocator(*sizes)
    ora = OA.Allocator(*sizes)
    for k, op in enumerate(ops):
        assert run_native(nat, op) == run_oracle(ora, op), (k, op)
        assert _state_native(nat, sizes) == _state_oracle(ora, sizes), (k, op)


def test_large_pool_decode_loop(api):
    """A decode-style loop at serving scale: 256 sequences admitted with
    prompts, then steps of reserve 1 / batch / commit 1 until the pool is
    full, with the oracle kept in lockstep on a sample of the calls."""
    sizes = (20000, 256, 512)
    nat, ora = api.PageAllocator(*sizes), OA.Allocator(*sizes)
    seqs = []
    for s in range(256):
        for a, run in ((nat, run_native), (ora, run_oracle)):
            assert run(a, {"op": "open"}) == s
            assert run(a, {"op": "reserve", "seq": s, "n": 100 + 7 * s}) is None
            assert run(a, {"op": "commit", "seq": s, "n": 100 + 7 * s}) is None
        seqs.append(s)
    for step in range(40):
        for s in seqs:
            r1 = run_native(nat, {"op": "reserve", "seq": s, "n": 1})
            r2 = run_oracle(ora, {"op": "reserve", "seq": s, "n": 1})
            assert r1 == r2
        b1 = run_native(nat, {"op": "batch", "seqs": seqs, "extra": 1, "stride": 512})
        b2 = run_oracle(ora, {"op": "batch", "seqs": seqs, "extra": 1, "stride": 512})
        assert b1 == b2
        for s in seqs:
            assert run_native(nat, {"op": "commit", "seq": s, "n": 1}) == \
                run_oracle(ora, {"op": "commit", "seq": s, "n": 1})
    assert list(nat.stats()) == list(ora.stats())
