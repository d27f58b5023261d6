"""Pins of oracle/policy.py (verify prices and the StairCut cut) to hand
calculations and to properties the pages state, independently of the
oracle's own code paths."""
import itertools
import math

import numpy as np
import pytest

from oracle import policy as P
from speculative_tree_verify_gb300 import synth

TABLE = {1024: {"chain": {8: 10.0, 16: 12.0, 32: 20.0}, "tree": {8: 11.0, 16: 14.0, 24: 16.0, 32: 21.0}},
         32768: {"chain": {8: 30.0, 16: 33.0}, "tree": {8: 31.0, 16: 36.0, 24: 52.0}}}


def test_price_lookup_by_hand():
    pr = P.Prices(TABLE, step_ms=0.0)
    assert pr.price(1024, "tree", 16) == 14.0                 # a measured count
    assert pr.price(1024, "tree", 12) == 12.5                 # halfway between 8 and 16
    assert pr.price(2000, "tree", 20) == 15.0                 # class 1024 (nearest lower), 16..24 interpolate
    assert pr.price(500, "chain", 8) == 10.0                  # below every class: the lowest
    assert pr.price(40000, "tree", 28) == 52.0 + 2.0 * 4      # past the last count: the last slope (16 ms / 8 rows)
    assert pr.price(1024, "chain", 4) == 10.0                 # below the first count: the first count's price
    stepped = P.Prices(TABLE, step_ms=0.5)
    assert stepped.price(32768, "chain", 20) == 33.0 + 0.5 * 4


def test_price_never_falls_with_more_rows():
    bumpy = {1024: {"tree": {8: 10.0, 16: 9.0, 24: 12.0, 32: 11.0}}}
    pr = P.Prices(bumpy)
    assert pr.price(1024, "tree", 16) == 10.0   # the 8-row price carries over the dip
    assert pr.price(1024, "tree", 32) == 12.0
    vals = [pr.price(1024, "tree", r) for r in range(1, 33)]
    assert all(b >= a for a, b in zip(vals, vals[1:]))


def test_online_update_is_an_exponential_average():
    pr = P.Prices(TABLE)
    pr.observe(1024, "tree", 16, 24.0)                 # prior 14: live 14 + 0.1 * 10
    assert math.isclose(pr.current(1024, "tree", 16), 15.0)
    assert math.isclose(pr.current(1024, "tree", 8), 11.0 + 1.0)    # unmeasured counts: + offset 0.1 * 10
    pr.observe(1024, "tree", 16, 24.0)
    assert math.isclose(pr.current(1024, "tree", 16), 15.0 + 0.1 * 9.0)
    assert math.isclose(pr.offset[(1024, "tree")], 1.0 + 0.1 * (10.0 - 1.0))
    assert pr.current(32768, "tree", 16) == 36.0                   # other classes untouched


def test_admission_order_is_ancestor_closed_and_follows_the_score():
    for seed in range(20):
        t = synth.tree_spine_random(20, 5, 100, seed)
        rng = np.random.default_rng(seed)
        score = rng.standard_normal(20)
        order = P.admission_order(t.parent, score)
        assert sorted(order) == list(range(1, 20))
        pos = {v: i for i, v in enumerate(order)}
        for v in order:   # every prefix is a tree: parents come first
            assert t.parent[v] == 0 or pos[t.parent[v]] < pos[v]
        # independently: a node enters when the best-scored node of its subtree
        # is taken, after its own ancestors: sort by (best rank in the subtree, depth)
        rank = {v: i for i, v in enumerate(sorted(range(1, 20), key=lambda i: (-score[i], i)))}
        best = {v: rank[v] for v in range(1, 20)}
        depth = {0: 0}
        for v in range(1, 20):
            depth[v] = depth[t.parent[v]] + 1
        for v in range(19, 0, -1):   # children have larger indices than parents
            if t.parent[v] > 0:
                best[t.parent[v]] = min(best[t.parent[v]], best[v])
        assert order == sorted(range(1, 20), key=lambda v: (best[v], depth[v]))


def test_staircut_by_hand():
    # a chain of 31 nodes with q falling by 0.9 a level; a flat price of 10 ms
    # up to 16 rows and 40 ms beyond: the 15-node cut wins
    n = 32
    parent = np.arange(-1, n - 1)
    q = np.array([1.0] + [0.9 ** d for d in range(1, n)])
    score = -np.arange(n, dtype=float)
    table = {0: {"tree": {1: 10.0, 16: 10.0, 17: 40.0, 32: 40.0}}}
    kept, val = P.staircut(parent, q, score, "tree", P.Prices(table), 0, draft_ms=2.0, commit_ms=1.0)
    assert kept == list(range(1, 16))
    assert math.isclose(val, (1.0 + sum(0.9 ** d for d in range(1, 16))) / 13.0)
    # a candidate smaller than 7 nodes is cut at its whole size
    small = P.staircut(parent[:5], q[:5], score[:5], "tree", P.Prices(table), 0, 2.0, 1.0)
    assert small[0] == [1, 2, 3, 4]
    # a chain pays the rollback weighted by the chance it is rejected
    kept_c, val_c = P.staircut(parent[:8], q[:8], score[:8], "chain",
                               P.Prices({0: {"chain": {1: 10.0, 32: 10.0}}}), 0, 2.0, 1.0, rollback_ms=5.0)
    assert kept_c == list(range(1, 8))
    assert math.isclose(val_c, (1.0 + sum(0.9 ** d for d in range(1, 8))) / (12.0 + (1 - 0.9 ** 7) * 5.0))


def test_staircut_is_the_best_of_its_counts():
    rng = np.random.default_rng(3)
    for seed in range(30):
        t = synth.tree_lattice(32, 15, 100, seed)
        score = rng.standard_normal(32)
        q = rng.uniform(0, 1, 32)
        table = {0: {"tree": {r: float(5 + 0.3 * r + (4 if r > 16 else 0)) for r in (1, 8, 16, 17, 24, 32)}}}
        pr = P.Prices(table)
        kept, val = P.staircut(t.parent, q, score, "tree", pr, 0, 1.5, 0.5)
        order = P.admission_order(t.parent, score)
        best = max((1 + min(sum(q[order[:c]]), c)) / (pr.price(0, "tree", c + 1) + 2.0) for c in (7, 15, 23, 31))
        assert math.isclose(val, best)
        assert kept == order[:len(kept)] and len(kept) in (7, 15, 23, 31)
