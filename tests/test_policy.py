"""The library's verify prices and StairCut cut (host code behind the C ABI)
against oracle/policy.py: the same doubles, the same kept nodes."""
import json
import math

import numpy as np
import pytest

from oracle import policy as P
from speculative_tree_verify_gb300 import abi, build, prices, synth


@pytest.fixture(scope="module")
def lib():
    build.build()
    return abi.load()


def _random_table(rng):
    classes = sorted(rng.choice([512, 1024, 2048, 4096, 8192, 16384, 32768, 65536], rng.integers(1, 6), replace=False))
    tab = {}
    for c in classes:
        kinds = {}
        for kind in ("chain", "tree"):
            if rng.random() < 0.15:
                continue
            rows = sorted(rng.choice(np.arange(1, 33), rng.integers(1, 8), replace=False))
            ms = np.cumsum(rng.uniform(-0.5, 3.0, len(rows))) + 5.0   # sometimes falling
            kinds[kind] = {int(r): float(v) for r, v in zip(rows, ms)}
        tab[int(c)] = kinds
    return tab, float(rng.choice([0.0, 0.0, 0.7]))


def _native(tab, step):
    obj = {str(c): {k: {str(r): v for r, v in rows.items()} for k, rows in kinds.items()} for c, kinds in tab.items()}
    obj["step_ms"] = step
    return prices.table_from_json(obj)


def test_prices_match_the_oracle(lib):
    rng = np.random.default_rng(0)
    for trial in range(200):
        tab, step = _random_table(rng)
        nat, orc = _native(tab, step), P.Prices(tab, step)
        for _ in range(40):
            ctx = int(rng.integers(0, 80000))
            kind = "chain" if rng.random() < 0.5 else "tree"
            rows = int(rng.integers(1, 33))
            rc, ms = abi.tv_price_lookup(nat, ctx, prices.KINDS[kind], rows)
            assert rc == abi.TV_OK
            assert ms == orc.price(ctx, kind, rows), (trial, ctx, kind, rows)
        for _ in range(10):   # observations, then lookups again
            ctx, kind, rows = int(rng.integers(0, 80000)), ("chain", "tree")[int(rng.integers(0, 2))], int(
                rng.integers(1, 33))
            ms = float(rng.uniform(1, 60))
            assert abi.tv_price_observe(nat, ctx, prices.KINDS[kind], rows, ms) == abi.TV_OK
            orc.observe(ctx, kind, rows, ms)
            for r in range(1, 33):
                assert abi.tv_price_lookup(nat, ctx, prices.KINDS[kind], r)[1] == orc.price(ctx, kind, r)


def test_staircut_matches_the_oracle(lib):
    rng = np.random.default_rng(1)
    for trial in range(300):
        n = int(rng.integers(1, 33))
        shape = trial % 3
        t = (synth.tree_lattice(n, 15, 100, trial) if shape == 0 else synth.tree_chain(n, 100, trial) if shape == 1
             else synth.tree_spine_random(n, max(1, n // 3), 100, trial))
        q = rng.uniform(0, 1.2, n).astype(np.float32)
        score = np.round(rng.standard_normal(n), 1).astype(np.float32)   # some ties
        tab, step = _random_table(rng)
        kind = "chain" if shape == 1 and rng.random() < 0.5 else "tree"
        if kind not in next(iter(tab.values())):
            tab[next(iter(tab))][kind] = {8: 9.0, 16: 10.0}
        ctx = int(rng.integers(0, 80000))
        draft, commit, rollback = float(rng.uniform(0, 5)), float(rng.uniform(0, 2)), float(rng.uniform(0, 5))
        rc, kept, val = abi.tv_staircut(t.parent, q, score, prices.KINDS[kind], _native(tab, step), ctx, draft,
                                        commit, rollback)
        assert rc == abi.TV_OK
        okept, oval = P.staircut(t.parent, q.astype(np.float64), score.astype(np.float64), kind, P.Prices(tab, step),
                                 ctx, draft, commit, rollback)
        assert kept == okept and val == oval, trial


def test_policy_rejects_bad_inputs(lib):
    t = abi.TvPriceTable()
    assert abi.tv_price_init(t) == abi.TV_OK
    assert abi.tv_price_lookup(t, 1024, 1, 8)[0] == abi.CODES["TV_E_ARG"]         # no classes
    t = _native({1024: {"tree": {8: 10.0}}}, 0.0)
    assert abi.tv_price_lookup(t, 1024, 2, 8)[0] == abi.CODES["TV_E_ARG"]         # kind
    assert abi.tv_price_lookup(t, 1024, 1, 33)[0] == abi.CODES["TV_E_ROWS"]
    assert abi.tv_price_observe(t, 1024, 1, 8, float("nan")) == abi.CODES["TV_E_ARG"]
    bad = np.array([-1, 0, 2], np.int32)
    assert abi.tv_staircut(bad, np.ones(3), np.ones(3), 1, t, 0, 1.0, 1.0)[0] == abi.CODES["TV_E_ORDER"]
    assert abi.tv_staircut(np.arange(-1, 32), np.ones(33), np.ones(33), 1, t, 0, 1.0, 1.0)[0] == abi.CODES["TV_E_ROWS"]
    unsorted = _native({1024: {"tree": {8: 1.0}}}, 0.0)
    unsorted.n_classes = 2
    unsorted.class_ctx[1] = 512
    assert abi.tv_price_lookup(unsorted, 1024, 1, 8)[0] == abi.CODES["TV_E_ARG"]


def test_price_file_round_trip(lib):
    tab = {1024: {"chain": {8: 10.5, 16: 12.25}, "tree": {8: 11.0, 32: 20.0}}, 32768: {"tree": {16: 40.0}}}
    obj = {str(c): {k: {str(r): v for r, v in rows.items()} for k, rows in kinds.items()} for c, kinds in tab.items()}
    obj["step_ms"] = 0.5
    t = prices.table_from_json(json.loads(json.dumps(obj)))
    back = prices.table_to_json(t)
    assert back == obj
