"""Pins of the oracle's accept walks, commit and input validation (CPU only).

* greedy walk: hand-derived cases of the rule in [Drafters and tree verify,
  §The round, step 3], and a brute-force enumeration of root paths;
* residual walk: the page's printed grid counts (2500/10000 and
  [2000, 500, 3000, 4500]) [Algorithm and correctness contract, §Evidence],
  and a Monte Carlo check that the walk reproduces p on a 16-token vocabulary,
  token after token;
* softmax against scipy;
* commit against the sequential decoder's K/V rows of the accepted path;
* validation against the rejections the pages list.
"""
import itertools
import json
import os

import numpy as np
import pytest
import scipy.special

import oracle
from speculative_tree_verify_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# greedy
# --------------------------------------------------------------------------
def test_greedy_hand_cases():
    # root 0 has children 1 (tok 5) and 2 (tok 7); node 1 has child 3 (tok 9).
    parent = [-1, 0, 0, 1]
    token = [100, 5, 7, 9]
    # row 0 picks 5 -> node 1; row 1 picks 9 -> node 3; row 3 picks 2: no child
    assert oracle.accept_greedy(parent, token, [5, 9, 4, 2]) == ([0, 1, 3], [5, 9, 2])
    # row 0 picks 7 -> node 2 (a leaf); its token 11 is kept
    assert oracle.accept_greedy(parent, token, [7, 0, 11, 0]) == ([0, 2], [7, 11])
    # row 0 picks a token no child carries: only the model's token comes out
    assert oracle.accept_greedy(parent, token, [8, 9, 4, 2]) == ([0], [8])


def _root_paths(parent):
    n = len(parent)
    paths = []
    for i in range(n):
        p, a = [], i
        while a >= 0:
            p.append(a)
            a = int(parent[a])
        paths.append(p[::-1])
    return paths


@pytest.mark.parametrize("seed", range(20))
def test_greedy_is_longest_matching_root_path(seed):
    rng = np.random.default_rng(seed)
    V = 6   # small vocabulary so that many drafts match
    n = int(rng.integers(1, 33))
    tree = synth.tree_spine_random(n, int(rng.integers(1, min(9, n) + 1)), V, seed)
    tree = synth.tree_star(tree.n, V, seed) if tree.n <= V and seed % 3 == 0 else tree
    argmax = rng.integers(0, V, size=tree.n)
    path, out = oracle.accept_greedy(tree.parent, tree.token, argmax)
    # brute force: among all root paths, those whose every step carries the
    # parent's argmax; the accepted one is the longest (unique: siblings differ)
    ok = [p for p in _root_paths(tree.parent)
          if all(int(tree.token[p[d]]) == int(argmax[p[d - 1]]) for d in range(1, len(p)))]
    best = max(ok, key=len)
    assert sum(len(p) == len(best) for p in ok) == 1
    assert path == best
    assert out == [int(tree.token[c]) for c in best[1:]] + [int(argmax[best[-1]])]
    last = best[-1]
    assert not any(int(tree.parent[c]) == last and int(tree.token[c]) == int(argmax[last])
                   for c in range(1, tree.n))


# --------------------------------------------------------------------------
# residual walk: the page's grid counts
# --------------------------------------------------------------------------
def _grid(k):
    return [(i + 0.5) / k for i in range(k)]


def test_grid_single_path():
    g = json.load(open(os.path.join(GOLDEN, "residual_grid_counts.json")))["single_path"]
    p = g["p_accept"]
    logits = np.log(np.array([[p, 1 - p], [0.5, 0.5]]))   # token 0 drafted at node 1
    parent, token = [-1, 0], [1, 0]
    acc = 0
    for u in _grid(g["grid_points"]):
        path, out, _ = oracle.accept_residual(parent, token, logits, 1.0, [u, 0.5])
        acc += len(path) == 2
    assert acc == g["accepted"]


def test_grid_two_level():
    g = json.load(open(os.path.join(GOLDEN, "residual_grid_counts.json")))["two_level"]
    rec = g["reconstruction"]
    # two-token vocabulary {A=0, B=1}; root offers A then B; each of them offers
    # A then B again.  Node order: 0 root, 1 A, 2 A.A, 3 A.B, 4 B, 5 B.A, 6 B.B
    parent = [-1, 0, 1, 1, 0, 4, 4]
    token = [0, 0, 0, 1, 1, 0, 1]
    rows = {0: rec["p_root"], 1: rec["p_after_A"], 4: rec["p_after_B"],
            2: [0.5, 0.5], 3: [0.5, 0.5], 5: [0.5, 0.5], 6: [0.5, 0.5]}
    logits = np.log(np.array([rows[i] for i in range(7)]))
    k = 100                                   # 100 x 100 grid of the draws that decide
    counts = {"AA": 0, "AB": 0, "BA": 0, "BB": 0}
    for u1, u2, u3 in itertools.product(_grid(k), _grid(k), [0.5]):
        # draw stream: test A at the root (u1); if rejected, B's test (always
        # accepted: r(B) = 1 after removing A, u3 = 0.5); then the first test at
        # the second level (u2); then whatever else follows.
        path, out, _ = oracle.accept_residual(parent, token, logits, 1.0,
                                              [u1, u2, 0.5, 0.5, 0.5] if u1 < rec["p_root"][0]
                                              else [u1, u3, u2, 0.5, 0.5])
        counts["AB"[out[0]] + "AB"[out[1]]] += 1
    total = k * k
    want = g["joint_counts_first_second"]
    scale = g["grid_points_per_level"] / total
    assert [counts[o] * scale for o in g["order"]] == want


def test_grid_residual_draw_counts():
    # a leaf row drawn by inverse CDF on a grid: exact p * grid counts
    p = np.array([0.1, 0.2, 0.3, 0.4])
    counts = np.zeros(4, int)
    for u in _grid(10000):
        _, out, _ = oracle.accept_residual([-1], [0], np.log(p)[None], 1.0, [u])
        counts[out[0]] += 1
    np.testing.assert_array_equal(counts, [1000, 2000, 3000, 4000])


def test_all_candidates_rejected_draws_from_residual():
    # every candidate of the root fails: the draw comes from p with them removed
    p = np.array([0.4, 0.3, 0.2, 0.1])
    parent, token = [-1, 0, 0], [0, 0, 1]
    counts = np.zeros(4, int)
    k = 1000
    for u in _grid(k):
        # u1 = 0.99 rejects token 0 (r=0.4); u2 = 0.99 rejects token 1 (r=0.5)
        path, out, _ = oracle.accept_residual(parent, token, np.log(p)[None].repeat(3, 0), 1.0, [0.99, 0.99, u])
        assert path == [0] and len(out) == 1
        counts[out[0]] += 1
    np.testing.assert_array_equal(counts, [0, 0, 667, 333])   # (i + 0.5) / 1000 < 2/3 for i <= 666


def test_leaf_without_bonus_ends_round():
    p = np.array([0.7, 0.3])
    path, out, _ = oracle.accept_residual([-1, 0], [1, 0], np.log(p)[None].repeat(2, 0), 1.0, [0.1, 0.5],
                                          bonus_at_leaf=False)
    assert path == [0, 1] and out == [0]


# --------------------------------------------------------------------------
# residual walk: Monte Carlo law on a 16-token vocabulary
# --------------------------------------------------------------------------
@pytest.mark.slow
def test_residual_walk_reproduces_p_monte_carlo():
    rng = np.random.default_rng(12345)
    V = 16
    # a three-level tree with distinct, random candidates per node
    parent = [-1]
    token = [0]

    def add_children(node, k, depth):
        toks = rng.choice(V, size=k, replace=False)
        ids = []
        for t in toks:
            parent.append(node)
            token.append(int(t))
            ids.append(len(parent) - 1)
        if depth > 1:
            for c in ids[:2]:
                add_children(c, 3, depth - 1)

    add_children(0, 4, 3)
    n = len(parent)
    assert n <= 32
    logits = (rng.standard_normal((n, V)) * 1.2).astype(np.float32)
    T = 0.8
    P = np.array([oracle.softmax_t(logits[i], T) for i in range(n)])
    kids = {i: {int(token[c]): c for c in range(1, n) if parent[c] == i} for i in range(n)}

    rounds = 200000
    us = rng.random((rounds, n)).astype(np.float32)
    first = np.zeros(V)
    pair = np.zeros((V, V))
    pair_seen = np.zeros(V)
    for r in range(rounds):
        path, out, _ = oracle.accept_residual(parent, token, logits, T, us[r])
        first[out[0]] += 1
        node = kids[0].get(out[0])
        if node is not None:           # a candidate was accepted: the next token scores at its row
            pair_seen[out[0]] += 1
            pair[out[0], out[1]] += 1

    def within(counts, total, probs, sig=5.0):
        sd = np.sqrt(total * probs * (1 - probs)) + 1e-9
        return np.all(np.abs(counts - total * probs) <= sig * sd + 1.0)

    assert within(first, rounds, P[0])
    for x, c in kids[0].items():
        tot = pair_seen[x]
        assert tot == first[x]                  # a candidate token only ever comes from acceptance
        assert within(pair[x], tot, P[c])


def test_softmax_matches_scipy():
    rng = np.random.default_rng(5)
    z = (rng.standard_normal(1000) * 4).astype(np.float32)
    for T in (1.0, 0.7, 2.5):
        np.testing.assert_allclose(oracle.softmax_t(z, T), scipy.special.softmax(z.astype(np.float64) / T),
                                   rtol=1e-12, atol=1e-300)
        assert abs(oracle.softmax_t(z, T).sum() - 1.0) < 1e-12


# --------------------------------------------------------------------------
# commit
# --------------------------------------------------------------------------
def test_commit_equals_sequential_decode_of_path():
    d = synth.TINY
    model = synth.gen_model(d, 31, random_gains=True)
    ctx = 40
    cache = synth.gen_cache(d, ctx, 80, 32)
    tree = synth.tree_lattice(16, 7, d.vocab, 33)
    ver = oracle.verify_tree(model, cache, tree)
    k, v = oracle.apply_tree_kv(cache, ver["k"], ver["v"])
    # a path that jumps over siblings: root -> a later child -> its child
    kids = [[c for c in range(1, tree.n) if tree.parent[c] == i] for i in range(tree.n)]
    path = [0, kids[0][-1]]
    if kids[path[-1]]:
        path.append(kids[path[-1]][0])
    k2, v2, src, new_ctx = oracle.commit_kv(k, v, ctx, path)
    assert src == [ctx + p for p in path] and new_ctx == ctx + len(path)
    dec = oracle.decode_sequence(model, cache, [int(tree.token[a]) for a in path])
    Hkv, D = d.n_kv_heads, d.head_dim
    for t in range(len(path)):
        np.testing.assert_array_equal(k2[:, ctx + t, :], dec["k"][t].reshape(Hkv, D))
        np.testing.assert_array_equal(v2[:, ctx + t, :], dec["v"][t].reshape(Hkv, D))
    np.testing.assert_array_equal(k2[:, :ctx], cache.k[:, :ctx])


def test_commit_reads_before_writing():
    # path [0, 2, 3]: slot ctx+2 is both the source of step 1 and the target of step 2
    k = np.arange(1 * 8 * 2, dtype=np.uint16).reshape(1, 8, 2)
    v = k + 100
    k2, v2, src, new_ctx = oracle.commit_kv(k, v, 2, [0, 2, 3])
    assert src == [2, 4, 5] and new_ctx == 5
    np.testing.assert_array_equal(k2[0, 2:5], k[0, [2, 4, 5]])
    np.testing.assert_array_equal(v2[0, 2:5], v[0, [2, 4, 5]])


# --------------------------------------------------------------------------
# validation
# --------------------------------------------------------------------------
def test_validation_rejections():
    V = 50
    assert oracle.validate([-1, 0, 1], [1, 2, 3], V) == "ok"
    assert oracle.validate([], [], V) == "rows"
    assert oracle.validate([-1] + [0] * 32, list(range(33)), V) == "rows"
    assert oracle.validate([0, 0], [1, 2], V) == "order"
    assert oracle.validate([-1, 1], [1, 2], V) == "order"         # parent not before child
    assert oracle.validate([-1, 0, 3, 0], [1, 2, 3, 4], V) == "order"
    assert oracle.validate([-1, 0], [1, V], V) == "token"
    assert oracle.validate([-1, 0], [-1, 2], V) == "token"
    assert oracle.validate([-1, 0, 0], [1, 7, 7], V) == "dup_sibling"
    assert oracle.validate([-1, 0, 1], [1, 7, 7], V) == "ok"       # same token, not siblings
    assert oracle.validate([-1, 0, 0], [1, 2, 3], V, ctx=10, capacity=12) == "capacity"
    assert oracle.validate([-1, 0, 0], [1, 2, 3], V, ctx=10, capacity=13) == "ok"
    assert oracle.validate_sampling([0.0, 0.5, 0.999], 1.0) == "ok"
    assert oracle.validate_sampling([1.0], 1.0) == "uniform"
    assert oracle.validate_sampling([-0.1], 1.0) == "uniform"
    assert oracle.validate_sampling([float("nan")], 1.0) == "uniform"
    assert oracle.validate_sampling([0.5], 0.0) == "temp"
    assert oracle.validate_sampling([0.5], float("nan")) == "temp"
