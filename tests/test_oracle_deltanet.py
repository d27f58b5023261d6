"""Pins of oracle/deltanet.py (the gated delta rule walked node by node) to
what the pages and the mathematics fix, independently of the oracle's own
recurrence:

* the pages' closed form of the state after any root path [Drafters and tree
  verify, §Tree verify through recurrent layers], built here from an
  ancestor-masked triangular solve (scipy), for every node's path;
* special cases: no writes (beta = 0) is pure decay; with g = 0, beta = 1 and
  orthonormal keys the delta rule stores each value exactly (read-back by its
  key returns it, keys orthogonal to all writes read the old state);
* a node's state depends only on its root path (siblings and other branches
  change nothing), and relabelling a tree keeps every node's state;
* one step by hand on 2 x 2 numbers;
* the grouping of value heads onto key heads.
"""
import numpy as np
import pytest
import scipy.linalg

from oracle import deltanet as DN
from speculative_tree_verify_gb300 import synth


def _inputs(n, dk, dv, seed, Hk=1, Hv=1):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((n, Hk, dk))
    q /= np.linalg.norm(q, axis=2, keepdims=True) * np.sqrt(dk)
    k = rng.standard_normal((n, Hk, dk))
    k /= np.linalg.norm(k, axis=2, keepdims=True)
    v = rng.standard_normal((n, Hv, dv))
    beta = rng.uniform(0.05, 0.95, (n, Hv))
    g = -rng.uniform(0.001, 0.4, (n, Hv))
    S0 = rng.standard_normal((Hv, dk, dv)) * 0.3
    return q, k, v, beta, g, S0


def _path(parent, t):
    p = []
    while t >= 0:
        p.append(t)
        t = parent[t]
    return p[::-1]


@pytest.mark.parametrize("shape", ["chain", "lattice", "star", "random"])
def test_state_after_any_path_is_the_pages_closed_form(shape):
    n, dk, dv = 12, 8, 6
    tree = {"chain": synth.tree_chain(n, 100, 1), "lattice": synth.tree_lattice(n, 5, 100, 2),
            "star": synth.tree_star(n, 100, 3), "random": synth.tree_spine_random(n, 3, 100, 4)}[shape]
    parent = tree.parent
    q, k, v, beta, g, S0 = _inputs(n, dk, dv, 10)
    res = DN.dn_verify_tree(parent, q, k, v, beta, g, S0)
    K, Q, Vv, B, G, S = k[:, 0], q[:, 0], v[:, 0], beta[:, 0], g[:, 0], S0[0]
    # cumulative gate along each node's path
    gc = np.zeros(n)
    for t in range(n):
        gc[t] = G[t] + (gc[parent[t]] if parent[t] >= 0 else 0.0)
    # pseudo-values: (I + A) U = diag(beta) (V - diag(exp gc) K S0), A ancestor-masked
    A = np.zeros((n, n))
    for t in range(n):
        for s in _path(parent, t)[:-1]:
            A[t, s] = B[t] * np.exp(gc[t] - gc[s]) * (K[t] @ K[s])
    rhs = B[:, None] * (Vv - np.exp(gc)[:, None] * (K @ S))
    U = scipy.linalg.solve_triangular(np.eye(n) + A, rhs, lower=True)
    for t in range(n):
        p = _path(parent, t)
        S_path = np.exp(gc[t]) * S + sum(np.exp(gc[t] - gc[s]) * np.outer(K[s], U[s]) for s in p)
        np.testing.assert_allclose(res["states"][t, 0], S_path, rtol=1e-11, atol=1e-12)
        o = np.exp(gc[t]) * (S.T @ Q[t]) + sum(np.exp(gc[t] - gc[s]) * (Q[t] @ K[s]) * U[s] for s in p)
        np.testing.assert_allclose(res["o"][t, 0], o, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(DN.dn_commit(S0[0], res["states"][:, 0], p), S_path, rtol=1e-11, atol=1e-12)


def test_no_writes_is_pure_decay():
    n, dk, dv = 9, 5, 4
    tree = synth.tree_spine_random(n, 4, 50, 7)
    q, k, v, beta, g, S0 = _inputs(n, dk, dv, 11)
    res = DN.dn_verify_tree(tree.parent, q, k, v, np.zeros_like(beta), g, S0)
    for t in range(n):
        gsum = sum(g[s, 0] for s in _path(tree.parent, t))
        np.testing.assert_allclose(res["states"][t, 0], np.exp(gsum) * S0[0], rtol=1e-13)
        np.testing.assert_allclose(res["o"][t, 0], np.exp(gsum) * S0[0].T @ q[t, 0], rtol=1e-12, atol=1e-15)


def test_unit_writes_with_orthonormal_keys_store_each_value():
    dk, dv, n = 8, 3, 5
    rng = np.random.default_rng(5)
    basis, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    k = basis[:, :n].T[:, None, :]             # n orthonormal keys
    v = rng.standard_normal((n, 1, dv))
    q = k.copy()
    S0 = rng.standard_normal((1, dk, dv))
    parent = np.arange(-1, n - 1)
    res = DN.dn_verify_tree(parent, q, k, v, np.ones((n, 1)), np.zeros((n, 1)), S0)
    S_last = res["states"][n - 1, 0]
    for j in range(n):
        np.testing.assert_allclose(S_last.T @ k[j, 0], v[j, 0], atol=1e-12)   # each write reads back
    for j in range(n, dk):
        np.testing.assert_allclose(S_last.T @ basis[:, j], S0[0].T @ basis[:, j], atol=1e-12)   # the rest is kept
    np.testing.assert_allclose(res["o"][:, 0], v[:, 0], atol=1e-12)   # q = k: each step reads its own value


def test_a_node_depends_only_on_its_path_and_labels_do_not_matter():
    n, dk, dv = 10, 6, 5
    tree = synth.tree_lattice(n, 4, 60, 9)
    q, k, v, beta, g, S0 = _inputs(n, dk, dv, 12)
    res = DN.dn_verify_tree(tree.parent, q, k, v, beta, g, S0)
    for t in range(n):
        p = _path(tree.parent, t)
        chain = DN.dn_verify_tree(np.arange(-1, len(p) - 1), q[p], k[p], v[p], beta[p], g[p], S0)
        assert np.array_equal(chain["states"][-1], res["states"][t])
        assert np.array_equal(chain["o"][-1], res["o"][t])
    # relabel: children of the root in reverse order (parents still before children)
    order = [0] + [c for c in range(n - 1, 0, -1) if tree.parent[c] == 0]
    rest = [c for c in range(1, n) if c not in order]
    while rest:
        c = next(c for c in rest if tree.parent[c] in order)
        order.append(c)
        rest.remove(c)
    new_index = {old: i for i, old in enumerate(order)}
    parent2 = np.array([-1] + [new_index[tree.parent[old]] for old in order[1:]])
    res2 = DN.dn_verify_tree(parent2, q[order], k[order], v[order], beta[order], g[order], S0)
    for old, new in new_index.items():
        assert np.array_equal(res2["states"][new], res["states"][old])


def test_one_step_by_hand():
    S0 = np.array([[[1.0, 2.0], [3.0, 4.0]]])
    k = np.array([[[0.6, 0.8]]])
    q = np.array([[[1.0, -1.0]]])
    v = np.array([[[0.5, -2.0]]])
    beta, g = np.array([[0.5]]), np.array([[np.log(0.5)]])
    res = DN.dn_verify_tree([-1], q, k, v, beta, g, S0)
    # k^T S0 = [3.0, 4.4]; S0 - 0.5 k (k^T S0) = [[0.1, 0.68], [1.8, 2.24]]
    # times 0.5 = [[0.05, 0.34], [0.9, 1.12]]; + 0.5 k v^T = [[0.15, -0.6], [0.2, -0.8]]
    want = np.array([[0.2, -0.26], [1.1, 0.32]])
    np.testing.assert_allclose(res["states"][0, 0], want, atol=1e-14)
    np.testing.assert_allclose(res["o"][0, 0], want.T @ np.array([1.0, -1.0]), atol=1e-14)


def test_value_heads_share_key_heads_in_groups():
    n, dk, dv, Hk, Hv = 4, 4, 3, 2, 4
    q, k, v, beta, g, S0 = _inputs(n, dk, dv, 13, Hk=Hk, Hv=Hv)
    parent = np.arange(-1, n - 1)
    base = DN.dn_verify_tree(parent, q, k, v, beta, g, S0)
    k2 = k.copy()
    k2[:, 1] = np.roll(k2[:, 1], 1, axis=1)   # change key head 1 only
    moved = DN.dn_verify_tree(parent, q, k2, v, beta, g, S0)
    for h in range(Hv):
        same = np.array_equal(base["o"][:, h], moved["o"][:, h])
        assert same == (h < Hv // Hk), h      # value heads 0, 1 read key head 0; 2, 3 read key head 1


def test_commit_of_an_empty_path_keeps_the_state():
    S0 = np.arange(6.0).reshape(2, 3)
    assert np.array_equal(DN.dn_commit(S0, np.zeros((0, 2, 3)), []), S0)
