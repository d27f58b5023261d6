"""CPU oracle of Gated DeltaNet tree verify and the path-state commit -- TEST
INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference leg may import this module; the CUDA library shares no code with it.

Written from [Drafters and tree verify, §Tree verify through recurrent layers]:
the state after node t of the tree is the state after t's parent, updated by
t; the state before the root is the state before the round, S0; the state
kept after a round is the state after the last node of the accepted path
(for a chain cut back to its first n nodes, the state after node n - 1).

The update is one step of the gated delta rule (Yang, Kautz and Hatamizadeh,
"Gated Delta Networks: Improving Mamba2 with Delta Rule", ICLR 2025), per
value head, with the state S a d_k x d_v matrix (keys to values):

    S_t = exp(g_t) (I - beta_t k_t k_t^T) S_parent + beta_t k_t v_t^T
    o_t = S_t^T q_t

g_t <= 0 is the step's log decay, beta_t in (0, 1) its write strength; q_t
and k_t come from the key head that serves the value head (value head h uses
key head h div (H_v / H_k)).  Inputs are taken as given (projections, the
short convolution, normalisation and scaling happen before this step).

Everything is fp64 and follows the definition node by node; no chunking, no
triangular solve, no reordering.  Pins: ``tests/test_oracle_deltanet.py``.
"""
from __future__ import annotations

from typing import Sequence

import numpy as np


def _key_head(h: int, n_k_heads: int, n_v_heads: int) -> int:
    return h // (n_v_heads // n_k_heads)


def dn_step(S: np.ndarray, q, k, v, beta: float, g: float):
    """One gated delta-rule step from state S: returns (S_new, o)."""
    S = np.asarray(S, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    q = np.asarray(q, np.float64)
    S_new = np.exp(g) * (S - beta * np.outer(k, k @ S)) + beta * np.outer(k, v)
    return S_new, S_new.T @ q


def dn_tree_states(parent: Sequence[int], q, k, v, beta, g, S0):
    """One value head over a tree.  q, k: [n][d_k]; v: [n][d_v]; beta, g: [n];
    S0: [d_k][d_v].  Returns (states [n][d_k][d_v], outputs [n][d_v]): the
    state after each node and its output."""
    n = len(parent)
    S0 = np.asarray(S0, np.float64)
    states = np.zeros((n,) + S0.shape)
    outs = np.zeros((n, S0.shape[1]))
    for t in range(n):
        before = S0 if parent[t] < 0 else states[parent[t]]
        states[t], outs[t] = dn_step(before, q[t], k[t], v[t], float(beta[t]), float(g[t]))
    return states, outs


def dn_verify_tree(parent, q, k, v, beta, g, S0):
    """All value heads.  q, k: [n][H_k][d_k]; v: [n][H_v][d_v]; beta, g:
    [n][H_v]; S0: [H_v][d_k][d_v].  Returns {"o": [n][H_v][d_v], "states":
    [n][H_v][d_k][d_v]}."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    n, Hk, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    o = np.zeros((n, Hv, dv))
    states = np.zeros((n, Hv, dk, dv))
    for h in range(Hv):
        kh = _key_head(h, Hk, Hv)
        st, oh = dn_tree_states(parent, q[:, kh], k[:, kh], v[:, h], np.asarray(beta)[:, h], np.asarray(g)[:, h],
                                np.asarray(S0)[h])
        states[:, h] = st
        o[:, h] = oh
    return {"o": o, "states": states}


def dn_commit(S0, states, path: Sequence[int]) -> np.ndarray:
    """The state kept after the round: the state after the last node of the
    accepted root path (path[0] is the root).  An empty path keeps S0."""
    if len(path) == 0:
        return np.asarray(S0, np.float64).copy()
    return np.asarray(states[path[-1]], np.float64).copy()
