"""CPU oracle of the sampled accept variants -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference leg may import this module; the CUDA library shares no code with it.

Written from the pages' statement of each method, in fp64 unless stated:

* ``sample_filter`` -- temperature, top_k, top_p and min_p applied through one
  function to a row of logits [Exactness, §Sampling, second paragraph].
* ``accept_single_draw`` -- the single-draw form of sampled tree verify: at each
  node the target draws its own token; a drafted child survives while the draw
  lands on it, otherwise the draw is the token [Exactness, §Sampling, first
  paragraph; Drafters and tree verify, §Sampling].
* ``philox4x32_10`` / ``gumbel_uniform`` / ``gumbel_draw`` / ``accept_gumbel``
  -- seeded sampling: the token at sequence index t is the argmax of
  log p_t + G_t, G_t Gumbel noise from a generator keyed by (seed, t)
  [Exactness, §Sampling, third paragraph].  The generator is Philox4x32-10
  (Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as easy as 1, 2,
  3", SC 2011), written here from that paper's definition.
* ``accept_rejection_chain`` -- the single-path rejection sampler: accept a
  draft x with probability min(1, p(x)/q(x)); on rejection draw from
  normalize(max(p - q, 0)) and stop; no extra token after a fully accepted
  path [Algorithm and correctness contract, §Single-path sampling].

Pins: ``tests/test_oracle_sampling.py`` (Philox known-answer vectors, exact
grid laws, Monte Carlo laws against p, sort-based definitions of the filters).
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

from . import _children, inverse_cdf

# ---------------------------------------------------------------------------
# filters
# ---------------------------------------------------------------------------


def sample_filter(logits_row, temperature: float, top_k: int = 0, top_p: float = 1.0,
                  min_p: float = 0.0) -> np.ndarray:
    """Scaled logits x = l / T with every token a filter removes set to -inf,
    so that softmax(x) is the filtered, renormalised distribution.

    Readings (the pages name the filters and their single function, not their
    order or ties):
      * order: temperature, then top_k, then top_p, then min_p; each filter
        sees the distribution renormalised over the tokens the previous ones
        kept;
      * top_k (0 = off): keep the tokens whose x is at least the k-th largest x;
        tokens tied with it are all kept;
      * top_p (1 = off): keep the fewest largest-probability tokens whose mass
        reaches top_p, i.e. every token whose probability is at least the
        probability of the token at which the running mass (largest first)
        first reaches top_p; ties with it are all kept;
      * min_p (0 = off): keep the tokens with p >= min_p * max p.
    """
    x = np.asarray(logits_row, np.float64) / float(temperature)
    keep = np.isfinite(x)
    if top_k and top_k > 0 and top_k < int(keep.sum()):
        kth = np.sort(x[keep])[::-1][top_k - 1]
        keep &= x >= kth
    if top_p < 1.0:
        z = np.where(keep, x - x[keep].max(), -np.inf)
        p = np.exp(z)
        p = p / p.sum()
        order = np.argsort(-p, kind="stable")
        c = np.cumsum(p[order])
        cut = int(np.searchsorted(c, top_p, side="left"))
        cut = min(cut, order.shape[0] - 1)
        keep &= p >= p[order[cut]]
    if min_p > 0.0:
        xm = x[keep].max()
        keep &= x >= xm + np.log(min_p)
    return np.where(keep, x, -np.inf)


def softmax_x(x) -> np.ndarray:
    """softmax of already-scaled logits (-inf entries get 0)."""
    x = np.asarray(x, np.float64)
    z = x - x[np.isfinite(x)].max()
    e = np.exp(z)
    return e / e.sum()


# ---------------------------------------------------------------------------
# single-draw walk
# ---------------------------------------------------------------------------


def accept_single_draw(parent, token, rows_x, uniforms, replay=None, eps: float = 0.0):
    """Single-draw sampled tree verify.  At node cur the target draws y from
    p = softmax(rows_x[cur]) by the inverse CDF with uniform ``uniforms[cur]``
    (one uniform per tree row; each visited row is drawn once).  If a child of
    cur carries y the walk moves there; otherwise y is the round's last token.
    At a leaf the draw is the last token.

    Returns (path, out_tokens, n_replayed).  ``replay`` = (path, out_tokens)
    of another implementation: where the scaled uniform lies within ``eps`` of a
    CDF boundary, its choice is taken if it is one of the boundary's two sides.
    """
    kids = _children(parent)
    path, out, cur, replayed = [0], [], 0, 0
    while True:
        p = softmax_x(rows_x[cur])
        u = float(uniforms[cur])
        y = inverse_cdf(p, u)
        if replay is not None and len(replay[1]) > len(out):
            yg = int(replay[1][len(out)])
            if yg != y and p[yg] > 0:
                c = np.cumsum(p)
                lo = c[yg - 1] if yg > 0 else 0.0
                t = u * c[-1]
                if lo - eps * c[-1] <= t < c[yg] + eps * c[-1]:
                    y = yg
                    replayed += 1
        nxt = next((c for c in kids[cur] if int(token[c]) == y), None)
        if nxt is None:
            out.append(y)
            return path, out, replayed
        path.append(nxt)
        out.append(y)
        cur = nxt


# ---------------------------------------------------------------------------
# seeded Gumbel-max
# ---------------------------------------------------------------------------
_M0, _M1 = 0xD2511F53, 0xCD9E8D57          # Philox4x32 round multipliers
_W0, _W1 = 0x9E3779B9, 0xBB67AE85          # Weyl key increments
_MASK = 0xFFFFFFFF


def philox4x32_10(ctr, key):
    """Philox4x32 with 10 rounds.  ``ctr`` = four uint32 words (scalars or
    equal-shape arrays), ``key`` = two uint32 words.  Each round:
      (hi0, lo0) = M0 * c0,  (hi1, lo1) = M1 * c2,
      c = (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0),
    and the key is bumped by (W0, W1) between rounds."""
    c0, c1, c2, c3 = (np.asarray(v, np.uint64) & _MASK for v in ctr)
    k0 = np.uint64(int(key[0]) & _MASK)
    k1 = np.uint64(int(key[1]) & _MASK)
    m0, m1 = np.uint64(_M0), np.uint64(_M1)
    mask = np.uint64(_MASK)
    for rnd in range(10):
        if rnd > 0:
            k0 = (k0 + np.uint64(_W0)) & mask
            k1 = (k1 + np.uint64(_W1)) & mask
        p0 = m0 * c0
        p1 = m1 * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & mask
        hi1, lo1 = p1 >> np.uint64(32), p1 & mask
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return c0, c1, c2, c3


def gumbel_uniform(seed: int, t: int, idx) -> np.ndarray:
    """U in (0, 1) for token ``idx`` at sequence index ``t``: word ``idx mod 4``
    of Philox4x32-10 at counter (idx div 4, t, 0, 0) under key (seed low,
    seed high), as (w + 0.5) / 2^32.  One generator block serves four
    consecutive tokens (the pages fix only that the noise is keyed by
    (seed, t); the layout of the generator's output is this reading)."""
    idx = np.asarray(idx, np.uint64)
    blk = idx >> np.uint64(2)
    words = philox4x32_10((blk, np.full_like(blk, int(t) & _MASK), np.zeros_like(blk), np.zeros_like(blk)),
                          (int(seed) & _MASK, (int(seed) >> 32) & _MASK))
    sel = (idx & np.uint64(3)).astype(np.int64)
    w = np.choose(sel, words)
    return (w.astype(np.float64) + 0.5) / 4294967296.0


def gumbel_scores(x, seed: int, t: int) -> np.ndarray:
    """x_i + G_i with G_i = -log(-log U_i); removed tokens (-inf) stay -inf."""
    x = np.asarray(x, np.float64)
    u = gumbel_uniform(seed, t, np.arange(x.shape[0]))
    return x - np.log(-np.log(u))


def gumbel_draw(x, seed: int, t: int) -> int:
    """The token at sequence index t: argmax of log p_t + G_t (log p and x differ
    by a constant), lowest index on ties."""
    return int(np.argmax(gumbel_scores(x, seed, t)))


def accept_gumbel(parent, token, rows_x, seed: int, ctx: int, choose=None):
    """Seeded sampled tree verify.  Row i holds node i at position ctx + depth(i)
    and scores the token at sequence index ctx + depth(i) + 1; that token is
    ``gumbel_draw(rows_x[i], seed, ctx + depth(i) + 1)``, whatever the tree.
    The walk moves to the child carrying the draw and stops where none does;
    the draw at the stopping node is the round's last token.  ``choose(i)``,
    when given, replaces row i's draw (near-tie replay)."""
    n = len(parent)
    depth = [0] * n
    for i in range(1, n):
        depth[i] = depth[int(parent[i])] + 1
    kids = _children(parent)
    path, out, cur = [0], [], 0
    while True:
        y = gumbel_draw(rows_x[cur], seed, ctx + depth[cur] + 1) if choose is None else int(choose(cur))
        out.append(y)
        nxt = next((c for c in kids[cur] if int(token[c]) == y), None)
        if nxt is None:
            return path, out
        path.append(nxt)
        cur = nxt


# ---------------------------------------------------------------------------
# single-path rejection sampler
# ---------------------------------------------------------------------------


def validate_proposal(q_rows, token, n: int, tol: float = 1e-3) -> str:
    """'ok' or the first broken rule for the proposal rows of nodes 1..n-1:
    finite, nonnegative, unit mass (|sum - 1| <= tol, summed in fp64), and
    q(x) > 0 at the drafted token (it was drawn from q)."""
    for i in range(1, n):
        q = np.asarray(q_rows[i], np.float64)
        if not np.all(np.isfinite(q)) or np.any(q < 0) or abs(q.sum() - 1.0) > tol or q[int(token[i])] <= 0:
            return "proposal"
    return "ok"


def accept_rejection_chain(token, rows_x, q_rows, uniforms, replay=None, eps: float = 0.0):
    """Single-path rejection sampling over a chain of drafts (node i's parent is
    i - 1).  Draft i (token[i], drawn from q_rows[i]) is tested against the
    target p = softmax(rows_x[i - 1]): accept iff uniforms[i] < p(x) / q(x)
    (probability min(1, p/q)).  On the first rejection one token is drawn from
    normalize(max(p - q, 0)) by the inverse CDF with uniforms[0] and the round
    ends.  A fully accepted chain ends with no extra token.

    Returns (path, out_tokens, n_replayed); ``replay`` / ``eps`` as in
    ``accept_single_draw`` (a test is replayed when |u - p/q| <= eps)."""
    n = len(token)
    path, out, replayed = [0], [], 0
    for i in range(1, n):
        p = softmax_x(rows_x[i - 1])
        q = np.asarray(q_rows[i], np.float64)
        x = int(token[i])
        ratio = p[x] / q[x]
        u = float(uniforms[i])
        ok = u < ratio
        if replay is not None and abs(u - ratio) <= eps:
            want = len(replay[0]) > len(path)
            if want != ok:
                ok = want
                replayed += 1
        if ok:
            path.append(i)
            out.append(x)
            continue
        r = np.maximum(p - q, 0.0)
        u0 = float(uniforms[0])
        y = inverse_cdf(r, u0)
        if replay is not None and len(replay[1]) > len(out):
            yg = int(replay[1][len(out)])
            if yg != y and r[yg] > 0:
                c = np.cumsum(r)
                lo = c[yg - 1] if yg > 0 else 0.0
                tt = u0 * c[-1]
                if lo - eps * c[-1] <= tt < c[yg] + eps * c[-1]:
                    y = yg
                    replayed += 1
        out.append(y)
        break
    return path, out, replayed
