"""Pins of the sampled-accept oracle (``oracle/sampling.py``) to things other
than itself: published Philox known-answer vectors, exact laws on uniform grids,
Monte Carlo laws against the target distribution (5 sigma), the sort-based
textbook definitions of the filters, and a reduction of the single-path
rejection sampler to the residual walk for a one-token drafter."""
import json
import os

import numpy as np
import pytest

import oracle
from oracle import sampling as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# Philox4x32-10 and the Gumbel draw
# ---------------------------------------------------------------------------
def test_philox_known_answers():
    kat = json.load(open(os.path.join(GOLDEN, "philox4x32_10_kat.json")))
    for v in kat["vectors"]:
        ctr = [int(w, 16) for w in v["ctr"]]
        key = [int(w, 16) for w in v["key"]]
        out = S.philox4x32_10(ctr, key)
        assert ["%08x" % int(w) for w in out] == v["out"]


def test_gumbel_uniform_word_layout():
    """token i uses word i mod 4 of the block at counter (i div 4, t, 0, 0)"""
    seed, t = 0x0123456789ABCDEF, 41
    u = S.gumbel_uniform(seed, t, np.arange(12))
    for i in range(12):
        w = S.philox4x32_10((i // 4, t, 0, 0), (seed & 0xFFFFFFFF, seed >> 32))[i % 4]
        assert u[i] == (int(w) + 0.5) / 2.0 ** 32
    # the all-zero known-answer vector of Salmon et al.: counter 0, key 0
    kat = S.philox4x32_10((0, 0, 0, 0), (0, 0))
    assert list(S.gumbel_uniform(0, 0, np.arange(4))) == [(int(w) + 0.5) / 2.0 ** 32 for w in kat]

def test_gumbel_uniforms_open_interval_and_keyed():
    u = S.gumbel_uniform(7, 3, np.arange(100000))
    assert np.all(u > 0) and np.all(u < 1)
    assert abs(u.mean() - 0.5) < 5 * np.sqrt(1 / 12 / u.size)
    assert not np.array_equal(u, S.gumbel_uniform(7, 4, np.arange(100000)))       # another position
    assert not np.array_equal(u, S.gumbel_uniform(8, 3, np.arange(100000)))       # another seed
    assert not np.array_equal(u, S.gumbel_uniform(7 + (1 << 32), 3, np.arange(100000)))   # the seed's high word


def _chi_ok(counts, p, n):
    """every count within 5 sigma of its multinomial mean"""
    sd = np.sqrt(n * p * (1 - p)) + 1e-9
    return np.all(np.abs(counts - n * p) <= 5 * sd + 1)


def test_gumbel_max_draws_follow_p():
    # argmax(x + G) over many positions t is a sample from softmax(x)
    rng = np.random.default_rng(0)
    x = rng.normal(0, 1.5, 12)
    p = S.softmax_x(x)
    T = 200000
    t = np.arange(T, dtype=np.uint64)[:, None]
    z = np.zeros((T, 3), np.uint64)
    # tokens 0..11 take the four words of the generator blocks 0, 1, 2
    words = S.philox4x32_10((np.broadcast_to(np.arange(3, dtype=np.uint64)[None, :], (T, 3)),
                             np.broadcast_to(t, (T, 3)), z, z), (99, 0))
    w = np.stack(words, axis=2).reshape(T, 12)
    u = (w.astype(np.float64) + 0.5) / 4294967296.0
    y = np.argmax(x[None, :] - np.log(-np.log(u)), axis=1)
    assert _chi_ok(np.bincount(y, minlength=12), p, T)
    # the same uniforms as gumbel_draw at a few positions
    for tt in (0, 5, 777):
        assert S.gumbel_draw(x, 99, tt) == int(y[tt])


def test_gumbel_walk_does_not_depend_on_the_drafts():
    rng = np.random.default_rng(1)
    V, n, ctx, seed = 32, 8, 40, 123456789
    rows = rng.normal(0, 2, (n, V))
    # a chain whose drafts are exactly the draws at their positions: all accepted
    parent = np.arange(-1, n - 1)
    tok = np.zeros(n, np.int64)
    for i in range(1, n):
        tok[i] = S.gumbel_draw(rows[i - 1], seed, ctx + i)
    path, out = S.accept_gumbel(parent, tok, rows, seed, ctx)
    assert path == list(range(n)) and out == [int(v) for v in tok[1:]] + [S.gumbel_draw(rows[n - 1], seed, ctx + n)]
    # any tree: the first token is the root row's draw, whatever was drafted
    for s in range(5):
        par = np.array([-1] + [int(rng.integers(0, i)) for i in range(1, n)])
        tk = rng.integers(0, V, n)
        _, out2 = S.accept_gumbel(par, tk, rows, seed, ctx)
        assert out2[0] == S.gumbel_draw(rows[0], seed, ctx + 1)


# ---------------------------------------------------------------------------
# single-draw walk
# ---------------------------------------------------------------------------
def test_single_draw_exact_grid_law():
    # root row p0 over 4 tokens; children of the root carry tokens 1 and 3 with
    # their own rows.  On a uniform grid the counts of (first, second) tokens are
    # exactly N0 * N1 * p0(y1) * p(y2 | y1's child), and N0 * p0(y1) where y1 has
    # no child (the walk ends there).
    p0 = np.array([0.1, 0.2, 0.3, 0.4])
    pa = np.array([0.5, 0.25, 0.125, 0.125])
    pb = np.array([0.25, 0.25, 0.25, 0.25])
    rows = np.log(np.stack([p0, pa, pb]))
    parent = [-1, 0, 0]
    token = [0, 1, 3]
    N0, N1 = 1000, 1000
    counts = {}
    for i in range(N0):
        for j in range(N1):
            u = [(i + 0.5) / N0, (j + 0.5) / N1, (j + 0.5) / N1]
            _, out, _ = S.accept_single_draw(parent, token, rows, u)
            counts[tuple(out)] = counts.get(tuple(out), 0) + 1
    for y1 in range(4):
        if y1 == 1:
            for y2 in range(4):
                assert counts.get((1, y2), 0) == round(N0 * N1 * p0[1] * pa[y2])
        elif y1 == 3:
            for y2 in range(4):
                assert counts.get((3, y2), 0) == round(N0 * N1 * p0[3] * pb[y2])
        else:
            assert counts.get((y1,), 0) == round(N0 * N1 * p0[y1])


def test_single_draw_and_residual_walk_share_one_law():
    rng = np.random.default_rng(3)
    V, n = 16, 7
    parent = [-1, 0, 0, 0, 1, 1, 2]
    token = [0, 3, 5, 9, 1, 2, 7]
    rows = rng.normal(0, 1.2, (n, V))
    R = 60000
    first = {"single": np.zeros(V), "residual": np.zeros(V)}
    second = {"single": {}, "residual": {}}
    for k in range(R):
        u = rng.random(n)
        _, o1, _ = S.accept_single_draw(parent, token, rows, u)
        _, o2, _ = oracle.accept_residual(parent, token, rows, 1.0, rng.random(n), bonus_at_leaf=True)
        for name, o in (("single", o1), ("residual", o2)):
            first[name][o[0]] += 1
            if len(o) > 1:
                second[name].setdefault(o[0], np.zeros(V))[o[1]] += 1
    p0 = S.softmax_x(rows[0])
    for name in first:
        assert _chi_ok(first[name], p0, R), name
        for y1, h in second[name].items():
            c = next(c for c in range(1, n) if parent[c] == 0 and token[c] == y1)
            assert _chi_ok(h, S.softmax_x(rows[c]), h.sum()), (name, y1)


# ---------------------------------------------------------------------------
# single-path rejection sampler
# ---------------------------------------------------------------------------
def test_rejection_chain_with_one_token_drafter_is_the_residual_walk():
    # q = one-hot at the draft: accept with p(x), else draw from p with x removed
    rng = np.random.default_rng(4)
    V, n = 20, 6
    rows = rng.normal(0, 1.5, (n, V))
    token = rng.integers(0, V, n)
    q = np.zeros((n, V))
    q[np.arange(n), token] = 1.0
    parent = np.arange(-1, n - 1)
    for k in range(400):
        u = rng.random(n)
        p1, o1, _ = S.accept_rejection_chain(token, rows, q, u)
        stream = list(u[1:len(p1) + 1]) + [u[0]]      # tests in order, then the residual draw
        p2, o2, _ = oracle.accept_residual(parent, token, rows, 1.0, stream, bonus_at_leaf=False)
        assert (p1, o1) == (p2, o2)


def test_rejection_chain_output_follows_the_target():
    # drafts drawn from q; the first output token is a sample from p_0 and, when
    # the first draft was kept, the second from p_1 (Leviathan et al., Thm 1)
    rng = np.random.default_rng(5)
    V = 10
    rows = rng.normal(0, 1.0, (3, V))
    q = np.stack([np.full(V, 1.0 / V), S.softmax_x(rng.normal(0, 1.0, V)), S.softmax_x(rng.normal(0, 1.0, V))])
    R = 120000
    first = np.zeros(V)
    second = {}
    for k in range(R):
        token = [0, int(rng.choice(V, p=q[1])), int(rng.choice(V, p=q[2]))]
        _, out, _ = S.accept_rejection_chain(token, rows, q, rng.random(3))
        first[out[0]] += 1
        if len(out) > 1:
            second.setdefault(out[0], np.zeros(V))[out[1]] += 1
    assert _chi_ok(first, S.softmax_x(rows[0]), R)
    p1 = S.softmax_x(rows[1])
    for y1, h in second.items():
        assert _chi_ok(h, p1, h.sum()), y1


def test_rejection_chain_perfect_drafter_keeps_everything():
    rng = np.random.default_rng(6)
    V, n = 12, 5
    rows = rng.normal(0, 1.0, (n, V))
    q = np.stack([S.softmax_x(rows[max(i - 1, 0)]) for i in range(n)])
    for k in range(50):
        token = [0] + [int(rng.choice(V, p=q[i])) for i in range(1, n)]
        path, out, _ = S.accept_rejection_chain(token, rows, q, rng.random(n) * 0.999)
        assert path == list(range(n)) and out == token[1:]


def test_validate_proposal():
    V = 6
    good = np.full((3, V), 1.0 / V)
    token = [0, 2, 4]
    assert S.validate_proposal(good, token, 3) == "ok"
    for bad in ("nan", "neg", "mass", "zero"):
        q = good.copy()
        if bad == "nan":
            q[1, 0] = np.nan
        elif bad == "neg":
            q[2, 1] = -0.01
            q[2, 0] += 0.01
        elif bad == "mass":
            q[1] *= 1.01
        else:
            q[2, 4] = 0.0
            q[2, 0] += 1.0 / V
        assert S.validate_proposal(q, token, 3) == "proposal", bad


# ---------------------------------------------------------------------------
# filters, against their sort-based definitions
# ---------------------------------------------------------------------------
def _kept(x):
    return set(np.nonzero(np.isfinite(x))[0].tolist())


def test_filters_off_scale_by_temperature():
    x = np.random.default_rng(7).normal(0, 3, 50)
    np.testing.assert_array_equal(S.sample_filter(x, 0.7), x / 0.7)


def test_top_k_keeps_the_k_largest():
    rng = np.random.default_rng(8)
    for k in (1, 3, 10, 49):
        x = rng.normal(0, 2, 50)
        assert _kept(S.sample_filter(x, 1.0, top_k=k)) == set(np.argsort(-x)[:k].tolist())
    x = np.array([3.0, 1.0, 3.0, 2.0, 3.0])        # ties at the k-th value are all kept
    assert _kept(S.sample_filter(x, 1.0, top_k=2)) == {0, 2, 4}


def test_top_p_is_the_shortest_prefix_of_the_sorted_distribution():
    rng = np.random.default_rng(9)
    for top_p in (0.05, 0.3, 0.6, 0.9, 0.999):
        x = rng.normal(0, 2, 40)
        p = np.exp(x - x.max())
        p /= p.sum()
        order = np.argsort(-p)
        m = 0.0
        want = set()
        for i in order:        # largest first until the mass reaches top_p
            want.add(int(i))
            m += p[i]
            if m >= top_p:
                break
        assert _kept(S.sample_filter(x, 1.0, top_p=top_p)) == want


def test_min_p_keeps_tokens_within_the_ratio_of_the_max():
    rng = np.random.default_rng(10)
    x = rng.normal(0, 2, 40)
    p = S.softmax_x(x)
    for mp in (0.01, 0.1, 0.5):
        assert _kept(S.sample_filter(x, 1.0, min_p=mp)) == set(np.nonzero(p >= mp * p.max())[0].tolist())


def test_filters_compose_in_order():
    rng = np.random.default_rng(11)
    x = rng.normal(0, 2, 60)
    f = S.sample_filter(x, 0.8, top_k=20, top_p=0.7, min_p=0.05)
    step = S.sample_filter(x, 0.8, top_k=20)
    step = S.sample_filter(step, 1.0, top_p=0.7)
    step = S.sample_filter(step, 1.0, min_p=0.05)
    np.testing.assert_array_equal(np.isfinite(f), np.isfinite(step))
    assert _kept(S.sample_filter(x, 1.0, top_k=1)) == {int(np.argmax(x))}
