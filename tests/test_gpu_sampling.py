"""GPU parity of the sampled accept variants against ``oracle/sampling.py``:
filters, single-draw walk, seeded Gumbel walk, single-path rejection sampler.
Integer outputs are compared exactly; where a float decides an integer (a CDF
boundary, an argmax of noisy scores, a p/q test) the oracle replays the GPU's
choice only inside a stated margin."""
import numpy as np
import pytest
import torch

import oracle
from oracle import sampling as S
from speculative_tree_verify_gb300 import abi, synth

from parity import to_np

pytestmark = pytest.mark.gpu


def _ok(rc, what="call"):
    assert rc == abi.TV_OK, f"{what}: {abi.STATUS.get(rc, rc)}"


def _trees(V, n_req, seed, n_each=8):
    out = []
    for i in range(n_req):
        out.append(synth.tree_lattice(n_each, 7, V, seed + i) if i % 2 == 0
                   else synth.tree_spine_random(n_each, 3, V, seed + i))
    return out


def _tv_trees(trees):
    keep = []
    tv = []
    for t in trees:
        p = torch.from_numpy(t.parent.astype(np.int32)).cuda()
        k = torch.from_numpy(t.token.astype(np.int32)).cuda()
        keep += [p, k]
        tv.append(abi.TvTree(p.data_ptr(), k.data_ptr(), t.n))
    return tv, keep


def _bufs(rows, n_req, V):
    rc, wsb = abi.tv_sample_workspace_size(V, rows)
    assert rc == 0
    z = lambda n, dt=torch.int32: torch.zeros(n, dtype=dt, device="cuda")
    return dict(row_tokens=z(rows), path=z(rows), accept_len=z(n_req), out_tokens=z(rows), out_count=z(n_req),
                status=z(1), ws=torch.zeros(wsb, dtype=torch.uint8, device="cuda"), wsb=wsb)


def _on_boundary(l, T, k, p, mp, j, tol=1e-5):
    """Token j sits within tol of the top_p cut (the running mass, largest
    first, before or after j) or of the min_p threshold, in fp64."""
    x = np.asarray(l, np.float64) / T
    keep = np.isfinite(x)
    if 0 < k < keep.sum():
        keep &= x >= np.sort(x)[::-1][k - 1]
    near = False
    if p < 1.0 and keep[j]:
        pr = np.where(keep, np.exp(x - x[keep].max()), 0.0)
        pr /= pr.sum()
        above = pr[pr > pr[j]].sum()
        near |= abs(above - p) < tol or abs(above + pr[j] - p) < tol
    if mp > 0.0:
        near |= abs(x[j] - (x[keep].max() + np.log(mp))) < tol
    return near


# ---------------------------------------------------------------------------
# filters
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("V", [1024, 151936])
@pytest.mark.parametrize("T,k,p,mp", [(0.7, 0, 1.0, 0.0), (1.0, 50, 1.0, 0.0), (0.8, 0, 0.9, 0.0),
                                      (1.2, 0, 1.0, 0.05), (0.9, 200, 0.8, 0.01), (1.0, 1, 1.0, 0.0)])
def test_filter_parity(gpu, V, T, k, p, mp):
    rows = 5
    logits = synth.logits_rows(rows, V, 11 + V % 7, scale=3.0)
    x = torch.from_numpy(logits).cuda()
    out = torch.empty_like(x)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    _ok(abi.tv_sample_filter(x, out, rows, V, T, k, p, mp, st))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    g = out.cpu().numpy()
    for r in range(rows):
        o = S.sample_filter(logits[r], T, top_k=k, top_p=p, min_p=mp)
        keep_o, keep_g = np.isfinite(o), np.isfinite(g[r])
        diff = np.nonzero(keep_o != keep_g)[0]
        for j in diff:   # fp32 against fp64: only a token on the top_p or min_p boundary may differ
            assert _on_boundary(logits[r], T, k, p, mp, j), (r, j)
        both = keep_o & keep_g
        np.testing.assert_allclose(g[r, both], o[both], rtol=3e-7, atol=0)


def _filter_check(logits, T, k, p, mp):
    rows, V = logits.shape
    x = torch.from_numpy(np.ascontiguousarray(logits)).cuda()
    out = torch.empty_like(x)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    _ok(abi.tv_sample_filter(x, out, rows, V, T, k, p, mp, st))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    g = out.cpu().numpy()
    for r in range(rows):
        o = S.sample_filter(logits[r], T, top_k=k, top_p=p, min_p=mp)
        keep_o, keep_g = np.isfinite(o), np.isfinite(g[r])
        for j in np.nonzero(keep_o != keep_g)[0]:
            assert _on_boundary(logits[r], T, k, p, mp, j), (r, j)
        both = keep_o & keep_g
        np.testing.assert_allclose(g[r, both], o[both], rtol=3e-7, atol=0)
        assert np.all(g[r, ~keep_g] == -np.inf)
    return g


@pytest.mark.parametrize("V", [2, 16, 4099, 262144])
def test_filter_vocab_sizes(gpu, V):
    logits = synth.logits_rows(3, V, 40 + V % 11, scale=2.0)
    _filter_check(logits, 0.9, min(7, V - 1), 0.85, 0.01)


@pytest.mark.parametrize("V", [151936, 262144])
@pytest.mark.parametrize("T,k,p,mp", [(0.8, 50, 0.9, 0.02), (0.8, 0, 0.9, 0.0)])
def test_filter_sixteen_rows(gpu, V, T, k, p, mp):
    # 16 rows: the launch takes smaller clusters, so a CTA holds a longer slice
    # (at 262144 past the part its threads keep in registers)
    logits = synth.logits_rows(16, V, 90 + V % 13, scale=1.5)
    _filter_check(logits, T, k, p, mp)


def test_filter_ties_and_masked_rows(gpu):
    V = 20000
    rng = np.random.default_rng(3)
    logits = (np.round(rng.standard_normal((4, V)) * 2) / 2).astype(np.float32)   # heavy ties
    logits[1, rng.random(V) < 0.3] = -np.inf                                       # an already-filtered row
    logits[2] = 1.25                                                               # one value everywhere
    logits[3, :V // 2] = -np.inf
    for T, k, p, mp in ((1.0, 10, 1.0, 0.0), (0.7, 0, 0.5, 0.0), (1.3, 300, 0.95, 0.1), (1.0, 0, 1e-6, 0.0)):
        g = _filter_check(logits, T, k, p, mp)
        if k == 10:   # every token tied with the 10th largest stays
            r0 = logits[0]
            kth = np.sort(r0)[::-1][9]
            assert np.isfinite(g[0]).sum() == (r0 >= kth).sum() > 10
        if p == 1e-6:   # only the largest logit (and its ties) stays
            assert np.array_equal(np.isfinite(g[0]), logits[0] == logits[0].max())


def test_filter_signed_zero_ties(gpu):
    """-0.0 and +0.0 compare equal, so both stay when they tie at the boundary"""
    V = 4096
    logits = np.full((1, V), -5.0, np.float32)
    logits[0, :3] = [3.0, 2.0, 1.0]
    logits[0, 10] = 0.0
    logits[0, 20] = -0.0
    g = _filter_check(logits, 1.0, 4, 1.0, 0.0)
    assert np.isfinite(g[0, 10]) and np.isfinite(g[0, 20]) and np.isfinite(g[0]).sum() == 5

def test_filter_large_logits(gpu):
    """logits near 1e7: the fast top_k cut's fixed grid (8 bins a unit of
    l / T) leaves float's exact integers there, so the three-level selection
    decides; a row with few tokens per slice and one small row take the fast cut"""
    V = 151936
    rng = np.random.default_rng(12)
    logits = np.empty((3, V), np.float32)
    logits[0] = (1e7 + rng.standard_normal(V) * 1e3).astype(np.float32)
    logits[1] = (rng.standard_normal(V) * 4.0).astype(np.float32)
    logits[2] = -np.inf
    logits[2, rng.choice(V, 40, replace=False)] = rng.standard_normal(40).astype(np.float32)
    for T, k, p, mp in ((1.0, 20, 1.0, 0.0), (0.8, 50, 0.9, 0.02), (1.0, 30, 0.7, 0.0)):
        _filter_check(logits, T, k, p, mp)


def test_filter_rejects_bad_arguments(gpu):
    x = torch.zeros(2, 16, device="cuda")
    out = torch.empty_like(x)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert abi.tv_sample_filter(x, out, 2, 16, 0.0, 0, 1.0, 0.0, st) == abi.CODES["TV_E_TEMP"]
    assert abi.tv_sample_filter(x, out, 2, 16, 1.0, -1, 1.0, 0.0, st) == abi.CODES["TV_E_ARG"]
    assert abi.tv_sample_filter(x, out, 2, 16, 1.0, 0, 0.0, 0.0, st) == abi.CODES["TV_E_ARG"]
    assert abi.tv_sample_filter(x, out, 2, 16, 1.0, 0, 1.0, 1.0, st) == abi.CODES["TV_E_ARG"]
    assert abi.tv_sample_filter(x, x, 2, 16, 1.0, 0, 1.0, 0.0, st) == abi.CODES["TV_E_ARG"]


# ---------------------------------------------------------------------------
# single-draw walk
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("V,T,seed", [(1024, 1.0, 0), (5003, 0.7, 1), (151936, 1.0, 2)])
def test_single_draw_parity(gpu, V, T, seed):
    trees = _trees(V, 3, 300 + seed)
    rows = sum(t.n for t in trees)
    logits = synth.logits_rows(rows, V, 310 + seed, scale=2.0)
    off = 0
    for t in trees:   # plausible drafts: each child's token among its parent row's best
        for c in range(1, t.n):
            logits[off + t.parent[c], t.token[c]] = logits[off + t.parent[c]].max() + 4.0
        off += t.n
    tv, keep = _tv_trees(trees)
    b = _bufs(rows, len(trees), V)
    lt = torch.from_numpy(logits).cuda()
    replays = 0
    for trial in range(4):
        u = synth.uniforms(rows, 320 + 17 * seed + trial)
        ut = torch.from_numpy(u).cuda()
        b["status"].zero_()
        _ok(abi.tv_accept_single_draw(tv, lt, V, T, ut, b["row_tokens"], b["path"], b["accept_len"],
                                      b["out_tokens"], b["status"], b["ws"], b["wsb"]))
        torch.cuda.synchronize()
        assert int(b["status"].item()) == 0
        off = 0
        for r, t in enumerate(trees):
            a = int(b["accept_len"][r])
            gpath = to_np(b["path"])[off:off + a + 1].tolist()
            gout = to_np(b["out_tokens"])[off:off + a + 1].tolist()
            x = logits[off:off + t.n].astype(np.float64) / T
            path, out, rep = S.accept_single_draw(t.parent, t.token, x, u[off:off + t.n], replay=(gpath, gout),
                                                  eps=1e-5)
            replays += rep
            assert (gpath, gout) == (path, out), (trial, r)
            off += t.n
    assert replays <= 2


# ---------------------------------------------------------------------------
# seeded Gumbel walk
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("V,T,seed", [(1024, 1.0, 0), (5003, 1.1, 2), (151936, 0.8, 1)])
def test_gumbel_parity(gpu, V, T, seed):
    trees = _trees(V, 3, 400 + seed)
    rows = sum(t.n for t in trees)
    logits = synth.logits_rows(rows, V, 410 + seed, scale=2.0)
    tv, keep = _tv_trees(trees)
    b = _bufs(rows, len(trees), V)
    lt = torch.from_numpy(logits).cuda()
    seeds = [123456789 + 7 * r + (seed << 40) for r in range(len(trees))]
    positions = [1000 + 37 * r for r in range(len(trees))]
    _ok(abi.tv_accept_gumbel(tv, lt, V, T, seeds, positions, b["row_tokens"], b["path"], b["accept_len"],
                             b["out_tokens"], b["status"], b["ws"], b["wsb"]))
    torch.cuda.synchronize()
    assert int(b["status"].item()) == 0
    grow = to_np(b["row_tokens"])
    off, near = 0, 0
    for r, t in enumerate(trees):
        depth = np.zeros(t.n, int)
        for i in range(1, t.n):
            depth[i] = depth[t.parent[i]] + 1
        x = logits[off:off + t.n].astype(np.float64) / T
        for i in range(t.n):
            sc = S.gumbel_scores(x[i], seeds[r], positions[r] + depth[i] + 1)
            y = int(np.argmax(sc))
            if int(grow[off + i]) != y:   # fp32 noise: only a near tie may differ
                assert sc[y] - sc[int(grow[off + i])] <= 1e-4, (r, i)
                near += 1
        a = int(b["accept_len"][r])
        path, out = S.accept_gumbel(t.parent, t.token, x, seeds[r], positions[r],
                                    choose=lambda i: int(grow[off + i]))
        assert to_np(b["path"])[off:off + a + 1].tolist() == path
        assert to_np(b["out_tokens"])[off:off + a + 1].tolist() == out
        off += t.n
    assert near <= 1


def test_gumbel_text_does_not_depend_on_the_drafts(gpu):
    V, n, seed, pos = 2048, 8, 987654321, 500
    logits = synth.logits_rows(n, V, 5, scale=1.0)
    lt = torch.from_numpy(logits).cuda()
    b = _bufs(n, 1, V)
    firsts = set()
    for s in range(6):
        t = synth.tree_spine_random(n, 3, V, 60 + s)
        tv, keep = _tv_trees([t])
        b["status"].zero_()
        _ok(abi.tv_accept_gumbel(tv, lt, V, 1.0, [seed], [pos], b["row_tokens"], b["path"], b["accept_len"],
                                 b["out_tokens"], b["status"], b["ws"], b["wsb"]))
        torch.cuda.synchronize()
        firsts.add(int(b["out_tokens"][0]))
    assert len(firsts) == 1                      # the root row's draw, whatever was drafted
    assert firsts.pop() == int(np.argmax(S.gumbel_scores(logits[0].astype(np.float64), seed, pos + 1)))


def test_gumbel_law_on_gpu(gpu):
    """Over many seeds the draw follows p (16 tokens, 5 sigma)."""
    V, R = 16, 4000
    x = synth.logits_rows(1, V, 9, scale=1.0)[0]
    p = S.softmax_x(x.astype(np.float64))
    t = synth.tree_chain(1, V, 0)
    tv, keep = _tv_trees([t])
    lt = torch.from_numpy(x[None, :]).cuda()
    b = _bufs(1, 1, V)
    draws = []
    for s in range(R):
        _ok(abi.tv_accept_gumbel(tv, lt, V, 1.0, [s * 2654435761], [s % 7], b["row_tokens"], b["path"],
                                 b["accept_len"], b["out_tokens"], b["status"], b["ws"], b["wsb"]))
        draws.append(b["row_tokens"][:1].clone())
    d = torch.cat(draws).cpu().numpy()
    assert int(b["status"].item()) == 0
    counts = np.bincount(d, minlength=V)
    sd = np.sqrt(R * p * (1 - p))
    assert np.all(np.abs(counts - R * p) <= 5 * sd + 1)


# ---------------------------------------------------------------------------
# single-path rejection sampler
# ---------------------------------------------------------------------------
def _chain_inputs(V, n, seed, T=1.0):
    rng = np.random.default_rng(seed)
    logits = synth.logits_rows(n, V, seed, scale=2.0)
    # proposals: a blend of the target row and noise, so that drafts are often kept
    q = np.zeros((n, V), np.float32)
    token = np.zeros(n, np.int32)
    for i in range(1, n):
        pt = S.softmax_x(logits[i - 1].astype(np.float64) / T)
        noise = rng.dirichlet(np.full(V, 0.5))
        qi = 0.7 * pt + 0.3 * noise
        qi = (qi / qi.sum()).astype(np.float32)
        q[i] = qi
        token[i] = int(rng.choice(V, p=qi.astype(np.float64) / qi.astype(np.float64).sum()))
    return logits, q, token


@pytest.mark.parametrize("V,T,seed", [(1024, 1.0, 0), (5003, 0.8, 1), (151936, 1.0, 2)])
def test_rejection_parity(gpu, V, T, seed):
    n, n_req = 8, 3
    trees, L, Q = [], [], []
    for r in range(n_req):
        lg, q, tok = _chain_inputs(V, n, 500 + 10 * seed + r, T)
        trees.append(synth.Tree(np.arange(-1, n - 1, dtype=np.int32), tok))
        L.append(lg)
        Q.append(q)
    logits = np.concatenate(L)
    qall = np.concatenate(Q)
    rows = n * n_req
    tv, keep = _tv_trees(trees)
    b = _bufs(rows, n_req, V)
    lt, qt = torch.from_numpy(logits).cuda(), torch.from_numpy(qall).cuda()
    replays, accepted = 0, 0
    for trial in range(5):
        u = synth.uniforms(rows, 520 + 13 * seed + trial)
        ut = torch.from_numpy(u).cuda()
        b["status"].zero_()
        _ok(abi.tv_accept_rejection(tv, lt, V, T, qt, ut, b["path"], b["accept_len"], b["out_tokens"],
                                    b["out_count"], b["status"], b["ws"], b["wsb"]))
        torch.cuda.synchronize()
        assert int(b["status"].item()) == 0, abi.STATUS.get(int(b["status"].item()))
        for r in range(n_req):
            off = r * n
            a, cnt = int(b["accept_len"][r]), int(b["out_count"][r])
            gpath = to_np(b["path"])[off:off + a + 1].tolist()
            gout = to_np(b["out_tokens"])[off:off + cnt].tolist()
            x = logits[off:off + n].astype(np.float64) / T
            path, out, rep = S.accept_rejection_chain(trees[r].token, x, qall[off:off + n].astype(np.float64),
                                                      u[off:off + n], replay=(gpath, gout), eps=1e-5)
            replays += rep
            accepted += a
            assert (gpath, gout) == (path, out), (trial, r)
    assert replays <= 2 and accepted > 0


@pytest.mark.parametrize("case,code", [("tree", "TV_E_CHAIN"), ("negative", "TV_E_PROPOSAL"),
                                       ("mass", "TV_E_PROPOSAL"), ("zero_at_draft", "TV_E_PROPOSAL"),
                                       ("uniform", "TV_E_UNIFORM")])
def test_rejection_rejects_bad_inputs(gpu, case, code):
    V, n = 256, 5
    logits, q, tok = _chain_inputs(V, n, 77)
    parent = np.arange(-1, n - 1, dtype=np.int32)
    u = synth.uniforms(n, 3)
    if case == "tree":
        parent[3] = 1
    elif case == "negative":
        q[2, 5] = -1e-3
    elif case == "mass":
        q[3] *= 1.01
    elif case == "zero_at_draft":
        q[2, tok[2]] = 0.0
        q[2] /= q[2].sum()
    else:
        u[4] = 1.0
    t = synth.Tree(parent, tok)
    tv, keep = _tv_trees([t])
    b = _bufs(n, 1, V)
    _ok(abi.tv_accept_rejection(tv, torch.from_numpy(logits).cuda(), V, 1.0, torch.from_numpy(q).cuda(),
                                torch.from_numpy(u).cuda(), b["path"], b["accept_len"], b["out_tokens"],
                                b["out_count"], b["status"], b["ws"], b["wsb"]))
    torch.cuda.synchronize()
    assert int(b["status"].item()) == abi.CODES[code]


# ---------------------------------------------------------------------------
# filters feeding a walk: the filtered rows at temperature 1
# ---------------------------------------------------------------------------
def test_filtered_rows_feed_the_residual_walk(gpu):
    V = 5003
    trees = _trees(V, 2, 900)
    rows = sum(t.n for t in trees)
    logits = synth.logits_rows(rows, V, 901, scale=3.0)
    lt = torch.from_numpy(logits).cuda()
    ft = torch.empty_like(lt)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    _ok(abi.tv_sample_filter(lt, ft, rows, V, 0.8, 40, 0.9, 0.02, st))
    tv, keep = _tv_trees(trees)
    b = _bufs(rows, len(trees), V)
    u = synth.uniforms(rows, 902)
    _ok(abi.tv_accept_single_draw(tv, ft, V, 1.0, torch.from_numpy(u).cuda(), b["row_tokens"], b["path"],
                                  b["accept_len"], b["out_tokens"], st, b["ws"], b["wsb"]))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    f = ft.cpu().numpy()
    grow = to_np(b["row_tokens"])
    for i in range(rows):
        assert np.isfinite(f[i, grow[i]])                     # every draw is a kept token
        o = S.sample_filter(logits[i], 0.8, 40, 0.9, 0.02)
        assert np.isfinite(o[grow[i]])
