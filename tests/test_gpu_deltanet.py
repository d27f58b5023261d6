"""GPU parity of Gated DeltaNet tree verify and the path-state commit
(tv_dn_verify_tree, tv_dn_commit) against oracle/deltanet.py, which applies
the gated delta rule node by node in fp64.

Tolerance, from the arithmetic: the GPU works in fp32 (unit roundoff 6e-8).
An output or state entry is a sum of at most 32 path terms, each built from
128-long dot products of unit keys with O(1) states and values, and the
pseudo-values come from a triangular solve whose coefficients are below 1 in
size; rounding then stays under ~1e-5 of the entries' scale.  The tests allow
2e-4 x (1 + |x|), ten times that with margin, and report the worst error."""
import numpy as np
import pytest
import torch

from oracle import deltanet as DN
from speculative_tree_verify_gb300 import abi, synth

pytestmark = pytest.mark.gpu

TOL = 2e-4


def _ok(rc, what="call"):
    assert rc == abi.TV_OK, f"{what}: {abi.STATUS.get(rc, rc)}"


def _tree(shape, n, seed):
    return {"chain": lambda: synth.tree_chain(n, 1000, seed), "lattice": lambda: synth.tree_lattice(n, 7, 1000, seed),
            "star": lambda: synth.tree_star(n, 1000, seed),
            "random": lambda: synth.tree_spine_random(n, max(1, n // 3), 1000, seed)}[shape]()


class Req:
    def __init__(self, tree, inp):
        self.tree, self.inp = tree, inp
        self.parent = torch.from_numpy(tree.parent.astype(np.int32)).cuda()
        self.token = torch.from_numpy(tree.token.astype(np.int32)).cuda()
        self.tv = abi.TvTree(self.parent.data_ptr(), self.token.data_ptr(), tree.n)
        self.S = torch.from_numpy(inp.S0.copy()).cuda()


def _run_verify(dims, reqs):
    cat = lambda name: torch.from_numpy(np.concatenate([getattr(r.inp, name) for r in reqs])).cuda()
    q, k, v, beta, g = (cat(x) for x in ("q", "k", "v", "beta", "g"))
    rows = q.shape[0]
    o = torch.full((rows, dims.n_v_heads, dims.d_v), float("nan"), device="cuda")
    u = torch.full_like(o, float("nan"))
    gc = torch.full((rows, dims.n_v_heads), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    _ok(abi.tv_dn_verify_tree(dims, [r.tv for r in reqs], [r.S for r in reqs], q, k, v, beta, g, o, u, gc, st))
    torch.cuda.synchronize()
    assert int(st.item()) == 0, abi.STATUS.get(int(st.item()))
    return dict(q=q, k=k, v=v, beta=beta, g=g, o=o, u=u, gc=gc, status=st)


def _oracle(r):
    x = r.inp
    return DN.dn_verify_tree(r.tree.parent, x.q.astype(np.float64), x.k.astype(np.float64), x.v.astype(np.float64),
                             x.beta.astype(np.float64), x.g.astype(np.float64), x.S0.astype(np.float64))


def _close(gpu, orc, what):
    err = np.abs(gpu.astype(np.float64) - orc) / (1.0 + np.abs(orc))
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite"
    assert err.max() <= TOL, f"{what}: worst error {err.max():.3e} x (1 + |x|) > {TOL}"
    print(f"{what}: worst error {err.max():.3e} x (1 + |x|)")
    return float(err.max())


def _root_path(parent, t):
    p = []
    while t >= 0:
        p.append(int(t))
        t = parent[t]
    return p[::-1]


@pytest.mark.parametrize("shape,n", [("chain", 1), ("chain", 32), ("lattice", 16), ("lattice", 32), ("star", 9),
                                     ("random", 24)])
@pytest.mark.parametrize("dimset", [(2, 4, 128, 128), (1, 2, 64, 32)])
def test_dn_verify_and_commit_parity(gpu, shape, n, dimset):
    Hk, Hv, dk, dv = dimset
    dims = abi.TvDnDims(Hk, Hv, dk, dv)
    tree = _tree(shape, n, 3 + n)
    r = Req(tree, synth.dn_inputs(n, Hk, Hv, dk, dv, 100 + n))
    out = _run_verify(dims, [r])
    orc = _oracle(r)
    _close(out["o"].cpu().numpy(), orc["o"], "outputs")
    # commit along several root paths: the root alone, a leaf's path, the deepest node's path
    depth = np.zeros(n, int)
    for t in range(1, n):
        depth[t] = depth[tree.parent[t]] + 1
    leaves = [t for t in range(n) if t not in set(tree.parent[1:].tolist())]
    for last in sorted({0, leaves[0], int(np.argmax(depth)), n - 1}):
        p = _root_path(tree.parent, last)
        S = torch.from_numpy(r.inp.S0.copy()).cuda()
        path = torch.full((n,), -1, dtype=torch.int32, device="cuda")
        path[:len(p)] = torch.tensor(p, dtype=torch.int32)
        alen = torch.tensor([len(p) - 1], dtype=torch.int32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        _ok(abi.tv_dn_commit(dims, [r.tv], 1, [S], out["k"], out["u"], out["gc"], path, alen, st))
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        _close(S.cpu().numpy(), DN.dn_commit(r.inp.S0, orc["states"], p), f"state after path to {last}")


def test_dn_chain_rollback_to_every_length(gpu):
    n, dims = 12, abi.TvDnDims(2, 4, 128, 64)
    tree = synth.tree_chain(n, 1000, 5)
    r = Req(tree, synth.dn_inputs(n, 2, 4, 128, 64, 7))
    out = _run_verify(dims, [r])
    orc = _oracle(r)
    for m in range(1, n + 1):   # keep the first m tokens of the block
        S = torch.from_numpy(r.inp.S0.copy()).cuda()
        path = torch.arange(n, dtype=torch.int32, device="cuda")
        alen = torch.tensor([m - 1], dtype=torch.int32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        _ok(abi.tv_dn_commit(dims, [r.tv], 1, [S], out["k"], out["u"], out["gc"], path, alen, st))
        torch.cuda.synchronize()
        _close(S.cpu().numpy(), orc["states"][m - 1], f"rollback to {m}")


def test_dn_joint_requests_and_layers(gpu):
    dims = abi.TvDnDims(2, 4, 128, 128)
    shapes = [("lattice", 16), ("random", 8), ("chain", 5)]
    reqs = [Req(_tree(s, n, 20 + i), synth.dn_inputs(n, 2, 4, 128, 128, 30 + i)) for i, (s, n) in enumerate(shapes)]
    out = _run_verify(dims, reqs)
    o = out["o"].cpu().numpy()
    row = 0
    for r in reqs:
        _close(o[row:row + r.tree.n], _oracle(r)["o"], "joint outputs")
        row += r.tree.n
    # three layers: layer l uses request inputs with another seed; one commit call for all of them
    L = 3
    layer_inputs = [[synth.dn_inputs(r.tree.n, 2, 4, 128, 128, 50 + 7 * l + i) for i, r in enumerate(reqs)]
                    for l in range(L)]
    ks, us, gcs, orcs = [], [], [], []
    for l in range(L):
        lr = [Req(r.tree, layer_inputs[l][i]) for i, r in enumerate(reqs)]
        res = _run_verify(dims, lr)
        ks.append(res["k"])
        us.append(res["u"])
        gcs.append(res["gc"])
        orcs.append([_oracle(x) for x in lr])
    states = [torch.from_numpy(np.stack([layer_inputs[l][i].S0 for l in range(L)])).cuda() for i in range(len(reqs))]
    paths, alens, want = [], [], []
    for i, r in enumerate(reqs):
        last = r.tree.n - 1
        p = _root_path(r.tree.parent, last)
        paths += p + [-1] * (r.tree.n - len(p))
        alens.append(len(p) - 1)
        want.append(np.stack([orcs[l][i]["states"][last] for l in range(L)]))
    path = torch.tensor(paths, dtype=torch.int32, device="cuda")
    alen = torch.tensor(alens, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    _ok(abi.tv_dn_commit(dims, [r.tv for r in reqs], L, states, torch.stack(ks), torch.stack(us), torch.stack(gcs),
                         path, alen, st))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for i in range(len(reqs)):
        _close(states[i].cpu().numpy(), want[i], f"request {i}, all layers")


def test_dn_full_dims(gpu):
    """16 key heads and 32 value heads of 128, a 32-node lattice"""
    dims = abi.TvDnDims(16, 32, 128, 128)
    tree = synth.tree_lattice(32, 15, 151936, 41)
    r = Req(tree, synth.dn_inputs(32, 16, 32, 128, 128, 77))
    out = _run_verify(dims, [r])
    orc = _oracle(r)
    _close(out["o"].cpu().numpy(), orc["o"], "outputs")
    _close(out["gc"].cpu().numpy(), np.array([[sum(r.inp.g[s, h].astype(np.float64)
                                                   for s in _root_path(tree.parent, t)) for h in range(32)]
                                                 for t in range(32)]), "cumulative gates")


def test_dn_rejects_bad_tree_and_bad_path(gpu):
    dims = abi.TvDnDims(1, 2, 32, 32)
    tree = synth.tree_chain(6, 1000, 9)
    bad = synth.Tree(tree.parent.copy(), tree.token.copy())
    bad.parent[4] = 5
    r = Req(bad, synth.dn_inputs(6, 1, 2, 32, 32, 1))
    q = torch.from_numpy(r.inp.q).cuda()
    k = torch.from_numpy(r.inp.k).cuda()
    v = torch.from_numpy(r.inp.v).cuda()
    beta, g = torch.from_numpy(r.inp.beta).cuda(), torch.from_numpy(r.inp.g).cuda()
    o = torch.zeros(6, 2, 32, device="cuda")
    u, gc = torch.zeros_like(o), torch.zeros(6, 2, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    _ok(abi.tv_dn_verify_tree(dims, [r.tv], [r.S], q, k, v, beta, g, o, u, gc, st))
    torch.cuda.synchronize()
    assert int(st.item()) == abi.CODES["TV_E_ORDER"]
    # a path that is not a root path leaves the state untouched
    good = Req(tree, r.inp)
    out = _run_verify(dims, [good])
    S = torch.from_numpy(r.inp.S0.copy()).cuda()
    path = torch.tensor([0, 2, -1, -1, -1, -1], dtype=torch.int32, device="cuda")   # node 2 is a grandchild
    alen = torch.tensor([1], dtype=torch.int32, device="cuda")
    st.zero_()
    _ok(abi.tv_dn_commit(dims, [good.tv], 1, [S], out["k"], out["u"], out["gc"], path, alen, st))
    torch.cuda.synchronize()
    assert int(st.item()) == abi.CODES["TV_E_PATH"]
    assert np.array_equal(S.cpu().numpy(), r.inp.S0)


def test_dn_full_size_48_layers_sampled(gpu):
    """The bench's configuration: 16 key / 32 value heads of 128, a 16-row
    lattice, the core of 48 layers (one call per layer, each on its own
    state), then one commit of all 48 layers along the deepest root path.
    Sampled (layer, head) pairs are checked against the oracle."""
    Hk, Hv, dk, dv, NL, n = 16, 32, 128, 128, 48, 16
    dims = abi.TvDnDims(Hk, Hv, dk, dv)
    tree = synth.tree_lattice(n, 7, 151936, 7)
    inps = [synth.dn_inputs(n, Hk, Hv, dk, dv, 900 + l) for l in range(NL)]
    par = torch.from_numpy(tree.parent.astype(np.int32)).cuda()
    tok = torch.from_numpy(tree.token.astype(np.int32)).cuda()
    tv = abi.TvTree(par.data_ptr(), tok.data_ptr(), n)
    S = torch.from_numpy(np.stack([x.S0 for x in inps])).cuda()
    k_all = torch.from_numpy(np.stack([x.k for x in inps])).cuda()
    u_all = torch.empty(NL, n, Hv, dv, device="cuda")
    gc_all = torch.empty(NL, n, Hv, device="cuda")
    o_all = torch.empty(NL, n, Hv, dv, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lb = Hv * dk * dv * 4
    for l, x in enumerate(inps):
        q, v, beta, g = (torch.from_numpy(a).cuda() for a in (x.q, x.v, x.beta, x.g))
        _ok(abi.tv_dn_verify_tree(dims, [tv], [S.data_ptr() + l * lb], q, k_all[l], v, beta, g, o_all[l], u_all[l],
                                  gc_all[l], st))
    depth = np.zeros(n, int)
    for t in range(1, n):
        depth[t] = depth[tree.parent[t]] + 1
    p = _root_path(tree.parent, int(np.argmax(depth)))
    path = torch.tensor(p + [-1] * (n - len(p)), dtype=torch.int32, device="cuda")
    alen = torch.tensor([len(p) - 1], dtype=torch.int32, device="cuda")
    _ok(abi.tv_dn_commit(dims, [tv], NL, [S], k_all, u_all, gc_all, path, alen, st))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    o_g, S_g = o_all.cpu().numpy(), S.cpu().numpy()
    rng = np.random.default_rng(0)
    for l, h in zip(rng.choice(NL, 6, replace=False), rng.choice(Hv, 6)):
        x = inps[l]
        kh = h // (Hv // Hk)
        states, outs = DN.dn_tree_states(tree.parent, x.q[:, kh].astype(np.float64), x.k[:, kh].astype(np.float64),
                                         x.v[:, h].astype(np.float64), x.beta[:, h].astype(np.float64),
                                         x.g[:, h].astype(np.float64), x.S0[h].astype(np.float64))
        _close(o_g[l][:, h], outs, f"layer {l} head {h} outputs")
        _close(S_g[l, h], DN.dn_commit(x.S0[h], states, p), f"layer {l} head {h} committed state")
