"""GPU parity of the tree verify round against the oracle, through the C ABI.

Sizes here are the ones the oracle finishes in seconds: the tiny random layer
(hidden 256, 4/2 heads of 64, vocab 1024, context 64) and a mid layer (hidden
512, 8/2 heads of 128, vocab 5003) that spans several GEMM tiles, several
attention chunks and ragged tails everywhere.  The hidden-5120 shapes are in
test_gpu_fullsize.py.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_tree_verify_gb300 import abi, build, synth
from speculative_tree_verify_gb300 import device as dv
from speculative_tree_verify_gb300.device import DeviceModel, DeviceRequest, RoundBuffers

from parity import (KV_TOL, _ok, check_close_bf16, check_verify, gpu_verify, greedy_replay, plant_spine,
                    to_np)

pytestmark = pytest.mark.gpu


# ---------------------------------------------------------------------------
# verify parity
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("seed", range(10))
def test_tiny_layer_parity(gpu, seed):
    d = synth.TINY
    model = synth.gen_model(d, seed, random_gains=True)
    cache = synth.gen_cache(d, 64, 96, 1000 + seed)
    tree = synth.tree_spine_random(8, 4, d.vocab, 2000 + seed)
    check_verify(model, [(cache, tree)])


@pytest.mark.parametrize("case", ["ctx0", "single_row", "chain32", "star32", "tight_capacity", "ctx1",
                                  "ctx_ragged", "lattice24"])
def test_tiny_edge_cases(gpu, case):
    d = synth.TINY
    model = synth.gen_model(d, 77, random_gains=True)
    ctx, cap, tree = {
        "ctx0": (0, 40, synth.tree_spine_random(8, 3, d.vocab, 1)),
        "single_row": (64, 65, synth.tree_chain(1, d.vocab, 2)),
        "chain32": (64, 96, synth.tree_chain(32, d.vocab, 3)),
        "star32": (64, 100, synth.tree_star(32, d.vocab, 4)),
        "tight_capacity": (37, 45, synth.tree_spine_random(8, 5, d.vocab, 5)),
        "ctx1": (1, 16, synth.tree_spine_random(8, 2, d.vocab, 6)),
        "ctx_ragged": (2049 + 65, 2200, synth.tree_lattice(16, 7, d.vocab, 7)),
        "lattice24": (200, 256, synth.tree_lattice(24, 7, d.vocab, 8)),
    }[case]
    cache = synth.gen_cache(d, ctx, cap, 500)
    check_verify(model, [(cache, tree)])


@pytest.mark.parametrize("ctx,n,seed", [(300, 32, 0), (1000, 8, 1), (4097, 24, 2)])
def test_mid_layer_parity(gpu, ctx, n, seed):
    d = synth.MID
    model = synth.gen_model(d, 40 + seed, random_gains=True)
    cache = synth.gen_cache(d, ctx, ctx + 40, 41 + seed)
    tree = synth.tree_lattice(n, 15, d.vocab, 42 + seed)
    _, _, _, stats = check_verify(model, [(cache, tree)])
    print(stats)


@pytest.mark.parametrize("layout", [(16, 16), (8, 8, 8, 8), (5, 1, 20)])
def test_joint_verify_parity(gpu, layout):
    d = synth.MID
    model = synth.gen_model(d, 60, random_gains=True)
    ctxs = synth.joint_contexts(len(layout), 61, lo=100, hi=900)
    host = [(synth.gen_cache(d, c, c + n + 5, 62 + i), synth.tree_lattice(n, 7, d.vocab, 63 + i))
            for i, (c, n) in enumerate(zip(ctxs, layout))]
    check_verify(model, host)


# ---------------------------------------------------------------------------
# the tile-packed weights
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("rows,cols", [(1, 64), (300, 192), (128, 5120), (1000, 320)])
def test_pack_weight_layout(gpu, rows, cols):
    w = torch.from_numpy(np.random.default_rng(rows + cols).standard_normal((rows, cols)).astype(np.float32))
    wt = w.to(torch.bfloat16).cuda()
    mt = (rows + 127) // 128
    out = torch.full((abi.tv_packed_weight_bytes(rows, cols) // 2,), float("nan"), dtype=torch.bfloat16,
                     device="cuda")   # every element must be written
    _ok(abi.tv_pack_weight(wt, rows, cols, out), "tv_pack_weight")
    torch.cuda.synchronize()
    # rows padded with zeros to 128 mt, cut into 128 x 64 tiles, tile (i, j) row-major at (i cols/64 + j) 8192
    wp = np.zeros((mt * 128, cols), np.uint16)
    wp[:rows] = wt.view(torch.int16).cpu().numpy().view(np.uint16)
    want = wp.reshape(mt, 128, cols // 64, 64).transpose(0, 2, 1, 3).reshape(-1)
    np.testing.assert_array_equal(out.view(torch.int16).cpu().numpy().view(np.uint16), want)


@pytest.mark.parametrize("dims", ["tiny", "mid"])
def test_packed_weights_give_the_same_verify(gpu, dims):
    d = {"tiny": synth.TINY, "mid": synth.MID}[dims]
    model = synth.gen_model(d, 90, random_gains=True)
    host = [(synth.gen_cache(d, 700, 760, 91), synth.tree_lattice(24, 7, d.vocab, 92))]
    _, bp = gpu_verify(DeviceModel.from_host(model, packed=True), host)
    _, br = gpu_verify(DeviceModel.from_host(model, packed=False), host)
    for name in ("logits", "argmax", "gap", "attn"):
        a, b = to_np(getattr(bp, name)), to_np(getattr(br, name))
        np.testing.assert_array_equal(a.view(np.uint8), b.view(np.uint8), err_msg=name)


# ---------------------------------------------------------------------------
# a row's results do not depend on the other rows of the pass
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dims", ["tiny", "mid"])
def test_rows_independent_of_the_rest_of_the_pass(gpu, dims):
    d = {"tiny": synth.TINY, "mid": synth.MID}[dims]
    model = synth.gen_model(d, 90)
    dm = DeviceModel.from_host(model)
    big = synth.tree_spine_random(32, 6, d.vocab, 91)
    small = synth.Tree(big.parent[:8].copy(), big.token[:8].copy())   # a prefix of a parent-before-child array
    cache = synth.gen_cache(d, 333, 400, 92)
    _, b_small = gpu_verify(dm, [(cache, small)])
    _, b_big = gpu_verify(dm, [(cache, big)])
    other = (synth.gen_cache(d, 150, 200, 93), synth.tree_star(24, d.vocab, 94))
    _, b_joint = gpu_verify(dm, [other, (cache, small)])
    ref = to_np(b_small.logits)
    np.testing.assert_array_equal(to_np(b_big.logits)[:8], ref)
    np.testing.assert_array_equal(to_np(b_joint.logits)[24:], ref)
    np.testing.assert_array_equal(to_np(b_big.argmax)[:8], to_np(b_small.argmax))
    np.testing.assert_array_equal(to_np(b_joint.attn)[24:], to_np(b_small.attn))


# ---------------------------------------------------------------------------
# greedy round: verify -> accept -> commit, with planted drafts
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dims,seed", [("tiny", 0), ("tiny", 1), ("tiny", 2), ("mid", 3)])
def test_greedy_round_parity(gpu, dims, seed):
    d = {"tiny": synth.TINY, "mid": synth.MID}[dims]
    model = synth.gen_model(d, 300 + seed, random_gains=True)
    ctx = 64 if dims == "tiny" else 700
    cache = synth.gen_cache(d, ctx, ctx + 40, 301 + seed)
    tree = synth.tree_lattice(16, 7, d.vocab, 302 + seed)
    plant_spine(model, cache, tree, depth=2 + seed)     # accept a few spine nodes
    dm = DeviceModel.from_host(model)
    orc, reqs, b, _ = check_verify(model, [(cache, tree)], dm=dm)
    _ok(dv.accept_greedy(reqs, b), "tv_accept_greedy")
    _ok(dv.commit(reqs, b), "tv_commit_kv")
    torch.cuda.synchronize()
    assert int(b.status.item()) == 0
    path, out = greedy_replay(tree.parent, tree.token, orc[0]["logits"], to_np(b.argmax))
    a = len(path) - 1
    assert int(b.accept_len[0]) == a
    assert to_np(b.path)[: a + 1].tolist() == path
    assert to_np(b.out_tokens)[: a + 1].tolist() == out
    assert to_np(b.committed_src)[: a + 1].tolist() == [ctx + p for p in path]
    assert int(b.new_ctx[0]) == ctx + a + 1
    assert a >= 1, "planted drafts were not accepted"
    # committed rows: slot ctx + d holds the oracle's K/V of path node d
    k, v = to_np(reqs[0].k), to_np(reqs[0].v)
    for dd, node in enumerate(path):
        check_close_bf16(orc[0]["k"][node], k[:, ctx + dd, :].reshape(-1), KV_TOL, "committed K", relative=True)
        check_close_bf16(orc[0]["v"][node], v[:, ctx + dd, :].reshape(-1), KV_TOL, "committed V", relative=True)
    np.testing.assert_array_equal(k[:, :ctx], cache.k[:, :ctx])


def test_greedy_joint_round(gpu):
    d = synth.TINY
    model = synth.gen_model(d, 400, random_gains=True)
    host = []
    for i in range(4):
        c = synth.gen_cache(d, 50 + 7 * i, 100, 401 + i)
        t = synth.tree_lattice(8, 7, d.vocab, 402 + i)
        plant_spine(model, c, t, depth=i + 1)
        host.append((c, t))
    dm = DeviceModel.from_host(model)
    orc, reqs, b, _ = check_verify(model, host, dm=dm)
    _ok(dv.accept_greedy(reqs, b))
    _ok(dv.commit(reqs, b))
    torch.cuda.synchronize()
    assert int(b.status.item()) == 0
    off = 0
    for r, ((c, t), o) in enumerate(zip(host, orc)):
        path, out = greedy_replay(t.parent, t.token, o["logits"], to_np(b.argmax)[off:off + t.n])
        a = len(path) - 1
        assert int(b.accept_len[r]) == a
        assert to_np(b.path)[off:off + a + 1].tolist() == path
        assert to_np(b.out_tokens)[off:off + a + 1].tolist() == out
        assert to_np(b.committed_src)[off:off + a + 1].tolist() == [c.ctx_len + p for p in path]
        assert int(b.new_ctx[r]) == c.ctx_len + a + 1
        off += t.n


@pytest.mark.parametrize("dims", ["tiny", "mid"])
def test_fused_greedy_commit_equals_the_two_calls(gpu, dims):
    """tv_accept_greedy_commit gives the bits of tv_accept_greedy followed by
    tv_commit_kv: walk outputs and every cache row."""
    d = {"tiny": synth.TINY, "mid": synth.MID}[dims]
    model = synth.gen_model(d, 450, random_gains=True)
    host = []
    for i in range(3):
        c = synth.gen_cache(d, 60 + 11 * i, 140, 451 + i)
        t = synth.tree_lattice(8 + 2 * i, 7, d.vocab, 452 + i)   # 30 rows in all
        plant_spine(model, c, t, depth=i + 1)
        host.append((c, t))
    dm = DeviceModel.from_host(model)
    reqs_a, b_a = gpu_verify(dm, host)
    reqs_b, b_b = gpu_verify(dm, host)
    _ok(dv.accept_greedy(reqs_a, b_a))
    _ok(dv.commit(reqs_a, b_a))
    _ok(dv.accept_greedy_commit(reqs_b, b_b))
    torch.cuda.synchronize()
    assert int(b_a.status.item()) == 0 and int(b_b.status.item()) == 0
    rows = sum(t.n for _, t in host)
    off = 0
    for r, (_, t) in enumerate(host):
        a = int(b_a.accept_len[r])
        assert int(b_b.accept_len[r]) == a and a >= 1
        for name in ("path", "out_tokens", "committed_src"):
            assert to_np(getattr(b_a, name))[off:off + a + 1].tolist() == to_np(getattr(b_b, name))[off:off + a + 1].tolist(), name
        off += t.n
    assert to_np(b_a.new_ctx).tolist() == to_np(b_b.new_ctx).tolist()
    for ra, rb in zip(reqs_a, reqs_b):
        np.testing.assert_array_equal(to_np(ra.k).view(np.uint16), to_np(rb.k).view(np.uint16))
        np.testing.assert_array_equal(to_np(ra.v).view(np.uint16), to_np(rb.v).view(np.uint16))
    assert rows == off


def test_fused_greedy_commit_reports_a_bad_tree(gpu):
    d = synth.TINY
    model = synth.gen_model(d, 460, random_gains=True)
    cache = synth.gen_cache(d, 40, 80, 461)
    tree = synth.tree_lattice(8, 7, d.vocab, 462)
    dm = DeviceModel.from_host(model)
    reqs, b = gpu_verify(dm, [(cache, tree)])
    k0, v0 = reqs[0].k.clone(), reqs[0].v.clone()
    reqs[0].parent[3] = 5   # parent after child: not in [0, 3)
    _ok(dv.accept_greedy_commit(reqs, b))
    torch.cuda.synchronize()
    assert int(b.status.item()) == abi.CODES["TV_E_ORDER"]
    assert torch.equal(reqs[0].k, k0) and torch.equal(reqs[0].v, v0)   # nothing committed


# ---------------------------------------------------------------------------
# accept walks on given logits (both sides read the same inputs)
# ---------------------------------------------------------------------------
def _walk_inputs(V, n_req, seed, n_each=8, scale=2.0):
    trees = []
    for i in range(n_req):
        t = synth.tree_lattice(n_each, 7, V, seed + i) if i % 2 == 0 else synth.tree_spine_random(
            n_each, 3, V, seed + i)
        trees.append(t)
    rows = sum(t.n for t in trees)
    logits = synth.logits_rows(rows, V, seed + 100, scale=scale)
    # make drafts plausible: each non-root node's token is one of its parent row's best tokens
    rng = np.random.default_rng(seed)
    off = 0
    for t in trees:
        for c in range(1, t.n):
            row = logits[off + t.parent[c]]
            logits[off + t.parent[c], t.token[c]] = row.max() + float(rng.uniform(-1.0, 0.5))
        off += t.n
    return trees, logits


def _device_walk_setup(V, trees, logits):
    d = synth.Dims(hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64, vocab=V)
    reqs = [DeviceRequest(torch.zeros(2, 1, 64, device="cuda", dtype=torch.bfloat16),
                          torch.zeros(2, 1, 64, device="cuda", dtype=torch.bfloat16), 0,
                          torch.from_numpy(t.parent).cuda(), torch.from_numpy(t.token).cuda()) for t in trees]
    b = RoundBuffers.alloc(d, sum(t.n for t in trees), len(trees), 0)
    b.logits.copy_(torch.from_numpy(logits))
    return reqs, b


@pytest.mark.parametrize("V,seed", [(1024, 0), (5003, 1), (151936, 2)])
def test_greedy_walk_on_given_argmax(gpu, V, seed):
    trees, logits = _walk_inputs(V, 4, 700 + seed)
    reqs, b = _device_walk_setup(V, trees, logits)
    am = np.argmax(logits, axis=1).astype(np.int32)
    b.argmax.copy_(torch.from_numpy(am))
    _ok(dv.accept_greedy(reqs, b))
    torch.cuda.synchronize()
    assert int(b.status.item()) == 0
    off = 0
    for r, t in enumerate(trees):
        path, out = oracle.accept_greedy(t.parent, t.token, am[off:off + t.n])
        a = len(path) - 1
        assert int(b.accept_len[r]) == a
        assert to_np(b.path)[off:off + a + 1].tolist() == path
        assert to_np(b.out_tokens)[off:off + a + 1].tolist() == out
        off += t.n


@pytest.mark.parametrize("V,T,bonus,seed", [(1024, 1.0, True, 0), (5003, 0.7, True, 1), (151936, 1.0, True, 2),
                                            (1024, 1.3, False, 3), (151936, 0.8, False, 4)])
def test_residual_walk_on_given_logits(gpu, V, T, bonus, seed):
    trees, logits = _walk_inputs(V, 4, 800 + seed, n_each=8)
    reqs, b = _device_walk_setup(V, trees, logits)
    total = sum(t.n for t in trees)
    replays = 0
    for trial in range(6):
        u = synth.uniforms(total, 900 + 31 * seed + trial)
        b.uniforms.copy_(torch.from_numpy(u))
        b.status.zero_()
        _ok(dv.accept_residual(reqs, b, T, bonus_at_leaf=bonus))
        torch.cuda.synchronize()
        assert int(b.status.item()) == 0
        off = 0
        for r, t in enumerate(trees):
            cnt = int(b.out_count[r])
            a = int(b.accept_len[r])
            gpu_path = to_np(b.path)[off:off + a + 1].tolist()
            gpu_out = to_np(b.out_tokens)[off:off + cnt].tolist()
            path, out, rep = oracle.accept_residual(t.parent, t.token, logits[off:off + t.n], T, u[off:off + t.n],
                                                    bonus_at_leaf=bonus, replay=(gpu_path, gpu_out), eps=1e-5)
            replays += rep
            assert gpu_path == path and gpu_out == out, (r, trial)
            off += t.n
    assert replays <= 2


def test_residual_walk_law_on_gpu(gpu):
    """The GPU walk reproduces p too: first-token histogram over many seeded
    rounds on a 16-token vocabulary, within 5 sigma."""
    V, T = 16, 1.0
    tree = synth.tree_star(5, V, 3)
    rng = np.random.default_rng(5)
    logits = (rng.standard_normal((5, V)) * 1.5).astype(np.float32)
    reqs, b = _device_walk_setup(V, [tree], logits)
    p = oracle.softmax_t(logits[0], T)
    rounds = 4000
    counts = np.zeros(V)
    us = synth.uniforms(rounds * 5, 17).reshape(rounds, 5)
    for i in range(rounds):
        b.uniforms.copy_(torch.from_numpy(us[i]))
        _ok(dv.accept_residual(reqs, b, T))
        counts[int(b.out_tokens[0])] += 1
    assert int(b.status.item()) == 0
    sd = np.sqrt(rounds * p * (1 - p))
    assert np.all(np.abs(counts - rounds * p) <= 5 * sd + 1)


# ---------------------------------------------------------------------------
# sampled round end to end (oracle logits vs GPU logits: wider replay window)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("seed", range(3))
def test_residual_round_parity(gpu, seed):
    d = synth.TINY
    model = synth.gen_model(d, 500 + seed, random_gains=True)
    cache = synth.gen_cache(d, 64, 100, 501 + seed)
    tree = synth.tree_lattice(16, 7, d.vocab, 502 + seed)
    plant_spine(model, cache, tree, depth=3)
    dm = DeviceModel.from_host(model)
    orc, reqs, b, _ = check_verify(model, [(cache, tree)], dm=dm)
    u = synth.uniforms(tree.n, 503 + seed)
    b.uniforms.copy_(torch.from_numpy(u))
    _ok(dv.accept_residual(reqs, b, 1.0))
    _ok(dv.commit(reqs, b))
    torch.cuda.synchronize()
    assert int(b.status.item()) == 0
    a, cnt = int(b.accept_len[0]), int(b.out_count[0])
    gpu_path = to_np(b.path)[: a + 1].tolist()
    gpu_out = to_np(b.out_tokens)[:cnt].tolist()
    path, out, rep = oracle.accept_residual(tree.parent, tree.token, orc[0]["logits"], 1.0, u,
                                            replay=(gpu_path, gpu_out), eps=2e-3)
    assert gpu_path == path and gpu_out == out
    assert to_np(b.committed_src)[: a + 1].tolist() == [64 + p for p in path]


# ---------------------------------------------------------------------------
# device-side validation and the sticky status word
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("case,code", [("order", "TV_E_ORDER"), ("root", "TV_E_ORDER"),
                                       ("dup", "TV_E_DUP_SIBLING"), ("token", "TV_E_TOKEN")])
def test_verify_rejects_bad_trees(gpu, case, code):
    d = synth.TINY
    model = synth.gen_model(d, 1)
    dm = DeviceModel.from_host(model)
    tree = synth.tree_spine_random(8, 4, d.vocab, 2)
    if case == "order":
        tree.parent[5] = 6
    elif case == "root":
        tree.parent[0] = 0
    elif case == "dup":
        tree.parent[6] = tree.parent[5]
        tree.token[6] = tree.token[5]
    else:
        tree.token[3] = d.vocab
    assert oracle.validate(tree.parent, tree.token, d.vocab) == code[5:].lower()
    cache = synth.gen_cache(d, 64, 96, 3)
    req = DeviceRequest.from_host(cache, tree)
    b = RoundBuffers.alloc(d, 8, 1, 64)
    b.logits.fill_(7.0)
    _ok(dv.verify(dm, [req], b))
    _ok(dv.accept_greedy([req], b))
    _ok(dv.commit([req], b))
    torch.cuda.synchronize()
    assert abi.STATUS[int(b.status.item())] == code
    # nothing ran after the prologue: outputs and cache untouched
    assert bool((b.logits == 7.0).all())
    np.testing.assert_array_equal(to_np(req.k), cache.k)
    assert int(b.accept_len[0]) == 0 and int(b.new_ctx[0]) == 0


@pytest.mark.parametrize("bad", [float("nan"), 1.0, -0.25, float("inf")])
def test_residual_rejects_bad_uniforms(gpu, bad):
    V = 1024
    trees, logits = _walk_inputs(V, 1, 11)
    reqs, b = _device_walk_setup(V, trees, logits)
    u = synth.uniforms(trees[0].n, 12)
    u[trees[0].n - 1] = bad      # even a draw the walk may never reach
    assert oracle.validate_sampling(u, 1.0) == "uniform"
    b.uniforms.copy_(torch.from_numpy(u))
    _ok(dv.accept_residual(reqs, b, 1.0))
    torch.cuda.synchronize()
    assert abi.STATUS[int(b.status.item())] == "TV_E_UNIFORM"


def test_commit_rejects_bad_path(gpu):
    d = synth.TINY
    cache = synth.gen_cache(d, 10, 40, 1)
    tree = synth.tree_chain(4, d.vocab, 2)
    req = DeviceRequest.from_host(cache, tree)
    b = RoundBuffers.alloc(d, 4, 1, 10)
    for accept, path in ((4, [0, 1, 2, 3]), (1, [0, 9, 0, 0]), (1, [1, 2, 0, 0])):
        b.status.zero_()
        b.accept_len.fill_(accept)
        b.path.copy_(torch.tensor(path, dtype=torch.int32))
        _ok(dv.commit([req], b))
        torch.cuda.synchronize()
        assert abi.STATUS[int(b.status.item())] == "TV_E_PATH"
    np.testing.assert_array_equal(to_np(req.k), cache.k)


def test_commit_reads_before_writing(gpu):
    """path [0, 2, 3, 5]: slot ctx+2 is the source of step 1 and the target of step 2."""
    d = synth.TINY
    ctx = 5
    cache = synth.gen_cache(d, ctx, 20, 7)
    tree = synth.tree_chain(8, d.vocab, 8)
    req = DeviceRequest.from_host(cache, tree)
    b = RoundBuffers.alloc(d, 8, 1, ctx)
    path = [0, 2, 3, 5]
    b.accept_len.fill_(3)
    b.path[:4].copy_(torch.tensor(path, dtype=torch.int32))
    _ok(dv.commit([req], b))
    torch.cuda.synchronize()
    assert int(b.status.item()) == 0
    k2, v2, src, new_ctx = oracle.commit_kv(cache.k, cache.v, ctx, path)
    np.testing.assert_array_equal(to_np(req.k), k2)
    np.testing.assert_array_equal(to_np(req.v), v2)
    assert to_np(b.committed_src)[:4].tolist() == src and int(b.new_ctx[0]) == new_ctx
