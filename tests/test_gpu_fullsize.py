"""GPU parity at the hidden-5120 shapes: 40 query / 8 KV heads of 128, vocab
151936, bf16 weights ~ N(0, 0.02).  The oracle computes every output of these
rounds in full (fp64, OpenMP over independent outputs), so the comparison is
element by element, not sampled.

  * one verify at 1k context with a 16-row lattice tree, planted drafts,
    greedy accept and commit;
  * the row sweep 8 / 16 / 24 / 32 at 1k context (spine of 15 + branches);
  * 32k context with a 32-row lattice tree (15 slots x 16 candidates),
    residual sampling at temperature 1 and commit;
  * joint verify: 2 requests x 16 rows and 4 x 8, contexts in 1024..8192.

The launch configuration is the one the benchmark times: same entry points,
same shapes, the same kernels.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_tree_verify_gb300 import synth
from speculative_tree_verify_gb300 import device as dv
from speculative_tree_verify_gb300.device import DeviceModel

from parity import KV_TOL, _ok, check_close_bf16, check_verify, gpu_verify, greedy_replay, plant_spine, to_np

pytestmark = pytest.mark.gpu

D = synth.FULL


@pytest.fixture(scope="module")
def full_model(gpu):
    model = synth.gen_model(D, 2026)
    return model, DeviceModel.from_host(model)


def test_hidden5120_greedy_round(full_model):
    model, dm = full_model
    ctx = 1024
    cache = synth.gen_cache(D, ctx, ctx + 64, 11)
    tree = synth.tree_lattice(16, 7, D.vocab, 12)
    plant_spine(model, cache, tree, depth=4)
    orc, reqs, b, stats = check_verify(model, [(cache, tree)], dm=dm)
    print("hidden-5120, 16 rows:", stats)
    _ok(dv.accept_greedy(reqs, b))
    _ok(dv.commit(reqs, b))
    torch.cuda.synchronize()
    assert int(b.status.item()) == 0
    path, out = greedy_replay(tree.parent, tree.token, orc[0]["logits"], to_np(b.argmax))
    a = len(path) - 1
    assert a >= 1
    assert int(b.accept_len[0]) == a
    assert to_np(b.path)[: a + 1].tolist() == path
    assert to_np(b.out_tokens)[: a + 1].tolist() == out
    assert to_np(b.committed_src)[: a + 1].tolist() == [ctx + p for p in path]
    k = to_np(reqs[0].k)
    for dd, node in enumerate(path):
        check_close_bf16(orc[0]["k"][node], k[:, ctx + dd, :].reshape(-1), KV_TOL, "committed K", relative=True)


def test_hidden5120_packed_weights_equal_row_major(full_model):
    """The tile-packed head / QKV / O weights the benchmark streams give the
    same bits as the row-major matrices."""
    model, dm = full_model
    assert dm.packed
    rm = DeviceModel(dm.dims, dm.t, packed=False)
    host = [(synth.gen_cache(D, 1024, 1100, 21), synth.tree_lattice(16, 7, D.vocab, 22))]
    _, bp = gpu_verify(dm, host)
    _, br = gpu_verify(rm, host)
    for name in ("logits", "argmax", "gap", "attn"):
        np.testing.assert_array_equal(to_np(getattr(bp, name)).view(np.uint8), to_np(getattr(br, name)).view(np.uint8),
                                      err_msg=name)


def test_hidden5120_fused_walk_commit_equals_the_two_calls(full_model):
    """The benchmark's round commits with tv_accept_greedy_commit: the same
    walk outputs and cache rows as tv_accept_greedy then tv_commit_kv."""
    model, dm = full_model
    cache = synth.gen_cache(D, 1024, 1100, 31)
    tree = synth.tree_lattice(16, 7, D.vocab, 32)
    plant_spine(model, cache, tree, depth=4)
    reqs_a, b_a = gpu_verify(dm, [(cache, tree)])
    reqs_b, b_b = gpu_verify(dm, [(cache, tree)])
    _ok(dv.accept_greedy(reqs_a, b_a))
    _ok(dv.commit(reqs_a, b_a))
    _ok(dv.accept_greedy_commit(reqs_b, b_b))
    torch.cuda.synchronize()
    assert int(b_a.status.item()) == 0 and int(b_b.status.item()) == 0
    a = int(b_a.accept_len[0])
    assert a >= 1 and int(b_b.accept_len[0]) == a
    for name in ("path", "out_tokens", "committed_src"):
        assert to_np(getattr(b_a, name))[: a + 1].tolist() == to_np(getattr(b_b, name))[: a + 1].tolist(), name
    assert int(b_a.new_ctx[0]) == int(b_b.new_ctx[0]) == 1024 + a + 1
    np.testing.assert_array_equal(to_np(reqs_a[0].k).view(np.uint16), to_np(reqs_b[0].k).view(np.uint16))
    np.testing.assert_array_equal(to_np(reqs_a[0].v).view(np.uint16), to_np(reqs_b[0].v).view(np.uint16))


@pytest.mark.parametrize("n", [8, 16, 24, 32])
def test_hidden5120_row_sweep(full_model, n):
    model, dm = full_model
    cache = synth.gen_cache(D, 1024, 1100, 20 + n)
    tree = synth.tree_spine_random(n, min(16, n), D.vocab, 30 + n)
    orc, reqs, b, stats = check_verify(model, [(cache, tree)], dm=dm)
    print(f"hidden-5120, {n} rows:", stats)
    _ok(dv.accept_greedy(reqs, b))
    torch.cuda.synchronize()
    path, out = greedy_replay(tree.parent, tree.token, orc[0]["logits"], to_np(b.argmax))
    assert to_np(b.path)[: len(path)].tolist() == path
    assert to_np(b.out_tokens)[: len(out)].tolist() == out


def test_hidden5120_long_context_sampled(full_model):
    model, dm = full_model
    ctx = 32768
    cache = synth.gen_cache(D, ctx, ctx + 32, 40)
    tree = synth.tree_lattice(32, 15, D.vocab, 41)
    plant_spine(model, cache, tree, depth=2)
    orc, reqs, b, stats = check_verify(model, [(cache, tree)], dm=dm)
    print("hidden-5120, 32k context, 32 rows:", stats)
    u = synth.uniforms(tree.n, 42)
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
    assert to_np(b.committed_src)[: a + 1].tolist() == [ctx + p for p in path]
    assert int(b.new_ctx[0]) == ctx + a + 1


@pytest.mark.parametrize("layout", [(16, 16), (8, 8, 8, 8)])
def test_hidden5120_joint_verify(full_model, layout):
    model, dm = full_model
    ctxs = synth.joint_contexts(len(layout), 50 + len(layout))
    host = [(synth.gen_cache(D, c, c + n + 8, 60 + i), synth.tree_lattice(n, 7, D.vocab, 70 + i))
            for i, (c, n) in enumerate(zip(ctxs, layout))]
    orc, reqs, b, stats = check_verify(model, host, dm=dm)
    print("hidden-5120 joint", layout, stats)
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
        assert int(b.new_ctx[r]) == c.ctx_len + a + 1
        off += t.n
