"""GPU parity of the tree verify through a decoder-layer stack (Gated DeltaNet
and attention layers, each with a SwiGLU MLP) against oracle/stack.py, through
the C ABI (tv_verify_stack with its residual-stream taps, tv_accept_greedy,
tv_commit_stack).

Two comparisons, both element by element.

* Layer by layer (teacher-forced): the oracle runs every residual sublayer of
  every tree row from the GPU's own input to it (the taps) and the GPU's
  output must agree within one bf16 step: 1e-2 x max(1, |value|), as the
  single layer's K/V.  The same forcing gives the reference for each attention
  layer's tree K/V, for each DeltaNet layer's state after every node (and so
  for the commit), and for the logits, from the GPU's last residual stream:
  2e-2 x the row's RMS logit (the verify's stated bound).  The argmax, the
  greedy walk (near ties replayed) and the committed slots are compared on
  those.
* End to end: the oracle's own, fully independent pass.  Its logits differ from
  the GPU's by the bf16 rounding differences of every sublayer, carried through
  the rest of the stack.  With random weights the stack's wide projections
  carry a one-step difference of a few activations into many outputs, so the
  bound grows with the number S of residual sublayers: 2e-2 x sqrt(S) x the
  row's RMS logit (S = 1 is the single-layer bound).  This is derived from
  the arithmetic; the pages give no figure for a stack.
DeltaNet states after the commit: 1e-3 x (1 + |s|), an fp32 sum of at most 33
terms of O(1) against fp64.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import stack as OS
from speculative_tree_verify_gb300 import abi, synth
from speculative_tree_verify_gb300 import device as dv

from parity import KV_TOL, LOGIT_TOL, check_argmax, check_close_bf16, check_logits, greedy_replay, to_np

pytestmark = pytest.mark.gpu

STATE_TOL = 1e-3


def end_to_end_tol(sd) -> float:
    return LOGIT_TOL * float(np.sqrt(2 * sd.n_layers))


def _ok(rc, what):
    assert rc == abi.TV_OK, f"{what}: {abi.STATUS.get(rc, rc)}"


def _requests(sd, host_reqs, device="cuda"):
    """host_reqs: list of (caches per attention layer, states per DeltaNet layer, tree)."""
    reqs = []
    for caches, states, tree in host_reqs:
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)
        ks = [t(c.k) for c in caches]
        vs = [t(c.v) for c in caches]
        ctx = caches[0].ctx_len if caches else 0
        st = torch.from_numpy(np.stack(states).astype(np.float32)).to(device) if states else \
            torch.zeros(1, device=device)
        reqs.append(dv.StackRequest(ks, vs, ctx, st, torch.from_numpy(tree.parent.copy()).to(device),
                                    torch.from_numpy(tree.token.copy()).to(device)))
    return reqs


def teacher_forced(m, host_req, taps):
    """The oracle's sublayers run from the GPU's inputs (taps [2L + 1][n][H],
    bf16 bits of this request's rows).  Returns the worst sublayer error (in
    units of 1e-2 x max(1, |value|)), the logits from the GPU's last stream,
    per attention layer the tree K/V (bits [n][Hkv][D]) and per DeltaNet layer
    the state after every node."""
    sd = m.dims
    d = sd.base
    caches, states, tree = host_req
    parent, n = tree.parent, tree.n
    ctx = caches[0].ctx_len if caches else 0
    depth = np.zeros(n, np.int64)
    for i in range(1, n):
        depth[i] = depth[parent[i]] + 1
    T = oracle.bf16_to_f64(taps)
    worst = 0.0
    kv, st = [], []
    ia = idn = 0

    def cmp(ref, gpu_bits, what):
        nonlocal worst
        worst = max(worst, check_close_bf16(OS.round_bf16_bits(np.stack(ref)), gpu_bits, KV_TOL, what,
                                            relative=True) / KV_TOL)

    for l, lay in enumerate(m.layers):
        x_in = T[2 * l]
        h = [OS._rms_bf16(x_in[i], lay.ln_mix, d.rms_eps) for i in range(n)]
        if lay.attn:
            Kc, Vc = OS._cache_rows(caches[ia])
            fr = [OS.attn_front(lay, d, h[i], ctx + int(depth[i])) for i in range(n)]
            out = []
            for i in range(n):
                p = OS._path(parent, i)
                K = np.concatenate([Kc, np.stack([fr[a][1] for a in p])])
                V = np.concatenate([Vc, np.stack([fr[a][2] for a in p])])
                out.append(OS.attn_back(lay, OS.attend(d, fr[i][0], K, V), x_in[i]))
            kv.append((OS.round_bf16_bits(np.stack([f[1] for f in fr])), OS.round_bf16_bits(np.stack([f[2] for f in fr]))))
            ia += 1
        else:
            S0 = np.asarray(states[idn], np.float64)
            Sn, out = [None] * n, []
            for i in range(n):
                f = OS.dn_front(lay, sd, h[i])
                Sn[i], o = OS.dn_core(sd, S0 if parent[i] < 0 else Sn[parent[i]], f)
                out.append(OS.dn_back(lay, sd, o, f.z, x_in[i]))
            st.append(np.stack(Sn))
            idn += 1
        cmp(out, taps[2 * l + 1], f"layer {l} mixer")
        cmp([OS.mlp_block(lay, sd, T[2 * l + 1][i]) for i in range(n)], taps[2 * l + 2], f"layer {l} MLP")
    hf = np.stack([OS._rms_bf16(T[2 * sd.n_layers][i], m.ln_f, d.rms_eps) for i in range(n)])
    return worst, OS._logits(m, hf), kv, st


def run_and_check(m, dm, host_reqs):
    sd = m.dims
    H = sd.base.hidden
    reqs = _requests(sd, host_reqs)
    rows = sum(r.n for r in reqs)
    b = dv.StackBuffers.alloc(dm, rows, len(reqs))
    taps = torch.zeros(2 * sd.n_layers + 1, rows, H, device="cuda", dtype=torch.bfloat16)
    _ok(dv.verify_stack(dm, reqs, b, x_taps=taps), "tv_verify_stack")
    torch.cuda.synchronize()
    assert int(b.status.item()) == 0, abi.STATUS.get(int(b.status.item()))
    taps_h = to_np(taps)
    tf, off = [], 0
    for hr, r in zip(host_reqs, reqs):
        tf.append(teacher_forced(m, hr, taps_h[:, off:off + r.n]))
        off += r.n
    logits_tf = np.concatenate([t[1] for t in tf])
    stats = {"sublayer_err_steps": max(t[0] for t in tf),
             "logit_err": check_logits(logits_tf, to_np(b.logits)),
             "swapped": check_argmax(logits_tf, to_np(b.argmax), to_np(b.gap))}
    # end to end: the oracle's own pass
    e2e = np.concatenate([OS.verify_stack(m, c, s_, t.parent, t.token)["logits"] for c, s_, t in host_reqs])
    stats["e2e_logit_err"] = check_logits(e2e, to_np(b.logits), end_to_end_tol(sd))
    kv_err = 0.0
    for (caches, states, tree), t, r in zip(host_reqs, tf, reqs):
        n = tree.n
        for j, c in enumerate(caches):
            ctx = c.ctx_len
            k, v = to_np(r.ks[j]), to_np(r.vs[j])
            kv_err = max(kv_err, check_close_bf16(t[2][j][0].reshape(n, -1),
                                                  k[:, ctx:ctx + n, :].transpose(1, 0, 2).reshape(n, -1), KV_TOL,
                                                  f"layer {j} tree K", relative=True))
            kv_err = max(kv_err, check_close_bf16(t[2][j][1].reshape(n, -1),
                                                  v[:, ctx:ctx + n, :].transpose(1, 0, 2).reshape(n, -1), KV_TOL,
                                                  f"layer {j} tree V", relative=True))
            np.testing.assert_array_equal(k[:, :ctx], c.k[:, :ctx])
            np.testing.assert_array_equal(k[:, ctx + n:], c.k[:, ctx + n:])
    stats["kv_err"] = kv_err
    # greedy walk and commit on the GPU, the oracle walk replaying near ties
    _ok(abi.tv_accept_greedy([r.tree() for r in reqs], b.argmax, b.path, b.accept_len, b.out_tokens, b.status),
        "tv_accept_greedy")
    _ok(dv.commit_stack(dm, reqs, b), "tv_commit_stack")
    torch.cuda.synchronize()
    assert int(b.status.item()) == 0, abi.STATUS.get(int(b.status.item()))
    off = 0
    st_err = 0.0
    for ri, ((caches, states, tree), t, r) in enumerate(zip(host_reqs, tf, reqs)):
        n = tree.n
        path, out = greedy_replay(tree.parent, tree.token, t[1], to_np(b.argmax)[off:off + n])
        a = len(path) - 1
        assert int(b.accept_len[ri]) == a
        assert to_np(b.path)[off:off + a + 1].tolist() == path
        assert to_np(b.out_tokens)[off:off + a + 1].tolist() == out
        for j, c in enumerate(caches):
            ctx = c.ctx_len
            assert int(b.new_ctx[ri]) == ctx + a + 1
            assert to_np(b.committed_src)[off:off + a + 1].tolist() == [ctx + p for p in path]
            gk, gv = to_np(r.ks[j]), to_np(r.vs[j])
            np.testing.assert_array_equal(gk[:, :ctx], c.k[:, :ctx])
            for dd, node in enumerate(path):
                check_close_bf16(t[2][j][0][node].reshape(-1), gk[:, ctx + dd, :].reshape(-1), KV_TOL, "committed K",
                                 relative=True)
                check_close_bf16(t[2][j][1][node].reshape(-1), gv[:, ctx + dd, :].reshape(-1), KV_TOL, "committed V",
                                 relative=True)
        gs = r.states.cpu().numpy().astype(np.float64)
        for ld, node_states in enumerate(t[3]):
            keep = node_states[path[-1]]
            st_err = max(st_err, float((np.abs(gs[ld] - keep) / (1.0 + np.abs(keep))).max()))
        off += n
    stats["state_err"] = st_err
    assert st_err <= STATE_TOL, f"DeltaNet state after commit: error {st_err:.3e} > {STATE_TOL}"
    return stats


def _host(sd, m, ctxs, trees, seed):
    out = []
    for i, (ctx, tree) in enumerate(zip(ctxs, trees)):
        caches = [synth.gen_cache(sd.base, ctx, ctx + 40, seed + 10 * i + j) for j in range(len(sd.attn_layers))]
        out.append((caches, synth.gen_dn_states(sd, seed + 100 + i), tree))
    return out


@pytest.fixture(scope="module")
def tiny(gpu):
    sd = synth.STACK_TINY
    m = synth.gen_stack(sd, 21, random_gains=True)
    return sd, m, dv.DeviceStack.from_host(m)


@pytest.mark.parametrize("shape", ["lattice", "random", "star", "chain", "single"])
def test_stack_tiny_parity(tiny, shape):
    sd, m, dm = tiny
    V = sd.base.vocab
    tree = {"lattice": synth.tree_lattice(12, 5, V, 1), "random": synth.tree_spine_random(11, 4, V, 2),
            "star": synth.tree_star(7, V, 3), "chain": synth.tree_chain(6, V, 4),
            "single": synth.tree_chain(1, V, 5)}[shape]
    stats = run_and_check(m, dm, _host(sd, m, [40], [tree], 300))
    print(f"stack {sd.n_layers} layers, hidden {sd.base.hidden}, {shape}:", stats)


def test_stack_tiny_joint_and_ragged_context(tiny):
    sd, m, dm = tiny
    V = sd.base.vocab
    trees = [synth.tree_lattice(9, 4, V, 7), synth.tree_spine_random(8, 3, V, 8), synth.tree_chain(5, V, 9)]
    stats = run_and_check(m, dm, _host(sd, m, [0, 77, 130], trees, 400))
    print("stack joint:", stats)


def test_stack_32_rows_dk128(gpu):
    # DeltaNet heads of 128 and a 32-row tree: the state loaded before the
    # programmatic-launch wait lands in both staging waves of the verify core
    sd = synth.StackDims(base=synth.MID, n_layers=4, attn_every=4, n_k_heads=2, n_v_heads=4, d_k=128, d_v=128,
                         intermediate=1024)
    m = synth.gen_stack(sd, 33, random_gains=True)
    dm = dv.DeviceStack.from_host(m)
    stats = run_and_check(m, dm, _host(sd, m, [96], [synth.tree_lattice(32, 15, sd.base.vocab, 13)], 800))
    print("stack hidden 512, DeltaNet heads of 128, 32 rows:", stats)


def test_stack_packed_equals_row_major(tiny):
    sd, m, dm = tiny
    assert dm.packed
    rm = dv.DeviceStack.from_host(m, packed=False)
    host = _host(sd, m, [64], [synth.tree_lattice(12, 5, sd.base.vocab, 11)], 500)
    outs = []
    for model in (dm, rm):
        reqs = _requests(sd, host)
        b = dv.StackBuffers.alloc(model, 12, 1)
        _ok(dv.verify_stack(model, reqs, b), "tv_verify_stack")
        torch.cuda.synchronize()
        outs.append((to_np(b.logits), to_np(b.argmax)))
    np.testing.assert_array_equal(outs[0][0].view(np.uint32), outs[1][0].view(np.uint32))
    np.testing.assert_array_equal(outs[0][1], outs[1][1])


def test_stack_rejects_bad_trees_and_bad_layers(tiny):
    sd, m, dm = tiny
    V = sd.base.vocab
    host = _host(sd, m, [16], [synth.tree_chain(4, V, 3)], 600)
    reqs = _requests(sd, host)
    b = dv.StackBuffers.alloc(dm, 4, 1)
    reqs[0].parent[2] = 3                     # a parent after its child
    _ok(dv.verify_stack(dm, reqs, b), "tv_verify_stack")
    torch.cuda.synchronize()
    assert abi.STATUS[int(b.status.item())] == "TV_E_ORDER"
    bad = abi.TvLayer(dm.c_layers[0].kind)    # null weights
    layers = (abi.TvLayer * 1)(bad)
    st = abi.TvStack(dm.c.dims, dm.c.dn, dm.c.intermediate, 1, layers, dm.c.embed, dm.c.ln_f, dm.c.lm_head, 1)
    rc, _ = abi.tv_stack_workspace_size(st)
    assert abi.STATUS[rc] == "TV_E_ARG"


# hidden 5120: 40/8 attention heads of 128, 16/32 DeltaNet heads of 128, vocab
# 151936; four layers (three DeltaNet, one attention) with the full MLP width
STACK_5120 = synth.StackDims(base=synth.FULL, n_layers=4, attn_every=4, n_k_heads=16, n_v_heads=32, d_k=128,
                             d_v=128, intermediate=17408)


def test_stack_hidden5120_parity(gpu):
    sd = STACK_5120
    m = synth.gen_stack(sd, 2027)
    dm = dv.DeviceStack.from_host(m)
    trees = [synth.tree_lattice(16, 7, sd.base.vocab, 12)]
    stats = run_and_check(m, dm, _host(sd, m, [1024], trees, 700))
    print("stack hidden 5120, 4 layers, 16 rows:", stats)
