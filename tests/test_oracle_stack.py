"""Pins of oracle/stack.py (the tree verify through a stack of Gated DeltaNet
and attention layers, each with an MLP) to what does not come from the oracle
itself:

* brute force: every tree row equals plain one-token-at-a-time decoding of its
  own root path through the stack, to the last bit -- logits, the K/V each
  attention layer writes, the state each DeltaNet layer reaches (the tree form
  attends to ancestors only and steps each node from its parent's state; the
  plain decoder appends and steps in sequence);
* on chains, an independent torch-fp64 stack: ``F.rms_norm``, ``F.linear``,
  complex-exponential RoPE, ``F.scaled_dot_product_attention`` with a causal
  mask over cache + chain, the Gated DeltaNet layer from the pages' closed form
  (the pseudo-values of an ancestor-masked -- here lower-triangular -- solve,
  ``torch.linalg.solve_triangular``, no recurrence), ``F.silu``/``F.softplus``;
* the commit keeps exactly what decoding the accepted path leaves: its K/V rows
  in every attention layer and its state in every DeltaNet layer.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import stack as ST
from speculative_tree_verify_gb300 import synth


def _setup(seed, ctx=40, cap=80, sd=synth.STACK_TINY, random_gains=True):
    m = synth.gen_stack(sd, seed, random_gains=random_gains)
    caches = [synth.gen_cache(sd.base, ctx, cap, 100 * seed + l) for l in range(len(sd.attn_layers))]
    states = synth.gen_dn_states(sd, seed + 1)
    return m, caches, states


@pytest.mark.parametrize("shape", ["lattice", "random", "star", "chain"])
def test_tree_rows_equal_sequential_decode(shape):
    m, caches, states = _setup(3)
    V = m.dims.base.vocab
    tree = {"lattice": synth.tree_lattice(12, 5, V, 1), "random": synth.tree_spine_random(11, 4, V, 2),
            "star": synth.tree_star(7, V, 3), "chain": synth.tree_chain(6, V, 4)}[shape]
    res = ST.verify_stack(m, caches, states, tree.parent, tree.token)
    for i in range(tree.n):
        p = ST._path(tree.parent, i)
        dec = ST.decode_stack(m, caches, states, [int(tree.token[a]) for a in p])
        assert np.array_equal(dec["logits"][-1], res["logits"][i]), f"logits of row {i}"
        assert np.array_equal(dec["hf"][-1], res["hf"][i])
        for la in range(len(caches)):
            assert np.array_equal(dec["k"][la][-1], res["k"][la][i]) and np.array_equal(dec["v"][la][-1], res["v"][la][i])
        for ld in range(len(states)):
            assert np.array_equal(dec["states"][ld][-1], res["states"][ld][i])


def test_empty_context_and_single_row():
    m, caches, states = _setup(5, ctx=0, cap=8)
    tree = synth.tree_chain(1, m.dims.base.vocab, 9)
    res = ST.verify_stack(m, caches, states, tree.parent, tree.token)
    dec = ST.decode_stack(m, caches, states, [int(tree.token[0])])
    assert np.array_equal(res["logits"], dec["logits"])


# ---- the independent torch-fp64 stack ------------------------------------------------
def _t(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(torch.float64)


def _r(t):
    return t.to(torch.float32).to(torch.bfloat16).to(torch.float64)


def _rope_complex(x, pos, theta):
    """x [n][heads][D]; pairs (d, d + D/2) as complex numbers times e^(i pos w_d)."""
    D = x.shape[-1]
    w = theta ** (-2.0 * torch.arange(D // 2, dtype=torch.float64) / D)
    rot = torch.polar(torch.ones(len(pos), D // 2, dtype=torch.float64), pos[:, None] * w[None, :])
    z = torch.complex(x[..., :D // 2], x[..., D // 2:]) * rot[:, None, :]
    return torch.cat([z.real, z.imag], dim=-1)


def torch_chain(m, caches, states, tokens):
    sd = m.dims
    d = sd.base
    H, Hq, Hkv, D, eps = d.hidden, d.n_q_heads, d.n_kv_heads, d.head_dim, d.rms_eps
    Hk, Hv, dk, dv, I = sd.n_k_heads, sd.n_v_heads, sd.d_k, sd.d_v, sd.intermediate
    n = len(tokens)
    ctx = caches[0].ctx_len
    pos = torch.arange(ctx, ctx + n, dtype=torch.float64)
    x = _t(m.embed)[torch.tensor(tokens)]
    ia = idn = 0
    kept_states = []
    for lay in m.layers:
        h = _r(F.rms_norm(x, (H,), _t(lay.ln_mix), eps))
        if lay.attn:
            y = F.linear(h, _t(lay.wqkv))
            q = _r(_rope_complex(y[:, :Hq * D].view(n, Hq, D), pos, d.rope_theta))
            k = _r(_rope_complex(y[:, Hq * D:(Hq + Hkv) * D].view(n, Hkv, D), pos, d.rope_theta))
            v = _r(y[:, (Hq + Hkv) * D:].view(n, Hkv, D))
            c = caches[ia]
            K = torch.cat([_t(c.k[:, :ctx]), k.transpose(0, 1)], dim=1).repeat_interleave(Hq // Hkv, dim=0)
            Vv = torch.cat([_t(c.v[:, :ctx]), v.transpose(0, 1)], dim=1).repeat_interleave(Hq // Hkv, dim=0)
            mask = torch.arange(ctx + n)[None, :] <= (ctx + torch.arange(n))[:, None]
            o = F.scaled_dot_product_attention(q.transpose(0, 1), K, Vv, attn_mask=mask)
            x = _r(x + F.linear(_r(o.transpose(0, 1).reshape(n, Hq * D)), _t(lay.wo)))
            ia += 1
        else:
            p = F.linear(h, _t(lay.w_in))
            sizes = [Hk * dk, Hk * dk, Hv * dv, Hv * dv, Hv, Hv]
            qr, kr, v, z, b, a = torch.split(p, sizes, dim=1)
            qr, kr = qr.view(n, Hk, dk), kr.view(n, Hk, dk)
            q = qr * torch.rsqrt((qr * qr).sum(-1, keepdim=True) + 1e-6) / math.sqrt(dk)
            k = kr * torch.rsqrt((kr * kr).sum(-1, keepdim=True) + 1e-6)
            v, z = v.view(n, Hv, dv), z.view(n, Hv, dv)
            beta, g = torch.sigmoid(b), -F.softplus(a)
            S0 = torch.from_numpy(np.asarray(states[idn], np.float64))
            gc = torch.cumsum(g, dim=0)
            o = torch.empty(n, Hv, dv, dtype=torch.float64)
            S_end = torch.empty_like(S0)
            for hh in range(Hv):
                kh = hh // (Hv // Hk)
                Kh, Qh, G = k[:, kh], q[:, kh], gc[:, hh]
                decay = torch.exp(G[:, None] - G[None, :])
                A = torch.tril(beta[:, hh, None] * decay * (Kh @ Kh.T), diagonal=-1)
                rhs = beta[:, hh, None] * (v[:, hh] - torch.exp(G)[:, None] * (Kh @ S0[hh]))
                U = torch.linalg.solve_triangular(torch.eye(n, dtype=torch.float64) + A, rhs, upper=False)
                o[:, hh] = torch.exp(G)[:, None] * (Qh @ S0[hh]) + torch.tril(decay * (Qh @ Kh.T)) @ U
                S_end[hh] = torch.exp(G[-1]) * S0[hh] + (torch.exp(G[-1] - G)[:, None] * Kh).T @ U
            kept_states.append(S_end)
            yv = o * torch.rsqrt((o * o).mean(-1, keepdim=True) + eps) * _t(lay.dn_norm) * F.silu(z)
            x = _r(x + F.linear(_r(yv).reshape(n, Hv * dv), _t(lay.w_out)))
            idn += 1
        h2 = _r(F.rms_norm(x, (H,), _t(lay.ln_mlp), eps))
        gu = F.linear(h2, _t(lay.w_gu))
        x = _r(x + F.linear(_r(F.silu(gu[:, :I]) * gu[:, I:]), _t(lay.w_down)))
    hf = _r(F.rms_norm(x, (H,), _t(m.ln_f), eps))
    return F.linear(hf, _t(m.lm_head)).to(torch.float32).numpy(), hf, kept_states


@pytest.mark.parametrize("seed,n,ctx", [(7, 6, 40), (8, 9, 0), (9, 4, 17)])
def test_chain_equals_torch_stack(seed, n, ctx):
    m, caches, states = _setup(seed, ctx=ctx, cap=ctx + 16)
    tokens = [int(t) for t in synth.tree_chain(n, m.dims.base.vocab, seed).token]
    dec = ST.decode_stack(m, caches, states, tokens)
    logits, hf, S_end = torch_chain(m, caches, states, tokens)
    hf_bits = _r(hf).to(torch.float32).view(torch.int32).numpy() >> 16
    assert np.count_nonzero((hf_bits & 0xFFFF).astype(np.uint16) != dec["hf"]) == 0, "bf16 hidden states differ"
    np.testing.assert_allclose(dec["logits"], logits, rtol=1e-12, atol=1e-12)
    for ld, S in enumerate(S_end):
        np.testing.assert_allclose(dec["states"][ld][-1], S.numpy(), rtol=1e-12, atol=1e-14)


def test_commit_keeps_what_decoding_the_path_leaves():
    import oracle
    m, caches, states = _setup(11)
    V = m.dims.base.vocab
    tree = synth.tree_lattice(10, 4, V, 5)
    res = ST.verify_stack(m, caches, states, tree.parent, tree.token)
    path = ST._path(tree.parent, 6)
    kept, kstates = ST.commit_stack(res, caches, path)
    dec = ST.decode_stack(m, caches, states, [int(tree.token[a]) for a in path])
    for la, c in enumerate(caches):
        k2, v2, src, new_ctx = kept[la]
        assert new_ctx == c.ctx_len + len(path)
        assert np.array_equal(k2[:, :c.ctx_len], c.k[:, :c.ctx_len])
        assert np.array_equal(k2[:, c.ctx_len:new_ctx].transpose(1, 0, 2), dec["k"][la])
        assert np.array_equal(v2[:, c.ctx_len:new_ctx].transpose(1, 0, 2), dec["v"][la])
    for ld in range(len(states)):
        assert np.array_equal(kstates[ld], dec["states"][ld][-1])
