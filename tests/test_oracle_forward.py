"""Pins of the oracle's forward pass (CPU only).

The oracle is checked against things other than itself:

* bf16 rounding against torch's conversion;
* every tree row against plain one-token-at-a-time decoding of that row's own
  root path ("each tree node's row equals a sequential one-token decode of that
  node's prefix"; the promise of [Exactness, §The promise]);
* chains against an independent torch-fp64 transformer layer built from
  library routines (rms_norm, linear, complex-exponential RoPE,
  scaled_dot_product_attention), with bf16 rounding at the same storage points;
* the head's argmax / top-2 gap against sorting, the BF16 step against the
  page's printed value and against bf16 bit patterns.
"""
import json
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from speculative_tree_verify_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# bf16 rounding
# --------------------------------------------------------------------------
def test_round_bf16_matches_torch_on_fp32_values():
    rng = np.random.default_rng(0)
    vals = list(rng.standard_normal(2000).astype(np.float32) * np.float32(3.0))
    # exact halfway cases: low 16 bits = 0x8000, both parities of the kept lsb
    for hi in (0x3F80, 0x3F81, 0xC2F7, 0x4000, 0x0001):
        vals.append(np.array([(hi << 16) | 0x8000], np.uint32).view(np.float32)[0])
    vals += [np.float32(0.0), np.float32(-0.0), np.float32(65504.0), np.float32(1e-40)]
    x = np.array(vals, np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.round_bf16(float(v)) for v in x], np.uint16)
    np.testing.assert_array_equal(got, want)


def test_round_bf16_goes_through_fp32():
    # a double just above a bf16 halfway point but below fp32's resolution there
    # rounds to the halfway fp32 value first, then ties to even
    half = np.array([(0x3F80 << 16) | 0x8000], np.uint32).view(np.float32)[0]   # 1 + 2^-8
    x = float(half) + 2.0 ** -40
    assert oracle.round_bf16(x) == 0x3F80        # tie -> even (1.0), not 0x3F81


# --------------------------------------------------------------------------
# tree rows == sequential decoding of each row's own path
# --------------------------------------------------------------------------
def _root_path(parent, i):
    p = []
    while i >= 0:
        p.append(i)
        i = int(parent[i])
    return p[::-1]


def _leaves(parent):
    n = len(parent)
    has_child = set(int(p) for p in parent[1:])
    return [i for i in range(n) if i not in has_child]


def _check_tree_against_decode(model, cache, tree):
    ver = oracle.verify_tree(model, cache, tree)
    seen = set()
    for leaf in _leaves(tree.parent):
        path = _root_path(tree.parent, leaf)
        dec = oracle.decode_sequence(model, cache, [int(tree.token[a]) for a in path])
        for t, node in enumerate(path):
            for key in ("logits", "k", "v", "attn", "hf"):
                np.testing.assert_array_equal(ver[key][node], dec[key][t], err_msg=f"{key} row {node}")
            seen.add(node)
    assert seen == set(range(tree.n))


@pytest.mark.parametrize("seed", range(6))
def test_tree_rows_equal_sequential_decode_tiny(seed):
    d = synth.TINY
    model = synth.gen_model(d, 100 + seed, random_gains=True)
    cache = synth.gen_cache(d, 64, 128, 200 + seed)
    tree = synth.tree_spine_random(8, 4, d.vocab, 300 + seed)
    _check_tree_against_decode(model, cache, tree)


@pytest.mark.parametrize("kind", ["star", "lattice", "chain32", "single"])
def test_tree_rows_equal_sequential_decode_shapes(kind):
    d = synth.TINY
    model = synth.gen_model(d, 7, random_gains=True)
    cache = synth.gen_cache(d, 19, 64, 8)
    tree = {"star": lambda: synth.tree_star(12, d.vocab, 9),
            "lattice": lambda: synth.tree_lattice(24, 7, d.vocab, 9),
            "chain32": lambda: synth.tree_chain(32, d.vocab, 9),
            "single": lambda: synth.tree_chain(1, d.vocab, 9)}[kind]()
    _check_tree_against_decode(model, cache, tree)


def test_empty_context_tree():
    d = synth.TINY
    model = synth.gen_model(d, 11)
    cache = synth.gen_cache(d, 0, 32, 12)
    tree = synth.tree_spine_random(8, 3, d.vocab, 13)
    _check_tree_against_decode(model, cache, tree)


# --------------------------------------------------------------------------
# chains == an independent torch-fp64 layer
# --------------------------------------------------------------------------
def _w(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(torch.float64)


def _rb(t):
    return t.to(torch.float32).to(torch.bfloat16).to(torch.float64)


def torch_layer_over_sequence(model, cache, tokens):
    """A textbook pre-norm attention layer + LM head over ``tokens`` appended
    after the cache, causal, in fp64 with bf16 stores at the same points."""
    d = model.dims
    H, D, Hq, Hkv = d.hidden, d.head_dim, d.n_q_heads, d.n_kv_heads
    L, ctx = len(tokens), cache.ctx_len
    E, Wqkv, Wo, Wl = _w(model.embed), _w(model.wqkv), _w(model.wo), _w(model.lm_head)
    g1, gf = _w(model.ln1), _w(model.ln_f)
    x = E[torch.tensor(tokens)]
    h = _rb(F.rms_norm(x, (H,), weight=g1, eps=d.rms_eps))
    qkv = F.linear(h, Wqkv)
    q = qkv[:, : Hq * D].reshape(L, Hq, D)
    k = qkv[:, Hq * D: (Hq + Hkv) * D].reshape(L, Hkv, D)
    v = qkv[:, (Hq + Hkv) * D:].reshape(L, Hkv, D)
    # RoPE as a complex rotation of (x[d], x[d + D/2]) by pos * theta^(-2d/D)
    inv_freq = torch.tensor(d.rope_theta, dtype=torch.float64) ** (-torch.arange(0, D, 2, dtype=torch.float64) / D)
    pos = torch.arange(ctx, ctx + L, dtype=torch.float64)
    rot = torch.polar(torch.ones(L, D // 2, dtype=torch.float64), pos[:, None] * inv_freq[None, :])

    def rope(t):
        z = torch.complex(t[..., : D // 2], t[..., D // 2:]) * rot[:, None, :]
        return torch.cat([z.real, z.imag], dim=-1)

    q, k, v = _rb(rope(q)), _rb(rope(k)), _rb(v)
    ck = _w(cache.k)[:, :ctx, :].permute(1, 0, 2)       # [ctx, Hkv, D]
    cv = _w(cache.v)[:, :ctx, :].permute(1, 0, 2)
    K = torch.cat([ck, k]).permute(1, 0, 2).repeat_interleave(Hq // Hkv, dim=0)   # [Hq, ctx+L, D]
    V = torch.cat([cv, v]).permute(1, 0, 2).repeat_interleave(Hq // Hkv, dim=0)
    mask = torch.ones(L, ctx + L, dtype=torch.bool).tril(diagonal=ctx)
    o = F.scaled_dot_product_attention(q.permute(1, 0, 2)[None], K[None], V[None], attn_mask=mask)[0]
    o = _rb(o.permute(1, 0, 2).reshape(L, Hq * D))
    r = _rb(x + F.linear(o, Wo))
    hf = _rb(F.rms_norm(r, (H,), weight=gf, eps=d.rms_eps))
    logits = F.linear(hf, Wl).to(torch.float32)

    def bits(t):
        return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)

    return {"logits": logits.numpy(), "k": bits(k.reshape(L, -1)), "v": bits(v.reshape(L, -1)),
            "attn": bits(o), "hf": bits(hf)}


@pytest.mark.parametrize("dims,ctx,L,seed", [(synth.TINY, 64, 8, 0), (synth.TINY, 0, 5, 1),
                                              (synth.MID, 37, 9, 2)])
def test_chain_equals_torch_layer(dims, ctx, L, seed):
    model = synth.gen_model(dims, seed, random_gains=True)
    cache = synth.gen_cache(dims, ctx, ctx + L + 3, seed + 50)
    tree = synth.tree_chain(L, dims.vocab, seed + 60)
    got = oracle.verify_tree(model, cache, tree)
    ref = torch_layer_over_sequence(model, cache, [int(t) for t in tree.token])
    for key in ("k", "v", "attn", "hf"):
        mism = np.count_nonzero(got[key] != ref[key])
        assert mism == 0, f"{key}: {mism} bf16 values differ"
    np.testing.assert_allclose(got["logits"], ref["logits"], rtol=3e-7, atol=1e-8)


# --------------------------------------------------------------------------
# argmax / top-2 / BF16 step
# --------------------------------------------------------------------------
def test_argmax_top2_against_sorting():
    rng = np.random.default_rng(3)
    lg = rng.standard_normal((40, 257)).astype(np.float32)
    lg[5, 17] = lg[5, 200] = lg[5].max() + 1.0          # equal maxima: lowest index, gap 0
    lg[6, :] = 0.25                                      # all equal
    idx, l1, l2, gap = oracle.argmax_top2(lg)
    for r in range(lg.shape[0]):
        order = sorted(range(lg.shape[1]), key=lambda j: (-float(lg[r, j]), j))
        assert idx[r] == order[0]
        assert l1[r] == float(lg[r, order[0]])
        assert l2[r] == float(lg[r, order[1]])
    assert idx[5] == 17 and gap[5] == 0.0
    assert idx[6] == 0 and gap[6] == 0.0


def test_bf16_step_matches_page():
    g = json.load(open(os.path.join(GOLDEN, "bf16_step.json")))
    lo, hi = g["magnitude_range"]
    for x in np.linspace(lo, hi, 50, endpoint=False):
        assert oracle.bf16_ulp(x) == g["bf16_step"]
        assert oracle.bf16_ulp(-x) == g["bf16_step"]


def test_bf16_ulp_is_spacing_of_bf16_values():
    rng = np.random.default_rng(4)
    x = (rng.standard_normal(500) * np.exp(rng.uniform(-8, 8, 500))).astype(np.float32)
    b = torch.from_numpy(x).to(torch.bfloat16)
    a = b.abs()
    nxt = (a.view(torch.int16) + 1).view(torch.bfloat16)       # next bf16 value above |x|
    spacing = (nxt.to(torch.float64) - a.to(torch.float64)).numpy()
    np.testing.assert_array_equal(oracle.bf16_ulp(a.to(torch.float64).numpy()), spacing)


def test_near_tie_rule():
    assert oracle.near_tie(20.0, 20.0 - 0.125)       # exactly one step at [16, 32)
    assert not oracle.near_tie(20.0, 20.0 - 0.126)
    assert oracle.near_tie(1.5, 1.5 - 2 ** -7)
    assert not oracle.near_tie(1.5, 1.5 - 2 ** -6)


def test_head_rows_match_full_head():
    d = synth.MID
    model = synth.gen_model(d, 21)
    cache = synth.gen_cache(d, 30, 64, 22)
    tree = synth.tree_spine_random(6, 3, d.vocab, 23)
    ver = oracle.verify_tree(model, cache, tree)
    ids = [0, 1, 17, d.vocab - 1, 4095, 2048]
    part = oracle.head_rows(model, ver["hf"], ids)
    np.testing.assert_array_equal(part, ver["logits"][:, ids])
