"""CPU oracle of the tree verify through a stack of decoder layers -- TEST
INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference leg may import this module; the CUDA library shares no code with it.

The pages verify a tree through the whole target model: "one forward pass of
the target model runs over the whole tree" [Drafters and tree verify, §The
round, step 2], a model with "48 Gated DeltaNet layers" besides its attention
layers [§Tree verify through recurrent layers], whose commit keeps "the KV
rows and the recurrent state of the accepted path" [§The round, step 4].  The
pages do not give the layers themselves; the reading taken (the plainest one
that the rest supports) is a pre-norm residual stack

    x = E[token]
    for each layer:   x = bf16( x + Mixer( bf16(RMSNorm(x) g_mix) ) )
                      x = bf16( x + MLP( bf16(RMSNorm(x) g_mlp) ) )
    hf = bf16( RMSNorm(x) g_f ),   logits = fp32( hf W_lm^T )

with MLP(h) = bf16( silu(h W_gate^T) * (h W_up^T) ) W_down^T, and the mixer
either

* the attention layer of the single-layer oracle (``tv_oracle.c``): q, k, v =
  h W_qkv^T, RoPE at the node's position ctx + depth, bf16 q/k/v, softmax over
  the cache plus the node's ancestors and itself, bf16 output, times W_o^T; or
* a Gated DeltaNet layer: [q, k, v, z, b, a] = h W_in^T; per key head q and k
  divided by sqrt(sum of squares + 1e-6), q also by sqrt(d_k); beta =
  sigmoid(b), g = -softplus(a) per value head; the gated delta rule
  (``oracle/deltanet.py``) from the state after the node's parent (the state
  before the round at the root); per value head y = bf16( RMSNorm(o) w * silu(z) );
  the mixer output is y W_out^T.

Row i of the tree processes node i's token at position ctx + depth(i); in
every layer it sees exactly what plain decoding of its own root path would
give it (the cache and its ancestors' K/V in attention layers, the state after
its parent in DeltaNet layers).  ``decode_stack`` is that plain decoding, one
token after the other, and each tree row must equal it on its own path
(``tests/test_oracle_stack.py``).

Arithmetic: fp64 everywhere; every projection output one sequential fp64 dot
product (``oracle.matvec_rows``); bf16 rounding (nearest-even through fp32)
only at the storage points named above; logits rounded to fp32.  Both the tree
and the sequential forms run every row through the same per-row functions, so
their results agree to the last bit.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Sequence

import numpy as np

from . import bf16_to_f64, matvec_rows
from .deltanet import dn_step


def round_bf16_bits(x) -> np.ndarray:
    """bf16 bits of fp64 values: to fp32 (nearest-even), then to bf16
    (nearest-even on the upper 16 bits); NaN stays NaN."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    nan = np.isnan(f)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    r[nan] = ((u[nan] >> 16) | 0x40).astype(np.uint16)
    return r


def rb(x) -> np.ndarray:
    """x rounded to bf16, as fp64 values."""
    return bf16_to_f64(round_bf16_bits(x))


def _rms_bf16(x: np.ndarray, g_bits: np.ndarray, eps: float) -> np.ndarray:
    ss = float(np.dot(x, x))
    return rb(x * (1.0 / np.sqrt(ss / x.shape[0] + eps)) * bf16_to_f64(g_bits))


def _rope(x: np.ndarray, pos: int, theta: float) -> np.ndarray:
    """Rotate-half RoPE of rows x [heads][D] at integer position pos."""
    D = x.shape[1]
    half = D // 2
    ang = pos * theta ** (-2.0 * np.arange(half) / D)
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[:, :half], x[:, half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=1)


def _silu(x):
    return x / (1.0 + np.exp(-x))


# ---- one row through one layer --------------------------------------------------
def attn_front(lay, d, h: np.ndarray, pos: int):
    """q [Hq][D], k, v [Hkv][D] of one row, bf16-rounded (k, v go to the cache)."""
    Hq, Hkv, D = d.n_q_heads, d.n_kv_heads, d.head_dim
    y = matvec_rows(lay.wqkv, h[None])[0]
    q = _rope(y[:Hq * D].reshape(Hq, D), pos, d.rope_theta)
    k = _rope(y[Hq * D:(Hq + Hkv) * D].reshape(Hkv, D), pos, d.rope_theta)
    v = y[(Hq + Hkv) * D:].reshape(Hkv, D)
    return rb(q), rb(k), rb(v)


def attend(d, q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """softmax(q k^T / sqrt(D)) V per query head over keys K, V [n][Hkv][D];
    query head hq reads KV head hq / (Hq / Hkv).  bf16-rounded [Hq][D]."""
    G = d.n_q_heads // d.n_kv_heads
    out = np.empty_like(q)
    for hq in range(d.n_q_heads):
        g = hq // G
        s = (K[:, g, :] @ q[hq]) / np.sqrt(d.head_dim)
        p = np.exp(s - s.max())
        p /= p.sum()
        out[hq] = p @ V[:, g, :]
    return rb(out)


def attn_back(lay, o: np.ndarray, x: np.ndarray) -> np.ndarray:
    return rb(x + matvec_rows(lay.wo, o.reshape(1, -1))[0])


@dataclass
class DnFront:
    q: np.ndarray      # [Hk][dk]
    k: np.ndarray      # [Hk][dk]
    v: np.ndarray      # [Hv][dv]
    z: np.ndarray      # [Hv][dv]
    beta: np.ndarray   # [Hv]
    g: np.ndarray      # [Hv]


def dn_front(lay, sd, h: np.ndarray) -> DnFront:
    Hk, Hv, dk, dv = sd.n_k_heads, sd.n_v_heads, sd.d_k, sd.d_v
    p = matvec_rows(lay.w_in, h[None])[0]
    o = 0
    q = p[o:o + Hk * dk].reshape(Hk, dk); o += Hk * dk
    k = p[o:o + Hk * dk].reshape(Hk, dk); o += Hk * dk
    v = p[o:o + Hv * dv].reshape(Hv, dv); o += Hv * dv
    z = p[o:o + Hv * dv].reshape(Hv, dv); o += Hv * dv
    b = p[o:o + Hv]; o += Hv
    a = p[o:o + Hv]
    q = q / np.sqrt(np.sum(q * q, axis=1, keepdims=True) + 1e-6) / np.sqrt(dk)
    k = k / np.sqrt(np.sum(k * k, axis=1, keepdims=True) + 1e-6)
    beta = 1.0 / (1.0 + np.exp(-b))
    g = -np.logaddexp(0.0, a)
    return DnFront(q, k, v, z, beta, g)


def dn_core(sd, S: np.ndarray, f: DnFront):
    """One gated delta-rule step of every value head from state S [Hv][dk][dv]:
    (state after, output [Hv][dv])."""
    G = sd.n_v_heads // sd.n_k_heads
    S_new = np.empty_like(S)
    o = np.empty((sd.n_v_heads, sd.d_v))
    for h in range(sd.n_v_heads):
        kh = h // G
        S_new[h], o[h] = dn_step(S[h], f.q[kh], f.k[kh], f.v[h], float(f.beta[h]), float(f.g[h]))
    return S_new, o


def dn_back(lay, sd, o: np.ndarray, z: np.ndarray, x: np.ndarray) -> np.ndarray:
    eps = sd.base.rms_eps
    ms = np.mean(o * o, axis=1, keepdims=True)
    y = rb(o / np.sqrt(ms + eps) * bf16_to_f64(lay.dn_norm)[None, :] * _silu(z))
    return rb(x + matvec_rows(lay.w_out, y.reshape(1, -1))[0])


def mlp_block(lay, sd, x: np.ndarray) -> np.ndarray:
    I = sd.intermediate
    h2 = _rms_bf16(x, lay.ln_mlp, sd.base.rms_eps)
    gu = matvec_rows(lay.w_gu, h2[None])[0]
    a = rb(_silu(gu[:I]) * gu[I:])
    return rb(x + matvec_rows(lay.w_down, a[None])[0])


def _cache_rows(cache) -> tuple:
    """Cached K/V [ctx][Hkv][D] as fp64."""
    c = cache.ctx_len
    K = bf16_to_f64(np.transpose(cache.k[:, :c, :], (1, 0, 2)))
    V = bf16_to_f64(np.transpose(cache.v[:, :c, :], (1, 0, 2)))
    return K, V


def _path(parent, i) -> list:
    p = []
    while i >= 0:
        p.append(i)
        i = int(parent[i])
    return p[::-1]


def _logits(model, hf: np.ndarray) -> np.ndarray:
    return matvec_rows(model.lm_head, hf).astype(np.float32)


# ---- the tree verify ------------------------------------------------------------
def verify_stack(model, caches: Sequence, states: Sequence, parent, token) -> dict:
    """One request's verify through the stack.

    caches: one ``synth.Cache`` per attention layer (same ctx_len); states: the
    state before the round of each DeltaNet layer, [Hv][dk][dv].  Returns
    logits [n][V] fp32, hf [n][H] bf16 bits, per attention layer the tree rows'
    K and V [n][Hkv][D] bf16 bits (what verify writes at slots ctx + i), and per
    DeltaNet layer the state after every node [n][Hv][dk][dv] (fp64)."""
    sd = model.dims
    d = sd.base
    parent = np.asarray(parent)
    n = len(parent)
    ctx = caches[0].ctx_len if caches else 0
    depth = np.zeros(n, np.int64)
    for i in range(1, n):
        depth[i] = depth[parent[i]] + 1
    x = [bf16_to_f64(model.embed[int(t)]) for t in token]
    out_k, out_v, out_states = [], [], []
    ia = idn = 0
    for lay in model.layers:
        h = [_rms_bf16(x[i], lay.ln_mix, d.rms_eps) for i in range(n)]
        if lay.attn:
            Kc, Vc = _cache_rows(caches[ia])
            fr = [attn_front(lay, d, h[i], ctx + int(depth[i])) for i in range(n)]
            for i in range(n):
                p = _path(parent, i)
                K = np.concatenate([Kc, np.stack([fr[a][1] for a in p])])
                V = np.concatenate([Vc, np.stack([fr[a][2] for a in p])])
                x[i] = attn_back(lay, attend(d, fr[i][0], K, V), x[i])
            out_k.append(round_bf16_bits(np.stack([f[1] for f in fr])))
            out_v.append(round_bf16_bits(np.stack([f[2] for f in fr])))
            ia += 1
        else:
            S0 = np.asarray(states[idn], np.float64)
            Sn = [None] * n
            for i in range(n):
                f = dn_front(lay, sd, h[i])
                Sn[i], o = dn_core(sd, S0 if parent[i] < 0 else Sn[parent[i]], f)
                x[i] = dn_back(lay, sd, o, f.z, x[i])
            out_states.append(np.stack(Sn))
            idn += 1
        x = [mlp_block(lay, sd, x[i]) for i in range(n)]
    hf = np.stack([_rms_bf16(x[i], model.ln_f, d.rms_eps) for i in range(n)])
    return {"logits": _logits(model, hf), "hf": round_bf16_bits(hf), "k": out_k, "v": out_v,
            "states": out_states}


def decode_stack(model, caches: Sequence, states: Sequence, tokens: Sequence[int]) -> dict:
    """Plain decoding of a token sequence after the cached context, one token
    after the other: token t sits at position ctx + t, every attention layer
    appends its K/V and every DeltaNet layer steps its state.  Outputs as
    ``verify_stack``, one row per token."""
    sd = model.dims
    d = sd.base
    ctx = caches[0].ctx_len if caches else 0
    kv = [list(_cache_rows(c)) for c in caches]
    S = [np.asarray(s, np.float64) for s in states]
    dec_k = [[] for _ in caches]
    dec_v = [[] for _ in caches]
    st_rows = [[] for _ in states]
    hf = []
    for t, tok in enumerate(tokens):
        x = bf16_to_f64(model.embed[int(tok)])
        ia = idn = 0
        for lay in model.layers:
            h = _rms_bf16(x, lay.ln_mix, d.rms_eps)
            if lay.attn:
                q, k, v = attn_front(lay, d, h, ctx + t)
                dec_k[ia].append(k)
                dec_v[ia].append(v)
                K = np.concatenate([kv[ia][0], np.stack(dec_k[ia])])
                V = np.concatenate([kv[ia][1], np.stack(dec_v[ia])])
                x = attn_back(lay, attend(d, q, K, V), x)
                ia += 1
            else:
                f = dn_front(lay, sd, h)
                S[idn], o = dn_core(sd, S[idn], f)
                st_rows[idn].append(S[idn])
                x = dn_back(lay, sd, o, f.z, x)
                idn += 1
            x = mlp_block(lay, sd, x)
        hf.append(_rms_bf16(x, model.ln_f, d.rms_eps))
    hf = np.stack(hf)
    return {"logits": _logits(model, hf), "hf": round_bf16_bits(hf),
            "k": [round_bf16_bits(np.stack(a)) for a in dec_k], "v": [round_bf16_bits(np.stack(a)) for a in dec_v],
            "states": [np.stack(a) for a in st_rows]}


def commit_stack(res: dict, caches: Sequence, path: Sequence[int]):
    """What the round keeps [Drafters and tree verify, §The round, step 4]: in
    every attention layer the accepted path's K/V rows at slots ctx .. ctx + a
    (``oracle.commit_kv``), in every DeltaNet layer the state after the path's
    last node.  Returns (per attention layer (k, v) caches, per DeltaNet layer
    the kept state)."""
    from . import apply_tree_kv, commit_kv
    kept = []
    for la, c in enumerate(caches):
        k, v = apply_tree_kv(c, res["k"][la].reshape(len(res["k"][la]), -1), res["v"][la].reshape(len(res["v"][la]), -1))
        kept.append(commit_kv(k, v, c.ctx_len, path))
    states = [st[path[-1]].copy() for st in res["states"]]
    return kept, states
