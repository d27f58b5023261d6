"""Seeded synthetic inputs for the tree verify round.

This module only draws numbers: model weights, KV caches, draft trees and
uniforms.  It holds none of the verify arithmetic, so both the CUDA path and the
CPU oracle can take their inputs from here without sharing any of the method.

Shapes and distributions follow the workloads the pages describe:

* weights ~ N(0, 0.02) in bf16, cached K/V ~ N(0, 1) in bf16;
* draft trees of at most 32 nodes given as a parent array in parent-before-child
  order [Algorithm and correctness contract, §Target position and batching];
* lattice trees: a spine (the greedy path through a slots x 16-candidates
  lattice) with next-best candidates as branches, siblings distinct and ordered
  by score [Drafters and tree verify, §The block drafter; Algorithm and
  correctness contract, §Deterministic tree candidates];
* a cut to 8, 16, 24 or 32 rows [Drafters and tree verify, §StairCut].

Everything is a pure function of its seed.  bf16 values are carried as uint16
bit patterns (numpy has no bf16 dtype); the rounding from the fp32 draw is done
by torch's own conversion.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Dims:
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    vocab: int
    rope_theta: float = 1.0e6
    rms_eps: float = 1.0e-6

    @property
    def qkv_out(self) -> int:
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.head_dim


# Tiny layer of the small random-model case: hidden 256, 4/2 heads of 64, vocab 1024.
TINY = Dims(hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64, vocab=1024)
# The hidden-5120 layer: 40 query heads / 8 KV heads of 128, vocab 151936.
FULL = Dims(hidden=5120, n_q_heads=40, n_kv_heads=8, head_dim=128, vocab=151936)
# A mid-size layer that still spans several GEMM tiles and has ragged tails
# everywhere (vocab and context not multiples of the tile sizes).
MID = Dims(hidden=512, n_q_heads=8, n_kv_heads=2, head_dim=128, vocab=5003)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round an fp32 array to bf16 (torch's round-to-nearest-even) -> uint16 bits."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _normal_bf16(rng: np.random.Generator, shape, std: float, chunk: int = 1 << 26) -> np.ndarray:
    """N(0, std) draws rounded to bf16, generated in chunks to bound host memory."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        x = rng.standard_normal(e - s, dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        out[s:e] = f32_to_bf16_bits(x)
    return out.reshape(shape)


@dataclass
class Model:
    dims: Dims
    embed: np.ndarray      # [V, H] bf16 bits
    ln1: np.ndarray        # [H] bf16 bits (RMSNorm gain before the projections)
    wqkv: np.ndarray       # [(Hq + 2 Hkv) D, H] bf16 bits, rows: Q heads, then K heads, then V heads
    wo: np.ndarray         # [H, Hq D] bf16 bits
    ln_f: np.ndarray       # [H] bf16 bits (final RMSNorm gain)
    lm_head: np.ndarray    # [V, H] bf16 bits


def gen_model(dims: Dims, seed: int, std: float = 0.02, random_gains: bool = False) -> Model:
    """A random-init layer + head.  Gains are 1.0 unless ``random_gains`` (tests
    use random gains so that a dropped gain multiply cannot go unnoticed)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    H, V = dims.hidden, dims.vocab
    embed = _normal_bf16(rng, (V, H), std)
    wqkv = _normal_bf16(rng, (dims.qkv_out, H), std)
    wo = _normal_bf16(rng, (H, dims.n_q_heads * dims.head_dim), std)
    lm_head = _normal_bf16(rng, (V, H), std)
    if random_gains:
        ln1 = f32_to_bf16_bits(1.0 + 0.25 * rng.standard_normal(H, dtype=np.float32))
        ln_f = f32_to_bf16_bits(1.0 + 0.25 * rng.standard_normal(H, dtype=np.float32))
    else:
        ln1 = f32_to_bf16_bits(np.ones(H, np.float32))
        ln_f = f32_to_bf16_bits(np.ones(H, np.float32))
    return Model(dims, embed, ln1, wqkv, wo, ln_f, lm_head)


@dataclass
class Cache:
    k: np.ndarray   # [Hkv, capacity, D] bf16 bits
    v: np.ndarray   # [Hkv, capacity, D] bf16 bits
    ctx_len: int
    capacity: int


def gen_cache(dims: Dims, ctx_len: int, capacity: int, seed: int) -> Cache:
    """Cached K/V ~ N(0, 1) in slots [0, ctx_len).  Slots past ctx_len hold other
    random values, so a kernel that reads a slot it should not read is caught."""
    assert capacity >= ctx_len
    rng = np.random.Generator(np.random.PCG64(seed))
    shape = (dims.n_kv_heads, capacity, dims.head_dim)
    k = _normal_bf16(rng, shape, 1.0)
    v = _normal_bf16(rng, shape, 1.0)
    return Cache(k, v, ctx_len, capacity)


@dataclass
class Tree:
    parent: np.ndarray  # [n] int32, parent[0] = -1, parent[i] < i
    token: np.ndarray   # [n] int32

    @property
    def n(self) -> int:
        return int(self.parent.shape[0])


def _distinct_sibling_tokens(rng, parent: np.ndarray, vocab: int) -> np.ndarray:
    """Tokens uniform in [0, vocab), re-drawn until no two siblings share one."""
    n = parent.shape[0]
    token = np.empty(n, np.int32)
    for i in range(n):
        while True:
            t = int(rng.integers(0, vocab))
            sib = [j for j in range(1, i) if parent[j] == parent[i]] if i > 0 else []
            if all(token[j] != t for j in sib):
                break
        token[i] = t
    return token


def tree_spine_random(n: int, spine: int, vocab: int, seed: int) -> Tree:
    """A spine of ``spine`` nodes (root included) chained 0 -> 1 -> ... -> spine-1,
    then nodes spine..n-1 with parents uniform over the earlier nodes."""
    assert 1 <= spine <= n <= 32
    rng = np.random.Generator(np.random.PCG64(seed))
    parent = np.empty(n, np.int32)
    parent[0] = -1
    for i in range(1, n):
        parent[i] = i - 1 if i < spine else int(rng.integers(0, i))
    return Tree(parent, _distinct_sibling_tokens(rng, parent, vocab))


def tree_chain(n: int, vocab: int, seed: int) -> Tree:
    return tree_spine_random(n, n, vocab, seed)


def tree_star(n: int, vocab: int, seed: int) -> Tree:
    """Root with n-1 children (a one-level bush)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    parent = np.full(n, 0, np.int32)
    parent[0] = -1
    return Tree(parent, _distinct_sibling_tokens(rng, parent, vocab))


def tree_lattice(n: int, slots: int, vocab: int, seed: int, width: int = 16) -> Tree:
    """A draft tree cut from a ``slots`` x ``width`` lattice of seeded scores.

    The spine is the best candidate of every slot (the greedy path); the other
    candidates of slot k are siblings of the spine node of slot k, admitted
    best-score-first until the tree holds ``n`` nodes (root included).  Nodes
    are emitted in depth-first pre-order with siblings in decreasing score.
    """
    assert 1 <= n <= 32
    rng = np.random.Generator(np.random.PCG64(seed))
    spine_len = min(slots, n - 1)
    scores = rng.standard_normal((slots, width))
    scores = -np.sort(-scores, axis=1)           # candidate 0 is the slot's best
    tokens = np.empty((slots, width), np.int64)
    for k in range(slots):
        tokens[k] = rng.choice(vocab, size=width, replace=False)
    # branch candidates (slot, rank>=1) ranked by score
    branches = sorted(((scores[k, c], k, c) for k in range(spine_len) for c in range(1, width)),
                      key=lambda t: -t[0])[: n - 1 - spine_len]
    # children lists: spine node of slot k-1 (root for k=0) holds slot k's candidates
    kids: dict[int, list] = {k: [(scores[k, 0], k, 0)] for k in range(spine_len)}
    for s, k, c in branches:
        kids[k].append((s, k, c))
    order_parent, order_token = [], []

    def emit(slot_parent_idx: int, k: int):
        if k >= spine_len:
            return
        for s, kk, c in sorted(kids[k], key=lambda t: -t[0]):
            idx = len(order_parent)
            order_parent.append(slot_parent_idx)
            order_token.append(int(tokens[kk, c]))
            if c == 0:
                emit(idx, k + 1)

    order_parent.append(-1)
    order_token.append(int(rng.integers(0, vocab)))   # the anchor token
    emit(0, 0)
    return Tree(np.array(order_parent, np.int32), np.array(order_token, np.int32))


def uniforms(n: int, seed: int) -> np.ndarray:
    """Uniform draws in [0, 1) as fp32 (never 1.0)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    u = rng.random(n, dtype=np.float32)
    return np.minimum(u, np.float32(np.nextafter(np.float32(1.0), np.float32(0.0))))


def logits_rows(n: int, vocab: int, seed: int, scale: float = 1.5) -> np.ndarray:
    """fp32 logit rows ~ N(0, scale) for walk-only tests."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return (rng.standard_normal((n, vocab), dtype=np.float32) * np.float32(scale)).astype(np.float32)


@dataclass
class DnInputs:
    q: np.ndarray      # [n][H_k][d_k] fp32, unit length / sqrt(d_k)
    k: np.ndarray      # [n][H_k][d_k] fp32, unit length
    v: np.ndarray      # [n][H_v][d_v] fp32 ~ N(0, 1)
    beta: np.ndarray   # [n][H_v] fp32 in (0.05, 0.95)
    g: np.ndarray      # [n][H_v] fp32 in (-0.4, -0.001)
    S0: np.ndarray     # [H_v][d_k][d_v] fp32 ~ N(0, 0.3^2)


def dn_inputs(n: int, n_k_heads: int, n_v_heads: int, d_k: int, d_v: int, seed: int) -> DnInputs:
    """Per-node inputs of one Gated DeltaNet layer's recurrent core and the
    state before the round, as fp32.  Keys and queries are unit vectors (the
    layer normalises them), queries scaled by 1/sqrt(d_k); write strengths and
    log decays span the ranges a sigmoid and a negative softplus give."""
    rng = np.random.Generator(np.random.PCG64(seed))
    q = rng.standard_normal((n, n_k_heads, d_k))
    q /= np.linalg.norm(q, axis=2, keepdims=True) * np.sqrt(d_k)
    k = rng.standard_normal((n, n_k_heads, d_k))
    k /= np.linalg.norm(k, axis=2, keepdims=True)
    v = rng.standard_normal((n, n_v_heads, d_v))
    beta = rng.uniform(0.05, 0.95, (n, n_v_heads))
    g = -rng.uniform(0.001, 0.4, (n, n_v_heads))
    S0 = rng.standard_normal((n_v_heads, d_k, d_v)) * 0.3
    f = lambda a: np.ascontiguousarray(a, dtype=np.float32)
    return DnInputs(f(q), f(k), f(v), f(beta), f(g), f(S0))


@dataclass
class Request:
    tree: Tree
    cache: Cache


@dataclass
class Workload:
    """One verify round's inputs: a model and one or more requests."""
    name: str
    model: Model
    requests: list = field(default_factory=list)


def joint_contexts(n_req: int, seed: int, lo: int = 1024, hi: int = 8192) -> list:
    rng = np.random.Generator(np.random.PCG64(seed))
    return [int(c) for c in rng.integers(lo, hi + 1, size=n_req)]


# ---------------------------------------------------------------------------
# the decoder-layer stack: Gated DeltaNet and attention layers, each followed by
# a SwiGLU MLP (the composition is a reading: the pages name the layer kinds,
# not the layers)
# ---------------------------------------------------------------------------
@dataclass(frozen=True)
class StackDims:
    base: Dims            # hidden, attention heads, vocab, RoPE base, RMSNorm eps
    n_layers: int
    attn_every: int       # layer l is an attention layer iff l % attn_every == attn_every - 1
    n_k_heads: int        # Gated DeltaNet key heads
    n_v_heads: int        # Gated DeltaNet value heads
    d_k: int
    d_v: int
    intermediate: int     # MLP width

    def is_attn(self, layer: int) -> bool:
        return layer % self.attn_every == self.attn_every - 1

    @property
    def attn_layers(self) -> list:
        return [l for l in range(self.n_layers) if self.is_attn(l)]

    @property
    def dn_layers(self) -> list:
        return [l for l in range(self.n_layers) if not self.is_attn(l)]

    @property
    def dn_in_out(self) -> int:
        """Rows of the DeltaNet input projection: q, k (key heads), v, z (value
        heads), then the write-strength and decay logits (one per value head)."""
        return 2 * self.n_k_heads * self.d_k + 2 * self.n_v_heads * self.d_v + 2 * self.n_v_heads


# small stack for the tests: 3 DeltaNet layers then an attention layer
STACK_TINY = StackDims(base=TINY, n_layers=4, attn_every=4, n_k_heads=2, n_v_heads=4, d_k=64, d_v=64,
                       intermediate=512)
# the hidden-5120 stack of the benchmark: 64 layers, every 4th an attention
# layer (48 DeltaNet layers), 16 key / 32 value heads of 128, MLP width 17408
STACK_FULL = StackDims(base=FULL, n_layers=64, attn_every=4, n_k_heads=16, n_v_heads=32, d_k=128, d_v=128,
                       intermediate=17408)


@dataclass
class StackLayer:
    attn: bool
    ln_mix: np.ndarray             # [H] gain of the norm before the mixer
    ln_mlp: np.ndarray             # [H] gain of the norm before the MLP
    w_gu: np.ndarray               # [2 I][H]: gate rows, then up rows
    w_down: np.ndarray             # [H][I]
    wqkv: np.ndarray = None        # attention: [(Hq + 2 Hkv) D][H]
    wo: np.ndarray = None          # attention: [H][Hq D]
    w_in: np.ndarray = None        # DeltaNet: [dn_in_out][H]
    w_out: np.ndarray = None       # DeltaNet: [H][Hv d_v]
    dn_norm: np.ndarray = None     # DeltaNet: [d_v] gain of the per-head output norm


@dataclass
class StackModel:
    dims: StackDims
    embed: np.ndarray              # [V][H]
    ln_f: np.ndarray               # [H]
    lm_head: np.ndarray            # [V][H]
    layers: list


def gen_stack(dims: StackDims, seed: int, std: float = 0.02, random_gains: bool = False) -> StackModel:
    """Random-init stack (bf16 bits), gains 1.0 unless ``random_gains``.  The
    matrices that write into the residual stream (the mixers' output
    projections and the MLP's down projection) draw with std / sqrt(2 L), L
    the number of layers (the GPT-2 initialisation of residual layers), so
    that the residual stream stays O(1) through the stack."""
    rng = np.random.Generator(np.random.PCG64(seed))
    b = dims.base
    H, V = b.hidden, b.vocab
    out_std = std / float(np.sqrt(2 * dims.n_layers))

    def gain(n):
        x = 1.0 + 0.25 * rng.standard_normal(n, dtype=np.float32) if random_gains else np.ones(n, np.float32)
        return f32_to_bf16_bits(x)

    embed = _normal_bf16(rng, (V, H), std)
    layers = []
    for l in range(dims.n_layers):
        if dims.is_attn(l):
            lay = StackLayer(True, gain(H), gain(H), None, None,
                             wqkv=_normal_bf16(rng, (b.qkv_out, H), std),
                             wo=_normal_bf16(rng, (H, b.n_q_heads * b.head_dim), out_std))
        else:
            lay = StackLayer(False, gain(H), gain(H), None, None,
                             w_in=_normal_bf16(rng, (dims.dn_in_out, H), std),
                             w_out=_normal_bf16(rng, (H, dims.n_v_heads * dims.d_v), out_std),
                             dn_norm=gain(dims.d_v))
        lay.w_gu = _normal_bf16(rng, (2 * dims.intermediate, H), std)
        lay.w_down = _normal_bf16(rng, (H, dims.intermediate), out_std)
        layers.append(lay)
    ln_f = gain(H)
    lm_head = _normal_bf16(rng, (V, H), std)
    return StackModel(dims, embed, ln_f, lm_head, layers)


def gen_dn_states(dims: StackDims, seed: int) -> list:
    """The recurrent state before the round of every DeltaNet layer, fp32
    [H_v][d_k][d_v] ~ N(0, 0.3^2)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return [np.ascontiguousarray(rng.standard_normal((dims.n_v_heads, dims.d_k, dims.d_v)) * 0.3, dtype=np.float32)
            for _ in dims.dn_layers]
