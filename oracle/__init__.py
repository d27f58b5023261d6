"""CPU oracle of the tree verify round -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference leg may import this package.  The product (the CUDA library and its
Python binding) never imports it and shares no code with it: no kernels,
headers, helpers, tables or pre/post-processing.  The only thing the two sides
share is the seeded input generator, which holds none of the method's
arithmetic.

What is here, each written from the pages' statement of the method:

* ``verify_tree`` / ``decode_sequence`` / ``head_rows`` -- the forward pass, in
  plain C (``tv_oracle.c``), fp64 accumulation, bf16 rounding only at the
  storage points, fp32 logits.
* ``validate`` -- the input rejections of [Algorithm and correctness contract,
  §Single-path sampling and §Target position and batching].
* ``argmax_top2`` / ``bf16_ulp`` / ``near_tie`` -- the greedy choice and the
  near-tie rule of [Exactness, §The one exception: near ties].
* ``accept_greedy`` -- [Drafters and tree verify, §The round, step 3].
* ``accept_residual`` -- deterministic-candidate residual sampling,
  [Algorithm and correctness contract, §Deterministic tree candidates and
  residual verification].
* ``commit_kv`` -- [Drafters and tree verify, §The round, step 4, and
  §Tree verify through recurrent layers, last paragraph].
* ``oracle.sampling`` -- the sampled accept variants and the filters.
* ``oracle.deltanet`` -- Gated DeltaNet tree verify and the path-state commit
  [Drafters and tree verify, §Tree verify through recurrent layers].

Parity pins: every function above is pinned in ``tests/test_oracle_*.py`` to
something other than itself (brute-force sequential decoding, an independent
torch-fp64 transformer layer on chains, the pages' printed grid counts, Monte
Carlo laws, closed forms).  Nothing here is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import sys
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (OpenMP when available).  -ffp-contract=off
    keeps every a*b+c unfused so the results are the same on every host."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    try:
        subprocess.run(base + ["-fopenmp", _SRC, "-o", tmp, "-lm"], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + [_SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Model(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("vocab", ctypes.c_int32),
                ("rope_theta", ctypes.c_double), ("rms_eps", ctypes.c_double),
                ("embed", ctypes.c_void_p), ("ln1", ctypes.c_void_p), ("wqkv", ctypes.c_void_p),
                ("wo", ctypes.c_void_p), ("ln_f", ctypes.c_void_p), ("lm_head", ctypes.c_void_p)]


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        I = ctypes.c_int
        lib.orc_verify_tree.argtypes = [ctypes.POINTER(_Model), P, P, I, I, P, P, I, P, P, P, P, P, P]
        lib.orc_decode_sequence.argtypes = [ctypes.POINTER(_Model), P, P, I, I, P, I, P, P, P, P, P]
        lib.orc_head_rows.argtypes = [ctypes.POINTER(_Model), P, I, P, I, P]
        lib.orc_matvec_rows.argtypes = [P, I, I, P, I, P]
        lib.orc_round_bf16.argtypes = [ctypes.c_double]
        lib.orc_round_bf16.restype = ctypes.c_uint16
        lib.orc_num_threads.restype = ctypes.c_int
        lib.orc_set_num_threads.argtypes = [ctypes.c_int]
        _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().orc_num_threads())


def set_num_threads(n: int) -> None:
    """Threads for the following calls (for timing; results do not depend on it)."""
    _load().orc_set_num_threads(int(n))


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


def _c_model(model):
    d = model.dims
    arrs = [np.ascontiguousarray(a, dtype=np.uint16) for a in
            (model.embed, model.ln1, model.wqkv, model.wo, model.ln_f, model.lm_head)]
    cm = _Model(d.hidden, d.n_q_heads, d.n_kv_heads, d.head_dim, d.vocab, float(d.rope_theta),
                float(d.rms_eps), *[a.ctypes.data for a in arrs])
    return cm, arrs   # keep the arrays alive with the struct


def matvec_rows(w_bits: np.ndarray, x: np.ndarray) -> np.ndarray:
    """y[i] = W x[i] for W given as bf16 bits [M][K] and x fp64 [n][K]; every
    output one sequential fp64 dot product (``tv_oracle.c``)."""
    w = np.ascontiguousarray(w_bits, dtype=np.uint16)
    xx = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float64)
    M, K = w.shape
    assert xx.shape[1] == K
    y = np.empty((xx.shape[0], M), dtype=np.float64)
    _load().orc_matvec_rows(w.ctypes.data, M, K, xx.ctypes.data, xx.shape[0], y.ctypes.data)
    return y


def round_bf16(x: float) -> int:
    """bf16 bits of x, rounded to nearest-even through fp32 (the C oracle's rule)."""
    return int(_load().orc_round_bf16(float(x)))


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# validation: what the pages reject
# ---------------------------------------------------------------------------
MAX_ROWS = 32


def validate(parent: Sequence[int], token: Sequence[int], vocab: int,
             ctx: int = 0, capacity: Optional[int] = None) -> str:
    """Name of the first rule a tree breaks, or "ok".

    * a tree of 1..32 nodes ("a draft tree of at most 32 nodes" [Drafters and
      tree verify, §The round]) -> "rows";
    * parent-before-child: parent[0] = -1, 0 <= parent[i] < i -> "order";
    * token ids inside the vocabulary -> "token";
    * no two siblings with the same token ("duplicate sibling token ids ... are
      rejected" [Algorithm and correctness contract, §Target position and
      batching]) -> "dup_sibling";
    * the tree's rows must fit in the cache: ctx + n <= capacity -> "capacity".
    """
    n = len(parent)
    if n < 1 or n > MAX_ROWS or len(token) != n:
        return "rows"
    if int(parent[0]) != -1:
        return "order"
    for i in range(1, n):
        if not (0 <= int(parent[i]) < i):
            return "order"
    for i in range(n):
        if not (0 <= int(token[i]) < vocab):
            return "token"
    for i in range(1, n):
        for j in range(1, i):
            if int(parent[j]) == int(parent[i]) and int(token[j]) == int(token[i]):
                return "dup_sibling"
    if capacity is not None and ctx + n > capacity:
        return "capacity"
    return "ok"


def validate_sampling(uniforms: Sequence[float], temperature: float) -> str:
    """Random inputs must be finite and in [0, 1) [Algorithm and correctness
    contract, §Single-path sampling]; a sampled walk needs a temperature above 0
    [Exactness, §Sampling]."""
    if not (math.isfinite(temperature) and temperature > 0.0):
        return "temp"
    for u in uniforms:
        u = float(u)
        if not (math.isfinite(u) and 0.0 <= u < 1.0):
            return "uniform"
    return "ok"


# ---------------------------------------------------------------------------
# the forward pass (C)
# ---------------------------------------------------------------------------
def verify_tree(model, cache, tree, want=("logits", "k", "v", "attn", "hf", "q")) -> dict:
    """One request's verify: every row's fp32 logits and the intermediate
    storage points.  ``cache`` holds K/V [Hkv][capacity][D] with ctx_len valid
    slots.  Returns arrays keyed by name (bf16 ones as uint16 bits)."""
    d = model.dims
    lib = _load()
    n = tree.n
    QD, KD = d.n_q_heads * d.head_dim, d.n_kv_heads * d.head_dim
    out = {
        "logits": np.empty((n, d.vocab), np.float32) if "logits" in want else None,
        "q": np.empty((n, QD), np.uint16) if "q" in want else None,
        "k": np.empty((n, KD), np.uint16) if "k" in want else None,
        "v": np.empty((n, KD), np.uint16) if "v" in want else None,
        "attn": np.empty((n, QD), np.uint16) if "attn" in want else None,
        "hf": np.empty((n, d.hidden), np.uint16) if "hf" in want else None,
    }
    cm, keep = _c_model(model)
    ck = np.ascontiguousarray(cache.k, np.uint16)
    cv = np.ascontiguousarray(cache.v, np.uint16)
    par = np.ascontiguousarray(tree.parent, np.int32)
    tok = np.ascontiguousarray(tree.token, np.int32)
    rc = lib.orc_verify_tree(ctypes.byref(cm), ck.ctypes.data, cv.ctypes.data, int(cache.ctx_len),
                             int(cache.capacity), par.ctypes.data, tok.ctypes.data, n,
                             _ptr(out["logits"]), _ptr(out["q"]), _ptr(out["k"]), _ptr(out["v"]),
                             _ptr(out["attn"]), _ptr(out["hf"]))
    if rc != 0:
        raise MemoryError("oracle verify failed")
    del keep
    return {k: v for k, v in out.items() if v is not None}


def decode_sequence(model, cache, tokens: Sequence[int]) -> dict:
    """Plain one-token-at-a-time decoding of ``tokens`` after the cached context
    (token t at position ctx + t).  Returns logits [len, V], k/v [len, Hkv*D],
    attn [len, Hq*D], hf [len, H]."""
    d = model.dims
    lib = _load()
    L = len(tokens)
    QD, KD = d.n_q_heads * d.head_dim, d.n_kv_heads * d.head_dim
    out = {"logits": np.empty((L, d.vocab), np.float32), "k": np.empty((L, KD), np.uint16),
           "v": np.empty((L, KD), np.uint16), "attn": np.empty((L, QD), np.uint16),
           "hf": np.empty((L, d.hidden), np.uint16)}
    cm, keep = _c_model(model)
    ck = np.ascontiguousarray(cache.k, np.uint16)
    cv = np.ascontiguousarray(cache.v, np.uint16)
    tok = np.ascontiguousarray(tokens, np.int32)
    rc = lib.orc_decode_sequence(ctypes.byref(cm), ck.ctypes.data, cv.ctypes.data, int(cache.ctx_len),
                                 int(cache.capacity), tok.ctypes.data, L, out["logits"].ctypes.data,
                                 out["k"].ctypes.data, out["v"].ctypes.data, out["attn"].ctypes.data,
                                 out["hf"].ctypes.data)
    if rc != 0:
        raise MemoryError("oracle decode failed")
    del keep
    return out


def head_rows(model, hf_bits: np.ndarray, vocab_ids: Sequence[int]) -> np.ndarray:
    """fp32 logits of the given hf rows ([n, H] bf16 bits) at the given vocab
    ids only -> [n, len(vocab_ids)]."""
    lib = _load()
    hf = np.ascontiguousarray(hf_bits, np.uint16)
    vid = np.ascontiguousarray(vocab_ids, np.int32)
    out = np.empty((hf.shape[0], vid.shape[0]), np.float32)
    cm, keep = _c_model(model)
    if lib.orc_head_rows(ctypes.byref(cm), hf.ctypes.data, hf.shape[0], vid.ctypes.data, vid.shape[0],
                         out.ctypes.data) != 0:
        raise MemoryError("oracle head failed")
    del keep
    return out


def verify_joint(model, requests) -> dict:
    """Joint verify of several requests [Exactness, §Parallel requests]: each
    request's rows see only its own cache and its own ancestors, so the joint
    result is every request's lone result, concatenated in request order."""
    parts = [verify_tree(model, r.cache, r.tree) for r in requests]
    return {k: np.concatenate([p[k] for p in parts]) for k in parts[0]}


# ---------------------------------------------------------------------------
# greedy choice and the near-tie rule
# ---------------------------------------------------------------------------
def argmax_top2(logits: np.ndarray):
    """Per row of fp32 logits: argmax (lowest index among equal maxima), the top
    value l1, the second value l2 (the largest value at any other index) and
    gap = l1 - l2.  The decision is taken on the fp32 values, the precision the
    head returns."""
    lg = np.asarray(logits, np.float32)
    idx = np.argmax(lg, axis=1)
    rows = np.arange(lg.shape[0])
    l1 = lg[rows, idx].astype(np.float64)
    rest = lg.astype(np.float64)
    rest[rows, idx] = -np.inf
    l2 = rest.max(axis=1)
    return idx.astype(np.int32), l1, l2, l1 - l2


def bf16_ulp(x) -> np.ndarray:
    """One BF16 step at x: 2^(floor(log2|x|) - 7).  BF16 keeps 8 significant
    bits, so a logit in [16, 32) moves in steps of 0.125 [Exactness, §Parallel
    requests]."""
    a = np.abs(np.asarray(x, np.float64))
    a = np.where(a > 0, a, np.finfo(np.float64).tiny)
    return np.exp2(np.floor(np.log2(a)) - 7.0)


def near_tie(l1, l2) -> np.ndarray:
    """True where the top-2 gap is within one BF16 ulp of the top logit; there
    either token is an acceptable greedy choice [Exactness, §The one exception:
    near ties]."""
    return (np.asarray(l1) - np.asarray(l2)) <= bf16_ulp(l1)


# ---------------------------------------------------------------------------
# accept walks
# ---------------------------------------------------------------------------
def _children(parent: Sequence[int]):
    n = len(parent)
    kids = [[] for _ in range(n)]
    for c in range(1, n):
        kids[int(parent[c])].append(c)      # increasing node index
    return kids


def accept_greedy(parent, token, argmax, choose=None):
    """Greedy accept [Drafters and tree verify, §The round, step 3]: start at the
    root; at each node take the model's token; move to the child carrying it;
    stop where no child does; the model's token at the stopping node is kept
    too, so a round yields at least one token.

    ``argmax[i]`` is row i's greedy token.  ``choose(i)``, when given, returns
    the token to take at row i instead (used to replay a near-tie choice).
    Returns (path, out_tokens): path = node indices root first (the rows whose
    KV is committed); out_tokens = tokens of the accepted non-root nodes, then
    the stopping node's token.
    """
    kids = _children(parent)
    path, cur = [0], 0
    while True:
        t = int(argmax[cur]) if choose is None else int(choose(cur))
        nxt = next((c for c in kids[cur] if int(token[c]) == t), None)
        if nxt is None:
            out = [int(token[c]) for c in path[1:]] + [t]
            return path, out
        path.append(nxt)
        cur = nxt


def softmax_t(logits_row: np.ndarray, temperature: float) -> np.ndarray:
    """p = softmax(logits / T) in fp64 (max subtracted)."""
    z = np.asarray(logits_row, np.float64) / float(temperature)
    z = z - z.max()
    e = np.exp(z)
    return e / e.sum()


def inverse_cdf(r: np.ndarray, u: float) -> int:
    """Smallest y with sum_{j<=y} r(j) > u * sum(r), summing in vocab order; if
    rounding leaves no such y, the last y with r(y) > 0."""
    c = np.cumsum(r)
    y = int(np.searchsorted(c, float(u) * c[-1], side="right"))
    if y >= r.shape[0]:
        y = int(np.nonzero(r > 0)[0][-1])
    return y


def accept_residual(parent, token, logits, temperature: float, uniforms, bonus_at_leaf: bool = True,
                    replay=None, eps: float = 0.0):
    """Deterministic-candidate residual sampling over a draft tree
    [Algorithm and correctness contract, §Deterministic tree candidates and
    residual verification].

    At the current node, r starts as the target distribution p of that node's
    row.  Its children (candidates, tried in increasing node index) are tested
    in turn: candidate x is accepted with probability r(x) (draw u, accept iff
    u < r(x)); on rejection x is removed from r and r renormalised before the
    next sibling.  On acceptance the walk follows only that branch.  If every
    candidate fails, one draw from the residual r is emitted and the round
    ends.  At a leaf the round ends; with ``bonus_at_leaf`` one draw from p is
    kept there too (the target's own token at the stopping point, as
    [Drafters and tree verify, §The round, step 3] keeps it; the MoonBit
    library ends a leaf round without it).

    Uniforms are consumed as one sequential stream: one per candidate test,
    one for the final residual / bonus draw.

    ``replay`` = (path, out_tokens) of another implementation: at a decision
    whose margin is within ``eps`` (|u - r(x)| for a test, the distance of the
    scaled draw to a CDF boundary for a draw), follow ``replay`` if its choice
    is one of the choices within ``eps``.  Returns (path, out_tokens, n_replayed).
    """
    kids = _children(parent)
    draws = iter([float(u) for u in uniforms])
    path, out, cur, replayed = [0], [], 0, 0
    while True:
        p = softmax_t(logits[cur], temperature)
        r = p.copy()
        accepted = None
        for c in kids[cur]:
            x = int(token[c])
            u = next(draws)
            ok = u < r[x]
            if replay is not None and abs(u - r[x]) <= eps:
                rp = replay[0]
                want = len(rp) > len(path) and rp[len(path)] == c
                if want != ok:
                    ok = want
                    replayed += 1
            if ok:
                accepted = c
                break
            r[x] = 0.0                      # remove x and renormalise
            r = r / r.sum()
        if accepted is not None:
            path.append(accepted)
            out.append(int(token[accepted]))
            cur = accepted
            continue
        if kids[cur] or bonus_at_leaf:
            u = next(draws)
            y = inverse_cdf(r, u)
            if replay is not None and len(replay[1]) > len(out):
                yg = int(replay[1][len(out)])
                if yg != y and r[yg] > 0:
                    c = np.cumsum(r)
                    lo = c[yg - 1] if yg > 0 else 0.0
                    t = u * c[-1]
                    if lo - eps * c[-1] <= t < c[yg] + eps * c[-1]:
                        y = yg
                        replayed += 1
            out.append(y)
        return path, out, replayed


# ---------------------------------------------------------------------------
# commit
# ---------------------------------------------------------------------------
def apply_tree_kv(cache, k_rows: np.ndarray, v_rows: np.ndarray):
    """The cache as verify leaves it: node i's K/V at slot ctx + i (the cache
    holds every node at its depth-first slot [Drafters and tree verify, §Tree
    verify through recurrent layers])."""
    Hkv = cache.k.shape[0]
    n = k_rows.shape[0]
    k = cache.k.copy()
    v = cache.v.copy()
    c = cache.ctx_len
    k[:, c:c + n, :] = k_rows.reshape(n, Hkv, -1).transpose(1, 0, 2)
    v[:, c:c + n, :] = v_rows.reshape(n, Hkv, -1).transpose(1, 0, 2)
    return k, v


def commit_kv(k: np.ndarray, v: np.ndarray, ctx: int, path: Sequence[int]):
    """Keep the accepted path's KV rows and drop the rest [Drafters and tree
    verify, §The round, step 4]: the commit gathers the accepted rows down into
    place, slot ctx + path[d] -> slot ctx + d for d = 0..a, every KV head.  All
    sources are read before any row is written.  Returns (k, v, committed_src,
    new_ctx) with committed_src[d] = ctx + path[d] and new_ctx = ctx + a + 1."""
    src = [ctx + int(p) for p in path]
    rows_k = [k[:, s, :].copy() for s in src]
    rows_v = [v[:, s, :].copy() for s in src]
    k2, v2 = k.copy(), v.copy()
    for d in range(len(src)):
        k2[:, ctx + d, :] = rows_k[d]
        v2[:, ctx + d, :] = rows_v[d]
    return k2, v2, src, ctx + len(src)
