"""Parity rules between the CUDA path and the oracle (shared by the GPU tests).

* fp32 logits: max |gpu - oracle| <= 2e-2 x the oracle row's RMS logit (the
  "logit scale");
* attention outputs: max abs error <= 1e-2;
* the tree rows' K/V (bf16 stores of values up to ~6 at hidden 5120): error
  <= 1e-2 x max(1, |oracle value|), which admits one bf16 step (2^-7 relative)
  where fp32 and fp64 accumulations round to different sides;
* greedy choice: the GPU's argmax equals the oracle's, except where the
  oracle's top-2 gap is within one BF16 ulp of its top logit, where the
  second token is accepted too [Exactness, §The one exception: near ties];
* accepted ids, accept lengths and committed indices: bit-exact after the
  oracle walk replays the GPU's choice at those near ties;
* sampled walks: bit-exact after replaying the GPU's choice where a decision
  lies within ``eps`` of its threshold.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from speculative_tree_verify_gb300 import abi
from speculative_tree_verify_gb300 import device as dv
from speculative_tree_verify_gb300.device import DeviceModel, DeviceRequest, RoundBuffers

LOGIT_TOL = 2e-2
ATTN_TOL = 1e-2
KV_TOL = 1e-2


def to_np(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return oracle.bf16_to_f64(bits)


def check_logits(orc: np.ndarray, gpu: np.ndarray, tol: float = LOGIT_TOL) -> float:
    """Returns the worst error as a fraction of the row's logit scale."""
    o = orc.astype(np.float64)
    g = gpu.astype(np.float64)
    assert np.all(np.isfinite(g)), "non-finite GPU logits"
    scale = np.sqrt((o * o).mean(axis=1))
    err = np.abs(g - o).max(axis=1)
    frac = err / scale
    assert np.all(frac <= tol), f"logit error {frac.max():.3e} x scale > {tol}"
    return float(frac.max())


def check_close_bf16(orc_bits: np.ndarray, gpu_bits: np.ndarray, tol: float, what: str,
                     relative: bool = False) -> float:
    """max |gpu - oracle| <= tol (absolute), or <= tol * max(1, |oracle|) when
    ``relative``.  Returns the worst error in those units."""
    o = bf16_to_f64(orc_bits)
    g = bf16_to_f64(gpu_bits)
    if not o.size:
        return 0.0
    denom = np.maximum(1.0, np.abs(o)) if relative else 1.0
    err = float((np.abs(g - o) / denom).max())
    assert err <= tol, f"{what}: max {'relative ' if relative else ''}error {err:.3e} > {tol}"
    return err


def second_index(logits: np.ndarray) -> np.ndarray:
    idx = np.argmax(logits, axis=1)
    m = logits.astype(np.float64).copy()
    m[np.arange(m.shape[0]), idx] = -np.inf
    return np.argmax(m, axis=1)


def check_argmax(orc_logits: np.ndarray, gpu_argmax: np.ndarray, gpu_gap: np.ndarray, gap_tol: float = None) -> int:
    """GPU argmax must be the oracle's, or its second token at a near tie.
    Returns the number of near-tie rows where the GPU took the second token."""
    idx, l1, l2, gap = oracle.argmax_top2(orc_logits)
    tie = oracle.near_tie(l1, l2)
    sec = second_index(orc_logits)
    swapped = 0
    for r in range(orc_logits.shape[0]):
        g = int(gpu_argmax[r])
        if g != int(idx[r]):
            assert tie[r] and g == int(sec[r]), (
                f"row {r}: gpu argmax {g}, oracle {idx[r]} (gap {gap[r]:.4g}, ulp {oracle.bf16_ulp(l1[r]):.4g})")
            swapped += 1
    scale = np.sqrt((orc_logits.astype(np.float64) ** 2).mean(axis=1))
    tol = (gap_tol if gap_tol is not None else 2 * LOGIT_TOL) * scale
    assert np.all(np.abs(gpu_gap.astype(np.float64) - gap) <= tol), "top-2 gap mismatch"
    return swapped


def greedy_replay(parent, token, orc_logits: np.ndarray, gpu_argmax: np.ndarray):
    """The oracle's greedy walk, taking the GPU's token where the oracle allows
    either (near ties)."""
    idx, l1, l2, _ = oracle.argmax_top2(orc_logits)
    tie = oracle.near_tie(l1, l2)
    sec = second_index(orc_logits)

    def choose(i):
        g = int(gpu_argmax[i])
        if g == int(idx[i]):
            return g
        assert tie[i] and g == int(sec[i]), f"row {i}: not a near tie"
        return g

    return oracle.accept_greedy(parent, token, idx, choose=choose)


def spine(parent) -> list:
    """Root, then the first child (lowest index) of each node, down to a leaf."""
    n = len(parent)
    path, cur = [0], 0
    while True:
        kids = [c for c in range(1, n) if int(parent[c]) == cur]
        if not kids:
            return path
        cur = kids[0]
        path.append(cur)


def plant_spine(model, cache, tree, depth: int = 1 << 30):
    """Teacher-forced drafts: write the oracle's own greedy token into the spine
    nodes (up to ``depth`` of them), so that the walk has something to accept.
    Siblings that collide with a planted token are re-drawn."""
    par = tree.parent
    tok = tree.token.copy()
    sp = spine(par)[: depth + 1]
    V = model.dims.vocab
    rng = np.random.default_rng(int(tok[0]) + 7)
    seq = [int(tok[0])]
    for d in range(1, len(sp)):
        dec = oracle.decode_sequence(model, cache, seq)
        t = int(np.argmax(dec["logits"][-1]))
        tok[sp[d]] = t
        for c in range(1, len(par)):
            if c != sp[d] and par[c] == par[sp[d]] and tok[c] == t:
                while True:
                    x = int(rng.integers(0, V))
                    if all(tok[s] != x for s in range(1, len(par)) if par[s] == par[c]):
                        tok[c] = x
                        break
        seq.append(t)
    tree.token[:] = tok
    return sp


# ---------------------------------------------------------------------------
# running a verify through the C ABI and comparing it with the oracle
# ---------------------------------------------------------------------------
def _ok(rc, what="call"):
    assert rc == abi.TV_OK, f"{what}: {abi.STATUS.get(rc, rc)}"


def gpu_verify(dm: DeviceModel, host_reqs, with_attn=True):
    reqs = [DeviceRequest.from_host(c, t) for c, t in host_reqs]
    rows = sum(r.n for r in reqs)
    b = RoundBuffers.alloc(dm.dims, rows, len(reqs), max(c.ctx_len for c, _ in host_reqs))
    _ok(dv.verify(dm, reqs, b, with_attn=with_attn), "tv_verify_tree")
    torch.cuda.synchronize()
    assert int(b.status.item()) == 0, abi.STATUS.get(int(b.status.item()))
    return reqs, b


def check_verify(model, host_reqs, dm=None, reqs_b=None):
    """Full comparison of one (joint) verify with the oracle."""
    dm = dm or DeviceModel.from_host(model)
    reqs, b = reqs_b or gpu_verify(dm, host_reqs)
    orc = [oracle.verify_tree(model, c, t) for c, t in host_reqs]
    logits = np.concatenate([o["logits"] for o in orc])
    stats = {"logit_err": check_logits(logits, to_np(b.logits)),
             "swapped": check_argmax(logits, to_np(b.argmax), to_np(b.gap)),
             "attn_err": check_close_bf16(np.concatenate([o["attn"] for o in orc]), to_np(b.attn), ATTN_TOL, "attn")}
    Hkv = model.dims.n_kv_heads
    stats["kv_err"] = 0.0
    for (c, t), o, r in zip(host_reqs, orc, reqs):
        ctx, n = c.ctx_len, t.n
        k, v = to_np(r.k), to_np(r.v)
        ek = check_close_bf16(o["k"], k[:, ctx:ctx + n, :].transpose(1, 0, 2).reshape(n, -1), KV_TOL, "tree K",
                              relative=True)
        ev = check_close_bf16(o["v"], v[:, ctx:ctx + n, :].transpose(1, 0, 2).reshape(n, -1), KV_TOL, "tree V",
                              relative=True)
        stats["kv_err"] = max(stats["kv_err"], ek, ev)
        np.testing.assert_array_equal(k[:, :ctx], c.k[:, :ctx])           # cached rows are only read
        np.testing.assert_array_equal(v[:, :ctx], c.v[:, :ctx])
        np.testing.assert_array_equal(k[:, ctx + n:], c.k[:, ctx + n:])   # nothing past the tree rows
        np.testing.assert_array_equal(v[:, ctx + n:], c.v[:, ctx + n:])
        assert k.shape[0] == Hkv
    return orc, reqs, b, stats
