#!/usr/bin/env python
"""Benchmark of the GB300 tree verify round.

One step = one verify round on one GPU at the hidden-5120 shapes (40/8 heads
of 128, vocab 151936, bf16 weights ~ N(0, 0.02) drawn on the device):
tv_verify_tree over a 16-row lattice tree (spine of 8 + 8 next-best branches)
at 1024 tokens of context, tv_accept_greedy_commit (the greedy walk and the KV
commit in one launch).  The drafts along
the spine are teacher-forced (the GPU's own greedy tokens, planted before
timing) so the walk and the commit do real work.  Inputs are synthetic.

Printed: one JSON line (rank 0).  value = ms per round from CUDA-graph replay
(the served configuration keeps verify in graphs), the mean over the timed
steps; step_ms_spread gives the median and 10th/90th percentiles of single
replays; clocks are sampled over the eager and the graph timed regions.  The
eager number, the row
sweep 8/16/24/32, a sampled round (residual walk), the sampled variants (filter,
single-draw, Gumbel and rejection walks alone and in rounds), the Gated DeltaNet
recurrent core of 48 layers and their path-state commit, per-stage times, the
roofline of the LM head kernel, end-to-end latency with host buffers, clocks
and the CPU oracle baseline ride along.

--impl reference times the CPU oracle (the only reference there is) on the
same workload on the host cores.

Under torchrun (N > 1) every rank runs an independent replica on its own GPU:
the round has no cross-GPU exchange, so there is no collective on the data
path ("replicas only"); the barrier and the max-over-ranks timing use a
process group.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "tree-verify latency (ms) at 8-32 nodes, 1k ctx; achieved HBM GB/s vs peak"
UNIT = "ms"
ROWS, CTX, SLOTS = 16, 1024, 7
WORKLOAD = "tree verify round (verify + greedy accept + commit), hidden 5120 layer + 151936-vocab head, " \
           "16-row lattice tree (spine 8 + 8 branches), 1024-token context"


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extras", action="store_true", help="only the headline number (for profiling runs)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--rows", type=int, default=ROWS, help="tree rows of the timed round (profiling runs)")
    ap.add_argument("--ctx", type=int, default=CTX, help="cached context of the timed round (profiling runs)")
    ap.add_argument("--no-stack", action="store_true", help="skip the 64-layer stack section")
    ap.add_argument("--only-stack", action="store_true", help="only the stack section (profiling runs)")
    ap.add_argument("--stack-layers", type=int, default=64, help="layers of the stack section (profiling runs)")
    return ap.parse_args()


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _max_over_ranks(vals, device):
    """Each value's maximum over the ranks (the slowest replica's time)."""
    t = torch.tensor(list(vals), dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t]


def _code_sha256() -> str:
    h = hashlib.sha256()
    for sub in ("include", os.path.join("speculative_tree_verify_gb300", "csrc")):
        d = os.path.join(ROOT, sub)
        for f in sorted(os.listdir(d)):
            with open(os.path.join(d, f), "rb") as fh:
                h.update(f.encode())
                h.update(fh.read())
    return h.hexdigest()


def _head_kernel_sha256() -> str:
    """sha256 over the sources the LM-head kernel is compiled from, in this
    order: tv_common.cuh, tv_gemm.cuh, tv_gemm.cu."""
    h = hashlib.sha256()
    for f in ("tv_common.cuh", "tv_gemm.cuh", "tv_gemm.cu"):
        with open(os.path.join(ROOT, "speculative_tree_verify_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            j = json.load(fh)
        return float(j["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def _ncu_traffic(kernel_sha: str):
    """DRAM bytes per launch of the LM head kernel from the committed ncu
    summary, if it was taken on the current kernel source."""
    p = os.path.join(ROOT, "profiles", "lm_head_hidden5120_ncu.md")
    if not os.path.exists(p):
        return None
    vals = {}
    for line in open(p):
        if ":" in line and line.strip().startswith(("traffic_bytes_per_launch", "kernel_source_sha256", "rows")):
            k, v = line.strip().split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_sha256") != kernel_sha or "traffic_bytes_per_launch" not in vals:
        return None
    return float(vals["traffic_bytes_per_launch"]), int(vals.get("rows", "0") or 0)


class Clocks:
    """nvidia-smi samples every 200 ms while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, local_rank: int):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        self.idx = vis.split(",")[local_rank] if vis else str(local_rank)
        self.f = tempfile.TemporaryFile(mode="w+")
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                       "-lms", "200", "-i", self.idx], stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return None
        time.sleep(0.25)
        self.p.terminate()
        self.p.wait()
        self.f.seek(0)
        sm, mx, reasons = [], [], set()
        for line in self.f:
            c = [x.strip() for x in line.split(",")]
            if len(c) < 9:
                continue
            try:
                sm.append(float(c[1]))
                mx.append(float(c[2]))
            except ValueError:
                continue
            for name, v in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"),
                               c[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# workload
# ---------------------------------------------------------------------------
def _make_request(dv, synth, D, tree, ctx, seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    cap = ctx + 64
    k = torch.randn(D.n_kv_heads, cap, D.head_dim, generator=g, device=device).to(torch.bfloat16)
    v = torch.randn(D.n_kv_heads, cap, D.head_dim, generator=g, device=device).to(torch.bfloat16)
    return dv.DeviceRequest(k, v, ctx, torch.from_numpy(tree.parent.copy()).to(device),
                            torch.from_numpy(tree.token.copy()).to(device))


def _plant(dv, dm, req, b, spine):
    """Teacher forcing on the GPU: spine node d+1 gets the token the model
    picks at spine node d (siblings re-drawn on a collision)."""
    par = req.parent.cpu().numpy()
    tok = req.token.cpu().numpy()
    rng = np.random.default_rng(0)
    for d in range(1, len(spine)):
        req.token.copy_(torch.from_numpy(tok))
        dv.check(dv.verify(dm, [req], b), "verify")
        t = int(b.argmax[spine[d - 1]])
        tok[spine[d]] = t
        for c in range(1, len(par)):
            if c != spine[d] and par[c] == par[spine[d]] and tok[c] == t:
                tok[c] = (t + 1 + int(rng.integers(0, 1000))) % dm.dims.vocab
    req.token.copy_(torch.from_numpy(tok))


def _spine(parent):
    path, cur = [0], 0
    while True:
        kids = [c for c in range(1, len(parent)) if int(parent[c]) == cur]
        if not kids:
            return path
        cur = kids[0]
        path.append(cur)


def _graph(fn, warm=3):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(warm):
            fn()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def _time_graph(g, steps):
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


class L2Flush:
    """Flushes the L2 between timed regions: a write of twice the L2 size
    (queried from the device, not assumed), then a read of another buffer of
    that size, so that the L2 holds none of the timed work's data and no
    dirty lines whose write-back the timed work would pay for."""

    def __init__(self, device):
        self.l2 = int(torch.cuda.get_device_properties(device).L2_cache_size)
        self.w = torch.empty(2 * self.l2, dtype=torch.uint8, device=device)
        self.r = torch.zeros(2 * self.l2 // 4, dtype=torch.int32, device=device)

    def __call__(self):
        self.w.zero_()
        self.r.max()


def _l2_flush_buffer(device):
    f = L2Flush(device)
    return f, f.l2


def _time_graph_flushed(g, steps, flush):
    """Mean per-replay time with the L2 flushed before every replay (outside
    the timed regions), CUDA events around each replay alone."""
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in ev:
        flush()
        a.record()
        g.replay()
        b.record()
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in ev) / steps


def _step_spread(g, steps):
    """Per-replay times of a graph (an event between consecutive replays):
    median and 10th/90th percentiles, for the spread behind the mean."""
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ev[0].record()
    for i in range(steps):
        g.replay()
        ev[i + 1].record()
    torch.cuda.synchronize()
    d = sorted(ev[i].elapsed_time(ev[i + 1]) for i in range(steps))
    pick = lambda f: round(d[min(steps - 1, int(f * steps))], 4)
    return {"median": pick(0.5), "p10": pick(0.1), "p90": pick(0.9), "samples": steps}


def verify_bytes(D, n, ctx):
    """Algorithmic bytes one verify must move: every weight once, the cached
    K/V once, the fp32 logits once; embeddings and tree K/V rows are < 0.5 MB."""
    H, V, QD = D.hidden, D.vocab, D.n_q_heads * D.head_dim
    weights = V * H * 2 + D.qkv_out * H * 2 + H * QD * 2
    kv = ctx * D.n_kv_heads * D.head_dim * 2 * 2
    return weights + kv + n * V * 4


def head_bytes(D, n):
    return D.vocab * D.hidden * 2 + n * D.vocab * 4 + n * D.hidden * 2


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------
def _host_model(dm, synth):
    def bits(t):
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return synth.Model(dm.dims, *(bits(dm.t[k]) for k in ("embed", "ln1", "wqkv", "wo", "ln_f", "lm_head")))


def _host_cache(req, synth):
    def bits(t):
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return synth.Cache(bits(req.k), bits(req.v), req.ctx_len, req.capacity)


def oracle_full_round(oracle, model, cache, tree):
    out = oracle.verify_tree(model, cache, tree, want=("logits", "k", "v"))
    idx, _, _, _ = oracle.argmax_top2(out["logits"])
    path, _ = oracle.accept_greedy(tree.parent, tree.token, idx)
    k, v = oracle.apply_tree_kv(cache, out["k"], out["v"])
    oracle.commit_kv(k, v, cache.ctx_len, path)


def oracle_sampled_step(oracle, model, cache, tree, r_rows, vocab_ids):
    """A bounded sample of one round: the layer over the first r_rows nodes (a
    valid smaller tree) and the head over a vocabulary slice.  Returns
    (layer seconds, head seconds)."""
    sub = type(tree)(tree.parent[:r_rows].copy(), tree.token[:r_rows].copy())
    t0 = time.perf_counter()
    out = oracle.verify_tree(model, cache, sub, want=("hf",))
    t1 = time.perf_counter()
    oracle.head_rows(model, out["hf"], vocab_ids)
    t2 = time.perf_counter()
    return t1 - t0, t2 - t1


def one_thread_round_ms(oracle, model, cache, tree, seconds):
    """The oracle on ONE host thread: a bounded sample of the round (the layer
    over a prefix of the tree's rows, the head over a vocabulary slice),
    scaled to ms per full round; the median of three samples.  Returns
    (ms, what the sample was)."""
    n, V = tree.n, model.dims.vocab
    prev = oracle.num_threads()
    oracle.set_num_threads(1)
    try:
        rng = np.random.default_rng(1)
        ids = np.sort(rng.choice(V, size=min(V, 512), replace=False)).astype(np.int32)
        r0 = min(n, 2)
        tl, th = oracle_sampled_step(oracle, model, cache, tree, r0, ids)
        per_row = tl / r0
        per_rv = th / (r0 * len(ids))
        budget = seconds / 6.0                 # three samples of a third each, half layer, half head
        r_rows = int(max(1, min(n, (budget / 2) / max(per_row, 1e-9))))
        s_voc = int(max(256, min(V, (budget / 2) / max(per_rv * r_rows, 1e-12))))
        vids = np.sort(rng.choice(V, size=s_voc, replace=False)).astype(np.int32)
        est = []
        for _ in range(3):
            a, h = oracle_sampled_step(oracle, model, cache, tree, r_rows, vids)
            est.append(1e3 * (a * n / r_rows + h * (n / r_rows) * (V / s_voc)))
    finally:
        oracle.set_num_threads(prev)
    return statistics.median(est), (f"1 thread: the layer over the first {r_rows} of {n} rows and the head over "
                                    f"{s_voc} of {V} vocabulary rows, scaled to a full round; median of 3")


def cpu_baseline(oracle, model, cache, tree, seconds):
    t0 = time.perf_counter()
    oracle_full_round(oracle, model, cache, tree)
    one = time.perf_counter() - t0
    reps = max(1, min(20, int(seconds / max(one, 1e-3))))
    ts = [one]
    for _ in range(reps - 1):
        t0 = time.perf_counter()
        oracle_full_round(oracle, model, cache, tree)
        ts.append(time.perf_counter() - t0)
    ms = 1e3 * statistics.median(ts)
    ms1, sample1 = one_thread_round_ms(oracle, model, cache, tree, seconds / 2)
    return {"value": ms, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{len(ts)} full rounds (verify of all {tree.n} rows over the full vocabulary, greedy walk, "
                      f"commit), median",
            "value_1_thread": round(ms1, 3), "sample_1_thread": sample1}


def stack_bytes(sd, n, ctx):
    """Algorithmic bytes of one verify through the stack: every GEMM weight
    once, each attention layer's cached K/V, each DeltaNet layer's state, the
    logits."""
    b = sd.base
    H, V = b.hidden, b.vocab
    attn = (b.qkv_out + H) * H * 2
    dn = (sd.dn_in_out * H + H * sd.n_v_heads * sd.d_v) * 2
    mlp = 3 * H * sd.intermediate * 2
    L_a, L_d = len(sd.attn_layers), len(sd.dn_layers)
    kv = L_a * ctx * b.n_kv_heads * b.head_dim * 2 * 2
    state = L_d * sd.n_v_heads * sd.d_k * sd.d_v * 4
    return L_a * attn + L_d * dn + sd.n_layers * mlp + V * H * 2 + kv + state + n * V * 4


def stack_bench(dv, synth, dev, peak, flush, n_layers=64, reps=10):
    """Round time of the 64-layer stack from a CUDA graph, L2 flushed before
    every replay; GB/s against the stack verify's algorithmic bytes."""
    import dataclasses
    sd = dataclasses.replace(synth.STACK_FULL, n_layers=n_layers)
    t0 = time.perf_counter()
    model = dv.DeviceStack.random(sd, 4321, device=dev)
    torch.cuda.synchronize()
    gen_s = time.perf_counter() - t0
    res = {"layers": sd.n_layers, "deltanet_layers": len(sd.dn_layers), "attention_layers": len(sd.attn_layers),
           "intermediate": sd.intermediate, "weights_GB": round(stack_bytes(sd, 0, 0) / 1e9, 3),
           "init_s": round(gen_s, 1), "rows": {}}
    ctx = CTX
    for n in (8, 16, 32):
        tree = synth.tree_lattice(n, SLOTS if n <= 16 else 15, sd.base.vocab, 7)
        gk = torch.Generator(device=dev)
        gk.manual_seed(77 + n)
        cap = ctx + 64
        ks = [torch.randn(sd.base.n_kv_heads, cap, sd.base.head_dim, generator=gk, device=dev).to(torch.bfloat16)
              for _ in sd.attn_layers]
        vs = [torch.randn_like(k) for k in ks]
        st = torch.randn(len(sd.dn_layers), sd.n_v_heads, sd.d_k, sd.d_v, generator=gk, device=dev) * 0.3
        req = dv.StackRequest(ks, vs, ctx, st, torch.from_numpy(tree.parent.copy()).to(dev),
                              torch.from_numpy(tree.token.copy()).to(dev))
        b = dv.StackBuffers.alloc(model, n, 1, device=dev)

        def round_():
            dv.run_stack_round(model, [req], b, stream=torch.cuda.current_stream())

        for _ in range(3):
            round_()
        torch.cuda.synchronize()
        if int(b.status.item()) != 0:
            raise RuntimeError(f"stack round: device status {int(b.status.item())}")
        gs = _graph(round_)
        ms = _time_graph_flushed(gs, reps, flush)
        del gs
        by = stack_bytes(sd, n, ctx)
        res["rows"][str(n)] = {"round_ms": round(ms, 4), "GB_per_s": round(by / ms / 1e6, 1),
                               "frac_of_peak": round(by / ms / 1e6 / peak, 4), "verify_bytes": by}
        del req, b, ks, vs, st
    res["ratio_32_over_8"] = round(res["rows"]["32"]["round_ms"] / res["rows"]["8"]["round_ms"], 4)
    del model
    torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------------------
def run_ours(args, world, rank, local):
    from speculative_tree_verify_gb300 import abi, build, synth
    from speculative_tree_verify_gb300 import device as dv

    build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if args.only_stack:
        peak, _ = _peaks()
        flush, _ = _l2_flush_buffer(dev)
        return {"stack": stack_bench(dv, synth, dev, peak, flush, args.stack_layers, args.steps)}
    D = synth.FULL
    dm = dv.DeviceModel.random(D, 1234 + rank, device=dev)
    rows, ctx = args.rows, args.ctx
    tree = synth.tree_lattice(rows, SLOTS if rows <= 16 else 15, D.vocab, 7)
    req = _make_request(dv, synth, D, tree, ctx, 99 + rank, dev)
    b = dv.RoundBuffers.alloc(D, rows, 1, ctx, device=dev)
    _plant(dv, dm, req, b, _spine(tree.parent))
    def round_():
        dv.run_round(dm, [req], b, stream=torch.cuda.current_stream())

    for _ in range(max(3, args.warmup)):
        round_()
    torch.cuda.synchronize()
    st = int(b.status.item())
    if st != 0:
        raise RuntimeError(f"device status {abi.STATUS.get(st, st)}")
    accept_len = int(b.accept_len[0])

    # ---- eager, K steps, clocks sampled during the timed region --------------
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clk = Clocks(local)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        round_()
    e1.record()
    torch.cuda.synchronize()
    eager_ms = e0.elapsed_time(e1) / args.steps

    # ---- the same round from a CUDA graph (the reported value); the clock
    #      samples cover both timed regions ------------------------------------------
    g = _graph(round_)
    graph_ms = _time_graph(g, args.steps)
    # the reported value: the same replays with the L2 flushed before each one
    flush, l2_bytes = _l2_flush_buffer(dev)
    flushed_ms = _time_graph_flushed(g, args.steps, flush)
    clocks = clk.stop()
    spread = _step_spread(g, min(args.steps, 500))
    if world > 1:
        flushed_ms, graph_ms, eager_ms = _max_over_ranks([flushed_ms, graph_ms, eager_ms], dev)
        torch.distributed.barrier()

    out = {"metric": METRIC, "value": round(flushed_ms, 4), "unit": UNIT, "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": round(flushed_ms, 4), "higher_is_better": False,
           "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
           "config": {"workload": WORKLOAD if (rows, ctx) == (ROWS, CTX) else
                      WORKLOAD.replace("16-row", f"{rows}-row").replace("1024-token", f"{ctx}-token"),
                      "hidden": D.hidden, "heads": f"{D.n_q_heads}/{D.n_kv_heads}x{D.head_dim}",
                      "vocab": D.vocab, "rows": rows, "ctx": ctx, "accept_len": accept_len,
                      "l2": f"flushed before every timed replay: {2 * l2_bytes} B (2x the queried L2) written, "
                            f"then another {2 * l2_bytes} B read; the 1.68 GB of weights exceed L2 either way",
                      "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
           "eager_ms_per_step": round(eager_ms, 4), "back_to_back_ms_per_step": round(graph_ms, 4),
           "step_ms_spread": spread, "clocks": clocks,
           "gpu_launches": 9 * args.steps, "code_sha256": _code_sha256()}
    if rank != 0 or args.no_extras:
        return out if rank == 0 else None

    # ---- per-stage times of the verify (eager, events on the launch stream) -----
    P = 200
    dv.check(abi.tv_profile_start(P), "tv_profile_start")
    for _ in range(P):
        dv.check(dv.verify(dm, [req], b, stream=torch.cuda.current_stream()), "verify")
    rc, stage_sum, calls = abi.tv_profile_stop()
    dv.check(rc, "tv_profile_stop")
    stage_us = {k: round(1e3 * v / calls, 2) for k, v in stage_sum.items()}
    peak, peak_kind = _peaks()
    head_s = stage_sum["lm_head"] / calls / 1e3
    hb = head_bytes(D, rows)
    achieved = hb / head_s / 1e9
    tr = _ncu_traffic(_head_kernel_sha256())
    out["roofline"] = {"kernel": "lm_head (tcgen05 skinny GEMM + fused argmax/top-2)", "bound": "hbm",
                       "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                       "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                       "algorithmic_bytes_per_launch": hb,
                       "traffic": None if tr is None else tr[0] * 1.0,
                       "launch_us": round(head_s * 1e6, 2)}
    out["stage_us"] = stage_us

    # ---- row sweep: verify-only latency from graphs -----------------------------
    sweep = {}
    for n in (8, 16, 24, 32):
        t = synth.tree_spine_random(n, min(16, n), D.vocab, 30 + n)
        r = _make_request(dv, synth, D, t, CTX, 200 + n, dev)
        bb = dv.RoundBuffers.alloc(D, n, 1, CTX, device=dev)

        def vf(r=r, bb=bb):
            dv.check(dv.verify(dm, [r], bb, stream=torch.cuda.current_stream()), "verify")

        gg = _graph(vf)
        ms = _time_graph(gg, max(200, args.steps // 4))
        vb = verify_bytes(D, n, CTX)
        sweep[str(n)] = {"verify_ms": round(ms, 4), "tree_rows_per_s": round(n / ms * 1e3, 1),
                         "GB_per_s": round(vb / ms / 1e6, 1), "frac_of_peak": round(vb / ms / 1e6 / peak, 4)}
        del gg
    sweep["ratio_32_over_8"] = round(sweep["32"]["verify_ms"] / sweep["8"]["verify_ms"], 4)
    out["sweep"] = sweep

    # ---- long context: 32768 cached tokens, 32-row lattice tree ------------------
    #      (attention graded here: its 134 MB of K/V stream from HBM; at 1k
    #      context the 4 MB of K/V are L2-sized)
    lc_ctx, lc_rows = 32768, 32
    lt = synth.tree_lattice(lc_rows, 15, D.vocab, 41)
    lr = _make_request(dv, synth, D, lt, lc_ctx, 300, dev)
    lb = dv.RoundBuffers.alloc(D, lc_rows, 1, lc_ctx, device=dev)

    def lvf():
        dv.check(dv.verify(dm, [lr], lb, stream=torch.cuda.current_stream()), "verify")

    gl = _graph(lvf)
    lc_ms = _time_graph(gl, max(100, args.steps // 10))
    del gl
    dv.check(abi.tv_profile_start(P), "tv_profile_start")
    for _ in range(P):
        lvf()
    rc, lsum, lcalls = abi.tv_profile_stop()
    dv.check(rc, "tv_profile_stop")
    kv_bytes = lc_ctx * D.n_kv_heads * D.head_dim * 2 * 2
    att_s = lsum["attention"] / lcalls / 1e3
    out["long_context"] = {
        "ctx": lc_ctx, "rows": lc_rows, "verify_ms": round(lc_ms, 4),
        "verify_GB_per_s": round(verify_bytes(D, lc_rows, lc_ctx) / lc_ms / 1e6, 1),
        "attention_us": round(att_s * 1e6, 2), "attention_kv_bytes": kv_bytes,
        "attention_GB_per_s": round(kv_bytes / att_s / 1e9, 1),
        "attention_frac_of_peak": round(kv_bytes / att_s / 1e9 / peak, 4),
        "stage_us": {k: round(1e3 * v / lcalls, 2) for k, v in lsum.items()}}
    del lr, lb

    # ---- sampled round: residual walk at T = 1 instead of the greedy walk -------
    b.uniforms.copy_(torch.from_numpy(synth.uniforms(rows, 5)))

    def sround():
        dv.run_round(dm, [req], b, sampled=1.0, stream=torch.cuda.current_stream())

    gs = _graph(sround)
    out["sampled_round_ms"] = round(_time_graph(gs, max(200, args.steps // 4)), 4)
    del gs

    # ---- sampled variants: each walk alone on the round's logits (L2-resident,
    #      as they are right after the LM head), then whole rounds with them ----------
    def ok_status(what):
        torch.cuda.synchronize()
        st = int(b.status.item())
        if st != 0:
            raise RuntimeError(f"{what}: device status {abi.STATUS.get(st, st)}")

    sb = dv.SampleBuffers.alloc(D.vocab, rows, device=dev)
    seeds, positions = [0x5EED5EED5EED], [ctx]
    filt = dict(temperature=0.8, top_k=50, top_p=0.9, min_p=0.02)
    cur = torch.cuda.current_stream
    sv = {"rows": rows, "vocab": D.vocab, "filter_params": filt}
    walks = {
        "filter": lambda: dv.check(dv.sample_filter(b, sb, rows, stream=cur(), **filt), "filter"),
        "single_draw": lambda: dv.check(dv.accept_single_draw([req], b, sb, 1.0, stream=cur()), "single_draw"),
        "gumbel": lambda: dv.check(dv.accept_gumbel([req], b, sb, 1.0, seeds, positions, stream=cur()), "gumbel"),
    }
    # single-path rejection: a chain of `rows` drafts, each drawn as its proposal row's mode
    gq = torch.Generator(device=dev)
    gq.manual_seed(17)
    prop = torch.softmax(2.0 * torch.randn(rows, D.vocab, device=dev, generator=gq), dim=1)
    ch_tok = torch.argmax(prop, dim=1).to(torch.int32)
    ch_tok[0] = 0
    chain = dv.DeviceRequest(req.k, req.v, ctx, torch.arange(-1, rows - 1, device=dev, dtype=torch.int32), ch_tok)
    walks["rejection"] = lambda: dv.check(dv.accept_rejection([chain], b, sb, 1.0, prop, stream=cur()), "rejection")
    for name, fn in walks.items():
        gw = _graph(fn)
        sv[name + "_us"] = round(1e3 * _time_graph(gw, 500), 2)
        del gw
        ok_status(name)
    lg = rows * D.vocab * 4
    sv["filter_GB_per_s"] = round(2 * lg / sv["filter_us"] / 1e3, 1)

    def gumbel_round():
        dv.check(dv.verify(dm, [req], b, stream=cur()), "verify")
        dv.check(dv.accept_gumbel([req], b, sb, 1.0, seeds, positions, stream=cur()), "gumbel")
        dv.check(dv.commit([req], b, stream=cur()), "commit")

    def filtered_round():
        dv.check(dv.verify(dm, [req], b, stream=cur()), "verify")
        dv.check(dv.sample_filter(b, sb, rows, stream=cur(), **filt), "filter")
        dv.check(dv.accept_single_draw([req], b, sb, 1.0, filtered=True, stream=cur()), "single_draw")
        dv.check(dv.commit([req], b, stream=cur()), "commit")

    for name, fn in (("gumbel_round_ms", gumbel_round), ("filtered_single_draw_round_ms", filtered_round)):
        gw = _graph(fn)
        sv[name] = round(_time_graph(gw, max(200, args.steps // 4)), 4)
        del gw
        ok_status(name)
    out["sampled_variants"] = sv
    del sb, prop, chain

    # ---- Gated DeltaNet: the recurrent core of 48 layers over the round's tree
    #      (one launch per layer, each on its own state) and the path-state
    #      commit of all 48 layers in one launch; 16 key / 32 value heads of 128 ----
    Hk, Hv, dkn, dvn, NL = 16, 32, 128, 128, 48
    dnd = abi.TvDnDims(Hk, Hv, dkn, dvn)
    dni = synth.dn_inputs(rows, Hk, Hv, dkn, dvn, 808)
    dq, dk_, dv_ = (torch.from_numpy(x).to(dev) for x in (dni.q, dni.k, dni.v))
    dbeta, dg = torch.from_numpy(dni.beta).to(dev), torch.from_numpy(dni.g).to(dev)
    gs = torch.Generator(device=dev)
    gs.manual_seed(909)
    dstate = torch.randn(NL, Hv, dkn, dvn, device=dev, generator=gs) * 0.3
    do_ = torch.empty(rows, Hv, dvn, device=dev)
    du = torch.empty(NL, rows, Hv, dvn, device=dev)
    dgc = torch.empty(NL, rows, Hv, device=dev)
    dks = dk_.unsqueeze(0).expand(NL, -1, -1, -1).contiguous()
    ptr0 = dstate.data_ptr()
    lbytes = Hv * dkn * dvn * 4

    def dn_layers():
        for l in range(NL):
            dv.check(abi.tv_dn_verify_tree(dnd, [req.tree()], [ptr0 + l * lbytes], dq, dk_, dv_, dbeta, dg, do_,
                                           du[l], dgc[l], b.status, stream=cur()), "tv_dn_verify_tree")

    def dn_commit():
        dv.check(abi.tv_dn_commit(dnd, [req.tree()], NL, [dstate], dks, du, dgc, b.path, b.accept_len, b.status,
                                  stream=cur()), "tv_dn_commit")

    round_()   # the greedy path of the round's tree
    gw = _graph(dn_layers)
    dn_v_us = 1e3 * _time_graph(gw, 100)
    del gw
    ok_status("dn verify")
    gw = _graph(dn_commit)
    reps = 200
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        gw.replay()
    e1.record()
    torch.cuda.synchronize()
    dn_c_us = 1e3 * e0.elapsed_time(e1) / reps
    del gw
    ok_status("dn commit")
    a_len = int(b.accept_len[0])
    cbytes = 2 * NL * lbytes + NL * (a_len + 1) * (Hk * dkn + Hv * dvn + Hv) * 4
    out["deltanet"] = {
        "dims": {"key_heads": Hk, "value_heads": Hv, "d_k": dkn, "d_v": dvn, "layers": NL, "rows": rows},
        "verify_48_layers_us": round(dn_v_us, 2), "verify_per_layer_us": round(dn_v_us / NL, 2),
        "verify_state_bytes_per_layer": lbytes,
        "commit_48_layers_us": round(dn_c_us, 2), "commit_accept_len": a_len,
        "commit_algorithmic_bytes": cbytes,
        "commit_GB_per_s": round(cbytes / dn_c_us / 1e3, 1),
        "commit_frac_of_peak": round(cbytes / dn_c_us / 1e3 / peak, 4)}
    del dstate, du, dgc, dks

    # ---- the full decoder-layer stack: 64 layers (48 Gated DeltaNet, 16
    #      attention, each with a SwiGLU MLP of width 17408) at hidden 5120, one
    #      round (verify through the stack, greedy walk, commit of every layer)
    #      from a CUDA graph, 16 and 32 rows, 1k context --------------------------
    if not args.no_stack:
        out["stack"] = stack_bench(dv, synth, dev, peak, flush)

    # ---- StairCut on the measured GB300 prices: the cut of a 31-node lattice
    #      (q = 0.85^depth, scores = q), its host cost through the C ABI ---------
    from speculative_tree_verify_gb300 import prices as pr
    if os.path.exists(pr.GB300_PRICES):
        ptab = pr.table_from_json(pr.GB300_PRICES)
        lat = synth.tree_lattice(32, 15, D.vocab, 77)
        depth = np.zeros(32)
        for i in range(1, 32):
            depth[i] = depth[lat.parent[i]] + 1
        qn = (0.85 ** depth).astype(np.float32)
        cuts = {}
        for cctx in (1024, 32768):
            rc, kept, val = abi.tv_staircut(lat.parent, qn, qn, abi.TV_KIND_TREE, ptab, cctx, 0.0, 0.0)
            dv.check(rc, "tv_staircut")
            cuts[str(cctx)] = {"nodes": len(kept), "tokens_per_ms": round(val, 3)}
        reps = 20000
        t0 = time.perf_counter()
        for _ in range(reps):
            abi.tv_staircut(lat.parent, qn, qn, abi.TV_KIND_TREE, ptab, 1024, 0.0, 0.0)
        out["staircut"] = {"cut_31_node_lattice": cuts,
                           "host_us_per_cut": round((time.perf_counter() - t0) / reps * 1e6, 2),
                           "note": "through the Python binding (argument marshalling included)"}

    # ---- end to end through the C ABI with host buffers --------------------------
    par_h = torch.from_numpy(req.parent.cpu().numpy()).pin_memory()
    tok_h = torch.from_numpy(req.token.cpu().numpy()).pin_memory()
    res_h = torch.empty(rows + 2, dtype=torch.int32).pin_memory()
    steps_e2e = max(50, args.steps // 4)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps_e2e):
        req.parent.copy_(par_h, non_blocking=True)
        req.token.copy_(tok_h, non_blocking=True)
        round_()
        res_h[:rows].copy_(b.out_tokens, non_blocking=True)
        res_h[rows:rows + 1].copy_(b.accept_len, non_blocking=True)
        res_h[rows + 1:].copy_(b.new_ctx, non_blocking=True)
        torch.cuda.current_stream().synchronize()
    e2e_eager_ms = (time.perf_counter() - t0) * 1e3 / steps_e2e

    # the same step captured once in a CUDA graph (the copies from and to the
    # pinned host buffers are nodes of the graph), replayed and synchronised
    # every step
    def e2e_step():
        req.parent.copy_(par_h, non_blocking=True)
        req.token.copy_(tok_h, non_blocking=True)
        round_()
        res_h[:rows].copy_(b.out_tokens, non_blocking=True)
        res_h[rows:rows + 1].copy_(b.accept_len, non_blocking=True)
        res_h[rows + 1:].copy_(b.new_ctx, non_blocking=True)

    ge = _graph(e2e_step)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps_e2e):
        ge.replay()
        torch.cuda.current_stream().synchronize()
    e2e_ms = (time.perf_counter() - t0) * 1e3 / steps_e2e
    dv.check(int(b.status.item()), "e2e round")
    out["e2e"] = {"value": round(e2e_ms, 4), "unit": UNIT, "h2d_bytes_per_step": 2 * rows * 4,
                  "d2h_bytes_per_step": (rows + 2) * 4, "steps": steps_e2e,
                  "eager_value": round(e2e_eager_ms, 4),
                  "note": "host clock per step: host tree -> device, the round, tokens/accept_len/new_ctx -> host, "
                          "stream synchronised; value: the step as one CUDA graph (copies included); eager_value: "
                          "the same calls launched one by one"}

    # ---- the CPU oracle on the host cores ----------------------------------------
    import oracle
    oracle.build()
    model_h = _host_model(dm, synth)
    cache_h = _host_cache(req, synth)     # slots below ctx are never written
    tree_h = synth.Tree(req.parent.cpu().numpy(), req.token.cpu().numpy())
    out["cpu_baseline"] = cpu_baseline(oracle, model_h, cache_h, tree_h, args.cpu_seconds)
    return out


def _reference_inputs(synth, oracle, D):
    """The timed arm's inputs for the oracle: the same weights and cache (the
    same torch draws on the device, seeds 1234 and 99, copied to the host), the
    same lattice tree, its spine planted with the oracle's own greedy tokens
    (the timed arm plants the GPU's, the same tokens except at near ties).
    Nothing of this library runs: torch draws the numbers, the oracle plants."""
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev)
    g.manual_seed(1234)
    H, V = D.hidden, D.vocab

    def w(*shape):
        t = (torch.randn(*shape, generator=g, device=dev, dtype=torch.float32) * 0.02).to(torch.bfloat16)
        return t.view(torch.int16).cpu().numpy().view(np.uint16)

    embed = w(V, H)
    wqkv = w(D.qkv_out, H)
    wo = w(H, D.n_q_heads * D.head_dim)
    lm_head = w(V, H)
    one = synth.f32_to_bf16_bits(np.ones(H, np.float32))
    model = synth.Model(D, embed, one, wqkv, wo, one.copy(), lm_head)
    gc = torch.Generator(device=dev)
    gc.manual_seed(99)
    cap = CTX + 64
    bits = lambda t: t.to(torch.bfloat16).view(torch.int16).cpu().numpy().view(np.uint16)
    k = bits(torch.randn(D.n_kv_heads, cap, D.head_dim, generator=gc, device=dev))
    v = bits(torch.randn(D.n_kv_heads, cap, D.head_dim, generator=gc, device=dev))
    cache = synth.Cache(k, v, CTX, cap)
    tree = synth.tree_lattice(ROWS, SLOTS, D.vocab, 7)
    par, tok = tree.parent, tree.token.copy()
    sp = _spine(par)
    rng = np.random.default_rng(0)
    seq = [int(tok[0])]
    for d in range(1, len(sp)):
        t = int(np.argmax(oracle.decode_sequence(model, cache, seq)["logits"][-1]))
        tok[sp[d]] = t
        for c in range(1, len(par)):
            if c != sp[d] and par[c] == par[sp[d]] and tok[c] == t:
                tok[c] = (t + 1 + int(rng.integers(0, 1000))) % V
        seq.append(t)
    return model, cache, synth.Tree(par.copy(), tok)


def run_reference(args, world, rank, local):
    """The oracle, as it stands, on the host cores: each step a bounded sample
    of the round scaled to ms per full round, on the timed arm's inputs."""
    if rank != 0:
        return None
    import oracle
    from speculative_tree_verify_gb300 import synth

    oracle.build()
    D = synth.FULL
    if torch.cuda.is_available():
        model, cache, tree = _reference_inputs(synth, oracle, D)
        same = True
    else:                                   # no device to draw the timed arm's numbers: numpy draws
        model = synth.gen_model(D, 1234)
        tree = synth.tree_lattice(ROWS, SLOTS, D.vocab, 7)
        cache = synth.gen_cache(D, CTX, CTX + 64, 99)
        same = False
    rng = np.random.default_rng(0)
    # calibrate: all rows, a 4096-entry vocabulary slice
    ids = np.sort(rng.choice(D.vocab, size=4096, replace=False)).astype(np.int32)
    tl, th = oracle_sampled_step(oracle, model, cache, tree, ROWS, ids)
    per_rv = th / (ROWS * len(ids))
    budget = min(2.0, 150.0 / max(1, args.steps + args.warmup))
    r_rows = int(max(1, min(ROWS, ROWS * (budget / 2) / max(tl, 1e-6))))
    s_voc = int(max(256, min(D.vocab, (budget / 2) / max(per_rv * r_rows, 1e-12))))
    vids = np.sort(rng.choice(D.vocab, size=s_voc, replace=False)).astype(np.int32)
    for _ in range(args.warmup):
        oracle_sampled_step(oracle, model, cache, tree, r_rows, vids)
    est = []
    for _ in range(args.steps):
        a, h = oracle_sampled_step(oracle, model, cache, tree, r_rows, vids)
        est.append(1e3 * (a * ROWS / r_rows + h * (ROWS / r_rows) * (D.vocab / s_voc)))
    ms = statistics.median(est)
    sample = (f"per step: the layer over the first {r_rows} of {ROWS} tree rows and the head over {s_voc} of "
              f"{D.vocab} vocabulary rows, scaled to a full round; median of {args.steps} steps")
    return {"metric": METRIC, "value": round(ms, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": WORKLOAD, "hidden": D.hidden, "vocab": D.vocab, "rows": ROWS, "ctx": CTX,
                       "inputs": "the timed arm's weights, cache and tree (spine planted by the oracle)" if same
                       else "numpy draws of the same shapes (no CUDA device for the timed arm's draws)"},
            "same_config": same,
            "cpu_baseline": {"value": round(ms, 3), "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(ms, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = _args()
    world, rank, local = _dist()
    if world > 1 and not torch.distributed.is_initialized():
        backend = "nccl" if args.impl == "ours" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        torch.distributed.init_process_group(backend=backend)
    if args.impl == "reference":
        out = run_reference(args, world, rank, local)
    else:
        out = run_ours(args, world, rank, local)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
