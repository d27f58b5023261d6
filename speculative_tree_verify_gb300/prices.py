"""Verify price files: the JSON format of the stair tables <-> tv_price_table,
and the measurement of this library's verify round on the GPU at hand.

Format [Drafters and tree verify, §StairCut on Flash-Next, and the shared
price files]:

    {"<context class>": {"<kind>": {"<rows>": ms, ...}, ...}, ...,
     "step_ms": 3.7, "measured": "how and when"}

kind is "chain" or "tree"; the context class is a context length.  Lookup,
interpolation, the online update and the cut run in the library
(tv_price_lookup, tv_price_observe, tv_staircut); this module only moves
numbers between the file and the table.

    python -m speculative_tree_verify_gb300.prices --measure --out prices.json
    python -m speculative_tree_verify_gb300.prices --measure --stack --out stack.json
"""
from __future__ import annotations

import argparse
import json
import math
import os
import time
from typing import Dict, Sequence

from . import abi

KINDS = {"chain": abi.TV_KIND_CHAIN, "tree": abi.TV_KIND_TREE}
HERE = os.path.dirname(os.path.abspath(__file__))
GB300_PRICES = os.path.join(HERE, "prices", "gb300.json")
GB300_STACK_PRICES = os.path.join(HERE, "prices", "gb300_stack.json")


def table_from_json(obj) -> abi.TvPriceTable:
    """A tv_price_table from a parsed price file (or its path)."""
    if isinstance(obj, str):
        with open(obj) as f:
            obj = json.load(f)
    t = abi.TvPriceTable()
    rc = abi.tv_price_init(t)
    if rc != abi.TV_OK:
        raise RuntimeError(abi.STATUS.get(rc, rc))
    classes = sorted(int(k) for k in obj if k.lstrip("-").isdigit())
    if not 1 <= len(classes) <= abi.PRICE_MAX_CLASSES:
        raise ValueError(f"{len(classes)} context classes (1..{abi.PRICE_MAX_CLASSES})")
    t.n_classes = len(classes)
    for i, c in enumerate(classes):
        t.class_ctx[i] = c
        for kind, rows in obj[str(c)].items():
            if kind not in KINDS:
                continue
            for r, ms in rows.items():
                r = int(r)
                if not 1 <= r <= abi.PRICE_MAX_ROWS:
                    raise ValueError(f"rows {r} outside 1..{abi.PRICE_MAX_ROWS}")
                t.prior[i][KINDS[kind]][r] = float(ms)
    t.step_ms = float(obj.get("step_ms", 0.0))
    return t


def table_to_json(t: abi.TvPriceTable, measured: str = "") -> dict:
    """The table's measured prices as a price file (the online state is not part of it)."""
    out: Dict[str, object] = {}
    for i in range(t.n_classes):
        kinds = {}
        for kind, k in KINDS.items():
            rows = {str(r): round(t.prior[i][k][r], 4) for r in range(1, abi.PRICE_MAX_ROWS + 1)
                    if not math.isnan(t.prior[i][k][r])}
            if rows:
                kinds[kind] = rows
        out[str(t.class_ctx[i])] = kinds
    out["step_ms"] = t.step_ms
    if measured:
        out["measured"] = measured
    return out


def measure(contexts: Sequence[int] = (1024, 4096, 8192, 16384, 32768),
            rows: Sequence[int] = (1, 2, 4, 8, 12, 16, 20, 24, 28, 32), reps: int = 100) -> dict:
    """Times one round (verify, greedy walk, commit) from a CUDA graph for a
    chain and a lattice tree of each row count at each context, on the hidden
    5120 / 151936-vocabulary shapes with random weights; returns a price file."""
    import torch

    from . import device as dv
    from . import synth

    D = synth.FULL
    dm = dv.DeviceModel.random(D, 1234)
    table: Dict[str, object] = {}
    for ctx in contexts:
        kinds: Dict[str, Dict[str, float]] = {"chain": {}, "tree": {}}
        for n in rows:
            for kind in ("chain", "tree"):
                tree = synth.tree_chain(n, D.vocab, 5 + n) if kind == "chain" else \
                    synth.tree_lattice(n, 15 if n > 16 else 7, D.vocab, 5 + n)
                g = torch.Generator(device="cuda")
                g.manual_seed(ctx + n)
                cap = ctx + 32
                k = (torch.randn(D.n_kv_heads, cap, D.head_dim, device="cuda", generator=g)).to(torch.bfloat16)
                v = (torch.randn(D.n_kv_heads, cap, D.head_dim, device="cuda", generator=g)).to(torch.bfloat16)
                req = dv.DeviceRequest(k, v, ctx, torch.from_numpy(tree.parent.copy()).cuda(),
                                       torch.from_numpy(tree.token.copy()).cuda())
                b = dv.RoundBuffers.alloc(D, n, 1, ctx)

                def round_():
                    dv.check(dv.verify(dm, [req], b, stream=torch.cuda.current_stream()), "verify")
                    dv.check(dv.accept_greedy_commit([req], b, stream=torch.cuda.current_stream()), "accept+commit")

                s = torch.cuda.Stream()
                s.wait_stream(torch.cuda.current_stream())
                with torch.cuda.stream(s):
                    for _ in range(3):
                        round_()
                torch.cuda.current_stream().wait_stream(s)
                gr = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gr):
                    round_()
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                for _ in range(reps):
                    gr.replay()
                e1.record()
                torch.cuda.synchronize()
                if int(b.status.item()) != 0:
                    raise RuntimeError(abi.STATUS.get(int(b.status.item())))
                kinds[kind][str(n)] = round(e0.elapsed_time(e1) / reps, 4)
                del gr, req, b, k, v
        table[str(ctx)] = kinds
    table["step_ms"] = 0.0
    table["measured"] = (f"{torch.cuda.get_device_name()}, {time.strftime('%Y-%m-%d')}: one round (verify + greedy "
                         f"walk + commit) from a CUDA graph, mean of {reps} replays, hidden 5120 layer + 151936 head, "
                         f"random weights; chain and lattice trees")
    return table


def measure_stack(contexts: Sequence[int] = (1024, 8192, 32768),
                  rows: Sequence[int] = (1, 2, 4, 8, 12, 16, 20, 24, 28, 32), reps: int = 10) -> dict:
    """Times one round of the whole decoder-layer stack (verify through every
    layer, greedy walk, commit of every layer) from a CUDA graph for a chain
    and a lattice tree of each row count at each context: the 64-layer stack at
    hidden 5120 (48 Gated DeltaNet and 16 attention layers, MLP width 17408,
    151936-vocabulary head), random weights; returns a price file."""
    import torch

    from . import device as dv
    from . import synth

    sd = synth.STACK_FULL
    model = dv.DeviceStack.random(sd, 1234)
    n_dn = len(sd.dn_layers)
    table: Dict[str, object] = {}
    for ctx in contexts:
        kinds: Dict[str, Dict[str, float]] = {"chain": {}, "tree": {}}
        g = torch.Generator(device="cuda")
        g.manual_seed(ctx)
        cap = ctx + 32
        ks = [torch.randn(sd.base.n_kv_heads, cap, sd.base.head_dim, device="cuda", generator=g).to(torch.bfloat16)
              for _ in sd.attn_layers]
        vs = [torch.randn_like(k) for k in ks]
        for n in rows:
            for kind in ("chain", "tree"):
                tree = synth.tree_chain(n, sd.base.vocab, 5 + n) if kind == "chain" else \
                    synth.tree_lattice(n, 15 if n > 16 else 7, sd.base.vocab, 5 + n)
                st = torch.randn(n_dn, sd.n_v_heads, sd.d_k, sd.d_v, device="cuda", generator=g) * 0.3
                req = dv.StackRequest(ks, vs, ctx, st, torch.from_numpy(tree.parent.copy()).cuda(),
                                      torch.from_numpy(tree.token.copy()).cuda())
                b = dv.StackBuffers.alloc(model, n, 1)

                def round_():
                    dv.run_stack_round(model, [req], b, stream=torch.cuda.current_stream())

                s = torch.cuda.Stream()
                s.wait_stream(torch.cuda.current_stream())
                with torch.cuda.stream(s):
                    for _ in range(2):
                        round_()
                torch.cuda.current_stream().wait_stream(s)
                gr = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gr):
                    round_()
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                for _ in range(reps):
                    gr.replay()
                e1.record()
                torch.cuda.synchronize()
                if int(b.status.item()) != 0:
                    raise RuntimeError(abi.STATUS.get(int(b.status.item())))
                kinds[kind][str(n)] = round(e0.elapsed_time(e1) / reps, 4)
                del gr, req, b, st
        table[str(ctx)] = kinds
        del ks, vs
    table["step_ms"] = 0.0
    table["measured"] = (f"{torch.cuda.get_device_name()}, {time.strftime('%Y-%m-%d')}: one round of the 64-layer "
                         f"stack (48 Gated DeltaNet + 16 attention layers, SwiGLU MLP 17408, hidden 5120, 151936 "
                         f"head; verify + greedy walk + commit of every layer) from a CUDA graph, mean of {reps} "
                         f"replays, random weights; chain and lattice trees")
    return table


def _main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--measure", action="store_true")
    ap.add_argument("--out", default=None)
    ap.add_argument("--reps", type=int, default=100)
    ap.add_argument("--stack", action="store_true", help="measure the 64-layer stack instead of one layer + head")
    a = ap.parse_args()
    if a.measure:
        tab = measure_stack(reps=min(a.reps, 10)) if a.stack else measure(reps=a.reps)
        text = json.dumps(tab, indent=1)
        if a.out:
            with open(a.out, "w") as f:
                f.write(text + "\n")
        print(text)


if __name__ == "__main__":
    _main()
