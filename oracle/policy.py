"""CPU oracle of the verify price model and the StairCut cut -- TEST
INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference leg may import this module; the library shares no code with it.

Written from [Drafters and tree verify, §StairCut: the node count, calculated
each round] and [§StairCut on Flash-Next, and the shared price files]:

* ``price`` -- V(rows) from a table of verify prices keyed by context class,
  kind (chain or tree) and measured row count: a class not in the table takes
  the nearest lower one; rows between two measured counts interpolate; rows
  past the last measured count add ``step_ms`` a row, else the slope of the
  last two counts; a price never falls with more rows.
* ``observe`` -- the online update: an observed count moves toward the live
  price by an exponential average of weight 0.1; counts never observed are
  shifted by the learned offset.
* ``staircut`` -- the cut: nodes are admitted in the order of the drafter's
  score, each with the ancestors it needs; the cut ends at 7, 15, 23 or 31
  nodes or at the whole candidate, and the count that maximises
  (1 + min(sum q, n)) / (V(rows) + draft + commit) is kept; a chain pays the
  rollback instead of the commit, weighted by the chance that it is rejected.

Readings where the pages are silent (each listed in the design notes):
rows below the first measured count take the first count's price; a context
below every class takes the lowest class; the learned offset of a (class,
kind) is the exponential average (weight 0.1) of observed minus prior price;
the chance a chain is rejected is 1 - q of its deepest kept node (q is a path
probability); ties between counts keep the smaller count.

Pins: ``tests/test_oracle_policy.py``.
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional, Sequence

EMA = 0.1
CUT_NODES = (7, 15, 23, 31)
MAX_ROWS = 32


class Prices:
    """A price table: {context class: {kind: {rows: ms}}}, step_ms, and the
    online state (live prices of observed counts, the learned offsets)."""

    def __init__(self, table: Dict[int, Dict[str, Dict[int, float]]], step_ms: float = 0.0):
        self.prior = {int(c): {k: {int(r): float(v) for r, v in rows.items()} for k, rows in kinds.items()}
                      for c, kinds in table.items()}
        self.step_ms = float(step_ms)
        self.live: Dict[tuple, float] = {}     # (class, kind, rows) -> ms
        self.offset: Dict[tuple, float] = {}   # (class, kind) -> ms

    def cls(self, context: int) -> int:
        keys = sorted(self.prior)
        lower = [c for c in keys if c <= context]
        return lower[-1] if lower else keys[0]

    def raw(self, c: int, kind: str, rows: int) -> float:
        """The table's price of one count, before the online state and the
        never-falls rule."""
        pts = sorted(self.prior[c].get(kind, {}).items())
        if not pts:
            return 0.0
        xs = [r for r, _ in pts]
        ys = [v for _, v in pts]
        if rows <= xs[0]:
            return ys[0]
        for (x0, y0), (x1, y1) in zip(pts, pts[1:]):
            if x0 <= rows <= x1:
                return y0 + (y1 - y0) * (rows - x0) / (x1 - x0)
        if self.step_ms > 0.0 or len(pts) == 1:
            return ys[-1] + self.step_ms * (rows - xs[-1])
        slope = (ys[-1] - ys[-2]) / (xs[-1] - xs[-2])
        return ys[-1] + slope * (rows - xs[-1])

    def current(self, c: int, kind: str, rows: int) -> float:
        """The price of one count with the online state: its live price if it
        was observed, else the table's plus the learned offset."""
        if (c, kind, rows) in self.live:
            return self.live[(c, kind, rows)]
        return self.raw(c, kind, rows) + self.offset.get((c, kind), 0.0)

    def price(self, context: int, kind: str, rows: int) -> float:
        c = self.cls(context)
        return max(self.current(c, kind, r) for r in range(1, rows + 1))   # never falls with more rows

    def observe(self, context: int, kind: str, rows: int, ms: float) -> None:
        c = self.cls(context)
        prior = self.raw(c, kind, rows)
        old = self.current(c, kind, rows)
        self.live[(c, kind, rows)] = old + EMA * (ms - old)
        off = self.offset.get((c, kind), 0.0)
        self.offset[(c, kind)] = off + EMA * ((ms - prior) - off)


def admission_order(parent: Sequence[int], score: Sequence[float]) -> List[int]:
    """Non-root nodes in the order of the drafter's score (highest first, lower
    index on ties), each preceded by its ancestors not yet admitted."""
    n = len(parent)
    order, seen = [], {0}
    for t in sorted(range(1, n), key=lambda i: (-float(score[i]), i)):
        chain = []
        a = t
        while a not in seen:
            chain.append(a)
            a = parent[a]
        for a in reversed(chain):
            seen.add(a)
            order.append(a)
    return order


def staircut(parent: Sequence[int], q: Sequence[float], score: Sequence[float], kind: str, prices: Prices,
             context: int, draft_ms: float, commit_ms: float, rollback_ms: float = 0.0):
    """Returns (kept nodes in admission order, value) for the best cut; the
    root is always kept (the cut counts nodes past the root: rows = nodes + 1)."""
    order = admission_order(parent, score)
    total = len(order)
    counts = sorted({c for c in CUT_NODES if c <= total} | {min(total, CUT_NODES[-1])})
    best, best_val = None, -math.inf
    for cnt in counts:
        kept = order[:cnt]
        gain = 1.0 + min(sum(min(1.0, float(q[i])) for i in kept), cnt)
        cost = prices.price(context, kind, cnt + 1) + draft_ms
        if kind == "chain":
            q_last = min(1.0, float(q[kept[-1]])) if kept else 1.0
            cost += (1.0 - q_last) * rollback_ms
        else:
            cost += commit_ms
        val = gain / cost
        if val > best_val:
            best, best_val = kept, val
    return best, best_val
