"""The forward pins catch plausible mistakes in the C oracle.

Each case plants one mistake in a copy of ``oracle/tv_oracle.c`` (a textual
edit that must match exactly once), builds the copy, points the oracle module
at it and runs two pins on a small layer with random norm gains:

* chain pin -- a chain's rows equal an independent torch-fp64 layer
  (rms_norm, linear, complex-exponential RoPE, scaled_dot_product_attention)
  bit for bit in every bf16 store;
* tree pin -- every row of a branched tree equals plain sequential decoding of
  the row's own root path, bit for bit.

The unedited copy passes both; every edited copy must fail at least one.  All
of it runs on the CPU.
"""
import os
import subprocess

import numpy as np
import pytest

import oracle
from speculative_tree_verify_gb300 import synth
from test_oracle_forward import _check_tree_against_decode, torch_layer_over_sequence

SRC = os.path.join(os.path.dirname(oracle.__file__), "tv_oracle.c")

# (name, exact text in the oracle, the planted mistake)
MUTATIONS = [
    ("rope_sign", "x[d] = x1 * c - x2 * s;", "x[d] = x1 * c + x2 * s;"),
    ("position_is_index", "(long)ctx + depth[i],", "(long)ctx + i,"),
    ("depth_from_previous_row", "depth[parent[i]] + 1", "depth[i - 1] + 1"),
    ("no_attention_scale", "s[j] = dot * scale;", "s[j] = dot;"),
    ("no_residual", "rb(x[c] + dot_w(m->wo", "rb(dot_w(m->wo"),
    ("dropped_norm_gain", "y[k] = rb(x[k] * inv * bf(g[k]));", "y[k] = rb(x[k] * inv);"),
    ("no_self_key", "for (int a = i; a >= 0; a = parent[a]) path[len++] = a;",
     "for (int a = parent[i]; a >= 0; a = parent[a]) path[len++] = a;"),
    ("gqa_head_map", "const int g = hq / group;", "const int g = hq % Hkv;"),
    ("no_norm_eps", "sqrt(ss / (double)H + eps)", "sqrt(ss / (double)H)"),
    ("qkv_store_scaled", "for (int d = 0; d < D; ++d) dst[d] = orc_round_bf16(t[d]);",
     "for (int d = 0; d < D; ++d) dst[d] = orc_round_bf16((float)t[d] * 1.0009765625f);"),
]


def _build_copy(tmp_path, name, old=None, new=None):
    text = open(SRC).read()
    if old is not None:
        assert text.count(old) == 1, f"{name}: the text to edit must occur exactly once"
        text = text.replace(old, new)
    src = tmp_path / f"{name}.c"
    lib = tmp_path / f"lib{name}.so"
    src.write_text(text)
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]
    try:
        subprocess.run(base + ["-fopenmp", str(src), "-o", str(lib), "-lm"], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + [str(src), "-o", str(lib), "-lm"], check=True)
    return str(lib)


def _use(monkeypatch, lib_path):
    monkeypatch.setattr(oracle, "build", lambda force=False: lib_path)
    monkeypatch.setattr(oracle, "_LIB_PATH", lib_path)
    monkeypatch.setattr(oracle, "_lib", None)


def _chain_pin():
    d = synth.TINY
    model = synth.gen_model(d, 0, random_gains=True)
    cache = synth.gen_cache(d, 64, 75, 50)
    tree = synth.tree_chain(8, d.vocab, 60)
    got = oracle.verify_tree(model, cache, tree)
    ref = torch_layer_over_sequence(model, cache, [int(t) for t in tree.token])
    for key in ("k", "v", "attn", "hf"):
        assert np.count_nonzero(got[key] != ref[key]) == 0, key
    np.testing.assert_allclose(got["logits"], ref["logits"], rtol=3e-7, atol=1e-8)


def _tree_pin():
    d = synth.TINY
    model = synth.gen_model(d, 101, random_gains=True)
    cache = synth.gen_cache(d, 64, 128, 201)
    tree = synth.tree_spine_random(12, 4, d.vocab, 301)
    assert any(int(tree.parent[i]) != i - 1 for i in range(1, tree.n))   # branched
    _check_tree_against_decode(model, cache, tree)


def _failed_pins():
    failed = []
    for name, pin in (("chain", _chain_pin), ("tree", _tree_pin)):
        try:
            with np.errstate(all="ignore"):
                pin()
        except AssertionError:
            failed.append(name)
    return failed


def test_unedited_copy_passes_the_pins(tmp_path, monkeypatch):
    _use(monkeypatch, _build_copy(tmp_path, "unedited"))
    assert _failed_pins() == []


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_fails_a_pin(tmp_path, monkeypatch, name, old, new):
    _use(monkeypatch, _build_copy(tmp_path, name, old, new))
    assert _failed_pins(), f"planted mistake {name} passed every forward pin"


# --------------------------------------------------------------------------
# the Gated DeltaNet oracle (oracle/deltanet.py) against its pins
# --------------------------------------------------------------------------
import inspect  # noqa: E402
import types  # noqa: E402

import test_oracle_deltanet as DNT  # noqa: E402
from oracle import deltanet as DN_REAL  # noqa: E402

DN_MUTATIONS = [
    ("dropped_decay", "S_new = np.exp(g) * (S - beta * np.outer(k, k @ S))", "S_new = (S - beta * np.outer(k, k @ S))"),
    ("flipped_erase_sign", "(S - beta * np.outer(k, k @ S))", "(S + beta * np.outer(k, k @ S))"),
    ("unscaled_write", "+ beta * np.outer(k, v)", "+ np.outer(k, v)"),
    ("previous_row_not_parent", "else states[parent[t]]", "else states[t - 1]"),
    ("wrong_head_map", "return h // (n_v_heads // n_k_heads)", "return h % n_k_heads"),
    ("output_before_update", "return S_new, S_new.T @ q", "return S_new, S.T @ q"),
    ("commit_keeps_the_root", "states[path[-1]]", "states[path[0]]"),
]


def _module_copy(real, old=None, new=None):
    """A fresh module built from ``real``'s source with one textual edit."""
    text = inspect.getsource(real)
    if old is not None:
        assert text.count(old) == 1, f"the text to edit must occur exactly once: {old!r}"
        text = text.replace(old, new)
    mod = types.ModuleType(real.__name__ + "_copy")
    mod.__file__ = real.__file__          # the copy finds the same C sources and library
    mod.__package__ = real.__package__    # and resolves relative imports in the same package
    exec(compile(text, mod.__name__, "exec"), mod.__dict__)
    return mod


def _deltanet_copy(old=None, new=None):
    return _module_copy(DN_REAL, old, new)


def _pins_failed(test_module, skip_slow=False, first_only=False, last=()):
    """Runs every test function of ``test_module`` (each parametrisation) and
    returns the names of those that fail.  ``last`` names pins to run after
    the others; ``first_only`` stops at the first failure."""
    failed = []
    fns = [(n, f) for n, f in inspect.getmembers(test_module, inspect.isfunction) if n.startswith("test_")]
    fns.sort(key=lambda nf: nf[0] in last)
    for name, fn in fns:
        if first_only and failed:
            break
        marks = getattr(fn, "pytestmark", [])
        if skip_slow and any(m.name == "slow" for m in marks):
            continue
        cases = [dict(zip([a.strip() for a in m.args[0].split(",")], vals if isinstance(vals, tuple) else (vals,)))
                 for m in marks if m.name == "parametrize" for vals in m.args[1]] or [{}]
        for kw in cases:
            try:
                with np.errstate(all="ignore"):
                    fn(**kw)
            except Exception:             # a failed assertion, or a pin that cannot run
                failed.append(name)
                break
    return failed


def _deltanet_pins_failed():
    return _pins_failed(DNT)


def test_unedited_deltanet_copy_passes_the_pins(monkeypatch):
    monkeypatch.setattr(DNT, "DN", _deltanet_copy())
    assert _deltanet_pins_failed() == []


@pytest.mark.parametrize("name,old,new", DN_MUTATIONS, ids=[m[0] for m in DN_MUTATIONS])
def test_planted_deltanet_mistake_fails_a_pin(monkeypatch, name, old, new):
    monkeypatch.setattr(DNT, "DN", _deltanet_copy(old, new))
    assert _deltanet_pins_failed(), f"planted mistake {name} passed every DeltaNet pin"


# --------------------------------------------------------------------------
# the walk and commit oracles (oracle/__init__.py) against their pins
# --------------------------------------------------------------------------
import test_oracle_walks as WT  # noqa: E402

# mistakes that would loop forever (a walk that never leaves the root's
# children) are left out: the harness runs pins, not a watchdog
WALK_MUTATIONS = [
    ("greedy_no_bonus", "out = [int(token[c]) for c in path[1:]] + [t]", "out = [int(token[c]) for c in path[1:]]"),
    ("greedy_first_child", "nxt = next((c for c in kids[cur] if int(token[c]) == t), None)",
     "nxt = next((c for c in kids[cur]), None)"),
    ("residual_no_renormalise", "r = r / r.sum()", "r = r"),
    ("residual_no_removal", "r[x] = 0.0                      # remove x and renormalise", "r[x] = r[x]"),
    ("residual_tests_against_p", "ok = u < r[x]", "ok = u < p[x]"),
    ("residual_draw_from_p", "y = inverse_cdf(r, u)", "y = inverse_cdf(p, u)"),
    ("inverse_cdf_off_by_one", 'y = int(np.searchsorted(c, float(u) * c[-1], side="right"))',
     'y = int(np.searchsorted(c, float(u) * c[-1], side="right")) - 1'),
    ("softmax_ignores_temperature", "z = np.asarray(logits_row, np.float64) / float(temperature)",
     "z = np.asarray(logits_row, np.float64)"),
    ("leaf_bonus_ignored", "if kids[cur] or bonus_at_leaf:", "if kids[cur]:"),
    ("commit_ignores_path", "src = [ctx + int(p) for p in path]", "src = [ctx + d for d in range(len(path))]"),
]


def test_unedited_walk_copy_passes_the_pins(monkeypatch):
    monkeypatch.setattr(WT, "oracle", _module_copy(oracle))
    assert _pins_failed(WT, skip_slow=True) == []


@pytest.mark.parametrize("name,old,new", WALK_MUTATIONS, ids=[m[0] for m in WALK_MUTATIONS])
def test_planted_walk_mistake_fails_a_pin(monkeypatch, name, old, new):
    monkeypatch.setattr(WT, "oracle", _module_copy(oracle, old, new))
    assert _pins_failed(WT, skip_slow=True), f"planted mistake {name} passed every walk pin"


# --------------------------------------------------------------------------
# the sampled-variant oracles (oracle/sampling.py) against their pins
# --------------------------------------------------------------------------
import test_oracle_sampling as ST  # noqa: E402
from oracle import sampling as SAMPLING_REAL  # noqa: E402

SAMPLING_SLOW = ("test_single_draw_exact_grid_law", "test_rejection_chain_output_follows_the_target",
                 "test_single_draw_and_residual_walk_share_one_law")
SAMPLING_MUTATIONS = [
    ("filter_ignores_temperature", "x = np.asarray(logits_row, np.float64) / float(temperature)",
     "x = np.asarray(logits_row, np.float64)"),
    ("top_k_off_by_one", "[::-1][top_k - 1]", "[::-1][top_k]"),
    ("top_p_drops_the_cut_token", "keep &= p >= p[order[cut]]", "keep &= p > p[order[cut]]"),
    ("min_p_not_relative_to_max", "keep &= x >= xm + np.log(min_p)", "keep &= x >= np.log(min_p)"),
    ("philox_wrong_key_bump", "k0 = (k0 + np.uint64(_W0)) & mask", "k0 = (k0 + np.uint64(_W1)) & mask"),
    ("philox_swapped_products", "c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0",
     "c0, c1, c2, c3 = hi0 ^ c1 ^ k0, lo0, hi1 ^ c3 ^ k1, lo1"),
    ("gumbel_noise_sign", "return x - np.log(-np.log(u))", "return x + np.log(-np.log(u))"),
    ("gumbel_position_off_by_one", "gumbel_draw(rows_x[cur], seed, ctx + depth[cur] + 1)",
     "gumbel_draw(rows_x[cur], seed, ctx + depth[cur])"),
    ("gumbel_uniform_not_centred", "return (w.astype(np.float64) + 0.5) / 4294967296.0",
     "return (w.astype(np.float64) + 1.0) / 4294967296.0"),
    ("rejection_ratio_inverted", "ratio = p[x] / q[x]", "ratio = q[x] / p[x]"),
    ("rejection_draws_from_p", "r = np.maximum(p - q, 0.0)", "r = p"),
]
# Which uniform a row consumes is a convention the laws cannot see (any
# independent uniform gives the same law): the GPU parity tests pin it.


def test_unedited_sampling_copy_passes_the_pins(monkeypatch):
    monkeypatch.setattr(ST, "S", _module_copy(SAMPLING_REAL))
    assert _pins_failed(ST) == []


@pytest.mark.parametrize("name,old,new", SAMPLING_MUTATIONS, ids=[m[0] for m in SAMPLING_MUTATIONS])
def test_planted_sampling_mistake_fails_a_pin(monkeypatch, name, old, new):
    monkeypatch.setattr(ST, "S", _module_copy(SAMPLING_REAL, old, new))
    assert _pins_failed(ST, first_only=True, last=SAMPLING_SLOW), f"planted mistake {name} passed every pin"


# --------------------------------------------------------------------------
# the price and StairCut oracles (oracle/policy.py) against their pins
# --------------------------------------------------------------------------
import test_oracle_policy as PT  # noqa: E402
from oracle import policy as POLICY_REAL  # noqa: E402

POLICY_MUTATIONS = [
    ("ema_weight", "EMA = 0.1", "EMA = 0.2"),
    ("cut_counts_taken_as_rows", "CUT_NODES = (7, 15, 23, 31)", "CUT_NODES = (8, 16, 24, 32)"),
    ("price_may_fall", "return max(self.current(c, kind, r) for r in range(1, rows + 1))",
     "return self.current(c, kind, rows)"),
    ("nearest_upper_class", "lower = [c for c in keys if c <= context]", "lower = [c for c in keys if c >= context][:1]"),
    ("rows_without_the_root", "cost = prices.price(context, kind, cnt + 1) + draft_ms",
     "cost = prices.price(context, kind, cnt) + draft_ms"),
    ("children_before_ancestors", "for a in reversed(chain):", "for a in chain:"),
    ("rollback_not_weighted", "cost += (1.0 - q_last) * rollback_ms", "cost += rollback_ms"),
    ("offset_never_learned", "self.offset[(c, kind)] = off + EMA * ((ms - prior) - off)", "self.offset[(c, kind)] = off"),
]


def test_unedited_policy_copy_passes_the_pins(monkeypatch):
    monkeypatch.setattr(PT, "P", _module_copy(POLICY_REAL))
    assert _pins_failed(PT) == []


@pytest.mark.parametrize("name,old,new", POLICY_MUTATIONS, ids=[m[0] for m in POLICY_MUTATIONS])
def test_planted_policy_mistake_fails_a_pin(monkeypatch, name, old, new):
    monkeypatch.setattr(PT, "P", _module_copy(POLICY_REAL, old, new))
    assert _pins_failed(PT), f"planted mistake {name} passed every price/StairCut pin"


# --------------------------------------------------------------------------
# the layer-stack oracle (oracle/stack.py) against its pins
# --------------------------------------------------------------------------
import test_oracle_stack as SKT  # noqa: E402
from oracle import stack as STACK_REAL  # noqa: E402

STACK_MUTATIONS = [
    ("mlp_no_residual", "return rb(x + matvec_rows(lay.w_down, a[None])[0])",
     "return rb(matvec_rows(lay.w_down, a[None])[0])"),
    ("swiglu_gate_on_up", "a = rb(_silu(gu[:I]) * gu[I:])", "a = rb(gu[:I] * _silu(gu[I:]))"),
    ("dn_state_of_previous_row", "S0 if parent[i] < 0 else Sn[parent[i]]", "S0 if parent[i] < 0 else Sn[i - 1]"),
    ("dn_q_not_scaled", "q = q / np.sqrt(np.sum(q * q, axis=1, keepdims=True) + 1e-6) / np.sqrt(dk)",
     "q = q / np.sqrt(np.sum(q * q, axis=1, keepdims=True) + 1e-6)"),
    ("dn_key_head_map", "kh = h // G", "kh = h % sd.n_k_heads"),
    ("dn_write_strength_not_sigmoid", "beta = 1.0 / (1.0 + np.exp(-b))", "beta = 1.0 / (1.0 + np.exp(b))"),
    ("dn_decay_sign", "g = -np.logaddexp(0.0, a)", "g = np.logaddexp(0.0, a) - 2.0 * np.logaddexp(0.0, a) + 0.01"),
    ("dn_output_gate_dropped", "* bf16_to_f64(lay.dn_norm)[None, :] * _silu(z))",
     "* bf16_to_f64(lay.dn_norm)[None, :])"),
    ("attn_position_is_index", "fr = [attn_front(lay, d, h[i], ctx + int(depth[i])) for i in range(n)]",
     "fr = [attn_front(lay, d, h[i], ctx + i) for i in range(n)]"),
    ("attn_key_of_wrong_node", "K = np.concatenate([Kc, np.stack([fr[a][1] for a in p])])",
     "K = np.concatenate([Kc, np.stack([fr[max(a - 1, 0)][1] for a in p])])"),
    ("commit_keeps_the_root_state", "states = [st[path[-1]].copy() for st in res[\"states\"]]",
     "states = [st[path[0]].copy() for st in res[\"states\"]]"),
    ("mlp_norm_gain_of_the_mixer", "h2 = _rms_bf16(x, lay.ln_mlp, sd.base.rms_eps)",
     "h2 = _rms_bf16(x, lay.ln_mix, sd.base.rms_eps)"),
]


def test_unedited_stack_copy_passes_the_pins(monkeypatch):
    monkeypatch.setattr(SKT, "ST", _module_copy(STACK_REAL))
    assert _pins_failed(SKT) == []


@pytest.mark.parametrize("name,old,new", STACK_MUTATIONS, ids=[m[0] for m in STACK_MUTATIONS])
def test_planted_stack_mistake_fails_a_pin(monkeypatch, name, old, new):
    monkeypatch.setattr(SKT, "ST", _module_copy(STACK_REAL, old, new))
    assert _pins_failed(SKT, first_only=True), f"planted mistake {name} passed every stack pin"
