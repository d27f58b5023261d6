"""The C-ABI library on a machine without a GPU: it builds, loads, exports
exactly the entry points include/tv.h declares, and its host-side argument
checks return the documented codes before anything is launched."""
import ctypes
import os
import re
import subprocess

import pytest

from speculative_tree_verify_gb300 import abi, build
from speculative_tree_verify_gb300.device import tv_dims
from speculative_tree_verify_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tv.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return abi.load()


def _declared():
    text = open(HEADER).read()
    return sorted(re.findall(r"TV_API\s+[\w\s\*]*?\b(tv_\w+)\s*\(", text))


def test_header_declares_the_four_round_calls():
    names = _declared()
    for n in ("tv_verify_tree", "tv_accept_greedy", "tv_accept_residual", "tv_commit_kv"):
        assert n in names
    assert sorted(abi.SYMBOLS) == names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", abi.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = sorted(l.split()[-1] for l in out.splitlines() if " T " in l)
    assert exported == _declared()
    for name in _declared():
        assert getattr(lib, name) is not None


def test_status_codes_match_header():
    defs = dict((name, int(val)) for name, val in re.findall(r"#define\s+(TV_OK|TV_E_\w+)\s+(-?\d+)", open(HEADER).read()))
    assert {v: k for k, v in defs.items()} == abi.STATUS
    for code, name in abi.STATUS.items():
        assert abi.tv_status_string(code) not in ("", "unknown status")


def test_workspace_size_host_only(lib):
    ws = abi.tv_workspace_size(tv_dims(synth.FULL), 32, 32768)
    assert ws > 0 and ws % 256 == 0
    small = abi.tv_workspace_size(tv_dims(synth.TINY), 8, 64)
    assert 0 < small < ws
    bad = tv_dims(synth.Dims(hidden=100, n_q_heads=4, n_kv_heads=2, head_dim=64, vocab=1024))
    with pytest.raises(ValueError, match="UNSUPPORTED"):
        abi.tv_workspace_size(bad, 8, 64)
    with pytest.raises(ValueError, match="ROWS"):
        abi.tv_workspace_size(tv_dims(synth.TINY), 33, 64)


FAKE = 0x10000   # a 16-byte aligned non-null address; never dereferenced on these paths


def _model(d=synth.TINY):
    return abi.TvModel(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, tv_dims(d))


def _kv(ctx, cap):
    return abi.TvKv(FAKE, FAKE, ctx, cap)


def _tree(n):
    return abi.TvTree(FAKE, FAKE, n)


def test_verify_host_checks(lib):
    d = synth.TINY
    ws = abi.tv_workspace_size(tv_dims(d), 32, 64)
    args = dict(logits=FAKE, argmax=FAKE, top2_gap=FAKE, attn_out=None, workspace=FAKE, workspace_bytes=ws,
                dev_status=FAKE)

    def call(model=None, kvs=None, trees=None, **over):
        a = dict(args)
        a.update(over)
        return abi.tv_verify_tree(model or _model(), kvs if kvs is not None else [_kv(64, 96)],
                                  trees if trees is not None else [_tree(8)], **a)

    assert call(logits=None) == abi.CODES["TV_E_ARG"]
    assert call(trees=[_tree(0)]) == abi.CODES["TV_E_ROWS"]
    assert call(trees=[_tree(33)], kvs=[_kv(0, 100)]) == abi.CODES["TV_E_ROWS"]
    assert call(trees=[_tree(20), _tree(13)], kvs=[_kv(0, 64), _kv(0, 64)]) == abi.CODES["TV_E_ROWS"]
    assert call(kvs=[_kv(90, 96)]) == abi.CODES["TV_E_CAPACITY"]
    assert call(workspace_bytes=ws - 1) == abi.CODES["TV_E_WORKSPACE"]
    assert call(workspace=None) == abi.CODES["TV_E_WORKSPACE"]
    assert call(kvs=[abi.TvKv(FAKE + 2, FAKE, 64, 96)]) == abi.CODES["TV_E_ARG"]   # misaligned cache
    bad = synth.Dims(hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=96, vocab=1024)
    assert call(model=_model(bad)) == abi.CODES["TV_E_UNSUPPORTED"]
    packed2 = _model()
    packed2.packed = 2
    assert call(model=packed2) == abi.CODES["TV_E_ARG"]                            # packed is 0 or 1
    wide = synth.Dims(hidden=512, n_q_heads=16, n_kv_heads=2, head_dim=64, vocab=1024)   # 8 heads per group
    assert call(model=_model(wide), trees=[_tree(21)], kvs=[_kv(0, 64)],
                workspace_bytes=abi.tv_workspace_size(tv_dims(wide), 32, 64)) == abi.CODES["TV_E_UNSUPPORTED"]


def test_packed_weight_host_checks(lib):
    # rows padded to a multiple of 128, bf16
    assert abi.tv_packed_weight_bytes(1, 64) == 128 * 64 * 2
    assert abi.tv_packed_weight_bytes(300, 192) == 384 * 192 * 2
    assert abi.tv_packed_weight_bytes(151936, 5120) == 151936 * 5120 * 2
    for rows, cols in ((0, 64), (128, 0), (128, 96), (128, 32)):
        with pytest.raises(ValueError, match="ARG"):
            abi.tv_packed_weight_bytes(rows, cols)
    assert abi.tv_pack_weight(None, 128, 64, FAKE) == abi.CODES["TV_E_ARG"]
    assert abi.tv_pack_weight(FAKE, 128, 64, None) == abi.CODES["TV_E_ARG"]
    assert abi.tv_pack_weight(FAKE + 2, 128, 64, FAKE) == abi.CODES["TV_E_ARG"]   # misaligned
    assert abi.tv_pack_weight(FAKE, 128, 96, FAKE) == abi.CODES["TV_E_ARG"]


def test_walk_and_commit_host_checks(lib):
    ws = abi.tv_workspace_size(tv_dims(synth.TINY), 32, 64)
    trees = [_tree(8)]
    assert abi.tv_accept_greedy(trees, None, FAKE, FAKE, FAKE, FAKE) == abi.CODES["TV_E_ARG"]
    assert abi.tv_accept_greedy([_tree(40)], FAKE, FAKE, FAKE, FAKE, FAKE) == abi.CODES["TV_E_ROWS"]
    for t in (0.0, -1.0, float("nan"), float("inf")):
        assert abi.tv_accept_residual(trees, FAKE, 1024, t, FAKE, True, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                      ws) == abi.CODES["TV_E_TEMP"]
    assert abi.tv_accept_residual(trees, FAKE, 1024, 1.0, FAKE, True, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                  16) == abi.CODES["TV_E_WORKSPACE"]
    dims = tv_dims(synth.TINY)
    assert abi.tv_commit_kv([_kv(64, 96)], dims, trees, None, FAKE, FAKE, FAKE, FAKE) == abi.CODES["TV_E_ARG"]
    assert abi.tv_commit_kv([_kv(64, 96)], dims, [_tree(33)], FAKE, FAKE, FAKE, FAKE, FAKE) == abi.CODES["TV_E_ROWS"]
    assert abi.tv_accept_greedy_commit([_kv(64, 96)], dims, trees, None, FAKE, FAKE, FAKE, FAKE, FAKE,
                                       FAKE) == abi.CODES["TV_E_ARG"]
    assert abi.tv_accept_greedy_commit([_kv(64, 96)], dims, [_tree(33)], FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                       FAKE) == abi.CODES["TV_E_ROWS"]
    assert abi.tv_accept_greedy_commit([_kv(90, 96)], dims, trees, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                       FAKE) == abi.CODES["TV_E_CAPACITY"]


def test_sampled_host_checks(lib):
    rc, wsb = abi.tv_sample_workspace_size(151936, 32)
    assert rc == abi.TV_OK and wsb > 0 and wsb % 256 == 0
    assert abi.tv_sample_workspace_size(151936, 33)[0] == abi.CODES["TV_E_ROWS"]
    assert abi.tv_sample_workspace_size(1, 8)[0] == abi.CODES["TV_E_ARG"]
    # filters: temperature, then the filter parameters, then in-place use
    for t in (0.0, -1.0, float("nan"), float("inf")):
        assert abi.tv_sample_filter(FAKE, FAKE + 256, 2, 16, t, 0, 1.0, 0.0, FAKE) == abi.CODES["TV_E_TEMP"]
    for k, p, mp in ((-1, 1.0, 0.0), (0, 0.0, 0.0), (0, 1.5, 0.0), (0, float("nan"), 0.0), (0, 1.0, 1.0),
                     (0, 1.0, -0.1)):
        assert abi.tv_sample_filter(FAKE, FAKE + 256, 2, 16, 1.0, k, p, mp, FAKE) == abi.CODES["TV_E_ARG"]
    assert abi.tv_sample_filter(FAKE, FAKE, 2, 16, 1.0, 0, 1.0, 0.0, FAKE) == abi.CODES["TV_E_ARG"]
    assert abi.tv_sample_filter(FAKE, FAKE + 256, 33, 16, 1.0, 0, 1.0, 0.0, FAKE) == abi.CODES["TV_E_ARG"]
    assert abi.tv_sample_filter(FAKE, FAKE + 256, 2, 262145, 1.0, 0, 1.0, 0.0, FAKE) == abi.CODES["TV_E_UNSUPPORTED"]
    # the walks: temperature, row count, workspace size, positions
    trees = [_tree(8)]
    _, ws8 = abi.tv_sample_workspace_size(1024, 8)
    args = (FAKE, FAKE, FAKE, FAKE, FAKE)
    assert abi.tv_accept_single_draw(trees, FAKE, 1024, 0.0, FAKE, *args, FAKE, ws8) == abi.CODES["TV_E_TEMP"]
    assert abi.tv_accept_single_draw([_tree(33)], FAKE, 1024, 1.0, FAKE, *args, FAKE, ws8) == abi.CODES["TV_E_ROWS"]
    assert abi.tv_accept_single_draw(trees, FAKE, 1024, 1.0, FAKE, *args, FAKE, ws8 - 256) == \
        abi.CODES["TV_E_WORKSPACE"]
    assert abi.tv_accept_gumbel(trees, FAKE, 1024, 1.0, [1], [-1], *args, FAKE, ws8) == abi.CODES["TV_E_ARG"]
    assert abi.tv_accept_gumbel(trees, FAKE, 1024, float("nan"), [1], [0], *args, FAKE, ws8) == \
        abi.CODES["TV_E_TEMP"]
    assert abi.tv_accept_gumbel(trees, FAKE, 1024, 1.0, [1], [0], *args, None, ws8) == abi.CODES["TV_E_WORKSPACE"]
    assert abi.tv_accept_rejection(trees, FAKE, 1024, 1.0, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                   ws8) == abi.CODES["TV_E_ARG"]
    assert abi.tv_accept_rejection(trees, FAKE, 1024, 1.0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                   16) == abi.CODES["TV_E_WORKSPACE"]


def test_deltanet_host_checks(lib):
    trees = [_tree(8)]
    ok = abi.TvDnDims(2, 4, 128, 128)
    args = (FAKE,) * 9   # q, k, v, beta, g, o, u, gc, dev_status
    call = lambda dims, trees=trees, states=(FAKE,): abi.tv_dn_verify_tree(dims, trees, list(states) * len(trees),
                                                                           *args[:9])
    for bad in (abi.TvDnDims(3, 4, 128, 128), abi.TvDnDims(0, 4, 128, 128), abi.TvDnDims(2, 4, 48, 128),
                abi.TvDnDims(2, 4, 128, 160), abi.TvDnDims(2, 4, 0, 128)):
        assert call(bad) == abi.CODES["TV_E_UNSUPPORTED"]
    assert call(ok, states=(FAKE + 4,)) == abi.CODES["TV_E_ARG"]          # misaligned state
    assert call(ok, trees=[_tree(40)]) == abi.CODES["TV_E_ROWS"]
    assert call(ok, trees=[_tree(20), _tree(20)]) == abi.CODES["TV_E_ROWS"]
    assert abi.tv_dn_verify_tree(ok, trees, [FAKE], None, *args[:8]) == abi.CODES["TV_E_ARG"]
    assert abi.tv_dn_commit(ok, trees, 0, [FAKE], FAKE, FAKE, FAKE, FAKE, FAKE, FAKE) == abi.CODES["TV_E_ARG"]
    assert abi.tv_dn_commit(abi.TvDnDims(2, 4, 96, 72), trees, 1, [FAKE], FAKE, FAKE, FAKE, FAKE, FAKE, FAKE) == \
        abi.CODES["TV_E_UNSUPPORTED"]
    assert abi.tv_dn_commit(ok, trees, 1, [FAKE], FAKE, FAKE, FAKE, None, FAKE, FAKE) == abi.CODES["TV_E_ARG"]


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(abi, "_lib", None)
    monkeypatch.setattr(abi, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(abi.LibraryMissing):
        abi.load()


def _param_kinds_from_header():
    """Every prototype's parameters, each as ptr / i32 / f32 / f64 / u64."""
    text = re.sub(r"/\*.*?\*/", " ", open(HEADER).read(), flags=re.S)
    out = {}
    for name, params in re.findall(r"TV_API\s+[\w\s\*]*?\b(tv_\w+)\s*\(([^)]*)\)\s*;", text):
        kinds = []
        for p in (x.strip() for x in params.split(",")):
            if not p or p == "void":
                continue
            if "*" in p:
                kinds.append("ptr")
            elif re.match(r"(const\s+)?(int|int32_t)\b", p):
                kinds.append("i32")
            elif re.match(r"(const\s+)?float\b", p):
                kinds.append("f32")
            elif re.match(r"(const\s+)?double\b", p):
                kinds.append("f64")
            elif re.match(r"(const\s+)?(size_t|uint64_t)\b", p):
                kinds.append("u64")
            else:
                raise AssertionError(f"{name}: unclassified parameter {p!r}")
        out[name] = kinds
    return out


def _ctypes_kind(t):
    if t in (ctypes.c_void_p, ctypes.c_char_p) or issubclass(t, ctypes._Pointer):
        return "ptr"
    if t in (ctypes.c_int, ctypes.c_int32):
        return "i32"
    if t is ctypes.c_float:
        return "f32"
    if t is ctypes.c_double:
        return "f64"
    if t in (ctypes.c_size_t, ctypes.c_uint64):
        return "u64"
    raise AssertionError(f"unclassified ctypes type {t}")


def test_binding_signatures_match_the_header(lib):
    """The binding's ctypes argument lists agree with include/tv.h parameter
    by parameter, so a prototype change cannot leave a stale binding."""
    header = _param_kinds_from_header()
    assert sorted(header) == _declared()
    for name, kinds in header.items():
        got = [_ctypes_kind(t) for t in getattr(lib, name).argtypes]
        assert got == kinds, (name, got, kinds)
