"""Python binding of the C ABI in include/tv.h -- argument marshalling only.

Every function here has the name of its C entry point and does nothing but
turn Python values (ints, torch tensors, lists of structs) into the C
arguments and call the CUDA library.  All computation happens in the
library's kernels.  If the library is missing the import of a function fails
loudly: there is no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtv.so")

TV_OK = 0
STATUS = {
    0: "TV_OK", -1: "TV_E_ARG", -2: "TV_E_ORDER", -3: "TV_E_DUP_SIBLING", -4: "TV_E_TOKEN",
    -5: "TV_E_CAPACITY", -6: "TV_E_ROWS", -7: "TV_E_UNIFORM", -8: "TV_E_TEMP", -9: "TV_E_WORKSPACE",
    -10: "TV_E_CUDA", -11: "TV_E_UNSUPPORTED", -12: "TV_E_TIMEOUT", -13: "TV_E_PATH", -14: "TV_E_CHAIN",
    -15: "TV_E_PROPOSAL",
}
CODES = {v: k for k, v in STATUS.items()}

# entry points declared in include/tv.h
SYMBOLS = ("tv_workspace_size", "tv_verify_tree", "tv_accept_greedy", "tv_accept_residual", "tv_commit_kv",
           "tv_profile_start", "tv_profile_stop", "tv_status_string", "tv_accept_residual_noalloc",
           "tv_sample_workspace_size", "tv_sample_filter", "tv_accept_single_draw", "tv_accept_gumbel",
           "tv_accept_rejection", "tv_dn_verify_tree", "tv_dn_commit", "tv_price_init", "tv_price_lookup",
           "tv_price_observe", "tv_staircut", "tv_packed_weight_bytes", "tv_pack_weight",
           "tv_accept_greedy_commit", "tv_stack_workspace_size", "tv_verify_stack", "tv_commit_stack")
PROFILE_STAGES = ("prologue+embed", "qkv_gemm", "qkv_finalize", "attention", "o_gemm", "o_finalize", "lm_head")


class TvDims(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("vocab", ctypes.c_int32), ("rope_theta", ctypes.c_float),
                ("rms_eps", ctypes.c_float)]


class TvModel(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("ln1", ctypes.c_void_p), ("wqkv", ctypes.c_void_p),
                ("wo", ctypes.c_void_p), ("ln_f", ctypes.c_void_p), ("lm_head", ctypes.c_void_p),
                ("dims", TvDims), ("packed", ctypes.c_int32)]


class TvKv(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("ctx_len", ctypes.c_int32),
                ("capacity", ctypes.c_int32)]


class TvTree(ctypes.Structure):
    _fields_ = [("parent", ctypes.c_void_p), ("token", ctypes.c_void_p), ("n", ctypes.c_int32)]


TV_KIND_CHAIN, TV_KIND_TREE = 0, 1
PRICE_MAX_CLASSES, PRICE_MAX_ROWS = 16, 32
_PriceRows = ctypes.c_double * (PRICE_MAX_ROWS + 1)


class TvPriceTable(ctypes.Structure):
    _fields_ = [("n_classes", ctypes.c_int32), ("class_ctx", ctypes.c_int32 * PRICE_MAX_CLASSES),
                ("step_ms", ctypes.c_double), ("prior", _PriceRows * 2 * PRICE_MAX_CLASSES),
                ("live", _PriceRows * 2 * PRICE_MAX_CLASSES), ("offset", ctypes.c_double * 2 * PRICE_MAX_CLASSES)]


class TvDnDims(ctypes.Structure):
    _fields_ = [("n_k_heads", ctypes.c_int32), ("n_v_heads", ctypes.c_int32), ("d_k", ctypes.c_int32),
                ("d_v", ctypes.c_int32)]


TV_LAYER_ATTN, TV_LAYER_DN = 0, 1


class TvLayer(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("ln_mix", ctypes.c_void_p), ("w_mix_in", ctypes.c_void_p),
                ("w_mix_out", ctypes.c_void_p), ("dn_norm", ctypes.c_void_p), ("ln_mlp", ctypes.c_void_p),
                ("w_gate_up", ctypes.c_void_p), ("w_down", ctypes.c_void_p)]


class TvStack(ctypes.Structure):
    _fields_ = [("dims", TvDims), ("dn", TvDnDims), ("intermediate", ctypes.c_int32), ("n_layers", ctypes.c_int32),
                ("layers", ctypes.POINTER(TvLayer)), ("embed", ctypes.c_void_p), ("ln_f", ctypes.c_void_p),
                ("lm_head", ctypes.c_void_p), ("packed", ctypes.c_int32)]


_lib = None


class LibraryMissing(RuntimeError):
    pass


def load():
    """Load libtv.so (built in-tree by speculative_tree_verify_gb300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise LibraryMissing(f"CUDA library not built: {LIB_PATH} is missing "
                                 "(run speculative_tree_verify_gb300.build.build())")
        lib = ctypes.CDLL(LIB_PATH)
        P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        lib.tv_workspace_size.argtypes = [ctypes.POINTER(TvDims), I, I, ctypes.POINTER(Z)]
        lib.tv_verify_tree.argtypes = [ctypes.POINTER(TvModel), ctypes.POINTER(TvKv), ctypes.POINTER(TvTree), I,
                                       P, P, P, P, P, Z, P, P]
        lib.tv_accept_greedy.argtypes = [ctypes.POINTER(TvTree), I, P, P, P, P, P, P]
        lib.tv_accept_residual.argtypes = [ctypes.POINTER(TvTree), I, P, ctypes.c_int32, ctypes.c_float, P, I,
                                           P, P, P, P, P, P, Z, P]
        lib.tv_accept_residual_noalloc.argtypes = [ctypes.POINTER(TvTree), I, P, ctypes.c_int32, ctypes.c_float, P,
                                                   I, P, P, P, P, P, P]
        lib.tv_commit_kv.argtypes = [ctypes.POINTER(TvKv), ctypes.POINTER(TvDims), ctypes.POINTER(TvTree), I,
                                     P, P, P, P, P, P]
        lib.tv_accept_greedy_commit.argtypes = [ctypes.POINTER(TvKv), ctypes.POINTER(TvDims), ctypes.POINTER(TvTree),
                                                I, P, P, P, P, P, P, P, P]
        lib.tv_packed_weight_bytes.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(Z)]
        lib.tv_pack_weight.argtypes = [P, ctypes.c_int32, ctypes.c_int32, P, P]
        lib.tv_profile_start.argtypes = [I]
        lib.tv_profile_stop.argtypes = [ctypes.POINTER(ctypes.c_float), I, ctypes.POINTER(I), ctypes.POINTER(I)]
        lib.tv_sample_workspace_size.argtypes = [ctypes.c_int32, I, ctypes.POINTER(Z)]
        lib.tv_sample_filter.argtypes = [P, P, I, ctypes.c_int32, ctypes.c_float, ctypes.c_int32, ctypes.c_float,
                                         ctypes.c_float, P, P]
        lib.tv_accept_single_draw.argtypes = [ctypes.POINTER(TvTree), I, P, ctypes.c_int32, ctypes.c_float, P, P,
                                              P, P, P, P, P, Z, P]
        lib.tv_accept_gumbel.argtypes = [ctypes.POINTER(TvTree), I, P, ctypes.c_int32, ctypes.c_float,
                                         ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_int32), P, P, P,
                                         P, P, P, Z, P]
        lib.tv_accept_rejection.argtypes = [ctypes.POINTER(TvTree), I, P, ctypes.c_int32, ctypes.c_float, P, P,
                                            P, P, P, P, P, P, Z, P]
        lib.tv_dn_verify_tree.argtypes = [ctypes.POINTER(TvDnDims), ctypes.POINTER(TvTree), I, ctypes.POINTER(P), P,
                                          P, P, P, P, P, P, P, P, P]
        lib.tv_dn_commit.argtypes = [ctypes.POINTER(TvDnDims), ctypes.POINTER(TvTree), I, I, ctypes.POINTER(P), P, P,
                                     P, P, P, P, P]
        lib.tv_stack_workspace_size.argtypes = [ctypes.POINTER(TvStack), ctypes.POINTER(Z)]
        lib.tv_verify_stack.argtypes = [ctypes.POINTER(TvStack), ctypes.POINTER(TvKv), ctypes.POINTER(P),
                                        ctypes.POINTER(TvTree), I, P, P, P, P, P, Z, P, P]
        lib.tv_commit_stack.argtypes = [ctypes.POINTER(TvStack), ctypes.POINTER(TvKv), ctypes.POINTER(P),
                                        ctypes.POINTER(TvTree), I, P, P, P, P, P, Z, P, P]
        D = ctypes.c_double
        lib.tv_price_init.argtypes = [ctypes.POINTER(TvPriceTable)]
        lib.tv_price_lookup.argtypes = [ctypes.POINTER(TvPriceTable), ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                        ctypes.POINTER(D)]
        lib.tv_price_observe.argtypes = [ctypes.POINTER(TvPriceTable), ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, D]
        lib.tv_staircut.argtypes = [P, P, P, ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(TvPriceTable),
                                    ctypes.c_int32, D, D, D, P, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(D)]
        lib.tv_status_string.argtypes = [I]
        lib.tv_status_string.restype = ctypes.c_char_p
        _lib = lib
    return _lib


def _p(x) -> Optional[int]:
    """Device/host address of a tensor, an int, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _arr(ctype, items: Sequence):
    return (ctype * len(items))(*items)


def _stream(stream) -> Optional[int]:
    if stream is None:
        return None
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def tv_status_string(code: int) -> str:
    return load().tv_status_string(int(code)).decode()


def tv_workspace_size(dims: TvDims, max_rows: int, max_ctx: int) -> int:
    out = ctypes.c_size_t(0)
    rc = load().tv_workspace_size(ctypes.byref(dims), int(max_rows), int(max_ctx), ctypes.byref(out))
    if rc != TV_OK:
        raise ValueError(f"tv_workspace_size: {STATUS.get(rc, rc)}")
    return int(out.value)


def tv_accept_greedy_commit(kvs: Sequence[TvKv], dims: TvDims, trees: Sequence[TvTree], argmax, path, accept_len,
                            out_tokens, committed_src, new_ctx, dev_status, stream=None) -> int:
    return load().tv_accept_greedy_commit(_arr(TvKv, kvs), ctypes.byref(dims), _arr(TvTree, trees), len(trees),
                                          _p(argmax), _p(path), _p(accept_len), _p(out_tokens), _p(committed_src),
                                          _p(new_ctx), _p(dev_status), _stream(stream))


def tv_packed_weight_bytes(rows: int, cols: int) -> int:
    out = ctypes.c_size_t(0)
    rc = load().tv_packed_weight_bytes(int(rows), int(cols), ctypes.byref(out))
    if rc != TV_OK:
        raise ValueError(f"tv_packed_weight_bytes: {STATUS.get(rc, rc)}")
    return int(out.value)


def tv_pack_weight(w, rows: int, cols: int, packed, stream=None) -> int:
    return load().tv_pack_weight(_p(w), int(rows), int(cols), _p(packed), _stream(stream))


def tv_verify_tree(model: TvModel, kvs: Sequence[TvKv], trees: Sequence[TvTree], logits, argmax, top2_gap,
                   attn_out, workspace, workspace_bytes: int, dev_status, stream=None) -> int:
    return load().tv_verify_tree(ctypes.byref(model), _arr(TvKv, kvs), _arr(TvTree, trees), len(trees),
                                 _p(logits), _p(argmax), _p(top2_gap), _p(attn_out), _p(workspace),
                                 int(workspace_bytes), _p(dev_status), _stream(stream))


def tv_accept_greedy(trees: Sequence[TvTree], argmax, path, accept_len, out_tokens, dev_status, stream=None) -> int:
    return load().tv_accept_greedy(_arr(TvTree, trees), len(trees), _p(argmax), _p(path), _p(accept_len),
                                   _p(out_tokens), _p(dev_status), _stream(stream))


def tv_accept_residual(trees: Sequence[TvTree], logits, vocab: int, temperature: float, uniforms,
                       bonus_at_leaf: bool, path, accept_len, out_tokens, out_count, dev_status, workspace,
                       workspace_bytes: int, stream=None) -> int:
    return load().tv_accept_residual(_arr(TvTree, trees), len(trees), _p(logits), int(vocab), float(temperature),
                                     _p(uniforms), 1 if bonus_at_leaf else 0, _p(path), _p(accept_len),
                                     _p(out_tokens), _p(out_count), _p(dev_status), _p(workspace),
                                     int(workspace_bytes), _stream(stream))


def tv_accept_residual_noalloc(trees: Sequence[TvTree], logits, vocab: int, temperature: float, uniforms,
                               bonus_at_leaf: bool, path, accept_len, out_tokens, out_count, dev_status,
                               stream=None) -> int:
    """tv_accept_residual for callers that cannot provide a workspace (the
    statistics live in a fixed 272 KB array inside the library; vocab <= 262144)."""
    return load().tv_accept_residual_noalloc(_arr(TvTree, trees), len(trees), _p(logits), int(vocab),
                                             float(temperature), _p(uniforms), 1 if bonus_at_leaf else 0,
                                             _p(path), _p(accept_len), _p(out_tokens), _p(out_count),
                                             _p(dev_status), _stream(stream))


def tv_sample_workspace_size(vocab: int, max_rows: int):
    """(rc, bytes) of workspace the sampled entry points need."""
    z = ctypes.c_size_t(0)
    rc = load().tv_sample_workspace_size(int(vocab), int(max_rows), ctypes.byref(z))
    return rc, int(z.value)


def tv_sample_filter(logits, filtered, rows: int, vocab: int, temperature: float, top_k: int, top_p: float,
                     min_p: float, dev_status, stream=None) -> int:
    return load().tv_sample_filter(_p(logits), _p(filtered), int(rows), int(vocab), float(temperature), int(top_k),
                                   float(top_p), float(min_p), _p(dev_status), _stream(stream))


def tv_accept_single_draw(trees: Sequence[TvTree], logits, vocab: int, temperature: float, uniforms, row_tokens,
                          path, accept_len, out_tokens, dev_status, workspace, workspace_bytes: int,
                          stream=None) -> int:
    return load().tv_accept_single_draw(_arr(TvTree, trees), len(trees), _p(logits), int(vocab), float(temperature),
                                        _p(uniforms), _p(row_tokens), _p(path), _p(accept_len), _p(out_tokens),
                                        _p(dev_status), _p(workspace), int(workspace_bytes), _stream(stream))


def tv_accept_gumbel(trees: Sequence[TvTree], logits, vocab: int, temperature: float, seeds: Sequence[int],
                     positions: Sequence[int], row_tokens, path, accept_len, out_tokens, dev_status, workspace,
                     workspace_bytes: int, stream=None) -> int:
    sd = (ctypes.c_uint64 * len(trees))(*[int(x) & 0xFFFFFFFFFFFFFFFF for x in seeds])
    ps = (ctypes.c_int32 * len(trees))(*[int(x) for x in positions])
    return load().tv_accept_gumbel(_arr(TvTree, trees), len(trees), _p(logits), int(vocab), float(temperature), sd,
                                   ps, _p(row_tokens), _p(path), _p(accept_len), _p(out_tokens), _p(dev_status),
                                   _p(workspace), int(workspace_bytes), _stream(stream))


def tv_accept_rejection(trees: Sequence[TvTree], logits, vocab: int, temperature: float, proposals, uniforms,
                        path, accept_len, out_tokens, out_count, dev_status, workspace, workspace_bytes: int,
                        stream=None) -> int:
    return load().tv_accept_rejection(_arr(TvTree, trees), len(trees), _p(logits), int(vocab), float(temperature),
                                      _p(proposals), _p(uniforms), _p(path), _p(accept_len), _p(out_tokens),
                                      _p(out_count), _p(dev_status), _p(workspace), int(workspace_bytes),
                                      _stream(stream))


def _ptrs(states):
    return (ctypes.c_void_p * len(states))(*[_p(x) for x in states])


def tv_dn_verify_tree(dims: TvDnDims, trees: Sequence[TvTree], states, q, k, v, beta, g, o, u, gc, dev_status,
                      stream=None) -> int:
    """states: one device buffer (tensor or address) per request."""
    return load().tv_dn_verify_tree(ctypes.byref(dims), _arr(TvTree, trees), len(trees), _ptrs(states), _p(q), _p(k),
                                    _p(v), _p(beta), _p(g), _p(o), _p(u), _p(gc), _p(dev_status), _stream(stream))


def tv_dn_commit(dims: TvDnDims, trees: Sequence[TvTree], n_layers: int, states, k, u, gc, path, accept_len,
                 dev_status, stream=None) -> int:
    return load().tv_dn_commit(ctypes.byref(dims), _arr(TvTree, trees), len(trees), int(n_layers), _ptrs(states),
                               _p(k), _p(u), _p(gc), _p(path), _p(accept_len), _p(dev_status), _stream(stream))


def tv_stack_workspace_size(stack: TvStack):
    """(rc, bytes) of workspace tv_verify_stack / tv_commit_stack need."""
    z = ctypes.c_size_t(0)
    rc = load().tv_stack_workspace_size(ctypes.byref(stack), ctypes.byref(z))
    return rc, int(z.value)


def tv_verify_stack(stack: TvStack, kvs: Sequence[TvKv], dn_states, trees: Sequence[TvTree], logits, argmax,
                    top2_gap, x_taps, workspace, workspace_bytes: int, dev_status, stream=None) -> int:
    """kvs: [n_attn_layers * n_req] (layer-major); dn_states: one device buffer
    per request; x_taps: bf16 [2 n_layers + 1][rows][hidden] or None."""
    return load().tv_verify_stack(ctypes.byref(stack), _arr(TvKv, kvs) if kvs else None,
                                  _ptrs(dn_states) if dn_states else None, _arr(TvTree, trees), len(trees),
                                  _p(logits), _p(argmax), _p(top2_gap), _p(x_taps), _p(workspace),
                                  int(workspace_bytes), _p(dev_status), _stream(stream))


def tv_commit_stack(stack: TvStack, kvs: Sequence[TvKv], dn_states, trees: Sequence[TvTree], path, accept_len,
                    committed_src, new_ctx, workspace, workspace_bytes: int, dev_status, stream=None) -> int:
    return load().tv_commit_stack(ctypes.byref(stack), _arr(TvKv, kvs) if kvs else None, _ptrs(dn_states) if dn_states else None,
                                  _arr(TvTree, trees), len(trees), _p(path), _p(accept_len), _p(committed_src),
                                  _p(new_ctx), _p(workspace), int(workspace_bytes), _p(dev_status), _stream(stream))


def tv_price_init(table: TvPriceTable) -> int:
    return load().tv_price_init(ctypes.byref(table))


def tv_price_lookup(table: TvPriceTable, context: int, kind: int, rows: int):
    """(rc, ms)"""
    ms = ctypes.c_double(0.0)
    rc = load().tv_price_lookup(ctypes.byref(table), int(context), int(kind), int(rows), ctypes.byref(ms))
    return rc, ms.value


def tv_price_observe(table: TvPriceTable, context: int, kind: int, rows: int, ms: float) -> int:
    return load().tv_price_observe(ctypes.byref(table), int(context), int(kind), int(rows), float(ms))


def tv_staircut(parent, q, score, kind: int, table: TvPriceTable, context: int, draft_ms: float, commit_ms: float,
                rollback_ms: float = 0.0):
    """Host arrays (numpy int32 / float32).  Returns (rc, kept nodes, value)."""
    import numpy as np
    par = np.ascontiguousarray(parent, dtype=np.int32)
    qq = np.ascontiguousarray(q, dtype=np.float32)
    sc = np.ascontiguousarray(score, dtype=np.float32)
    n = int(par.shape[0])
    keep = np.zeros(max(n, 1), dtype=np.int32)
    nk, val = ctypes.c_int32(0), ctypes.c_double(0.0)
    rc = load().tv_staircut(par.ctypes.data, qq.ctypes.data, sc.ctypes.data, n, int(kind), ctypes.byref(table),
                            int(context), float(draft_ms), float(commit_ms), float(rollback_ms), keep.ctypes.data,
                            ctypes.byref(nk), ctypes.byref(val))
    return rc, keep[:nk.value].tolist(), val.value


def tv_commit_kv(kvs: Sequence[TvKv], dims: TvDims, trees: Sequence[TvTree], path, accept_len, committed_src,
                 new_ctx, dev_status, stream=None) -> int:
    return load().tv_commit_kv(_arr(TvKv, kvs), ctypes.byref(dims), _arr(TvTree, trees), len(trees), _p(path),
                               _p(accept_len), _p(committed_src), _p(new_ctx), _p(dev_status), _stream(stream))


def tv_profile_start(max_calls: int) -> int:
    return load().tv_profile_start(int(max_calls))


def tv_profile_stop():
    """-> (rc, {stage name: summed ms}, recorded calls)"""
    ms = (ctypes.c_float * len(PROFILE_STAGES))()
    ns, nc = ctypes.c_int(0), ctypes.c_int(0)
    rc = load().tv_profile_stop(ms, len(PROFILE_STAGES), ctypes.byref(ns), ctypes.byref(nc))
    return rc, {name: float(ms[i]) for i, name in enumerate(PROFILE_STAGES)}, int(nc.value)
