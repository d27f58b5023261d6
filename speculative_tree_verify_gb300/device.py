"""Device-memory plumbing around the C ABI: torch allocates and holds the
buffers, the C library computes.  Nothing here does any of the method's
arithmetic.

  DeviceModel   -- the layer's weights on the GPU + its TvModel struct
  DeviceRequest -- one request's KV cache and draft tree on the GPU
  RoundBuffers  -- every output and the workspace of one verify round
  run_round     -- verify -> accept -> commit through the C ABI on one stream
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional, Sequence

import numpy as np
import torch

from . import abi
from .synth import Cache, Dims, Model, Tree


def _bf16_tensor(bits: np.ndarray, device) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device=device, non_blocking=False).view(torch.bfloat16)


def tv_dims(d: Dims) -> abi.TvDims:
    return abi.TvDims(d.hidden, d.n_q_heads, d.n_kv_heads, d.head_dim, d.vocab, float(d.rope_theta),
                      float(d.rms_eps))


PACKED = ("wqkv", "wo", "lm_head")


class DeviceModel:
    """The layer + head on the GPU.  packed=True (the default) also makes the
    tile-packed copies of wqkv, wo and lm_head (tv_pack_weight) and hands
    those to the verify; the row-major tensors stay in ``t``."""

    def __init__(self, dims: Dims, tensors: dict, packed: bool = True):
        self.dims = dims
        self.t = tensors    # name -> bf16 tensor on the GPU, row-major
        self.p = {}         # name -> packed copy (packed=True)
        ptr = {k: self.t[k].data_ptr() for k in ("embed", "ln1", "wqkv", "wo", "ln_f", "lm_head")}
        if packed:
            for k in PACKED:
                w = self.t[k]
                rows, cols = int(w.shape[0]), int(w.shape[1])
                buf = torch.empty(abi.tv_packed_weight_bytes(rows, cols) // 2, dtype=torch.bfloat16, device=w.device)
                check(abi.tv_pack_weight(w, rows, cols, buf, stream=torch.cuda.current_stream(w.device)),
                      "tv_pack_weight")
                self.p[k] = buf
                ptr[k] = buf.data_ptr()
        self.packed = bool(packed)
        self.c = abi.TvModel(*(ptr[k] for k in ("embed", "ln1", "wqkv", "wo", "ln_f", "lm_head")), tv_dims(dims),
                             1 if packed else 0)

    @classmethod
    def from_host(cls, m: Model, device="cuda", packed: bool = True) -> "DeviceModel":
        return cls(m.dims, {k: _bf16_tensor(getattr(m, k), device)
                            for k in ("embed", "ln1", "wqkv", "wo", "ln_f", "lm_head")}, packed)

    @classmethod
    def random(cls, dims: Dims, seed: int, device="cuda", std: float = 0.02, packed: bool = True) -> "DeviceModel":
        """Random-init weights drawn on the device (torch's generator), gains 1."""
        g = torch.Generator(device=device)
        g.manual_seed(seed)
        H, V = dims.hidden, dims.vocab

        def w(*shape):
            return (torch.randn(*shape, generator=g, device=device, dtype=torch.float32) * std).to(torch.bfloat16)

        t = {"embed": w(V, H), "wqkv": w(dims.qkv_out, H), "wo": w(H, dims.n_q_heads * dims.head_dim),
             "lm_head": w(V, H), "ln1": torch.ones(H, device=device, dtype=torch.bfloat16),
             "ln_f": torch.ones(H, device=device, dtype=torch.bfloat16)}
        return cls(dims, t, packed)


class DeviceRequest:
    def __init__(self, k: torch.Tensor, v: torch.Tensor, ctx_len: int, parent: torch.Tensor, token: torch.Tensor):
        self.k, self.v = k, v
        self.ctx_len = int(ctx_len)
        self.capacity = int(k.shape[1])
        self.parent, self.token = parent, token

    @classmethod
    def from_host(cls, cache: Cache, tree: Tree, device="cuda") -> "DeviceRequest":
        return cls(_bf16_tensor(cache.k, device), _bf16_tensor(cache.v, device), cache.ctx_len,
                   torch.from_numpy(np.ascontiguousarray(tree.parent, np.int32)).to(device),
                   torch.from_numpy(np.ascontiguousarray(tree.token, np.int32)).to(device))

    @property
    def n(self) -> int:
        return int(self.parent.shape[0])

    def kv(self) -> abi.TvKv:
        return abi.TvKv(self.k.data_ptr(), self.v.data_ptr(), self.ctx_len, self.capacity)

    def tree(self) -> abi.TvTree:
        return abi.TvTree(self.parent.data_ptr(), self.token.data_ptr(), self.n)


@dataclass
class RoundBuffers:
    dims: Dims
    rows: int
    ws: torch.Tensor
    logits: torch.Tensor
    argmax: torch.Tensor
    gap: torch.Tensor
    attn: torch.Tensor
    status: torch.Tensor
    path: torch.Tensor
    accept_len: torch.Tensor
    out_tokens: torch.Tensor
    out_count: torch.Tensor
    committed_src: torch.Tensor
    new_ctx: torch.Tensor
    uniforms: torch.Tensor

    @classmethod
    def alloc(cls, dims: Dims, rows: int, n_req: int, max_ctx: int, device="cuda") -> "RoundBuffers":
        ws_bytes = abi.tv_workspace_size(tv_dims(dims), rows, max_ctx)
        i32 = dict(device=device, dtype=torch.int32)
        return cls(dims, rows,
                   ws=torch.empty(ws_bytes, device=device, dtype=torch.uint8),
                   logits=torch.empty(rows, dims.vocab, device=device, dtype=torch.float32),
                   argmax=torch.empty(rows, **i32), gap=torch.empty(rows, device=device, dtype=torch.float32),
                   attn=torch.empty(rows, dims.n_q_heads * dims.head_dim, device=device, dtype=torch.bfloat16),
                   status=torch.zeros(1, **i32), path=torch.full((rows,), -1, **i32),
                   accept_len=torch.zeros(n_req, **i32), out_tokens=torch.full((rows,), -1, **i32),
                   out_count=torch.zeros(n_req, **i32), committed_src=torch.full((rows,), -1, **i32),
                   new_ctx=torch.zeros(n_req, **i32),
                   uniforms=torch.zeros(rows, device=device, dtype=torch.float32))


def check(rc: int, what: str):
    if rc != abi.TV_OK:
        raise RuntimeError(f"{what}: {abi.STATUS.get(rc, rc)}")


def verify(model: DeviceModel, reqs: Sequence[DeviceRequest], b: RoundBuffers, stream=None, with_attn=True) -> int:
    return abi.tv_verify_tree(model.c, [r.kv() for r in reqs], [r.tree() for r in reqs], b.logits, b.argmax, b.gap,
                              b.attn if with_attn else None, b.ws, b.ws.numel(), b.status, stream)


def accept_greedy(reqs: Sequence[DeviceRequest], b: RoundBuffers, stream=None) -> int:
    return abi.tv_accept_greedy([r.tree() for r in reqs], b.argmax, b.path, b.accept_len, b.out_tokens, b.status,
                                stream)


def accept_residual(reqs: Sequence[DeviceRequest], b: RoundBuffers, temperature: float, bonus_at_leaf=True,
                    stream=None) -> int:
    return abi.tv_accept_residual([r.tree() for r in reqs], b.logits, b.dims.vocab, temperature, b.uniforms,
                                  bonus_at_leaf, b.path, b.accept_len, b.out_tokens, b.out_count, b.status, b.ws,
                                  b.ws.numel(), stream)


def commit(reqs: Sequence[DeviceRequest], b: RoundBuffers, stream=None) -> int:
    return abi.tv_commit_kv([r.kv() for r in reqs], tv_dims(b.dims), [r.tree() for r in reqs], b.path,
                            b.accept_len, b.committed_src, b.new_ctx, b.status, stream)


def accept_greedy_commit(reqs: Sequence[DeviceRequest], b: RoundBuffers, stream=None) -> int:
    """The greedy walk and the commit in one launch (tv_accept_greedy_commit)."""
    return abi.tv_accept_greedy_commit([r.kv() for r in reqs], tv_dims(b.dims), [r.tree() for r in reqs], b.argmax,
                                       b.path, b.accept_len, b.out_tokens, b.committed_src, b.new_ctx, b.status,
                                       stream)


@dataclass
class SampleBuffers:
    """Workspace and outputs of the sampled entry points (filters, single-draw,
    Gumbel and rejection walks) for up to ``rows`` tree rows."""
    ws: torch.Tensor
    row_tokens: torch.Tensor
    filtered: torch.Tensor

    @classmethod
    def alloc(cls, vocab: int, rows: int, device="cuda") -> "SampleBuffers":
        rc, nbytes = abi.tv_sample_workspace_size(vocab, rows)
        check(rc, "tv_sample_workspace_size")
        return cls(ws=torch.empty(nbytes, device=device, dtype=torch.uint8),
                   row_tokens=torch.empty(rows, device=device, dtype=torch.int32),
                   filtered=torch.empty(rows, vocab, device=device, dtype=torch.float32))


def sample_filter(b: RoundBuffers, sb: SampleBuffers, rows: int, temperature: float, top_k: int = 0,
                  top_p: float = 1.0, min_p: float = 0.0, stream=None) -> int:
    return abi.tv_sample_filter(b.logits, sb.filtered, rows, b.dims.vocab, temperature, top_k, top_p, min_p,
                                b.status, stream)


def accept_single_draw(reqs: Sequence[DeviceRequest], b: RoundBuffers, sb: SampleBuffers, temperature: float,
                       filtered: bool = False, stream=None) -> int:
    return abi.tv_accept_single_draw([r.tree() for r in reqs], sb.filtered if filtered else b.logits, b.dims.vocab,
                                     temperature, b.uniforms, sb.row_tokens, b.path, b.accept_len, b.out_tokens,
                                     b.status, sb.ws, sb.ws.numel(), stream)


def accept_gumbel(reqs: Sequence[DeviceRequest], b: RoundBuffers, sb: SampleBuffers, temperature: float,
                  seeds: Sequence[int], positions: Sequence[int], filtered: bool = False, stream=None) -> int:
    return abi.tv_accept_gumbel([r.tree() for r in reqs], sb.filtered if filtered else b.logits, b.dims.vocab,
                                temperature, seeds, positions, sb.row_tokens, b.path, b.accept_len, b.out_tokens,
                                b.status, sb.ws, sb.ws.numel(), stream)


def accept_rejection(reqs: Sequence[DeviceRequest], b: RoundBuffers, sb: SampleBuffers, temperature: float,
                     proposals: torch.Tensor, stream=None) -> int:
    return abi.tv_accept_rejection([r.tree() for r in reqs], b.logits, b.dims.vocab, temperature, proposals,
                                   b.uniforms, b.path, b.accept_len, b.out_tokens, b.out_count, b.status, sb.ws,
                                   sb.ws.numel(), stream)


def run_round(model: DeviceModel, reqs: Sequence[DeviceRequest], b: RoundBuffers, sampled: Optional[float] = None,
              stream=None):
    """One round on one stream: verify, accept (greedy, or residual sampling at
    temperature ``sampled``), commit; the greedy walk and the commit are one
    launch (tv_accept_greedy_commit).  Raises on a host-side error code."""
    check(verify(model, reqs, b, stream), "tv_verify_tree")
    if sampled is None:
        check(accept_greedy_commit(reqs, b, stream), "tv_accept_greedy_commit")
    else:
        check(accept_residual(reqs, b, sampled, stream=stream), "tv_accept_residual")
        check(commit(reqs, b, stream), "tv_commit_kv")


# ---------------------------------------------------------------------------
# the decoder-layer stack (tv_verify_stack / tv_commit_stack)
# ---------------------------------------------------------------------------
def _stack_weight_names(attn: bool):
    return ("w_mix_in", "w_mix_out", "w_gate_up", "w_down")


class DeviceStack:
    """A layer stack on the GPU and its TvStack struct.  ``layers`` holds per
    layer a dict of bf16 tensors (ln_mix, ln_mlp, w_mix_in, w_mix_out, dn_norm,
    w_gate_up, w_down); with packed=True the four GEMM weights of every layer
    and the head are handed to the library as tile-packed copies (the
    row-major tensors are dropped when ``keep_rowmajor`` is False)."""

    def __init__(self, dims, embed, ln_f, lm_head, layers: list, packed: bool = True, keep_rowmajor: bool = True):
        from .synth import StackDims  # noqa: F401  (type only)
        self.dims = dims
        self.embed, self.ln_f = embed, ln_f
        self.layers = layers
        self.packed = bool(packed)
        self.head = self._pack(lm_head, keep_rowmajor) if packed else lm_head
        self.head_rowmajor = lm_head if (keep_rowmajor or not packed) else None
        self.c_layers = (abi.TvLayer * len(layers))()
        for i, L in enumerate(layers):
            if packed:
                for k in _stack_weight_names(L["attn"]):
                    L["p_" + k] = self._pack(L[k], keep_rowmajor)
                    if not keep_rowmajor:
                        L[k] = None
            ptr = lambda k: (L["p_" + k] if packed else L[k]).data_ptr()
            self.c_layers[i] = abi.TvLayer(abi.TV_LAYER_ATTN if L["attn"] else abi.TV_LAYER_DN, L["ln_mix"].data_ptr(),
                                           ptr("w_mix_in"), ptr("w_mix_out"),
                                           L["dn_norm"].data_ptr() if L.get("dn_norm") is not None else None,
                                           L["ln_mlp"].data_ptr(), ptr("w_gate_up"), ptr("w_down"))
        b = dims.base
        self.c = abi.TvStack(tv_dims(b), abi.TvDnDims(dims.n_k_heads, dims.n_v_heads, dims.d_k, dims.d_v),
                             dims.intermediate, len(layers), self.c_layers, embed.data_ptr(), ln_f.data_ptr(),
                             self.head.data_ptr(), 1 if packed else 0)

    @staticmethod
    def _pack(w: torch.Tensor, keep: bool) -> torch.Tensor:
        rows, cols = int(w.shape[0]), int(w.shape[1])
        buf = torch.empty(abi.tv_packed_weight_bytes(rows, cols) // 2, dtype=torch.bfloat16, device=w.device)
        check(abi.tv_pack_weight(w, rows, cols, buf, stream=torch.cuda.current_stream(w.device)), "tv_pack_weight")
        return buf

    @classmethod
    def from_host(cls, m, device="cuda", packed: bool = True) -> "DeviceStack":
        t = lambda a: _bf16_tensor(a, device)
        layers = []
        for L in m.layers:
            d = {"attn": bool(L.attn), "ln_mix": t(L.ln_mix), "ln_mlp": t(L.ln_mlp), "w_gate_up": t(L.w_gu),
                 "w_down": t(L.w_down)}
            if L.attn:
                d.update(w_mix_in=t(L.wqkv), w_mix_out=t(L.wo), dn_norm=None)
            else:
                d.update(w_mix_in=t(L.w_in), w_mix_out=t(L.w_out), dn_norm=t(L.dn_norm))
            layers.append(d)
        return cls(m.dims, t(m.embed), t(m.ln_f), t(m.lm_head), layers, packed)

    @classmethod
    def random(cls, dims, seed: int, device="cuda", std: float = 0.02, packed: bool = True,
               keep_rowmajor: bool = False) -> "DeviceStack":
        """Random-init weights drawn on the device, gains 1, the residual
        output projections with std / sqrt(2 L) as in synth.gen_stack; with
        packed and not keep_rowmajor, each weight is packed as it is drawn and
        only the packed copy is kept (a 64-layer stack at hidden 5120 then
        holds ~46 GB)."""
        g = torch.Generator(device=device)
        g.manual_seed(seed)
        b = dims.base
        H = b.hidden
        out_std = std / float(np.sqrt(2 * dims.n_layers))

        def w(*shape, sd=std):
            return (torch.randn(*shape, generator=g, device=device, dtype=torch.float32) * sd).to(torch.bfloat16)

        ones = lambda n: torch.ones(n, device=device, dtype=torch.bfloat16)
        embed = w(b.vocab, H)
        layers = []
        for l in range(dims.n_layers):
            a = dims.is_attn(l)
            d = {"attn": a, "ln_mix": ones(H), "ln_mlp": ones(H)}
            if a:
                d.update(w_mix_in=w(b.qkv_out, H), w_mix_out=w(H, b.n_q_heads * b.head_dim, sd=out_std), dn_norm=None)
            else:
                d.update(w_mix_in=w(dims.dn_in_out, H), w_mix_out=w(H, dims.n_v_heads * dims.d_v, sd=out_std),
                         dn_norm=ones(dims.d_v))
            d.update(w_gate_up=w(2 * dims.intermediate, H), w_down=w(H, dims.intermediate, sd=out_std))
            if packed and not keep_rowmajor:
                for k in _stack_weight_names(a):
                    d["p_" + k] = cls._pack(d[k], False)
                    d[k] = None
            layers.append(d)
        lm_head = w(b.vocab, H)
        obj = cls.__new__(cls)
        if packed and not keep_rowmajor:
            # already packed: build the struct without packing again
            obj.dims, obj.embed, obj.ln_f, obj.layers, obj.packed = dims, embed, ones(H), layers, True
            obj.head = cls._pack(lm_head, False)
            obj.head_rowmajor = None
            del lm_head
            obj.c_layers = (abi.TvLayer * len(layers))()
            for i, L in enumerate(layers):
                obj.c_layers[i] = abi.TvLayer(abi.TV_LAYER_ATTN if L["attn"] else abi.TV_LAYER_DN,
                                              L["ln_mix"].data_ptr(), L["p_w_mix_in"].data_ptr(),
                                              L["p_w_mix_out"].data_ptr(),
                                              L["dn_norm"].data_ptr() if L["dn_norm"] is not None else None,
                                              L["ln_mlp"].data_ptr(), L["p_w_gate_up"].data_ptr(),
                                              L["p_w_down"].data_ptr())
            obj.c = abi.TvStack(tv_dims(b), abi.TvDnDims(dims.n_k_heads, dims.n_v_heads, dims.d_k, dims.d_v),
                                dims.intermediate, len(layers), obj.c_layers, embed.data_ptr(), obj.ln_f.data_ptr(),
                                obj.head.data_ptr(), 1)
            return obj
        cls.__init__(obj, dims, embed, ones(H), lm_head, layers, packed, keep_rowmajor)
        return obj


class StackRequest:
    """One request of a stack verify: a KV cache per attention layer (k, v
    [Hkv][capacity][D] bf16, one ctx_len), the DeltaNet states [n_dn][Hv][dk][dv]
    fp32 and the draft tree."""

    def __init__(self, ks: list, vs: list, ctx_len: int, states: torch.Tensor, parent: torch.Tensor,
                 token: torch.Tensor):
        self.ks, self.vs = ks, vs
        self.ctx_len = int(ctx_len)
        self.states = states
        self.parent, self.token = parent, token

    @property
    def n(self) -> int:
        return int(self.parent.shape[0])

    def kv(self, j: int) -> abi.TvKv:
        return abi.TvKv(self.ks[j].data_ptr(), self.vs[j].data_ptr(), self.ctx_len, int(self.ks[j].shape[1]))

    def tree(self) -> abi.TvTree:
        return abi.TvTree(self.parent.data_ptr(), self.token.data_ptr(), self.n)


def stack_kvs(model: DeviceStack, reqs: Sequence[StackRequest]) -> list:
    n_attn = len(model.dims.attn_layers)
    return [r.kv(j) for j in range(n_attn) for r in reqs]


@dataclass
class StackBuffers:
    ws: torch.Tensor
    logits: torch.Tensor
    argmax: torch.Tensor
    gap: torch.Tensor
    status: torch.Tensor
    path: torch.Tensor
    accept_len: torch.Tensor
    out_tokens: torch.Tensor
    committed_src: torch.Tensor
    new_ctx: torch.Tensor

    @classmethod
    def alloc(cls, model: DeviceStack, rows: int, n_req: int, device="cuda") -> "StackBuffers":
        rc, nbytes = abi.tv_stack_workspace_size(model.c)
        check(rc, "tv_stack_workspace_size")
        i32 = dict(device=device, dtype=torch.int32)
        return cls(ws=torch.empty(nbytes, device=device, dtype=torch.uint8),
                   logits=torch.empty(rows, model.dims.base.vocab, device=device, dtype=torch.float32),
                   argmax=torch.empty(rows, **i32), gap=torch.empty(rows, device=device, dtype=torch.float32),
                   status=torch.zeros(1, **i32), path=torch.full((rows,), -1, **i32),
                   accept_len=torch.zeros(n_req, **i32), out_tokens=torch.full((rows,), -1, **i32),
                   committed_src=torch.full((rows,), -1, **i32), new_ctx=torch.zeros(n_req, **i32))


def verify_stack(model: DeviceStack, reqs: Sequence[StackRequest], b: StackBuffers, stream=None,
                 x_taps: Optional[torch.Tensor] = None) -> int:
    return abi.tv_verify_stack(model.c, stack_kvs(model, reqs), [r.states for r in reqs], [r.tree() for r in reqs],
                               b.logits, b.argmax, b.gap, x_taps, b.ws, b.ws.numel(), b.status, stream)


def commit_stack(model: DeviceStack, reqs: Sequence[StackRequest], b: StackBuffers, stream=None) -> int:
    return abi.tv_commit_stack(model.c, stack_kvs(model, reqs), [r.states for r in reqs], [r.tree() for r in reqs],
                               b.path, b.accept_len, b.committed_src, b.new_ctx, b.ws, b.ws.numel(), b.status, stream)


def run_stack_round(model: DeviceStack, reqs: Sequence[StackRequest], b: StackBuffers, stream=None):
    """Verify through the stack, greedy walk, commit of every layer."""
    check(verify_stack(model, reqs, b, stream), "tv_verify_stack")
    check(abi.tv_accept_greedy([r.tree() for r in reqs], b.argmax, b.path, b.accept_len, b.out_tokens, b.status,
                               stream), "tv_accept_greedy")
    check(commit_stack(model, reqs, b, stream), "tv_commit_stack")
