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
