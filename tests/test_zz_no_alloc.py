"""tv_accept_residual_noalloc against tv_accept_residual.

The no-workspace entry point exists for callers that cannot give the library
device memory: a step running inside another framework's executor that may not
call cudaMalloc, or a loop with a no-allocation rule.  It must return exactly
what the workspace version returns on the same inputs, and keep doing so on the
next call, which finds the previous call's statistics still in the library's
fixed array.  Integer outputs, so the comparison is exact.
"""
import numpy as np
import pytest
import torch

from speculative_tree_verify_gb300 import abi, synth
from speculative_tree_verify_gb300.device import DeviceRequest, RoundBuffers

pytestmark = pytest.mark.gpu


def _inputs(V, seed):
    trees = [synth.tree_lattice(8, 7, V, seed), synth.tree_spine_random(12, 4, V, seed + 1),
             synth.tree_star(6, V, seed + 2)]
    rows = sum(t.n for t in trees)
    logits = synth.logits_rows(rows, V, seed + 3, scale=2.0)
    rng = np.random.default_rng(seed)
    off = 0
    for t in trees:                       # make some drafts likely to be accepted
        for c in range(1, t.n):
            r = off + int(t.parent[c])
            logits[r, t.token[c]] = logits[r].max() + float(rng.uniform(-1.0, 0.5))
        off += t.n
    return trees, logits, synth.uniforms(rows, seed + 4)


def _outputs(b, n_req, trees):
    out = []
    off = 0
    for r in range(n_req):
        a, cnt = int(b.accept_len[r]), int(b.out_count[r])
        out.append((a, cnt, b.path[off:off + a + 1].cpu().tolist(), b.out_tokens[off:off + cnt].cpu().tolist()))
        off += trees[r].n
    return out


@pytest.mark.parametrize("V", [151936, 1024])
def test_noalloc_walk_matches_workspace_walk(gpu, V):
    d = synth.Dims(hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64, vocab=V)
    for call in range(2):
        trees, logits, u = _inputs(V, 1000 * call + V % 97)
        reqs = [DeviceRequest(torch.zeros(2, 1, 64, device="cuda", dtype=torch.bfloat16),
                              torch.zeros(2, 1, 64, device="cuda", dtype=torch.bfloat16), 0,
                              torch.from_numpy(t.parent).cuda(), torch.from_numpy(t.token).cuda()) for t in trees]
        tt = [r.tree() for r in reqs]
        rows = sum(t.n for t in trees)
        ref = RoundBuffers.alloc(d, rows, len(trees), 0)
        new = RoundBuffers.alloc(d, rows, len(trees), 0)
        for b in (ref, new):
            b.logits.copy_(torch.from_numpy(logits))
            b.uniforms.copy_(torch.from_numpy(u))
        rc = abi.tv_accept_residual(tt, ref.logits, V, 1.0, ref.uniforms, True, ref.path, ref.accept_len,
                                    ref.out_tokens, ref.out_count, ref.status, ref.ws, ref.ws.numel())
        assert rc == abi.TV_OK
        # the second call runs on a stream of its own: the entry point takes the
        # caller's stream and needs nothing else from it
        side = torch.cuda.Stream() if call == 1 else None
        if side is not None:
            side.wait_stream(torch.cuda.current_stream())
        rc = abi.tv_accept_residual_noalloc(tt, new.logits, V, 1.0, new.uniforms, True, new.path, new.accept_len,
                                            new.out_tokens, new.out_count, new.status, stream=side)
        assert rc == abi.TV_OK
        torch.cuda.synchronize()
        assert int(ref.status.item()) == 0 and int(new.status.item()) == 0
        assert _outputs(new, len(trees), trees) == _outputs(ref, len(trees), trees), f"call {call}"


def test_noalloc_rejects_vocab_beyond_its_array(gpu):
    t = synth.tree_chain(2, 8, 0)
    req = DeviceRequest(torch.zeros(2, 1, 64, device="cuda", dtype=torch.bfloat16),
                        torch.zeros(2, 1, 64, device="cuda", dtype=torch.bfloat16), 0,
                        torch.from_numpy(t.parent).cuda(), torch.from_numpy(t.token).cuda())
    buf = torch.zeros(8, device="cuda", dtype=torch.int32)
    rc = abi.tv_accept_residual_noalloc([req.tree()], buf, 262145, 1.0, buf, True, buf, buf, buf, buf, buf)
    assert rc == abi.CODES["TV_E_UNSUPPORTED"]
