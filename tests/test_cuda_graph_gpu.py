"""The C-ABI calls can be captured into a CUDA graph and replayed (the pages'
audit times prepared launches under CUDA-graph replay).  Each entry is called
once before capture (per-device set-up), then captured on torch's capture
stream and replayed; the replay must match the eager call."""
import numpy as np
import pytest
import torch

import workloads
from parity import assert_parity

pytestmark = pytest.mark.gpu


def f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def capture_and_replay(call, out, replays=3):
    call()                                   # eager, also the per-device set-up
    torch.cuda.synchronize()
    eager = out.clone()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call(s)                              # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        call(torch.cuda.current_stream())
    first = None
    for _ in range(replays):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        if first is None:
            first = out.clone()
        assert torch.equal(out, first), "graph replays differ"
    return eager, out.clone()


def test_graph_dense(cuda_lib):
    w = workloads.custom("dense", 1, 1000, 1000, 4, 128)   # 16 units: split into key pieces
    q, k, v = (t.cuda() for t in workloads.make_inputs(w, seed_base=17000))
    out = torch.empty_like(q)
    eager, replay = capture_and_replay(
        lambda s=None: cuda_lib.attn_dense_fwd(q, k, v, out, stream=s), out)
    assert_parity(f64(replay), f64(eager), "graph replay vs eager (dense)")


def test_graph_prefix_and_block_causal(cuda_lib):
    B, Nq, Np, H, D = 1, 384, 200, 2, 64
    ts = [workloads.randn_bf16(s, 1.0, 17100 + i) for i, s in enumerate(
        [(B, Nq, H, D), (B, Np, H, D), (B, Np, H, D), (B, Nq, H, D), (B, Nq, H, D)])]
    q, kp, vp, kc, vc = (t.cuda() for t in ts)
    out = torch.empty_like(q)
    eager, replay = capture_and_replay(
        lambda s=None: cuda_lib.attn_prefix_fwd(q, kp, vp, kc, vc, out, stream=s), out)
    assert_parity(f64(replay), f64(eager), "graph replay vs eager (prefix)")

    ids = torch.tensor([-1] * 100 + [0] * 284, dtype=torch.int32, device="cuda")
    out2 = torch.empty_like(q)
    eager, replay = capture_and_replay(
        lambda s=None: cuda_lib.attn_block_causal_fwd(q, kc, vc, ids, out2, stream=s), out2)
    assert_parity(f64(replay), f64(eager), "graph replay vs eager (block-causal)")


def test_graph_keeps_its_split_workspace(cuda_lib):
    """Captured on a stream that has just made the same call eagerly, the
    graph takes that stream's split workspace (and clears its arrival
    counters in a captured step, since every replay repeats the captured
    launch): replays are bit-identical to the eager call, also with eager
    calls on another stream in between, which get a workspace of their own."""
    w = workloads.custom("dense", 1, 1000, 1000, 4, 128)   # 16 units: split into key pieces
    q, k, v = (t.cuda() for t in workloads.make_inputs(w, seed_base=17200))
    out = torch.empty_like(q)
    other = torch.empty_like(q)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        cuda_lib.attn_dense_fwd(q, k, v, out, stream=s)
    s.synchronize()
    eager = out.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        cuda_lib.attn_dense_fwd(q, k, v, out, stream=s)
    side = torch.cuda.Stream()
    for _ in range(3):
        out.zero_()
        g.replay()
        cuda_lib.attn_dense_fwd(q, k, v, other, stream=side)
        torch.cuda.synchronize()
        assert torch.equal(out, eager)
        assert torch.equal(other, eager)
