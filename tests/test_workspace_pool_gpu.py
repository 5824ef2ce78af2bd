"""The split workspaces form a bounded pool per device.

Calls on many streams at once must neither grow device memory past the pool
(at most four workspaces per device) nor share a workspace between calls in
flight: when every workspace is busy a call runs its units whole instead, and
its result differs from a split call's only by rounding order.
"""
import numpy as np
import pytest
import torch

import workloads
from parity import assert_parity

pytestmark = pytest.mark.gpu

POOL = 4


def f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def workspace_bytes() -> int:
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    partials = 2 * sms * 2 * 128 * (128 + 4) * 4
    counters = 2 * sms * 8
    return partials + counters


def test_pool_bounded_under_stream_churn(cuda_lib, oracle_mod):
    w = workloads.custom("dense", 1, 2048, 2048, 3, 128)   # 24 units: all split
    ins = workloads.make_inputs(w, seed_base=14000)
    q, k, v = (t.cuda() for t in ins)
    ref = torch.empty_like(q)
    cuda_lib.attn_dense_fwd(q, k, v, ref)
    outs = [torch.empty_like(q) for _ in range(64)]
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        streams = [torch.cuda.Stream() for _ in range(64)]
        for s, o in zip(streams, outs):
            s.wait_stream(torch.cuda.current_stream())
            cuda_lib.attn_dense_fwd(q, k, v, o, stream=s)
        torch.cuda.synchronize()
        del streams
    free1 = torch.cuda.mem_get_info()[0]
    assert cuda_lib.device_status()[0] == cuda_lib.ATTN_OK
    grown = free0 - free1
    assert grown <= (POOL - 1) * workspace_bytes() + (16 << 20), grown
    expected = oracle_mod.dense_attention(*(workloads.bf16_bits(t) for t in ins))
    assert_parity(f64(ref), expected, "reference call")
    for n, o in enumerate(outs):
        if not torch.equal(o, ref):   # ran unsplit: another rounding order
            assert_parity(f64(o), expected, f"call on stream {n}")


def test_sequential_streams_reuse_one_workspace(cuda_lib):
    """Calls on fresh streams that do not overlap in time keep taking free
    workspaces, so memory does not grow, and every call splits (bit-identical
    results)."""
    w = workloads.custom("dense", 1, 2048, 2048, 3, 128)
    q, k, v = (t.cuda() for t in workloads.make_inputs(w, seed_base=14100))
    ref = torch.empty_like(q)
    cuda_lib.attn_dense_fwd(q, k, v, ref)
    out = torch.empty_like(q)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(64):
        s = torch.cuda.Stream()
        cuda_lib.attn_dense_fwd(q, k, v, out, stream=s)
        s.synchronize()
        assert torch.equal(out, ref)
    assert torch.cuda.mem_get_info()[0] >= free0 - (16 << 20)
