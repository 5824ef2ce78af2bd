"""attn_dense_fwd_noalloc: dense attention for callers that cannot allocate
device memory (an engine whose pool owns the GPU memory, a plugin given only
its buffers, a loop that cannot pay for cudaMalloc's synchronisation).

It runs the same kernel and schedule as attn_dense_fwd, with the split
workspace in the library's static device scratch instead of a cudaMalloc'd
buffer.  Each case calls it twice in a row through the C ABI; both outputs
must be bit-identical to attn_dense_fwd's (same schedule, same merge order),
and one case is compared with the FP64 oracle directly.  A call whose launch
gave up on a bounded wait must not disturb the next one, which clears the
scratch's arrival counters first.
This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from parity import assert_parity

pytestmark = pytest.mark.gpu

CASES = [  # (B, N, H, D): all cut their units into key-range pieces
    (1, 2048, 3, 128),
    (1, 4096, 32, 128),
    (1, 4096, 1, 64),
    (2, 1000, 1, 128),
]


def noalloc(cuda_lib, q, k, v, out):
    """One call of the C entry point on the current stream; returns its status."""
    B, N, H, D = q.shape
    stream = torch.cuda.current_stream().cuda_stream
    return cuda_lib.load_library().attn_dense_fwd_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
        ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(out.data_ptr()), B, N, H, D,
        ctypes.c_void_p(stream))


def f64(t):
    return t.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("B,N,H,D", CASES)
def test_noalloc_matches_dense_twice(cuda_lib, B, N, H, D):
    w = workloads.custom("dense", B, N, N, H, D)
    q, k, v = (t.cuda() for t in workloads.make_inputs(w, seed_base=13000 + N + D))
    ref = torch.empty_like(q)
    cuda_lib.attn_dense_fwd(q, k, v, ref)
    outs = []
    for _ in range(2):
        out = torch.full_like(q, float("nan"))
        rc = noalloc(cuda_lib, q, k, v, out)
        assert rc == cuda_lib.ATTN_OK, cuda_lib.status_string(rc)
        outs.append(out)
    torch.cuda.synchronize()
    assert cuda_lib.device_status()[0] == cuda_lib.ATTN_OK
    for out in outs:
        assert torch.equal(out, ref), f"noalloc differs from attn_dense_fwd on {w.describe()}"


def test_noalloc_matches_oracle(cuda_lib, oracle_mod):
    w = workloads.custom("dense", 2, 1000, 1000, 1, 128)
    ins = workloads.make_inputs(w, seed_base=13500)
    q, k, v = (t.cuda() for t in ins)
    out = torch.full_like(q, float("nan"))
    assert noalloc(cuda_lib, q, k, v, out) == cuda_lib.ATTN_OK
    torch.cuda.synchronize()
    ref = oracle_mod.dense_attention(*(workloads.bf16_bits(t) for t in ins))
    assert_parity(f64(out), ref, f"noalloc {w.describe()}")


def test_noalloc_after_timeout(cuda_lib, oracle_mod):
    """A launch that gives up (the loader of block 0 skips a value tile on
    purpose, so a bounded wait runs out) leaves some tail units' pieces
    counted in; the next call must still merge correctly."""
    w = workloads.custom("dense", 2, 1000, 1000, 1, 128)   # 16 tail CTAs of 4 key tiles
    ins = workloads.make_inputs(w, seed_base=13600)
    q, k, v = (t.cuda() for t in ins)
    good = torch.empty_like(q)
    assert noalloc(cuda_lib, q, k, v, good) == cuda_lib.ATTN_OK
    torch.cuda.synchronize()
    assert cuda_lib.device_status()[0] == cuda_lib.ATTN_OK
    cuda_lib.debug_set_fault(1, 50_000)
    try:
        bad = torch.empty_like(q)
        assert noalloc(cuda_lib, q, k, v, bad) == cuda_lib.ATTN_OK
        rc, _ = cuda_lib.device_status()
    finally:
        cuda_lib.debug_set_fault(0, 0)
    assert rc == cuda_lib.ATTN_ERR_TIMEOUT
    out = torch.full_like(q, float("nan"))
    assert noalloc(cuda_lib, q, k, v, out) == cuda_lib.ATTN_OK
    torch.cuda.synchronize()
    assert cuda_lib.device_status()[0] == cuda_lib.ATTN_OK
    assert torch.equal(out, good)
    ref = oracle_mod.dense_attention(*(workloads.bf16_bits(t) for t in ins))
    assert_parity(f64(out), ref, "noalloc after a timeout")


def test_noalloc_rejects_like_dense(cuda_lib):
    lib = cuda_lib.load_library()
    a, b, c, o = 0x10000000, 0x20000000, 0x30000000, 0x40000000
    assert lib.attn_dense_fwd_noalloc(a, b, c, o, 1, 128, 32, 96, None) == cuda_lib.ATTN_ERR_HEADDIM
    assert lib.attn_dense_fwd_noalloc(a, None, c, o, 1, 128, 32, 64, None) == cuda_lib.ATTN_ERR_NULL
    assert lib.attn_dense_fwd_noalloc(a, b, c, a, 1, 128, 32, 64, None) == cuda_lib.ATTN_ERR_ALIAS
