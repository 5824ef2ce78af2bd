"""attn_dense_fwd_noalloc: dense attention for callers that cannot allocate
device memory (an engine whose pool owns the GPU memory, a plugin given only
its buffers, a loop that cannot pay for cudaMalloc's synchronisation).

It runs the same kernel and schedule as attn_dense_fwd, with the split
workspace in the library's static device scratch instead of a cudaMalloc'd
buffer.  Each case calls it twice in a row through the C ABI and compares both
outputs with attn_dense_fwd's under the parity tolerance of the other tests.
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


@pytest.mark.parametrize("B,N,H,D", CASES)
def test_noalloc_matches_dense_twice(cuda_lib, B, N, H, D):
    w = workloads.custom("dense", B, N, N, H, D)
    q, k, v = (t.cuda() for t in workloads.make_inputs(w, seed_base=13000 + N + D))
    ref = torch.empty_like(q)
    cuda_lib.attn_dense_fwd(q, k, v, ref)
    lib = cuda_lib.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    outs = []
    for _ in range(2):
        out = torch.full_like(q, float("nan"))
        rc = lib.attn_dense_fwd_noalloc(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
                                        ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                        B, N, H, D, ctypes.c_void_p(stream))
        assert rc == cuda_lib.ATTN_OK, cuda_lib.status_string(rc)
        outs.append(out)
    torch.cuda.synchronize()
    assert cuda_lib.device_status()[0] == cuda_lib.ATTN_OK
    expected = ref.float().cpu().numpy().astype(np.float64)
    for out in outs:
        assert_parity(out.float().cpu().numpy().astype(np.float64), expected, f"noalloc {w.describe()}")
    assert torch.equal(outs[0], outs[1])


def test_noalloc_rejects_like_dense(cuda_lib):
    lib = cuda_lib.load_library()
    a, b, c, o = 0x10000000, 0x20000000, 0x30000000, 0x40000000
    assert lib.attn_dense_fwd_noalloc(a, b, c, o, 1, 128, 32, 96, None) == cuda_lib.ATTN_ERR_HEADDIM
    assert lib.attn_dense_fwd_noalloc(a, None, c, o, 1, 128, 32, 64, None) == cuda_lib.ATTN_ERR_NULL
    assert lib.attn_dense_fwd_noalloc(a, b, c, a, 1, 128, 32, 64, None) == cuda_lib.ATTN_ERR_ALIAS
