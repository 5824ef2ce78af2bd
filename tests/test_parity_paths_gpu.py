"""Both kernels on the same shapes: the CTA-pair kernel (units of 512 query
rows on SM pairs, D = 128, every key visible) and the single-CTA kernel,
forced through the library's path hook, each against the FP64 oracle.

Shapes span ragged lengths in N, Nq, Np and Nc, pair units whose odd CTA holds
only padding rows, single-tile units, split tails (fewer units than pairs) and
prefix segments that end inside a tile."""
import numpy as np
import pytest
import torch

import workloads
from parity import assert_parity, stats

pytestmark = pytest.mark.gpu

DENSE = [  # (B, Nq, Nk, H)
    (1, 1, 1, 1), (1, 2, 2, 1), (1, 128, 128, 2), (1, 129, 129, 2), (1, 256, 256, 1),
    (1, 257, 300, 2), (2, 300, 300, 2), (1, 511, 511, 1), (1, 512, 512, 1), (1, 513, 513, 3),
    (1, 1000, 1000, 2), (2, 1536, 700, 3), (1, 2048, 2048, 3), (1, 64, 3000, 2),
    (1, 4096, 4096, 2),
]
PREFIX = [  # (B, Nq, Np, Nc, H)
    (1, 128, 1, 128, 2), (1, 300, 129, 300, 1), (2, 200, 128, 200, 2), (1, 64, 1024, 64, 2),
    (1, 700, 300, 500, 2), (1, 1024, 640, 1024, 2), (2, 1, 1, 1, 3),
]


@pytest.fixture
def path(cuda_lib):
    yield cuda_lib.debug_set_path
    cuda_lib.debug_set_path(0)


def f64(t):
    return t.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("B,Nq,Nk,H", DENSE)
def test_dense_both_paths(cuda_lib, oracle_mod, path, B, Nq, Nk, H):
    shapes = [(B, Nq, H, 128), (B, Nk, H, 128), (B, Nk, H, 128)]
    ins = [workloads.randn_bf16(s, 1.0, 15000 + 7 * Nq + Nk + i) for i, s in enumerate(shapes)]
    q, k, v = (t.cuda() for t in ins)
    ref = oracle_mod.dense_attention(*(workloads.bf16_bits(t) for t in ins))
    outs = {}
    for mode in (1, 2):
        path(mode)
        out = torch.full_like(q, float("nan"))
        cuda_lib.attn_dense_cross_fwd(q, k, v, out)
        torch.cuda.synchronize()
        assert cuda_lib.device_status()[0] == cuda_lib.ATTN_OK
        outs[mode] = f64(out)
        assert_parity(outs[mode], ref, f"path {mode} dense B={B} Nq={Nq} Nk={Nk} H={H}")
    s = stats(outs[2], outs[1])
    assert s["max_abs_err"] < 2e-2, s


@pytest.mark.parametrize("B,Nq,Np,Nc,H", PREFIX)
def test_prefix_both_paths(cuda_lib, oracle_mod, path, B, Nq, Np, Nc, H):
    shapes = [(B, Nq, H, 128), (B, Np, H, 128), (B, Np, H, 128), (B, Nc, H, 128), (B, Nc, H, 128)]
    ins = [workloads.randn_bf16(s, 1.0, 16000 + Nq + 3 * Np + i) for i, s in enumerate(shapes)]
    dev = [t.cuda() for t in ins]
    ref = oracle_mod.prefix_attention(*(workloads.bf16_bits(t) for t in ins))
    for mode in (1, 2):
        path(mode)
        out = torch.full_like(dev[0], float("nan"))
        cuda_lib.attn_prefix_fwd(*dev, out)
        torch.cuda.synchronize()
        assert cuda_lib.device_status()[0] == cuda_lib.ATTN_OK
        assert_parity(f64(out), ref, f"path {mode} prefix B={B} Nq={Nq} Np={Np} Nc={Nc} H={H}")


def test_pair_path_deterministic(cuda_lib, path):
    """The pair kernel's split tail merges in piece order: repeated calls are
    bit-identical."""
    path(2)
    w = workloads.custom("dense", 1, 2048, 2048, 3, 128)
    q, k, v = (t.cuda() for t in workloads.make_inputs(w, seed_base=16500))
    first = torch.empty_like(q)
    cuda_lib.attn_dense_fwd(q, k, v, first)
    for _ in range(3):
        out = torch.empty_like(q)
        cuda_lib.attn_dense_fwd(q, k, v, out)
        torch.cuda.synchronize()
        assert torch.equal(out, first)


def test_pair_path_timeout_recovers(cuda_lib, oracle_mod, path):
    """Bounded waits on the pair kernel: the even CTA of the first pair skips
    a value half on purpose, its wait runs out, both CTAs of every pair exit,
    and the next call on the same context is exact."""
    path(2)
    w = workloads.custom("dense", 1, 1024, 1024, 4, 128)
    ins = workloads.make_inputs(w, seed_base=16600)
    q, k, v = (t.cuda() for t in ins)
    good = torch.empty_like(q)
    cuda_lib.attn_dense_fwd(q, k, v, good)
    assert cuda_lib.device_status()[0] == cuda_lib.ATTN_OK
    cuda_lib.debug_set_fault(1, 50_000)
    try:
        cuda_lib.attn_dense_fwd(q, k, v, torch.empty_like(q))
        rc, info = cuda_lib.device_status()
    finally:
        cuda_lib.debug_set_fault(0, 0)
    assert rc == cuda_lib.ATTN_ERR_TIMEOUT and info & 0xff != 0
    out = torch.empty_like(q)
    cuda_lib.attn_dense_fwd(q, k, v, out)
    torch.cuda.synchronize()
    assert cuda_lib.device_status()[0] == cuda_lib.ATTN_OK
    assert torch.equal(out, good)
    assert_parity(f64(out), oracle_mod.dense_attention(*(workloads.bf16_bits(t) for t in ins)),
                  "pair path after a timeout")
