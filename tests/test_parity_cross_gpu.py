"""GPU parity of dense cross attention (Nq != Nk; the dense definitions'
"cross attention allows unequal lengths") against the FP64 oracle, through the
C ABI.  Short-query, long-context shapes have fewer work units than SMs, so
their keys are cut into pieces on separate SMs and merged (split-KV)."""
import numpy as np
import pytest
import torch

import workloads
from parity import assert_parity

pytestmark = pytest.mark.gpu

CASES = [  # (B, Nq, Nk, H, D)
    (1, 300, 1, 2, 128), (1, 1, 700, 2, 64), (2, 1000, 130, 2, 128),
    (1, 129, 4000, 3, 128), (1, 4096, 256, 2, 64), (2, 64, 9000, 1, 64),
]


def run(ncp, w, seed):
    ins = workloads.make_inputs(w, seed_base=seed)
    q, k, v = (t.cuda() for t in ins)
    out = torch.empty_like(q)
    ncp.attn_dense_cross_fwd(q, k, v, out)
    torch.cuda.synchronize()
    return ins, out


def f64(t):
    return t.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("B,Nq,Nk,H,D", CASES)
def test_cross_small(cuda_lib, oracle_mod, B, Nq, Nk, H, D):
    w = workloads.custom("cross", B, Nq, Nk, H, D)
    ins, out = run(cuda_lib, w, 14000 + Nq + Nk)
    ref = oracle_mod.dense_attention(*(workloads.bf16_bits(t) for t in ins))
    assert_parity(f64(out), ref, w.describe())


@pytest.mark.parametrize("cid", [7, 8])
def test_cross_workloads(cuda_lib, oracle_mod, cid):
    w = workloads.WORKLOADS[cid]
    ins, out = run(cuda_lib, w, None)
    ref = oracle_mod.dense_attention(*(workloads.bf16_bits(t) for t in ins))
    s = assert_parity(f64(out), ref, w.describe())
    print(w.name, s)


def test_cross_with_equal_lengths_is_the_dense_entry(cuda_lib):
    w = workloads.custom("dense", 1, 777, 777, 3, 128)
    q, k, v = (t.cuda() for t in workloads.make_inputs(w, seed_base=14900))
    a, b = torch.empty_like(q), torch.empty_like(q)
    cuda_lib.attn_dense_fwd(q, k, v, a)
    cuda_lib.attn_dense_cross_fwd(q, k, v, b)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
