"""Key sequences past the largest workload: dense attention over ~100 000
tokens and a prefix of ~70 000 tokens, both ragged (the last key tile of each
segment is partial, so every prefix row crosses a partial tile between the
segments), against the FP64 oracle on sampled rows (tile edges, the ragged end
and a seeded random spread)."""
import numpy as np
import pytest
import torch

import workloads
from parity import assert_parity, sample_rows

pytestmark = pytest.mark.gpu


def f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def test_dense_very_long_sampled(cuda_lib, oracle_mod):
    B, N, H, D = 1, 100003, 2, 128
    w = workloads.custom("dense", B, N, N, H, D)
    q, k, v = (workloads.randn_bf16((B, N, H, D), 1.0, 17000 + i) for i in range(3))
    out = torch.empty((B, N, H, D), dtype=torch.bfloat16, device="cuda")
    cuda_lib.attn_dense_fwd(q.cuda(), k.cuda(), v.cuda(), out)
    torch.cuda.synchronize()
    rows = sample_rows(B, N, H, n_random=60, seed=17)
    got = f64(out).reshape(-1, D)[rows]
    b = workloads.bf16_bits
    ref = oracle_mod.dense_attention_rows(b(q), b(k), b(v), rows)
    s = assert_parity(got, ref, w.describe())
    print(w.name, s)


def test_prefix_very_long_sampled(cuda_lib, oracle_mod):
    B, Nq, Np, Nc, H, D = 1, 3001, 70001, 3001, 2, 64
    w = workloads.custom("prefix", B, Nq, Nc, H, D, Np=Np)
    shapes = [(B, Nq, H, D), (B, Np, H, D), (B, Np, H, D), (B, Nc, H, D), (B, Nc, H, D)]
    q, kp, vp, kc, vc = (workloads.randn_bf16(s, 1.0, 17100 + i) for i, s in enumerate(shapes))
    out = torch.empty((B, Nq, H, D), dtype=torch.bfloat16, device="cuda")
    cuda_lib.attn_prefix_fwd(q.cuda(), kp.cuda(), vp.cuda(), kc.cuda(), vc.cuda(), out)
    torch.cuda.synchronize()
    rows = sample_rows(B, Nq, H, n_random=60, seed=18)
    got = f64(out).reshape(-1, D)[rows]
    b = workloads.bf16_bits
    ref = oracle_mod.prefix_attention_rows(b(q), b(kp), b(vp), b(kc), b(vc), rows)
    s = assert_parity(got, ref, w.describe())
    print(w.name, s)
