"""D = 128 cross and prefix-cached attention on ragged shapes against the FP64
oracle: lengths in Nq, Nk, Np and Nc that end inside a tile, single-tile
units, units whose second query tile holds only padding rows, split tails
(fewer units than SMs) and prefix segments that end inside a tile."""
import numpy as np
import pytest
import torch

import workloads
from parity import assert_parity

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


def f64(t):
    return t.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("B,Nq,Nk,H", DENSE)
def test_cross_ragged(cuda_lib, oracle_mod, B, Nq, Nk, H):
    shapes = [(B, Nq, H, 128), (B, Nk, H, 128), (B, Nk, H, 128)]
    ins = [workloads.randn_bf16(s, 1.0, 15000 + 7 * Nq + Nk + i) for i, s in enumerate(shapes)]
    q, k, v = (t.cuda() for t in ins)
    ref = oracle_mod.dense_attention(*(workloads.bf16_bits(t) for t in ins))
    out = torch.full_like(q, float("nan"))
    cuda_lib.attn_dense_cross_fwd(q, k, v, out)
    torch.cuda.synchronize()
    assert cuda_lib.device_status()[0] == cuda_lib.ATTN_OK
    assert_parity(f64(out), ref, f"cross B={B} Nq={Nq} Nk={Nk} H={H}")


@pytest.mark.parametrize("B,Nq,Np,Nc,H", PREFIX)
def test_prefix_ragged(cuda_lib, oracle_mod, B, Nq, Np, Nc, H):
    shapes = [(B, Nq, H, 128), (B, Np, H, 128), (B, Np, H, 128), (B, Nc, H, 128), (B, Nc, H, 128)]
    ins = [workloads.randn_bf16(s, 1.0, 16000 + Nq + 3 * Np + i) for i, s in enumerate(shapes)]
    dev = [t.cuda() for t in ins]
    ref = oracle_mod.prefix_attention(*(workloads.bf16_bits(t) for t in ins))
    out = torch.full_like(dev[0], float("nan"))
    cuda_lib.attn_prefix_fwd(*dev, out)
    torch.cuda.synchronize()
    assert cuda_lib.device_status()[0] == cuda_lib.ATTN_OK
    assert_parity(f64(out), ref, f"prefix B={B} Nq={Nq} Np={Np} Nc={Nc} H={H}")
