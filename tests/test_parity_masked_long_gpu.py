"""Long masked-form calls (block-causal over 16 384 tokens, masked prefix with
a 4 000-token prefix): many key tiles per unit, units of very unequal work
handed out longest first.  Compared with the FP64 oracle on sampled rows
(tile edges, block boundaries and a seeded random spread)."""
import numpy as np
import pytest
import torch

import workloads
from parity import assert_parity

pytestmark = pytest.mark.gpu


def boundary_rows(B, Nq, H, edges, n_random, seed):
    rng = np.random.default_rng(seed)
    qs = set()
    for e in edges:
        qs.update(q for q in (e - 129, e - 128, e - 1, e, e + 1, e + 127, e + 128) if 0 <= q < Nq)
    qs.update((0, 1, Nq - 1))
    rows = [(b * Nq + q) * H + h for b in range(B) for h in sorted({0, H - 1}) for q in sorted(qs)]
    rows += list(rng.integers(0, B * Nq * H, size=n_random))
    return np.unique(np.array(rows, dtype=np.int64))


def test_block_causal_long_sampled(cuda_lib, oracle_mod):
    segs = ((-1, 1000), (0, 6000), (-1, 77), (1, 9307))
    N = sum(n for _, n in segs)
    w = workloads.custom("block_causal", 1, N, N, 8, 128, segments=segs)
    ins = workloads.make_inputs(w, seed_base=16000)
    ids = workloads.image_ids(w)
    q, k, v = (t.cuda() for t in ins)
    out = torch.empty_like(q)
    cuda_lib.attn_block_causal_fwd(q, k, v, ids.cuda(), out)
    torch.cuda.synchronize()
    edges = np.cumsum([n for _, n in segs])[:-1].tolist()
    rows = boundary_rows(1, N, 8, edges, 300, 1)
    got = out.float().cpu().numpy().astype(np.float64).reshape(-1, 128)[rows]
    ref = oracle_mod.block_causal_attention_rows(*(workloads.bf16_bits(t) for t in ins),
                                                 ids.numpy(), rows)
    assert_parity(got, ref, w.describe())


def test_masked_prefix_long_sampled(cuda_lib, oracle_mod):
    B, Nq, Np, H, D = 2, 6000, 4000, 4, 64
    segs = ((-1, 700), (0, 3300), (1, 6000))
    shapes = [(B, Nq, H, D)] * 3 + [(B, Np, H, D)] * 2
    q, kc, vc, kp, vp = (workloads.randn_bf16(s, 1.0, 16100 + i) for i, s in enumerate(shapes))
    ids = torch.cat([torch.full((n,), k, dtype=torch.int32) for k, n in segs])
    valid = torch.ones((B, Np + Nq), dtype=torch.bool)
    valid[0, 600:700] = False
    valid[1, 3000:3500] = False
    d = [t.cuda() for t in (q, kc, vc, kp, vp)]
    out = torch.empty_like(d[0])
    cuda_lib.attn_masked_prefix_fwd(d[0], d[1], d[2], d[3], d[4], ids.cuda(), valid.cuda(), 0.11,
                                    out)
    torch.cuda.synchronize()
    rows = boundary_rows(B, Nq, H, [0, 3000, 5999], 300, 2)
    got = out.float().cpu().numpy().astype(np.float64).reshape(-1, D)[rows]
    b = workloads.bf16_bits
    ref = oracle_mod.masked_prefix_attention_rows(b(q), b(kc), b(vc), b(kp), b(vp), ids.numpy(),
                                                  valid.numpy().astype(np.uint8),
                                                  float(np.float32(0.11)), rows)
    assert_parity(got, ref, "masked prefix long")


def test_block_causal_max_length_sampled(cuda_lib, oracle_mod):
    """The longest sequence the masked forms accept, 131 072 tokens (1 024 key
    tiles): the per-item key-tile masks use every word, and an image block
    runs over the last tile edges up to the end."""
    segs = ((-1, 60000), (3, 40000), (-1, 1000), (4, 30000), (-1, 5), (5, 67))
    N = sum(n for _, n in segs)
    assert N == 131072
    w = workloads.custom("block_causal", 1, N, N, 2, 128, segments=segs)
    ins = workloads.make_inputs(w, seed_base=16200)
    ids = workloads.image_ids(w)
    q, k, v = (t.cuda() for t in ins)
    out = torch.empty_like(q)
    cuda_lib.attn_block_causal_fwd(q, k, v, ids.cuda(), out)
    torch.cuda.synchronize()
    edges = np.cumsum([n for _, n in segs])[:-1].tolist() + [126976, 130944]
    rows = boundary_rows(1, N, 2, edges, 60, 3)
    got = out.float().cpu().numpy().astype(np.float64).reshape(-1, 128)[rows]
    ref = oracle_mod.block_causal_attention_rows(*(workloads.bf16_bits(t) for t in ins),
                                                 ids.numpy(), rows)
    assert_parity(got, ref, w.describe())


def test_masked_prefix_max_tiles_sampled(cuda_lib, oracle_mod):
    """Prefix and query tiles together at the limit of 1 024 key tiles, the
    prefix ending inside a tile, with invalid keys in both segments."""
    B, Nq, Np, H, D = 1, 126900, 4000, 2, 64
    assert (Np + 127) // 128 + (Nq + 127) // 128 == 1024
    segs = ((-1, 3000), (0, 2000), (-1, 90000), (1, 35900))
    shapes = [(B, Nq, H, D)] * 3 + [(B, Np, H, D)] * 2
    q, kc, vc, kp, vp = (workloads.randn_bf16(s, 1.0, 16300 + i) for i, s in enumerate(shapes))
    ids = torch.cat([torch.full((n,), k, dtype=torch.int32) for k, n in segs])
    assert ids.numel() == Np + Nq
    valid = torch.ones((B, Np + Nq), dtype=torch.bool)
    valid[0, 100:300] = False
    valid[0, 128000:128100] = False
    d = [t.cuda() for t in (q, kc, vc, kp, vp)]
    out = torch.empty_like(d[0])
    cuda_lib.attn_masked_prefix_fwd(d[0], d[1], d[2], d[3], d[4], ids.cuda(), valid.cuda(), 0.125,
                                    out)
    torch.cuda.synchronize()
    rows = boundary_rows(B, Nq, H, [0, 1000, 91000, 124000, Nq - 1], 60, 4)
    got = out.float().cpu().numpy().astype(np.float64).reshape(-1, D)[rows]
    b = workloads.bf16_bits
    ref = oracle_mod.masked_prefix_attention_rows(b(q), b(kc), b(vc), b(kp), b(vp), ids.numpy(),
                                                  valid.numpy().astype(np.uint8),
                                                  float(np.float32(0.125)), rows)
    assert_parity(got, ref, "masked prefix at 1024 key tiles")
