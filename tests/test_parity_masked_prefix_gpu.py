"""GPU parity of the masked prefix-cached form (the pre-audit definition
prefix_cached_block_causal_h32_d128: keys cat(prefix, current), query i at
position Np + i sees key j iff (j <= Np + i or the same image id >= 0) and
key_valid[b, j]; runtime sm_scale) against the FP64 oracle, through the C ABI.
Cases cover an empty prefix, prefixes whose length is not a multiple of 4
(unaligned id loads) or of 128 (tiles straddling the segment boundary),
per-batch key padding and D = 64."""
import dataclasses

import numpy as np
import pytest
import torch

import workloads
from parity import assert_parity

pytestmark = pytest.mark.gpu

CASES = [  # (B, Nq, Np, H, D, segments over Np + Nq, invalid fraction, sm_scale)
    (1, 200, 0, 2, 128, ((-1, 50), (0, 150)), 0.0, 128 ** -0.5),
    (2, 300, 300, 2, 128, ((-1, 120), (3, 180), (4, 300)), 0.1, 128 ** -0.5),
    (1, 129, 1, 2, 128, ((-1, 130),), 0.0, 0.1),
    (1, 257, 301, 3, 64, ((-1, 301), (9, 257)), 0.2, 0.125),
    (2, 100, 777, 1, 128, ((-1, 77), (1, 700), (2, 100)), 0.3, 0.05),
]


def make(B, Nq, Np, H, D, segs, frac, seed):
    shapes = [(B, Nq, H, D)] * 3 + [(B, Np, H, D)] * 2
    q, kc, vc, kp, vp = (workloads.randn_bf16(s, 1.0, seed + i) for i, s in enumerate(shapes))
    ids = torch.cat([torch.full((n,), k, dtype=torch.int32) for k, n in segs])
    g = torch.Generator().manual_seed(seed)
    valid = torch.rand((B, Np + Nq), generator=g) >= frac
    valid[:, 0] = True   # every query sees key 0 (the definition requires a visible key)
    return q, kc, vc, kp, vp, ids, valid


def gpu(ncp, q, kc, vc, kp, vp, ids, valid, scale):
    d = [t.cuda() for t in (q, kc, vc)]
    dkp, dvp = (kp.cuda(), vp.cuda()) if kp.shape[1] else (None, None)
    out = torch.empty_like(d[0])
    ncp.attn_masked_prefix_fwd(d[0], d[1], d[2], dkp, dvp, ids.cuda(), valid.cuda(), scale, out)
    torch.cuda.synchronize()
    return out


def oracle_of(o, q, kc, vc, kp, vp, ids, valid, scale):
    b = workloads.bf16_bits
    kp_, vp_ = (b(kp), b(vp)) if kp.shape[1] else (None, None)
    return o.masked_prefix_attention(b(q), b(kc), b(vc), kp_, vp_, ids.numpy(),
                                     valid.numpy().astype(np.uint8), scale)


@pytest.mark.parametrize("case", CASES)
def test_masked_prefix_small(cuda_lib, oracle_mod, case):
    B, Nq, Np, H, D, segs, frac, scale = case
    ins = make(B, Nq, Np, H, D, segs, frac, 15000 + Nq + Np)
    out = gpu(cuda_lib, *ins, scale)
    ref = oracle_of(oracle_mod, *ins, float(np.float32(scale)))
    assert_parity(out.float().cpu().numpy().astype(np.float64), ref, str(case[:5]))


def test_masked_prefix_workload(cuda_lib, oracle_mod):
    w = workloads.WORKLOADS[9]
    q, kc, vc, kp, vp = workloads.make_inputs(w)
    ids, valid = workloads.image_ids(w), workloads.key_valid(w)
    out = gpu(cuda_lib, q, kc, vc, kp, vp, ids, valid, w.sm_scale)
    ref = oracle_of(oracle_mod, q, kc, vc, kp, vp, ids, valid, float(np.float32(w.sm_scale)))
    s = assert_parity(out.float().cpu().numpy().astype(np.float64), ref, w.describe())
    print(w.name, s)


def test_masked_prefix_workload_d64(cuda_lib, oracle_mod):
    """The workload's prefix, ids and padding at D = 64 (scale 1/8), where P
    has TMEM columns of its own and the next S goes out ahead of the P V."""
    w9 = workloads.WORKLOADS[9]
    w = dataclasses.replace(w9, D=64, sm_scale=0.125, name=w9.name.replace("d128", "d64"))
    q, kc, vc, kp, vp = workloads.make_inputs(w, seed_base=15900)
    ids, valid = workloads.image_ids(w), workloads.key_valid(w)
    out = gpu(cuda_lib, q, kc, vc, kp, vp, ids, valid, w.sm_scale)
    ref = oracle_of(oracle_mod, q, kc, vc, kp, vp, ids, valid, float(np.float32(w.sm_scale)))
    s = assert_parity(out.float().cpu().numpy().astype(np.float64), ref, w.describe())
    print(w.name, s)


def test_masked_prefix_without_prefix_or_padding_is_block_causal(cuda_lib):
    segs = ((-1, 90), (5, 300), (-1, 10))
    B, N, H, D = 1, 400, 2, 64
    q, kc, vc, kp, vp, ids, valid = make(B, N, 0, H, D, segs, 0.0, 15900)
    a = gpu(cuda_lib, q, kc, vc, kp, vp, ids, valid, 0.125)
    b = torch.empty_like(a)
    cuda_lib.attn_block_causal_fwd(q.cuda(), kc.cuda(), vc.cuda(), ids.cuda(), b)
    torch.cuda.synchronize()
    assert torch.equal(a, b)   # D = 64: sm_scale 1/8 is D^-0.5 exactly


def test_masked_prefix_rejects(cuda_lib):
    lib = cuda_lib.load_library()
    q = torch.zeros(1, 128, 2, 128, device="cuda", dtype=torch.bfloat16)
    ids = torch.zeros(128, device="cuda", dtype=torch.int32)
    out = torch.empty_like(q)
    P = lambda t: t.data_ptr()  # noqa: E731
    for scale, want in ((0.0, cuda_lib.ATTN_ERR_SHAPE), (float("nan"), cuda_lib.ATTN_ERR_SHAPE),
                        (-1.0, cuda_lib.ATTN_ERR_SHAPE)):
        assert lib.attn_masked_prefix_fwd(P(q), P(q), P(q), None, None, P(ids), None, scale,
                                          P(out), 1, 128, 0, 2, 128, None) == want
    assert lib.attn_masked_prefix_fwd(P(q), P(q), P(q), None, None, P(ids) + 4, None, 0.1,
                                      P(out), 1, 128, 0, 2, 128, None) == cuda_lib.ATTN_ERR_ALIGN
    assert lib.attn_masked_prefix_fwd(P(q), P(q), P(q), None, None, None, None, 0.1,
                                      P(out), 1, 128, 0, 2, 128, None) == cuda_lib.ATTN_ERR_NULL
