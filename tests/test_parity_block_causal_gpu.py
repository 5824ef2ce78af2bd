"""GPU parity of the block-causal form (definition prefix_cached_block_causal_
h32_d128_prefix0) against the FP64 oracle, through the C ABI.

The id layouts cover text only (pure causal), one image (dense), text and
image runs that start and end inside 128-token tiles, an id reused by two
separate blocks (outside the definition's contiguity promise: the kernel is
exact for any ids), single tokens and a one-token sequence.
"""
import dataclasses

import numpy as np
import pytest
import torch

import workloads
from parity import assert_parity, sample_rows

pytestmark = pytest.mark.gpu

CASES = [  # (B, H, D, segments)
    (1, 2, 128, ((-1, 300),)),
    (1, 2, 64, ((7, 260),)),
    (2, 2, 128, ((-1, 100), (0, 150), (-1, 30), (1, 200))),
    (1, 3, 64, ((-1, 120), (5, 20), (-1, 3), (2, 300), (-1, 1))),
    (1, 2, 128, ((0, 100), (-1, 50), (0, 100), (-1, 10))),
    (1, 1, 128, ((-1, 1),)),
    (1, 2, 128, ((3, 1), (-1, 128), (4, 129))),
    (2, 1, 64, ((-1, 513), (9, 640), (-1, 7))),
]


def run(ncp, w, seed):
    ins = workloads.make_inputs(w, seed_base=seed)
    ids = workloads.image_ids(w)
    q, k, v = (t.cuda() for t in ins)
    out = torch.empty_like(q)
    ncp.attn_block_causal_fwd(q, k, v, ids.cuda(), out)
    torch.cuda.synchronize()
    return ins, ids, out


def bits(ts):
    return [workloads.bf16_bits(t) for t in ts]


@pytest.mark.parametrize("case", CASES)
def test_block_causal_small(cuda_lib, oracle_mod, case):
    B, H, D, segs = case
    N = sum(n for _, n in segs)
    w = workloads.custom("block_causal", B, N, N, H, D, segments=segs)
    ins, ids, out = run(cuda_lib, w, 12000 + N + D)
    ref = oracle_mod.block_causal_attention(*bits(ins), ids.numpy())
    assert_parity(out.float().cpu().numpy().astype(np.float64), ref, w.describe())


def test_block_causal_workload(cuda_lib, oracle_mod):
    w = workloads.WORKLOADS[6]
    ins, ids, out = run(cuda_lib, w, None)
    ref = oracle_mod.block_causal_attention(*bits(ins), ids.numpy())
    s = assert_parity(out.float().cpu().numpy().astype(np.float64), ref, w.describe())
    print(w.name, s)


def test_block_causal_workload_d64(cuda_lib, oracle_mod):
    """The workload's ids at D = 64, where P has TMEM columns of its own and
    the next S goes out ahead of the P V: 32 heads give each CTA several work
    items and a split tail, so the per-tile barrier phases carry across items."""
    w6 = workloads.WORKLOADS[6]
    w = dataclasses.replace(w6, D=64, name=w6.name.replace("d128", "d64"))
    ins, ids, out = run(cuda_lib, w, 12900)
    ref = oracle_mod.block_causal_attention(*bits(ins), ids.numpy())
    s = assert_parity(out.float().cpu().numpy().astype(np.float64), ref, w.describe())
    print(w.name, s)


def test_block_causal_text_only_matches_prefix_dense(cuda_lib):
    """Text only: row i is dense attention over keys 0..i; the first rows are
    checked against the dense entry on the truncated keys."""
    w = workloads.custom("block_causal", 1, 256, 256, 2, 128, segments=((-1, 256),))
    ins, _, out = run(cuda_lib, w, 12500)
    q, k, v = (t.cuda() for t in ins)
    for i in (0, 1, 127, 128, 255):
        o = torch.empty_like(q[:, i:i + 1])
        cuda_lib.attn_prefix_fwd(q[:, i:i + 1].contiguous(), None, None,
                                 k[:, :i + 1].contiguous(), v[:, :i + 1].contiguous(), o)
        torch.cuda.synchronize()
        assert (o.float() - out[:, i:i + 1].float()).abs().max().item() < 2e-2


def test_block_causal_rejects(cuda_lib):
    q = torch.zeros(1, 128, 2, 128, device="cuda", dtype=torch.bfloat16)
    ids = torch.zeros(128, device="cuda", dtype=torch.int32)
    with pytest.raises(ValueError):
        cuda_lib.attn_block_causal_fwd(q, q, q, ids.long(), torch.empty_like(q))
    with pytest.raises(ValueError):
        cuda_lib.attn_block_causal_fwd(q, q, q, ids[:64], torch.empty_like(q))
    lib = cuda_lib.load_library()
    big = 131072 + 1
    assert lib.attn_block_causal_fwd(q.data_ptr(), q.data_ptr(), q.data_ptr(), ids.data_ptr(),
                                     torch.empty_like(q).data_ptr(), 1, big, 2, 128,
                                     None) == cuda_lib.ATTN_ERR_SHAPE
    assert lib.attn_block_causal_fwd(q.data_ptr(), q.data_ptr(), q.data_ptr(),
                                     ids.data_ptr() + 4, torch.empty_like(q).data_ptr(), 1, 128, 2,
                                     128, None) == cuda_lib.ATTN_ERR_ALIGN
