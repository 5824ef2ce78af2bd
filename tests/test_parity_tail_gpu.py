"""GPU parity of split tails on small, ragged shapes: each case has a few more
work units than SMs, so its last units are cut into key-range pieces (dense
forms: weighted ranges chosen on the host; masked forms: ranges of visited
key tiles chosen in the kernel) and merged through the workspace.  The
launch's schedule comes from the library's host hook; every row of every
tail unit, and of one whole unit, is compared with the FP64 oracle."""
import numpy as np
import pytest
import torch

import workloads
from parity import assert_parity

pytestmark = pytest.mark.gpu

# kind, B, Nq, Np (prefix keys), Nk (current keys; masked forms: Nq), H, D, segments
CASES = [
    ("dense", 1, 1280, 0, 1280, 31, 128, ()),
    ("dense", 2, 1000, 0, 1000, 39, 64, ()),
    ("prefix", 1, 700, 300, 700, 53, 128, ()),
    ("cross", 1, 300, 0, 3000, 81, 128, ()),
    ("block_causal", 1, 2000, 0, 2000, 20, 64, ((-1, 100), (2, 1900))),
    ("block_causal", 2, 1200, 0, 1200, 21, 128, ((-1, 240), (0, 600), (-1, 13), (1, 347))),
    ("masked_prefix", 2, 600, 200, 600, 26, 128, ((-1, 120), (3, 80), (-1, 100), (4, 500))),
]


def ptr_rows(rows_sched, B, Nq, H):
    """Flat output rows (b*Nq + q)*H + h of the units in `rows_sched`."""
    out = []
    for b, h, q0 in rows_sched:
        for q in range(q0, min(q0 + 256, Nq)):
            out.append((b * Nq + q) * H + h)
    return np.array(sorted(set(out)), dtype=np.int64)


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-{c[5]}h" for c in CASES])
def test_split_tail_rows(cuda_lib, oracle_mod, case):
    kind, B, Nq, Np, Nk, H, D, segs = case
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    q_pairs = -(-Nq // 256)
    masked = kind in ("block_causal", "masked_prefix")
    ids = (torch.cat([torch.full((n,), k, dtype=torch.int32) for k, n in segs])
           if segs else None)
    T = -(-Np // 128) + -(-Nk // 128)
    sched, grid, _ = cuda_lib.debug_schedule(B, Nq, H, T, sms, masked,
                                             ids.numpy() if masked else None, Np)
    tail = sched[sched[:, 8] >= 0]
    if B * H * q_pairs <= sms or len(tail) == 0:
        pytest.skip(f"no split tail with {sms} SMs")
    units = {(int(r[2]), int(r[3]), int(r[4])) for r in tail}
    whole = sched[sched[:, 8] < 0][0]
    units.add((int(whole[2]), int(whole[3]), int(whole[4])))
    rows = ptr_rows(units, B, Nq, H)

    seed = 19000 + 10 * CASES.index(case)
    if kind in ("dense", "cross"):
        q, k, v = (workloads.randn_bf16(s, 1.0, seed + i) for i, s in
                   enumerate([(B, Nq, H, D), (B, Nk, H, D), (B, Nk, H, D)]))
        out = torch.empty(B, Nq, H, D, dtype=torch.bfloat16, device="cuda")
        if kind == "dense":
            cuda_lib.attn_dense_fwd(q.cuda(), k.cuda(), v.cuda(), out)
        else:
            cuda_lib.attn_dense_cross_fwd(q.cuda(), k.cuda(), v.cuda(), out)
        ref = oracle_mod.dense_attention_rows(*(workloads.bf16_bits(t) for t in (q, k, v)), rows)
    elif kind == "prefix":
        shapes = [(B, Nq, H, D), (B, Np, H, D), (B, Np, H, D), (B, Nk, H, D), (B, Nk, H, D)]
        q, kp, vp, kc, vc = (workloads.randn_bf16(s, 1.0, seed + i) for i, s in enumerate(shapes))
        out = torch.empty(B, Nq, H, D, dtype=torch.bfloat16, device="cuda")
        cuda_lib.attn_prefix_fwd(*(t.cuda() for t in (q, kp, vp, kc, vc)), out)
        ref = oracle_mod.prefix_attention_rows(
            *(workloads.bf16_bits(t) for t in (q, kp, vp, kc, vc)), rows)
    elif kind == "block_causal":
        q, k, v = (workloads.randn_bf16((B, Nq, H, D), 1.0, seed + i) for i in range(3))
        out = torch.empty(B, Nq, H, D, dtype=torch.bfloat16, device="cuda")
        cuda_lib.attn_block_causal_fwd(q.cuda(), k.cuda(), v.cuda(), ids.cuda(), out)
        ref = oracle_mod.block_causal_attention_rows(
            *(workloads.bf16_bits(t) for t in (q, k, v)), ids.numpy(), rows)
    else:
        shapes = [(B, Nq, H, D)] * 3 + [(B, Np, H, D)] * 2
        q, kc, vc, kp, vp = (workloads.randn_bf16(s, 1.0, seed + i) for i, s in enumerate(shapes))
        valid = torch.ones((B, Np + Nq), dtype=torch.bool)
        valid[1, 50:90] = False
        out = torch.empty(B, Nq, H, D, dtype=torch.bfloat16, device="cuda")
        cuda_lib.attn_masked_prefix_fwd(*(t.cuda() for t in (q, kc, vc, kp, vp)), ids.cuda(),
                                        valid.cuda(), 0.09, out)
        ref = oracle_mod.masked_prefix_attention_rows(
            *(workloads.bf16_bits(t) for t in (q, kc, vc, kp, vp)), ids.numpy(),
            valid.numpy(), 0.09, rows)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().astype(np.float64).reshape(-1, D)[rows]
    assert_parity(got, ref, f"{kind} B={B} Nq={Nq} Np={Np} Nk={Nk} H={H} D={D} (split tail rows)")


def test_masked_split_tail_deterministic_and_per_stream(cuda_lib):
    """A block-causal call whose tail is split: repeated calls are
    bit-identical, and calls on two streams at once (separate workspaces)
    agree with them."""
    B, N, H, D = 1, 2000, 20, 64
    segs = ((-1, 100), (2, 1900))
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    ids = torch.cat([torch.full((n,), k, dtype=torch.int32) for k, n in segs])
    sched, _, _ = cuda_lib.debug_schedule(B, N, H, 0, sms, True, ids.numpy(), 0)
    if not (sched[:, 8] >= 0).any():
        pytest.skip(f"no split tail with {sms} SMs")
    q, k, v = (workloads.randn_bf16((B, N, H, D), 1.0, 19500 + i).cuda() for i in range(3))
    dids = ids.cuda()
    first = torch.empty_like(q)
    cuda_lib.attn_block_causal_fwd(q, k, v, dids, first)
    torch.cuda.synchronize()
    for _ in range(3):
        again = torch.empty_like(q)
        cuda_lib.attn_block_causal_fwd(q, k, v, dids, again)
        torch.cuda.synchronize()
        assert torch.equal(again, first)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [torch.empty_like(q) for _ in streams]
    for _ in range(4):
        for s, o in zip(streams, outs):
            cuda_lib.attn_block_causal_fwd(q, k, v, dids, o, stream=s)
    torch.cuda.synchronize()
    for o in outs:
        assert torch.equal(o, first)
