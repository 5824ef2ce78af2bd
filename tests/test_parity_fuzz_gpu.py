"""Seeded random shapes through every entry point, sized to have a little more
work than one round of CTAs so that the last round is split in varied ways
(pieces of one or two key tiles, several pieces per CTA, prefix and current
segments, ragged query pairs).  Every row of every split unit, plus a random
spread of other rows, is compared with the FP64 oracle."""
import numpy as np
import pytest
import torch

import workloads
from parity import assert_parity

pytestmark = pytest.mark.gpu

KINDS = ("dense", "cross", "prefix", "block_causal", "masked_prefix")


def draw_case(seed, sms):
    """A shape whose units slightly exceed a multiple of the SM count."""
    rng = np.random.default_rng(seed)
    kind = KINDS[seed % len(KINDS)]
    D = int(rng.choice([64, 128]))
    B = int(rng.integers(1, 3))
    Nq = int(rng.integers(129, 1400))
    q_pairs = -(-Nq // 256)
    # H so that B * H * q_pairs lands just past a multiple of the SM count
    target = sms * int(rng.integers(1, 3)) + int(rng.integers(1, 40))
    H = max(1, target // (B * q_pairs))
    Np = int(rng.integers(1, 700)) if kind in ("prefix", "masked_prefix") else 0
    Nk = int(rng.integers(1, 3000)) if kind == "cross" else Nq
    segs = ()
    if kind in ("block_causal", "masked_prefix"):
        n, pos, segs = Np + Nq, 0, []
        while pos < n:
            L = min(int(rng.integers(1, 500)), n - pos)
            segs.append((int(rng.integers(-1, 3)) if rng.random() < 0.6 else -1, L))
            pos += L
        segs = tuple(segs)
    return kind, B, Nq, Np, Nk, H, D, segs


@pytest.mark.parametrize("seed", range(10))
def test_fuzz_split_tails(cuda_lib, oracle_mod, seed):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    kind, B, Nq, Np, Nk, H, D, segs = draw_case(7000 + seed, sms)
    masked = kind in ("block_causal", "masked_prefix")
    ids = (torch.cat([torch.full((n,), k, dtype=torch.int32) for k, n in segs])
           if segs else None)
    T = -(-Np // 128) + -(-Nk // 128)
    sched, _, _ = cuda_lib.debug_schedule(B, Nq, H, T, sms, masked,
                                          ids.numpy() if masked else None, Np)
    units = {(int(r[2]), int(r[3]), int(r[4])) for r in sched if r[8] >= 0}
    rng = np.random.default_rng(seed)
    rows = [(b * Nq + q) * H + h for b, h, q0 in units for q in range(q0, min(q0 + 256, Nq))]
    rows += rng.integers(0, B * Nq * H, size=200).tolist()
    rows = np.unique(np.array(rows, dtype=np.int64))

    base = 30000 + 10 * seed
    if kind in ("dense", "cross"):
        q, k, v = (workloads.randn_bf16(s, 1.0, base + i) for i, s in
                   enumerate([(B, Nq, H, D), (B, Nk, H, D), (B, Nk, H, D)]))
        out = torch.empty(B, Nq, H, D, dtype=torch.bfloat16, device="cuda")
        if kind == "dense":
            cuda_lib.attn_dense_fwd(q.cuda(), k.cuda(), v.cuda(), out)
        else:
            cuda_lib.attn_dense_cross_fwd(q.cuda(), k.cuda(), v.cuda(), out)
        ref = oracle_mod.dense_attention_rows(*(workloads.bf16_bits(t) for t in (q, k, v)), rows)
    elif kind == "prefix":
        shapes = [(B, Nq, H, D), (B, Np, H, D), (B, Np, H, D), (B, Nk, H, D), (B, Nk, H, D)]
        q, kp, vp, kc, vc = (workloads.randn_bf16(s, 1.0, base + i) for i, s in enumerate(shapes))
        out = torch.empty(B, Nq, H, D, dtype=torch.bfloat16, device="cuda")
        cuda_lib.attn_prefix_fwd(*(t.cuda() for t in (q, kp, vp, kc, vc)), out)
        ref = oracle_mod.prefix_attention_rows(
            *(workloads.bf16_bits(t) for t in (q, kp, vp, kc, vc)), rows)
    elif kind == "block_causal":
        q, k, v = (workloads.randn_bf16((B, Nq, H, D), 1.0, base + i) for i in range(3))
        out = torch.empty(B, Nq, H, D, dtype=torch.bfloat16, device="cuda")
        cuda_lib.attn_block_causal_fwd(q.cuda(), k.cuda(), v.cuda(), ids.cuda(), out)
        ref = oracle_mod.block_causal_attention_rows(
            *(workloads.bf16_bits(t) for t in (q, k, v)), ids.numpy(), rows)
    else:
        shapes = [(B, Nq, H, D)] * 3 + [(B, Np, H, D)] * 2
        q, kc, vc, kp, vp = (workloads.randn_bf16(s, 1.0, base + i) for i, s in enumerate(shapes))
        valid = torch.rand((B, Np + Nq), generator=torch.Generator().manual_seed(base)) >= 0.1
        valid[:, 0] = True  # every query sees key 0
        out = torch.empty(B, Nq, H, D, dtype=torch.bfloat16, device="cuda")
        cuda_lib.attn_masked_prefix_fwd(*(t.cuda() for t in (q, kc, vc, kp, vp)), ids.cuda(),
                                        valid.cuda(), 0.1, out)
        ref = oracle_mod.masked_prefix_attention_rows(
            *(workloads.bf16_bits(t) for t in (q, kc, vc, kp, vp)), ids.numpy(),
            valid.numpy(), 0.1, rows)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().astype(np.float64).reshape(-1, D)[rows]
    assert_parity(got, ref, f"{kind} B={B} Nq={Nq} Np={Np} Nk={Nk} H={H} D={D} "
                            f"({len(units)} split units)")
