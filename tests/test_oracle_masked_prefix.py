"""Pins of the FP64 oracle for the masked prefix-cached form (the definition
prefix_cached_block_causal_h32_d128 as it stood before the audit, field
"reference"): keys cat(K_prefix, K_current), query i at position Np + i sees
key j iff (j <= Np + i, or both carry the same image id >= 0) and
key_valid[b, j]; runtime sm_scale.

The pins: a pure-Python brute force of that rule on tiny mixed inputs; the
empty-prefix, all-valid case equals the block-causal oracle (pinned on its
own); text only is dense attention over cat(prefix, current[:i+1]); masking a
prefix key with key_valid equals deleting it; doubling Q while halving
sm_scale changes nothing; a row with no visible key is an error.  Each C
mutant in MUTANTS fails at least one pin.
"""
import math

import numpy as np
import pytest
import torch

import workloads


def rnd(shape, seed, sigma=1.0):
    return workloads.bf16_bits(workloads.randn_bf16(shape, sigma, seed))


def f(x):
    return torch.from_numpy(x.astype(np.uint16).view(np.int16)).view(torch.bfloat16).double().numpy()


def brute(Q, Kc, Vc, Kp, Vp, ids, valid, scale):
    q, kc, vc = f(Q), f(Kc), f(Vc)
    B, Nq, H, D = q.shape
    Np = Kp.shape[1]
    k = np.concatenate([f(Kp), kc], 1)
    v = np.concatenate([f(Vp), vc], 1)
    out = np.zeros((B, Nq, H, D))
    for b in range(B):
        for h in range(H):
            for i in range(Nq):
                qp = Np + i
                vis = [j for j in range(Np + Nq)
                       if (j <= qp or (ids[qp] >= 0 and ids[j] == ids[qp])) and valid[b, j]]
                s = [math.fsum(q[b, i, h, d] * k[b, j, h, d] for d in range(D)) * scale for j in vis]
                mx = max(s)
                w = [math.exp(x - mx) for x in s]
                tot = math.fsum(w)
                for d in range(D):
                    out[b, i, h, d] = math.fsum(wj * v[b, j, h, d] for wj, j in zip(w, vis)) / tot
    return out


def inputs(B, Nq, Np, H, D, seed):
    return (rnd((B, Nq, H, D), seed), rnd((B, Nq, H, D), seed + 1), rnd((B, Nq, H, D), seed + 2),
            rnd((B, Np, H, D), seed + 3), rnd((B, Np, H, D), seed + 4))


def pin_brute_force(o):
    B, Nq, Np, H, D = 2, 6, 4, 2, 4
    Q, Kc, Vc, Kp, Vp = inputs(B, Nq, Np, H, D, 1)
    ids = np.array([-1, 3, 3, -1, 5, 5, 5, -1, 3, 3], dtype=np.int32)
    valid = np.random.default_rng(0).random((B, Np + Nq)) < 0.75
    valid[:, 0] = True
    got = o.masked_prefix_attention(Q, Kc, Vc, Kp, Vp, ids, valid, 0.4)
    want = brute(Q, Kc, Vc, Kp, Vp, ids, valid, float(np.float32(0.4)))
    assert np.allclose(got, want, rtol=1e-12, atol=1e-13)


def pin_empty_prefix_is_block_causal(o):
    B, Nq, H, D = 1, 40, 2, 64
    Q, Kc, Vc, Kp, Vp = inputs(B, Nq, 0, H, D, 10)
    ids = np.array([-1] * 7 + [2] * 20 + [-1] * 3 + [4] * 10, dtype=np.int32)
    valid = np.ones((B, Nq), dtype=bool)
    got = o.masked_prefix_attention(Q, Kc, Vc, Kp, Vp, ids, valid, 0.125)
    assert np.array_equal(got, o.block_causal_attention(Q, Kc, Vc, ids))


def pin_text_only_is_dense_on_the_causal_keys(o):
    B, Nq, Np, H, D = 1, 9, 12, 2, 8
    Q, Kc, Vc, Kp, Vp = inputs(B, Nq, Np, H, D, 20)
    ids = np.full(Np + Nq, -1, dtype=np.int32)
    valid = np.ones((B, Np + Nq), dtype=bool)
    got = o.masked_prefix_attention(Q, Kc, Vc, Kp, Vp, ids, valid, float(np.float32(8 ** -0.5)))
    for i in (0, 4, Nq - 1):
        keys = np.concatenate([Kp, Kc[:, :i + 1]], 1)
        vals = np.concatenate([Vp, Vc[:, :i + 1]], 1)
        want = o.dense_attention(Q[:, i:i + 1], keys, vals)
        assert np.allclose(got[:, i:i + 1], want, rtol=1e-6, atol=1e-7)   # scale: fp32 vs D^-0.5


def pin_masking_a_prefix_key_is_deleting_it(o):
    B, Nq, Np, H, D = 1, 8, 10, 2, 8
    Q, Kc, Vc, Kp, Vp = inputs(B, Nq, Np, H, D, 30)
    ids = np.array([-1] * 4 + [1] * 6 + [1] * 3 + [-1] * 5, dtype=np.int32)
    j0 = 2
    valid = np.ones((B, Np + Nq), dtype=bool)
    valid[:, j0] = False
    got = o.masked_prefix_attention(Q, Kc, Vc, Kp, Vp, ids, valid, 0.3)
    keep = [j for j in range(Np) if j != j0]
    want = o.masked_prefix_attention(Q, Kc, Vc, np.ascontiguousarray(Kp[:, keep]),
                                     np.ascontiguousarray(Vp[:, keep]), np.delete(ids, j0),
                                     np.delete(valid, j0, axis=1), 0.3)
    assert np.array_equal(got, want)


def pin_scale_moves_into_q(o):
    B, Nq, Np, H, D = 1, 7, 5, 1, 8
    Q, Kc, Vc, Kp, Vp = inputs(B, Nq, Np, H, D, 40)
    ids = np.array([-1] * 5 + [0] * 7, dtype=np.int32)
    valid = np.ones((B, Np + Nq), dtype=bool)
    a = o.masked_prefix_attention(Q, Kc, Vc, Kp, Vp, ids, valid, 0.5)
    q2 = workloads.bf16_bits(torch.from_numpy(f(Q) * 2).to(torch.bfloat16))
    b = o.masked_prefix_attention(q2, Kc, Vc, Kp, Vp, ids, valid, 0.25)
    assert np.array_equal(a, b)
    c = o.masked_prefix_attention(Q, Kc, Vc, Kp, Vp, ids, valid, 0.25)
    assert not np.allclose(a, c)


def pin_row_without_a_visible_key_fails(o):
    B, Nq, Np, H, D = 1, 3, 2, 1, 4
    Q, Kc, Vc, Kp, Vp = inputs(B, Nq, Np, H, D, 50)
    ids = np.full(Np + Nq, -1, dtype=np.int32)
    valid = np.zeros((B, Np + Nq), dtype=bool)
    with pytest.raises(RuntimeError):
        o.masked_prefix_attention(Q, Kc, Vc, Kp, Vp, ids, valid, 0.5)


PINS = [pin_brute_force, pin_empty_prefix_is_block_causal, pin_text_only_is_dense_on_the_causal_keys,
        pin_masking_a_prefix_key_is_deleting_it, pin_scale_moves_into_q,
        pin_row_without_a_visible_key_fails]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(oracle_mod, pin):
    pin(oracle_mod.default())


def test_rows_match_full(oracle_mod):
    B, Nq, Np, H, D = 2, 20, 9, 2, 8
    Q, Kc, Vc, Kp, Vp = inputs(B, Nq, Np, H, D, 60)
    ids = np.array([-1] * 9 + [6] * 20, dtype=np.int32)
    valid = np.random.default_rng(1).random((B, Np + Nq)) < 0.8
    valid[:, 0] = True
    full = oracle_mod.masked_prefix_attention(Q, Kc, Vc, Kp, Vp, ids, valid, 0.3).reshape(-1, D)
    rows = np.array([0, 5, 41, 79], dtype=np.int64)
    got = oracle_mod.masked_prefix_attention_rows(Q, Kc, Vc, Kp, Vp, ids, valid, 0.3, rows)
    assert np.array_equal(got, full[rows])


MUTANTS = {
    "strict_causal": ("j <= qpos ||", "j < qpos ||"),
    "text_as_image": ("(image_ids[qpos] >= 0 && image_ids[j] == image_ids[qpos])",
                      "(image_ids[j] == image_ids[qpos])"),
    "key_valid_ignored": ("return causal_or_image && key_valid[b * Nall + j] != 0;",
                          "return causal_or_image;"),
    "key_valid_wrong_batch": ("key_valid[b * Nall + j]", "key_valid[j]"),
    "query_position_without_prefix": ("qpos = Np + i;", "qpos = i;"),
    "segments_swapped": ("if (j < Np)\n        return Xp", "if (j >= Nq)\n        return Xp"),
    "scale_ignored": ("s[j] = dot * scale;", "s[j] = dot;"),
    "no_max_subtraction": ("exp(s[j] - top)", "exp(s[j])"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(oracle_mod, name):
    import os
    import shutil
    import tempfile
    old, new = MUTANTS[name]
    src = open(oracle_mod.SOURCE_MASKED_PREFIX).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    tmp = tempfile.mkdtemp(prefix="oracle_mp_mutant_")
    try:
        path = os.path.join(tmp, "mutant.c")
        with open(path, "w") as fh:
            fh.write(src.replace(old, new))
        lib = oracle_mod.compile_source([oracle_mod.SOURCE, oracle_mod.SOURCE_BLOCK_CAUSAL, path],
                                        os.path.join(tmp, "libmutant.so"))
        mutant = oracle_mod.Oracle(lib)
        caught = []
        for pin in PINS:
            try:
                with np.errstate(all="ignore"):
                    pin(mutant)
            except (AssertionError, RuntimeError, ValueError):
                caught.append(pin.__name__)
            except BaseException as e:  # pytest.raises failing inside a pin is a catch too
                if type(e).__name__ == "Failed":
                    caught.append(pin.__name__)
                else:
                    raise
        assert caught, f"no pin catches mutant {name}"
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
