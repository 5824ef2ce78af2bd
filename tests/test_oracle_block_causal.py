"""Pins of the FP64 oracle for block-causal attention with image segments
(definition prefix_cached_block_causal_h32_d128_prefix0, field "reference":
query i sees key j iff j <= i, or image_ids[i] == image_ids[j] >= 0).

Each pin comes from outside the oracle's own code: special cases that reduce
to the dense oracle (one image: every key visible) or to a truncated dense
problem (text only: causal), a closed form (row 0 of a text sequence is v_0),
an invariance the definition implies (shuffling key/value rows inside one
image block changes nothing), and a pure-Python brute force written from the
definition on tiny mixed inputs.  Two planted mistakes (strict causality;
text tokens treated as one image) each fail a pin.
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


def brute(Q, K, V, ids, causal_strict=False, text_is_image=False):
    """Pure-Python restatement of the definition, math.fsum sums."""
    q, k, v = f(Q), f(K), f(V)
    B, N, H, D = q.shape
    out = np.zeros((B, N, H, D))
    for b in range(B):
        for h in range(H):
            for i in range(N):
                vis = []
                for j in range(N):
                    causal = j < i if causal_strict else j <= i
                    same = ids[i] == ids[j] and (text_is_image or ids[i] >= 0)
                    if causal or same:
                        vis.append(j)
                if not vis:
                    out[b, i, h] = np.nan
                    continue
                s = [math.fsum(q[b, i, h, d] * k[b, j, h, d] for d in range(D)) / math.sqrt(D)
                     for j in vis]
                mx = max(s)
                w = [math.exp(x - mx) for x in s]
                tot = math.fsum(w)
                for d in range(D):
                    out[b, i, h, d] = math.fsum(wj * v[b, j, h, d] for wj, j in zip(w, vis)) / tot
    return out


IDS_MIXED = np.array([-1, -1, 0, 0, 0, -1, 2, 2, -1], dtype=np.int32)


def test_brute_force_tiny_mixed(oracle_mod):
    B, N, H, D = 2, 9, 2, 4
    Q, K, V = rnd((B, N, H, D), 1), rnd((B, N, H, D), 2), rnd((B, N, H, D), 3)
    got = oracle_mod.block_causal_attention(Q, K, V, IDS_MIXED)
    assert np.allclose(got, brute(Q, K, V, IDS_MIXED), rtol=1e-12, atol=1e-13)


def test_text_only_is_causal_dense_on_the_prefix(oracle_mod):
    B, N, H, D = 1, 37, 2, 8
    Q, K, V = rnd((B, N, H, D), 4), rnd((B, N, H, D), 5), rnd((B, N, H, D), 6)
    ids = np.full(N, -1, dtype=np.int32)
    got = oracle_mod.block_causal_attention(Q, K, V, ids)
    for i in (0, 1, 17, N - 1):
        want = oracle_mod.dense_attention(Q[:, i:i + 1], K[:, :i + 1], V[:, :i + 1])
        assert np.allclose(got[:, i:i + 1], want, rtol=1e-13, atol=1e-14)
    # Closed form: the first text token sees only itself.
    assert np.array_equal(got[:, 0], f(V)[:, 0])


def test_one_image_is_dense(oracle_mod):
    B, N, H, D = 2, 40, 2, 8
    Q, K, V = rnd((B, N, H, D), 7), rnd((B, N, H, D), 8), rnd((B, N, H, D), 9)
    ids = np.full(N, 3, dtype=np.int32)
    got = oracle_mod.block_causal_attention(Q, K, V, ids)
    assert np.array_equal(got, oracle_mod.dense_attention(Q, K, V))


def test_shuffling_inside_an_image_block_changes_nothing(oracle_mod):
    B, N, H, D = 1, 30, 2, 8
    ids = np.array([-1] * 6 + [0] * 10 + [-1] * 4 + [1] * 10, dtype=np.int32)
    Q, K, V = rnd((B, N, H, D), 10), rnd((B, N, H, D), 11), rnd((B, N, H, D), 12)
    base = oracle_mod.block_causal_attention(Q, K, V, ids)
    perm = np.arange(N)
    perm[6:16] = np.random.default_rng(0).permutation(np.arange(6, 16))
    got = oracle_mod.block_causal_attention(Q, K[:, perm], V[:, perm], ids)
    assert np.allclose(got, base, rtol=1e-12, atol=1e-13)
    # ... while shuffling across the block boundary does change a later text row.
    perm2 = np.arange(N)
    perm2[[0, 20]] = perm2[[20, 0]]
    moved = oracle_mod.block_causal_attention(Q, K[:, perm2], V[:, perm2], ids)
    assert not np.allclose(moved[:, 5], base[:, 5])


def test_rows_match_full(oracle_mod):
    B, N, H, D = 2, 50, 3, 8
    ids = np.array([-1] * 5 + [4] * 20 + [-1] * 5 + [7] * 20, dtype=np.int32)
    Q, K, V = rnd((B, N, H, D), 13), rnd((B, N, H, D), 14), rnd((B, N, H, D), 15)
    full = oracle_mod.block_causal_attention(Q, K, V, ids).reshape(-1, D)
    rows = np.array([0, 7, 151, 299], dtype=np.int64)
    got = oracle_mod.block_causal_attention_rows(Q, K, V, ids, rows)
    assert np.array_equal(got, full[rows])


@pytest.mark.parametrize("mistake", ["causal_strict", "text_is_image"])
def test_planted_mistakes_fail_a_pin(oracle_mod, mistake):
    B, N, H, D = 1, 9, 1, 4
    Q, K, V = rnd((B, N, H, D), 16), rnd((B, N, H, D), 17), rnd((B, N, H, D), 18)
    wrong = brute(Q, K, V, IDS_MIXED, **{mistake: True})
    right = oracle_mod.block_causal_attention(Q, K, V, IDS_MIXED)
    assert not np.allclose(np.nan_to_num(wrong, nan=1e9), right, rtol=1e-6, atol=1e-6)


def test_one_image_is_dense_with_large_logits(oracle_mod):
    """Logits of several hundred: the max subtraction keeps exp finite; the
    dense oracle (pinned separately on a dominant-logit closed form) agrees."""
    B, N, H, D = 1, 24, 1, 8
    Q, K, V = rnd((B, N, H, D), 19, 30.0), rnd((B, N, H, D), 20, 30.0), rnd((B, N, H, D), 21)
    ids = np.full(N, 0, dtype=np.int32)
    got = oracle_mod.block_causal_attention(Q, K, V, ids)
    assert np.isfinite(got).all()
    assert np.array_equal(got, oracle_mod.dense_attention(Q, K, V))


# --------------------------------------------------------------------------
# Planted mistakes in the C source: each mutant must fail at least one pin.
# --------------------------------------------------------------------------

PINS = [test_brute_force_tiny_mixed, test_text_only_is_causal_dense_on_the_prefix,
        test_one_image_is_dense, test_shuffling_inside_an_image_block_changes_nothing,
        test_rows_match_full, test_one_image_is_dense_with_large_logits]

MUTANTS = {
    "strict_causal": ("return j <= i ||", "return j < i ||"),
    "anti_causal": ("return j <= i ||", "return j >= i ||"),
    "text_tokens_as_one_image": ("(image_ids[i] >= 0 && image_ids[j] == image_ids[i])",
                                 "(image_ids[j] == image_ids[i])"),
    "no_max_subtraction": ("exp(s[j] - mx)", "exp(s[j])"),
    "value_uses_key": ("const uint16_t *vr = V +", "const uint16_t *vr = K +"),
    "key_row_is_query_row": ("const uint16_t *kr = K + ((b * N + j)",
                             "const uint16_t *kr = K + ((b * N + i)"),
    "no_normalisation": ("o_row[d] = acc[d] / total;", "o_row[d] = acc[d];"),
    "mask_missing_in_pass_2": ("if (!visible(image_ids, i, j))\n            continue;\n"
                               "        const double wj",
                               "if (0)\n            continue;\n        const double wj"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(oracle_mod, name):
    import os
    import shutil
    import tempfile
    old, new = MUTANTS[name]
    src = open(oracle_mod.SOURCE_BLOCK_CAUSAL).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    tmp = tempfile.mkdtemp(prefix="oracle_bc_mutant_")
    try:
        path = os.path.join(tmp, "mutant.c")
        with open(path, "w") as fh:
            fh.write(src.replace(old, new))
        lib = oracle_mod.compile_source([oracle_mod.SOURCE, path],
                                        os.path.join(tmp, "libmutant.so"))
        mutant = oracle_mod.Oracle(lib)
        caught = []
        for pin in PINS:
            try:
                with np.errstate(all="ignore"):
                    pin(mutant)
            except (AssertionError, RuntimeError, ValueError):
                caught.append(pin.__name__)
        assert caught, f"no pin catches mutant {name}"
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
