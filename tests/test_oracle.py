"""Pins of the FP64 oracle against facts that do not come from the oracle itself.

The pages print no worked numbers for the attention leaf, so every pin is a
closed form, an invariant, a brute force on tiny inputs or a library special
case of the definition (page "Audit SGLang interfaces and refresh validated
kernel solutions", definitions noncausal_dense_attention_h32_d{128,64}.json
and prefix_cached_block_causal_h32_d128.json, field "reference").  The last
test plants plausible mistakes in a copy of the oracle's C source and checks
that at least one pin fails for each.
"""
import math
import os
import random
import shutil
import subprocess
import tempfile

import numpy as np
import pytest
import torch

import workloads


def bits(x) -> np.ndarray:
    """bf16 bit patterns of values that are exactly representable in bf16."""
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    back = t.float().numpy()
    assert np.array_equal(back, np.asarray(x, dtype=np.float32)), "not exact in bf16"
    return workloads.bf16_bits(t)


def rand_bits(shape, seed, sigma=1.0):
    return workloads.bf16_bits(workloads.randn_bf16(shape, sigma, seed))


def values(u16: np.ndarray) -> np.ndarray:
    return (u16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------
# Pins, written against an oracle object so the mutant check can reuse them.
# --------------------------------------------------------------------------

def pin_single_key(o):
    """Nk = 1: the only weight is 1, so O[b,i,h] == V[b,0,h] exactly."""
    for D in (8, 64, 128):
        Q = rand_bits((2, 5, 3, D), 11)
        K = rand_bits((2, 1, 3, D), 12)
        V = rand_bits((2, 1, 3, D), 13)
        out = o.dense_attention(Q, K, V)
        want = np.broadcast_to(values(V), out.shape)
        assert np.array_equal(out, want)


def pin_identical_keys(o):
    """All keys equal within a (b, h): uniform weights, O = mean_j V[b,j,h]."""
    B, Nq, Nk, H, D = 2, 4, 37, 3, 64
    Q = rand_bits((B, Nq, H, D), 21)
    k_one = rand_bits((B, 1, H, D), 22)
    K = np.ascontiguousarray(np.broadcast_to(k_one, (B, Nk, H, D)))
    V = rand_bits((B, Nk, H, D), 23)
    out = o.dense_attention(Q, K, V)
    Vv = values(V)
    for b in range(B):
        for h in range(H):
            mean = np.array([math.fsum(Vv[b, :, h, d]) / Nk for d in range(D)])
            for i in range(Nq):
                np.testing.assert_allclose(out[b, i, h], mean, rtol=0, atol=1e-14)


def pin_dominant_logit(o):
    """One key aligned with a large query: its weight is 1 - O(e^-1000).

    q = 128 e_0 and k_{j*} = 128 e_0 give a score of 128^2 D^-0.5 (>= 1448),
    every other key is zero (score 0).  exp of the raw score overflows a
    double, so this also fails an oracle that skips the max subtraction.
    """
    for D in (64, 128):
        B, Nq, Nk, H = 2, 3, 9, 4
        Q = np.zeros((B, Nq, H, D), np.float32)
        Q[..., 0] = 128.0
        K = np.zeros((B, Nk, H, D), np.float32)
        star = {}
        for b in range(B):
            for h in range(H):
                j = (3 * b + 5 * h + 1) % Nk
                star[b, h] = j
                K[b, j, h, 0] = 128.0
        V = rand_bits((B, Nk, H, D), 31)
        out = o.dense_attention(bits(Q), bits(K), V)
        Vv = values(V)
        for (b, h), j in star.items():
            for i in range(Nq):
                assert np.array_equal(out[b, i, h], Vv[b, j, h])


def pin_two_key_logistic(o):
    """Nk = 2: O = v0 + sigmoid(d) (v1 - v0), d = (q.k1 - q.k0) D^-0.5.

    Products of bf16 values are exact in double and summed with fsum, so the
    closed form is accurate to a few ulp; the scale D^-0.5 and the pairing of
    weights with values are what it pins.
    """
    for D in (64, 128):
        B, Nq, H = 1, 6, 2
        Q = rand_bits((B, Nq, H, D), 41, 0.5)
        K = rand_bits((B, 2, H, D), 42, 0.5)
        V = rand_bits((B, 2, H, D), 43)
        out = o.dense_attention(Q, K, V)
        q, k, v = values(Q), values(K), values(V)
        for i in range(Nq):
            for h in range(H):
                d = (math.fsum(q[0, i, h] * k[0, 1, h]) - math.fsum(q[0, i, h] * k[0, 0, h]))
                d /= math.sqrt(D)
                w1 = 1.0 / (1.0 + math.exp(-d))
                want = v[0, 0, h] + w1 * (v[0, 1, h] - v[0, 0, h])
                np.testing.assert_allclose(out[0, i, h], want, rtol=1e-12, atol=1e-14)


def pin_joint_permutation(o):
    """Permuting K and V rows together leaves O unchanged (up to rounding)."""
    B, Nq, Nk, H, D = 2, 7, 50, 3, 64
    Q, K, V = (rand_bits((B, n, H, D), 51 + t) for t, n in enumerate((Nq, Nk, Nk)))
    perm = np.random.default_rng(5).permutation(Nk)
    a = o.dense_attention(Q, K, V)
    b = o.dense_attention(Q, np.ascontiguousarray(K[:, perm]), np.ascontiguousarray(V[:, perm]))
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-14)
    # Permuting V alone changes the result: the pairing of k_j with v_j matters.
    c = o.dense_attention(Q, K, np.ascontiguousarray(V[:, perm]))
    assert np.abs(a - c).max() > 1e-3


def pin_row_independence(o):
    """Each output row depends only on its own (b, i, h): slicing the problem
    by batch, query rows or heads gives bit-identical rows."""
    B, Nq, Nk, H, D = 2, 9, 13, 3, 64
    Q, K, V = (rand_bits((B, n, H, D), 61 + t) for t, n in enumerate((Nq, Nk, Nk)))
    full = o.dense_attention(Q, K, V)
    for b in range(B):
        for h in range(H):
            sl = o.dense_attention(np.ascontiguousarray(Q[b:b + 1, :, h:h + 1]),
                                   np.ascontiguousarray(K[b:b + 1, :, h:h + 1]),
                                   np.ascontiguousarray(V[b:b + 1, :, h:h + 1]))
            assert np.array_equal(sl[0, :, 0], full[b, :, h])
    perm = np.random.default_rng(6).permutation(Nq)
    pq = o.dense_attention(np.ascontiguousarray(Q[:, perm]), K, V)
    assert np.array_equal(pq, full[:, perm])


def brute_force(Q, K, V, scale=None):
    """Pure-Python softmax attention with fsum; Q [B,Nq,H,D], K/V [B,Nk,H,D]."""
    q, k, v = values(Q), values(K), values(V)
    B, Nq, H, D = q.shape
    Nk = k.shape[1]
    scale = D ** -0.5 if scale is None else scale
    out = np.zeros((B, Nq, H, D))
    for b in range(B):
        for h in range(H):
            for i in range(Nq):
                s = [math.fsum(q[b, i, h, d] * k[b, j, h, d] for d in range(D)) * scale
                     for j in range(Nk)]
                m = max(s)
                w = [math.exp(x - m) for x in s]
                l = math.fsum(w)
                for d in range(D):
                    out[b, i, h, d] = math.fsum(w[j] * v[b, j, h, d] for j in range(Nk)) / l
    return out


def pin_brute_force(o):
    """Tiny shapes, self and cross attention, against the pure-Python sum."""
    rng = random.Random(7)
    for case in range(8):
        B, H = rng.randint(1, 2), rng.randint(1, 2)
        Nq, Nk = rng.randint(1, 9), rng.randint(1, 9)
        D = rng.choice((1, 2, 8))
        Q, K, V = (rand_bits((B, n, H, D), 70 + 3 * case + t)
                   for t, n in enumerate((Nq, Nk, Nk)))
        np.testing.assert_allclose(o.dense_attention(Q, K, V), brute_force(Q, K, V),
                                   rtol=1e-12, atol=1e-14)


def pin_torch_float64(o):
    """The definition's own expression (einsum, softmax, einsum) in float64."""
    for (B, Nq, Nk, H, D) in ((1, 128, 128, 4, 64), (2, 33, 70, 3, 128)):
        ts = [workloads.randn_bf16((B, n, H, D), 1.0, 80 + t)
              for t, n in enumerate((Nq, Nk, Nk))]
        q, k, v = (t.double() for t in ts)
        scores = torch.einsum("bqhd,bkhd->bhqk", q, k) * D ** -0.5
        want = torch.einsum("bhqk,bkhd->bqhd", scores.softmax(-1), v).numpy()
        got = o.dense_attention(*(workloads.bf16_bits(t) for t in ts))
        np.testing.assert_allclose(got, want, rtol=1e-11, atol=1e-13)


def pin_prefix_is_dense_on_concat(o):
    """prefix_attention(Q, Kp, Vp, Kc, Vc) == attention(Q, cat(Kp,Kc), cat(Vp,Vc))."""
    for (B, Nq, Np, Nc, H, D) in ((1, 5, 3, 4, 2, 8), (2, 17, 9, 17, 3, 128)):
        Q = rand_bits((B, Nq, H, D), 91)
        Kp, Vp = rand_bits((B, Np, H, D), 92), rand_bits((B, Np, H, D), 93)
        Kc, Vc = rand_bits((B, Nc, H, D), 94), rand_bits((B, Nc, H, D), 95)
        got = o.prefix_attention(Q, Kp, Vp, Kc, Vc)
        K = np.ascontiguousarray(np.concatenate([Kp, Kc], axis=1))
        V = np.ascontiguousarray(np.concatenate([Vp, Vc], axis=1))
        assert np.array_equal(got, o.dense_attention(Q, K, V))
        # Brute force on the concatenation for the small case.
        if D == 8:
            np.testing.assert_allclose(got, brute_force(Q, K, V), rtol=1e-12, atol=1e-14)
        # The prefix keys are visible: dropping them changes the output.
        assert np.abs(got - o.dense_attention(Q, Kc, Vc)).max() > 1e-3


def pin_prefix_pairs_segments(o):
    """K_prefix pairs with V_prefix and K_current with V_current: a prefix key
    that dominates selects its prefix value row, a current key its current row."""
    B, Nq, Np, Nc, H, D = 1, 2, 3, 4, 2, 128
    Q = np.zeros((B, Nq, H, D), np.float32)
    Q[..., 0] = 128.0
    Vp, Vc = rand_bits((B, Np, H, D), 96), rand_bits((B, Nc, H, D), 97)
    for seg, j in (("prefix", 1), ("current", 2)):
        Kp = np.zeros((B, Np, H, D), np.float32)
        Kc = np.zeros((B, Nc, H, D), np.float32)
        (Kp if seg == "prefix" else Kc)[0, j, :, 0] = 128.0
        out = o.prefix_attention(bits(Q), bits(Kp), Vp, bits(Kc), Vc)
        want = values(Vp if seg == "prefix" else Vc)[0, j]
        for i in range(Nq):
            assert np.array_equal(out[0, i], want)


def pin_prefix_empty(o):
    """Np = 0 reduces to dense attention over the current keys."""
    Q, Kc, Vc = (rand_bits((2, n, 2, 64), 98 + t) for t, n in enumerate((6, 11, 11)))
    got = o.prefix_attention(Q, None, None, Kc, Vc)
    assert np.array_equal(got, o.dense_attention(Q, Kc, Vc))


def pin_rows_match_full(o):
    """Sampled rows are the same computation as the full output."""
    B, Nq, Nk, H, D = 2, 9, 21, 3, 64
    Q, K, V = (rand_bits((B, n, H, D), 101 + t) for t, n in enumerate((Nq, Nk, Nk)))
    full = o.dense_attention(Q, K, V).reshape(-1, D)
    rows = np.array([0, 5, B * Nq * H - 1, 17, 17])
    assert np.array_equal(o.dense_attention_rows(Q, K, V, rows), full[rows])
    Kp, Vp = rand_bits((B, 4, H, D), 104), rand_bits((B, 4, H, D), 105)
    fullp = o.prefix_attention(Q, Kp, Vp, K, V).reshape(-1, D)
    assert np.array_equal(o.prefix_attention_rows(Q, Kp, Vp, K, V, rows), fullp[rows])


PINS = [pin_single_key, pin_identical_keys, pin_dominant_logit, pin_two_key_logistic,
        pin_joint_permutation, pin_row_independence, pin_brute_force, pin_torch_float64,
        pin_prefix_is_dense_on_concat, pin_prefix_pairs_segments, pin_prefix_empty,
        pin_rows_match_full]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(oracle_mod, pin):
    pin(oracle_mod.default())


def test_oracle_rejects_bad_shapes(oracle_mod):
    o = oracle_mod.default()
    z = np.zeros((1, 1, 1, 8), np.uint16)
    rc = o.lib.oracle_dense_attention(None, None, None, None, 1, 1, 1, 1, 8)
    assert rc == -1
    with pytest.raises(RuntimeError):
        o.dense_attention_rows(z, z, z, np.array([5]))     # row out of range
    with pytest.raises(ValueError):
        o.dense_attention(z, np.zeros((1, 1, 2, 8), np.uint16), z)


def test_oracle_output_finite_on_workload_shapes(oracle_mod):
    """Config 1 in full and sampled rows of the others: finite, and |O| is
    bounded by max |V| (O is a convex combination of value rows)."""
    o = oracle_mod.default()
    w = workloads.WORKLOADS[1]
    ins = [workloads.bf16_bits(t) for t in workloads.make_inputs(w)]
    out = o.dense_attention(*ins)
    assert np.isfinite(out).all()
    vmax = np.abs(values(ins[2])).max(axis=1, keepdims=True)
    assert (np.abs(out) <= vmax + 1e-12).all()


# --------------------------------------------------------------------------
# Planted mistakes: each mutant of the C source must fail at least one pin.
# --------------------------------------------------------------------------

MUTANTS = {
    "no_max_subtraction": ("exp(s[j] - m)", "exp(s[j])"),
    "scale_one_over_d": ("pow((double)D, -0.5)", "pow((double)D, -1.0)"),
    "no_scale": ("s[j] = dot * scale;", "s[j] = dot;"),
    "no_normalisation": ("o_row[d] = acc[d] / l;", "o_row[d] = acc[d];"),
    "value_uses_key": ("const uint16_t *v = V + ((b * Nk + j) * H + h) * D;",
                       "const uint16_t *v = K + ((b * Nk + j) * H + h) * D;"),
    "value_wrong_head": ("const uint16_t *v = V + ((b * Nk + j) * H + h) * D;",
                         "const uint16_t *v = V + ((b * Nk + j) * H + 0) * D;"),
    "key_wrong_batch": ("const uint16_t *k = K + ((b * Nk + j) * H + h) * D;",
                        "const uint16_t *k = K + ((0 * Nk + j) * H + h) * D;"),
    "query_layout_bhnd": ("const uint16_t *q = Q + ((b * Nq + i) * H + h) * D;",
                          "const uint16_t *q = Q + ((b * H + h) * Nq + i) * D;"),
    "sign_flip": ("s[j] = dot * scale;", "s[j] = -dot * scale;"),
    "last_key_dropped": ("for (int64_t j = 0; j < Nk; ++j) {\n        const double w",
                         "for (int64_t j = 0; j < Nk - 1; ++j) {\n        const double w"),
    "prefix_segments_unpaired": (
        "uint16_t *values = concat_tokens(V_prefix, V_current, B, Np, Nc, H, D);",
        "uint16_t *values = concat_tokens(V_current, V_prefix, B, Nc, Np, H, D);"),
    "prefix_dropped": (
        "rc = oracle_dense_attention_rows(Q, keys, values, O_rows, B, Nq, Np + Nc, H, D,",
        "rc = oracle_dense_attention_rows(Q, keys + (int64_t)Np * H * D, "
        "values + (int64_t)Np * H * D, O_rows, B, Nq, Nc, H, D,"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(oracle_mod, name):
    old, new = MUTANTS[name]
    src = open(oracle_mod.SOURCE).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    tmp = tempfile.mkdtemp(prefix="oracle_mutant_")
    try:
        path = os.path.join(tmp, "mutant.c")
        with open(path, "w") as f:
            f.write(src.replace(old, new))
        lib = oracle_mod.compile_source(path, os.path.join(tmp, "libmutant.so"))
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


def test_oracle_matches_frozen_fixture(oracle_mod):
    """The oracle still produces the rows frozen in tests/golden (bitwise)."""
    import json
    path = os.path.join(os.path.dirname(__file__), "golden",
                        "oracle_dense_b1_n128_h32_d64_rows.json")
    doc = json.load(open(path))
    w = workloads.WORKLOADS[1]
    q, k, v = (workloads.bf16_bits(t) for t in workloads.make_inputs(w))
    got = oracle_mod.dense_attention_rows(q, k, v, np.array(doc["rows_flat_index"]))
    want = np.array([[float.fromhex(x) for x in row] for row in doc["values"]])
    assert np.array_equal(got, want)
