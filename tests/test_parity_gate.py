"""Negative and positive controls of the parity gate (CPU only).

The acceptance rule of the task-acceptance checker (page "Audit SGLang
interfaces and refresh validated kernel solutions", scripts/task_acceptance.py
compare_output, dataset README "Task acceptance configs") is an element rule:
|a - e| <= atol + rtol |e| for at least 99.99 % of the elements.  At the long
workload (dense B=1 N=32768 H=32 D=128, inputs N(0, 0.5^2)) the logits have a
standard deviation of about 0.25, so the softmax weights are nearly uniform
and |O| is about 3e-3, below atol = 1e-2.  The element rule alone then accepts
an output that ignores Q K^T altogether.  The internal gate
rel_rms = ||a - e|| / ||e|| <= 1e-2 closes that hole.

These tests build wrong outputs from the oracle's own inputs and show that
each one fails the gate:
  - an all-zero output;
  - the mean of V (uniform weights: a kernel blind to Q K^T);
  - a prefix-cached call that skips the prefix keys;
  - a prefix-cached call whose value segments are swapped against the key
    segments (key j of cat(K_prefix, K_current) paired with value j of
    cat(V_current, V_prefix)).
They also show that the mean-of-V output passes the element rule at the long
workload (the reason the gate exists), and that correct outputs pass the gate:
the oracle rounded to bf16, and the prefix-cached call with both segments
swapped together (for the full-visibility form that is a joint permutation of
the key/value pairs, which leaves the softmax unchanged).
"""
import numpy as np
import pytest
import torch

import workloads
from parity import bf16_round, passes, passes_element_rule, sample_rows, stats


def bits(ts):
    return [workloads.bf16_bits(t) for t in ts]


def mean_of_v(V: torch.Tensor, rows: np.ndarray, Nq: int, H: int) -> np.ndarray:
    """The output of uniform weights for flat rows (b * Nq + i) * H + h: the
    mean over all keys of V[b, :, h, :], in FP64."""
    b_idx = rows // (Nq * H)
    h_idx = rows % H
    out = np.empty((rows.size, V.shape[-1]), dtype=np.float64)
    cache = {}
    for n, (b, h) in enumerate(zip(b_idx, h_idx)):
        key = (int(b), int(h))
        if key not in cache:
            cache[key] = V[key[0], :, key[1], :].double().mean(0).numpy()
        out[n] = cache[key]
    return out


@pytest.fixture(scope="module")
def long_dense(oracle_mod):
    w = workloads.WORKLOADS[5]
    ins = workloads.make_inputs(w)
    rows = sample_rows(w.B, w.Nq, w.H, n_random=150, seed=5)
    ref = oracle_mod.dense_attention_rows(*bits(ins), rows)
    return w, ins, rows, ref


@pytest.fixture(scope="module")
def prefix_case(oracle_mod):
    w = workloads.WORKLOADS[4]
    ins = workloads.make_inputs(w)  # Q, K_prefix, V_prefix, K_current, V_current
    rows = sample_rows(w.B, w.Nq, w.H, n_random=150, seed=4)
    ref = oracle_mod.prefix_attention_rows(*bits(ins), rows)
    return w, ins, rows, ref


def test_long_workload_output_is_below_atol(long_dense):
    """The premise: at N = 32768, sigma = 0.5 the outputs sit below atol."""
    _, _, _, ref = long_dense
    assert np.sqrt(np.mean(ref ** 2)) < 5e-3


def test_long_all_zero_fails_gate(long_dense):
    _, _, _, ref = long_dense
    s = stats(np.zeros_like(ref), ref)
    assert s["rel_rms"] == pytest.approx(1.0)
    assert not passes(s)


def test_long_mean_of_v_passes_element_rule_but_fails_gate(long_dense):
    w, ins, rows, ref = long_dense
    s = stats(mean_of_v(ins[2], rows, w.Nq, w.H), ref)
    print("mean-of-V at N=32768:", s)
    assert passes_element_rule(s), s   # the hole in the element rule
    assert s["rel_rms"] > 0.1          # far outside the gate
    assert not passes(s)


def test_long_rounded_oracle_passes_gate(long_dense):
    _, _, _, ref = long_dense
    s = stats(bf16_round(ref), ref)
    assert passes(s), s
    assert s["rel_rms"] < 2e-3


def test_prefix_all_zero_and_mean_of_v_fail_gate(prefix_case):
    w, ins, rows, ref = prefix_case
    assert not passes(stats(np.zeros_like(ref), ref))
    v_all = torch.cat([ins[2], ins[4]], dim=1)  # cat(V_prefix, V_current)
    s = stats(mean_of_v(v_all, rows, w.Nq, w.H), ref)
    assert not passes(s), s


def test_prefix_dropped_fails_gate(oracle_mod, prefix_case):
    """A prefix path that skips the prefix tiles: dense attention over the
    current keys alone."""
    w, ins, rows, ref = prefix_case
    q, kp, vp, kc, vc = bits(ins)
    s = stats(oracle_mod.dense_attention_rows(q, kc, vc, rows), ref)
    print("prefix dropped:", s)
    assert not passes(s), s


def test_prefix_value_segments_swapped_fails_gate(oracle_mod, prefix_case):
    """Keys walked prefix first, values current first: every key paired with
    the wrong value row."""
    w, ins, rows, ref = prefix_case
    q, kp, vp, kc, vc = ins
    v_swapped = torch.cat([vc, vp], dim=1)
    vp_bad = v_swapped[:, :w.Np].contiguous()
    vc_bad = v_swapped[:, w.Np:].contiguous()
    s = stats(oracle_mod.prefix_attention_rows(*bits([q, kp, vp_bad, kc, vc_bad]), rows), ref)
    print("value segments swapped:", s)
    assert not passes(s), s


def test_prefix_joint_segment_swap_passes_gate(oracle_mod, prefix_case):
    """Swapping both segments together permutes (key, value) pairs jointly:
    the full-visibility softmax is unchanged, so the gate must accept it."""
    w, ins, rows, ref = prefix_case
    q, kp, vp, kc, vc = bits(ins)
    s = stats(oracle_mod.prefix_attention_rows(q, kc, vc, kp, vp, rows), ref)
    assert passes(s), s
    assert s["max_abs_err"] < 1e-12
