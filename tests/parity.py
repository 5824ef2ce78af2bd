"""Acceptance arithmetic shared by the parity tests and the bench.

The element rule is the pages' task acceptance (page "Audit SGLang interfaces
and refresh validated kernel solutions", scripts/task_acceptance.py
compare_output; dataset README "Task acceptance configs"): an element matches
when |a - e| <= atol + rtol * |e|; the matched count is an integer; any
non-finite value fails.  The thresholds are the target tolerance of this
build: max |err| <= 2e-2 and at least 99.99 % of elements within
atol = rtol = 1e-2.  An internal gate adds rel_rms = ||a - e|| / ||e|| <= 1e-2,
because at N = 32768 with sigma = 0.5 the outputs (~3e-3) sit below atol and
the element rule alone would accept a kernel that ignores Q K^T.
"""
from __future__ import annotations

import numpy as np

MAX_ABS = 2e-2
ATOL = 1e-2
RTOL = 1e-2
MATCHED_RATIO = 0.9999
REL_RMS = 1e-2


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float64 values to bf16 (nearest even) and return them as float64."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).double().numpy()


def stats(actual: np.ndarray, expected: np.ndarray) -> dict:
    """Comparison statistics of ``actual`` (GPU, any float) against FP64 ``expected``."""
    a = np.asarray(actual, dtype=np.float64)
    e = np.asarray(expected, dtype=np.float64)
    assert a.shape == e.shape, (a.shape, e.shape)
    finite = bool(np.isfinite(a).all() and np.isfinite(e).all())
    err = np.abs(a - e)
    close = err <= ATOL + RTOL * np.abs(e)
    matched = int(np.count_nonzero(close))
    n = close.size
    ref_norm = float(np.sqrt(np.sum(e * e)))
    return {
        "finite": finite,
        "max_abs_err": float(err.max()) if n else 0.0,
        "matched": matched,
        "elements": n,
        "matched_ratio": matched / n if n else 1.0,
        "rel_rms": float(np.sqrt(np.sum((a - e) ** 2)) / ref_norm) if ref_norm > 0 else 0.0,
    }


def passes_element_rule(s: dict) -> bool:
    """The pages' element rule alone: finite, max |err| and the matched count."""
    return (s["finite"] and s["max_abs_err"] <= MAX_ABS and
            s["matched"] * 10000 >= s["elements"] * 9999)


def passes(s: dict) -> bool:
    """The element rule and the internal rel_rms gate."""
    return passes_element_rule(s) and s["rel_rms"] <= REL_RMS


def assert_parity(actual, expected, what: str = "") -> dict:
    s = stats(actual, expected)
    assert passes(s), f"{what} parity failed: {s}"
    return s


def sample_rows(B: int, Nq: int, H: int, n_random: int, seed: int) -> np.ndarray:
    """Flat row indices (b*Nq + i)*H + h: tile edges, the ragged end and a
    seeded random spread over every (b, h)."""
    rng = np.random.default_rng(seed)
    qs = {0, 1, 127, 128, 129, 255, 256, Nq // 2, Nq - 129, Nq - 128, Nq - 1}
    qs = sorted(q for q in qs if 0 <= q < Nq)
    rows = []
    for b in range(B):
        for h in sorted({0, H // 2, H - 1}):
            rows += [(b * Nq + q) * H + h for q in qs]
    rows += list(rng.integers(0, B * Nq * H, size=n_random))
    return np.unique(np.array(rows, dtype=np.int64))
