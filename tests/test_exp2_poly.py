"""The polynomial exp2 that the softmax uses for part of its exponentials.

CPU: the coefficients in the CUDA source are the minimax solution the
generator script computes, and an fp32 restatement of the algorithm (clamp,
round-to-integer by the 1.5 * 2^23 trick, cubic, exponent-field add) meets its
error bound against float64 2^x.  GPU: the kernel's own evaluation meets the
same bound, through the C ABI's test probe.
"""
import os
import re
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "non_causal_prefix_gb300", "csrc")
sys.path.insert(0, CSRC)

BOUND = 1.02e-4


def source_coeffs():
    text = open(os.path.join(CSRC, "sm103_ptx.cuh")).read()
    out = []
    for name in ("EXP2_C1", "EXP2_C2", "EXP2_C3"):
        m = re.search(name + r"\s*=\s*(0x[0-9a-fA-Fp.+-]+)f;", text)
        assert m, name
        out.append(float.fromhex(m.group(1)))
    return out


def poly_fp32(x, coeffs):
    """fp32 restatement of the kernel's exp2 path (no fused FMA: a bound check)."""
    f32 = np.float32
    x = np.maximum(np.asarray(x, dtype=f32), f32(-127.0))
    t = (x + f32(12582912.0)).astype(f32)
    j = (t - f32(12582912.0)).astype(f32)
    f = (x - j).astype(f32)
    c1, c2, c3 = (f32(c) for c in coeffs)
    p = f32(1) + f * (c1 + f * (c2 + f * c3))
    bits = p.view(np.uint32) + (t.view(np.uint32) << np.uint32(23))
    return bits.astype(np.uint32).view(f32)


def probe_inputs():
    rng = np.random.default_rng(5)
    xs = [np.linspace(-126.0, 127.0, 200_001), rng.uniform(-30, 8, 100_000),
          np.arange(-126, 128, dtype=np.float64), np.arange(-126, 127) + 0.5,
          np.arange(-125, 127) - 0.5 + 1e-6]
    return np.concatenate(xs).astype(np.float32)


def sub_normal_inputs():
    # -127 < x < -126: the result is below the smallest normal fp32 (the
    # exponent-field add cannot encode it exactly); only 0 <= y < 2^-125 holds.
    return np.linspace(-126.999, -126.001, 1001).astype(np.float32)


def test_source_coefficients_are_the_minimax_solution():
    pytest.importorskip("scipy")
    import exp2_poly_coeffs as gen
    want, err = gen.solve()
    got = source_coeffs()
    assert np.allclose(got, want, rtol=2e-6, atol=0), (got, want)
    assert err < BOUND
    assert gen.max_rel_error_fp32(got) < BOUND


def test_fp32_restatement_meets_the_bound():
    coeffs = source_coeffs()
    x = probe_inputs()
    y = poly_fp32(x, coeffs).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    assert np.max(np.abs(y / ref - 1)) < BOUND
    ints = np.arange(-126, 128).astype(np.float32)
    exact = np.exp2(ints.astype(np.float64)).astype(np.float32)
    assert np.array_equal(poly_fp32(ints, coeffs), exact)     # p(0) = 1
    low = np.array([-127.0, -128.0, -1e30, -np.inf], dtype=np.float32)
    assert np.all(poly_fp32(low, coeffs) == 0.0)
    tiny = poly_fp32(sub_normal_inputs(), coeffs).astype(np.float64)
    assert np.all((tiny >= 0) & (tiny < 2.0 ** -125))


@pytest.mark.gpu
def test_kernel_polynomial_meets_the_bound(cuda_lib):
    import torch
    x = probe_inputs()
    for extra in ([], [3.25]):   # even and odd element counts
        xe = np.concatenate([x, np.float32(extra)]).astype(np.float32)
        y = cuda_lib.debug_exp2(torch.from_numpy(xe).cuda(), 0).cpu().numpy()
        ref = np.exp2(xe.astype(np.float64))
        assert np.max(np.abs(y.astype(np.float64) / ref - 1)) < BOUND
    ints = torch.arange(-126, 128, dtype=torch.float32, device="cuda")
    assert torch.equal(cuda_lib.debug_exp2(ints, 0), torch.exp2(ints.double()).float())
    low = torch.tensor([-127.0, -128.0, -1e30, -float("inf")], device="cuda")
    assert torch.all(cuda_lib.debug_exp2(low, 0) == 0)
    tiny = cuda_lib.debug_exp2(torch.from_numpy(sub_normal_inputs()).cuda(), 0).double()
    assert torch.all((tiny >= 0) & (tiny < 2.0 ** -125))


@pytest.mark.gpu
def test_kernel_mufu_exp2(cuda_lib):
    import torch
    x = np.linspace(-100.0, 100.0, 100_001).astype(np.float32)
    y = cuda_lib.debug_exp2(torch.from_numpy(x).cuda(), 1).cpu().numpy()
    ref = np.exp2(x.astype(np.float64))
    assert np.max(np.abs(y.astype(np.float64) / ref - 1)) < 1e-6
