"""The Python binding checks its tensors before it calls the library: CPU
tensors, other dtypes and mismatched shapes raise at once (the product path
has no CPU fallback).  No GPU is needed: the checks run before any CUDA call."""
import pytest
import torch

import non_causal_prefix_gb300 as ncp


@pytest.fixture(scope="module", autouse=True)
def built():
    ncp.build(quiet=True)


def bf16(*shape):
    return torch.zeros(*shape, dtype=torch.bfloat16)


Q = (1, 256, 2, 64)


def calls(make):
    """Every tensor entry of the binding, with tensors from make(shape)."""
    q, k, v, o = (make(Q) for _ in range(4))
    kp, vp = make((1, 128, 2, 64)), make((1, 128, 2, 64))
    ids = torch.zeros(256, dtype=torch.int32)
    ids_all = torch.zeros(384, dtype=torch.int32)
    return {
        "attn_dense_fwd": lambda: ncp.attn_dense_fwd(q, k, v, o),
        "attn_dense_fwd_noalloc": lambda: ncp.attn_dense_fwd_noalloc(q, k, v, o),
        "attn_dense_cross_fwd": lambda: ncp.attn_dense_cross_fwd(q, kp, vp, o),
        "attn_prefix_fwd": lambda: ncp.attn_prefix_fwd(q, kp, vp, k, v, o),
        "attn_block_causal_fwd": lambda: ncp.attn_block_causal_fwd(q, k, v, ids, o),
        "attn_masked_prefix_fwd": lambda: ncp.attn_masked_prefix_fwd(
            q, k, v, kp, vp, ids_all, None, 0.125, o),
        "dense_attention": lambda: ncp.dense_attention(q, k, v),
        "prefix_attention": lambda: ncp.prefix_attention(q, kp, vp, k, v),
    }


ENTRIES = sorted(calls(bf16))


@pytest.mark.parametrize("name", ENTRIES)
def test_cpu_tensors_are_refused(name):
    with pytest.raises(ValueError, match="CUDA"):
        calls(lambda s: bf16(*s))[name]()


@pytest.mark.parametrize("name", ENTRIES)
def test_other_dtypes_are_refused(name):
    with pytest.raises((TypeError, ValueError)):
        calls(lambda s: torch.zeros(*s, dtype=torch.float32))[name]()


def test_shapes_are_checked():
    q, k, v = bf16(*Q), bf16(*Q), bf16(*Q)
    with pytest.raises(ValueError, match="shape"):
        ncp.attn_dense_fwd(q, k, v, bf16(1, 256, 2, 128))
    with pytest.raises(ValueError, match="B, N, H, D"):
        ncp.attn_dense_fwd(bf16(256, 2, 64), k, v, q)
    with pytest.raises(ValueError):
        ncp.attn_dense_cross_fwd(q, bf16(1, 128, 3, 64), bf16(1, 128, 3, 64), bf16(*Q))
    with pytest.raises(ValueError):
        ncp.attn_prefix_fwd(q, bf16(1, 128, 2, 128), bf16(1, 128, 2, 128), k, v, bf16(*Q))
    with pytest.raises(ValueError, match="image_ids"):
        ncp.attn_block_causal_fwd(q, k, v, torch.zeros(255, dtype=torch.int32), bf16(*Q))
