"""Seeded synthetic inputs for the attention leaf, shared by the tests, the bench
and the oracle's callers.

This module holds no attention arithmetic: it only draws random tensors.  The
pages' workloads are captured engine tensors that are not available here
(dense LTX video/audio attention and Qwen-Image prefix attention, page 2,
dataset README "Sources and scope"); the five configurations below stand in
for them with the same layout ``[B, N, H, D]`` (bf16, contiguous), the same
head count H=32 and the same head dims D in {64, 128}.

Recipe (one generator per tensor, so tensors are independent of each other):
    g = torch.Generator("cpu").manual_seed(1000 * config_id + tensor_index)
    x = (torch.randn(shape, dtype=float32, generator=g) * sigma).to(bfloat16)
Tensor order is (Q, K, V) for dense and (Q, K_prefix, V_prefix, K_current,
V_current) for the prefix-cached form, the operand order of the definitions
(noncausal_dense_attention_h32_d128 and prefix_cached_block_causal_h32_d128,
"inputs" and "reference" fields).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    """One synthetic workload.  ``kind`` is "dense" or "prefix"."""

    config_id: int
    name: str
    kind: str
    B: int
    Nq: int
    Nk: int          # dense: key count (== Nq for self-attention); prefix: Nc
    H: int
    D: int
    sigma: float
    Np: int = 0      # prefix length (prefix form only)
    # Block-causal and masked prefix forms: the key positions as (image id,
    # length) runs; -1 = text.
    segments: tuple = ()
    # Masked prefix form: runtime scale and [start, end) runs of padded keys.
    sm_scale: float = 0.0
    invalid: tuple = ()

    @property
    def n_keys(self) -> int:
        """Total visible keys per query (Np + Nc for prefix, Nk for dense)."""
        return self.Np + self.Nk

    @property
    def visible_pairs(self) -> int:
        """(query, key) pairs that enter the softmax, per (batch, head)."""
        if self.kind == "masked_prefix":
            ids = np.concatenate([np.full(n, k, dtype=np.int64) for k, n in self.segments])
            valid = np.ones(ids.size, dtype=bool)
            for a, b in self.invalid:
                valid[a:b] = False
            j = np.arange(ids.size)
            total = 0
            for i in range(self.Nq):
                qp = self.Np + i
                vis = (j <= qp) | ((ids[qp] >= 0) & (ids == ids[qp]))
                total += int(np.count_nonzero(vis & valid))
            return total
        if self.kind != "block_causal":
            return self.Nq * self.n_keys
        total, pos = 0, 0
        for ident, length in self.segments:
            if ident < 0:          # text: token i sees keys 0..i
                total += sum(pos + r + 1 for r in range(length))
            else:                  # an image block [pos, pos+length): every token sees 0..end-1
                total += length * (pos + length)
            pos += length
        return total

    @property
    def flops(self) -> int:
        """Algorithmic FLOPs: 2*D per visible score (QK^T) + 2*D per visible score (PV)."""
        return 4 * self.B * self.H * self.visible_pairs * self.D

    @property
    def hbm_bytes(self) -> int:
        """Algorithmic HBM bytes: every input read once, O written once (bf16)."""
        rows = self.Nq + self.Np * 2 + self.Nk * 2 + self.Nq  # Q, K, V (+prefix), O
        return 2 * self.B * self.H * self.D * rows

    def shapes(self):
        """Shapes of the inputs, in operand order."""
        q = (self.B, self.Nq, self.H, self.D)
        kv = (self.B, self.Nk, self.H, self.D)
        if self.kind in ("dense", "cross", "block_causal"):
            return [q, kv, kv]
        if self.kind == "masked_prefix":   # the old definition's operand order
            p = (self.B, self.Np, self.H, self.D)
            return [q, q, q, p, p]
        p = (self.B, self.Np, self.H, self.D)
        return [q, p, p, kv, kv]

    def describe(self) -> str:
        if self.kind == "block_causal":
            runs = "+".join(f"{'text' if i < 0 else 'img' + str(i)}:{n}" for i, n in self.segments)
            return (f"block-causal B={self.B} N={self.Nq} ({runs}) H={self.H} D={self.D} "
                    f"sigma={self.sigma}")
        if self.kind == "dense":
            return (f"dense B={self.B} N={self.Nq} H={self.H} D={self.D} "
                    f"sigma={self.sigma}")
        if self.kind == "masked_prefix":
            return (f"masked prefix B={self.B} Nq={self.Nq} Np={self.Np} H={self.H} D={self.D} "
                    f"padding={list(self.invalid)} sm_scale={self.sm_scale:.6g}")
        if self.kind == "cross":
            return (f"cross B={self.B} Nq={self.Nq} Nk={self.Nk} H={self.H} D={self.D} "
                    f"sigma={self.sigma}")
        return (f"prefix B={self.B} Nq=Nc={self.Nq} Np={self.Np} H={self.H} "
                f"D={self.D} sigma={self.sigma}")


# The five synthetic configurations of the dense and prefix-cached forms:
# 1-3 and 5 are dense self-attention, 4 is the prefix-cached form with a
# 1024-token prefix.  6-8 cover the further forms.  6 is the block-causal
# (empty-prefix) form of the same model's first evaluation: a text prompt, a
# condition image, a short text run and the target image, each image a
# contiguous block with its own id (definition prefix_cached_block_causal_h32_
# d128_prefix0: "image_ids still represents the engine segment list").
WORKLOADS = {
    1: Workload(1, "dense_b1_n128_h32_d64", "dense", 1, 128, 128, 32, 64, 1.0),
    2: Workload(2, "dense_b1_n4096_h32_d128", "dense", 1, 4096, 4096, 32, 128, 1.0),
    3: Workload(3, "dense_b2_n8192_h32_d64", "dense", 2, 8192, 8192, 32, 64, 1.0),
    4: Workload(4, "prefix_b1_nq4096_np1024_h32_d128", "prefix", 1, 4096, 4096, 32,
                128, 1.0, Np=1024),
    5: Workload(5, "dense_b1_n32768_h32_d128", "dense", 1, 32768, 32768, 32, 128, 0.5),
    6: Workload(6, "block_causal_b1_n4448_h32_d128", "block_causal", 1, 4448, 4448, 32, 128,
                1.0, segments=((-1, 333), (0, 2048), (-1, 19), (1, 2048))),
    # Cross attention (the dense definition's Nq != Nk case): video queries
    # over a short conditioning sequence, and a short query block over a long
    # context (fewer work units than SMs: the keys are split across SMs).
    7: Workload(7, "cross_b1_nq8192_nk512_h32_d128", "cross", 1, 8192, 512, 32, 128, 1.0),
    8: Workload(8, "cross_b1_nq256_nk32768_h32_d128", "cross", 1, 256, 32768, 32, 128, 1.0),
    # The pre-audit prefix form: a 1024-token prefix (a 256-token prompt whose
    # last 56 tokens are padding, then a 768-token condition image) and a
    # 4096-token target image as the current block; runtime scale 128^-0.5.
    9: Workload(9, "masked_prefix_b1_nq4096_np1024_h32_d128", "masked_prefix", 1, 4096, 4096, 32,
                128, 1.0, Np=1024, segments=((-1, 256), (0, 768), (1, 4096)),
                sm_scale=128 ** -0.5, invalid=((200, 256),)),
}


def randn_bf16(shape, sigma: float, seed: int) -> torch.Tensor:
    """N(0, sigma^2) float32 draws rounded to bf16 (round-to-nearest-even)."""
    g = torch.Generator("cpu").manual_seed(int(seed))
    x = torch.randn(tuple(shape), dtype=torch.float32, generator=g)
    if sigma != 1.0:
        x = x * sigma
    return x.to(torch.bfloat16).contiguous()


def make_inputs(w: Workload, seed_base: int | None = None):
    """CPU bf16 tensors for workload ``w`` in operand order."""
    base = 1000 * w.config_id if seed_base is None else seed_base
    return [randn_bf16(s, w.sigma, base + i) for i, s in enumerate(w.shapes())]


def custom(kind: str, B: int, Nq: int, Nk: int, H: int, D: int, sigma: float = 1.0,
           Np: int = 0, config_id: int = 0, segments: tuple = ()) -> Workload:
    """A workload of arbitrary shape (used for small parity and edge cases)."""
    name = f"{kind}_b{B}_nq{Nq}_nk{Nk}_np{Np}_h{H}_d{D}"
    if segments:
        assert sum(n for _, n in segments) == Nq == Nk
    return Workload(config_id, name, kind, B, Nq, Nk, H, D, sigma, Np=Np, segments=segments)


def key_valid(w: Workload) -> torch.Tensor:
    """The [B, Np + Nq] key-valid mask of a masked prefix workload (CPU bool)."""
    valid = torch.ones((w.B, w.Np + w.Nq), dtype=torch.bool)
    for a, b in w.invalid:
        valid[:, a:b] = False
    return valid


def image_ids(w: Workload) -> torch.Tensor:
    """The [N] int32 image-id vector of a block-causal workload (CPU)."""
    parts = [torch.full((n,), ident, dtype=torch.int32) for ident, n in w.segments]
    return torch.cat(parts) if parts else torch.empty(0, dtype=torch.int32)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bit patterns of a CPU bf16 tensor as a contiguous uint16 array."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)
