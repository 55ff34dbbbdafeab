"""Seeded synthetic workloads for rotary position embedding.

This module is shared by the tests, the bench and the smoke check, and feeds
the same bits to the CUDA library and to the CPU oracle.  It holds only
shapes, seeds and random draws: none of the method's arithmetic (no
frequencies, no angles, no rotation).

Workload shapes follow the pages' examples:
  * "How Unsloth Optimizes RoPE Embedding Computations in Triton Kernels",
    Usage Examples: Q, K [batch, n_heads, seq_len, head_dim]; optional
    [seq_len] position ids (prefix shift ``arange(seq_len) + prefix_len``).
  * "rotary-embedding-torch", flash_attn_with_rotary: q [1, 8, 1024 + 2, 64]
    with a 32-wide rotary part and the first two tokens left unrotated;
    RotaryEmbedding: ``seq_before_head_dim`` gives [batch, seq, heads, dim].
  * "Rotary Embedding (RoPE) Kernel Optimization", Paired Element Layout:
    split-half and interleaved pairs.
Values are N(0, 1), drawn in fp32 on the CPU from ``torch.Generator`` seeded
with the workload's seed, then cast to the workload's dtype.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

# enum values of the C ABI (include/rope.h); repeated here as plain numbers
DTYPES = {"f32": 0, "bf16": 1, "f16": 2}
TORCH_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}
LAYOUTS = {"split_half": 0, "interleaved": 1}
ELEM_BYTES = {"f32": 4, "bf16": 2, "f16": 2}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hk: int
    S: int
    D: int
    rotary_dim: int
    theta: float
    dtype: str              # "f32" | "bf16" | "f16"
    layout: str             # "split_half" | "interleaved"
    seq_before_head: bool   # False: [B,H,S,D]; True: [B,S,H,D]
    table_rows: int
    positions: str          # "none" | "masked_prefix" | "random_sorted"
    seed: int
    interpolate_factor: float = 1.0
    mask_prefix: int = 0    # tokens at the start with position -1 (masked_prefix only)

    @property
    def q_shape(self):
        return ((self.B, self.S, self.Hq, self.D) if self.seq_before_head
                else (self.B, self.Hq, self.S, self.D))

    @property
    def k_shape(self):
        return ((self.B, self.S, self.Hk, self.D) if self.seq_before_head
                else (self.B, self.Hk, self.S, self.D))

    def with_sizes(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads: a tiny fp32 case; a Llama-3-8B-shaped GQA layer (bf16);
# interleaved fp16 in [B,S,H,D]; partial rotary with masked prefix tokens and
# gathered positions; long-context prefill with random sorted positions.
WORKLOADS = [
    Workload("tiny_f32_split_half", 1, 8, 8, 128, 64, 64, 1e4, "f32", "split_half",
             False, 128, "none", seed=1),
    Workload("llama3_8b_gqa_bf16", 4, 32, 8, 4096, 128, 128, 5e5, "bf16", "split_half",
             False, 4096, "none", seed=2),
    Workload("interleaved_f16_bshd", 8, 32, 32, 2048, 128, 128, 1e4, "f16", "interleaved",
             True, 2048, "none", seed=3),
    Workload("partial_rd32_masked_bf16", 16, 16, 16, 1026, 64, 32, 1e4, "bf16", "split_half",
             False, 8192, "masked_prefix", seed=4, mask_prefix=2),
    Workload("long_context_gqa_bf16", 1, 32, 8, 131072, 128, 128, 5e5, "bf16", "split_half",
             False, 262144, "random_sorted", seed=5),
]
BY_NAME = {w.name: w for w in WORKLOADS}

# Launch-bound single calls of the Llama-3-8B-shaped layer: one decode step of
# 64 sequences (one token each) and a short prefill.  Not among the five
# workloads; the bench times them for the per-call cost of small calls.
SMALL_CALLS = [
    Workload("decode_b64_llama_bf16", 64, 32, 8, 1, 128, 128, 5e5, "bf16", "split_half",
             False, 4096, "none", seed=7),
    Workload("prefill_b1_s512_llama_bf16", 1, 32, 8, 512, 128, 128, 5e5, "bf16", "split_half",
             False, 4096, "none", seed=8),
]
ALL_BY_NAME = dict(BY_NAME, **{w.name: w for w in SMALL_CALLS})


def positions(w: Workload, gen: torch.Generator | None = None) -> np.ndarray | None:
    """int32 [S] position indices of the workload, or None for rows 0..S-1."""
    if w.positions == "none":
        return None
    if w.positions == "masked_prefix":
        p = np.arange(-w.mask_prefix, w.S - w.mask_prefix, dtype=np.int32)
        p[: w.mask_prefix] = -1
        return p
    if w.positions == "random_sorted":
        g = gen if gen is not None else torch.Generator().manual_seed(w.seed + 1000)
        perm = torch.randperm(w.table_rows, generator=g)[: w.S]
        return np.sort(perm.numpy()).astype(np.int32)
    raise ValueError(w.positions)


def draw(shape, dtype: str, gen: torch.Generator) -> torch.Tensor:
    """N(0,1) fp32 on the CPU from ``gen``, cast to ``dtype``."""
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(TORCH_DTYPES[dtype])


def make_inputs(w: Workload, seed_offset: int = 0):
    """Q, K (CPU torch tensors) and int32 positions (numpy or None)."""
    g = torch.Generator().manual_seed(w.seed + seed_offset)
    q = draw(w.q_shape, w.dtype, g)
    k = draw(w.k_shape, w.dtype, g) if w.Hk > 0 else None
    return q, k, positions(w)


def bits(t: torch.Tensor) -> np.ndarray:
    """Element bits of a CPU tensor as numpy (float32 or uint16), no copy of values."""
    t = t.contiguous()
    if t.dtype == torch.float32:
        return t.numpy()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view(np.uint16)
    raise TypeError(t.dtype)


def algorithmic_bytes(w: Workload) -> int:
    """Bytes one fused Q+K call must move: the rotary span of every Q and K row
    read and written, each distinct cos/sin row read once, and the position
    vector read once."""
    e = ELEM_BYTES[w.dtype]
    pos = positions(w)
    rotated_tokens = w.S if pos is None else int(np.count_nonzero(pos != -1))
    rows = w.B * rotated_tokens * (w.Hq + w.Hk)
    span = rows * w.rotary_dim * e * 2
    if pos is None:
        unique_rows = w.S
    else:
        unique_rows = int(np.unique(pos[pos >= 0]).size)
    table = unique_rows * (w.rotary_dim // 2) * 4 * 2
    return span + table + (0 if pos is None else w.S * 4)
