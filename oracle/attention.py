"""fp64 oracle of attention with rotary embeddings applied to Q and K --
TEST INFRASTRUCTURE ONLY (tests, smoke check, bench CPU leg).

"rotary-embedding-torch", flash_attn_with_rotary: the rotation is applied to
the loaded blocks of Q and K inside the attention kernel, so the rotated Q
and K are never written to global memory.  The result is
    O = softmax(scale * rot(Q) rot(K)^T + mask) V
with GQA/MQA (heads_q != heads_kv: each K/V head serves Hq/Hk query heads,
same page, Key Features), a causal mask (is_causal), and per-token positions
where -1 leaves the token unrotated (pos_mask / rotary_pos_emb_indices,
Input Tensor Shapes).

Readings (the page prints no formula for these):
  * the rotated Q and K are rounded to the input type (bf16/fp16) before the
    products, as they would be if written out by the separate rotation;
  * causal masking is aligned to the bottom right: query i (of Sq) may see
    key j (of Sk) when j <= i + Sk - Sq, the usual convention when Sq < Sk;
  * a query row with no visible key outputs zeros;
  * the default scale is 1/sqrt(D).
The rotation itself is the CPU oracle's (rope_oracle.c); the softmax and the
two products are plain numpy fp64.
"""
from __future__ import annotations

import numpy as np

from . import BF16, F16, F64, INTERLEAVED, SPLIT_HALF, load  # noqa: F401


_DECODE_CACHE = {}


def decode16(bits: np.ndarray, dtype: int) -> np.ndarray:
    """Exact fp64 values of bf16/fp16 bit patterns."""
    if dtype not in _DECODE_CACHE:
        o = load()
        conv = o.bf16_to_f64 if dtype == BF16 else o.f16_to_f64
        _DECODE_CACHE[dtype] = np.array([conv(i) for i in range(65536)], dtype=np.float64)
    return _DECODE_CACHE[dtype][bits.astype(np.int64)]


def rotate_rounded(x_bits, dtype, pos, rotary_dim, layout, cos32, sin32):
    """Rotate one [B,H,S,D] tensor with the oracle and round to the element type
    (dtype F64: fp64 values in, fp64 out, nothing rounded)."""
    B, H, S, D = x_bits.shape
    rc, yb, y64 = load().apply(x_bits, dtype, B, H, S, D, rotary_dim, layout, False, False, pos,
                               cos32, sin32, want_f64=(dtype == F64), want_bits=(dtype != F64))
    if rc != 0:
        raise ValueError("rotation rejected the positions (code %d)" % rc)
    return y64 if dtype == F64 else decode16(yb, dtype)


def attention(q_bits, k_bits, v_bits, dtype, rotary_dim, layout, cos32, sin32,
              pos_q=None, pos_k=None, causal=False, scale=None):
    """O (fp64) for q [B,Hq,Sq,D], k/v [B,Hk,Sk,D] given as element bits."""
    B, Hq, Sq, D = q_bits.shape
    _, Hk, Sk, _ = k_bits.shape
    if Hq % Hk:
        raise ValueError("Hq must be a multiple of Hk")
    scale = 1.0 / np.sqrt(D) if scale is None else scale
    q = rotate_rounded(q_bits, dtype, pos_q, rotary_dim, layout, cos32, sin32)
    k = rotate_rounded(k_bits, dtype, pos_k, rotary_dim, layout, cos32, sin32)
    v = np.asarray(v_bits, dtype=np.float64) if dtype == F64 else decode16(v_bits, dtype)
    group = Hq // Hk
    out = np.zeros((B, Hq, Sq, D))
    visible = np.ones((Sq, Sk), dtype=bool)
    if causal:
        visible = np.arange(Sk)[None, :] <= (np.arange(Sq)[:, None] + (Sk - Sq))
    for b in range(B):
        for h in range(Hq):
            kh = h // group
            s = (q[b, h] @ k[b, kh].T) * scale
            s = np.where(visible, s, -np.inf)
            m = s.max(axis=1, keepdims=True)
            has = np.isfinite(m[:, 0])
            p = np.where(visible, np.exp(s - np.where(np.isfinite(m), m, 0.0)), 0.0)
            l = p.sum(axis=1, keepdims=True)
            o = np.where(has[:, None], (p @ v[b, kh]) / np.where(l > 0, l, 1.0), 0.0)
            out[b, h] = o
    return out
