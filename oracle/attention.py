"""fp64 oracle of attention with rotary embeddings applied to Q and K --
TEST INFRASTRUCTURE ONLY (tests, smoke check, bench CPU leg).

"rotary-embedding-torch", flash_attn_with_rotary: the rotation is applied to
the loaded blocks of Q and K inside the attention kernel, so the rotated Q
and K are never written to global memory.  The result is
    O = softmax(scale * rot(Q) rot(K)^T + mask) V
with GQA/MQA (heads_q != heads_kv: each K/V head serves Hq/Hk query heads,
same page, Key Features), a causal mask (is_causal), a boolean attn_mask of
shape (batch, seq_len_k) or (batch, seq_len_q, seq_len_k) whose False entries
are excluded like masked scores (Input Tensor Shapes), and per-token
positions where -1 leaves the token unrotated (pos_mask /
rotary_pos_emb_indices, Input Tensor Shapes).

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
              pos_q=None, pos_k=None, causal=False, scale=None, want_bounds=False,
              attn_mask=None):
    """O (fp64) for q [B,Hq,Sq,D], k/v [B,Hk,Sk,D] given as element bits.

    attn_mask: None, or booleans [B, Sk] (one per key: key padding) or
    [B, Sq, Sk] (one per query and key); a False entry hides that key from
    that query, as the causal mask does (its score becomes -inf).  Both masks
    apply together.

    want_bounds: also return, like O, the two weights an implementation that
    rounds the softmax probabilities P and the output O is measured by:
        W[i, d] = sum_j p_ij |v_jd| / l_i   (what rounding P perturbs), and
        A[i, d] = sum_j vis_ij |v_jd| / l_i (what an absolute error in each p
                                             of the visible keys perturbs),
    with p_ij = exp(s_ij - max_j s_ij) over the visible keys and l_i = sum_j
    p_ij; zero for rows that see no key.  Rounding every p to a relative
    error e and O to a relative error e changes O by at most e (W + |O|),
    since |sum_j dp_j v_jd| / l <= e sum_j p_j |v_jd| / l."""
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
    w_abs = np.zeros((B, Hq, Sq, D)) if want_bounds else None
    a_abs = np.zeros((B, Hq, Sq, D)) if want_bounds else None
    vis_causal = np.ones((Sq, Sk), dtype=bool)
    if causal:
        vis_causal = np.arange(Sk)[None, :] <= (np.arange(Sq)[:, None] + (Sk - Sq))
    if attn_mask is not None:
        attn_mask = np.asarray(attn_mask, dtype=bool)
        if attn_mask.shape not in ((B, Sk), (B, Sq, Sk)):
            raise ValueError("attn_mask must be [B, Sk] or [B, Sq, Sk]")
    for b in range(B):
        visible = vis_causal
        if attn_mask is not None:
            mb = attn_mask[b]
            visible = visible & (mb[None, :] if mb.ndim == 1 else mb)
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
            if want_bounds:
                av = np.abs(v[b, kh])
                inv_l = np.where(has, 1.0 / np.where(l[:, 0] > 0, l[:, 0], 1.0), 0.0)[:, None]
                w_abs[b, h] = (p @ av) * inv_l
                a_abs[b, h] = (visible.astype(np.float64) @ av) * inv_l
    return (out, w_abs, a_abs) if want_bounds else out
