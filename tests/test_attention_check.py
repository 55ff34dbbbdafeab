"""The fused-attention comparison rule (attention_check.py) can fail: on the
full-length Llama-shaped causal prefill (Sq = Sk = 4096, GQA 32/8, D = 128,
bf16), at sampled query rows, it rejects an all-zero output and the result of
an attention that skips one key tile of 128 keys, and accepts the oracle's
result rounded once to bf16 and the worst case its two roundings allow.  Two
value tensors: N(0,1), and a tile indicator v[j, d] = 1 when
(j // 128) % D == d, so that output column d carries the softmax mass of key
tile d alone.  Runs on the CPU (oracle only)."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from oracle import attention as OA

import attention_check as AC

B, HQ, HK, S, D, RD, THETA = 1, 32, 8, 4096, 128, 128, 5e5
ROWS = [(0, 4095), (5, 2047), (31, 1000), (17, 129), (3, 3900), (12, 640)]


def tile_indicator_values(Sk, D):
    v = np.zeros((Sk, D), dtype=np.float32)
    v[np.arange(Sk), (np.arange(Sk) // 128) % D] = 1.0
    return v


@pytest.fixture(scope="module")
def inputs():
    g = torch.Generator().manual_seed(6)
    q = W.draw((B, HQ, S, D), "bf16", g)
    k = W.draw((B, HK, S, D), "bf16", g)
    v = W.draw((B, HK, S, D), "bf16", g)
    vt = torch.from_numpy(tile_indicator_values(S, D)).to(torch.bfloat16)[None, None].expand(
        B, HK, S, D).contiguous()
    c32, s32 = O.load().tables(THETA, RD, S, 1.0, "f32")
    return q, k, v, vt, c32, s32


def row_ref(q, k, v, c32, s32, h, i, keep=None):
    """The oracle's row i of query head h at position i, against the keys it
    sees (keys 0..i, or the subset `keep` of them, at their own positions)."""
    kv = h // (HQ // HK)
    keys = np.arange(i + 1) if keep is None else keep
    kb = np.ascontiguousarray(W.bits(k[:, kv:kv + 1])[:, :, keys])
    vb = np.ascontiguousarray(W.bits(v[:, kv:kv + 1])[:, :, keys])
    return OA.attention(W.bits(q[:, h:h + 1, i:i + 1]), kb, vb, O.BF16, RD, O.SPLIT_HALF, c32,
                        s32, np.array([i], dtype=np.int32), keys.astype(np.int32), False,
                        want_bounds=True)


def to_bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).double().numpy()


@pytest.mark.parametrize("values", ["normal", "tile_indicator"])
def test_rule_rejects_zero_and_a_skipped_key_tile(inputs, values):
    q, k, v, vt, c32, s32 = inputs
    vv = v if values == "normal" else vt
    for h, i in ROWS:
        o, w, a = row_ref(q, k, vv, c32, s32, h, i)
        # accepted: the exact result rounded once, and the worst case of both roundings
        AC.check(to_bf16(o), o, w, a, "bf16", "rounded oracle row")
        u = AC.U["bf16"]
        sgn = np.where(o >= 0, 1.0, -1.0)
        worst = (o + sgn * u * w) * (1 + sgn * u)
        AC.check(worst, o, w, a, "bf16", "worst-case roundings")
        # rejected: zeros
        assert AC.rejects(np.zeros_like(o), o, w, a, "bf16"), (values, h, i)
        # rejected: the first, a middle and the last whole key tile skipped
        full = (i + 1) // 128
        for t in sorted({0, full // 2, full - 1}):
            keep = np.setdiff1d(np.arange(i + 1), np.arange(128 * t, 128 * t + 128))
            skipped = row_ref(q, k, vv, c32, s32, h, i, keep)[0]
            assert AC.rejects(skipped, o, w, a, "bf16"), (values, h, i, t)


def test_rule_is_tighter_than_the_value_range_bound(inputs):
    """The value-range rule u (max|v| + |O|) lets an all-zero output through on
    most elements of a late row; the weighted rule only where |O| is itself
    below u W, the resolution any implementation that rounds P has."""
    q, k, v, vt, c32, s32 = inputs
    o, w, a = row_ref(q, k, v, c32, s32, 0, 4095)
    u = AC.U["bf16"]
    old = u * (float(v.float().abs().max()) + np.abs(o))
    new = AC.tolerance("bf16", o, w, a)
    assert np.mean(np.abs(o) <= old) > 0.3
    assert np.mean(np.abs(o) <= new) < 0.15
    assert np.all(np.abs(o)[np.abs(o) <= new] <= 2 * AC.U["bf16"] * w[np.abs(o) <= new])
    assert np.all(new < old)


def test_fp16_subnormal_term():
    """fp16: probabilities below 2^-14 are subnormal, with an absolute error
    of up to 2^-25 each; the rule's A term covers a row of such keys."""
    o = np.array([[[[1e-3, -2e-3]]]])
    w = np.array([[[[0.5, 0.5]]]])
    a = np.array([[[[4096.0, 4096.0]]]])
    tol = AC.tolerance("f16", o, w, a)
    assert np.allclose(tol - (AC.U["f16"] + AC.ARITH) * (w + np.abs(o)), 2.0 ** -25 * a)
    assert np.allclose(AC.tolerance("bf16", o, w, a), (AC.U["bf16"] + AC.ARITH) * (w + np.abs(o)))
