"""Pins of the rotary-attention oracle (oracle/attention.py), no GPU."""
import math

import numpy as np
import pytest

import oracle as O
from oracle import attention as A


def _tables(rd, rows, prec="f64"):
    return O.load().tables(1e4, rd, rows, 1.0, prec)


def _x(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


@pytest.mark.parametrize("layout", [O.SPLIT_HALF, O.INTERLEAVED])
@pytest.mark.parametrize("causal", [False, True])
def test_shifting_all_positions_leaves_attention_unchanged(layout, causal):
    # <R_m q, R_n k> depends on m - n only, so a common shift of every position
    # changes nothing
    B, Hq, Hk, Sq, Sk, D, rd = 1, 4, 2, 9, 13, 16, 16
    c, s = _tables(rd, 128)
    q, k, v = _x((B, Hq, Sq, D), 1), _x((B, Hk, Sk, D), 2), _x((B, Hk, Sk, D), 3)
    pq = np.arange(Sk - Sq, Sk, dtype=np.int32)
    pk = np.arange(Sk, dtype=np.int32)
    o0 = A.attention(q, k, v, O.F64, rd, layout, c, s, pq, pk, causal)
    for t in (1, 7, 50):
        o1 = A.attention(q, k, v, O.F64, rd, layout, c, s, pq + t, pk + t, causal)
        assert np.max(np.abs(o1 - o0)) <= 1e-12
    o2 = A.attention(q, k, v, O.F64, rd, layout, c, s, pq + 3, pk, causal)
    assert np.max(np.abs(o2 - o0)) > 1e-6          # a relative shift does change it


def test_constant_values_give_the_constant():
    B, H, S, D = 2, 3, 10, 8
    c, s = _tables(D, S)
    q, k = _x((B, H, S, D), 4), _x((B, H, S, D), 5)
    v = np.broadcast_to(np.arange(D, dtype=np.float64), (B, H, S, D)).copy()
    for causal in (False, True):
        o = A.attention(q, k, v, O.F64, D, O.SPLIT_HALF, c, s, None, None, causal)
        assert np.allclose(o, v, atol=1e-12)


def test_causal_first_query_sees_only_first_key():
    B, H, S, D = 1, 2, 6, 8
    c, s = _tables(D, S)
    q, k, v = _x((B, H, S, D), 6), _x((B, H, S, D), 7), _x((B, H, S, D), 8)
    o = A.attention(q, k, v, O.F64, D, O.SPLIT_HALF, c, s, None, None, True)
    assert np.array_equal(o[:, :, 0], v[:, :, 0])
    o_full = A.attention(q, k, v, O.F64, D, O.SPLIT_HALF, c, s, None, None, False)
    assert np.allclose(o[:, :, -1], o_full[:, :, -1], atol=1e-12)   # last query sees every key


def test_gqa_equals_repeated_kv_heads():
    B, Hq, Hk, S, D = 1, 6, 2, 7, 16
    c, s = _tables(D, S)
    q, k, v = _x((B, Hq, S, D), 9), _x((B, Hk, S, D), 10), _x((B, Hk, S, D), 11)
    o = A.attention(q, k, v, O.F64, D, O.SPLIT_HALF, c, s)
    kr, vr = np.repeat(k, Hq // Hk, axis=1), np.repeat(v, Hq // Hk, axis=1)
    o2 = A.attention(q, kr, vr, O.F64, D, O.SPLIT_HALF, c, s)
    assert np.array_equal(o, o2)


def test_key_permutation_invariance():
    B, H, Sq, Sk, D = 1, 2, 5, 11, 8
    c, s = _tables(D, Sk)
    q, k, v = _x((B, H, Sq, D), 12), _x((B, H, Sk, D), 13), _x((B, H, Sk, D), 14)
    pk = np.arange(Sk, dtype=np.int32)
    perm = np.random.default_rng(0).permutation(Sk)
    o = A.attention(q, k, v, O.F64, D, O.SPLIT_HALF, c, s, None, pk)
    o2 = A.attention(q, k[:, :, perm], v[:, :, perm], O.F64, D, O.SPLIT_HALF, c, s, None,
                     pk[perm].copy())
    assert np.max(np.abs(o - o2)) <= 1e-12


def test_unrotated_positions_give_plain_attention_and_zero_scale_averages():
    B, H, S, D = 1, 2, 6, 8
    c, s = _tables(D, S)
    q, k, v = _x((B, H, S, D), 15), _x((B, H, S, D), 16), _x((B, H, S, D), 17)
    none = np.full(S, -1, dtype=np.int32)
    o = A.attention(q, k, v, O.F64, D, O.SPLIT_HALF, c, s, none, none)
    for h in range(H):
        sc = q[0, h] @ k[0, h].T / math.sqrt(D)
        w = np.exp(sc - sc.max(axis=1, keepdims=True))
        assert np.allclose(o[0, h], (w / w.sum(axis=1, keepdims=True)) @ v[0, h], atol=1e-12)
    oz = A.attention(q, k, v, O.F64, D, O.SPLIT_HALF, c, s, None, None, True, scale=0.0)
    for i in range(S):
        assert np.allclose(oz[0, :, i], v[0, :, : i + 1].mean(axis=1), atol=1e-12)


def test_brute_force_scalar_loops_tiny_case():
    B, Hq, Hk, Sq, Sk, D, rd = 1, 2, 1, 3, 4, 4, 2
    c, s = _tables(rd, 8)
    q, k, v = _x((B, Hq, Sq, D), 18), _x((B, Hk, Sk, D), 19), _x((B, Hk, Sk, D), 20)
    pq = np.array([2, -1, 5], dtype=np.int32)
    pk = np.array([0, 1, -1, 7], dtype=np.int32)
    o = A.attention(q, k, v, O.F64, rd, O.SPLIT_HALF, c, s, pq, pk, True)

    def rot(x, p):
        x = list(x)
        if p < 0:
            return x
        # rd = 2: one pair (x[0], x[1]) rotated by p radians (inverse frequency 1)
        a = float(p)
        return [x[0] * math.cos(a) - x[1] * math.sin(a), x[0] * math.sin(a) + x[1] * math.cos(a)] + x[2:]

    for h in range(Hq):
        for i in range(Sq):
            qi = rot(q[0, h, i], pq[i])
            sc = []
            for j in range(Sk):
                if j > i + Sk - Sq:
                    continue
                kj = rot(k[0, 0, j], pk[j])
                sc.append((j, sum(a * b for a, b in zip(qi, kj)) / math.sqrt(D)))
            mx = max(x for _, x in sc)
            w = [(j, math.exp(x - mx)) for j, x in sc]
            tot = sum(x for _, x in w)
            for d in range(D):
                want = sum(wj * v[0, 0, j, d] for j, wj in w) / tot
                assert abs(o[0, h, i, d] - want) <= 1e-12
