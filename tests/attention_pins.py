"""Pins of the rotary-attention oracle, as functions of the oracle module.

Each pin takes the module (``oracle.attention``, or a copy with a planted
mistake) and raises AssertionError when the module breaks what it checks.
test_oracle_attention.py runs them on the oracle; test_oracle_attention_mutants.py
runs them on mutants.  What fixes each expected value:
  * relative positions: <R_m q, R_n k> depends on m - n only (RoFormer's
    property, restated by the pages), so shifting every position together
    changes nothing;
  * closed forms: constant values average to the constant; a causal first
    query sees only the first key; zero scale gives the mean of the visible
    values; unrotated tokens give plain softmax attention (written out here
    with numpy); a query row that sees no key gives zeros (the reading the
    oracle states);
  * GQA is the same as repeating each key/value head over its query group;
  * brute force: scalar Python loops on tiny cases, in fp64 and in bf16 with
    the rotated rows rounded as the oracle's reading says;
  * the attn_mask: an all-True mask is no mask, hiding a key is deleting it
    (with its position), a per-query mask shaped like the causal pattern is
    the causal mask, and a row whose keys are all hidden gives zeros;
  * the bound weights W = sum p |v| / l and A = sum_vis |v| / l: constant
    values give W = |c|, one visible key gives W = A = |v_0|, and always
    |O| <= W <= A with W blind to the sign of V.
"""
import math

import numpy as np

import oracle as O


def _tables(rd, rows, prec="f64"):
    return O.load().tables(1e4, rd, rows, 1.0, prec)


def _x(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def pin_shifting_all_positions_leaves_attention_unchanged(A):
    B, Hq, Hk, Sq, Sk, D, rd = 1, 4, 2, 9, 13, 16, 16
    c, s = _tables(rd, 128)
    q, k, v = _x((B, Hq, Sq, D), 1), _x((B, Hk, Sk, D), 2), _x((B, Hk, Sk, D), 3)
    pq = np.arange(Sk - Sq, Sk, dtype=np.int32)
    pk = np.arange(Sk, dtype=np.int32)
    for layout in (O.SPLIT_HALF, O.INTERLEAVED):
        for causal in (False, True):
            o0 = A.attention(q, k, v, O.F64, rd, layout, c, s, pq, pk, causal)
            for t in (1, 7, 50):
                o1 = A.attention(q, k, v, O.F64, rd, layout, c, s, pq + t, pk + t, causal)
                assert np.max(np.abs(o1 - o0)) <= 1e-12
            o2 = A.attention(q, k, v, O.F64, rd, layout, c, s, pq + 3, pk, causal)
            assert np.max(np.abs(o2 - o0)) > 1e-6      # a relative shift does change it


def pin_constant_values_give_the_constant(A):
    B, H, S, D = 2, 3, 10, 8
    c, s = _tables(D, S)
    q, k = _x((B, H, S, D), 4), _x((B, H, S, D), 5)
    v = np.broadcast_to(np.arange(D, dtype=np.float64), (B, H, S, D)).copy()
    for causal in (False, True):
        o = A.attention(q, k, v, O.F64, D, O.SPLIT_HALF, c, s, None, None, causal)
        assert np.allclose(o, v, atol=1e-12)


def pin_causal_first_query_sees_only_first_key(A):
    B, H, S, D = 1, 2, 6, 8
    c, s = _tables(D, S)
    q, k, v = _x((B, H, S, D), 6), _x((B, H, S, D), 7), _x((B, H, S, D), 8)
    o = A.attention(q, k, v, O.F64, D, O.SPLIT_HALF, c, s, None, None, True)
    assert np.array_equal(o[:, :, 0], v[:, :, 0])
    o_full = A.attention(q, k, v, O.F64, D, O.SPLIT_HALF, c, s, None, None, False)
    assert np.allclose(o[:, :, -1], o_full[:, :, -1], atol=1e-12)   # the last query sees every key


def pin_rows_that_see_no_key_are_zero(A):
    # Sq > Sk, causal, bottom-right aligned: query i sees key j when j <= i + Sk - Sq, so the
    # first Sq - Sk queries see nothing and give zeros; query Sq - Sk sees key 0 only
    B, H, Sq, Sk, D = 1, 2, 7, 3, 8
    c, s = _tables(D, Sq)
    q, k, v = _x((B, H, Sq, D), 21), _x((B, H, Sk, D), 22), _x((B, H, Sk, D), 23)
    o = A.attention(q, k, v, O.F64, D, O.SPLIT_HALF, c, s, None, None, True)
    assert np.all(np.isfinite(o))
    assert np.array_equal(o[:, :, : Sq - Sk], np.zeros((B, H, Sq - Sk, D)))
    assert np.array_equal(o[:, :, Sq - Sk], v[:, :, 0])


def pin_gqa_equals_repeated_kv_heads(A):
    B, Hq, Hk, S, D = 1, 6, 2, 7, 16
    c, s = _tables(D, S)
    q, k, v = _x((B, Hq, S, D), 9), _x((B, Hk, S, D), 10), _x((B, Hk, S, D), 11)
    o = A.attention(q, k, v, O.F64, D, O.SPLIT_HALF, c, s)
    kr, vr = np.repeat(k, Hq // Hk, axis=1), np.repeat(v, Hq // Hk, axis=1)
    o2 = A.attention(q, kr, vr, O.F64, D, O.SPLIT_HALF, c, s)
    assert np.array_equal(o, o2)


def pin_key_permutation_invariance(A):
    B, H, Sq, Sk, D = 1, 2, 5, 11, 8
    c, s = _tables(D, Sk)
    q, k, v = _x((B, H, Sq, D), 12), _x((B, H, Sk, D), 13), _x((B, H, Sk, D), 14)
    pk = np.arange(Sk, dtype=np.int32)
    perm = np.random.default_rng(0).permutation(Sk)
    o = A.attention(q, k, v, O.F64, D, O.SPLIT_HALF, c, s, None, pk)
    o2 = A.attention(q, k[:, :, perm], v[:, :, perm], O.F64, D, O.SPLIT_HALF, c, s, None,
                     pk[perm].copy())
    assert np.max(np.abs(o - o2)) <= 1e-12


def pin_unrotated_positions_give_plain_attention_and_zero_scale_averages(A):
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


def _rot2(x, p):
    """rd = 2: the pair (x[0], x[1]) rotated by p radians (inverse frequency 1)."""
    x = list(x)
    if p < 0:
        return x
    a = float(p)
    return [x[0] * math.cos(a) - x[1] * math.sin(a), x[0] * math.sin(a) + x[1] * math.cos(a)] + x[2:]


def _loop_attention(qrows, krows, vrows, Sq, Sk, D, causal):
    """Scalar softmax attention of one head: lists of rows in, rows out."""
    out = []
    for i in range(Sq):
        sc = []
        for j in range(Sk):
            if causal and j > i + Sk - Sq:
                continue
            sc.append((j, sum(a * b for a, b in zip(qrows[i], krows[j])) / math.sqrt(D)))
        if not sc:
            out.append([0.0] * D)
            continue
        mx = max(x for _, x in sc)
        w = [(j, math.exp(x - mx)) for j, x in sc]
        tot = sum(x for _, x in w)
        out.append([sum(wj * vrows[j][d] for j, wj in w) / tot for d in range(D)])
    return out


def pin_brute_force_scalar_loops_tiny_case(A):
    B, Hq, Hk, Sq, Sk, D, rd = 1, 2, 1, 3, 4, 4, 2
    c, s = _tables(rd, 8)
    q, k, v = _x((B, Hq, Sq, D), 18), _x((B, Hk, Sk, D), 19), _x((B, Hk, Sk, D), 20)
    pq = np.array([2, -1, 5], dtype=np.int32)
    pk = np.array([0, 1, -1, 7], dtype=np.int32)
    o = A.attention(q, k, v, O.F64, rd, O.SPLIT_HALF, c, s, pq, pk, True)
    krows = [_rot2(k[0, 0, j], pk[j]) for j in range(Sk)]
    for h in range(Hq):
        qrows = [_rot2(q[0, h, i], pq[i]) for i in range(Sq)]
        want = _loop_attention(qrows, krows, v[0, 0].tolist(), Sq, Sk, D, True)
        assert np.max(np.abs(o[0, h] - np.array(want))) <= 1e-12


def pin_bf16_rotated_rows_are_rounded_before_the_products(A):
    # bf16 inputs: the rotated q and k rows are rounded to bf16 (the oracle's reading) before
    # S = q k^T; checked against scalar loops over the rotation's own rounded output, and
    # against the unrounded result, which differs
    B, H, Sq, Sk, D, rd = 1, 1, 3, 5, 8, 8
    c32, s32 = _tables(rd, 16, "f32")
    g = np.random.default_rng(24)
    to_bits = O.load().f64_to_bf16
    bits = lambda shape: np.array([to_bits(x) for x in g.standard_normal(int(np.prod(shape)))],
                                  dtype=np.uint16).reshape(shape)
    qb, kb, vb = bits((B, H, Sq, D)), bits((B, H, Sk, D)), bits((B, H, Sk, D))
    pq = np.array([3, 4, 9], dtype=np.int32)
    pk = np.array([0, 2, 5, 6, 11], dtype=np.int32)
    o = A.attention(qb, kb, vb, O.BF16, rd, O.SPLIT_HALF, c32, s32, pq, pk, True)
    rot = lambda xb, p: A.decode16(
        O.load().apply(xb, O.BF16, B, H, xb.shape[2], D, rd, O.SPLIT_HALF, False, False, p, c32,
                       s32, want_bits=True)[1], O.BF16)
    qr, kr, vv = rot(qb, pq)[0, 0], rot(kb, pk)[0, 0], A.decode16(vb, O.BF16)[0, 0]
    want = np.array(_loop_attention(qr.tolist(), kr.tolist(), vv.tolist(), Sq, Sk, D, True))
    assert np.max(np.abs(o[0, 0] - want)) <= 1e-12
    rot64 = lambda xb, p: O.load().apply(xb, O.BF16, B, H, xb.shape[2], D, rd, O.SPLIT_HALF, False,
                                         False, p, c32, s32, want_f64=True)[2]
    unrounded = np.array(_loop_attention(rot64(qb, pq)[0, 0].tolist(), rot64(kb, pk)[0, 0].tolist(),
                                         vv.tolist(), Sq, Sk, D, True))
    assert np.max(np.abs(o[0, 0] - unrounded)) > 1e-6


def pin_default_scale_is_inverse_sqrt_d(A):
    B, H, S, D = 1, 1, 5, 16
    c, s = _tables(D, S)
    q, k, v = _x((B, H, S, D), 25), _x((B, H, S, D), 26), _x((B, H, S, D), 27)
    o = A.attention(q, k, v, O.F64, D, O.SPLIT_HALF, c, s)
    o2 = A.attention(q, k, v, O.F64, D, O.SPLIT_HALF, c, s, scale=1.0 / math.sqrt(D))
    assert np.array_equal(o, o2)
    o3 = A.attention(q, k, v, O.F64, D, O.SPLIT_HALF, c, s, scale=1.0 / D)
    assert np.max(np.abs(o - o3)) > 1e-6


def pin_bound_weights_closed_forms(A):
    B, H, Sq, Sk, D = 1, 2, 6, 9, 8
    c, s = _tables(D, Sk)
    q, k, v = _x((B, H, Sq, D), 31), _x((B, H, Sk, D), 32), _x((B, H, Sk, D), 33)
    for causal in (False, True):
        o, w, a = A.attention(q, k, v, O.F64, D, O.SPLIT_HALF, c, s, None, None, causal,
                              want_bounds=True)
        assert np.array_equal(o, A.attention(q, k, v, O.F64, D, O.SPLIT_HALF, c, s, None, None,
                                             causal))
        assert np.all(np.abs(o) <= w + 1e-12) and np.all(w <= a + 1e-12)
        # the sign of V changes O's sign, not the weights
        o2, w2, a2 = A.attention(q, k, -v, O.F64, D, O.SPLIT_HALF, c, s, None, None, causal,
                                 want_bounds=True)
        assert np.allclose(o2, -o, atol=1e-12) and np.allclose(w2, w, atol=1e-12)
        assert np.allclose(a2, a, atol=1e-12)
        # constant values: W is |c| whatever the weights, A is |c| times the
        # visible keys over the softmax sum (>= |c|, = |c| for one key)
        cv = np.broadcast_to(np.linspace(-2.0, 1.5, D), (B, H, Sk, D)).copy()
        _, wc, ac = A.attention(q, k, cv, O.F64, D, O.SPLIT_HALF, c, s, None, None, causal,
                                want_bounds=True)
        assert np.allclose(wc, np.abs(cv[:, :, :Sq]), atol=1e-12)
        assert np.all(ac >= np.abs(cv[:, :, :Sq]) - 1e-12)
    # causal with Sq = Sk: the first query sees key 0 alone (p = 1, l = 1)
    o, w, a = A.attention(q, k[:, :, :Sq], v[:, :, :Sq], O.F64, D, O.SPLIT_HALF, c, s, None, None,
                          True, want_bounds=True)
    assert np.array_equal(w[:, :, 0], np.abs(v[:, :, 0])) and np.array_equal(a[:, :, 0],
                                                                             np.abs(v[:, :, 0]))


def pin_attn_mask_hides_keys(A):
    B, Hq, Hk, Sq, Sk, D = 2, 4, 2, 5, 11, 8
    c, s = _tables(D, 32)
    q, k, v = _x((B, Hq, Sq, D), 34), _x((B, Hk, Sk, D), 35), _x((B, Hk, Sk, D), 36)
    pq = np.arange(Sk - Sq, Sk, dtype=np.int32)
    pk = np.arange(Sk, dtype=np.int32)
    for causal in (False, True):
        base = A.attention(q, k, v, O.F64, D, O.SPLIT_HALF, c, s, pq, pk, causal)
        ones = np.ones((B, Sk), dtype=bool)
        assert np.array_equal(base, A.attention(q, k, v, O.F64, D, O.SPLIT_HALF, c, s, pq, pk,
                                                causal, attn_mask=ones))
        # batch 0 hides keys 1 and 6, batch 1 hides its last three: the same as
        # deleting those keys (with their positions) from each batch entry
        mask = ones.copy()
        mask[0, [1, 6]] = False
        mask[1, Sk - 3:] = False
        got = A.attention(q, k, v, O.F64, D, O.SPLIT_HALF, c, s, pq, pk, causal, attn_mask=mask)
        for b in range(B):
            keep = np.flatnonzero(mask[b])
            want = A.attention(q[b:b + 1], k[b:b + 1][:, :, keep], v[b:b + 1][:, :, keep], O.F64, D,
                               O.SPLIT_HALF, c, s, pq, pk[keep].copy(), False,
                               attn_mask=None if not causal else
                               (keep[None, None, :] <= (np.arange(Sq)[None, :, None] + Sk - Sq)))
            assert np.max(np.abs(got[b] - want[0])) <= 1e-12
        # a [B, Sq, Sk] mask equal to the causal pattern is the causal mask; the
        # same key mask broadcast over the queries is the key mask
        pat = np.arange(Sk)[None, :] <= (np.arange(Sq)[:, None] + (Sk - Sq))
        full = np.broadcast_to(pat, (B, Sq, Sk)).copy()
        assert np.max(np.abs(A.attention(q, k, v, O.F64, D, O.SPLIT_HALF, c, s, pq, pk, False,
                                         attn_mask=full) -
                             A.attention(q, k, v, O.F64, D, O.SPLIT_HALF, c, s, pq, pk, True))) == 0
        bcast = np.broadcast_to(mask[:, None, :], (B, Sq, Sk)).copy()
        assert np.array_equal(got, A.attention(q, k, v, O.F64, D, O.SPLIT_HALF, c, s, pq, pk,
                                               causal, attn_mask=bcast))
    # every key of batch 1 hidden: zeros there, batch 0 unchanged
    mask = np.ones((B, Sk), dtype=bool)
    mask[1] = False
    got = A.attention(q, k, v, O.F64, D, O.SPLIT_HALF, c, s, pq, pk, False, attn_mask=mask)
    assert np.array_equal(got[1], np.zeros_like(got[1]))
    assert np.array_equal(got[0], A.attention(q, k, v, O.F64, D, O.SPLIT_HALF, c, s, pq, pk)[0])
    # one query row of batch 0 with all its keys hidden
    m3 = np.ones((B, Sq, Sk), dtype=bool)
    m3[0, 2] = False
    got = A.attention(q, k, v, O.F64, D, O.SPLIT_HALF, c, s, pq, pk, False, attn_mask=m3)
    assert np.array_equal(got[0, :, 2], np.zeros((Hq, D)))
    assert np.array_equal(np.delete(got, 2, axis=2)[0],
                          np.delete(A.attention(q, k, v, O.F64, D, O.SPLIT_HALF, c, s, pq, pk), 2,
                                    axis=2)[0])


ALL_PINS = [
    pin_shifting_all_positions_leaves_attention_unchanged,
    pin_constant_values_give_the_constant,
    pin_causal_first_query_sees_only_first_key,
    pin_rows_that_see_no_key_are_zero,
    pin_gqa_equals_repeated_kv_heads,
    pin_key_permutation_invariance,
    pin_unrotated_positions_give_plain_attention_and_zero_scale_averages,
    pin_brute_force_scalar_loops_tiny_case,
    pin_bf16_rotated_rows_are_rounded_before_the_products,
    pin_default_scale_is_inverse_sqrt_d,
    pin_bound_weights_closed_forms,
    pin_attn_mask_hides_keys,
]
