"""Pins for the CPU oracle: checks against facts fixed outside the oracle.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when the oracle disagrees with what the pages or mathematics fix.  The same
functions run against the real oracle (all must pass) and against mutated
copies of it (at least one must fail), see test_oracle_mutants.py.

Independent references used here:
  * library routines: torch (bfloat16 decode), numpy (float16 / float32
    conversions), Python's complex arithmetic and ``math.cos``/``math.sin``;
  * brute force: nearest representable value found by exact rational
    comparison over the full list of finite bfloat16 / float16 values;
  * closed forms evaluated with sympy at 40 significant digits;
  * invariants of a rotation: identity at position 0, norm preservation,
    backward after forward, relative-position property, layout permutation.
"""
from __future__ import annotations

import bisect
import math
from fractions import Fraction

import numpy as np

import oracle as O

RNG_SEED = 1234


# --------------------------------------------------------------------------
# helpers (no oracle arithmetic repeated here)
# --------------------------------------------------------------------------
def _finite_values(kind: str):
    """All non-negative finite values of a 16-bit format, ascending, as floats,
    decoded by a library routine."""
    import torch

    if kind == "bf16":
        b = np.arange(0, 0x7F80, dtype=np.int32).astype(np.int16)
        vals = torch.from_numpy(b).view(torch.bfloat16).to(torch.float64).numpy()
    else:
        b = np.arange(0, 0x7C00, dtype=np.uint16)
        vals = b.view(np.float16).astype(np.float64)
    return list(vals), list(range(len(vals)))


_TABLES = {}


def _values(kind):
    if kind not in _TABLES:
        _TABLES[kind] = _finite_values(kind)
    return _TABLES[kind]


def _bruteforce_rne(y: float, kind: str) -> int:
    """Bits of the nearest value of the format to y (ties to even mantissa),
    overflow to infinity per IEEE 754 round-to-nearest."""
    vals, codes = _values(kind)
    inf_bits = 0x7F80 if kind == "bf16" else 0x7C00
    sign = 0x8000 if math.copysign(1.0, y) < 0 else 0
    a = abs(y)
    top = vals[-1]
    ulp_top = top - vals[-2]
    if Fraction(a) >= Fraction(top) + Fraction(ulp_top) / 2:
        return sign | inf_bits
    j = bisect.bisect_left(vals, a)
    if j < len(vals) and vals[j] == a:
        return sign | codes[j]
    lo, hi = vals[j - 1], vals[j] if j < len(vals) else None
    if hi is None:
        return sign | codes[j - 1]
    dlo = Fraction(a) - Fraction(lo)
    dhi = Fraction(hi) - Fraction(a)
    if dlo < dhi:
        return sign | codes[j - 1]
    if dhi < dlo:
        return sign | codes[j]
    return sign | (codes[j - 1] if codes[j - 1] % 2 == 0 else codes[j])


def _rounding_probes(kind: str, n_random: int, seed: int):
    """Doubles covering the whole range of a 16-bit format: random values,
    exact midpoints, midpoints +/- one fp64 ulp, extremes."""
    rng = np.random.default_rng(seed)
    vals, _ = _values(kind)
    lo_exp, hi_exp = (-140, 130) if kind == "bf16" else (-27, 17)
    out = list(rng.uniform(1, 2, n_random) * np.exp2(rng.integers(lo_exp, hi_exp, n_random)))
    idx = rng.integers(0, len(vals) - 1, n_random)
    for j in idx:
        mid = (vals[j] + vals[j + 1]) / 2          # exact in fp64
        out += [mid, np.nextafter(mid, 0.0), np.nextafter(mid, np.inf)]
    top = vals[-1]
    half = (top - vals[-2]) / 2
    out += [0.0, vals[1], vals[1] / 2, vals[1] / 4, top, top + half,
            np.nextafter(top + half, 0.0), top * 4, 1.0, 1.5]
    out = np.array(out, dtype=np.float64)
    signs = np.where(rng.random(out.size) < 0.5, -1.0, 1.0)
    return out * signs


def _tensor_f64(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _apply64(o, x, rd, layout, seq_first, backward, pos, cos, sin):
    """Run the oracle on an fp64 tensor of shape [B,H,S,D] (or [B,S,H,D])."""
    if seq_first:
        B, S, H, D = x.shape
    else:
        B, H, S, D = x.shape
    rc, _, y = o.apply(x, O.F64, B, H, S, D, rd, layout, seq_first, backward, pos,
                       cos, sin, want_bits=False)
    return rc, y


# --------------------------------------------------------------------------
# pins: number formats
# --------------------------------------------------------------------------
def pin_decode_bf16_all(o):
    import torch

    b = np.arange(0, 65536, dtype=np.int32).astype(np.int16)
    ref = torch.from_numpy(b).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([o.bf16_to_f64(int(v) & 0xFFFF) for v in b], dtype=np.float64)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    m = ~np.isnan(ref)
    assert np.array_equal(ref[m], got[m])
    assert np.array_equal(np.signbit(ref[m]), np.signbit(got[m]))


def pin_decode_f16_all(o):
    b = np.arange(0, 65536, dtype=np.uint32).astype(np.uint16)
    ref = b.view(np.float16).astype(np.float64)
    got = np.array([o.f16_to_f64(int(v)) for v in b], dtype=np.float64)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    m = ~np.isnan(ref)
    assert np.array_equal(ref[m], got[m])
    assert np.array_equal(np.signbit(ref[m]), np.signbit(got[m]))


def pin_round_bf16_bruteforce(o):
    for y in _rounding_probes("bf16", 400, RNG_SEED):
        want = _bruteforce_rne(float(y), "bf16")
        got = o.f64_to_bf16(float(y))
        assert got == want, (float(y).hex(), hex(got), hex(want))


def pin_round_f16_bruteforce(o):
    for y in _rounding_probes("f16", 400, RNG_SEED + 1):
        want = _bruteforce_rne(float(y), "f16")
        got = o.f64_to_f16(float(y))
        assert got == want, (float(y).hex(), hex(got), hex(want))


def pin_round_f16_numpy(o):
    y = _rounding_probes("f16", 3000, RNG_SEED + 2)
    with np.errstate(over="ignore"):
        ref = y.astype(np.float16).view(np.uint16)
    got = np.array([o.f64_to_f16(float(v)) for v in y], dtype=np.uint16)
    assert np.array_equal(ref, got)


def pin_round_f32_numpy(o):
    rng = np.random.default_rng(RNG_SEED + 3)
    y = rng.standard_normal(5000) * np.exp2(rng.integers(-60, 60, 5000))
    ref = y.astype(np.float32)
    got = np.array([o.f64_to_f32(float(v)) for v in y], dtype=np.float32)
    assert np.array_equal(ref.view(np.uint32), got.view(np.uint32))


# --------------------------------------------------------------------------
# pins: frequencies and tables
# --------------------------------------------------------------------------
def _exact_inv(theta, rd, i, digits=40):
    import sympy

    return sympy.N(sympy.Integer(int(theta)) ** sympy.Rational(-2 * i, rd), digits)


def pin_inv_freq_closed_form(o):
    import sympy  # noqa: F401  (pin needs it; skip cleanly if absent)

    for theta in (10.0, 1e4, 5e5):
        for rd in (2, 8, 32, 64, 128):
            h = rd // 2
            assert o.inv_freq(theta, rd, 0) == 1.0           # theta^0 exactly
            for i in sorted({0, 1, h // 2, h - 1}):
                exact = float(_exact_inv(theta, rd, i))
                got = o.inv_freq(theta, rd, i)
                assert abs(got - exact) <= 2 * math.ulp(exact), (theta, rd, i, got, exact)


def pin_angle_first_pair_is_position(o):
    # pair 0 has frequency 1: its angle is the (scaled) position itself
    for m in (0, 1, 7, 4095, 262143):
        for f in (1.0, 2.0, 4.0):
            assert o.angle(m, f, o.inv_freq(5e5, 128, 0)) == m / f


def pin_tables_high_precision(o):
    import sympy

    rng = np.random.default_rng(RNG_SEED + 4)
    for theta, rd, rows, f in ((1e4, 64, 128, 1.0), (5e5, 128, 262144, 1.0),
                               (1e4, 32, 8192, 2.0)):
        h = rd // 2
        ms = sorted({0, 1, rows - 1, *rng.integers(0, rows, 6).tolist()})
        c64, s64 = o.tables(theta, rd, rows, f, "f64")
        c32, s32 = o.tables(theta, rd, rows, f, "f32")
        for m in ms:
            for i in sorted({0, 1, h - 1, int(rng.integers(0, h))}):
                ang = sympy.Rational(m) / sympy.Rational(f) * _exact_inv(theta, rd, i, 45)
                ec = float(sympy.cos(ang).evalf(40))
                es = float(sympy.sin(ang).evalf(40))
                tol64 = 4 * 2.0 ** -52 * (abs(float(ang)) + 1.0)
                assert abs(c64[m, i] - ec) <= tol64, (theta, rd, m, i, c64[m, i], ec)
                assert abs(s64[m, i] - es) <= tol64, (theta, rd, m, i, s64[m, i], es)
                tol32 = tol64 + 2.0 ** -24
                assert abs(float(c32[m, i]) - ec) <= tol32
                assert abs(float(s32[m, i]) - es) <= tol32
        # the fp32 table is the fp64 table rounded once (library conversion)
        assert np.array_equal(c64.astype(np.float32), c32)
        assert np.array_equal(s64.astype(np.float32), s32)


def pin_interpolate_factor_scales_positions(o):
    # position m with factor 2 has the angles of position m/2 with factor 1
    c2, s2 = o.tables(1e4, 64, 256, 2.0, "f64")
    c1, s1 = o.tables(1e4, 64, 128, 1.0, "f64")
    assert np.array_equal(c2[0::2], c1) and np.array_equal(s2[0::2], s1)


# --------------------------------------------------------------------------
# pins: the rotation
# --------------------------------------------------------------------------
def pin_rd2_rotates_by_position(o):
    # one pair, frequency theta^0 = 1: position m rotates by exactly m radians
    for theta in (10.0, 1e4, 5e5):
        S = 50
        c, s = o.tables(theta, 2, S, 1.0, "f64")
        x = _tensor_f64((1, 1, S, 2), 7)
        rc, y = _apply64(o, x, 2, O.SPLIT_HALF, False, False, None, c, s)
        assert rc == O.OK
        for m in range(S):
            x1, x2 = x[0, 0, m]
            want = (x1 * math.cos(m) - x2 * math.sin(m), x1 * math.sin(m) + x2 * math.cos(m))
            assert abs(y[0, 0, m, 0] - want[0]) <= 1e-14 and abs(y[0, 0, m, 1] - want[1]) <= 1e-14


def pin_complex_multiply(o):
    # an interleaved pair is the complex number x1 + i x2 times exp(i angle)
    import cmath

    rd, D, S = 16, 16, 40
    c, s = o.tables(1e4, rd, S, 1.0, "f64")
    x = _tensor_f64((1, 2, S, D), 11)
    for backward in (False, True):
        rc, y = _apply64(o, x, rd, O.INTERLEAVED, False, backward, None, c, s)
        assert rc == O.OK
        for h in range(2):
            for m in range(S):
                for i in range(rd // 2):
                    ang = o.angle(m, 1.0, o.inv_freq(1e4, rd, i))
                    z = complex(x[0, h, m, 2 * i], x[0, h, m, 2 * i + 1]) * cmath.rect(
                        1.0, -ang if backward else ang)
                    tol = 4e-16 * (abs(z) + 1e-300)
                    assert abs(y[0, h, m, 2 * i] - z.real) <= tol
                    assert abs(y[0, h, m, 2 * i + 1] - z.imag) <= tol


def pin_position_zero_identity(o):
    c, s = o.tables(5e5, 128, 4, 1.0, "f32")
    g = np.random.default_rng(3)
    x = g.standard_normal((2, 3, 1, 128)).astype(np.float32)
    for layout in (O.SPLIT_HALF, O.INTERLEAVED):
        for dt, xb in ((O.F32, x), (O.F16, x.astype(np.float16).view(np.uint16))):
            rc, yb, y64 = o.apply(xb, dt, 2, 3, 1, 128, 128, layout, False, False, None, c, s)
            assert rc == O.OK
            ref = x if dt == O.F32 else xb.view(np.float16).astype(np.float32)
            assert np.array_equal(y64, ref.astype(np.float64))


def pin_norm_preserved(o):
    rd, D, S = 64, 64, 300
    c, s = o.tables(1e4, rd, S, 1.0, "f64")
    x = _tensor_f64((2, 3, S, D), 5)
    for layout in (O.SPLIT_HALF, O.INTERLEAVED):
        rc, y = _apply64(o, x, rd, layout, False, False, None, c, s)
        assert rc == O.OK
        if layout == O.SPLIT_HALF:
            nx = x[..., :32] ** 2 + x[..., 32:] ** 2
            ny = y[..., :32] ** 2 + y[..., 32:] ** 2
        else:
            nx = x[..., 0::2] ** 2 + x[..., 1::2] ** 2
            ny = y[..., 0::2] ** 2 + y[..., 1::2] ** 2
        assert np.all(np.abs(ny - nx) <= 1e-15 * nx + 1e-300)
        assert not np.allclose(y, x)       # it did rotate


def pin_backward_inverts_forward(o):
    rd, D, S = 32, 48, 200
    c, s = o.tables(1e4, rd, S, 1.0, "f64")
    x = _tensor_f64((1, 4, S, D), 9)
    for layout in (O.SPLIT_HALF, O.INTERLEAVED):
        _, y = _apply64(o, x, rd, layout, False, False, None, c, s)
        _, z = _apply64(o, y, rd, layout, False, True, None, c, s)
        assert np.all(np.abs(z - x) <= 1e-15 * (np.abs(x).max() + 1))
        _, y_b = _apply64(o, x, rd, layout, False, True, None, c, s)
        assert not np.allclose(y_b, y)      # backward is not forward


def pin_backward_is_negated_sin(o):
    rd, D, S = 64, 64, 64
    c, s = o.tables(1e4, rd, S, 1.0, "f32")
    x = np.random.default_rng(2).standard_normal((1, 2, S, D)).astype(np.float32)
    xb = x.astype(np.float16).view(np.uint16)
    for layout in (O.SPLIT_HALF, O.INTERLEAVED):
        _, b1, _ = o.apply(xb, O.F16, 1, 2, S, D, rd, layout, False, True, None, c, s)
        _, b2, _ = o.apply(xb, O.F16, 1, 2, S, D, rd, layout, False, False, None, c, -s)
        assert np.array_equal(b1, b2)


def pin_relative_position(o):
    # <R_m q, R_n k> depends on m - n only: brute force over tiny inputs
    rows = 96
    for rd in (2, 8, 64):
        c, s = o.tables(1e4, rd, rows, 1.0, "f64")
        g = np.random.default_rng(rd)
        q = g.standard_normal(rd)
        k = g.standard_normal(rd)
        for layout in (O.SPLIT_HALF, O.INTERLEAVED):
            xq = np.broadcast_to(q, (1, 1, rows, rd)).copy()
            xk = np.broadcast_to(k, (1, 1, rows, rd)).copy()
            _, rq = _apply64(o, xq, rd, layout, False, False, None, c, s)
            _, rk = _apply64(o, xk, rd, layout, False, False, None, c, s)
            G = rq[0, 0] @ rk[0, 0].T                    # G[m, n] = <R_m q, R_n k>
            tol = 1e-12 * np.linalg.norm(q) * np.linalg.norm(k)
            for t in range(64):
                assert np.all(np.abs(G[t:t + 32, t:t + 32] - G[:32, :32]) <= tol), (rd, layout, t)
            assert not np.allclose(G[0, 1], G[0, 2])      # it is not trivially constant


def pin_layout_permutation(o):
    # split-half of x equals interleaved of P x, with P: 2i -> i, 2i+1 -> i+h
    rd, D, S = 32, 40, 50
    h = rd // 2
    c, s = o.tables(1e4, rd, S, 1.0, "f64")
    x = _tensor_f64((2, 2, S, D), 13)
    perm = np.arange(D)
    perm[0:rd:2] = np.arange(h)
    perm[1:rd:2] = np.arange(h) + h             # interleaved slot j takes split-half element perm[j]
    _, ys = _apply64(o, x, rd, O.SPLIT_HALF, False, False, None, c, s)
    _, yi = _apply64(o, x[..., perm], rd, O.INTERLEAVED, False, False, None, c, s)
    assert np.array_equal(yi, ys[..., perm])


def pin_seq_before_head_transpose(o):
    rd, D, S = 16, 16, 30
    c, s = o.tables(1e4, rd, S, 1.0, "f64")
    x = _tensor_f64((2, 3, S, D), 17)                  # [B,H,S,D]
    pos = np.random.default_rng(0).integers(0, S, S).astype(np.int32)
    _, y = _apply64(o, x, rd, O.SPLIT_HALF, False, False, pos, c, s)
    xt = np.ascontiguousarray(x.transpose(0, 2, 1, 3))  # [B,S,H,D]
    _, yt = _apply64(o, xt, rd, O.SPLIT_HALF, True, False, pos, c, s)
    assert np.array_equal(yt, y.transpose(0, 2, 1, 3))


def pin_gather_prefix_shift(o):
    # "Custom Position IDs for Prefix-Tuning": ids = arange(S) + prefix_len
    # equals rows 0..S-1 of the table shifted by prefix_len
    rd, D, S, p = 32, 64, 40, 7
    c, s = o.tables(1e4, rd, S + p, 1.0, "f32")
    x = np.random.default_rng(4).standard_normal((1, 2, S, D)).astype(np.float32)
    xb = x.astype(np.float16).view(np.uint16)
    ids = (np.arange(S) + p).astype(np.int32)
    _, a, _ = o.apply(xb, O.F16, 1, 2, S, D, rd, O.SPLIT_HALF, False, False, ids, c, s)
    _, b, _ = o.apply(xb, O.F16, 1, 2, S, D, rd, O.SPLIT_HALF, False, False, None, c[p:], s[p:])
    assert np.array_equal(a, b)
    _, z, _ = o.apply(xb, O.F16, 1, 2, S, D, rd, O.SPLIT_HALF, False, False, None, c, s)
    assert not np.array_equal(a, z)


def pin_tail_and_mask_passthrough(o):
    rd, D, S = 32, 64, 12
    c, s = o.tables(1e4, rd, 64, 1.0, "f32")
    x = np.random.default_rng(6).standard_normal((2, 3, S, D)).astype(np.float32)
    xb = x.astype(np.float16).view(np.uint16).copy()
    xb.reshape(-1)[::97] = 0x8000            # some negative zeros, which arithmetic would turn to +0
    pos = np.arange(-2, S - 2, dtype=np.int32)
    pos[:2] = -1
    pos[5] = -1
    for layout in (O.SPLIT_HALF, O.INTERLEAVED):
        rc, yb, _ = o.apply(xb, O.F16, 2, 3, S, D, rd, layout, False, False, pos, c, s)
        assert rc == O.OK
        assert np.array_equal(yb[..., rd:], xb[..., rd:])            # tail untouched
        assert np.array_equal(yb[:, :, pos == -1], xb[:, :, pos == -1])  # masked tokens untouched
        assert not np.array_equal(yb[:, :, 3, :rd], xb[:, :, 3, :rd])


def pin_out_of_range_rejected(o):
    rd, D, S = 8, 8, 6
    c, s = o.tables(1e4, rd, 10, 1.0, "f64")
    x = _tensor_f64((1, 1, S, D), 1)
    for bad in (10, -2, 1 << 30):
        pos = np.arange(S, dtype=np.int32)
        pos[3] = bad
        rc, y = _apply64(o, x, rd, O.SPLIT_HALF, False, False, pos, c, s)
        assert rc == O.POS_OUT_OF_RANGE
        assert np.array_equal(y[0, 0, 3], x[0, 0, 3])


def pin_rounded_outputs_are_rne_of_f64(o):
    rd, D, S = 64, 64, 64
    c, s = o.tables(1e4, rd, S, 1.0, "f32")
    x = np.random.default_rng(8).standard_normal((1, 2, S, D)).astype(np.float32)
    # fp32 and fp16: library conversions of the fp64 result
    rc, y32, y64 = o.apply(x, O.F32, 1, 2, S, D, rd, O.SPLIT_HALF, False, False, None, c, s)
    assert np.array_equal(y32, y64.astype(np.float32))
    xh = x.astype(np.float16).view(np.uint16)
    rc, y16, y64 = o.apply(xh, O.F16, 1, 2, S, D, rd, O.SPLIT_HALF, False, False, None, c, s)
    assert np.array_equal(y16, y64.astype(np.float16).view(np.uint16))
    # bf16: brute force on a sample
    import torch

    xb = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    rc, yb, y64 = o.apply(xb, O.BF16, 1, 2, S, D, rd, O.SPLIT_HALF, False, False, None, c, s)
    flat_b, flat_y = yb.reshape(-1), y64.reshape(-1)
    for j in np.random.default_rng(9).integers(0, flat_y.size, 300):
        assert flat_b[j] == _bruteforce_rne(float(flat_y[j]), "bf16")


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
