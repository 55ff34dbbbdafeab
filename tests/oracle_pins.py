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
    backward after forward, relative-position property, layout permutation;
  * defining properties of the frequency modes and of XPOS: linear pixel
    spacing with fixed endpoints, the constant mode's closed form, query and
    key scales that cancel, a log-scale linear in the position, an affine
    zeta reaching 1, and the relative-position property with scaling.
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


# --------------------------------------------------------------------------
# frequency modes, row positions and the XPOS scale
# ("rotary-embedding-torch", RotaryEmbedding / Key Parameters names them;
# Perceiver's Fourier features and the XPOS paper define them)
# --------------------------------------------------------------------------
def pin_freq_lang_mode_is_the_plain_table(o):
    # lang mode at positions m / f is exactly the table of rope_tables_build
    for f in (1.0, 2.0, 3.0):
        for prec in ("f64", "f32"):
            c0, s0 = o.tables(1e4, 64, 50, f, prec)
            c1, s1 = o.tables_ex(O.FREQ_LANG, 64, 50, theta=1e4, pos_divisor=f, precision=prec)
            assert np.array_equal(c0, c1) and np.array_equal(s0, s1), (f, prec)


def pin_freq_constant_mode_closed_form(o):
    # every pair turns at frequency 1: the angle is the position itself
    c, s = o.tables_ex(O.FREQ_CONSTANT, 8, 20, pos_offset=-3.5, pos_divisor=4.0)
    for m in range(20):
        p = -3.5 + m / 4.0
        assert np.all(np.abs(c[m] - math.cos(p)) <= 1e-15) and np.all(np.abs(s[m] - math.sin(p)) <= 1e-15)
    with_theta = o.tables_ex(O.FREQ_CONSTANT, 8, 20, theta=3.0, pos_offset=-3.5, pos_divisor=4.0)
    assert np.array_equal(with_theta[0], c)            # theta plays no part


def pin_freq_pixel_mode_spacing(o):
    # Perceiver: frequencies spaced linearly from 1 to max_freq / 2, times pi
    for mu, rd in ((10.0, 16), (224.0, 64), (3.0, 4)):
        h = rd // 2
        w = np.array([o.freq_ex(O.FREQ_PIXEL, 1e4, mu, rd, i) for i in range(h)])
        assert abs(w[0] - math.pi) <= 1e-15 * math.pi
        assert abs(w[-1] - math.pi * mu / 2) <= 4e-16 * math.pi * mu
        d = np.diff(w)
        assert np.all(np.abs(d - d[0]) <= 1e-13 * abs(w[-1])), (mu, rd)
    assert o.freq_ex(O.FREQ_PIXEL, 1e4, 10.0, 2, 0) == math.pi      # one pair: the start
    # max_freq 2: every frequency is pi, so positions -1 and 1 give cos = -1, sin ~ 0
    c, s = o.tables_ex(O.FREQ_PIXEL, 8, 2, max_freq=2.0, pos_offset=-1.0, pos_divisor=0.5)
    assert np.all(np.abs(c + 1.0) <= 1e-15) and np.all(np.abs(s) <= 1e-15)
    # positions span [-1, 1] with divisor (rows - 1) / 2
    assert o.position(0, -1.0, 3.5) == -1.0 and o.position(7, -1.0, 3.5) == 1.0


def _xpos_magnitude(c, s):
    return np.sqrt(c * c + s * s)


def pin_xpos_identity_at_centre(o):
    # at the centre the scale is zeta^0 = 1: the table is the unscaled one
    base = o.tables_ex(O.FREQ_LANG, 16, 9, theta=1e4, pos_offset=0.0)
    for sign in (1, -1):
        xs = o.tables_ex(O.FREQ_LANG, 16, 9, theta=1e4, xpos_sign=sign, xpos_center=4.0)
        assert np.array_equal(xs[0][4], base[0][4]) and np.array_equal(xs[1][4], base[1][4])


def pin_xpos_query_key_scales_cancel(o):
    # the query is scaled by zeta^(n/B) and the key by zeta^(-n/B): at one
    # position the magnitudes multiply to 1, and the phases are the plain ones
    kw = dict(theta=1e4, xpos_base=64.0, xpos_center=10.0)
    cq, sq = o.tables_ex(O.FREQ_LANG, 32, 40, xpos_sign=1, **kw)
    ck, sk = o.tables_ex(O.FREQ_LANG, 32, 40, xpos_sign=-1, **kw)
    c0, s0 = o.tables_ex(O.FREQ_LANG, 32, 40, theta=1e4)
    assert np.all(np.abs(_xpos_magnitude(cq, sq) * _xpos_magnitude(ck, sk) - 1.0) <= 1e-13)
    assert np.all(np.abs(np.arctan2(sq, cq) - np.arctan2(s0, c0)) <= 1e-13)
    # past the centre the query shrinks and the key grows (zeta < 1)
    mq = _xpos_magnitude(cq, sq)
    assert np.all(mq[11:] < 1.0) and np.all(mq[:10] > 1.0)


def pin_xpos_log_scale_linear_in_position(o):
    # log|scale| = (p - c) / B * log(zeta): linear in p, with slope 1/B
    for B in (8.0, 512.0):
        c, s = o.tables_ex(O.FREQ_CONSTANT, 16, 30, pos_divisor=1.0, xpos_sign=1, xpos_base=B,
                           xpos_center=3.0)
        L = np.log(_xpos_magnitude(c, s))                # [rows, pairs]
        assert np.all(np.abs(np.diff(L, n=2, axis=0)) <= 1e-12)
        # one base length past the centre, the scale is zeta itself, whatever B is
        cB, sB = o.tables_ex(O.FREQ_CONSTANT, 16, 1, pos_offset=3.0 + B, xpos_sign=1, xpos_base=B,
                             xpos_center=3.0)
        z = _xpos_magnitude(cB, sB)[0]
        if B == 8.0:
            z8 = z
        else:
            assert np.all(np.abs(z - z8) <= 1e-14)


def pin_xpos_zeta_affine_reaching_one(o):
    # zeta_i is affine in i/rd, zeta_0 / (1 - zeta_0) = gamma, and it would
    # reach exactly 1 at i = rd/2 (one pair past the last)
    for rd, gamma in ((16, 0.4), (64, 0.4), (8, 1.5)):
        h = rd // 2
        z = np.array([o.xpos_scale(rd, i, 1.0, 1, 1.0, gamma, 0.0) for i in range(h)])
        d = np.diff(z)
        assert np.all(np.abs(d - d[0]) <= 1e-15), (rd, gamma)
        assert abs(z[-1] + d[0] - 1.0) <= 1e-14
        assert abs(z[0] / (1.0 - z[0]) - gamma) <= 1e-14
    # the same fraction i / rd gives the same zeta
    assert o.xpos_scale(16, 3, 1.0, 1, 1.0, 0.4, 0.0) == o.xpos_scale(32, 6, 1.0, 1, 1.0, 0.4, 0.0)


def pin_xpos_relative_position(o):
    # <f_q(q, m), f_k(k, n)> depends on m - n only (brute force)
    rows, rd = 64, 16
    kw = dict(theta=1e4, xpos_base=32.0, xpos_center=0.0)
    cq, sq = o.tables_ex(O.FREQ_LANG, rd, rows, xpos_sign=1, **kw)
    ck, sk = o.tables_ex(O.FREQ_LANG, rd, rows, xpos_sign=-1, **kw)
    g = np.random.default_rng(17)
    q, k = g.standard_normal(rd), g.standard_normal(rd)
    for layout in (O.SPLIT_HALF, O.INTERLEAVED):
        xq = np.broadcast_to(q, (1, 1, rows, rd)).copy()
        xk = np.broadcast_to(k, (1, 1, rows, rd)).copy()
        _, rq = _apply64(o, xq, rd, layout, False, False, None, cq, sq)
        _, rk = _apply64(o, xk, rd, layout, False, False, None, ck, sk)
        G = rq[0, 0] @ rk[0, 0].T
        tol = 1e-11 * np.linalg.norm(q) * np.linalg.norm(k)
        for t in range(32):
            assert np.all(np.abs(G[t:t + 32, t:t + 32] - G[:32, :32]) <= tol), (layout, t)
        # a plain rotation of the key breaks it
        c0, s0 = o.tables_ex(O.FREQ_LANG, rd, rows, theta=1e4)
        _, rk0 = _apply64(o, xk, rd, layout, False, False, None, c0, s0)
        G0 = rq[0, 0] @ rk0[0, 0].T
        assert np.max(np.abs(G0[5:37, 5:37] - G0[:32, :32])) > 1e-6


def pin_tables_ex_rejects_bad_arguments(o):
    good = dict(theta=1e4, max_freq=10.0, pos_offset=0.0, pos_divisor=1.0, xpos_sign=0,
                xpos_base=512.0, xpos_gamma=0.4, xpos_center=0.0)
    bad = [(3, {}), (O.FREQ_LANG, dict(theta=0.0)), (O.FREQ_PIXEL, dict(max_freq=-1.0)),
           (O.FREQ_LANG, dict(pos_divisor=0.0)), (O.FREQ_LANG, dict(pos_offset=float("nan"))),
           (O.FREQ_LANG, dict(xpos_sign=2)), (O.FREQ_LANG, dict(xpos_sign=1, xpos_base=0.0)),
           (O.FREQ_LANG, dict(xpos_sign=-1, xpos_gamma=0.0))]
    for mode, over in bad:
        args = dict(good, **over)
        try:
            o.tables_ex(mode, 8, 4, **args)
        except ValueError:
            continue
        raise AssertionError("accepted %r %r" % (mode, over))
    o.tables_ex(O.FREQ_PIXEL, 8, 4, **dict(good, theta=0.0))   # theta unused by pixel mode


def pin_tables_ex_f32_is_f64_rounded_once(o):
    # the stored fp32 tables of every mode, scaled or not, are the fp64 ones
    # rounded once to nearest (numpy's conversion)
    cases = [dict(mode=O.FREQ_LANG, theta=5e5), dict(mode=O.FREQ_PIXEL, max_freq=64.0, pos_offset=-1.0,
                                                     pos_divisor=15.5),
             dict(mode=O.FREQ_CONSTANT, pos_offset=2.0), dict(mode=O.FREQ_LANG, xpos_sign=1, xpos_center=7.0),
             dict(mode=O.FREQ_PIXEL, xpos_sign=-1, xpos_base=16.0, pos_divisor=3.0)]
    for kw in cases:
        kw = dict(kw)
        mode = kw.pop("mode")
        c64, s64 = o.tables_ex(mode, 32, 32, precision="f64", **kw)
        c32, s32 = o.tables_ex(mode, 32, 32, precision="f32", **kw)
        assert np.array_equal(c64.astype(np.float32), c32) and np.array_equal(s64.astype(np.float32), s32), kw


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
