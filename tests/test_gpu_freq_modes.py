"""Frequency modes and XPOS on the GPU against the oracle.

Tables (rope_tables_build_ex): each entry within 1 fp32 ulp of the oracle's
fp64 value plus 2^-48 s (|angle| + |ln s| + 1), s the entry's XPOS scale.
Both sides evaluate pow, sincos and (for XPOS) pow in fp64 with their own
libraries, whose results may differ by a few fp64 ulp: that perturbs the angle
by ~2^-51 |angle| and the scale by ~2^-51 s |ln s|, which only matters near
zeros of cos/sin.  Rotations with XPOS tables: the rotation rule of every
other GPU test (1 ulp of the oracle's once-rounded result, on the same fp32
tables).
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
import attention_check as AC
from gpu_util import assert_matches, gpu_bits, lib, require_gpu

pytestmark = pytest.mark.gpu

MODES = {"lang": O.FREQ_LANG, "pixel": O.FREQ_PIXEL, "constant": O.FREQ_CONSTANT}

TABLE_CASES = [
    dict(mode="lang", rd=128, rows=4096, theta=5e5),
    dict(mode="lang", rd=64, rows=1000, theta=1e4, pos_offset=-7.0, pos_divisor=2.5),
    dict(mode="pixel", rd=64, rows=257, max_freq=224.0, pos_offset=-1.0, pos_divisor=128.0),
    dict(mode="pixel", rd=2, rows=9, max_freq=10.0, pos_offset=-1.0, pos_divisor=4.0),
    dict(mode="constant", rd=16, rows=100, pos_offset=-50.0, pos_divisor=7.0),
    dict(mode="lang", rd=128, rows=4096, theta=5e5, xpos_sign=1, xpos_scale_base=512.0,
         xpos_center=2048.0),
    dict(mode="lang", rd=128, rows=4096, theta=5e5, xpos_sign=-1, xpos_scale_base=512.0,
         xpos_center=2048.0),
    dict(mode="pixel", rd=32, rows=65, max_freq=64.0, pos_offset=-1.0, pos_divisor=32.0,
         xpos_sign=-1, xpos_scale_base=8.0, xpos_gamma=1.5),
]


def _oracle_kwargs(c):
    kw = dict(c)
    mode = MODES[kw.pop("mode")]
    rd, rows = kw.pop("rd"), kw.pop("rows")
    if "xpos_scale_base" in kw:
        kw["xpos_base"] = kw.pop("xpos_scale_base")
    return mode, rd, rows, kw


def _gpu_tables(R, c):
    kw = dict(c)
    return R.build_tables_ex(kw.pop("mode"), kw.pop("rd"), kw.pop("rows"), **kw)


@pytest.mark.parametrize("c", TABLE_CASES, ids=lambda c: "%s_rd%d_rows%d_xpos%d" % (
    c["mode"], c["rd"], c["rows"], c.get("xpos_sign", 0)))
def test_tables_ex_match_oracle(c):
    require_gpu()
    R = lib()
    cos, sin = _gpu_tables(R, c)
    torch.cuda.synchronize()
    mode, rd, rows, kw = _oracle_kwargs(c)
    o = O.load()
    c64, s64 = o.tables_ex(mode, rd, rows, precision="f64", **kw)
    h = rd // 2
    w = np.array([o.freq_ex(mode, kw.get("theta", 1e4), kw.get("max_freq", 10.0), rd, i)
                  for i in range(h)])
    p = kw.get("pos_offset", 0.0) + np.arange(rows, dtype=np.float64) / kw.get("pos_divisor", 1.0)
    angle = np.abs(p[:, None] * w[None, :])
    smag = np.sqrt(c64 * c64 + s64 * s64)
    extra = 2.0 ** -48 * smag * (angle + np.abs(np.log(smag)) + 1.0)
    for name, g, e in (("cos", cos.cpu().numpy(), c64), ("sin", sin.cpu().numpy(), s64)):
        ulp32 = np.spacing(np.abs(e).astype(np.float32)).astype(np.float64)
        err = np.abs(g.astype(np.float64) - e)
        bad = err > ulp32 + extra
        assert not bad.any(), "%s %s: %d entries beyond the bar (max err %.3g)" % (
            c, name, np.count_nonzero(bad), err.max())


def test_lang_mode_is_rope_tables_build_bit_for_bit():
    require_gpu()
    R = lib()
    for f in (1.0, 3.0):
        a = R.build_tables(5e5, 128, 3000, f)
        b = R.build_tables_ex("lang", 128, 3000, theta=5e5, pos_divisor=f)
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def _xpos_inputs(dtype, seed):
    g = torch.Generator().manual_seed(seed)
    q = W.draw((2, 4, 300, 128), dtype, g)
    k = W.draw((2, 2, 300, 128), dtype, g)
    return q, k


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("backward", [False, True])
def test_xpos_rotation_matches_oracle(dtype, backward):
    """Q rotated with the +1 table and K with the -1 table (one launch each),
    on the oracle's fp32 tables, against the oracle's rotation of the same
    bits; backward negates the sine of the same tables."""
    require_gpu()
    R = lib()
    o = O.load()
    kw = dict(theta=1e4, xpos_base=512.0, xpos_center=150.0)
    cq, sq = o.tables_ex(O.FREQ_LANG, 128, 300, xpos_sign=1, precision="f32", **kw)
    ck, sk = o.tables_ex(O.FREQ_LANG, 128, 300, xpos_sign=-1, precision="f32", **kw)
    q, k = _xpos_inputs(dtype, 41)
    qg, kg = q.cuda(), k.cuda()
    tq = (torch.from_numpy(cq).cuda(), torch.from_numpy(sq).cuda())
    tk = (torch.from_numpy(ck).cuda(), torch.from_numpy(sk).cuda())
    R.apply_qk_xpos(qg, kg, tq, tk, backward=backward)
    assert R.rope_check_errors() == R.ROPE_OK
    code = {"f32": O.F32, "bf16": O.BF16, "f16": O.F16}[dtype]
    for name, x, xg, H, c, s in (("q", q, qg, 4, cq, sq), ("k", k, kg, 2, ck, sk)):
        rc, yb, y64 = o.apply(W.bits(x), code, 2, H, 300, 128, 128, O.SPLIT_HALF, False, backward,
                              None, c, s)
        assert rc == O.OK
        assert_matches(dtype, gpu_bits(xg), yb, y64, "xpos %s %s bwd=%d" % (name, dtype, backward))


def test_xpos_scores_depend_on_distance_only():
    """With XPOS tables from the GPU builder, the query-key products of the
    rotated tensors (fp32) are unchanged by a common shift of all positions."""
    require_gpu()
    R = lib()
    rows, S, shift = 600, 64, 200
    tq = R.build_tables_ex("lang", 64, rows, theta=1e4, xpos_sign=1, xpos_scale_base=256.0,
                           xpos_center=300.0)
    tk = R.build_tables_ex("lang", 64, rows, theta=1e4, xpos_sign=-1, xpos_scale_base=256.0,
                           xpos_center=300.0)
    g = torch.Generator().manual_seed(5)
    q0 = torch.randn(1, 1, S, 64, generator=g).cuda()
    k0 = torch.randn(1, 1, S, 64, generator=g).cuda()
    scores = []
    for base in (0, shift):
        pos = torch.arange(base, base + S, dtype=torch.int32).cuda()
        q, k = q0.clone(), k0.clone()
        R.apply_qk_xpos(q, k, tq, tk, pos_idx=pos)
        scores.append((q[0, 0].double() @ k[0, 0].double().T).cpu())
    assert R.rope_check_errors() == R.ROPE_OK
    ref = float(scores[0].abs().max())
    assert float((scores[0] - scores[1]).abs().max()) <= 1e-5 * ref


def test_attention_with_pixel_tables():
    """The fused attention with a pixel-mode table (two-dimensional image
    positions flattened to rows of one table, gathered by pos_q / pos_k)."""
    require_gpu()
    R = lib()
    from oracle import attention as OA

    o = O.load()
    c32, s32 = o.tables_ex(O.FREQ_PIXEL, 64, 33, max_freq=32.0, pos_offset=-1.0, pos_divisor=16.0,
                           precision="f32")
    g = torch.Generator().manual_seed(23)
    S = 200
    q = W.draw((1, 2, S, 64), "bf16", g)
    k = W.draw((1, 2, S, 64), "bf16", g)
    v = W.draw((1, 2, S, 64), "bf16", g)
    pos = np.random.default_rng(2).integers(0, 33, S).astype(np.int32)
    pg = torch.from_numpy(pos).cuda()
    out = R.attention(q.cuda(), k.cuda(), v.cuda(), torch.from_numpy(c32).cuda(),
                      torch.from_numpy(s32).cuda(), pos_q=pg, pos_k=pg, rotary_dim=64, causal=False)
    assert R.rope_check_errors() == R.ROPE_OK
    ref, w, a = OA.attention(W.bits(q), W.bits(k), W.bits(v), O.BF16, 64, O.SPLIT_HALF, c32, s32,
                             pos, pos, False, want_bounds=True)
    AC.check(out.float().cpu().numpy(), ref, w, a, "bf16", "pixel tables")


def _table_fuzz(n=16, seed=77):
    g = np.random.default_rng(seed)
    out = []
    for i in range(n):
        mode = str(g.choice(["lang", "pixel", "constant"]))
        c = dict(mode=mode, rd=2 * int(g.integers(1, 65)), rows=int(g.integers(1, 3000)),
                 pos_offset=float(g.uniform(-100, 100)), pos_divisor=float(g.uniform(0.25, 8.0)))
        if mode == "lang":
            c["theta"] = float(10 ** g.uniform(2, 6))
        if mode == "pixel":
            c["max_freq"] = float(g.uniform(1.0, 256.0))
        if g.integers(0, 2):
            # a base of at least the rows' largest distance from the centre keeps
            # the scale within [zeta, 1 / zeta], inside fp32's range
            centre = float(g.uniform(-50, 50))
            p_lo = c["pos_offset"]
            p_hi = c["pos_offset"] + (c["rows"] - 1) / c["pos_divisor"]
            reach = max(abs(p_lo - centre), abs(p_hi - centre), 1.0)
            c.update(xpos_sign=int(g.choice([-1, 1])), xpos_scale_base=reach * float(g.uniform(1, 4)),
                     xpos_gamma=float(g.uniform(0.1, 2.0)), xpos_center=centre)
        out.append(c)
    return out


@pytest.mark.parametrize("c", _table_fuzz(), ids=lambda c: "%s_rd%d_rows%d_x%d" % (
    c["mode"], c["rd"], c["rows"], c.get("xpos_sign", 0)))
def test_tables_ex_fuzz(c):
    """Seeded random modes, widths, positions and XPOS parameters."""
    test_tables_ex_match_oracle(c)
