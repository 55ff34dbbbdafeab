"""CUDA library against the CPU oracle on the five workloads.

* Tables: every entry of the GPU-built cos/sin table within one fp32 ulp of
  the oracle's fp64 value (and the count of entries that differ from the
  oracle's own fp32 rounding is reported).
* Rotation at reduced sizes (several tiles, ragged last tile): every output
  element compared, forward and backward.
* Rotation at full sizes, in the bench's launch configuration: sampled rows
  compared with the oracle, and the pass-through properties checked on every
  element.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from gpu_util import (all_finite16, assert_matches, gpu_bits, lib, oracle_apply, oracle_tables, pos_tensor,
                      require_gpu, run_apply)

pytestmark = pytest.mark.gpu

NAMES = [w.name for w in W.WORKLOADS]
# reduced sizes: several CTAs per batch with a ragged last tile
REDUCED = {
    "tiny_f32_split_half": {},
    "llama3_8b_gqa_bf16": dict(B=2, S=333),
    "interleaved_f16_bshd": dict(B=2, S=157),
    "partial_rd32_masked_bf16": dict(B=3),
    "long_context_gqa_bf16": dict(S=777),
}


def seq_axis(w):
    return 1 if w.seq_before_head else 2


def check_tensor(w, x_cpu, x_gpu, H, pos, backward, cos32, sin32, what):
    xb = W.bits(x_cpu)
    got = gpu_bits(x_gpu)
    yb, y64 = oracle_apply(w, xb, H, pos, backward, cos32, sin32)
    assert_matches(w.dtype, got, yb, y64, what)
    if w.dtype == "f32":
        c64, s64 = oracle_tables(w.theta, w.rotary_dim, w.table_rows, w.interpolate_factor, "f64")
        _, y64_exact = oracle_apply(w, xb, H, pos, backward, c64, s64)
        assert_matches("f32", got, None, y64_exact, what + " (fp64 cos/sin)")
    # pass-through: tail features and masked tokens keep their bits
    assert np.array_equal(got[..., w.rotary_dim:], xb[..., w.rotary_dim:]), what
    if pos is not None and np.any(pos == -1):
        idx = np.flatnonzero(pos == -1)
        assert np.array_equal(np.take(got, idx, axis=seq_axis(w)),
                              np.take(xb, idx, axis=seq_axis(w))), what


@pytest.mark.parametrize("theta,rd,rows,f", sorted(
    {(w.theta, w.rotary_dim, w.table_rows, w.interpolate_factor) for w in W.WORKLOADS}
    | {(1e4, 2, 1, 1.0), (1e4, 6, 37, 2.0), (10.0, 130, 100, 1.0), (5e5, 128, 5000, 4.0)}))
def test_table_matches_oracle(theta, rd, rows, f):
    require_gpu()
    R = lib()
    cos, sin = R.build_tables(theta, rd, rows, f)
    torch.cuda.synchronize()
    c64, s64 = oracle_tables(theta, rd, rows, f, "f64")
    # Both sides evaluate theta^(-2i/rd) with their platform's fp64 pow (CUDA:
    # within 2 ulp; glibc: within 1), so their fp64 angles may differ by up to
    # about 2^-51 |angle|, and cos/sin by as much.  Bar per entry: 1 fp32 ulp
    # of the oracle's fp64 value plus 2^-50 |angle|.  The angle term matters
    # only near zeros of cos/sin at large angles (long-context tables).
    h = rd // 2
    angle = (np.arange(rows, dtype=np.float64)[:, None] / f) * \
        np.power(float(theta), -2.0 * np.arange(h, dtype=np.float64) / rd)[None, :]
    angle_term = 2.0 ** -50 * np.abs(angle)
    for name, g, e in (("cos", cos.cpu().numpy(), c64), ("sin", sin.cpu().numpy(), s64)):
        ulp32 = np.spacing(np.abs(e).astype(np.float32)).astype(np.float64)
        err = np.abs(g.astype(np.float64) - e)
        bad = err > ulp32 + angle_term
        assert not bad.any(), "%s: %d entries beyond the bar" % (name, np.count_nonzero(bad))
        off = int(np.count_nonzero(g != e.astype(np.float32)))
        beyond_ulp = int(np.count_nonzero(err > ulp32))
        print("table theta=%g rd=%d rows=%d f=%g %s: %d of %d entries differ from the oracle's "
              "fp32 rounding; %d need the angle term" % (theta, rd, rows, f, name, off, g.size,
                                                         beyond_ulp))


@pytest.mark.parametrize("backward", [False, True], ids=["fwd", "bwd"])
@pytest.mark.parametrize("name", NAMES)
def test_rotation_reduced_all_elements(name, backward):
    require_gpu()
    R = lib()
    w = W.BY_NAME[name].with_sizes(**REDUCED[name])
    q, k, pos = W.make_inputs(w)
    cos32, sin32 = oracle_tables(w.theta, w.rotary_dim, w.table_rows, w.interpolate_factor)
    qg, kg = q.cuda(), k.cuda()
    run_apply(w, qg, kg, torch.from_numpy(cos32).cuda(), torch.from_numpy(sin32).cuda(),
              pos_tensor(pos), backward)
    assert R.rope_check_errors() == R.ROPE_OK
    check_tensor(w, q, qg, w.Hq, pos, backward, cos32, sin32, name + " Q")
    check_tensor(w, k, kg, w.Hk, pos, backward, cos32, sin32, name + " K")


@pytest.mark.parametrize("name", NAMES)
def test_full_path_reduced_gpu_table(name):
    """Table built by the library, then forward: against the oracle end to end."""
    require_gpu()
    R = lib()
    w = W.BY_NAME[name].with_sizes(**REDUCED[name])
    q, k, pos = W.make_inputs(w)
    cos, sin = R.build_tables(w.theta, w.rotary_dim, w.table_rows, w.interpolate_factor)
    qg, kg = q.cuda(), k.cuda()
    run_apply(w, qg, kg, cos, sin, pos_tensor(pos), False)
    assert R.rope_check_errors() == R.ROPE_OK
    cos32, sin32 = oracle_tables(w.theta, w.rotary_dim, w.table_rows, w.interpolate_factor)
    check_tensor(w, q, qg, w.Hq, pos, False, cos32, sin32, name + " Q")
    check_tensor(w, k, kg, w.Hk, pos, False, cos32, sin32, name + " K")


def _sample_rows(w, H, n, rng):
    """(b, h, s) of n random rows plus the corner rows."""
    b = rng.integers(0, w.B, n)
    h = rng.integers(0, H, n)
    s = rng.integers(0, w.S, n)
    corners = [(0, 0, 0), (w.B - 1, H - 1, w.S - 1), (0, H - 1, w.S - 1), (w.B - 1, 0, 0)]
    b = np.concatenate([b, [c[0] for c in corners]])
    h = np.concatenate([h, [c[1] for c in corners]])
    s = np.concatenate([s, [c[2] for c in corners]])
    return b, h, s


def _rows(w, x, b, h, s):
    return x[b, s, h] if w.seq_before_head else x[b, h, s]


@pytest.mark.parametrize("name", NAMES)
def test_full_size_sampled(name):
    """Full-size workload, same calls as the bench: forward on (Q, K) and
    backward on a second pair (the gradients), table built by the library."""
    require_gpu()
    R = lib()
    w = W.BY_NAME[name]
    q, k, pos = W.make_inputs(w)
    cos, sin = R.build_tables(w.theta, w.rotary_dim, w.table_rows, w.interpolate_factor)
    cos32, sin32 = oracle_tables(w.theta, w.rotary_dim, w.table_rows, w.interpolate_factor)
    rows_of_token = np.arange(w.S) if pos is None else pos
    pos_g = pos_tensor(pos)
    rng = np.random.default_rng(w.seed)
    for backward in (False, True):
        qg, kg = q.cuda(), k.cuda()
        run_apply(w, qg, kg, cos, sin, pos_g, backward)
        assert R.rope_check_errors() == R.ROPE_OK
        for x, xg, H, tag in ((q, qg, w.Hq, "Q"), (k, kg, w.Hk, "K")):
            what = "%s %s %s" % (name, tag, "bwd" if backward else "fwd")
            b, h, s = _sample_rows(w, H, 3000, rng)
            xb = W.bits(x)
            got_all = gpu_bits(xg)
            inp = _rows(w, xb, b, h, s)                     # [n, D] input rows
            got = _rows(w, got_all, b, h, s)
            r = rows_of_token[s].astype(np.int32)
            n = inp.shape[0]
            rc, yb, y64 = O.load().apply(inp.reshape(1, 1, n, w.D), {"f32": O.F32, "bf16": O.BF16,
                                         "f16": O.F16}[w.dtype], 1, 1, n, w.D, w.rotary_dim,
                                         W.LAYOUTS[w.layout], False, backward, r, cos32, sin32)
            assert rc == O.OK
            assert_matches(w.dtype, got.reshape(1, 1, n, w.D), yb, y64, what)
            # properties on every element
            assert np.array_equal(got_all[..., w.rotary_dim:], xb[..., w.rotary_dim:]), what
            if pos is not None and np.any(pos == -1):
                idx = np.flatnonzero(pos == -1)
                assert np.array_equal(np.take(got_all, idx, axis=seq_axis(w)),
                                      np.take(xb, idx, axis=seq_axis(w))), what
            if w.dtype != "f32":
                assert all_finite16(w.dtype, got_all), what
            del got_all, xb
        del qg, kg
        torch.cuda.empty_cache()


@pytest.mark.parametrize("backward", [False, True], ids=["fwd", "bwd"])
@pytest.mark.parametrize("name", [w.name for w in W.SMALL_CALLS])
def test_small_calls_all_elements(name, backward):
    """The launch-bound calls the bench times (a decode step of 64 sequences
    with one token each; a 512-token prefill), at their full size: they take
    the launch rule's small-call branch (balanced runs over the resident
    lane groups, runs shorter than a tile).  Every element against the
    oracle."""
    require_gpu()
    w = W.ALL_BY_NAME[name]
    q, k, pos = W.make_inputs(w)
    cos32, sin32 = oracle_tables(w.theta, w.rotary_dim, w.table_rows)
    cg, sg = torch.from_numpy(cos32).cuda(), torch.from_numpy(sin32).cuda()
    qg, kg = q.cuda(), k.cuda()
    run_apply(w, qg, kg, cg, sg, pos_tensor(pos), backward)
    assert lib().rope_check_errors() == lib().ROPE_OK
    for x, xg, H in ((q, qg, w.Hq), (k, kg, w.Hk)):
        yb, y64 = oracle_apply(w, W.bits(x), H, pos, backward, cos32, sin32)
        assert_matches(w.dtype, gpu_bits(xg), yb, y64, "%s %s" % (name, "bwd" if backward else "fwd"))
