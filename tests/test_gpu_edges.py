"""Edge cases of the CUDA library, through the C ABI.

Vectorised vs element-wise kernels (bit-identical), odd and maximum sizes,
layout permutation, backward as the negated sine, position gathers, the
out-of-range flag, guard bands around every buffer, empty problems, streams.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from gpu_util import (assert_matches, gpu_bits, lib, oracle_apply, oracle_tables, pos_tensor,
                      require_gpu)

pytestmark = pytest.mark.gpu

GUARD = 4096
FILL = 0xA5


def case(B, Hq, Hk, S, D, rd, dtype, layout="split_half", sbh=False, rows=None, theta=1e4, seed=7):
    return W.Workload("edge", B, Hq, Hk, S, D, rd, theta, dtype, layout, sbh,
                      rows if rows is not None else S, "none", seed)


class Guarded:
    """A tensor placed inside a larger byte buffer filled with a sentinel."""

    def __init__(self, src: torch.Tensor, byte_offset: int = 0):
        nbytes = src.numel() * src.element_size()
        self.buf = torch.full((2 * GUARD + nbytes + 64,), FILL, dtype=torch.uint8, device="cuda")
        self.start = GUARD + byte_offset
        self.nbytes = nbytes
        raw = self.buf[self.start:self.start + nbytes]
        self.t = raw.view(src.dtype).view(src.shape) if nbytes else torch.empty_like(src, device="cuda")
        self.t.copy_(src)

    def intact(self) -> bool:
        torch.cuda.synchronize()
        before = self.buf[:self.start]
        after = self.buf[self.start + self.nbytes:]
        return bool((before == FILL).all()) and bool((after == FILL).all())


def apply(w, q, k, cos, sin, pos=None, backward=False, stream=None, rows=None):
    R = lib()
    R.rope_apply_qk(q, k, cos, sin, pos, w.B, w.Hq, w.Hk if k is not None else 0, w.S, w.D,
                    w.rotary_dim, W.LAYOUTS[w.layout], int(w.seq_before_head), int(backward),
                    W.DTYPES[w.dtype], rows if rows is not None else cos.shape[0], stream)


def variant(w, q, k, cos, sin, pos=None):
    R = lib()
    return R.rope_qk_kernel_variant(q, k, cos, sin, pos, w.B, w.Hq, w.Hk, w.S, w.D, w.rotary_dim,
                                    W.LAYOUTS[w.layout], int(w.seq_before_head), 0,
                                    W.DTYPES[w.dtype], cos.shape[0])


def tables(w):
    c, s = oracle_tables(w.theta, w.rotary_dim, w.table_rows)
    return c, s, torch.from_numpy(c).cuda(), torch.from_numpy(s).cuda()


def check_vs_oracle(w, x_cpu, x_gpu, H, pos, backward, c32, s32, what=""):
    yb, y64 = oracle_apply(w, W.bits(x_cpu), H, pos, backward, c32, s32)
    assert_matches(w.dtype, gpu_bits(x_gpu), yb, y64, what)


@pytest.mark.parametrize("sbh", [False, True])
@pytest.mark.parametrize("layout", ["split_half", "interleaved"])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_vector_and_elementwise_kernels_bit_identical(dtype, layout, sbh):
    require_gpu()
    w = case(2, 5, 3, 37, 128, 96, dtype, layout, sbh)
    q, k, _ = W.make_inputs(w)
    c32, s32, cg, sg = tables(w)
    e = q.element_size()
    for backward in (False, True):
        qa, ka = Guarded(q), Guarded(k)                 # 16-byte aligned
        qm, km = Guarded(q, e), Guarded(k, e)           # one element off
        assert variant(w, qa.t, ka.t, cg, sg) == 3
        assert variant(w, qm.t, km.t, cg, sg) == 2
        apply(w, qa.t, ka.t, cg, sg, backward=backward)
        apply(w, qm.t, km.t, cg, sg, backward=backward)
        assert np.array_equal(gpu_bits(qa.t), gpu_bits(qm.t))
        assert np.array_equal(gpu_bits(ka.t), gpu_bits(km.t))
        for g in (qa, ka, qm, km):
            assert g.intact()
        check_vs_oracle(w, q, qa.t, w.Hq, None, backward, c32, s32, "Q")
        check_vs_oracle(w, k, ka.t, w.Hk, None, backward, c32, s32, "K")


@pytest.mark.parametrize("D,rd,dtype,layout,want_variant", [
    (34, 2, "bf16", "split_half", 2),
    (10, 6, "f16", "interleaved", 2),
    (8, 8, "bf16", "split_half", 2),            # 16-byte rotary span
    (6, 4, "f32", "interleaved", 2),
    (130, 130, "f16", "split_half", 2),
    (64, 16, "bf16", "interleaved", 3),         # smallest vector span: one pair of vectors
    (40, 32, "bf16", "split_half", 3),          # 80-byte rows
    (1024, 1024, "f32", "split_half", 3),       # 128 vectors per half: widest vector CTA row
    (1032, 1032, "f32", "interleaved", 2),      # 129 vectors per half: element-wise
    (2048, 2048, "f32", "split_half", 2),
    (1024, 512, "bf16", "interleaved", 3),
])
def test_odd_and_large_shapes(D, rd, dtype, layout, want_variant):
    require_gpu()
    w = case(2, 3, 2, 19, D, rd, dtype, layout)
    q, k, _ = W.make_inputs(w)
    c32, s32, cg, sg = tables(w)
    qg, kg = Guarded(q), Guarded(k)
    assert variant(w, qg.t, kg.t, cg, sg) == want_variant
    for backward in (False, True):
        qg.t.copy_(q)
        kg.t.copy_(k)
        apply(w, qg.t, kg.t, cg, sg, backward=backward)
        check_vs_oracle(w, q, qg.t, w.Hq, None, backward, c32, s32, "Q")
        check_vs_oracle(w, k, kg.t, w.Hk, None, backward, c32, s32, "K")
        assert np.array_equal(gpu_bits(qg.t)[..., rd:], W.bits(q)[..., rd:])
    assert qg.intact() and kg.intact()


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_layout_permutation_bit_exact(dtype):
    """Split-half of x equals interleaved of P x (P: 2i -> i, 2i+1 -> i + rd/2)."""
    require_gpu()
    w = case(1, 4, 2, 50, 128, 128, dtype)
    q, k, _ = W.make_inputs(w)
    _, _, cg, sg = tables(w)
    h = w.rotary_dim // 2
    perm = torch.arange(w.D)
    perm[0:w.rotary_dim:2] = torch.arange(h)
    perm[1:w.rotary_dim:2] = torch.arange(h) + h
    qs, ks = q.cuda(), k.cuda()
    qi, ki = q[..., perm].contiguous().cuda(), k[..., perm].contiguous().cuda()
    apply(w, qs, ks, cg, sg)
    apply(w.with_sizes(layout="interleaved"), qi, ki, cg, sg)
    assert np.array_equal(gpu_bits(qi), gpu_bits(qs[..., perm].contiguous()))
    assert np.array_equal(gpu_bits(ki), gpu_bits(ks[..., perm].contiguous()))


@pytest.mark.parametrize("layout", ["split_half", "interleaved"])
def test_backward_is_forward_with_negated_sine(layout):
    require_gpu()
    w = case(2, 4, 4, 64, 64, 64, "bf16", layout)
    q, k, _ = W.make_inputs(w)
    _, _, cg, sg = tables(w)
    a, b = q.cuda(), k.cuda()
    c, d = q.cuda(), k.cuda()
    apply(w, a, b, cg, sg, backward=True)
    apply(w, c, d, cg, -sg, backward=False)
    assert torch.equal(a, c) and torch.equal(b, d)


def test_gather_identity_and_prefix_shift():
    """pos_idx = arange(S) equals no index; arange(S) + p equals rows p.. of
    the table ("Custom Position IDs for Prefix-Tuning")."""
    require_gpu()
    p = 5
    w = case(2, 6, 2, 100, 128, 128, "bf16", rows=100 + p)
    q, k, _ = W.make_inputs(w)
    _, _, cg, sg = tables(w)
    ref_q, ref_k = q.cuda(), k.cuda()
    apply(w, ref_q, ref_k, cg, sg)
    a_q, a_k = q.cuda(), k.cuda()
    apply(w, a_q, a_k, cg, sg, pos=pos_tensor(np.arange(w.S)))
    assert torch.equal(a_q, ref_q) and torch.equal(a_k, ref_k)
    s_q, s_k = q.cuda(), k.cuda()
    apply(w, s_q, s_k, cg, sg, pos=pos_tensor(np.arange(w.S) + p))
    t_q, t_k = q.cuda(), k.cuda()
    apply(w, t_q, t_k, cg[p:].contiguous(), sg[p:].contiguous())
    assert torch.equal(s_q, t_q) and torch.equal(s_k, t_k)
    assert not torch.equal(s_q, ref_q)


@pytest.mark.parametrize("misaligned", [False, True])
def test_out_of_range_positions_flagged_and_untouched(misaligned):
    require_gpu()
    R = lib()
    assert R.rope_check_errors() == R.ROPE_OK
    w = case(2, 4, 2, 20, 64, 64, "f16", rows=16)
    q, k, _ = W.make_inputs(w)
    c32, s32, cg, sg = tables(w)
    pos = np.arange(w.S, dtype=np.int32) % 16
    pos[3] = 16            # one past the table
    pos[5] = -7            # negative, not the -1 mask
    pos[8] = -1            # masked: fine
    qg, kg = Guarded(q, 2 if misaligned else 0), Guarded(k)
    assert variant(w, qg.t, kg.t, cg, sg, pos_tensor(pos)) == (2 if misaligned else 3)
    apply(w, qg.t, kg.t, cg, sg, pos=pos_tensor(pos))
    assert R.rope_check_errors() == R.ROPE_ERR_POS_OUT_OF_RANGE
    assert R.rope_check_errors() == R.ROPE_OK            # reading clears the flag
    got = gpu_bits(qg.t)
    xb = W.bits(q)
    for s in (3, 5, 8):
        assert np.array_equal(got[:, :, s], xb[:, :, s])
    good = np.flatnonzero((pos >= 0) & (pos < 16))
    yb, y64 = oracle_apply(w.with_sizes(S=len(good)), np.ascontiguousarray(xb[:, :, good]), w.Hq,
                           pos[good], False, c32, s32)
    assert_matches("f16", np.ascontiguousarray(got[:, :, good]), yb, y64)
    assert qg.intact() and kg.intact()


@pytest.mark.parametrize("vector", [True, False])
def test_guard_bands_untouched(vector):
    require_gpu()
    w = case(3, 7, 3, 41, 64, 32, "bf16", rows=64)
    q, k, _ = W.make_inputs(w)
    c32, s32, _, _ = tables(w)
    off = 0 if vector else 2
    qg, kg = Guarded(q, off), Guarded(k, off)
    cg, sg = Guarded(torch.from_numpy(c32)), Guarded(torch.from_numpy(s32))
    pos = np.arange(w.S, dtype=np.int32) + 3
    pos[0] = -1
    pg = Guarded(torch.from_numpy(pos))
    assert variant(w, qg.t, kg.t, cg.t, sg.t, pg.t) == (3 if vector else 2)
    for backward in (False, True):
        apply(w, qg.t, kg.t, cg.t, sg.t, pos=pg.t, backward=backward)
    for g in (qg, kg, cg, sg, pg):
        assert g.intact()
    assert torch.equal(cg.t.cpu(), torch.from_numpy(c32)) and torch.equal(pg.t.cpu(), torch.from_numpy(pos))


def test_empty_problems_change_nothing():
    require_gpu()
    R = lib()
    w = case(1, 2, 2, 8, 64, 64, "bf16")
    q, k, _ = W.make_inputs(w)
    _, _, cg, sg = tables(w)
    qg, kg = q.cuda(), k.cuda()
    for B, S, Hq, Hk in ((0, 8, 2, 2), (1, 0, 2, 2), (1, 8, 0, 0)):
        R.rope_apply_qk(qg, kg, cg, sg, None, B, Hq, Hk, S, 64, 64, 0, 0, 0, R.ROPE_BF16, 8)
    assert R.rope_check_errors() == R.ROPE_OK
    assert torch.equal(qg.cpu(), q) and torch.equal(kg.cpu(), k)


def test_q_only_entry_and_gqa_without_k():
    require_gpu()
    R = lib()
    w = case(2, 8, 0, 33, 128, 128, "bf16")
    q, _, _ = W.make_inputs(w)
    c32, s32, cg, sg = tables(w)
    a, b = q.cuda(), q.cuda()
    R.apply_q(a, cg, sg)
    R.rope_apply_qk(b, None, cg, sg, None, w.B, w.Hq, 0, w.S, w.D, w.rotary_dim, 0, 0, 0,
                    R.ROPE_BF16, cg.shape[0])
    assert torch.equal(a, b)
    check_vs_oracle(w, q, a, w.Hq, None, False, c32, s32)


def test_single_token_single_head():
    require_gpu()
    w = case(1, 1, 1, 1, 128, 128, "f16")
    q, k, _ = W.make_inputs(w)
    c32, s32, cg, sg = tables(w)
    qg, kg = q.cuda(), k.cuda()
    apply(w, qg, kg, cg, sg)
    check_vs_oracle(w, q, qg, 1, None, False, c32, s32)
    assert torch.equal(qg.cpu(), q)           # position 0 is the identity


def test_runs_on_the_given_stream():
    require_gpu()
    w = case(2, 8, 2, 300, 128, 128, "bf16")
    q, k, _ = W.make_inputs(w)
    _, _, cg, sg = tables(w)
    a, b = q.cuda(), k.cuda()
    c, d = q.cuda(), k.cuda()
    apply(w, a, b, cg, sg)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        apply(w, c, d, cg, sg, stream=side)
    side.synchronize()
    torch.cuda.synchronize()
    assert torch.equal(a, c) and torch.equal(b, d)


def test_interpolate_factor_halves_positions_on_gpu():
    require_gpu()
    R = lib()
    c2, s2 = R.build_tables(1e4, 64, 200, 2.0)
    c1, s1 = R.build_tables(1e4, 64, 100, 1.0)
    assert torch.equal(c2[0::2], c1) and torch.equal(s2[0::2], s1)


def test_convenience_wrappers_match_abi_call():
    require_gpu()
    R = lib()
    w = case(2, 4, 2, 64, 128, 128, "f16", layout="interleaved", sbh=True)
    q, k, _ = W.make_inputs(w)
    cos, sin = R.build_tables(w.theta, w.rotary_dim, w.table_rows)
    a, b = q.cuda(), k.cuda()
    c, d = q.cuda(), k.cuda()
    R.apply_qk(a, b, cos, sin, layout="interleaved", seq_before_head=True)
    apply(w, c, d, cos, sin)
    assert torch.equal(a, c) and torch.equal(b, d)


@pytest.fixture
def restore_variant():
    yield
    lib().rope_force_kernel_variant(0)


@pytest.mark.parametrize("cfg", [
    dict(B=2, Hq=5, Hk=3, S=70, D=128, rd=128, dtype="bf16", layout="split_half", sbh=False),
    dict(B=3, Hq=4, Hk=2, S=45, D=128, rd=128, dtype="f16", layout="interleaved", sbh=True),
    dict(B=2, Hq=6, Hk=6, S=300, D=64, rd=32, dtype="bf16", layout="split_half", sbh=False),
    dict(B=1, Hq=3, Hk=0, S=33, D=64, rd=64, dtype="f32", layout="interleaved", sbh=False),
    dict(B=2, Hq=2, Hk=1, S=17, D=96, rd=64, dtype="f32", layout="split_half", sbh=True),
    dict(B=1, Hq=2, Hk=2, S=9, D=1024, rd=1024, dtype="f32", layout="split_half", sbh=False),
])
@pytest.mark.parametrize("positions", ["none", "masked", "out_of_range"])
def test_all_kernel_variants_bit_identical(cfg, positions, restore_variant):
    """Register-vector and element-wise kernels give the same bits, and touch
    nothing outside the rotated spans."""
    require_gpu()
    R = lib()
    rows = cfg["S"] + 8
    w = case(cfg["B"], cfg["Hq"], cfg["Hk"], cfg["S"], cfg["D"], cfg["rd"], cfg["dtype"],
             cfg["layout"], cfg["sbh"], rows=rows)
    q, k, _ = W.make_inputs(w)
    c32, s32, cg, sg = tables(w)
    pos = None
    if positions != "none":
        pos = (np.arange(w.S, dtype=np.int32) * 7 + 3) % rows
        pos[:2] = -1
        pos[w.S // 2] = -1
        if positions == "out_of_range":
            pos[w.S - 1] = rows + 5
    pos_g = None if pos is None else pos_tensor(pos)
    results = {}
    for v in (3, 2):
        R.rope_force_kernel_variant(v)
        for backward in (False, True):
            qg = Guarded(q)
            kg = Guarded(k) if k is not None else None
            assert variant(w, qg.t, None if kg is None else kg.t, cg, sg, pos_g) == v
            apply(w, qg.t, None if kg is None else kg.t, cg, sg, pos=pos_g, backward=backward)
            st = R.rope_check_errors()
            want = R.ROPE_ERR_POS_OUT_OF_RANGE if positions == "out_of_range" else R.ROPE_OK
            assert st == want, (v, st)
            assert qg.intact() and (kg is None or kg.intact())
            results[(v, backward)] = (gpu_bits(qg.t), None if kg is None else gpu_bits(kg.t))
    for backward in (False, True):
        a, b = results[(3, backward)], results[(2, backward)]
        assert np.array_equal(a[0], b[0]), backward
        if a[1] is not None:
            assert np.array_equal(a[1], b[1]), backward
    # and the vector result against the oracle on the rows the oracle accepts
    good = np.ones(w.S, bool) if pos is None else (pos >= 0) & (pos < rows)
    sa = 1 if w.seq_before_head else 2
    for x, H, got in ((q, w.Hq, results[(3, False)][0]), (k, w.Hk, results[(3, False)][1])):
        if x is None or H == 0:
            continue
        idx = np.flatnonzero(good)
        xb = np.ascontiguousarray(np.take(W.bits(x), idx, axis=sa))
        yb, y64 = oracle_apply(w.with_sizes(S=len(idx)), xb, H, None if pos is None else pos[idx],
                               False, c32, s32)
        assert_matches(w.dtype, np.ascontiguousarray(np.take(got, idx, axis=sa)), yb, y64)
        bad = np.flatnonzero(~good)
        assert np.array_equal(np.take(got, bad, axis=sa), np.take(W.bits(x), bad, axis=sa))


@pytest.fixture
def restore_tuning():
    yield
    lib().rope_tune_rotation_launch(0, 0, 0)


@pytest.mark.parametrize("cfg", [
    dict(B=3, Hq=5, Hk=3, S=70, D=128, rd=128, dtype="bf16", layout="split_half", sbh=False),
    dict(B=2, Hq=4, Hk=2, S=45, D=128, rd=128, dtype="f16", layout="interleaved", sbh=True),
    dict(B=5, Hq=6, Hk=6, S=301, D=64, rd=32, dtype="bf16", layout="split_half", sbh=False),
    dict(B=1, Hq=3, Hk=1, S=33, D=64, rd=64, dtype="f32", layout="interleaved", sbh=False),
])
@pytest.mark.parametrize("tuning", [(1, 1, 0), (1, 7, -1), (2, 1000, 0), (0, 3, -1), (64, 1, 0)],
                         ids=lambda t: "ctas%d_units%d_pf%d" % t)
def test_vector_grid_sizing_does_not_change_results(cfg, tuning, restore_tuning):
    """The vector kernel splits its (token tile, head) units into balanced
    runs, one per lane group; a run may start and end inside a tile and cross
    several tiles (and batch entries).  However the grid is sized -- one CTA
    per SM, runs of 7 or 1000 units, more CTAs than are resident -- the bits
    are those of the default launch, with positions gathered and masked, and
    nothing outside the rotated spans is touched."""
    require_gpu()
    R = lib()
    rows = cfg["S"] + 8
    w = case(cfg["B"], cfg["Hq"], cfg["Hk"], cfg["S"], cfg["D"], cfg["rd"], cfg["dtype"],
             cfg["layout"], cfg["sbh"], rows=rows)
    q, k, _ = W.make_inputs(w)
    c32, s32, cg, sg = tables(w)
    pos = (np.arange(w.S, dtype=np.int32) * 5 + 1) % rows
    pos[0] = -1
    pos[w.S // 3] = -1
    pos_g = pos_tensor(pos)
    got = {}
    for t in ((0, 0, 0), tuning):
        R.rope_tune_rotation_launch(*t)
        qg, kg = Guarded(q), Guarded(k)
        assert variant(w, qg.t, kg.t, cg, sg, pos_g) == 3
        apply(w, qg.t, kg.t, cg, sg, pos=pos_g, backward=False)
        first = (gpu_bits(qg.t), gpu_bits(kg.t))
        apply(w, qg.t, kg.t, cg, sg, pos=pos_g, backward=True)
        apply(w, qg.t, kg.t, cg, sg, pos=pos_g, backward=False)
        assert R.rope_check_errors() == R.ROPE_OK
        assert qg.intact() and kg.intact()
        got[t] = first + (gpu_bits(qg.t), gpu_bits(kg.t))
    a, b = got[(0, 0, 0)], got[tuning]
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    # the first forward against the oracle; unrotated tokens bit-exact
    sa = 1 if w.seq_before_head else 2
    good = pos >= 0
    idx, bad = np.flatnonzero(good), np.flatnonzero(~good)
    for x, H, g in ((q, w.Hq, b[0]), (k, w.Hk, b[1])):
        xb = np.ascontiguousarray(np.take(W.bits(x), idx, axis=sa))
        yb, y64 = oracle_apply(w.with_sizes(S=len(idx)), xb, H, pos[idx], False, c32, s32)
        assert_matches(w.dtype, np.ascontiguousarray(np.take(g, idx, axis=sa)), yb, y64,
                       "tuning %s" % (tuning,))
        assert np.array_equal(np.take(g, bad, axis=sa), np.take(W.bits(x), bad, axis=sa))


def test_calls_replay_in_a_cuda_graph():
    """Forward/backward calls captured in a CUDA graph (programmatic launches
    become graph edges) and replayed give the eager results."""
    require_gpu()
    R = lib()
    w = case(2, 8, 2, 96, 128, 128, "bf16")
    q, k, _ = W.make_inputs(w)
    dq, dk, _ = W.make_inputs(w, seed_offset=3)
    cos, sin = R.build_tables(w.theta, w.rotary_dim, w.table_rows)
    # eager
    eq, ek, edq, edk = q.cuda(), k.cuda(), dq.cuda(), dk.cuda()
    for _ in range(3):
        R.apply_qk(eq, ek, cos, sin)
        R.apply_qk(edq, edk, cos, sin, backward=True)
    # captured
    gq, gk, gdq, gdk = q.cuda(), k.cuda(), dq.cuda(), dk.cuda()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            R.apply_qk(gq, gk, cos, sin, stream=s)
            R.apply_qk(gdq, gdk, cos, sin, backward=True, stream=s)
    torch.cuda.synchronize()
    # capture does not execute: replay three times
    gq.copy_(q.cuda()); gk.copy_(k.cuda()); gdq.copy_(dq.cuda()); gdk.copy_(dk.cuda())
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert R.rope_check_errors() == R.ROPE_OK
    assert torch.equal(gq, eq) and torch.equal(gk, ek)
    assert torch.equal(gdq, edq) and torch.equal(gdk, edk)


@pytest.mark.parametrize("delta", [-1, 0, 1])
def test_launch_rule_boundary_against_oracle(delta):
    """The launch rule switches from balanced runs over the resident lane
    groups to one tile per lane group when the call has as many tiles as
    there are resident lane groups (SM count x 4 CTAs x 4 lane groups for
    bf16 rd = 128).  One tile below, at and above that count (4 tokens per
    tile), against the oracle, forward and backward."""
    require_gpu()
    R = lib()
    lanes = torch.cuda.get_device_properties(0).multi_processor_count * 4 * 4
    S = 4 * (lanes + delta) - 2                    # ragged last tile
    w = case(1, 2, 1, S, 128, 128, "bf16", rows=S)
    q, k, _ = W.make_inputs(w)
    c32, s32, cg, sg = tables(w)
    for backward in (False, True):
        qg, kg = q.cuda(), k.cuda()
        apply(w, qg, kg, cg, sg, backward=backward)
        assert R.rope_check_errors() == R.ROPE_OK
        check_vs_oracle(w, q, qg, w.Hq, None, backward, c32, s32, "Q delta %d" % delta)
        check_vs_oracle(w, k, kg, w.Hk, None, backward, c32, s32, "K delta %d" % delta)
