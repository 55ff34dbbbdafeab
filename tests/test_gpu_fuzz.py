"""Seeded random shapes through rope_apply_qk_out: every case against the
oracle (per sequence) and against the element-wise kernel bit for bit."""
import numpy as np
import pytest
import torch

import workloads as W
from gpu_util import assert_matches, gpu_bits, lib, oracle_apply, oracle_tables, require_gpu

pytestmark = pytest.mark.gpu


def _cases(n=48, seed=20261202):
    g = np.random.default_rng(seed)
    out = []
    for i in range(n):
        dtype = ["f32", "bf16", "f16"][g.integers(3)]
        D = int(g.choice([8, 16, 34, 40, 64, 96, 128, 136, 256]))
        rd = int(D if g.random() < 0.5 else 2 * g.integers(1, D // 2 + 1))
        out.append(dict(
            id=i, dtype=dtype, layout=["split_half", "interleaved"][g.integers(2)],
            sbh=bool(g.integers(2)), D=D, rd=rd, B=int(g.integers(1, 4)), S=int(g.integers(1, 71)),
            Hq=int(g.integers(1, 10)), Hk=int(g.integers(0, 6)),
            pos=["none", "shared", "per_seq"][g.integers(3)], oop=bool(g.integers(2)),
            backward=bool(g.integers(2)), misalign=bool(g.random() < 0.25)))
    return out


CASES = _cases()


@pytest.fixture
def restore_variant():
    yield
    lib().rope_force_kernel_variant(0)


def _run(R, w, q, k, cg, sg, pos_g, stride, oop, backward, misalign):
    """Rotate copies of q, k on the GPU; returns the output tensors."""
    e = q.element_size()

    def place(t):
        if t is None:
            return None
        if not misalign:
            return t.cuda()
        buf = torch.empty(t.numel() * e + 16, dtype=torch.uint8, device="cuda")
        v = buf[e:e + t.numel() * e].view(t.dtype).view(t.shape)
        v.copy_(t)
        return v

    qi, ki = place(q), place(k)
    qo = torch.empty_like(qi) if oop else qi
    ko = (torch.empty_like(ki) if oop else ki) if ki is not None else None
    R.rope_apply_qk_out(qi, ki, qo, ko, cg, sg, pos_g, stride, w.B, w.Hq, w.Hk, w.S, w.D,
                        w.rotary_dim, W.LAYOUTS[w.layout], int(w.seq_before_head), int(backward),
                        W.DTYPES[w.dtype], cg.shape[0])
    assert R.rope_check_errors() == R.ROPE_OK
    if oop:
        assert np.array_equal(gpu_bits(qi), W.bits(q))
    return qo, ko


@pytest.mark.parametrize("c", CASES, ids=lambda c: "case%d" % c["id"])
def test_random_shape(c, restore_variant):
    require_gpu()
    R = lib()
    rows = c["S"] + 9
    w = W.Workload("fuzz", c["B"], c["Hq"], c["Hk"], c["S"], c["D"], c["rd"], 1e4, c["dtype"],
                   c["layout"], c["sbh"], rows, "none", 1000 + c["id"])
    q, k, _ = W.make_inputs(w)
    c32, s32 = oracle_tables(w.theta, w.rotary_dim, rows)
    cg, sg = torch.from_numpy(c32).cuda(), torch.from_numpy(s32).cuda()
    g = np.random.default_rng(c["id"])
    if c["pos"] == "none":
        pos2d, pos_g, stride = None, None, 0
    elif c["pos"] == "shared":
        p = g.integers(-1, rows, w.S).astype(np.int32)
        pos2d, pos_g, stride = np.tile(p, (w.B, 1)), torch.from_numpy(p).cuda(), 0
    else:
        stride = w.S + int(g.integers(0, 3))
        pos2d = g.integers(-1, rows, (w.B, stride)).astype(np.int32)
        pos_g = torch.from_numpy(pos2d).cuda()
    got = _run(R, w, q, k, cg, sg, pos_g, stride, c["oop"], c["backward"], c["misalign"])
    R.rope_force_kernel_variant(2)
    ref = _run(R, w, q, k, cg, sg, pos_g, stride, c["oop"], c["backward"], False)
    R.rope_force_kernel_variant(0)
    sa = 1 if w.seq_before_head else 2
    for x, y, y2, H in ((q, got[0], ref[0], w.Hq), (k, got[1], ref[1], w.Hk)):
        if x is None or H == 0:
            continue
        yb_gpu = gpu_bits(y)
        assert np.array_equal(yb_gpu, gpu_bits(y2))             # same bits as element-wise
        for b in range(w.B):
            one = w.with_sizes(B=1)
            xs = np.ascontiguousarray(W.bits(x)[b:b + 1])
            pb = None if pos2d is None else np.ascontiguousarray(pos2d[b, :w.S])
            yb, y64 = oracle_apply(one, xs, H, pb, c["backward"], c32, s32)
            assert_matches(w.dtype, np.ascontiguousarray(yb_gpu[b:b + 1]), yb, y64,
                           "case %d batch %d" % (c["id"], b))
