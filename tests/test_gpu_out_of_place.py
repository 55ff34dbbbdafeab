"""Out-of-place rotation, per-sequence position indices and the autograd
binding, through the C ABI, against in-place calls and the CPU oracle."""
import numpy as np
import pytest
import torch

import workloads as W
from gpu_util import (assert_matches, gpu_bits, lib, oracle_apply, oracle_tables, pos_tensor,
                      require_gpu)

pytestmark = pytest.mark.gpu


def case(B, Hq, Hk, S, D, rd, dtype, layout="split_half", sbh=False, rows=None, seed=11):
    return W.Workload("oop", B, Hq, Hk, S, D, rd, 1e4, dtype, layout, sbh,
                      rows if rows is not None else S, "none", seed)


@pytest.fixture
def restore_variant():
    yield
    lib().rope_force_kernel_variant(0)


def _oracle_per_sequence(w, x, H, pos2d, backward, c32, s32):
    """Oracle on each sequence b with its own position row (pos2d[b, :S])."""
    xb = W.bits(x)
    sa = 1 if w.seq_before_head else 2
    ys, y64s = [], []
    for b in range(w.B):
        one = w.with_sizes(B=1)
        xs = np.ascontiguousarray(xb[b:b + 1])
        yb, y64 = oracle_apply(one, xs, H, None if pos2d is None else pos2d[b, :w.S], backward,
                               c32, s32)
        ys.append(yb)
        y64s.append(y64)
    return np.concatenate(ys), np.concatenate(y64s)


@pytest.mark.parametrize("variant", [3, 2])
@pytest.mark.parametrize("cfg", [
    dict(B=2, Hq=6, Hk=2, S=40, D=128, rd=128, dtype="bf16", layout="split_half", sbh=False),
    dict(B=3, Hq=4, Hk=4, S=25, D=64, rd=32, dtype="f16", layout="interleaved", sbh=True),
    dict(B=2, Hq=3, Hk=1, S=19, D=96, rd=64, dtype="f32", layout="split_half", sbh=False),
])
def test_out_of_place_matches_in_place_and_passes_through(cfg, variant, restore_variant):
    require_gpu()
    R = lib()
    R.rope_force_kernel_variant(variant)
    rows = cfg["S"] + 4
    w = case(cfg["B"], cfg["Hq"], cfg["Hk"], cfg["S"], cfg["D"], cfg["rd"], cfg["dtype"],
             cfg["layout"], cfg["sbh"], rows=rows)
    q, k, _ = W.make_inputs(w)
    c32, s32 = oracle_tables(w.theta, w.rotary_dim, w.table_rows)
    cg, sg = torch.from_numpy(c32).cuda(), torch.from_numpy(s32).cuda()
    pos = (np.arange(w.S, dtype=np.int32) + 2) % rows
    pos[0] = -1
    pos[3] = rows + 7                                  # out of range: unrotated, flagged
    pg = pos_tensor(pos)
    for backward in (False, True):
        qi, ki = q.cuda(), k.cuda()
        qin, kin = q.cuda(), k.cuda()
        qo, ko = torch.full_like(qin, 7.0), torch.full_like(kin, 7.0)
        R.rope_apply_qk(qi, ki, cg, sg, pg, w.B, w.Hq, w.Hk, w.S, w.D, w.rotary_dim,
                        W.LAYOUTS[w.layout], int(w.seq_before_head), int(backward),
                        W.DTYPES[w.dtype], rows)
        R.rope_apply_qk_out(qin, kin, qo, ko, cg, sg, pg, 0, w.B, w.Hq, w.Hk, w.S, w.D,
                            w.rotary_dim, W.LAYOUTS[w.layout], int(w.seq_before_head),
                            int(backward), W.DTYPES[w.dtype], rows)
        assert R.rope_check_errors() == R.ROPE_ERR_POS_OUT_OF_RANGE
        # out of place gives every element of the in-place result; inputs untouched
        assert np.array_equal(gpu_bits(qo), gpu_bits(qi)) and np.array_equal(gpu_bits(ko), gpu_bits(ki))
        assert np.array_equal(gpu_bits(qin), W.bits(q)) and np.array_equal(gpu_bits(kin), W.bits(k))


@pytest.mark.parametrize("stride_pad", [0, 5])
@pytest.mark.parametrize("cfg", [
    dict(B=4, Hq=8, Hk=2, S=33, D=128, rd=128, dtype="bf16", layout="split_half", sbh=False),
    dict(B=3, Hq=4, Hk=4, S=17, D=64, rd=64, dtype="f16", layout="interleaved", sbh=True),
    dict(B=64, Hq=32, Hk=8, S=1, D=128, rd=128, dtype="bf16", layout="split_half", sbh=False),  # decode
])
def test_per_sequence_positions_against_oracle(cfg, stride_pad):
    require_gpu()
    R = lib()
    rows = 4096
    w = case(cfg["B"], cfg["Hq"], cfg["Hk"], cfg["S"], cfg["D"], cfg["rd"], cfg["dtype"],
             cfg["layout"], cfg["sbh"], rows=rows)
    q, k, _ = W.make_inputs(w)
    c32, s32 = oracle_tables(w.theta, w.rotary_dim, rows)
    cg, sg = torch.from_numpy(c32).cuda(), torch.from_numpy(s32).cuda()
    g = np.random.default_rng(w.B * 100 + w.S)
    stride = w.S + stride_pad
    pos2d = np.full((w.B, stride), -5, dtype=np.int32)     # padding never read
    starts = g.integers(0, rows - w.S, w.B)
    pos2d[:, :w.S] = starts[:, None] + np.arange(w.S)[None, :]   # context shifted per sequence
    if w.S > 2:
        pos2d[0, 1] = -1
    qo, ko = R.rotate_qk(q.cuda(), k.cuda(), cg, sg, pos_idx=torch.from_numpy(pos2d).cuda(),
                         layout=w.layout, seq_before_head=w.seq_before_head)
    assert R.rope_check_errors() == R.ROPE_OK
    for x, got, H in ((q, qo, w.Hq), (k, ko, w.Hk)):
        yb, y64 = _oracle_per_sequence(w, x, H, pos2d, False, c32, s32)
        assert_matches(w.dtype, gpu_bits(got), yb, y64)
    # in place through the same entry point (q_out = q)
    qi, ki = q.cuda(), k.cuda()
    R.rotate_qk(qi, ki, cg, sg, pos_idx=torch.from_numpy(pos2d).cuda(), layout=w.layout,
                seq_before_head=w.seq_before_head, q_out=qi, k_out=ki)
    assert torch.equal(qi, qo) and torch.equal(ki, ko)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_autograd_forward_and_backward(dtype):
    require_gpu()
    R = lib()
    from rotary_position_embedding_rope_gb300.autograd import rotary_qk

    w = case(2, 4, 2, 48, 64, 64, dtype, rows=64)
    q, k, _ = W.make_inputs(w)
    gq, gk, _ = W.make_inputs(w, seed_offset=50)            # upstream gradients
    c32, s32 = oracle_tables(w.theta, w.rotary_dim, w.table_rows)
    cg, sg = torch.from_numpy(c32).cuda(), torch.from_numpy(s32).cuda()
    qg = q.cuda().requires_grad_(True)
    kg = k.cuda().requires_grad_(True)
    qr, kr = rotary_qk(qg, kg, cg, sg)
    fq, fk = R.rotate_qk(q.cuda(), k.cuda(), cg, sg)
    assert torch.equal(qr.detach(), fq) and torch.equal(kr.detach(), fk)
    ((qr * gq.cuda()).sum() + (kr * gk.cuda()).sum()).backward()
    # d/dx of sum(G * R(t) x) is R(-t) G: the oracle's backward rotation of G
    for g_in, grad, H in ((gq, qg.grad, w.Hq), (gk, kg.grad, w.Hk)):
        yb, y64 = oracle_apply(w, W.bits(g_in), H, None, True, c32, s32)
        assert_matches(dtype, gpu_bits(grad), yb, y64)
    # a loss that uses only q leaves k's gradient None-free and zero
    qg2 = q.cuda().requires_grad_(True)
    kg2 = k.cuda().requires_grad_(True)
    qr2, _ = rotary_qk(qg2, kg2, cg, sg)
    (qr2 * gq.cuda()).sum().backward()
    assert kg2.grad is None or torch.count_nonzero(kg2.grad) == 0
    yb, y64 = oracle_apply(w, W.bits(gq), w.Hq, None, True, c32, s32)
    assert_matches(dtype, gpu_bits(qg2.grad), yb, y64)


@pytest.mark.parametrize("chunks", [1, 2, 4, 10])
def test_host_pipeline_matches_device_call(chunks):
    """Pinned host tensors rotated through the chunked copy/rotate/copy pipeline
    give the same bits as the device call (10 pieces: each batch entry's heads
    in two groups)."""
    require_gpu()
    R = lib()
    from rotary_position_embedding_rope_gb300.host import HostRotator

    w = case(5, 4, 2, 64, 128, 128, "bf16", rows=64)
    q, k, _ = W.make_inputs(w)
    cos, sin = R.build_tables(w.theta, w.rotary_dim, w.table_rows)
    rot = HostRotator(chunks=chunks)
    hq, hk = q.pin_memory(), k.pin_memory()
    oq, ok_ = torch.empty_like(q).pin_memory(), torch.empty_like(k).pin_memory()
    for backward in (False, True):
        done = rot.apply_qk(hq, hk, cos, sin, oq, ok_, backward=backward)
        done.synchronize()
        dq, dk = q.cuda(), k.cuda()
        R.apply_qk(dq, dk, cos, sin, backward=backward)
        assert torch.equal(oq, dq.cpu()) and torch.equal(ok_, dk.cpu())
        assert torch.equal(hq, q) and torch.equal(hk, k)


@pytest.mark.parametrize("sbh,with_k", [(False, False), (True, True)])
def test_host_pipeline_head_pieces_q_only_and_seq_first(sbh, with_k):
    """More pieces than batch entries: Q alone is split by head groups; the
    [B,S,H,D] layout (heads not contiguous per entry) falls back to batch
    pieces.  Both give the device call's bits."""
    require_gpu()
    R = lib()
    from rotary_position_embedding_rope_gb300.host import HostRotator

    w = case(3, 4, 2, 48, 64, 64, "f16", sbh=sbh, rows=48)
    q, k, _ = W.make_inputs(w)
    cos, sin = R.build_tables(w.theta, w.rotary_dim, w.table_rows)
    rot = HostRotator(chunks=12)
    hq = q.pin_memory()
    hk = k.pin_memory() if with_k else None
    oq = torch.empty_like(q).pin_memory()
    ok_ = torch.empty_like(k).pin_memory() if with_k else None
    rot.apply_qk(hq, hk, cos, sin, oq, ok_, seq_before_head=sbh).synchronize()
    dq = q.cuda()
    dk = k.cuda() if with_k else None
    R.apply_qk(dq, dk, cos, sin, seq_before_head=sbh)
    assert torch.equal(oq, dq.cpu())
    if with_k:
        assert torch.equal(ok_, dk.cpu())


def test_host_pipeline_shape_change_without_sync():
    """Back-to-back pipeline calls with different shapes and no wait between
    them: the second call's new staging buffers must not reuse the first
    call's memory while its copies are still queued.  Both results equal the
    device calls bit for bit."""
    require_gpu()
    R = lib()
    from rotary_position_embedding_rope_gb300.host import HostRotator

    rot = HostRotator(chunks=4)
    outs = []
    for i, (B, S) in enumerate(((4, 512), (2, 96), (4, 512))):
        w = case(B, 8, 2, S, 128, 128, "bf16", rows=512, seed=30 + i)
        q, k, _ = W.make_inputs(w)
        cos, sin = R.build_tables(w.theta, w.rotary_dim, w.table_rows)
        hq, hk = q.pin_memory(), k.pin_memory()
        oq, ok_ = torch.empty_like(q).pin_memory(), torch.empty_like(k).pin_memory()
        done = rot.apply_qk(hq, hk, cos, sin, oq, ok_)
        outs.append((w, q, k, cos, sin, oq, ok_, done))
    for w, q, k, cos, sin, oq, ok_, done in outs:
        done.synchronize()
        dq, dk = q.cuda(), k.cuda()
        R.apply_qk(dq, dk, cos, sin)
        assert torch.equal(oq, dq.cpu()) and torch.equal(ok_, dk.cpu())


@pytest.mark.parametrize("slots,chunks", [(3, 5), (4, 4)])
def test_host_pipeline_more_staging_slots(slots, chunks):
    """With more staging slots than two, the pieces of successive calls take
    the slots in turn; two calls back to back (forward, then backward on other
    tensors) give the device calls' bits."""
    require_gpu()
    R = lib()
    from rotary_position_embedding_rope_gb300.host import HostRotator

    w = case(5, 4, 2, 64, 128, 128, "bf16", rows=64)
    q, k, _ = W.make_inputs(w)
    dq, dk, _ = W.make_inputs(w, seed_offset=9)
    cos, sin = R.build_tables(w.theta, w.rotary_dim, w.table_rows)
    rot = HostRotator(chunks=chunks, slots=slots)
    outs = []
    for x, y, backward in ((q, k, False), (dq, dk, True)):
        hx, hy = x.pin_memory(), y.pin_memory()
        ox, oy = torch.empty_like(x).pin_memory(), torch.empty_like(y).pin_memory()
        outs.append((x, y, backward, ox, oy, rot.apply_qk(hx, hy, cos, sin, ox, oy,
                                                         backward=backward)))
    for x, y, backward, ox, oy, done in outs:
        done.synchronize()
        gx, gy = x.cuda(), y.cuda()
        R.apply_qk(gx, gy, cos, sin, backward=backward)
        assert torch.equal(ox, gx.cpu()) and torch.equal(oy, gy.cpu())
