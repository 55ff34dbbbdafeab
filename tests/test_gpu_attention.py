"""Attention with the rotation fused into the Q/K tile loads (tcgen05) against
the fp64 rotary-attention oracle, on both key paths: keys rotated inside the
attention kernel (no workspace) and keys rotated once into a workspace by the
rotation kernel.  The two paths give the same bits.

Tolerance: the kernel rounds P to the element type before the P.V product and
rounds O once; each is within half a unit in the last place, so per element
|o - o_ref| <= u * (max|v| + |o_ref|) with u = 2^-8 (bf16) or 2^-10 (fp16),
a bound twice the two roundings' sum.  Everything else (fp32 accumulation,
exp2) is far below it.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from gpu_util import lib, oracle_tables, require_gpu
from oracle import attention as OA

pytestmark = pytest.mark.gpu
U = {"bf16": 2.0 ** -8, "f16": 2.0 ** -10}
CODE = {"bf16": O.BF16, "f16": O.F16}


def _inputs(B, Hq, Hk, Sq, Sk, D, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    q = W.draw((B, Hq, Sq, D), dtype, g)
    k = W.draw((B, Hk, Sk, D), dtype, g)
    v = W.draw((B, Hk, Sk, D), dtype, g)
    return q, k, v


def _check(got, q, k, v, dtype, rd, layout, c32, s32, pq, pk, causal, what=""):
    ref = OA.attention(W.bits(q), W.bits(k), W.bits(v), CODE[dtype], rd, layout, c32, s32,
                       pq, pk, causal)
    g = got.float().cpu().numpy().astype(np.float64)
    vmax = float(v.float().abs().max()) if v.numel() else 0.0
    tol = U[dtype] * (vmax + np.abs(ref))
    err = np.abs(g - ref)
    assert np.all(np.isfinite(g)), what
    assert np.all(err <= tol), "%s: %d of %d beyond tolerance, max err %.3g" % (
        what, np.count_nonzero(err > tol), err.size, err.max())


CASES = [
    dict(B=1, Hq=4, Hk=2, Sq=200, Sk=200, D=128, rd=128, dtype="bf16", layout="split_half", causal=True),
    dict(B=2, Hq=2, Hk=2, Sq=130, Sk=257, D=128, rd=64, dtype="bf16", layout="split_half", causal=False),
    dict(B=1, Hq=8, Hk=1, Sq=129, Sk=129, D=64, rd=32, dtype="f16", layout="interleaved", causal=True),
    dict(B=1, Hq=2, Hk=1, Sq=64, Sk=300, D=64, rd=64, dtype="bf16", layout="interleaved", causal=False),
    dict(B=1, Hq=2, Hk=2, Sq=1, Sk=300, D=128, rd=128, dtype="bf16", layout="split_half", causal=True),
    dict(B=1, Hq=2, Hk=2, Sq=300, Sk=100, D=128, rd=128, dtype="f16", layout="split_half", causal=True),
    # eight key tiles: both value buffers alternate several times; Sq < Sk
    dict(B=1, Hq=4, Hk=2, Sq=520, Sk=1000, D=128, rd=128, dtype="bf16", layout="split_half", causal=True),
    # odd group (3): pairs of query tiles, the last CTA's second block past Sq
    dict(B=2, Hq=6, Hk=2, Sq=300, Sk=300, D=64, rd=32, dtype="f16", layout="split_half", causal=False),
    dict(B=1, Hq=3, Hk=1, Sq=257, Sk=390, D=128, rd=64, dtype="bf16", layout="interleaved", causal=True),
    # interleaved, full rotary span: table chunks from the second staged table box
    dict(B=1, Hq=4, Hk=1, Sq=300, Sk=300, D=128, rd=128, dtype="bf16", layout="interleaved", causal=True),
    # more work units than pairs of SMs (144 and 180): the persistent kernel of
    # the workspace path runs several units per cluster, back to back
    dict(B=24, Hq=4, Hk=2, Sq=300, Sk=400, D=128, rd=128, dtype="bf16", layout="split_half", causal=False),
    dict(B=30, Hq=3, Hk=1, Sq=260, Sk=260, D=128, rd=64, dtype="f16", layout="interleaved", causal=True),
]


WS = {"ws": "auto", "inkernel": None}     # key workspace, or keys rotated in the kernel


@pytest.mark.parametrize("ws", sorted(WS))
@pytest.mark.parametrize("c", CASES, ids=lambda c: "Sq%d_Sk%d_D%d_rd%d_%s_%s_c%d" % (
    c["Sq"], c["Sk"], c["D"], c["rd"], c["dtype"], c["layout"], c["causal"]))
def test_attention_against_oracle(c, ws):
    require_gpu()
    R = lib()
    q, k, v = _inputs(c["B"], c["Hq"], c["Hk"], c["Sq"], c["Sk"], c["D"], c["dtype"], 31)
    rows = max(c["Sq"], c["Sk"]) + 8
    c32, s32 = oracle_tables(1e4, c["rd"], rows)
    cg, sg = torch.from_numpy(c32).cuda(), torch.from_numpy(s32).cuda()
    o = R.attention(q.cuda(), k.cuda(), v.cuda(), cg, sg, rotary_dim=c["rd"], layout=c["layout"],
                    causal=c["causal"], k_workspace=WS[ws])
    assert R.rope_check_errors() == R.ROPE_OK
    _check(o, q, k, v, c["dtype"], c["rd"], W.LAYOUTS[c["layout"]], c32, s32, None, None,
           c["causal"], str(c))


@pytest.mark.parametrize("ws", sorted(WS))
def test_pages_example_cls_tokens_unrotated(ws):
    """q, k, v [1, 8, 1024 + 2, 64], rotary dim 32, the first 2 tokens not
    rotated and the rest at positions 0..1023 ("rotary-embedding-torch",
    flash_attn_with_rotary example), causal."""
    require_gpu()
    R = lib()
    q, k, v = _inputs(1, 8, 8, 1026, 1026, 64, "bf16", 7)
    pos = np.arange(-2, 1024, dtype=np.int32)
    pos[:2] = -1
    c32, s32 = oracle_tables(1e4, 32, 1024)
    cg, sg = torch.from_numpy(c32).cuda(), torch.from_numpy(s32).cuda()
    pg = torch.from_numpy(pos).cuda()
    o = R.attention(q.cuda(), k.cuda(), v.cuda(), cg, sg, pos_q=pg, pos_k=pg, rotary_dim=32,
                    causal=True, k_workspace=WS[ws])
    assert R.rope_check_errors() == R.ROPE_OK
    _check(o, q, k, v, "bf16", 32, O.SPLIT_HALF, c32, s32, pos, pos, True, "pages example")


def test_attention_with_no_keys_is_zero_and_shift_invariant():
    require_gpu()
    R = lib()
    q, k, v = _inputs(1, 2, 2, 100, 0, 128, "bf16", 3)
    c32, s32 = oracle_tables(1e4, 128, 512)
    cg, sg = torch.from_numpy(c32).cuda(), torch.from_numpy(s32).cuda()
    o = R.attention(q.cuda(), k.cuda(), v.cuda(), cg, sg, causal=False)
    assert torch.count_nonzero(o) == 0
    # a common shift of every position changes only rounding
    q, k, v = _inputs(1, 2, 2, 160, 160, 128, "bf16", 4)
    p0 = torch.arange(160, dtype=torch.int32).cuda()
    a = R.attention(q.cuda(), k.cuda(), v.cuda(), cg, sg, pos_q=p0, pos_k=p0, causal=True)
    b = R.attention(q.cuda(), k.cuda(), v.cuda(), cg, sg, pos_q=p0 + 300, pos_k=p0 + 300,
                    causal=True)
    assert float((a.float() - b.float()).abs().max()) < 0.05


@pytest.mark.parametrize("ws", sorted(WS))
def test_attention_gathered_positions_interleaved(ws):
    """Per-token positions (a shuffled set, some -1) with the interleaved
    layout: the key rotation reads each row's table row by its position."""
    require_gpu()
    R = lib()
    q, k, v = _inputs(1, 4, 2, 200, 333, 64, "f16", 11)
    g = np.random.default_rng(5)
    pq = g.permutation(600)[:200].astype(np.int32)
    pk = g.permutation(600)[:333].astype(np.int32)
    pq[::17] = -1
    pk[::13] = -1
    c32, s32 = oracle_tables(1e4, 64, 600)
    cg, sg = torch.from_numpy(c32).cuda(), torch.from_numpy(s32).cuda()
    o = R.attention(q.cuda(), k.cuda(), v.cuda(), cg, sg, pos_q=torch.from_numpy(pq).cuda(),
                    pos_k=torch.from_numpy(pk).cuda(), rotary_dim=64, layout="interleaved",
                    causal=False, k_workspace=WS[ws])
    assert R.rope_check_errors() == R.ROPE_OK
    _check(o, q, k, v, "f16", 64, O.INTERLEAVED, c32, s32, pq, pk, False, "gathered positions")


def _fuzz_cases(n=24, seed=2024):
    g = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        D = int(g.choice([64, 128]))
        Hk = int(g.integers(1, 4))
        cases.append(dict(
            i=i, B=int(g.integers(1, 3)), Hk=Hk, Hq=Hk * int(g.integers(1, 5)), D=D,
            rd=16 * int(g.integers(1, D // 16 + 1)), layout=str(g.choice(["split_half", "interleaved"])),
            dtype=str(g.choice(["bf16", "f16"])), Sq=int(g.integers(1, 400)), Sk=int(g.integers(1, 400)),
            causal=bool(g.integers(0, 2)), pos=str(g.choice(["none", "none", "random"])),
            seed=int(g.integers(0, 2 ** 31))))
    return cases


@pytest.mark.parametrize("c", _fuzz_cases(), ids=lambda c: "fuzz%02d" % c["i"])
def test_attention_fuzz(c):
    """Seeded random shapes, spans, layouts, types, masks and positions; the
    workspace path against the oracle, the in-kernel key path bit for bit
    against it."""
    require_gpu()
    R = lib()
    q, k, v = _inputs(c["B"], c["Hq"], c["Hk"], c["Sq"], c["Sk"], c["D"], c["dtype"], c["seed"])
    g = np.random.default_rng(c["seed"])
    rows = max(c["Sq"], c["Sk"]) + 16
    pq = pk = None
    if c["pos"] == "random":
        pq = g.integers(-1, rows, c["Sq"]).astype(np.int32)
        pk = g.integers(-1, rows, c["Sk"]).astype(np.int32)
    c32, s32 = oracle_tables(1e4, c["rd"], rows)
    cg, sg = torch.from_numpy(c32).cuda(), torch.from_numpy(s32).cuda()
    args = (q.cuda(), k.cuda(), v.cuda(), cg, sg)
    kw = dict(pos_q=None if pq is None else torch.from_numpy(pq).cuda(),
              pos_k=None if pk is None else torch.from_numpy(pk).cuda(),
              rotary_dim=c["rd"], layout=c["layout"], causal=c["causal"])
    o = R.attention(*args, **kw)
    o_in = R.attention(*args, k_workspace=None, **kw)
    assert R.rope_check_errors() == R.ROPE_OK
    assert torch.equal(o.view(torch.int16), o_in.view(torch.int16)), "key paths differ"
    _check(o, q, k, v, c["dtype"], c["rd"], W.LAYOUTS[c["layout"]], c32, s32, pq, pk, c["causal"],
           str(c))


def test_attention_full_size_sampled_rows():
    """The bench's attention workload at full size (Q [4,32,4096,128], K/V
    [4,8,4096,128] bf16, causal, theta 5e5) through the workspace path, in
    the configuration the bench times (2048 work units on the persistent
    clusters).  Sampled query rows against the oracle: row i at its own
    position, against the keys 0..i it can see, is exactly that row of the
    causal attention."""
    require_gpu()
    R = lib()
    B, Hq, Hk, S, D, rd = 4, 32, 8, 4096, 128, 128
    q, k, v = _inputs(B, Hq, Hk, S, S, D, "bf16", 6)
    c32, s32 = oracle_tables(5e5, rd, S)
    cg, sg = torch.from_numpy(c32).cuda(), torch.from_numpy(s32).cuda()
    o = R.attention(q.cuda(), k.cuda(), v.cuda(), cg, sg, causal=True).cpu()
    assert R.rope_check_errors() == R.ROPE_OK
    rng = np.random.default_rng(11)
    rows = [(0, 0, 0), (3, 31, S - 1), (1, 5, 127), (2, 17, 128), (0, 30, 2047), (3, 2, 4095)]
    rows += [(int(rng.integers(B)), int(rng.integers(Hq)), int(rng.integers(S))) for _ in range(18)]
    group = Hq // Hk
    for b, h, i in rows:
        kv = h // group
        ref = OA.attention(W.bits(q[b:b + 1, h:h + 1, i:i + 1]), W.bits(k[b:b + 1, kv:kv + 1, :i + 1]),
                           W.bits(v[b:b + 1, kv:kv + 1, :i + 1]), O.BF16, rd, O.SPLIT_HALF, c32, s32,
                           np.array([i], dtype=np.int32), None, True)
        got = o[b:b + 1, h:h + 1, i:i + 1].float().numpy().astype(np.float64)
        vmax = float(v[b, kv, :i + 1].float().abs().max())
        tol = U["bf16"] * (vmax + np.abs(ref))
        assert np.all(np.abs(got - ref) <= tol), "row (%d, %d, %d): max err %.3g" % (
            b, h, i, np.abs(got - ref).max())


@pytest.mark.parametrize("chunks", [1, 2, 3, 6])
def test_host_attention_pipeline_matches_device_call(chunks):
    """Pinned host Q, K, V through the chunked copy/attend/copy pipeline give
    the device call's bits, and leave the host inputs untouched (6 pieces:
    each batch entry's two key/value heads apart)."""
    require_gpu()
    R = lib()
    from rotary_position_embedding_rope_gb300.host import HostAttention

    q, k, v = _inputs(3, 4, 2, 200, 230, 128, "bf16", seed=17)
    cos, sin = R.build_tables(10000.0, 128, 256)
    hq, hk, hv = q.pin_memory(), k.pin_memory(), v.pin_memory()
    ho = torch.full_like(q, float("nan")).pin_memory()
    hat = HostAttention(chunks=chunks)
    for causal in (True, False):
        hat.forward(hq, hk, hv, ho, cos, sin, causal=causal).synchronize()
        want = R.attention(q.cuda(), k.cuda(), v.cuda(), cos, sin, causal=causal)
        torch.cuda.synchronize()
        assert R.rope_check_errors() == R.ROPE_OK
        assert torch.equal(ho, want.cpu())
    assert torch.equal(hq, q) and torch.equal(hk, k) and torch.equal(hv, v)
