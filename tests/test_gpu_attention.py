"""Attention with the rotation fused into the Q/K tile loads (tcgen05) against
the fp64 rotary-attention oracle, on both key paths: keys rotated inside the
attention kernel (no workspace) and keys rotated once into a workspace by the
rotation kernel.  The two paths give the same bits.

Tolerance (attention_check.py): the kernel rounds P to the element type
before the P.V product and rounds O once, so per output element
|o - O| <= (u + 2^-14)(W + |O|) (+ 2^-25 A for fp16's subnormal P), with
u = 2^-8 (bf16) or 2^-11 (fp16) and W = sum_j p_j |v_j| / l,
A = sum_j vis_j |v_j| / l from the oracle.
"""
import numpy as np
import pytest
import torch

import attention_check as AC
import oracle as O
import workloads as W
from gpu_util import lib, oracle_tables, require_gpu
from oracle import attention as OA

pytestmark = pytest.mark.gpu
CODE = {"bf16": O.BF16, "f16": O.F16}


def _inputs(B, Hq, Hk, Sq, Sk, D, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    q = W.draw((B, Hq, Sq, D), dtype, g)
    k = W.draw((B, Hk, Sk, D), dtype, g)
    v = W.draw((B, Hk, Sk, D), dtype, g)
    return q, k, v


def _check(got, q, k, v, dtype, rd, layout, c32, s32, pq, pk, causal, what="", attn_mask=None):
    ref, w, a = OA.attention(W.bits(q), W.bits(k), W.bits(v), CODE[dtype], rd, layout, c32, s32,
                             pq, pk, causal, want_bounds=True, attn_mask=attn_mask)
    return AC.check(got.float().cpu().numpy(), ref, w, a, dtype, what)


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


def _cid(c):
    return "B%d_Hq%d_Hk%d_Sq%d_Sk%d_D%d_rd%d_%s_%s_c%d" % (
        c["B"], c["Hq"], c["Hk"], c["Sq"], c["Sk"], c["D"], c["rd"], c["dtype"], c["layout"],
        c["causal"])


@pytest.mark.parametrize("ws", sorted(WS))
@pytest.mark.parametrize("c", CASES, ids=_cid)
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
           c["causal"], "case %s %s" % (_cid(c), ws))


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
           "fuzz%02d" % c["i"])


def _masked_fuzz_cases(n=16, seed=4048):
    g = np.random.default_rng(seed)
    cases = _fuzz_cases(n, seed)
    for c in cases:
        c["mask"] = str(g.choice(["keys", "query_keys"]))
        c["density"] = float(g.choice([0.1, 0.5, 0.9, 1.0]))
    return cases


@pytest.mark.parametrize("c", _masked_fuzz_cases(), ids=lambda c: "mfuzz%02d" % c["i"])
def test_attention_masked_fuzz(c):
    """Seeded random shapes, spans, layouts, types, positions and attn_masks
    ([B, Sk] or [B, Sq, Sk], 10 % to all keys visible, byte-aligned or not):
    the workspace path against the oracle, the in-kernel key path bit for bit
    against it."""
    require_gpu()
    R = lib()
    q, k, v = _inputs(c["B"], c["Hq"], c["Hk"], c["Sq"], c["Sk"], c["D"], c["dtype"], c["seed"])
    g = np.random.default_rng(c["seed"] + 1)
    rows = max(c["Sq"], c["Sk"]) + 16
    pq = pk = None
    if c["pos"] == "random":
        pq = g.integers(-1, rows, c["Sq"]).astype(np.int32)
        pk = g.integers(-1, rows, c["Sk"]).astype(np.int32)
    shape = (c["B"], c["Sk"]) if c["mask"] == "keys" else (c["B"], c["Sq"], c["Sk"])
    m = g.random(shape) < c["density"]
    c32, s32 = oracle_tables(1e4, c["rd"], rows)
    cg, sg = torch.from_numpy(c32).cuda(), torch.from_numpy(s32).cuda()
    args = (q.cuda(), k.cuda(), v.cuda(), cg, sg)
    kw = dict(pos_q=None if pq is None else torch.from_numpy(pq).cuda(),
              pos_k=None if pk is None else torch.from_numpy(pk).cuda(),
              rotary_dim=c["rd"], layout=c["layout"], causal=c["causal"],
              attn_mask=torch.from_numpy(m).cuda())
    o = R.attention(*args, **kw)
    o_in = R.attention(*args, k_workspace=None, **kw)
    assert R.rope_check_errors() == R.ROPE_OK
    assert torch.equal(o.view(torch.int16), o_in.view(torch.int16)), "key paths differ"
    _check(o, q, k, v, c["dtype"], c["rd"], W.LAYOUTS[c["layout"]], c32, s32, pq, pk, c["causal"],
           "mfuzz%02d" % c["i"], attn_mask=m)


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
        ref, w, a = OA.attention(W.bits(q[b:b + 1, h:h + 1, i:i + 1]),
                                 W.bits(k[b:b + 1, kv:kv + 1, :i + 1]),
                                 W.bits(v[b:b + 1, kv:kv + 1, :i + 1]), O.BF16, rd, O.SPLIT_HALF,
                                 c32, s32, np.array([i], dtype=np.int32), None, True,
                                 want_bounds=True)
        AC.check(o[b:b + 1, h:h + 1, i:i + 1].float().numpy(), ref, w, a, "bf16",
                 "full size sampled rows: row (%d, %d, %d)" % (b, h, i))


def tile_indicator_values(Sk, D):
    """v[j, d] = 1 when (j // 128) % D == d: output column d of a row is the
    softmax mass of the key tiles d, d + D, ... alone."""
    v = torch.zeros((Sk, D), dtype=torch.bfloat16)
    v[torch.arange(Sk), (torch.arange(Sk) // 128) % D] = 1.0
    return v


@pytest.mark.parametrize("ws", sorted(WS))
def test_attention_full_length_tile_indicator_values(ws):
    """The Llama-shaped causal prefill at full length (Sq = Sk = 4096, GQA
    32/8, D = 128, bf16) with values that mark their key tile: each output
    column carries one key tile's softmax mass, so a skipped, repeated or
    misplaced key tile moves whole columns far outside the bound (the CPU
    test of attention_check shows the rule rejecting a skipped tile and a zero
    output on these rows).  Sampled query rows against the oracle, on both
    key paths."""
    require_gpu()
    R = lib()
    B, Hq, Hk, S, D, rd = 1, 32, 8, 4096, 128, 128
    g = torch.Generator().manual_seed(6)
    q = W.draw((B, Hq, S, D), "bf16", g)
    k = W.draw((B, Hk, S, D), "bf16", g)
    v = tile_indicator_values(S, D)[None, None].expand(B, Hk, S, D).contiguous()
    c32, s32 = oracle_tables(5e5, rd, S)
    cg, sg = torch.from_numpy(c32).cuda(), torch.from_numpy(s32).cuda()
    o = R.attention(q.cuda(), k.cuda(), v.cuda(), cg, sg, causal=True, k_workspace=WS[ws]).cpu()
    assert R.rope_check_errors() == R.ROPE_OK
    rng = np.random.default_rng(13)
    rows = [(0, 0), (31, 4095), (5, 127), (17, 128), (30, 2047), (2, 4000), (9, 255), (12, 3071)]
    rows += [(int(rng.integers(Hq)), int(rng.integers(S))) for _ in range(16)]
    for h, i in rows:
        kv = h // (Hq // Hk)
        ref, w, a = OA.attention(W.bits(q[:, h:h + 1, i:i + 1]), W.bits(k[:, kv:kv + 1, :i + 1]),
                                 W.bits(v[:, kv:kv + 1, :i + 1]), O.BF16, rd, O.SPLIT_HALF, c32,
                                 s32, np.array([i], dtype=np.int32), None, True, want_bounds=True)
        AC.check(o[:, h:h + 1, i:i + 1].float().numpy(), ref, w, a, "bf16",
                 "tile indicator values (%s): head %d row %d" % (ws, h, i))


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


MASK_CASES = [
    dict(B=3, Hq=4, Hk=2, Sq=300, Sk=300, D=128, rd=128, dtype="bf16", layout="split_half", causal=True),
    dict(B=3, Hq=4, Hk=2, Sq=200, Sk=333, D=128, rd=64, dtype="f16", layout="interleaved", causal=False),
    dict(B=3, Hq=6, Hk=2, Sq=260, Sk=260, D=64, rd=32, dtype="bf16", layout="split_half", causal=True),
    dict(B=3, Hq=3, Hk=1, Sq=129, Sk=400, D=64, rd=64, dtype="f16", layout="split_half", causal=False),
]


def _key_mask(B, Sk, seed):
    """Per batch entry: all keys, a padded tail, a hidden whole key tile plus
    scattered keys."""
    m = np.ones((B, Sk), dtype=bool)
    if B > 1:
        m[1, Sk - 77:] = False
    if B > 2:
        m[2, 10:140] = False
        m[2, np.random.default_rng(seed).integers(0, Sk, Sk // 5)] = False
    return m


@pytest.mark.parametrize("ws", sorted(WS))
@pytest.mark.parametrize("c", MASK_CASES, ids=_cid)
def test_attention_key_padding_mask(c, ws):
    """attn_mask [B, Sk] ("rotary-embedding-torch", Input Tensor Shapes):
    padded batches, a whole key tile hidden, scattered keys; with and without
    the causal mask, on both key paths."""
    require_gpu()
    R = lib()
    q, k, v = _inputs(c["B"], c["Hq"], c["Hk"], c["Sq"], c["Sk"], c["D"], c["dtype"], 51)
    m = _key_mask(c["B"], c["Sk"], 5)
    rows = max(c["Sq"], c["Sk"]) + 8
    c32, s32 = oracle_tables(1e4, c["rd"], rows)
    cg, sg = torch.from_numpy(c32).cuda(), torch.from_numpy(s32).cuda()
    o = R.attention(q.cuda(), k.cuda(), v.cuda(), cg, sg, rotary_dim=c["rd"], layout=c["layout"],
                    causal=c["causal"], k_workspace=WS[ws], attn_mask=torch.from_numpy(m).cuda())
    assert R.rope_check_errors() == R.ROPE_OK
    _check(o, q, k, v, c["dtype"], c["rd"], W.LAYOUTS[c["layout"]], c32, s32, None, None,
           c["causal"], "key mask %s %s" % (_cid(c), ws), attn_mask=m)


@pytest.mark.parametrize("ws", sorted(WS))
@pytest.mark.parametrize("Sk", [320, 333])
def test_attention_per_query_mask(Sk, ws):
    """attn_mask [B, Sq, Sk]: random visibility, one query row with every key
    hidden (zeros), one batch entry all visible; rows read as 16-byte vectors
    (Sk = 320) or byte by byte (Sk = 333)."""
    require_gpu()
    R = lib()
    B, Hq, Hk, Sq, D, rd = 2, 4, 2, 200, 128, 128
    q, k, v = _inputs(B, Hq, Hk, Sq, Sk, D, "bf16", 52)
    g = np.random.default_rng(9)
    m = g.random((B, Sq, Sk)) < 0.7
    m[0, 17] = False
    m[1] = True
    c32, s32 = oracle_tables(1e4, rd, Sk + 8)
    cg, sg = torch.from_numpy(c32).cuda(), torch.from_numpy(s32).cuda()
    for causal in (False, True):
        o = R.attention(q.cuda(), k.cuda(), v.cuda(), cg, sg, causal=causal, k_workspace=WS[ws],
                        attn_mask=torch.from_numpy(m).cuda())
        assert R.rope_check_errors() == R.ROPE_OK
        _check(o, q, k, v, "bf16", rd, O.SPLIT_HALF, c32, s32, None, None, causal,
               "query mask Sk%d %s" % (Sk, ws), attn_mask=m)
        if not causal:
            assert torch.count_nonzero(o[0, :, 17]) == 0


@pytest.mark.parametrize("ws", sorted(WS))
def test_attention_mask_causal_pattern_equals_causal(ws):
    """A [B, Sq, Sk] mask shaped like the causal pattern gives the causal
    call's bits: the hidden keys contribute exact zeros (p = 2^-inf) to the
    sums and products the causal call skips; an all-False mask gives zeros."""
    require_gpu()
    R = lib()
    B, Hq, Hk, Sq, Sk, D = 1, 4, 2, 250, 390, 128
    q, k, v = _inputs(B, Hq, Hk, Sq, Sk, D, "bf16", 53)
    c32, s32 = oracle_tables(1e4, 128, Sk + 8)
    cg, sg = torch.from_numpy(c32).cuda(), torch.from_numpy(s32).cuda()
    qg, kg, vg = q.cuda(), k.cuda(), v.cuda()
    pat = torch.arange(Sk)[None, :] <= (torch.arange(Sq)[:, None] + (Sk - Sq))
    a = R.attention(qg, kg, vg, cg, sg, causal=True, k_workspace=WS[ws])
    b = R.attention(qg, kg, vg, cg, sg, causal=False, k_workspace=WS[ws],
                    attn_mask=pat[None].expand(B, Sq, Sk).contiguous().cuda())
    z = R.attention(qg, kg, vg, cg, sg, causal=True, k_workspace=WS[ws],
                    attn_mask=torch.zeros((B, Sk), dtype=torch.bool, device="cuda"))
    assert R.rope_check_errors() == R.ROPE_OK
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.count_nonzero(z) == 0


def test_host_attention_shape_change_without_sync():
    """HostAttention calls with different shapes back to back, no wait
    between them: each equals the device call bit for bit (the staging and
    workspace buffers of a replaced shape are not reused while queued work
    still reads or writes them)."""
    require_gpu()
    R = lib()
    from rotary_position_embedding_rope_gb300.host import HostAttention

    hat = HostAttention(chunks=2)
    cos, sin = R.build_tables(10000.0, 128, 512)
    outs = []
    for i, (B, S) in enumerate(((2, 400), (3, 130), (2, 400))):
        q, k, v = _inputs(B, 4, 2, S, S, 128, "bf16", seed=60 + i)
        hq, hk, hv = q.pin_memory(), k.pin_memory(), v.pin_memory()
        ho = torch.empty_like(hq).pin_memory()
        outs.append((q, k, v, ho, hat.forward(hq, hk, hv, ho, cos, sin, causal=True)))
    for q, k, v, ho, done in outs:
        done.synchronize()
        want = R.attention(q.cuda(), k.cuda(), v.cuda(), cos, sin, causal=True)
        torch.cuda.synchronize()
        assert torch.equal(ho, want.cpu())
    assert R.rope_check_errors() == R.ROPE_OK


@pytest.mark.parametrize("ws", sorted(WS))
def test_attention_full_size_key_padding_sampled_rows(ws):
    """The bench's masked attention call at full size: the Llama-shaped causal
    prefill with a [B, Sk] key-padding mask (batch entry b keeps its first
    S - 512 b keys).  Sampled query rows against the oracle: row i at its own
    position against the keys 0..i with the batch entry's mask."""
    require_gpu()
    R = lib()
    B, Hq, Hk, S, D, rd = 4, 32, 8, 4096, 128, 128
    q, k, v = _inputs(B, Hq, Hk, S, S, D, "bf16", 6)
    keep = S - 512 * np.arange(B)
    m = np.arange(S)[None, :] < keep[:, None]
    c32, s32 = oracle_tables(5e5, rd, S)
    cg, sg = torch.from_numpy(c32).cuda(), torch.from_numpy(s32).cuda()
    o = R.attention(q.cuda(), k.cuda(), v.cuda(), cg, sg, causal=True, k_workspace=WS[ws],
                    attn_mask=torch.from_numpy(m).cuda()).cpu()
    assert R.rope_check_errors() == R.ROPE_OK
    rng = np.random.default_rng(21)
    rows = [(0, 0, 4095), (3, 31, 4095), (3, 5, 2560), (2, 9, 3000), (1, 17, 3583), (1, 2, 3584)]
    rows += [(int(rng.integers(B)), int(rng.integers(Hq)), int(rng.integers(S))) for _ in range(12)]
    group = Hq // Hk
    for b, h, i in rows:
        kv = h // group
        ref, w, a = OA.attention(W.bits(q[b:b + 1, h:h + 1, i:i + 1]),
                                 W.bits(k[b:b + 1, kv:kv + 1, :i + 1]),
                                 W.bits(v[b:b + 1, kv:kv + 1, :i + 1]), O.BF16, rd, O.SPLIT_HALF,
                                 c32, s32, np.array([i], dtype=np.int32), None, False,
                                 want_bounds=True, attn_mask=m[b:b + 1, :i + 1])
        AC.check(o[b:b + 1, h:h + 1, i:i + 1].float().numpy(), ref, w, a, "bf16",
                 "full size key padding (%s): row (%d, %d, %d)" % (ws, b, h, i))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [64, 128])
def test_attention_skips_key_tiles_a_key_mask_hides(D, causal):
    """With room for them after rot(K) in the workspace, a [B, Sk] mask's
    per-entry key-tile counts are written there and the kernels skip the
    tiles past each entry's last visible key.  Entries: all keys visible;
    the first 130 (two tiles); none (zero tiles, an entry in the middle);
    exactly the first tile; only the last key.  After the counts come the
    entries' prefix lengths (-1 for the last entry, whose mask is not a
    prefix).  The call with both, one with room for the counts only (every
    mask byte read), one with a workspace of rot(K)'s size only (no counts,
    every tile computed) and the in-kernel key path give the same bits, and
    match the oracle."""
    require_gpu()
    R = lib()
    B, Hq, Hk, Sq, Sk = 5, 4, 2, 300, 700
    q, k, v = _inputs(B, Hq, Hk, Sq, Sk, D, "bf16", 71)
    m = np.zeros((B, Sk), dtype=bool)
    m[0] = True
    m[1, :130] = True
    m[3, :128] = True
    m[4, Sk - 1] = True
    c32, s32 = oracle_tables(1e4, D, Sk + 8)
    cg, sg = torch.from_numpy(c32).cuda(), torch.from_numpy(s32).cuda()
    qg, kg, vg, mg = q.cuda(), k.cuda(), v.cuda(), torch.from_numpy(m).cuda()
    ws = R.attention_workspace(kg, mg)
    kb = kg.numel() * kg.element_size()
    w0 = (kb + 15) // 16 * 16
    assert ws.numel() == w0 + 8 * B
    kw = dict(rotary_dim=D, causal=causal, attn_mask=mg)
    skip = R.attention(qg, kg, vg, cg, sg, k_workspace=ws, **kw)
    torch.cuda.synchronize()
    tiles = ws[w0:w0 + 4 * B].view(torch.int32).cpu().tolist()
    assert tiles == [6, 2, 0, 1, 6]
    assert ws[w0 + 4 * B:].view(torch.int32).cpu().tolist() == [Sk, 130, 0, 128, -1]
    counts = R.attention(qg, kg, vg, cg, sg, k_workspace=ws[:w0 + 4 * B].clone(), **kw)
    full = R.attention(qg, kg, vg, cg, sg, k_workspace=torch.empty_like(kg), **kw)
    inker = R.attention(qg, kg, vg, cg, sg, k_workspace=None, **kw)
    assert R.rope_check_errors() == R.ROPE_OK
    assert torch.equal(skip.view(torch.int16), full.view(torch.int16))
    assert torch.equal(skip.view(torch.int16), counts.view(torch.int16))
    assert torch.equal(skip.view(torch.int16), inker.view(torch.int16))
    assert torch.count_nonzero(skip[2]) == 0
    _check(skip, q, k, v, "bf16", D, O.SPLIT_HALF, c32, s32, None, None, causal,
           "tile skipping D%d c%d" % (D, causal), attn_mask=m)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("D", [64, 128])
def test_key_mask_prefix_lengths(D, dtype):
    """Prefix lengths of a [B, Sk] mask whose rows are 16-byte aligned (Sk =
    1024: read 16 bytes at a time): all keys visible (1024); the first 1000
    (1000, the first hidden key in another 16-byte chunk than the last
    visible one); the first 1000 and key 1020 (not a prefix: -1); all but
    key 5 (-1).  Entries with a length are computed without reading their
    mask: the same bits as the call that reads every byte (room for the
    counts only) and as the in-kernel key path, and the oracle's result."""
    require_gpu()
    R = lib()
    B, Hq, Hk, Sq, Sk = 4, 4, 2, 200, 1024
    q, k, v = _inputs(B, Hq, Hk, Sq, Sk, D, dtype, 79)
    m = np.ones((B, Sk), dtype=bool)
    m[1, 1000:] = False
    m[2, 1000:] = False
    m[2, 1020] = True
    m[3, 5] = False
    c32, s32 = oracle_tables(1e4, D, Sk + 8)
    cg, sg = torch.from_numpy(c32).cuda(), torch.from_numpy(s32).cuda()
    qg, kg, vg, mg = q.cuda(), k.cuda(), v.cuda(), torch.from_numpy(m).cuda()
    ws = R.attention_workspace(kg, mg)
    kb = kg.numel() * kg.element_size()
    w0 = (kb + 15) // 16 * 16
    kw = dict(rotary_dim=D, causal=False, attn_mask=mg)
    got = R.attention(qg, kg, vg, cg, sg, k_workspace=ws, **kw)
    torch.cuda.synchronize()
    assert ws[w0:w0 + 4 * B].view(torch.int32).cpu().tolist() == [8, 8, 8, 8]
    assert ws[w0 + 4 * B:].view(torch.int32).cpu().tolist() == [1024, 1000, -1, -1]
    counts = R.attention(qg, kg, vg, cg, sg, k_workspace=ws[:w0 + 4 * B].clone(), **kw)
    inker = R.attention(qg, kg, vg, cg, sg, k_workspace=None, **kw)
    assert R.rope_check_errors() == R.ROPE_OK
    assert torch.equal(got.view(torch.int16), counts.view(torch.int16))
    assert torch.equal(got.view(torch.int16), inker.view(torch.int16))
    _check(got, q, k, v, dtype, D, O.SPLIT_HALF, c32, s32, None, None, False,
           "prefix lengths D%d %s" % (D, dtype), attn_mask=m)
