"""The C-ABI library without a GPU: it loads, exports every symbol the
header declares, rejects bad arguments before touching the device, and picks
the kernel variant by its documented rules.  No call here launches work."""
import ctypes
import os
import re

import pytest

import rotary_position_embedding_rope_gb300 as R
from rotary_position_embedding_rope_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rope.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return R.load_library()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rope_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = header_functions()
    for want in ("rope_tables_build", "rope_apply_qk", "rope_apply_q", "rope_check_errors",
                 "rope_status_string"):
        assert want in names


def test_library_exports_every_header_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name
        assert isinstance(getattr(lib, name), ctypes._CFuncPtr)


def test_status_strings(lib):
    assert R.rope_status_string(R.ROPE_OK) == "ROPE_OK"
    assert R.rope_status_string(R.ROPE_ERR_POS_OUT_OF_RANGE) == "ROPE_ERR_POS_OUT_OF_RANGE"
    assert R.rope_status_string(99) == "ROPE_STATUS_UNKNOWN"


A16 = 0x10000  # fake, 16-byte aligned "device" addresses: never dereferenced on these paths
GOOD = dict(q=A16 * 1, k=A16 * 1000, cos=A16 * 2000, sin=A16 * 3000, pos=None, B=2, Hq=4, Hk=2,
            S=16, D=64, rd=64, layout=0, sbh=0, bwd=0, dtype=1, rows=16)


def qk_args(**over):
    a = dict(GOOD, **over)
    return (a["q"], a["k"], a["cos"], a["sin"], a["pos"], a["B"], a["Hq"], a["Hk"], a["S"],
            a["D"], a["rd"], a["layout"], a["sbh"], a["bwd"], a["dtype"], a["rows"])


@pytest.mark.parametrize("over,status", [
    (dict(dtype=3), R.ROPE_ERR_UNSUPPORTED),
    (dict(dtype=-1), R.ROPE_ERR_UNSUPPORTED),
    (dict(layout=2), R.ROPE_ERR_UNSUPPORTED),
    (dict(sbh=2), R.ROPE_ERR_INVALID_ARG),
    (dict(bwd=-1), R.ROPE_ERR_INVALID_ARG),
    (dict(B=-1), R.ROPE_ERR_INVALID_ARG),
    (dict(S=-5), R.ROPE_ERR_INVALID_ARG),
    (dict(Hq=-1), R.ROPE_ERR_INVALID_ARG),
    (dict(Hk=-1), R.ROPE_ERR_INVALID_ARG),
    (dict(D=0), R.ROPE_ERR_INVALID_ARG),
    (dict(rd=0), R.ROPE_ERR_INVALID_ARG),
    (dict(rd=63), R.ROPE_ERR_INVALID_ARG),
    (dict(rd=66), R.ROPE_ERR_INVALID_ARG),
    (dict(q=None), R.ROPE_ERR_INVALID_ARG),
    (dict(k=None), R.ROPE_ERR_INVALID_ARG),
    (dict(cos=None), R.ROPE_ERR_INVALID_ARG),
    (dict(sin=None), R.ROPE_ERR_INVALID_ARG),
    (dict(rows=0), R.ROPE_ERR_INVALID_ARG),
    (dict(rows=15), R.ROPE_ERR_INVALID_ARG),             # S > table_rows without pos_idx
    (dict(rows=-1), R.ROPE_ERR_INVALID_ARG),
    (dict(k=A16 * 1 + 64), R.ROPE_ERR_INVALID_ARG),      # q and k overlap
    (dict(cos=A16 * 1 + 128), R.ROPE_ERR_INVALID_ARG),   # q overlaps the table
    (dict(B=1 << 40, S=1 << 40), R.ROPE_ERR_INVALID_ARG),  # size overflow
])
def test_apply_rejects_bad_arguments(lib, over, status):
    args = qk_args(**over)
    assert lib.rope_qk_kernel_variant(*args) == 0
    assert lib.rope_apply_qk(*args, None) == status


@pytest.mark.parametrize("over", [dict(B=0), dict(S=0), dict(Hq=0, Hk=0),
                                  dict(B=0, q=None, k=None, cos=None, sin=None)])
def test_empty_problems_are_noops(lib, over):
    args = qk_args(**over)
    assert lib.rope_qk_kernel_variant(*args) == 0
    assert lib.rope_apply_qk(*args, None) == R.ROPE_OK


def test_q_only_rejects_bad_arguments(lib):
    assert lib.rope_apply_q(None, A16, A16 * 2, None, 1, 4, 8, 64, 64, 0, 0, 0, 1, 8, None) \
        == R.ROPE_ERR_INVALID_ARG
    assert lib.rope_apply_q(A16, A16 * 2, A16 * 3, None, 1, 4, 8, 64, 64, 0, 0, 0, 7, 8, None) \
        == R.ROPE_ERR_UNSUPPORTED
    assert lib.rope_apply_q(A16, A16 * 20, A16 * 30, None, 0, 4, 8, 64, 64, 0, 0, 0, 1, 8, None) \
        == R.ROPE_OK


@pytest.mark.parametrize("theta,rd,max_pos,f,cos,sin,status", [
    (0.0, 64, 8, 1.0, A16, A16 * 2, R.ROPE_ERR_INVALID_ARG),
    (-1.0, 64, 8, 1.0, A16, A16 * 2, R.ROPE_ERR_INVALID_ARG),
    (float("nan"), 64, 8, 1.0, A16, A16 * 2, R.ROPE_ERR_INVALID_ARG),
    (float("inf"), 64, 8, 1.0, A16, A16 * 2, R.ROPE_ERR_INVALID_ARG),
    (1e4, 64, 8, 0.0, A16, A16 * 2, R.ROPE_ERR_INVALID_ARG),
    (1e4, 63, 8, 1.0, A16, A16 * 2, R.ROPE_ERR_INVALID_ARG),
    (1e4, 0, 8, 1.0, A16, A16 * 2, R.ROPE_ERR_INVALID_ARG),
    (1e4, 64, -1, 1.0, A16, A16 * 2, R.ROPE_ERR_INVALID_ARG),
    (1e4, 64, 8, 1.0, None, A16 * 2, R.ROPE_ERR_INVALID_ARG),
    (1e4, 64, 8, 1.0, A16, A16 + 16, R.ROPE_ERR_INVALID_ARG),   # cos and sin overlap
    (1e4, 64, 0, 1.0, None, None, R.ROPE_OK),                  # empty table: no-op
])
def test_tables_build_rejects_bad_arguments(lib, theta, rd, max_pos, f, cos, sin, status):
    assert lib.rope_tables_build(theta, rd, max_pos, f, cos, sin, None) == status


TEX = dict(mode=0, theta=1e4, max_freq=10.0, rd=64, rows=16, off=0.0, div=1.0, sign=0, base=512.0,
           gamma=0.4, centre=0.0, cos=A16 * 2000, sin=A16 * 3000)


def tex_args(**over):
    a = dict(TEX, **over)
    return (a["mode"], a["theta"], a["max_freq"], a["rd"], a["rows"], a["off"], a["div"], a["sign"],
            a["base"], a["gamma"], a["centre"], a["cos"], a["sin"], None)


@pytest.mark.parametrize("over,status", [
    (dict(mode=3), R.ROPE_ERR_UNSUPPORTED),
    (dict(mode=-1), R.ROPE_ERR_UNSUPPORTED),
    (dict(rd=7), R.ROPE_ERR_INVALID_ARG),
    (dict(rd=0), R.ROPE_ERR_INVALID_ARG),
    (dict(rows=-1), R.ROPE_ERR_INVALID_ARG),
    (dict(theta=0.0), R.ROPE_ERR_INVALID_ARG),            # lang needs theta > 0
    (dict(mode=1, max_freq=0.0), R.ROPE_ERR_INVALID_ARG),  # pixel needs max_freq > 0
    (dict(div=0.0), R.ROPE_ERR_INVALID_ARG),
    (dict(div=float("inf")), R.ROPE_ERR_INVALID_ARG),
    (dict(off=float("nan")), R.ROPE_ERR_INVALID_ARG),
    (dict(sign=2), R.ROPE_ERR_INVALID_ARG),
    (dict(sign=1, base=0.0), R.ROPE_ERR_INVALID_ARG),
    (dict(sign=-1, gamma=0.0), R.ROPE_ERR_INVALID_ARG),
    (dict(sign=1, centre=float("inf")), R.ROPE_ERR_INVALID_ARG),
    (dict(cos=None), R.ROPE_ERR_INVALID_ARG),
    (dict(sin=A16 * 2000), R.ROPE_ERR_INVALID_ARG),        # outputs overlap
    (dict(rows=0, cos=None, sin=None), R.ROPE_OK),         # empty: no-op
])
def test_tables_build_ex_rejects_bad_arguments(lib, over, status):
    assert lib.rope_tables_build_ex(*tex_args(**over)) == status


@pytest.mark.parametrize("over,variant", [
    (dict(), 3),                                   # bf16 split-half, rd*2 = 128 B: vectorised
    (dict(layout=1), 3),
    (dict(dtype=0), 3),                            # fp32 rd=64: 256 B span
    (dict(dtype=2, sbh=1), 3),
    (dict(q=A16 + 2), 2),                          # q not 16-byte aligned
    (dict(k=A16 * 1000 + 8), 2),
    (dict(cos=A16 * 2000 + 4), 2),
    (dict(sin=A16 * 3000 + 4), 2),
    (dict(rd=8, D=64), 2),                         # 16-byte span: not whole vector pairs
    (dict(rd=16, D=64), 3),                        # 32-byte span (bf16)
    (dict(rd=16, D=64, dtype=0), 3),               # 64-byte span (fp32)
    (dict(rd=8, D=64, dtype=0), 3),                # 32-byte span (fp32)
    (dict(rd=2, D=34), 2),                         # odd sizes
    (dict(rd=32, D=36), 2),                        # rows of 72 B: not 16-byte aligned
    (dict(rd=32, D=40), 3),                        # rows of 80 B
    (dict(Hk=0, k=None), 3),
    (dict(pos=A16 * 4000, rows=8), 3),             # gather: S may exceed table_rows
    (dict(rd=1024, D=1024, dtype=0, cos=A16 * 2000, sin=A16 * 2100), 3),   # 128 vectors per half
    (dict(rd=1032, D=1032, dtype=0, cos=A16 * 2000, sin=A16 * 2100), 2),   # 129: element-wise
])
def test_kernel_variant_rules(lib, over, variant):
    assert lib.rope_qk_kernel_variant(*qk_args(**over)) == variant


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(R, "_lib", None)
    monkeypatch.setattr(R, "library_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        R.load_library()


def test_force_kernel_variant_rules(lib):
    try:
        for bad in (4, -1, 1):
            assert lib.rope_force_kernel_variant(bad) == R.ROPE_ERR_INVALID_ARG
        for forced, aligned_want, unaligned_want in ((0, 3, 2), (2, 2, 2), (3, 3, 0)):
            assert lib.rope_force_kernel_variant(forced) == R.ROPE_OK
            assert lib.rope_qk_kernel_variant(*qk_args()) == aligned_want
            assert lib.rope_qk_kernel_variant(*qk_args(q=A16 + 2)) == unaligned_want
        assert lib.rope_force_kernel_variant(3) == R.ROPE_OK
        # a forced kernel that does not fit the arguments is refused before any launch
        assert lib.rope_apply_qk(*qk_args(q=A16 + 2), None) == R.ROPE_ERR_UNSUPPORTED
    finally:
        lib.rope_force_kernel_variant(0)
    assert R.rope_status_string(R.ROPE_ERR_KERNEL_TIMEOUT) == "ROPE_ERR_KERNEL_TIMEOUT"


def out_args(**over):
    a = dict(q=A16 * 1, k=A16 * 1000, qo=A16 * 5000, ko=A16 * 6000, cos=A16 * 2000, sin=A16 * 3000,
             pos=None, stride=0, B=2, Hq=4, Hk=2, S=16, D=64, rd=64, layout=0, sbh=0, bwd=0,
             dtype=1, rows=16)
    a.update(over)
    return (a["q"], a["k"], a["qo"], a["ko"], a["cos"], a["sin"], a["pos"], a["stride"], a["B"],
            a["Hq"], a["Hk"], a["S"], a["D"], a["rd"], a["layout"], a["sbh"], a["bwd"], a["dtype"],
            a["rows"], None)


@pytest.mark.parametrize("over,status", [
    (dict(pos=A16 * 4000, stride=5), R.ROPE_ERR_INVALID_ARG),       # 0 < stride < S
    (dict(pos=A16 * 4000, stride=-1), R.ROPE_ERR_INVALID_ARG),
    (dict(qo=None), R.ROPE_ERR_INVALID_ARG),
    (dict(ko=None), R.ROPE_ERR_INVALID_ARG),
    (dict(qo=A16 * 1 + 64), R.ROPE_ERR_INVALID_ARG),                 # q_out overlaps q, not equal
    (dict(qo=A16 * 1000), R.ROPE_ERR_INVALID_ARG),                   # q_out over k
    (dict(ko=A16 * 5000 + 32), R.ROPE_ERR_INVALID_ARG),              # outputs overlap
    (dict(qo=A16 * 2000), R.ROPE_ERR_INVALID_ARG),                   # output over the table
    (dict(pos=A16 * 4000, stride=16, qo=A16 * 4000), R.ROPE_ERR_INVALID_ARG),  # output over positions
    (dict(dtype=9), R.ROPE_ERR_UNSUPPORTED),
])
def test_apply_out_rejects_bad_arguments(lib, over, status):
    assert lib.rope_apply_qk_out(*out_args(**over)) == status


def test_tune_rotation_launch_rules(lib):
    try:
        for bad in ((-1, 0, 0), (65, 0, 0), (0, -1, 0), (0, 0, 2), (0, 0, -2)):
            assert lib.rope_tune_rotation_launch(*bad) == R.ROPE_ERR_INVALID_ARG
        for good in ((0, 0, 0), (1, 1, -1), (64, 1000, 1), (3, 4, 0)):
            assert lib.rope_tune_rotation_launch(*good) == R.ROPE_OK
            # the kernel choice does not depend on the grid sizing
            assert lib.rope_qk_kernel_variant(*qk_args()) == 3
    finally:
        lib.rope_tune_rotation_launch(0, 0, 0)


def test_apply_out_empty_is_noop(lib):
    assert lib.rope_apply_qk_out(*out_args(B=0, qo=None, ko=None)) == R.ROPE_OK


def attn_args(**over):
    a = dict(q=A16 * 1, k=A16 * 100, v=A16 * 200, o=A16 * 300, cos=A16 * 400, sin=A16 * 500,
             pq=None, pk=None, B=1, Hq=4, Hk=2, Sq=64, Sk=64, D=128, rd=128, layout=0, causal=1,
             scale=-1.0, dtype=1, rows=64, ws=None, ws_bytes=0)
    a.update(over)
    return (a["q"], a["k"], a["v"], a["o"], a["cos"], a["sin"], a["pq"], a["pk"], a["B"], a["Hq"],
            a["Hk"], a["Sq"], a["Sk"], a["D"], a["rd"], a["layout"], a["causal"], a["scale"],
            a["dtype"], a["rows"], a["ws"], a["ws_bytes"], None)


@pytest.mark.parametrize("over,status", [
    (dict(dtype=0), R.ROPE_ERR_UNSUPPORTED),          # fp32 attention not offered
    (dict(D=96, rd=96), R.ROPE_ERR_UNSUPPORTED),
    (dict(rd=8), R.ROPE_ERR_UNSUPPORTED),
    (dict(rd=40), R.ROPE_ERR_UNSUPPORTED),
    (dict(layout=2), R.ROPE_ERR_UNSUPPORTED),
    (dict(Hq=3), R.ROPE_ERR_INVALID_ARG),              # not a multiple of Hk
    (dict(Hk=0), R.ROPE_ERR_INVALID_ARG),
    (dict(causal=2), R.ROPE_ERR_INVALID_ARG),
    (dict(o=None), R.ROPE_ERR_INVALID_ARG),
    (dict(o=A16 * 1), R.ROPE_ERR_INVALID_ARG),          # o over q
    (dict(o=A16 * 200 + 64), R.ROPE_ERR_INVALID_ARG),   # o over v
    (dict(rows=32), R.ROPE_ERR_INVALID_ARG),            # positions past the table
    (dict(q=A16 + 8), R.ROPE_ERR_UNSUPPORTED),          # not 16-byte aligned
    (dict(scale=float("nan")), R.ROPE_ERR_INVALID_ARG),
    # key workspace: B * Hk * Sk * D * 2 = 32768 bytes, aligned, disjoint
    (dict(ws=A16 * 600, ws_bytes=32767), R.ROPE_ERR_INVALID_ARG),       # too small
    (dict(ws=A16 * 600 + 8, ws_bytes=32768), R.ROPE_ERR_UNSUPPORTED),   # not 16-byte aligned
    (dict(ws=A16 * 100 + 16, ws_bytes=32768), R.ROPE_ERR_INVALID_ARG),  # over k
    (dict(ws=A16 * 300 + 16, ws_bytes=32768), R.ROPE_ERR_INVALID_ARG),  # over o
    (dict(ws=A16 * 400, ws_bytes=32768), R.ROPE_ERR_INVALID_ARG),       # over the cos table
])
def test_attention_rejects_bad_arguments(lib, over, status):
    assert lib.rope_attention_fwd(*attn_args(**over)) == status


def test_attention_empty_is_noop(lib):
    assert lib.rope_attention_fwd(*attn_args(Sq=0, q=None, o=None)) == R.ROPE_OK
    assert lib.rope_attention_fwd(*attn_args(B=0)) == R.ROPE_OK


@pytest.mark.parametrize("cycles", [0, -5, 4000000001])
def test_wait_probe_rejects_cycles_out_of_range(lib, cycles):
    # checked before any CUDA call: nothing is launched
    assert lib.rope_probe_wait_expiry(cycles, None) == R.ROPE_ERR_INVALID_ARG


def masked_args(mask=A16 * 700, kind=1, **over):
    a = list(attn_args(**over))
    # rope_attention_fwd's arguments with (attn_mask, mask_kind) before the workspace
    return tuple(a[:20] + [mask, kind] + a[20:])


@pytest.mark.parametrize("kw,status", [
    (dict(kind=3), R.ROPE_ERR_UNSUPPORTED),                       # mask kind outside the enum
    (dict(kind=-1), R.ROPE_ERR_UNSUPPORTED),
    (dict(mask=None, kind=1), R.ROPE_ERR_INVALID_ARG),            # a mask kind needs a mask
    (dict(mask=None, kind=2), R.ROPE_ERR_INVALID_ARG),
    (dict(mask=A16 * 300 + 16, kind=1), R.ROPE_ERR_INVALID_ARG),   # mask inside o
    (dict(mask=A16 * 300 - 64 * 64 + 16, kind=2), R.ROPE_ERR_INVALID_ARG),   # [B,Sq,Sk] reaches o
    (dict(mask=A16 * 800, kind=1, ws=A16 * 800 - 16 * 1024, ws_bytes=1 << 20), R.ROPE_ERR_INVALID_ARG),
    (dict(dtype=0), R.ROPE_ERR_UNSUPPORTED),                      # the plain call's rules apply
    (dict(Hq=3), R.ROPE_ERR_INVALID_ARG),
])
def test_masked_attention_rejects_bad_arguments(lib, kw, status):
    assert lib.rope_attention_fwd_masked(*masked_args(**kw)) == status


def test_masked_attention_empty_and_no_mask(lib):
    assert lib.rope_attention_fwd_masked(*masked_args(Sq=0, q=None, o=None)) == R.ROPE_OK
    # kind 0 ignores the pointer: the same checks as rope_attention_fwd
    assert lib.rope_attention_fwd_masked(*masked_args(mask=None, kind=0, dtype=0)) == \
        lib.rope_attention_fwd(*attn_args(dtype=0))


def test_masked_attention_workspace_with_key_tiles(lib):
    """A workspace with room for the key-tile counts of a [B, Sk] mask is
    checked over its whole used extent: rot(K), then B int32 counts from the
    next 16-byte boundary."""
    kb = 1 * 2 * 64 * 128 * 2                 # B * Hk * Sk * D * 2
    used = (kb + 15) // 16 * 16 + 4 * 1
    ws = A16 * 800
    # a mask right after rot(K) overlaps the counts of a workspace with room
    # for them (refused before anything touches the device)
    assert lib.rope_attention_fwd_masked(*masked_args(mask=ws + kb, kind=1, ws=ws,
                                                      ws_bytes=used)) == R.ROPE_ERR_INVALID_ARG
    # a per-query mask never uses the counts: the same placement then only
    # has to clear rot(K)'s kb bytes -- checked here through the overlap with
    # o instead, which is refused either way
    assert lib.rope_attention_fwd_masked(*masked_args(mask=A16 * 300, kind=2, ws=ws,
                                                      ws_bytes=used)) == R.ROPE_ERR_INVALID_ARG
    # with room for the prefix lengths too (4 bytes per entry), the extent
    # grows by them: a mask right after the counts now overlaps
    assert lib.rope_attention_fwd_masked(*masked_args(mask=ws + used, kind=1, ws=ws,
                                                      ws_bytes=used + 4)) == R.ROPE_ERR_INVALID_ARG


def test_attention_workspace_sizes():
    """attention_workspace: rot(K)'s bytes; for a [B, Sk] mask also the B
    key-tile counts from the next 16-byte boundary and the B prefix lengths
    after them; a [B, Sq, Sk] mask uses neither."""
    import torch
    B, Hk, Sk, D = 3, 2, 37, 64
    k = torch.empty((B, Hk, Sk, D), dtype=torch.bfloat16)
    kb = B * Hk * Sk * D * 2
    assert R.attention_workspace(k).numel() == kb
    assert R.attention_workspace(k, torch.ones((B, Sk), dtype=torch.bool)).numel() == \
        (kb + 15) // 16 * 16 + 8 * B
    assert R.attention_workspace(k, torch.ones((B, 5, Sk), dtype=torch.bool)).numel() == kb
    assert R.attention_workspace(k).dtype == torch.uint8


def test_attention_binding_names_the_dtypes_it_takes():
    """The Python attention call refuses fp32 tensors before any device work,
    naming bf16 / fp16 (the C entry point returns ROPE_ERR_UNSUPPORTED)."""
    import torch
    q = torch.zeros(1, 8, 16, 64)
    c = torch.zeros(16, 32)
    with pytest.raises(TypeError, match="bf16 or fp16"):
        R.attention(q, q.clone(), q.clone(), c, c.clone())


def test_rope_library_override(lib):
    """ROPE_LIBRARY makes the binding load another build (here the in-tree one
    under its own path); a missing file is named in the error.  Subprocesses:
    the binding keeps the library it loaded first."""
    import subprocess
    import sys
    code = ("import rotary_position_embedding_rope_gb300 as R; L = R.load_library(); "
            "print(L._name)")
    env = dict(os.environ, ROPE_LIBRARY=_build.LIBRARY)
    p = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       cwd=ROOT)
    assert p.returncode == 0, p.stderr
    assert p.stdout.strip() == _build.LIBRARY
    env["ROPE_LIBRARY"] = os.path.join(ROOT, "no_such_dir", "librope.so")
    p = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       cwd=ROOT)
    assert p.returncode != 0 and "ROPE_LIBRARY names" in p.stderr
