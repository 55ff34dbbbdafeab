"""rope_attention_fwd_noalloc: the rotary attention with its key workspace
in a fixed 32 MiB device array of the library, for callers that cannot
allocate device memory at call time (an engine that keeps all device memory
in its own pool, a plugin limited to the buffers its host framework hands
it).  The GPU test compares it with rope_attention_fwd given a
caller-allocated workspace, on two calls in a row with different shapes and
data, so the second call also shows that the shared array left over from the
first does not leak into its result.  Both entry points run the same two
kernels on the same inputs, so their outputs must be equal bit for bit: any
difference would mean the shared array changed the result.

The file is named to be collected last: if it fails, a run that stops at the
first failure has already run every other test.
"""
import ctypes

import pytest
import torch

import workloads as W
from gpu_util import lib, oracle_tables, require_gpu
from rotary_position_embedding_rope_gb300 import _build

DTYPE_CODE = {"bf16": 1, "f16": 2}
SCRATCH_BYTES = 32 << 20

CALLS = [
    dict(B=1, Hq=4, Hk=2, Sq=300, Sk=300, D=128, rd=128, dtype="bf16", causal=True, seed=41),
    dict(B=2, Hq=6, Hk=3, Sq=200, Sk=517, D=64, rd=32, dtype="f16", causal=False, seed=42),
]


def _run(R, c, noalloc):
    g = torch.Generator().manual_seed(c["seed"])
    q = W.draw((c["B"], c["Hq"], c["Sq"], c["D"]), c["dtype"], g).cuda()
    k = W.draw((c["B"], c["Hk"], c["Sk"], c["D"]), c["dtype"], g).cuda()
    v = W.draw((c["B"], c["Hk"], c["Sk"], c["D"]), c["dtype"], g).cuda()
    rows = max(c["Sq"], c["Sk"]) + 8
    c32, s32 = oracle_tables(1e4, c["rd"], rows)
    cg, sg = torch.from_numpy(c32).cuda(), torch.from_numpy(s32).cuda()
    o = torch.empty_like(q)
    args = (q, k, v, o, cg, sg, None, None, c["B"], c["Hq"], c["Hk"], c["Sq"], c["Sk"], c["D"],
            c["rd"], R.ROPE_SPLIT_HALF, int(c["causal"]), -1.0, DTYPE_CODE[c["dtype"]], rows)
    if noalloc:
        R.rope_attention_fwd_noalloc(*args)
    else:
        ws = torch.empty_like(k)
        R.rope_attention_fwd(*args, ws, ws.numel() * ws.element_size())
    torch.cuda.synchronize()
    assert R.rope_check_errors() == R.ROPE_OK
    return o, v


@pytest.mark.gpu
def test_noalloc_matches_the_workspace_entry_point_on_two_calls():
    require_gpu()
    R = lib()
    for c in CALLS:
        got, _ = _run(R, c, noalloc=True)
        want, _ = _run(R, c, noalloc=False)
        assert torch.equal(got.view(torch.int16), want.view(torch.int16)), str(c)
        assert torch.isfinite(got.float()).all(), str(c)


def test_noalloc_rejects_keys_beyond_its_array():
    """B * Hk * Sk * D * 2 bytes above 32 MiB: ROPE_ERR_UNSUPPORTED before
    the device is touched (the pointers here are never dereferenced); the
    arguments are checked first, as rope_attention_fwd checks them, so an
    oversized call that is also invalid (Hq not a multiple of Hk) gets that
    error instead."""
    import rotary_position_embedding_rope_gb300 as R

    _build.build()
    L = R.load_library()
    A = 1 << 32                                    # buffers 4 GiB apart: none overlaps
    Sk = SCRATCH_BYTES // (128 * 2) + 1            # one key row past the array
    st = L.rope_attention_fwd_noalloc(A, A * 2, A * 3, A * 4, A * 5, A * 6, None, None,
                                      1, 1, 1, 1, Sk, 128, 128, 0, 0, ctypes.c_float(-1.0), 1,
                                      Sk, None)
    assert st == R.ROPE_ERR_UNSUPPORTED
    st = L.rope_attention_fwd_noalloc(A, A * 2, A * 3, A * 4, A * 5, A * 6, None, None,
                                      1, 3, 2, 1, Sk, 128, 128, 0, 0, ctypes.c_float(-1.0), 1,
                                      Sk, None)
    assert st == R.ROPE_ERR_INVALID_ARG
