"""rope_attention_fwd_noalloc: the rotary attention with its key workspace
in a fixed 32 MiB device array of the library, for callers that cannot
allocate device memory at call time (an engine that keeps all device memory
in its own pool, a plugin limited to the buffers its host framework hands
it).  The GPU test compares it with rope_attention_fwd given a
caller-allocated workspace, on two calls in a row with different shapes and
data, so the second call also shows that the shared array left over from the
first does not leak into its result.  Tolerance: the attention tests' bound,
|o - o_ref| <= u (max|v| + |o_ref|), u = 2^-8 (bf16) or 2^-10 (fp16).

The file is named to be collected last: if it fails, a run that stops at the
first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from gpu_util import lib, oracle_tables, require_gpu
from rotary_position_embedding_rope_gb300 import _build

U = {"bf16": 2.0 ** -8, "f16": 2.0 ** -10}
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
        got, v = _run(R, c, noalloc=True)
        want, _ = _run(R, c, noalloc=False)
        g = got.float().cpu().numpy().astype(np.float64)
        w = want.float().cpu().numpy().astype(np.float64)
        tol = U[c["dtype"]] * (float(v.float().abs().max()) + np.abs(w))
        assert np.all(np.isfinite(g)), str(c)
        err = np.abs(g - w)
        assert np.all(err <= tol), "%s: %d beyond tolerance, max err %.3g" % (
            c, np.count_nonzero(err > tol), err.max())


def test_noalloc_rejects_keys_beyond_its_array():
    """B * Hk * Sk * D * 2 bytes above 32 MiB: ROPE_ERR_UNSUPPORTED before
    the device is touched (the pointers here are never dereferenced)."""
    import rotary_position_embedding_rope_gb300 as R

    _build.build()
    L = R.load_library()
    A = 0x10000
    Sk = SCRATCH_BYTES // (128 * 2) + 1            # one key row past the array
    st = L.rope_attention_fwd_noalloc(A, A * 100, A * 200, A * 300, A * 400, A * 500, None, None,
                                      1, 1, 1, 1, Sk, 128, 128, 0, 0, ctypes.c_float(-1.0), 1,
                                      Sk, None)
    assert st == R.ROPE_ERR_UNSUPPORTED
