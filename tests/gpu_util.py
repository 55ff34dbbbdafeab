"""Helpers for the GPU tests: building/loading the CUDA library, moving the
same input bits to the GPU and to the oracle, and the comparison rules.

Comparison rules (tolerances written here, used by every GPU test):
  * fp32 outputs: max |gpu - y| <= 2e-6, y the oracle's fp64 result computed
    with fp64 cos/sin (the exact method) -- and also against the oracle run
    on the same fp32 table.
  * bf16/fp16 outputs: every element within 1 unit in the last place of the
    oracle's fp64 result rounded once to the output type, the oracle using
    the same fp32 table values as the GPU (an fp32 table entry carries an
    error of up to |x| 2^-25, larger than one bf16 ulp of y when x1 c and
    x2 s nearly cancel, so the table is part of the method's input).
  * pass-through tail, masked tokens, position gathers: bit-exact.
"""
from __future__ import annotations

import functools

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W

FP32_ABS_TOL = 2e-6
ULP_TOL_16 = 1

ORACLE_DTYPE = {"f32": O.F32, "bf16": O.BF16, "f16": O.F16}


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@functools.lru_cache(maxsize=None)
def lib():
    import rotary_position_embedding_rope_gb300 as R
    from rotary_position_embedding_rope_gb300 import _build

    _build.build()
    R.load_library()
    return R


@functools.lru_cache(maxsize=8)
def oracle_tables(theta, rd, rows, f=1.0, precision="f32"):
    return O.load().tables(theta, rd, rows, f, precision)


def ordered16(bits: np.ndarray) -> np.ndarray:
    """Map 16-bit float patterns to integers ordered like their values (-0 == +0)."""
    v = bits.astype(np.int64)
    return np.where(v < 0x8000, v, 0x8000 - v)


def ulp_distance16(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    return np.abs(ordered16(a_bits) - ordered16(b_bits))


def gpu_bits(t: torch.Tensor) -> np.ndarray:
    return W.bits(t.detach().cpu())


def assert_matches(dtype: str, got_bits: np.ndarray, want_bits: np.ndarray,
                   want_f64: np.ndarray | None, what: str = ""):
    """Apply the comparison rule of the output type."""
    if dtype == "f32":
        err = np.abs(got_bits.astype(np.float64) - want_f64)
        assert np.all(np.isfinite(got_bits)), what
        assert err.max(initial=0.0) <= FP32_ABS_TOL, "%s: max abs error %.3g" % (what, err.max())
    else:
        d = ulp_distance16(got_bits, want_bits)
        bad = np.count_nonzero(d > ULP_TOL_16)
        assert bad == 0, "%s: %d elements beyond %d ulp (max %d)" % (what, bad, ULP_TOL_16, d.max())
        assert all_finite16(dtype, got_bits), what


def all_finite16(dtype: str, bits: np.ndarray) -> bool:
    """No infinity or NaN among 16-bit float patterns (exponent field not all ones)."""
    e = np.uint16(0x7F80 if dtype == "bf16" else 0x7C00)
    return not np.any((bits & e) == e)


def to_gpu(t):
    return None if t is None else t.cuda()


def pos_tensor(pos: np.ndarray | None):
    return None if pos is None else torch.from_numpy(np.ascontiguousarray(pos, dtype=np.int32)).cuda()


def run_apply(w: W.Workload, q: torch.Tensor, k: torch.Tensor | None, cos: torch.Tensor,
              sin: torch.Tensor, pos: torch.Tensor | None, backward: bool, stream=None):
    R = lib()
    R.rope_apply_qk(q, k, cos, sin, pos, w.B, w.Hq, w.Hk if k is not None else 0, w.S, w.D,
                    w.rotary_dim, W.LAYOUTS[w.layout], int(w.seq_before_head), int(backward),
                    W.DTYPES[w.dtype], cos.shape[0], stream)


def oracle_apply(w: W.Workload, x_bits: np.ndarray, H: int, pos, backward: bool,
                 cos: np.ndarray, sin: np.ndarray):
    rc, yb, y64 = O.load().apply(x_bits, ORACLE_DTYPE[w.dtype], w.B, H, w.S, w.D, w.rotary_dim,
                                 W.LAYOUTS[w.layout], w.seq_before_head, backward, pos, cos, sin)
    assert rc == O.OK, rc
    return yb, y64
