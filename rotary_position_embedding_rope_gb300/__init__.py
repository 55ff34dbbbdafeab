"""Python binding of librope: rotary position embedding on GB300 (sm_103a).

The functions named like the C ABI (``rope_tables_build``, ``rope_apply_qk``,
``rope_apply_q``, ``rope_check_errors``, ``rope_status_string``,
``rope_qk_kernel_variant``) take the same arguments as ``include/rope.h``,
with torch tensors (or raw integer addresses) in place of pointers and a
torch stream (or raw handle, or None for torch's current stream) in place of
``void* stream``.  They only marshal arguments: every step runs in the CUDA
library, and a missing library is an error, never a fallback.

``build_tables``, ``apply_qk``, ``apply_q`` and ``rotate_qk`` are conveniences
that read the sizes from tensor shapes and allocate tables and outputs with
torch; ``PreparedApply`` checks a rotation's arguments once for calls
repeated on tensors of one shape.  ``autograd.rotary_qk`` wraps the out-of-place call in a
``torch.autograd.Function`` (backward = rotation by the negated angle).
``build_tables_ex`` builds the table of a frequency mode ('lang', 'pixel',
'constant') at given positions, optionally XPOS-scaled; ``apply_qk_xpos``
rotates Q and K with their own XPOS tables.  ``attention`` calls
``rope_attention_fwd`` (``rope_attention_fwd_masked`` with an ``attn_mask``):
attention with the rotation fused into the Q/K tile loads (or, with a key
workspace, keys rotated once beforehand).
``host.HostRotator`` and ``host.HostAttention`` run the rotation and the
attention on tensors that live in pinned host memory, overlapping the copies
with the calls.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

__all__ = [
    "RopeError", "ROPE_OK", "ROPE_ERR_INVALID_ARG", "ROPE_ERR_UNSUPPORTED", "ROPE_ERR_CUDA",
    "ROPE_ERR_POS_OUT_OF_RANGE", "ROPE_ERR_KERNEL_TIMEOUT", "VARIANT_ELEMENTWISE", "VARIANT_VECTOR",
    "ROPE_SPLIT_HALF", "ROPE_INTERLEAVED", "ROPE_F32", "ROPE_BF16", "ROPE_F16", "ROPE_FREQ_LANG",
    "ROPE_FREQ_PIXEL", "ROPE_FREQ_CONSTANT", "ROPE_MASK_NONE", "ROPE_MASK_KEYS",
    "ROPE_MASK_QUERY_KEYS", "library_path", "load_library",
    # the C ABI, same names
    "rope_tables_build", "rope_tables_build_ex", "rope_apply_qk", "rope_apply_q",
    "rope_apply_qk_out", "rope_attention_fwd", "rope_attention_fwd_masked",
    "rope_attention_fwd_noalloc", "rope_check_errors", "rope_probe_wait_expiry",
    "rope_status_string", "rope_qk_kernel_variant", "rope_force_kernel_variant",
    "rope_tune_rotation_launch",
    # conveniences
    "build_tables", "build_tables_ex", "apply_qk", "apply_q", "apply_qk_xpos", "rotate_qk",
    "attention", "attention_workspace", "PreparedApply",
]

(ROPE_OK, ROPE_ERR_INVALID_ARG, ROPE_ERR_UNSUPPORTED, ROPE_ERR_CUDA, ROPE_ERR_POS_OUT_OF_RANGE,
 ROPE_ERR_KERNEL_TIMEOUT) = range(6)
VARIANT_ELEMENTWISE, VARIANT_VECTOR = 2, 3
ROPE_SPLIT_HALF, ROPE_INTERLEAVED = 0, 1
ROPE_F32, ROPE_BF16, ROPE_F16 = 0, 1, 2
ROPE_FREQ_LANG, ROPE_FREQ_PIXEL, ROPE_FREQ_CONSTANT = 0, 1, 2
ROPE_MASK_NONE, ROPE_MASK_KEYS, ROPE_MASK_QUERY_KEYS = 0, 1, 2
_FREQ_CODE = {"lang": ROPE_FREQ_LANG, "pixel": ROPE_FREQ_PIXEL, "constant": ROPE_FREQ_CONSTANT}
_DTYPE_CODE = {torch.float32: ROPE_F32, torch.bfloat16: ROPE_BF16, torch.float16: ROPE_F16}
_LAYOUT_CODE = {"split_half": ROPE_SPLIT_HALF, "interleaved": ROPE_INTERLEAVED}


class RopeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s" % (where, rope_status_string(status)))


_lib = None


def library_path() -> str:
    """lib/librope.so, or the library ROPE_LIBRARY names (a build of the same
    sources with other compile-time settings, made with
    ``_build.build(extra_flags=[...], output=...)``, for timing variants)."""
    return os.environ.get("ROPE_LIBRARY") or _build.LIBRARY


def load_library() -> ctypes.CDLL:
    """Load lib/librope.so (built by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path) and os.environ.get("ROPE_LIBRARY"):
        raise RuntimeError("ROPE_LIBRARY names %s, which does not exist" % path)
    if not os.path.exists(path):
        raise RuntimeError(
            "librope.so is not built (%s); run `python -c \"import __graft_entry__ as g; "
            "g.build()\"` first" % path)
    lib = ctypes.CDLL(path)
    c = ctypes
    P = c.c_void_p
    lib.rope_tables_build.argtypes = [c.c_double, c.c_int32, c.c_int64, c.c_double, P, P, P]
    lib.rope_tables_build.restype = c.c_int
    lib.rope_tables_build_ex.argtypes = [c.c_int32, c.c_double, c.c_double, c.c_int32, c.c_int64,
                                         c.c_double, c.c_double, c.c_int32, c.c_double, c.c_double,
                                         c.c_double, P, P, P]
    lib.rope_tables_build_ex.restype = c.c_int
    lib.rope_apply_qk.argtypes = [P, P, P, P, P, c.c_int64, c.c_int32, c.c_int32, c.c_int64,
                                  c.c_int32, c.c_int32, c.c_int32, c.c_int32, c.c_int32,
                                  c.c_int32, c.c_int64, P]
    lib.rope_apply_qk.restype = c.c_int
    lib.rope_apply_q.argtypes = [P, P, P, P, c.c_int64, c.c_int32, c.c_int64, c.c_int32,
                                 c.c_int32, c.c_int32, c.c_int32, c.c_int32, c.c_int32,
                                 c.c_int64, P]
    lib.rope_apply_q.restype = c.c_int
    lib.rope_check_errors.argtypes = [P]
    lib.rope_check_errors.restype = c.c_int
    lib.rope_probe_wait_expiry.argtypes = [c.c_int64, P]
    lib.rope_probe_wait_expiry.restype = c.c_int
    lib.rope_status_string.argtypes = [c.c_int]
    lib.rope_status_string.restype = c.c_char_p
    lib.rope_qk_kernel_variant.argtypes = [P, P, P, P, P, c.c_int64, c.c_int32, c.c_int32,
                                           c.c_int64, c.c_int32, c.c_int32, c.c_int32,
                                           c.c_int32, c.c_int32, c.c_int32, c.c_int64]
    lib.rope_qk_kernel_variant.restype = c.c_int32
    lib.rope_apply_qk_out.argtypes = [P, P, P, P, P, P, P, c.c_int64, c.c_int64, c.c_int32,
                                      c.c_int32, c.c_int64, c.c_int32, c.c_int32, c.c_int32,
                                      c.c_int32, c.c_int32, c.c_int32, c.c_int64, P]
    lib.rope_apply_qk_out.restype = c.c_int
    lib.rope_attention_fwd.argtypes = [P, P, P, P, P, P, P, P, c.c_int64, c.c_int32, c.c_int32,
                                       c.c_int64, c.c_int64, c.c_int32, c.c_int32, c.c_int32,
                                       c.c_int32, c.c_float, c.c_int32, c.c_int64, P,
                                       c.c_int64, P]
    lib.rope_attention_fwd.restype = c.c_int
    lib.rope_attention_fwd_masked.argtypes = [P, P, P, P, P, P, P, P, c.c_int64, c.c_int32,
                                              c.c_int32, c.c_int64, c.c_int64, c.c_int32,
                                              c.c_int32, c.c_int32, c.c_int32, c.c_float,
                                              c.c_int32, c.c_int64, P, c.c_int32, P, c.c_int64, P]
    lib.rope_attention_fwd_masked.restype = c.c_int
    lib.rope_attention_fwd_noalloc.argtypes = [P, P, P, P, P, P, P, P, c.c_int64, c.c_int32,
                                               c.c_int32, c.c_int64, c.c_int64, c.c_int32,
                                               c.c_int32, c.c_int32, c.c_int32, c.c_float,
                                               c.c_int32, c.c_int64, P]
    lib.rope_attention_fwd_noalloc.restype = c.c_int
    lib.rope_force_kernel_variant.argtypes = [c.c_int32]
    lib.rope_force_kernel_variant.restype = c.c_int
    lib.rope_tune_rotation_launch.argtypes = [c.c_int32, c.c_int32, c.c_int32]
    lib.rope_tune_rotation_launch.restype = c.c_int
    _lib = lib
    return lib


# --------------------------------------------------------------------------
# marshalling
# --------------------------------------------------------------------------
def _addr(x, name: str, device_required: bool = True):
    """Device address of a tensor (checked contiguous, on CUDA) or a raw int."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if isinstance(x, torch.Tensor):
        if device_required and not x.is_cuda:
            raise ValueError("%s must be a CUDA tensor" % name)
        if not x.is_contiguous():
            raise ValueError("%s must be contiguous" % name)
        return x.data_ptr() if x.numel() > 0 else None
    raise TypeError("%s: expected a tensor, an int address or None" % name)


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str):
    if status != ROPE_OK:
        raise RopeError(status, where)


# --------------------------------------------------------------------------
# functions of the C ABI, same names and arguments
# --------------------------------------------------------------------------
def rope_tables_build(theta, rotary_dim, max_pos, interpolate_factor, cos_out, sin_out,
                      stream=None):
    lib = load_library()
    for t, n in ((cos_out, "cos_out"), (sin_out, "sin_out")):
        if isinstance(t, torch.Tensor) and (t.dtype != torch.float32 or
                                            t.numel() < max_pos * (rotary_dim // 2)):
            raise ValueError("%s must be float32 with at least max_pos*rotary_dim/2 elements" % n)
    st = lib.rope_tables_build(float(theta), int(rotary_dim), int(max_pos),
                               float(interpolate_factor), _addr(cos_out, "cos_out"),
                               _addr(sin_out, "sin_out"), _stream(stream))
    _check(st, "rope_tables_build")


def rope_tables_build_ex(freq_mode, theta, max_freq, rotary_dim, rows, pos_offset, pos_divisor,
                         xpos_sign, xpos_scale_base, xpos_gamma, xpos_center, cos_out, sin_out,
                         stream=None):
    lib = load_library()
    for t, n in ((cos_out, "cos_out"), (sin_out, "sin_out")):
        if isinstance(t, torch.Tensor) and (t.dtype != torch.float32 or
                                            t.numel() < rows * (rotary_dim // 2)):
            raise ValueError("%s must be float32 with at least rows*rotary_dim/2 elements" % n)
    st = lib.rope_tables_build_ex(int(freq_mode), float(theta), float(max_freq), int(rotary_dim),
                                  int(rows), float(pos_offset), float(pos_divisor), int(xpos_sign),
                                  float(xpos_scale_base), float(xpos_gamma), float(xpos_center),
                                  _addr(cos_out, "cos_out"), _addr(sin_out, "sin_out"),
                                  _stream(stream))
    _check(st, "rope_tables_build_ex")


def rope_apply_qk(q, k, cos, sin, pos_idx, B, Hq, Hk, S, D, rotary_dim, layout,
                  seq_before_head, backward, dtype, table_rows, stream=None):
    lib = load_library()
    st = lib.rope_apply_qk(_addr(q, "q"), _addr(k, "k"), _addr(cos, "cos"), _addr(sin, "sin"),
                           _addr(pos_idx, "pos_idx"), int(B), int(Hq), int(Hk), int(S), int(D),
                           int(rotary_dim), int(layout), int(seq_before_head), int(backward),
                           int(dtype), int(table_rows), _stream(stream))
    _check(st, "rope_apply_qk")


def rope_apply_qk_out(q, k, q_out, k_out, cos, sin, pos_idx, pos_batch_stride, B, Hq, Hk, S, D,
                      rotary_dim, layout, seq_before_head, backward, dtype, table_rows,
                      stream=None):
    lib = load_library()
    st = lib.rope_apply_qk_out(_addr(q, "q"), _addr(k, "k"), _addr(q_out, "q_out"),
                               _addr(k_out, "k_out"), _addr(cos, "cos"), _addr(sin, "sin"),
                               _addr(pos_idx, "pos_idx"), int(pos_batch_stride), int(B), int(Hq),
                               int(Hk), int(S), int(D), int(rotary_dim), int(layout),
                               int(seq_before_head), int(backward), int(dtype), int(table_rows),
                               _stream(stream))
    _check(st, "rope_apply_qk_out")


def rope_apply_q(x, cos, sin, pos_idx, B, H, S, D, rotary_dim, layout, seq_before_head,
                 backward, dtype, table_rows, stream=None):
    lib = load_library()
    st = lib.rope_apply_q(_addr(x, "x"), _addr(cos, "cos"), _addr(sin, "sin"),
                          _addr(pos_idx, "pos_idx"), int(B), int(H), int(S), int(D),
                          int(rotary_dim), int(layout), int(seq_before_head), int(backward),
                          int(dtype), int(table_rows), _stream(stream))
    _check(st, "rope_apply_q")


def rope_check_errors(stream=None) -> int:
    """Synchronise the stream; returns the status (does not raise)."""
    return load_library().rope_check_errors(_stream(stream))


def rope_probe_wait_expiry(cycles: int, stream=None) -> int:
    """Launch one bounded wait that expires after `cycles` clock cycles and
    sets the timeout bit of the device flag (the next rope_check_errors
    returns ROPE_ERR_KERNEL_TIMEOUT).  Returns the launch status."""
    return load_library().rope_probe_wait_expiry(int(cycles), _stream(stream))


def rope_status_string(status: int) -> str:
    return load_library().rope_status_string(int(status)).decode()


def rope_qk_kernel_variant(q, k, cos, sin, pos_idx, B, Hq, Hk, S, D, rotary_dim, layout,
                           seq_before_head, backward, dtype, table_rows) -> int:
    lib = load_library()
    return lib.rope_qk_kernel_variant(
        _addr(q, "q", False), _addr(k, "k", False), _addr(cos, "cos", False),
        _addr(sin, "sin", False), _addr(pos_idx, "pos_idx", False), int(B), int(Hq), int(Hk),
        int(S), int(D), int(rotary_dim), int(layout), int(seq_before_head), int(backward),
        int(dtype), int(table_rows))


def rope_force_kernel_variant(variant: int):
    _check(load_library().rope_force_kernel_variant(int(variant)), "rope_force_kernel_variant")


def rope_tune_rotation_launch(ctas_per_sm: int = 0, min_units: int = 0, prefetch_next: int = 0):
    """Grid sizing of the vector rotation kernel (0 = defaults); results do
    not depend on it."""
    _check(load_library().rope_tune_rotation_launch(int(ctas_per_sm), int(min_units),
                                                    int(prefetch_next)),
           "rope_tune_rotation_launch")


# --------------------------------------------------------------------------
# conveniences
# --------------------------------------------------------------------------
def build_tables(theta: float, rotary_dim: int, max_pos: int, interpolate_factor: float = 1.0,
                 device=None, stream=None):
    """Allocate and fill fp32 cos/sin tables [max_pos, rotary_dim // 2]."""
    device = torch.device("cuda") if device is None else torch.device(device)
    h = rotary_dim // 2
    cos = torch.empty((max_pos, h), dtype=torch.float32, device=device)
    sin = torch.empty((max_pos, h), dtype=torch.float32, device=device)
    rope_tables_build(theta, rotary_dim, max_pos, interpolate_factor, cos, sin, stream)
    return cos, sin


def build_tables_ex(freqs_for: str, rotary_dim: int, rows: int, theta: float = 10000.0,
                    max_freq: float = 10.0, pos_offset: float = 0.0, pos_divisor: float = 1.0,
                    xpos_sign: int = 0, xpos_scale_base: float = 512.0, xpos_gamma: float = 0.4,
                    xpos_center: float = 0.0, device=None, stream=None):
    """Allocate and fill fp32 cos/sin tables [rows, rotary_dim // 2] of the mode
    ``freqs_for`` ('lang', 'pixel' or 'constant'), row m at position
    pos_offset + m / pos_divisor, XPOS-scaled when xpos_sign is +1 (queries) or
    -1 (keys)."""
    device = torch.device("cuda") if device is None else torch.device(device)
    h = rotary_dim // 2
    cos = torch.empty((rows, h), dtype=torch.float32, device=device)
    sin = torch.empty((rows, h), dtype=torch.float32, device=device)
    rope_tables_build_ex(_FREQ_CODE[freqs_for], theta, max_freq, rotary_dim, rows, pos_offset,
                         pos_divisor, xpos_sign, xpos_scale_base, xpos_gamma, xpos_center, cos,
                         sin, stream)
    return cos, sin


def _shape4(x: torch.Tensor, seq_before_head: bool):
    if x.dim() != 4:
        raise ValueError("expected a 4-D tensor, got shape %s" % (tuple(x.shape),))
    if seq_before_head:
        B, S, H, D = x.shape
    else:
        B, H, S, D = x.shape
    return B, H, S, D


def apply_qk(q: torch.Tensor, k: torch.Tensor | None, cos: torch.Tensor, sin: torch.Tensor,
             pos_idx: torch.Tensor | None = None, rotary_dim: int | None = None,
             layout: str = "split_half", seq_before_head: bool = False, backward: bool = False,
             stream=None):
    """Rotate q and k in place; sizes are read from the tensors.

    q: [B, Hq, S, D] (or [B, S, Hq, D] with seq_before_head); k likewise with
    Hk heads, or None.  cos/sin: float32 [rows, rotary_dim // 2].
    pos_idx: int32 [S] or None.  rotary_dim defaults to 2 * cos.shape[1].
    """
    B, Hq, S, D = _shape4(q, seq_before_head)
    Hk = 0
    if k is not None:
        Bk, Hk, Sk, Dk = _shape4(k, seq_before_head)
        if (Bk, Sk, Dk) != (B, S, D) or k.dtype != q.dtype:
            raise ValueError("q and k must agree in batch, sequence, head_dim and dtype")
    if q.dtype not in _DTYPE_CODE:
        raise TypeError("unsupported dtype %s" % q.dtype)
    if cos.dtype != torch.float32 or sin.dtype != torch.float32 or cos.shape != sin.shape:
        raise ValueError("cos and sin must be float32 tables of the same shape")
    rd = 2 * cos.shape[1] if rotary_dim is None else rotary_dim
    if cos.shape[1] != rd // 2:
        raise ValueError("table width %d does not match rotary_dim %d" % (cos.shape[1], rd))
    if pos_idx is not None and (pos_idx.dtype != torch.int32 or pos_idx.numel() != S):
        raise ValueError("pos_idx must be int32 with S elements")
    rope_apply_qk(q, k, cos, sin, pos_idx, B, Hq, Hk, S, D, rd, _LAYOUT_CODE[layout],
                  int(seq_before_head), int(backward), _DTYPE_CODE[q.dtype], cos.shape[0],
                  stream)
    return q, k


class PreparedApply:
    """rope_apply_qk with every argument but q and k checked and converted
    once, for calls repeated on tensors of one shape (a model layer, a decode
    loop): each call marshals two pointers and the fixed rest.

        f = PreparedApply(q, k, cos, sin, stream=s)   # shapes, tables, layout
        f(q, k)                  # forward, in place
        f(dq, dk, backward=True)

    q and k of later calls must have the shapes and dtype of the ones given
    here (their element counts are checked; raw integer addresses are passed
    as they are).  The stream is fixed here (None: torch's current stream at
    this point).  Only marshalling: the library does the work."""

    def __init__(self, q, k, cos, sin, pos_idx=None, rotary_dim=None, layout="split_half",
                 seq_before_head=False, stream=None):
        B, Hq, S, D = _shape4(q, seq_before_head)
        Hk = 0
        if k is not None:
            Bk, Hk, Sk, Dk = _shape4(k, seq_before_head)
            if (Bk, Sk, Dk) != (B, S, D) or k.dtype != q.dtype:
                raise ValueError("q and k must agree in batch, sequence, head_dim and dtype")
        if q.dtype not in _DTYPE_CODE:
            raise TypeError("unsupported dtype %s" % q.dtype)
        if cos.dtype != torch.float32 or sin.dtype != torch.float32 or cos.shape != sin.shape:
            raise ValueError("cos and sin must be float32 tables of the same shape")
        rd = 2 * cos.shape[1] if rotary_dim is None else rotary_dim
        if cos.shape[1] != rd // 2:
            raise ValueError("table width %d does not match rotary_dim %d" % (cos.shape[1], rd))
        if pos_idx is not None and (pos_idx.dtype != torch.int32 or pos_idx.numel() != S):
            raise ValueError("pos_idx must be int32 with S elements")
        c = ctypes
        self._fn = load_library().rope_apply_qk
        self._keep = (cos, sin, pos_idx)
        self._nq, self._nk = q.numel(), 0 if k is None else k.numel()
        head = [c.c_void_p(_addr(cos, "cos")), c.c_void_p(_addr(sin, "sin")),
                c.c_void_p(_addr(pos_idx, "pos_idx")), c.c_int64(B), c.c_int32(Hq),
                c.c_int32(Hk), c.c_int64(S), c.c_int32(D), c.c_int32(rd),
                c.c_int32(_LAYOUT_CODE[layout]), c.c_int32(int(seq_before_head))]
        tail = [c.c_int32(_DTYPE_CODE[q.dtype]), c.c_int64(cos.shape[0]),
                c.c_void_p(_stream(stream))]
        self._fwd = tuple(head + [c.c_int32(0)] + tail)
        self._bwd = tuple(head + [c.c_int32(1)] + tail)

    def __call__(self, q, k=None, backward: bool = False):
        if isinstance(q, int):
            qp = q
        else:
            if q.numel() != self._nq:
                raise ValueError("q does not have the prepared shape")
            qp = q.data_ptr()
        if k is None or isinstance(k, int):
            kp = k
        else:
            if k.numel() != self._nk:
                raise ValueError("k does not have the prepared shape")
            kp = k.data_ptr()
        st = self._fn(qp, kp, *(self._bwd if backward else self._fwd))
        if st != ROPE_OK:
            raise RopeError(st, "rope_apply_qk")


def apply_q(x: torch.Tensor, cos: torch.Tensor, sin: torch.Tensor,
            pos_idx: torch.Tensor | None = None, rotary_dim: int | None = None,
            layout: str = "split_half", seq_before_head: bool = False, backward: bool = False,
            stream=None):
    """Rotate one tensor in place through the query-only entry point."""
    B, H, S, D = _shape4(x, seq_before_head)
    if x.dtype not in _DTYPE_CODE:
        raise TypeError("unsupported dtype %s" % x.dtype)
    if cos.dtype != torch.float32 or sin.dtype != torch.float32 or cos.shape != sin.shape:
        raise ValueError("cos and sin must be float32 tables of the same shape")
    rd = 2 * cos.shape[1] if rotary_dim is None else rotary_dim
    if cos.shape[1] != rd // 2:
        raise ValueError("table width %d does not match rotary_dim %d" % (cos.shape[1], rd))
    if pos_idx is not None and (pos_idx.dtype != torch.int32 or pos_idx.numel() != S):
        raise ValueError("pos_idx must be int32 with S elements")
    rope_apply_q(x, cos, sin, pos_idx, B, H, S, D, rd, _LAYOUT_CODE[layout],
                 int(seq_before_head), int(backward), _DTYPE_CODE[x.dtype], cos.shape[0], stream)
    return x


def apply_qk_xpos(q: torch.Tensor, k: torch.Tensor, tables_q, tables_k,
                  pos_idx: torch.Tensor | None = None, rotary_dim: int | None = None,
                  layout: str = "split_half", seq_before_head: bool = False,
                  backward: bool = False, stream=None):
    """XPOS: rotate Q with its table (xpos_sign +1) and K with its table
    (xpos_sign -1), in place: one launch per tensor."""
    apply_q(q, tables_q[0], tables_q[1], pos_idx, rotary_dim, layout, seq_before_head, backward,
            stream)
    apply_q(k, tables_k[0], tables_k[1], pos_idx, rotary_dim, layout, seq_before_head, backward,
            stream)
    return q, k


def _positions(pos_idx, B: int, S: int):
    """(tensor, batch stride) for an int32 [S] or [B, S'] (S' >= S) position tensor."""
    if pos_idx is None:
        return None, 0
    if pos_idx.dtype != torch.int32:
        raise ValueError("pos_idx must be int32")
    if pos_idx.dim() == 1:
        if pos_idx.numel() != S:
            raise ValueError("pos_idx [S] must have S elements")
        return pos_idx, 0
    if pos_idx.dim() == 2 and pos_idx.shape[0] == B and pos_idx.shape[1] >= S:
        return pos_idx, pos_idx.shape[1]
    raise ValueError("pos_idx must be [S] or [B, >=S]")


def rotate_qk(q: torch.Tensor, k: torch.Tensor | None, cos: torch.Tensor, sin: torch.Tensor,
              pos_idx: torch.Tensor | None = None, rotary_dim: int | None = None,
              layout: str = "split_half", seq_before_head: bool = False, backward: bool = False,
              q_out: torch.Tensor | None = None, k_out: torch.Tensor | None = None, stream=None):
    """Out-of-place rotation: returns (q_out, k_out), allocated when not given.

    pos_idx: int32 [S] (shared by all sequences) or [B, S] (one row per
    sequence).  Passing q_out=q (k_out=k) rotates that tensor in place.
    """
    B, Hq, S, D = _shape4(q, seq_before_head)
    Hk = 0
    if k is not None:
        Bk, Hk, Sk, Dk = _shape4(k, seq_before_head)
        if (Bk, Sk, Dk) != (B, S, D) or k.dtype != q.dtype:
            raise ValueError("q and k must agree in batch, sequence, head_dim and dtype")
    if q.dtype not in _DTYPE_CODE:
        raise TypeError("unsupported dtype %s" % q.dtype)
    if cos.dtype != torch.float32 or sin.dtype != torch.float32 or cos.shape != sin.shape:
        raise ValueError("cos and sin must be float32 tables of the same shape")
    rd = 2 * cos.shape[1] if rotary_dim is None else rotary_dim
    if cos.shape[1] != rd // 2:
        raise ValueError("table width %d does not match rotary_dim %d" % (cos.shape[1], rd))
    pos, stride = _positions(pos_idx, B, S)
    q_out = torch.empty_like(q) if q_out is None else q_out
    if k is not None and k_out is None:
        k_out = torch.empty_like(k)
    for o, x, n in ((q_out, q, "q_out"), (k_out, k, "k_out")):
        if x is not None and (o.shape != x.shape or o.dtype != x.dtype):
            raise ValueError("%s must match its input's shape and dtype" % n)
    rope_apply_qk_out(q, k, q_out, k_out if k is not None else None, cos, sin, pos, stride, B, Hq,
                      Hk, S, D, rd, _LAYOUT_CODE[layout], int(seq_before_head), int(backward),
                      _DTYPE_CODE[q.dtype], cos.shape[0], stream)
    return q_out, k_out


def rope_attention_fwd(q, k, v, o, cos, sin, pos_q, pos_k, B, Hq, Hk, Sq, Sk, D, rotary_dim,
                       layout, causal, softmax_scale, dtype, table_rows, k_workspace=None,
                       workspace_bytes=0, stream=None):
    lib = load_library()
    st = lib.rope_attention_fwd(_addr(q, "q"), _addr(k, "k"), _addr(v, "v"), _addr(o, "o"),
                                _addr(cos, "cos"), _addr(sin, "sin"), _addr(pos_q, "pos_q"),
                                _addr(pos_k, "pos_k"), int(B), int(Hq), int(Hk), int(Sq), int(Sk),
                                int(D), int(rotary_dim), int(layout), int(causal),
                                float(softmax_scale), int(dtype), int(table_rows),
                                _addr(k_workspace, "k_workspace"), int(workspace_bytes),
                                _stream(stream))
    _check(st, "rope_attention_fwd")


def rope_attention_fwd_masked(q, k, v, o, cos, sin, pos_q, pos_k, B, Hq, Hk, Sq, Sk, D, rotary_dim,
                              layout, causal, softmax_scale, dtype, table_rows, attn_mask,
                              mask_kind, k_workspace=None, workspace_bytes=0, stream=None):
    lib = load_library()
    st = lib.rope_attention_fwd_masked(_addr(q, "q"), _addr(k, "k"), _addr(v, "v"), _addr(o, "o"),
                                       _addr(cos, "cos"), _addr(sin, "sin"), _addr(pos_q, "pos_q"),
                                       _addr(pos_k, "pos_k"), int(B), int(Hq), int(Hk), int(Sq),
                                       int(Sk), int(D), int(rotary_dim), int(layout), int(causal),
                                       float(softmax_scale), int(dtype), int(table_rows),
                                       _addr(attn_mask, "attn_mask"), int(mask_kind),
                                       _addr(k_workspace, "k_workspace"), int(workspace_bytes),
                                       _stream(stream))
    _check(st, "rope_attention_fwd_masked")


def rope_attention_fwd_noalloc(q, k, v, o, cos, sin, pos_q, pos_k, B, Hq, Hk, Sq, Sk, D,
                               rotary_dim, layout, causal, softmax_scale, dtype, table_rows,
                               stream=None):
    """rope_attention_fwd with the rot(K) buffer taken from the library's own
    32 MiB device array: for callers that cannot allocate device memory when
    they call (their memory is all reserved by their own pool, or they may
    only use buffers their host framework gives them).  Allocates nothing."""
    lib = load_library()
    st = lib.rope_attention_fwd_noalloc(_addr(q, "q"), _addr(k, "k"), _addr(v, "v"),
                                        _addr(o, "o"), _addr(cos, "cos"), _addr(sin, "sin"),
                                        _addr(pos_q, "pos_q"), _addr(pos_k, "pos_k"), int(B),
                                        int(Hq), int(Hk), int(Sq), int(Sk), int(D),
                                        int(rotary_dim), int(layout), int(causal),
                                        float(softmax_scale), int(dtype), int(table_rows),
                                        _stream(stream))
    _check(st, "rope_attention_fwd_noalloc")


def attention_workspace(k: torch.Tensor, attn_mask: torch.Tensor | None = None) -> torch.Tensor:
    """A key workspace for rope_attention_fwd(_masked) on keys like k: rot(K)
    and, for a [B, Sk] attn_mask, the per-batch key-tile counts after it (with
    them the kernels skip the key tiles the mask hides entirely), then the
    per-batch prefix lengths (an entry whose mask shows exactly its first L
    keys, as padding does, is then computed without reading the mask)."""
    kb = k.numel() * k.element_size()
    n = kb
    if attn_mask is not None and attn_mask.dim() == 2:
        n = (kb + 15) // 16 * 16 + 8 * k.shape[0]
    return torch.empty(n, dtype=torch.uint8, device=k.device)


def attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cos: torch.Tensor,
              sin: torch.Tensor, pos_q: torch.Tensor | None = None,
              pos_k: torch.Tensor | None = None, rotary_dim: int | None = None,
              layout: str = "split_half", causal: bool = False, scale: float | None = None,
              out: torch.Tensor | None = None, k_workspace="auto",
              attn_mask: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """softmax(scale * rot(q) rot(k)^T + mask) v with q [B,Hq,Sq,D], k/v [B,Hk,Sk,D].

    k_workspace: "auto" allocates a buffer (attention_workspace) that receives
    rot(K) (the keys are rotated once, then read rotated by the attention
    kernel); a tensor of at least k's size is used as that buffer; None
    rotates the key tiles inside the attention kernel instead (nothing extra
    is written).  The result is the same bit for bit.
    attn_mask: None, or a bool (or uint8) CUDA tensor [B, Sk] (one entry per
    key) or [B, Sq, Sk] (one per query and key); False hides the key from the
    query, together with the causal mask.
    """
    B, Hq, Sq, D = q.shape
    _, Hk, Sk, _ = k.shape
    if v.shape != k.shape or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("k and v must have the same shape, and q, k, v the same dtype")
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise TypeError("attention takes bf16 or fp16 q, k, v (the tensor-core products are 16-bit); "
                        "got %s: convert the inputs first (e.g. q.bfloat16()), a rounding that is "
                        "the caller's choice" % q.dtype)
    rd = 2 * cos.shape[1] if rotary_dim is None else rotary_dim
    o = torch.empty_like(q) if out is None else out
    if isinstance(k_workspace, str):
        if k_workspace != "auto":
            raise ValueError("k_workspace must be 'auto', None or a tensor")
        k_workspace = attention_workspace(k, attn_mask)
    ws_bytes = 0 if k_workspace is None else k_workspace.numel() * k_workspace.element_size()
    args = (q, k, v, o, cos, sin, pos_q, pos_k, B, Hq, Hk, Sq, Sk, D, rd, _LAYOUT_CODE[layout],
            int(causal), -1.0 if scale is None else scale, _DTYPE_CODE[q.dtype], cos.shape[0])
    if attn_mask is None:
        rope_attention_fwd(*args, k_workspace, ws_bytes, stream)
        return o
    if attn_mask.dtype not in (torch.bool, torch.uint8):
        raise TypeError("attn_mask must be bool or uint8")
    if tuple(attn_mask.shape) == (B, Sk):
        kind = ROPE_MASK_KEYS
    elif tuple(attn_mask.shape) == (B, Sq, Sk):
        kind = ROPE_MASK_QUERY_KEYS
    else:
        raise ValueError("attn_mask must be [B, Sk] or [B, Sq, Sk], got %s" %
                         (tuple(attn_mask.shape),))
    rope_attention_fwd_masked(*args, attn_mask, kind, k_workspace, ws_bytes, stream)
    return o
