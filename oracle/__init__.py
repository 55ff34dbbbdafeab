"""fp64 CPU oracle for rotary position embedding -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It wraps ``rope_oracle.c`` (plain C,
single-threaded, fp64) through ctypes and shares no code with the CUDA
library.  See the header of ``rope_oracle.c`` for the sources it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "rope_oracle.c")
LIBRARY = os.path.join(HERE, "librope_oracle.so")

F32, BF16, F16, F64 = 0, 1, 2, 3
SPLIT_HALF, INTERLEAVED = 0, 1
FREQ_LANG, FREQ_PIXEL, FREQ_CONSTANT = 0, 1, 2
OK, BAD_ARG, POS_OUT_OF_RANGE = 0, 1, 4

# numpy container type used for the element bits of each oracle dtype
_STORAGE = {F32: np.float32, BF16: np.uint16, F16: np.uint16, F64: np.float64}

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def compile_library(source: str = SOURCE, output: str = LIBRARY) -> str:
    """Compile ``source`` with gcc into the shared library ``output``.

    ``-ffp-contract=off`` keeps every product and sum a separate IEEE
    operation, so x86-64 and aarch64 hosts compute identical results.
    """
    os.makedirs(os.path.dirname(output) or ".", exist_ok=True)
    tmp = output + ".tmp%d" % os.getpid()
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, source, "-lm"], check=True)
    os.replace(tmp, output)
    return output


def build(force: bool = False) -> str:
    """Build ``librope_oracle.so`` next to its source if missing or stale."""
    if force or not os.path.exists(LIBRARY) or (
        os.path.getmtime(LIBRARY) < os.path.getmtime(SOURCE)
    ):
        compile_library()
    return LIBRARY


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        c = ctypes
        lib.oracle_bf16_to_f64.argtypes = [c.c_uint16]
        lib.oracle_bf16_to_f64.restype = c.c_double
        lib.oracle_f16_to_f64.argtypes = [c.c_uint16]
        lib.oracle_f16_to_f64.restype = c.c_double
        lib.oracle_f64_to_bf16.argtypes = [c.c_double]
        lib.oracle_f64_to_bf16.restype = c.c_uint16
        lib.oracle_f64_to_f16.argtypes = [c.c_double]
        lib.oracle_f64_to_f16.restype = c.c_uint16
        lib.oracle_f64_to_f32.argtypes = [c.c_double]
        lib.oracle_f64_to_f32.restype = c.c_float
        lib.oracle_inv_freq.argtypes = [c.c_double, c.c_int32, c.c_int32]
        lib.oracle_inv_freq.restype = c.c_double
        lib.oracle_angle.argtypes = [c.c_int64, c.c_double, c.c_double]
        lib.oracle_angle.restype = c.c_double
        for name in ("oracle_tables_f64", "oracle_tables_f32"):
            fn = getattr(lib, name)
            fn.argtypes = [c.c_double, c.c_int32, c.c_int64, c.c_double, c.c_void_p, c.c_void_p]
            fn.restype = c.c_int
        lib.oracle_freq_ex.argtypes = [c.c_int32, c.c_double, c.c_double, c.c_int32, c.c_int32]
        lib.oracle_freq_ex.restype = c.c_double
        lib.oracle_position.argtypes = [c.c_int64, c.c_double, c.c_double]
        lib.oracle_position.restype = c.c_double
        lib.oracle_xpos_scale.argtypes = [c.c_int32, c.c_int32, c.c_double, c.c_int32, c.c_double,
                                          c.c_double, c.c_double]
        lib.oracle_xpos_scale.restype = c.c_double
        for name in ("oracle_tables_ex_f64", "oracle_tables_ex_f32"):
            fn = getattr(lib, name)
            fn.argtypes = [c.c_int32, c.c_double, c.c_double, c.c_int32, c.c_int64, c.c_double,
                           c.c_double, c.c_int32, c.c_double, c.c_double, c.c_double, c.c_void_p,
                           c.c_void_p]
            fn.restype = c.c_int
        lib.oracle_rotate_row_f64.argtypes = [
            c.c_void_p, c.c_void_p, c.c_int32, c.c_int32, c.c_int32,
            c.c_void_p, c.c_void_p, c.c_int32,
        ]
        lib.oracle_rotate_row_f64.restype = None
        lib.oracle_apply.argtypes = [
            c.c_int32, c.c_void_p, c.c_void_p, c.c_void_p,
            c.c_int64, c.c_int32, c.c_int64, c.c_int32, c.c_int32,
            c.c_int32, c.c_int32, c.c_int32,
            c.c_void_p, c.c_void_p, c.c_void_p, c.c_int64,
        ]
        lib.oracle_apply.restype = c.c_int
        self.lib = lib
        self.path = path

    # --- scalar conversions -------------------------------------------------
    def bf16_to_f64(self, bits: int) -> float:
        return self.lib.oracle_bf16_to_f64(bits)

    def f16_to_f64(self, bits: int) -> float:
        return self.lib.oracle_f16_to_f64(bits)

    def f64_to_bf16(self, y: float) -> int:
        return self.lib.oracle_f64_to_bf16(y)

    def f64_to_f16(self, y: float) -> int:
        return self.lib.oracle_f64_to_f16(y)

    def f64_to_f32(self, y: float) -> float:
        return self.lib.oracle_f64_to_f32(y)

    def inv_freq(self, theta: float, rotary_dim: int, i: int) -> float:
        return self.lib.oracle_inv_freq(theta, rotary_dim, i)

    def angle(self, m: int, interpolate_factor: float, inv_freq: float) -> float:
        return self.lib.oracle_angle(m, interpolate_factor, inv_freq)

    # --- tables ---------------------------------------------------------------
    def tables(self, theta: float, rotary_dim: int, max_pos: int,
               interpolate_factor: float = 1.0, precision: str = "f64"):
        """cos, sin tables [max_pos, rotary_dim // 2] in fp64 or fp32."""
        h = rotary_dim // 2
        dt = np.float64 if precision == "f64" else np.float32
        cos = np.empty((max_pos, h), dtype=dt)
        sin = np.empty((max_pos, h), dtype=dt)
        fn = self.lib.oracle_tables_f64 if precision == "f64" else self.lib.oracle_tables_f32
        rc = fn(theta, rotary_dim, max_pos, interpolate_factor, _ptr(cos), _ptr(sin))
        if rc != OK:
            raise ValueError("oracle tables: bad arguments (code %d)" % rc)
        return cos, sin

    def freq_ex(self, mode: int, theta: float, max_freq: float, rotary_dim: int, i: int) -> float:
        return self.lib.oracle_freq_ex(mode, theta, max_freq, rotary_dim, i)

    def position(self, m: int, pos_offset: float, pos_divisor: float) -> float:
        return self.lib.oracle_position(m, pos_offset, pos_divisor)

    def xpos_scale(self, rotary_dim: int, i: int, p: float, sign: int, base: float, gamma: float,
                   center: float) -> float:
        return self.lib.oracle_xpos_scale(rotary_dim, i, p, sign, base, gamma, center)

    def tables_ex(self, mode: int, rotary_dim: int, rows: int, theta: float = 10000.0,
                  max_freq: float = 10.0, pos_offset: float = 0.0, pos_divisor: float = 1.0,
                  xpos_sign: int = 0, xpos_base: float = 512.0, xpos_gamma: float = 0.4,
                  xpos_center: float = 0.0, precision: str = "f64"):
        """cos, sin tables [rows, rotary_dim // 2] of a frequency mode, row m at
        position pos_offset + m / pos_divisor, optionally XPOS-scaled."""
        h = rotary_dim // 2
        dt = np.float64 if precision == "f64" else np.float32
        cos = np.empty((rows, h), dtype=dt)
        sin = np.empty((rows, h), dtype=dt)
        fn = self.lib.oracle_tables_ex_f64 if precision == "f64" else self.lib.oracle_tables_ex_f32
        rc = fn(mode, theta, max_freq, rotary_dim, rows, pos_offset, pos_divisor, xpos_sign,
                xpos_base, xpos_gamma, xpos_center, _ptr(cos), _ptr(sin))
        if rc != OK:
            raise ValueError("oracle tables_ex: bad arguments (code %d)" % rc)
        return cos, sin

    # --- rotation -------------------------------------------------------------
    def rotate_row(self, x: np.ndarray, rotary_dim: int, layout: int,
                   c_row: np.ndarray, s_row: np.ndarray, backward: bool = False) -> np.ndarray:
        x = np.ascontiguousarray(x, dtype=np.float64)
        c_row = np.ascontiguousarray(c_row, dtype=np.float64)
        s_row = np.ascontiguousarray(s_row, dtype=np.float64)
        y = np.empty_like(x)
        self.lib.oracle_rotate_row_f64(_ptr(x), _ptr(y), x.shape[-1], rotary_dim, layout,
                                       _ptr(c_row), _ptr(s_row), int(backward))
        return y

    def apply(self, x_bits: np.ndarray, dtype: int, B: int, H: int, S: int, D: int,
              rotary_dim: int, layout: int, seq_before_head: bool, backward: bool,
              pos_idx: np.ndarray | None, cos_tab: np.ndarray, sin_tab: np.ndarray,
              want_f64: bool = True, want_bits: bool = True):
        """Rotate one tensor.  Returns (status, y_bits or None, y_f64 or None).

        ``x_bits`` holds the element bits (float32 for F32, uint16 for BF16 and
        F16, float64 for F64).  ``cos_tab``/``sin_tab`` are widened to fp64
        (exactly) before the call.
        """
        x_bits = np.ascontiguousarray(x_bits, dtype=_STORAGE[dtype])
        n = B * H * S * D
        assert x_bits.size == n, (x_bits.size, n)
        cos64 = np.ascontiguousarray(cos_tab, dtype=np.float64)
        sin64 = np.ascontiguousarray(sin_tab, dtype=np.float64)
        y_bits = np.empty_like(x_bits) if want_bits else None
        y_f64 = np.empty(x_bits.shape, dtype=np.float64) if want_f64 else None
        pos = None if pos_idx is None else np.ascontiguousarray(pos_idx, dtype=np.int32)
        rc = self.lib.oracle_apply(dtype, _ptr(x_bits), _ptr(y_bits), _ptr(y_f64),
                                   B, H, S, D, rotary_dim, layout, int(seq_before_head),
                                   int(backward), _ptr(pos), _ptr(cos64), _ptr(sin64),
                                   cos64.shape[0])
        return rc, y_bits, y_f64


_default: Oracle | None = None


def load() -> Oracle:
    """The oracle built from ``rope_oracle.c`` in this folder (built on demand)."""
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def load_mutant(replacements: list[tuple[str, str]], workdir: str | None = None) -> Oracle:
    """Compile a copy of the oracle source with textual replacements applied.

    Used by the tests to plant a mistake in the oracle, on the CPU, and check
    that at least one pin catches it.  Each ``old`` string must occur in the
    source.
    """
    with open(SOURCE) as f:
        text = f.read()
    for old, new in replacements:
        if old not in text:
            raise ValueError("mutation target not found: %r" % old)
        text = text.replace(old, new)
    workdir = workdir or tempfile.mkdtemp(prefix="rope_oracle_mutant_")
    src = os.path.join(workdir, "mutant.c")
    with open(src, "w") as f:
        f.write(text)
    return Oracle(compile_library(src, os.path.join(workdir, "libmutant.so")))
