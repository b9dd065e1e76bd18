"""The plain CPU oracle for the low-precision MoE expert path (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never does, and this
package never touches it: the two share no code.

The arithmetic lives in ``fme_oracle.c`` (scalar C, fp32 steps as IEEE binary32
operations, fp64 GEMM on exactly dequantized operands).  This module only
compiles that file with gcc and marshals numpy arrays into it.

Sources for what is computed (full citations in the C file's header):
  * "Composer 2 Technical Report", section 6.1: NVFP4 variant (E2M1 codes,
    E4M3 scale per 16 along K, FP32 per-token scale, IEEE division) for the MoE
    forward; standard MXFP8 (E4M3 codes, E8M0 scale per 32) for the backward.
  * "Scaling and Optimizing Frontier Model Training", "MXFP8 expert kernels":
    block-scaled grouped GEMMs over expert-grouped tokens.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "fme_oracle.c")
LIBRARY = os.path.join(_HERE, "libfme_oracle.so")
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

_lib = None
_lock = threading.Lock()


def build(source: str = SOURCE, output: str = LIBRARY) -> str:
    """Compile the oracle with gcc (no fused multiply-add, no fast math)."""
    cmd = ["gcc", *CFLAGS, "-o", output, source, "-lm"]
    scratch = os.path.join(_HERE, "_build")  # gcc's intermediates stay in the tree (git-ignored)
    os.makedirs(scratch, exist_ok=True)
    subprocess.run(cmd, check=True, env=dict(os.environ, TMPDIR=scratch))
    return output


def _stale() -> bool:
    return (not os.path.exists(LIBRARY)) or os.path.getmtime(LIBRARY) < os.path.getmtime(SOURCE)


def load(path: str | None = None):
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if _stale():
                build()
            _lib = _declare(ctypes.CDLL(LIBRARY))
    return _lib


def _declare(lib):
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    I32 = ctypes.c_int32
    U8 = ctypes.c_uint8
    D = ctypes.c_double
    lib.fme_orc_e2m1_value.argtypes = [U8]
    lib.fme_orc_e2m1_value.restype = D
    lib.fme_orc_e4m3_value.argtypes = [U8]
    lib.fme_orc_e4m3_value.restype = D
    lib.fme_orc_e8m0_value.argtypes = [U8]
    lib.fme_orc_e8m0_value.restype = D
    lib.fme_orc_e2m1_encode.argtypes = [D]
    lib.fme_orc_e2m1_encode.restype = U8
    lib.fme_orc_e4m3_encode.argtypes = [D]
    lib.fme_orc_e4m3_encode.restype = U8
    lib.fme_orc_e2m1_encode_array.argtypes = [P, I64, P]
    lib.fme_orc_e4m3_encode_array.argtypes = [P, I64, P]
    lib.fme_orc_quant_nvfp4.argtypes = [P, I64, I64, P, P, P]
    lib.fme_orc_quant_nvfp4_pertensor.argtypes = [P, I64, I64, P, P, P]
    lib.fme_orc_dequant_nvfp4.argtypes = [P, P, P, I64, I64, P]
    lib.fme_orc_quant_mxfp8_rows.argtypes = [P, I64, I64, P, P]
    lib.fme_orc_quant_mxfp8_cols.argtypes = [P, I64, I64, P, I32, I64, P, P, P]
    lib.fme_orc_quant_mxfp8_rows_ceil.argtypes = [P, I64, I64, P, P]
    lib.fme_orc_quant_mxfp8_cols_ceil.argtypes = [P, I64, I64, P, I32, I64, P, P, P]
    lib.fme_orc_dequant_mxfp8.argtypes = [P, P, I64, I64, P]
    lib.fme_orc_gemm_abt.argtypes = [P, P, I64, I64, I64, P]
    lib.fme_orc_swiglu.argtypes = [P, I64, I64, P]
    lib.fme_orc_swiglu_f64.argtypes = [P, I64, I64, P]
    lib.fme_orc_route.argtypes = [P, I64, I32, P, P, P]
    lib.fme_orc_swiglu_bwd.argtypes = [P, P, I64, I64, P]
    lib.fme_orc_combine.argtypes = [P, P, P, I64, I32, I64, P]
    for name in ("fme_orc_e2m1_encode_array", "fme_orc_e4m3_encode_array", "fme_orc_quant_nvfp4",
                 "fme_orc_dequant_nvfp4", "fme_orc_quant_mxfp8_rows", "fme_orc_quant_mxfp8_cols",
                 "fme_orc_dequant_mxfp8", "fme_orc_gemm_abt", "fme_orc_swiglu", "fme_orc_swiglu_f64", "fme_orc_route", "fme_orc_swiglu_bwd",
                 "fme_orc_quant_nvfp4_pertensor", "fme_orc_quant_mxfp8_rows_ceil", "fme_orc_quant_mxfp8_cols_ceil",
                 "fme_orc_combine"):
        getattr(lib, name).restype = None
    return lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _bits(x) -> np.ndarray:
    """bf16 input as its uint16 bit patterns, C-contiguous."""
    x = np.asarray(x)
    if x.dtype != np.uint16:
        raise TypeError("oracle inputs are bf16 bit patterns (uint16)")
    return np.ascontiguousarray(x)


class Oracle:
    """numpy front end of the C oracle.  ``lib`` lets a test load a rebuilt copy."""

    def __init__(self, lib=None):
        self.lib = lib if lib is not None else load()

    # code tables --------------------------------------------------------
    def e2m1_value(self, codes) -> np.ndarray:
        return np.array([self.lib.fme_orc_e2m1_value(int(c)) for c in np.ravel(codes)]).reshape(np.shape(codes))

    def e4m3_value(self, codes) -> np.ndarray:
        return np.array([self.lib.fme_orc_e4m3_value(int(c)) for c in np.ravel(codes)]).reshape(np.shape(codes))

    def e8m0_value(self, codes) -> np.ndarray:
        return np.array([self.lib.fme_orc_e8m0_value(int(c)) for c in np.ravel(codes)]).reshape(np.shape(codes))

    def e2m1_encode(self, v) -> np.ndarray:
        v = np.ascontiguousarray(v, dtype=np.float64)
        out = np.empty(v.shape, np.uint8)
        self.lib.fme_orc_e2m1_encode_array(_p(v), v.size, _p(out))
        return out

    def e4m3_encode(self, v) -> np.ndarray:
        v = np.ascontiguousarray(v, dtype=np.float64)
        out = np.empty(v.shape, np.uint8)
        self.lib.fme_orc_e4m3_encode_array(_p(v), v.size, _p(out))
        return out

    # quantizers ---------------------------------------------------------
    def quant_nvfp4(self, x_bits):
        """-> codes [rows, k/2] uint8, sf [rows, k/16] uint8 (E4M3), scale [rows] float32."""
        x = _bits(x_bits)
        rows, k = x.shape
        if k % 16:
            raise ValueError("k must be a multiple of 16")
        codes = np.zeros((rows, k // 2), np.uint8)
        sf = np.zeros((rows, k // 16), np.uint8)
        scale = np.zeros(rows, np.float32)
        self.lib.fme_orc_quant_nvfp4(_p(x), rows, k, _p(codes), _p(sf), _p(scale))
        return codes, sf, scale

    def quant_nvfp4_pertensor(self, x_bits):
        """Standard NVFP4 (one scale for the tensor) -> codes, sf, scale [rows] (all S)."""
        x = _bits(x_bits)
        rows, k = x.shape
        if k % 16:
            raise ValueError("k must be a multiple of 16")
        codes = np.zeros((rows, k // 2), np.uint8)
        sf = np.zeros((rows, k // 16), np.uint8)
        scale = np.zeros(rows, np.float32)
        self.lib.fme_orc_quant_nvfp4_pertensor(_p(x), rows, k, _p(codes), _p(sf), _p(scale))
        return codes, sf, scale

    def dequant_nvfp4(self, codes, sf, scale) -> np.ndarray:
        codes = np.ascontiguousarray(codes, np.uint8)
        sf = np.ascontiguousarray(sf, np.uint8)
        scale = np.ascontiguousarray(scale, np.float32)
        rows, half = codes.shape
        out = np.empty((rows, 2 * half), np.float64)
        self.lib.fme_orc_dequant_nvfp4(_p(codes), _p(sf), _p(scale), rows, 2 * half, _p(out))
        return out

    def quant_mxfp8_rows(self, x_bits, ceil_scale: bool = False):
        """-> codes [rows, cols] uint8 (E4M3), sf [rows, cols/32] uint8 (E8M0).
        ``ceil_scale``: the round-up scale rule X = 2^ceil(log2(amax / 448))."""
        x = _bits(x_bits)
        rows, cols = x.shape
        if cols % 32:
            raise ValueError("cols must be a multiple of 32")
        codes = np.zeros((rows, cols), np.uint8)
        sf = np.zeros((rows, cols // 32), np.uint8)
        fn = self.lib.fme_orc_quant_mxfp8_rows_ceil if ceil_scale else self.lib.fme_orc_quant_mxfp8_rows
        fn(_p(x), rows, cols, _p(codes), _p(sf))
        return codes, sf

    def quant_mxfp8_cols(self, x_bits, offsets, ld: int | None = None, ceil_scale: bool = False):
        """Column-wise MXFP8 over row groups.

        -> codes_t [cols, ld] uint8, sf_t [cols, ld/32] uint8, poff [G+1] int32.
        ``ld`` defaults to the padded total ``poff[G]``.
        """
        x = _bits(x_bits)
        rows, cols = x.shape
        offsets = np.ascontiguousarray(offsets, np.int32)
        g = len(offsets) - 1
        if offsets[0] != 0 or offsets[-1] != rows or np.any(np.diff(offsets) < 0):
            raise ValueError("offsets must rise from 0 to rows")
        padded = int(sum(((int(n) + 127) // 128) * 128 for n in np.diff(offsets)))
        if ld is None:
            ld = padded
        if ld < padded or ld % 128:
            raise ValueError("ld must be a multiple of 128 no smaller than the padded total")
        codes = np.zeros((cols, ld), np.uint8)
        sf = np.zeros((cols, ld // 32), np.uint8)
        poff = np.zeros(g + 1, np.int32)
        fn = self.lib.fme_orc_quant_mxfp8_cols_ceil if ceil_scale else self.lib.fme_orc_quant_mxfp8_cols
        fn(_p(x), rows, cols, _p(offsets), g, ld, _p(codes), _p(sf), _p(poff))
        return codes, sf, poff

    def dequant_mxfp8(self, codes, sf) -> np.ndarray:
        codes = np.ascontiguousarray(codes, np.uint8)
        sf = np.ascontiguousarray(sf, np.uint8)
        rows, cols = codes.shape
        out = np.empty((rows, cols), np.float64)
        self.lib.fme_orc_dequant_mxfp8(_p(codes), _p(sf), rows, cols, _p(out))
        return out

    # SwiGLU --------------------------------------------------------------
    def swiglu(self, y_gu_bits) -> np.ndarray:
        """h = silu(g) * u in fp64 for bf16 rows [g | u] (bit patterns)."""
        y = _bits(y_gu_bits)
        rows, two_inter = y.shape
        inter = two_inter // 2
        h = np.empty((rows, inter), np.float64)
        self.lib.fme_orc_swiglu(_p(y), rows, inter, _p(h))
        return h

    def swiglu_f64(self, y_gu) -> np.ndarray:
        """h = silu(g) * u in fp64 for fp64 rows [g | u] (e.g. the fp64 gate/up GEMM)."""
        y = np.ascontiguousarray(y_gu, np.float64)
        rows, two_inter = y.shape
        inter = two_inter // 2
        h = np.empty((rows, inter), np.float64)
        self.lib.fme_orc_swiglu_f64(_p(y), rows, inter, _p(h))
        return h

    def swiglu_bwd(self, y_gu_bits, dh_bits) -> np.ndarray:
        """d(gate/up) = [dg | du] in fp64 of h = silu(g) * u for upstream dh (bf16 bits)."""
        y = _bits(y_gu_bits)
        dh = _bits(dh_bits)
        rows, two_inter = y.shape
        inter = two_inter // 2
        if dh.shape != (rows, inter):
            raise ValueError("dh must be [rows x inter]")
        out = np.empty((rows, two_inter), np.float64)
        self.lib.fme_orc_swiglu_bwd(_p(y), _p(dh), rows, inter, _p(out))
        return out

    # routing -------------------------------------------------------------
    def route(self, ids, num_experts: int):
        """Stable grouping of assignments a (row-major over [tokens, top_k]) by
        expert -> offsets [E+1], row_of (shape of ids), src_row [ids.size], int32."""
        ids = np.ascontiguousarray(ids, np.int32)
        n = ids.size
        offsets = np.zeros(num_experts + 1, np.int32)
        row_of = np.zeros(ids.shape, np.int32)
        src_row = np.zeros(n, np.int32)
        self.lib.fme_orc_route(_p(ids), n, num_experts, _p(offsets), _p(row_of), _p(src_row))
        valid = int(offsets[-1])
        return offsets, row_of, src_row[:valid] if valid < n else src_row

    def combine(self, y_bits, row_of, weights):
        """out [tokens, n] bf16 bits = fp32 in-order weighted sum of the rows of
        y (bf16 bits) picked by row_of [tokens, top_k], rounded once to bf16."""
        y = _bits(y_bits)
        row_of = np.ascontiguousarray(row_of, np.int32)
        w = np.ascontiguousarray(weights, np.float32)
        tokens, top_k = row_of.shape
        n = y.shape[1]
        if np.any(row_of >= y.shape[0]):
            raise ValueError("row_of points past y")
        out = np.zeros((tokens, n), np.uint16)
        self.lib.fme_orc_combine(_p(y), _p(row_of), _p(w), tokens, top_k, n, _p(out))
        return out

    # GEMM ----------------------------------------------------------------
    def gemm_abt(self, a, b) -> np.ndarray:
        """y = a @ b.T in fp64, plain loops."""
        a = np.ascontiguousarray(a, np.float64)
        b = np.ascontiguousarray(b, np.float64)
        m, k = a.shape
        n, k2 = b.shape
        assert k == k2
        y = np.empty((m, n), np.float64)
        self.lib.fme_orc_gemm_abt(_p(a), _p(b), m, n, k, _p(y))
        return y
