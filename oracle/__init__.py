"""TEST INFRASTRUCTURE ONLY -- the CPU oracle for the BitDelta hot path.

A thin ctypes wrapper around ``bitdelta_oracle.c``: a plain fp64 statement of
the formulas on the web page "BitDelta: serving 14 Zen models from one GPU
cluster" (Hanzo blog, 2026-02-28):

* section "The mathematical foundation": delta = W_ft - W_base,
  alpha = (1/n)*||delta||_1 (one scale per matrix), one sign bit per entry;
* section "Serving architecture": W_eff = W_base + alpha_v * sign(delta_v),
  then y = x * W_eff^T (the conceptual ``fused_bitdelta_linear`` listing);
* section "Infrastructure details": sign bits packed 8 per byte, alpha in f32.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It never touches a GPU and shares no
code with the CUDA library in ``bit_delta_compressed_gb300``.

Arrays: bf16 matrices are passed as ``numpy.uint16`` arrays holding the bf16
bit patterns; f32 as ``numpy.float32``; packed sign bits as ``numpy.uint32``
``[N, K/32]`` (bit j of word w in row n is column 32*w + j; 1 means the delta is
>= 0).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
SOURCE = _HERE / "bitdelta_oracle.c"
_BUILD_DIR = _HERE / "_build"
_DEFAULT_LIB = _BUILD_DIR / "liboracle_bitdelta.so"

# -ffp-contract=off: no fused multiply-add, so x86 and Arm builds round alike.
CFLAGS = ["-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off", "-pthread"]


def build(src: Path = SOURCE, out: Path = _DEFAULT_LIB, force: bool = False) -> Path:
    """Compile the oracle C source with gcc into a shared library."""
    out = Path(out)
    if not force and out.exists() and out.stat().st_mtime >= Path(src).stat().st_mtime:
        return out
    out.parent.mkdir(parents=True, exist_ok=True)
    tmp = out.with_suffix(".so.tmp%d" % os.getpid())
    subprocess.run(["gcc", *CFLAGS, "-o", str(tmp), str(src), "-lm"], check=True)
    os.replace(tmp, out)
    return out


def host_threads() -> int:
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


_p = ctypes.c_void_p
_i64 = ctypes.c_int64


class Oracle:
    """Handle on one compiled copy of the oracle library."""

    def __init__(self, lib_path: Path | str | None = None):
        path = Path(lib_path) if lib_path is not None else build()
        self.lib = ctypes.CDLL(str(path))
        L = self.lib
        for name in ("bdo_compress_f32", "bdo_compress_bf16"):
            fn = getattr(L, name)
            fn.argtypes = [_p, _p, _i64, _i64, _p, _p, _p]
            fn.restype = ctypes.c_int
        L.bdo_compress_rows.argtypes = [_p, _p, ctypes.c_int, _i64, _i64, _p, _p, _p]
        L.bdo_compress_rows.restype = ctypes.c_int
        L.bdo_reconstruct.argtypes = [_p, _p, ctypes.c_int, _p, _i64, _i64, _p]
        L.bdo_reconstruct.restype = ctypes.c_int
        L.bdo_linear.argtypes = [_p, _p, _i64, _i64, _i64, _p, _p, ctypes.c_int,
                                 _p, ctypes.c_int32, _p, _i64, _p, ctypes.c_int]
        L.bdo_linear.restype = ctypes.c_int

    # -- compression -----------------------------------------------------
    def compress(self, w_ft: np.ndarray, w_base: np.ndarray):
        """Return (alpha_f64, alpha_f32, bits[N, K/32] uint32).

        ``w_ft``/``w_base``: float32 arrays, or uint16 arrays of bf16 bits."""
        w_ft = np.ascontiguousarray(w_ft)
        w_base = np.ascontiguousarray(w_base)
        if w_ft.shape != w_base.shape or w_ft.ndim != 2 or w_ft.dtype != w_base.dtype:
            raise ValueError("w_ft and w_base must be 2-D arrays of one shape and dtype")
        N, K = w_ft.shape
        if K % 32:
            raise ValueError("K must be a multiple of 32")
        bits = np.zeros((N, K // 32), dtype=np.uint32)
        a64 = ctypes.c_double()
        a32 = ctypes.c_float()
        fn = {np.dtype(np.float32): self.lib.bdo_compress_f32,
              np.dtype(np.uint16): self.lib.bdo_compress_bf16}[w_ft.dtype]
        rc = fn(w_ft.ctypes.data, w_base.ctypes.data, N, K,
                ctypes.addressof(a64), ctypes.addressof(a32), bits.ctypes.data)
        if rc != 0:
            raise ValueError("oracle compress failed: %d" % rc)
        return a64.value, np.float32(a32.value), bits

    def compress_rows(self, w_ft: np.ndarray, w_base: np.ndarray):
        """Per-output-row scale: (alpha_f64[N], alpha_f32[N], bits)."""
        w_ft = np.ascontiguousarray(w_ft)
        w_base = np.ascontiguousarray(w_base)
        N, K = w_ft.shape
        bits = np.zeros((N, K // 32), dtype=np.uint32)
        a64 = np.zeros(N, dtype=np.float64)
        a32 = np.zeros(N, dtype=np.float32)
        is_bf16 = int(w_ft.dtype == np.uint16)
        rc = self.lib.bdo_compress_rows(w_ft.ctypes.data, w_base.ctypes.data, is_bf16, N, K,
                                        a64.ctypes.data, a32.ctypes.data, bits.ctypes.data)
        if rc != 0:
            raise ValueError("oracle compress_rows failed: %d" % rc)
        return a64, a32, bits

    # -- multi-variant linear --------------------------------------------
    def reconstruct(self, w_base: np.ndarray, alpha, bits: np.ndarray, per_row: bool = False) -> np.ndarray:
        """bf16 bits [N, K] of the nearest bf16 (ties to even) of
        W_base + a * s, a = alpha (scalar) or alpha[n] with ``per_row``."""
        w_base = np.ascontiguousarray(w_base, dtype=np.uint16)
        bits = np.ascontiguousarray(bits, dtype=np.uint32)
        N, K = w_base.shape
        al = np.ascontiguousarray(np.atleast_1d(alpha), dtype=np.float32)
        if bits.shape != (N, K // 32) or al.shape[0] != (N if per_row else 1):
            raise ValueError("shape mismatch")
        out = np.empty((N, K), dtype=np.uint16)
        rc = self.lib.bdo_reconstruct(w_base.ctypes.data, al.ctypes.data, int(per_row), bits.ctypes.data, N, K,
                                      out.ctypes.data)
        if rc != 0:
            raise ValueError("oracle reconstruct failed: %d" % rc)
        return out

    def linear(self, x: np.ndarray, variant_ids: np.ndarray, w_base: np.ndarray,
               alphas: np.ndarray, bits: list, rows=None, nthreads: int | None = None,
               per_row_alpha: bool = False) -> np.ndarray:
        """y[t, i] = sum_k x[t,k] * W_eff_{v(t)}[rows[i], k] in fp64.

        ``x``: uint16 bf16 bits [M, K]; ``w_base``: uint16 bf16 bits [N, K];
        ``alphas``: float32 [V] (or [V, N] with ``per_row_alpha``);
        ``bits``: list of V uint32 arrays [N, K/32]; ``rows``: output rows
        (default all).  Returns float64 [M, len(rows)]."""
        x = np.ascontiguousarray(x, dtype=np.uint16)
        w_base = np.ascontiguousarray(w_base, dtype=np.uint16)
        vid = np.ascontiguousarray(variant_ids, dtype=np.int32)
        alphas = np.ascontiguousarray(alphas, dtype=np.float32)
        M, K = x.shape
        N, K2 = w_base.shape
        if K2 != K or vid.shape != (M,):
            raise ValueError("shape mismatch")
        bits = [np.ascontiguousarray(b, dtype=np.uint32) for b in bits]
        for b in bits:
            if b.shape != (N, K // 32):
                raise ValueError("bits must be [N, K/32]")
        V = len(bits)
        rows = np.arange(N, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        ptrs = (ctypes.c_void_p * max(V, 1))(*[b.ctypes.data for b in bits])
        y = np.zeros((M, rows.shape[0]), dtype=np.float64)
        nt = host_threads() if nthreads is None else int(nthreads)
        rc = self.lib.bdo_linear(x.ctypes.data, vid.ctypes.data, M, N, K, w_base.ctypes.data,
                                 alphas.ctypes.data, int(per_row_alpha), ctypes.addressof(ptrs),
                                 V, rows.ctypes.data, rows.shape[0], y.ctypes.data, nt)
        if rc == -3:
            raise ValueError("variant id outside [-1, V)")
        if rc != 0:
            raise ValueError("oracle linear failed: %d" % rc)
        return y


_default: Oracle | None = None


def get() -> Oracle:
    """The oracle built from this directory's source (compiled on first use)."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def packed_bytes(N: int, K: int) -> int:
    """Storage of one packed sign matrix: one bit per weight, 8 per byte."""
    return N * K // 8
