"""BitDelta on GB300: Python binding of the C-ABI library ``libbitdelta.so``.

The method (web page "BitDelta: serving 14 Zen models from one GPU cluster",
sections "The mathematical foundation" and "Serving architecture"):
compress a fine-tuned matrix to one f32 scale alpha = mean|W_ft - W_base| and
one sign bit per weight, and serve many variants from one resident base with a
fused linear y = x (W_base + alpha_v sign(delta_v))^T that never writes the
reconstructed weights to memory.

This module only marshals arguments: every step runs in the library's CUDA
kernels.  The first use loads the library and raises ImportError if it is
missing (build it with ``python -m bit_delta_compressed_gb300.build``); there
is no CPU fallback.

Two layers:
* ``lib`` and the functions named like the C entry points
  (``bitdelta_compress``, ``bitdelta_linear``, ...) take raw integers
  (device pointers, sizes, a stream handle) exactly as the C ABI does;
* ``compress``, ``compress_rows`` and ``linear`` take torch CUDA tensors,
  allocate outputs and workspace with torch, and call the C ABI on the
  current torch stream.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

_PKG = Path(__file__).resolve().parent
LIB_PATH = _PKG / "libbitdelta.so"

BD_OK, BD_ERR_NULL, BD_ERR_ALIGN, BD_ERR_SHAPE, BD_ERR_DTYPE, BD_ERR_VARIANT, \
    BD_ERR_WORKSPACE, BD_ERR_CUDA, BD_ERR_TIMEOUT, BD_ERR_UNSUPPORTED = range(10)
BD_F32, BD_BF16 = 0, 1
BD_PATH_AUTO, BD_PATH_SIMT, BD_PATH_DECODE_TC, BD_PATH_PREFILL_TC, BD_PATH_DECODE_FOLD, BD_PATH_DECODE_WEFF = range(6)
MAX_VARIANTS = 64
PATHS = {"auto": BD_PATH_AUTO, "simt": BD_PATH_SIMT, "decode_tc": BD_PATH_DECODE_TC,
         "prefill_tc": BD_PATH_PREFILL_TC, "decode_fold": BD_PATH_DECODE_FOLD,
         "decode_weff": BD_PATH_DECODE_WEFF}

# name -> (restype, argtypes), in the order of include/bitdelta.h
_P, _I64, _I32, _SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
_ST = ctypes.c_int
SIGNATURES = {
    "bitdelta_compress_workspace": (_SZ, [_I64, _I64]),
    "bitdelta_compress": (_ST, [_P, _P, _ST, _I64, _I64, _P, _P, _P, _SZ, _P]),
    "bitdelta_compress_rows": (_ST, [_P, _P, _ST, _I64, _I64, _P, _P, _P]),
    "bitdelta_compress_noalloc": (_ST, [_P, _P, _ST, _I64, _I64, _P, _P, _P]),
    "bitdelta_reconstruct": (_ST, [_P, _P, _I32, _P, _I64, _I64, _P, _P]),
    "bitdelta_linear_workspace": (_SZ, [_I64, _I64, _I64, _I32]),
    "bitdelta_linear": (_ST, [_P, _P, _I64, _I64, _I64, _P, _P, _P, _I32, _P, _ST, _P, _SZ, _P]),
    "bitdelta_linear_ex": (_ST, [_P, _P, _I64, _I64, _I64, _P, _P, _P, _I32, _P, _ST, _P, _SZ,
                                 _P, _ST]),
    "bitdelta_group": (_ST, [_P, _I64, _I32, _P, _SZ, _P]),
    "bitdelta_linear_grouped": (_ST, [_P, _I64, _I64, _I64, _P, _P, _P, _I32, _P, _ST, _P, _SZ,
                                      _P, _ST]),
    "bitdelta_linear_rows": (_ST, [_P, _P, _I64, _I64, _I64, _P, _P, _P, _I32, _P, _ST, _P, _SZ,
                                   _P, _ST]),
    "bitdelta_device_status": (_ST, [_P, _P]),
    "bitdelta_check_bounded_wait": (_ST, [_P, ctypes.c_uint32, ctypes.c_int, _P]),
    "bitdelta_launch_count": (ctypes.c_uint64, []),
    "bitdelta_status_string": (ctypes.c_char_p, [_ST]),
    "bitdelta_abi_version": (ctypes.c_int, []),
}


class BitDeltaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__("%s: %s (status %d)" % (where, status_string(code), code))


_LIB = None


def get_lib() -> ctypes.CDLL:
    """The loaded library; raises ImportError if it has not been built."""
    global _LIB
    if _LIB is None:
        if not LIB_PATH.exists():
            raise ImportError("libbitdelta.so is not built (%s); run "
                              "`python -m bit_delta_compressed_gb300.build`" % LIB_PATH)
        lib = ctypes.CDLL(str(LIB_PATH))
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
    return _LIB


def __getattr__(name):
    # `lib` and the raw C entry points resolve on first use, so the build
    # submodule can be imported before the library exists.
    if name == "lib":
        return get_lib()
    if name in SIGNATURES:
        return getattr(get_lib(), name)
    raise AttributeError(name)


def status_string(code: int) -> str:
    return get_lib().bitdelta_status_string(int(code)).decode()


def check(code: int, where: str) -> None:
    if code != BD_OK:
        raise BitDeltaError(code, where)


# -- torch layer ---------------------------------------------------------------

def _torch():
    import torch
    return torch


def _stream(stream=None) -> int:
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _dtype_code(t) -> int:
    torch = _torch()
    if t == torch.float32:
        return BD_F32
    if t == torch.bfloat16:
        return BD_BF16
    raise TypeError("unsupported dtype %s" % t)


def _need_cuda(*ts):
    for t in ts:
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("tensors must be contiguous CUDA tensors")


def compress_workspace(N: int, K: int, device=None):
    torch = _torch()
    n = int(get_lib().bitdelta_compress_workspace(N, K))
    if n == 0:
        raise BitDeltaError(BD_ERR_SHAPE, "bitdelta_compress_workspace")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def compress(w_ft, w_base, workspace=None, alpha_out=None, bits_out=None, stream=None):
    """(alpha [1] f32, bits int32 [N, K/32]) for one fine-tuned matrix."""
    torch = _torch()
    _need_cuda(w_ft, w_base)
    if w_ft.shape != w_base.shape or w_ft.dtype != w_base.dtype or w_ft.dim() != 2:
        raise ValueError("w_ft and w_base must be 2-D of one shape and dtype")
    N, K = w_ft.shape
    dev = w_ft.device
    ws = compress_workspace(N, K, dev) if workspace is None else workspace
    alpha = torch.empty(1, dtype=torch.float32, device=dev) if alpha_out is None else alpha_out
    bits = torch.empty((N, K // 32), dtype=torch.int32, device=dev) if bits_out is None else bits_out
    check(get_lib().bitdelta_compress(w_ft.data_ptr(), w_base.data_ptr(), _dtype_code(w_ft.dtype), N, K,
                                alpha.data_ptr(), bits.data_ptr(), ws.data_ptr(), ws.numel(),
                                _stream(stream)), "bitdelta_compress")
    return alpha, bits


def compress_rows(w_ft, w_base, stream=None):
    """(alpha [N] f32, bits int32 [N, K/32]) with one scale per output row."""
    torch = _torch()
    _need_cuda(w_ft, w_base)
    N, K = w_ft.shape
    alpha = torch.empty(N, dtype=torch.float32, device=w_ft.device)
    bits = torch.empty((N, K // 32), dtype=torch.int32, device=w_ft.device)
    check(get_lib().bitdelta_compress_rows(w_ft.data_ptr(), w_base.data_ptr(), _dtype_code(w_ft.dtype),
                                     N, K, alpha.data_ptr(), bits.data_ptr(), _stream(stream)),
          "bitdelta_compress_rows")
    return alpha, bits


def reconstruct(w_base, alpha, bits, out=None, stream=None):
    """bf16 W_eff [N, K] = nearest bf16 of W_base + alpha * s (``alpha``: a
    float32 tensor of 1 or N values; see ``bitdelta_reconstruct``)."""
    torch = _torch()
    _need_cuda(w_base, alpha, bits)
    N, K = w_base.shape
    if alpha.dtype != torch.float32 or alpha.numel() not in (1, N) or not alpha.is_contiguous():
        raise ValueError("alpha must be a contiguous float32 tensor of 1 or N values")
    per_row = 1 if (alpha.numel() == N and N != 1) else 0
    out = torch.empty((N, K), dtype=torch.bfloat16, device=w_base.device) if out is None else out
    check(get_lib().bitdelta_reconstruct(w_base.data_ptr(), alpha.data_ptr(), per_row, bits.data_ptr(), N, K,
                                         out.data_ptr(), _stream(stream)), "bitdelta_reconstruct")
    return out


def linear_workspace(M: int, N: int, K: int, V: int, device=None):
    torch = _torch()
    n = int(get_lib().bitdelta_linear_workspace(M, N, K, V))
    if n == 0:
        raise BitDeltaError(BD_ERR_SHAPE, "bitdelta_linear_workspace")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def bits_pointer_array(bits_list):
    """HOST array of the variants' device pointers, as the C ABI takes it."""
    arr = (ctypes.c_void_p * max(1, len(bits_list)))(*[b.data_ptr() for b in bits_list])
    return arr


def linear(x, variant_ids, w_base, alphas, bits_list, out_dtype=None, workspace=None,
           out=None, path: str = "auto", stream=None, bits_ptrs=None):
    """y [M, N] = per-token fused BitDelta linear (see ``bitdelta_linear``)."""
    torch = _torch()
    _need_cuda(x, variant_ids, w_base)
    M, K = x.shape
    N = w_base.shape[0]
    V = len(bits_list)
    if V > MAX_VARIANTS:
        raise ValueError("at most %d variants" % MAX_VARIANTS)
    out_dtype = out_dtype or torch.float32
    y = torch.empty((M, N), dtype=out_dtype, device=x.device) if out is None else out
    ws = linear_workspace(M, N, K, V, x.device) if workspace is None else workspace
    ptrs = bits_pointer_array(bits_list) if bits_ptrs is None else bits_ptrs
    al = alphas.data_ptr() if V > 0 else None
    check(get_lib().bitdelta_linear_ex(x.data_ptr(), variant_ids.data_ptr(), M, N, K, w_base.data_ptr(),
                                 al, ctypes.cast(ptrs, ctypes.c_void_p), V, y.data_ptr(),
                                 _dtype_code(out_dtype), ws.data_ptr(), ws.numel(),
                                 _stream(stream), PATHS[path]), "bitdelta_linear")
    return y


def linear_rows(x, variant_ids, w_base, alpha_rows, bits_list, out_dtype=None, workspace=None,
                out=None, path: str = "auto", stream=None, bits_ptrs=None):
    """y [M, N] with one scale per (variant, output row): ``alpha_rows`` is a
    float32 [V, N] device tensor (see ``bitdelta_linear_rows``)."""
    torch = _torch()
    _need_cuda(x, variant_ids, w_base)
    M, K = x.shape
    N = w_base.shape[0]
    V = len(bits_list)
    if V > MAX_VARIANTS:
        raise ValueError("at most %d variants" % MAX_VARIANTS)
    if V > 0 and (alpha_rows.dtype != torch.float32 or alpha_rows.numel() != V * N
                  or not alpha_rows.is_contiguous()):
        raise ValueError("alpha_rows must be a contiguous float32 [V, N] tensor")
    out_dtype = out_dtype or torch.float32
    y = torch.empty((M, N), dtype=out_dtype, device=x.device) if out is None else out
    ws = linear_workspace(M, N, K, V, x.device) if workspace is None else workspace
    ptrs = bits_pointer_array(bits_list) if bits_ptrs is None else bits_ptrs
    al = alpha_rows.data_ptr() if V > 0 else None
    check(get_lib().bitdelta_linear_rows(x.data_ptr(), variant_ids.data_ptr(), M, N, K, w_base.data_ptr(),
                                         al, ctypes.cast(ptrs, ctypes.c_void_p), V, y.data_ptr(),
                                         _dtype_code(out_dtype), ws.data_ptr(), ws.numel(),
                                         _stream(stream), PATHS[path]), "bitdelta_linear_rows")
    return y


def group(variant_ids, V: int, workspace, stream=None) -> None:
    """Group one batch's tokens by variant into ``workspace``."""
    _need_cuda(variant_ids)
    check(get_lib().bitdelta_group(variant_ids.data_ptr(), variant_ids.numel(), V,
                                   workspace.data_ptr(), workspace.numel(), _stream(stream)),
          "bitdelta_group")


def linear_grouped(x, w_base, alphas, bits_ptrs, V: int, y, workspace, path: str = "auto",
                   stream=None) -> None:
    """The fused linear on a batch grouped by ``group`` (outputs into ``y``).
    ``bits_ptrs`` is the host pointer array from ``bits_pointer_array``."""
    M, K = x.shape
    N = w_base.shape[0]
    al = alphas.data_ptr() if V > 0 else None
    check(get_lib().bitdelta_linear_grouped(x.data_ptr(), M, N, K, w_base.data_ptr(), al,
                                            ctypes.cast(bits_ptrs, ctypes.c_void_p), V,
                                            y.data_ptr(), _dtype_code(y.dtype),
                                            workspace.data_ptr(), workspace.numel(),
                                            _stream(stream), PATHS[path]),
          "bitdelta_linear_grouped")


def device_status(workspace, stream=None) -> int:
    """Synchronise, read and clear the status word of a workspace."""
    return int(get_lib().bitdelta_device_status(workspace.data_ptr(), _stream(stream)))
