"""The C-ABI library loads, exports every declared entry point, and rejects bad
arguments on the host before touching a GPU (no compute calls here)."""
import ctypes
import re
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]
HEADER = ROOT / "include" / "bitdelta.h"


@pytest.fixture(scope="module")
def bd():
    from bit_delta_compressed_gb300 import build
    build.build()
    import bit_delta_compressed_gb300 as bd
    return bd


def declared_functions():
    text = re.sub(r"/\*.*?\*/", "", HEADER.read_text(), flags=re.S)
    return sorted(set(re.findall(r"\b(bitdelta_\w+)\s*\(", text)))


def test_header_declares_entry_points():
    names = declared_functions()
    for must in ("bitdelta_compress", "bitdelta_linear", "bitdelta_compress_workspace",
                 "bitdelta_linear_workspace", "bitdelta_device_status"):
        assert must in names


def test_every_declared_symbol_is_exported(bd):
    lib = ctypes.CDLL(str(bd.LIB_PATH))
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in bd.SIGNATURES, "binding lacks " + name


def test_version_and_strings(bd):
    assert bd.bitdelta_abi_version() == 1
    for code in range(10):
        assert bd.status_string(code)
    assert bd.status_string(0) == "ok"


def test_workspace_sizes(bd):
    assert bd.bitdelta_compress_workspace(4096, 4096) > 0
    assert bd.bitdelta_compress_workspace(4096, 4095) == 0
    assert bd.bitdelta_compress_workspace(0, 4096) == 0
    assert bd.bitdelta_linear_workspace(64, 4096, 4096, 14) > 0
    assert bd.bitdelta_linear_workspace(64, 4096, 4100, 14) == 0
    assert bd.bitdelta_linear_workspace(64, 4096, 4096, 65) == 0
    assert bd.bitdelta_linear_workspace(0, 4096, 4096, 1) > 0


FAKE = 0x10000          # 16-byte aligned, never dereferenced: validation fails first
MISALIGNED = 0x10008


def test_compress_argument_errors(bd):
    c = bd.bitdelta_compress
    assert c(None, FAKE, bd.BD_BF16, 64, 64, FAKE, FAKE, FAKE, 1 << 20, None) == bd.BD_ERR_NULL
    assert c(FAKE, FAKE, 7, 64, 64, FAKE, FAKE, FAKE, 1 << 20, None) == bd.BD_ERR_DTYPE
    assert c(FAKE, FAKE, bd.BD_BF16, 64, 48, FAKE, FAKE, FAKE, 1 << 20, None) == bd.BD_ERR_SHAPE
    assert c(FAKE, FAKE, bd.BD_BF16, 0, 64, FAKE, FAKE, FAKE, 1 << 20, None) == bd.BD_ERR_SHAPE
    assert c(MISALIGNED, FAKE, bd.BD_BF16, 64, 64, FAKE, FAKE, FAKE, 1 << 20, None) == bd.BD_ERR_ALIGN
    assert c(FAKE, FAKE, bd.BD_BF16, 64, 64, FAKE, FAKE, None, 1 << 20, None) == bd.BD_ERR_WORKSPACE
    assert c(FAKE, FAKE, bd.BD_BF16, 64, 64, FAKE, FAKE, FAKE, 8, None) == bd.BD_ERR_WORKSPACE
    r = bd.bitdelta_compress_rows
    assert r(FAKE, None, bd.BD_F32, 4, 64, FAKE, FAKE, None) == bd.BD_ERR_NULL
    assert r(FAKE, FAKE, bd.BD_F32, 4, 65, FAKE, FAKE, None) == bd.BD_ERR_SHAPE


def _lin(bd, x=FAKE, ids=FAKE, M=4, N=64, K=64, w=FAKE, al=FAKE, bits="ok", V=1, y=FAKE,
         ydt=None, ws=FAKE, wsb=1 << 24, path=0):
    ydt = bd.BD_F32 if ydt is None else ydt
    if bits == "ok":
        bits = (ctypes.c_void_p * max(1, V))(*([FAKE] * max(1, V)))
    elif bits == "null_entry":
        bits = (ctypes.c_void_p * 1)(None)
    elif bits == "misaligned":
        bits = (ctypes.c_void_p * 1)(MISALIGNED)
    ptr = ctypes.cast(bits, ctypes.c_void_p) if bits is not None else None
    return bd.bitdelta_linear_ex(x, ids, M, N, K, w, al, ptr, V, y, ydt, ws, wsb, None, path)


def test_linear_argument_errors(bd):
    assert _lin(bd, x=None) == bd.BD_ERR_NULL
    assert _lin(bd, bits=None) == bd.BD_ERR_NULL
    assert _lin(bd, bits="null_entry") == bd.BD_ERR_NULL
    assert _lin(bd, al=None) == bd.BD_ERR_NULL
    assert _lin(bd, K=48) == bd.BD_ERR_SHAPE
    assert _lin(bd, N=0) == bd.BD_ERR_SHAPE
    assert _lin(bd, M=-1) == bd.BD_ERR_SHAPE
    assert _lin(bd, V=65) == bd.BD_ERR_SHAPE
    assert _lin(bd, ydt=5) == bd.BD_ERR_DTYPE
    assert _lin(bd, x=MISALIGNED) == bd.BD_ERR_ALIGN
    assert _lin(bd, bits="misaligned") == bd.BD_ERR_ALIGN
    assert _lin(bd, ws=None) == bd.BD_ERR_WORKSPACE
    assert _lin(bd, wsb=16) == bd.BD_ERR_WORKSPACE
    assert _lin(bd, M=0, x=None, y=None) == bd.BD_OK          # empty batch: no-op
    assert _lin(bd, path=9) == bd.BD_ERR_UNSUPPORTED


def test_status_needs_workspace(bd):
    assert bd.bitdelta_device_status(None, None) == bd.BD_ERR_NULL
    assert bd.bitdelta_check_bounded_wait(None, 16, 0, None) == bd.BD_ERR_NULL
    assert bd.bitdelta_check_bounded_wait(MISALIGNED, 16, 0, None) == bd.BD_ERR_ALIGN
    assert bd.bitdelta_check_bounded_wait(FAKE, 0, 0, None) == bd.BD_ERR_SHAPE
    assert bd.bitdelta_check_bounded_wait(FAKE, (1 << 24) + 1, 0, None) == bd.BD_ERR_SHAPE
