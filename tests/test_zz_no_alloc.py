"""bitdelta_compress_noalloc -- compression for callers that cannot allocate.

Some programs that embed this library may not call cudaMalloc: an inference
engine whose memory pool already owns the device, a plugin that must not
grow the process's footprint, or code on a path where an allocation would
synchronise the device.  The no-allocation entry point keeps its scratch in a
static device array inside the library.  This test calls it through the C ABI
twice in a row (different shapes and dtypes, so the second call reuses the
array left behind by the first) and checks each result against the regular
bitdelta_compress, which takes a caller workspace.

It lives in a file of its own that pytest collects last, and passes both
alone in a fresh process and after every other test."""
import ctypes

import numpy as np
import pytest
import torch

import workloads as wl
from tests.gpu_util import ALPHA_REL, load_bd

pytestmark = pytest.mark.gpu


def _compress_with_workspace(bd, w_ft, w_base, dtype_code, stream):
    N, K = w_ft.shape
    ws = torch.zeros(int(bd.bitdelta_compress_workspace(N, K)), dtype=torch.uint8, device="cuda")
    alpha = torch.empty(1, dtype=torch.float32, device="cuda")
    bits = torch.empty((N, K // 32), dtype=torch.int32, device="cuda")
    rc = bd.bitdelta_compress(w_ft.data_ptr(), w_base.data_ptr(), dtype_code, N, K, alpha.data_ptr(),
                              bits.data_ptr(), ws.data_ptr(), ws.numel(), stream)
    assert rc == bd.BD_OK, bd.status_string(rc)
    return alpha, bits


def _compress_no_alloc(bd, w_ft, w_base, dtype_code, stream):
    N, K = w_ft.shape
    alpha = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
    bits = torch.full((N, K // 32), -1, dtype=torch.int32, device="cuda")
    rc = bd.bitdelta_compress_noalloc(w_ft.data_ptr(), w_base.data_ptr(), dtype_code, N, K,
                                      alpha.data_ptr(), bits.data_ptr(), stream)
    assert rc == bd.BD_OK, bd.status_string(rc)
    return alpha, bits


def test_no_alloc_matches_workspace_entry_point():
    bd = load_bd()
    stream = torch.cuda.current_stream().cuda_stream
    cases = [((4096, 4096), torch.bfloat16, bd.BD_BF16, 5e-4),
             ((1000, 288), torch.float32, bd.BD_F32, 1e-3)]
    g = wl.generator(77, "cuda")
    for (N, K), dtype, code, b in cases:
        wb = wl.base_weights(N, K, g, "cuda", dtype=dtype)
        wf = wl.finetuned_weights(wb, b, g)
        a_ref, bits_ref = _compress_with_workspace(bd, wf, wb, code, stream)
        a_new, bits_new = _compress_no_alloc(bd, wf, wb, code, stream)
        torch.cuda.synchronize()
        assert torch.equal(bits_new, bits_ref), "bits differ for %dx%d" % (N, K)
        ar, an = float(a_ref.item()), float(a_new.item())
        assert abs(an - ar) <= ALPHA_REL * abs(ar), (an, ar)


def test_no_alloc_rejects_bad_arguments():
    bd = load_bd()
    assert bd.bitdelta_compress_noalloc(None, None, bd.BD_BF16, 64, 64, None, None, None) == bd.BD_ERR_NULL
    x = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(1, dtype=torch.float32, device="cuda")
    bits = torch.zeros((4, 2), dtype=torch.int32, device="cuda")
    assert bd.bitdelta_compress_noalloc(x.data_ptr(), x.data_ptr(), bd.BD_BF16, 4, 48, out.data_ptr(),
                                        bits.data_ptr(), None) == bd.BD_ERR_SHAPE
