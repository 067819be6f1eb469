"""GPU parity: bitdelta_compress against the CPU oracle.

Bits must match bit for bit; alpha within 1e-6 relative of the oracle's fp64
mean.  Inputs come from the seeded generators in ``workloads``."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests.gpu_util import assert_alpha_close, bf16_np, bits_np, f32_np, load_bd

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def bd():
    return load_bd()


@pytest.fixture(scope="module")
def o():
    return oracle.get()


def _host(t):
    return f32_np(t) if t.dtype == torch.float32 else bf16_np(t)


def _check(bd, o, w_ft, w_base, what):
    alpha, bits = bd.compress(w_ft, w_base)
    torch.cuda.synchronize()
    a64, _, rbits = o.compress(_host(w_ft), _host(w_base))
    got = bits_np(bits)
    assert np.array_equal(got, rbits), "%s: %d words differ" % (what, int((got != rbits).sum()))
    assert_alpha_close(float(alpha.item()), a64, what)
    return alpha, bits


def test_tiny_f32(bd, o):
    g = wl.generator(0, DEV)
    wb = wl.base_weights(256, 256, g, DEV, dtype=torch.float32)
    wf = wl.finetuned_weights(wb, 1e-3, g)
    alpha, bits = _check(bd, o, wf, wb, "tiny f32")
    assert bits.numel() == 2048


def test_single_bf16(bd, o):
    g = wl.generator(1, DEV)
    wb = wl.base_weights(4096, 4096, g, DEV)
    wf = wl.finetuned_weights(wb, 5e-4, g)
    _check(bd, o, wf, wb, "single bf16")


def test_single_f32_finetuned(bd, o):
    g = wl.generator(2, DEV)
    wb = wl.base_weights(4096, 4096, g, DEV, dtype=torch.float32)
    wf = wl.finetuned_weights(wb, 5e-4, g, out_dtype=torch.float32)
    _check(bd, o, wf, wb, "single f32")


@pytest.mark.parametrize("N,K", [(1, 32), (3, 96), (5, 160), (7, 4096), (129, 288), (1, 65536)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_ragged_shapes(bd, o, N, K, dtype):
    g = wl.generator(N * 7919 + K, DEV)
    wb = wl.base_weights(N, K, g, DEV, dtype=dtype)
    wf = wl.finetuned_weights(wb, 1e-3, g)
    _check(bd, o, wf, wb, "ragged %dx%d" % (N, K))


def test_zero_delta_and_signed_zero(bd, o):
    wb = torch.zeros((8, 64), dtype=torch.float32, device=DEV)
    wf = torch.zeros_like(wb)
    wf[0] = -0.0
    wb[1] = -0.0
    wf[2, 3] = -1.0
    alpha, bits = _check(bd, o, wf, wb, "zeros")
    b = bits_np(bits)
    assert b[0, 0] == 0xFFFFFFFF and b[1, 0] == 0xFFFFFFFF
    assert b[2, 0] == 0xFFFFFFFF ^ (1 << 3)


def test_deterministic(bd, o):
    g = wl.generator(3, DEV)
    wb = wl.base_weights(2048, 4096, g, DEV)
    wf = wl.finetuned_weights(wb, 1e-3, g)
    a1, b1 = bd.compress(wf, wb)
    a2, b2 = bd.compress(wf, wb)
    torch.cuda.synchronize()
    assert a1.view(torch.int32).item() == a2.view(torch.int32).item()
    assert torch.equal(b1, b2)


def test_rows_alpha(bd, o):
    g = wl.generator(4, DEV)
    wb = wl.base_weights(300, 1024, g, DEV)
    wf = wl.finetuned_weights(wb, 1e-3, g)
    alpha, bits = bd.compress_rows(wf, wb)
    torch.cuda.synchronize()
    a64, _, rbits = o.compress_rows(bf16_np(wf), bf16_np(wb))
    assert np.array_equal(bits_np(bits), rbits)
    got = f32_np(alpha).astype(np.float64)
    assert np.all(np.abs(got - a64) <= 1e-6 * np.abs(a64))


def test_prefill_matrix_fourteen_variants(bd, o):
    """Full size: 14 variants of one 28672 x 8192 bf16 matrix, bits compared
    in full for every variant, alpha for every variant."""
    g = wl.generator(5, DEV)
    wb = wl.base_weights(28672, 8192, g, DEV)
    wb_h = bf16_np(wb)
    for v in range(14):
        wf = wl.finetuned_weights(wb, 1e-3, g)
        alpha, bits = bd.compress(wf, wb)
        torch.cuda.synchronize()
        a64, _, rbits = o.compress(bf16_np(wf), wb_h)
        assert np.array_equal(bits_np(bits), rbits), "variant %d" % v
        assert_alpha_close(float(alpha.item()), a64, "variant %d" % v)
        del wf, alpha, bits
