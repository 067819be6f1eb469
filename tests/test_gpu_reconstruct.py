"""GPU parity: materialised effective weights (bitdelta_reconstruct) against
the CPU oracle, bit for bit (the nearest bf16 of the exact sum, ties to even),
with per-matrix and per-row scales, hand-made ties, a ragged shape and sampled
rows of a full-size matrix."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests.gpu_util import bf16_np, bits_np, f32_np, load_bd

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def bd():
    return load_bd()


@pytest.fixture(scope="module")
def o():
    return oracle.get()


def bits_of(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("N,K", [(1, 32), (1000, 512), (4096, 4096)])
def test_reconstruct_per_matrix(bd, o, N, K):
    g = wl.generator(200 + N, DEV)
    wb = wl.base_weights(N, K, g, DEV)
    wf = wl.finetuned_weights(wb, 1e-3, g)
    alpha, bits = bd.compress(wf, wb)
    we = bd.reconstruct(wb, alpha, bits)
    ref = o.reconstruct(bf16_np(wb), f32_np(alpha), bits_np(bits))
    assert np.array_equal(bits_of(we), ref)


def test_reconstruct_per_row(bd, o):
    g = wl.generator(210, DEV)
    N, K = 777, 1024
    wb = wl.base_weights(N, K, g, DEV)
    wf = wl.finetuned_weights(wb, 7e-4, g)
    arow, bits = bd.compress_rows(wf, wb)
    we = bd.reconstruct(wb, arow, bits)
    ref = o.reconstruct(bf16_np(wb), f32_np(arow), bits_np(bits), per_row=True)
    assert np.array_equal(bits_of(we), ref)


def test_reconstruct_ties(bd, o):
    """Rows whose sums land exactly on, just above and just below bf16
    midpoints, positive and negative."""
    vals = [(0x3F80, 2.0 ** -8), (0x3F81, 2.0 ** -8), (0x3F80, 2.0 ** -8 + 2.0 ** -20),
            (0x3F80, 2.0 ** -8 - 2.0 ** -20), (0xBF80, 2.0 ** -8), (0xBF80, 2.0 ** -8 + 2.0 ** -20),
            (0x3C00, 2.0 ** -16), (0x4120, 2.0 ** -5)]
    N, K = len(vals), 64
    wb_np = np.array([[w] * K for w, _ in vals], dtype=np.uint16)
    arow = torch.tensor([a for _, a in vals], dtype=torch.float32, device=DEV)
    bits_np_ = np.zeros((N, K // 32), dtype=np.uint32)
    bits_np_[:, 0] = 0xAAAAAAAA                        # alternate +- in the first word
    bits_np_[:, 1] = 0xFFFF0000
    wb = torch.from_numpy(wb_np.view(np.int16)).to(DEV).view(torch.bfloat16)
    bits = torch.from_numpy(bits_np_.view(np.int32)).to(DEV)
    we = bd.reconstruct(wb, arow, bits)
    ref = o.reconstruct(wb_np, f32_np(arow), bits_np_, per_row=True)
    assert np.array_equal(bits_of(we), ref)


def test_reconstruct_full_size_sampled_rows(bd, o):
    g = wl.generator(220, DEV)
    N, K = 28672, 8192
    wb = wl.base_weights(N, K, g, DEV)
    wf = wl.finetuned_weights(wb, 1e-3, g)
    alpha, bits = bd.compress(wf, wb)
    del wf
    we = bd.reconstruct(wb, alpha, bits)
    rows = np.sort(np.random.default_rng(221).choice(N, 64, replace=False))
    r = torch.from_numpy(rows).to(DEV)
    ref = o.reconstruct(bf16_np(wb[r]), f32_np(alpha), bits_np(bits[r]))
    assert np.array_equal(bits_of(we[r]), ref)


def test_reconstruct_rejects_overlap(bd):
    wb = torch.zeros((64, 64), dtype=torch.bfloat16, device=DEV)
    alpha = torch.ones(1, device=DEV)
    bits = torch.zeros((64, 2), dtype=torch.int32, device=DEV)
    with pytest.raises(bd.BitDeltaError) as e:
        bd.reconstruct(wb, alpha, bits, out=wb)
    assert e.value.code == bd.BD_ERR_ALIGN
