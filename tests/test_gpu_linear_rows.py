"""GPU parity: the fused linear with one scale per (variant, output row)
(bitdelta_linear_rows) against the CPU oracle, on every kernel path.

Scales come from the GPU's own row compression (bitdelta_compress_rows) of
Laplace deltas whose width differs from row to row, and the oracle is given
the same f32 scales and bits (compression parity is tested elsewhere).  Same
tolerances as the per-matrix linear: max|y - y_ref| <= 1e-2 * max|y_ref| and
relative Frobenius error <= 5e-3."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests.gpu_util import assert_y_close, bf16_np, bits_np, f32_np, load_bd

pytestmark = pytest.mark.gpu
DEV = "cuda"
ROW_PATHS = ["auto", "simt", "decode_tc", "prefill_tc", "decode_fold", "decode_weff"]


@pytest.fixture(scope="module")
def bd():
    return load_bd()


@pytest.fixture(scope="module")
def o():
    return oracle.get()


def row_case(bd, g, N, K, V):
    """W_base, and V variants with per-row Laplace widths b_n in [2e-4, 2e-3]:
    (alpha_rows [V, N] f32 from row compression, bits list)."""
    wb = wl.base_weights(N, K, g, DEV)
    arows, bits = [], []
    for _ in range(V):
        b = 2e-4 + 1.8e-3 * torch.rand(N, 1, generator=g, device=DEV)
        delta = wl.laplace((N, K), 1.0, g, device=DEV) * b          # Laplace(0, b_n) per row
        wf = (wb.float() + delta).to(torch.bfloat16)
        a, bt = bd.compress_rows(wf, wb)
        arows.append(a)
        bits.append(bt)
    return wb, torch.stack(arows).contiguous(), bits


def run_rows(bd, path, x, ids, wb, arows, bits, out_dtype=torch.float32):
    ws = bd.linear_workspace(x.shape[0], wb.shape[0], x.shape[1], len(bits), DEV)
    try:
        y = bd.linear_rows(x, ids, wb, arows, bits, out_dtype=out_dtype, workspace=ws, path=path)
    except bd.BitDeltaError as e:
        if e.code == bd.BD_ERR_UNSUPPORTED:
            pytest.skip("path %s does not take this shape" % path)
        raise
    assert bd.device_status(ws) == 0
    return y.float().cpu().numpy().astype(np.float64)


def oracle_rows(o, x, ids, wb, arows, bits, rows=None):
    return o.linear(bf16_np(x), ids.cpu().numpy(), bf16_np(wb), f32_np(arows), [bits_np(b) for b in bits],
                    rows=rows, per_row_alpha=True)


@pytest.mark.parametrize("path", ROW_PATHS)
@pytest.mark.parametrize("M,N,K,V", [(1, 300, 256, 2), (4, 1000, 512, 3), (37, 1366, 640, 5), (128, 2048, 1024, 14)])
def test_rows_small(bd, o, path, M, N, K, V):
    """Ragged shapes (N not a multiple of 128, several K blocks), base-model
    tokens (id -1) mixed in."""
    g = wl.generator(100 + M, DEV)
    wb, arows, bits = row_case(bd, g, N, K, V)
    x = wl.activations(M, K, g, DEV)
    ids = torch.randint(-1, V, (M,), generator=g, device=DEV, dtype=torch.int32)
    y = run_rows(bd, path, x, ids, wb, arows, bits)
    ref = oracle_rows(o, x, ids, wb, arows, bits)
    assert_y_close(y, ref, "rows %s M=%d" % (path, M))


@pytest.mark.parametrize("path", ROW_PATHS)
def test_rows_prefill_shape(bd, o, path):
    """Large grouped batch (4 variants x 512 tokens) through 4096 x 2048;
    64 sampled rows, all tokens."""
    g = wl.generator(120, DEV)
    N, K, V, per = 4096, 2048, 4, 512
    wb, arows, bits = row_case(bd, g, N, K, V)
    ids = torch.arange(V, device=DEV, dtype=torch.int32).repeat_interleave(per)
    x = wl.activations(V * per, K, g, DEV)
    y = run_rows(bd, path, x, ids, wb, arows, bits, torch.bfloat16)
    rows = np.sort(np.random.default_rng(121).choice(N, 64, replace=False))
    ref = oracle_rows(o, x, ids, wb, arows, bits, rows)
    assert_y_close(y[:, rows], ref, "rows prefill %s" % path)


def test_rows_constant_equals_per_matrix(bd):
    """Per-row scales that repeat one value per variant give exactly the
    per-matrix result (same arithmetic) on the CUDA-core and both decode
    kernels."""
    g = wl.generator(130, DEV)
    M, N, K, V = 64, 1024, 1024, 6
    wb = wl.base_weights(N, K, g, DEV)
    bits = [torch.randint(-2 ** 31, 2 ** 31, (N, K // 32), generator=g, device=DEV,
                          dtype=torch.int64).to(torch.int32) for _ in range(V)]
    alphas = 1e-3 * (1 + torch.rand(V, generator=g, device=DEV))
    arows = alphas[:, None].expand(V, N).contiguous()
    x = wl.activations(M, K, g, DEV)
    ids = torch.randint(-1, V, (M,), generator=g, device=DEV, dtype=torch.int32)
    for path in ("simt", "decode_tc", "decode_fold"):
        y1 = bd.linear(x, ids, wb, alphas, bits, path=path)
        y2 = bd.linear_rows(x, ids, wb, arows, bits, path=path)
        assert torch.equal(y1, y2), path


@pytest.mark.parametrize("per_row", [False, True])
def test_prefill_materialised(bd, o, per_row):
    """Prefill with >= 2048 tokens per variant: each present variant's W_eff is
    materialised once (nearest bf16) and multiplied without the in-tile
    rewrite; ragged N, base-model tokens mixed in, 64 sampled rows."""
    g = wl.generator(150 + int(per_row), DEV)
    N, K, V, per = 1000, 1024, 2, 2304
    wb = wl.base_weights(N, K, g, DEV)
    bits, alphas, arows = [], [], []
    for _ in range(V):
        wf = wl.finetuned_weights(wb, 8e-4, g)
        if per_row:
            a, b = bd.compress_rows(wf, wb)
            arows.append(a)
        else:
            a, b = bd.compress(wf, wb)
            alphas.append(a)
        bits.append(b)
    ids = torch.cat([torch.full((per,), v, dtype=torch.int32, device=DEV) for v in range(V)] +
                    [torch.full((100,), -1, dtype=torch.int32, device=DEV)])
    ids = ids[torch.randperm(ids.numel(), generator=torch.Generator().manual_seed(151)).to(DEV)]
    x = wl.activations(ids.numel(), K, g, DEV)
    rows = np.sort(np.random.default_rng(152).choice(N, 64, replace=False))
    if per_row:
        al = torch.stack(arows).contiguous()
        y = bd.linear_rows(x, ids, wb, al, bits, path="prefill_tc").float().cpu().numpy()
        ref = o.linear(bf16_np(x), ids.cpu().numpy(), bf16_np(wb), f32_np(al), [bits_np(b) for b in bits],
                       rows=rows, per_row_alpha=True)
    else:
        al = torch.cat(alphas)
        y = bd.linear(x, ids, wb, al, bits, path="prefill_tc").float().cpu().numpy()
        ref = o.linear(bf16_np(x), ids.cpu().numpy(), bf16_np(wb), f32_np(al), [bits_np(b) for b in bits],
                       rows=rows)
    assert_y_close(y.astype(np.float64)[:, rows], ref, "prefill materialised per_row=%s" % per_row)


@pytest.mark.parametrize("M", [1, 8, 64])
def test_rows_single_variant(bd, o, M):
    """Per-row scales on the single-variant kernel (V = 1), base-model tokens
    mixed in, a 2048 x 4096 matrix split over several K slices."""
    g = wl.generator(140 + M, DEV)
    N, K = 2048, 4096
    wb, arows, bits = row_case(bd, g, N, K, 1)
    x = wl.activations(M, K, g, DEV)
    ids = torch.zeros(M, dtype=torch.int32, device=DEV)
    ids[::5] = -1
    y = run_rows(bd, "decode_weff", x, ids, wb, arows, bits)
    rows = np.arange(0, N, 7)
    ref = oracle_rows(o, x, ids, wb, arows, bits, rows)
    assert_y_close(y[:, rows], ref, "rows single variant M=%d" % M)
