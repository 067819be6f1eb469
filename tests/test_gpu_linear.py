"""GPU parity: bitdelta_linear (every kernel path) against the CPU oracle.

y must satisfy max|y - y_ref| <= 1e-2 * max|y_ref| and relative Frobenius
error <= 5e-3 (fp32 accumulation).  Small cases compare every output; the
full-size workloads compare sampled output rows (all tokens) that the oracle
computes one by one."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests.gpu_util import assert_y_close, bf16_np, bits_np, f32_np, load_bd

pytestmark = pytest.mark.gpu
DEV = "cuda"
PATHS = ["simt", "decode_tc", "prefill_tc", "decode_fold", "decode_weff"]


@pytest.fixture(scope="module")
def bd():
    return load_bd()


@pytest.fixture(scope="module")
def o():
    return oracle.get()


def run(bd, path, x, ids, wb, alphas, bits, out_dtype=torch.float32, expect_status=0):
    """Run one path; skip if that path does not take this shape."""
    ws = bd.linear_workspace(x.shape[0], wb.shape[0], x.shape[1], len(bits), DEV)
    try:
        y = bd.linear(x, ids, wb, alphas, bits, out_dtype=out_dtype, workspace=ws, path=path)
    except bd.BitDeltaError as e:
        if e.code == bd.BD_ERR_UNSUPPORTED:
            pytest.skip("path %s does not take this shape" % path)
        raise
    st = bd.device_status(ws)
    assert st == expect_status, bd.status_string(st)
    return y.float().cpu().numpy().astype(np.float64)


def random_bits(g, N, K, V):
    return [torch.randint(-2 ** 31, 2 ** 31, (N, K // 32), generator=g, device=DEV,
                          dtype=torch.int64).to(torch.int32) for _ in range(V)]


def oracle_y(o, x, ids, wb, alphas, bits, rows=None):
    return o.linear(bf16_np(x), ids.cpu().numpy(), bf16_np(wb), f32_np(alphas),
                    [bits_np(b) for b in bits], rows=rows)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_tiny_end_to_end(bd, o, path, out_dtype):
    """f32 256x256 compress on each side, then the linear on bf16(W_base)."""
    g = wl.generator(0, DEV)
    wb32 = wl.base_weights(256, 256, g, DEV, dtype=torch.float32)
    wf32 = wl.finetuned_weights(wb32, 1e-3, g)
    x = wl.activations(4, 256, g, DEV)
    ids = torch.zeros(4, dtype=torch.int32, device=DEV)
    alpha, bits = bd.compress(wf32, wb32)
    wb = wb32.to(torch.bfloat16)
    y = run(bd, path, x, ids, wb, alpha, [bits], out_dtype)
    _, a32, rbits = o.compress(f32_np(wf32), f32_np(wb32))
    ref = o.linear(bf16_np(x), np.zeros(4, np.int32), bf16_np(wb), np.array([a32]), [rbits])
    assert_y_close(y, ref, "tiny")


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("M", [1, 8, 32, 64])
def test_single_linear_decode(bd, o, path, M):
    g = wl.generator(10 + M, DEV)
    wb = wl.base_weights(4096, 4096, g, DEV)
    wf = wl.finetuned_weights(wb, 5e-4, g)
    x = wl.activations(M, 4096, g, DEV)
    ids = torch.zeros(M, dtype=torch.int32, device=DEV)
    alpha, bits = bd.compress(wf, wb)
    y = run(bd, path, x, ids, wb, alpha, [bits])
    _, a32, rbits = o.compress(bf16_np(wf), bf16_np(wb))
    rows = np.arange(0, 4096, 3)
    ref = o.linear(bf16_np(x), np.zeros(M, np.int32), bf16_np(wb), np.array([a32]), [rbits], rows=rows)
    assert_y_close(y[:, rows], ref, "single M=%d" % M)


@pytest.mark.parametrize("path", PATHS)
def test_ffn_fourteen_variants(bd, o, path):
    """14336 x 4096 up-projection, 14 variants, 64 tokens with uniform ids."""
    g = wl.generator(20, DEV)
    N, K, V, M = 14336, 4096, 14, 64
    wb = wl.base_weights(N, K, g, DEV)
    bs = wl.scales_uniform(V, 2e-4, 2e-3, wl.generator(21))
    alphas, bits, ralphas, rbits = [], [], [], []
    wb_h = bf16_np(wb)
    for v in range(V):
        wf = wl.finetuned_weights(wb, bs[v], g)
        a, b = bd.compress(wf, wb)
        alphas.append(a)
        bits.append(b)
        _, a32, rb = o.compress(bf16_np(wf), wb_h)
        ralphas.append(a32)
        rbits.append(rb)
    alphas = torch.cat(alphas)
    x = wl.activations(M, K, g, DEV)
    ids = wl.variant_ids_uniform(M, V, wl.generator(22)).to(DEV)
    y = run(bd, path, x, ids, wb, alphas, bits)
    rows = np.sort(np.random.default_rng(23).choice(N, 1024, replace=False))
    ref = o.linear(bf16_np(x), ids.cpu().numpy(), wb_h, np.array(ralphas), rbits, rows=rows)
    assert_y_close(y[:, rows], ref, "ffn14")


@pytest.mark.parametrize("path", PATHS)
def test_stack70b_one_layer(bd, o, path):
    """The seven linears of one 70B-shaped layer at full size, 14 variants,
    128 tokens with Zipf(1.1) ids; 192 sampled rows per linear."""
    g = wl.generator(30, DEV)
    V, M = 14, 128
    ids = wl.variant_ids_zipf(M, V, 1.1, wl.generator(31)).to(DEV)
    rng = np.random.default_rng(32)
    for name, N, K in wl.LAYER_LINEARS:
        wb = wl.base_weights(N, K, g, DEV)
        bits = random_bits(g, N, K, V)
        alphas = torch.full((V,), 1e-3, device=DEV) * (1 + torch.rand(V, generator=g, device=DEV))
        x = wl.activations(M, K, g, DEV)
        y = run(bd, path, x, ids, wb, alphas, bits, torch.bfloat16)
        rows = np.sort(rng.choice(N, 192, replace=False))
        ref = oracle_y(o, x, ids, wb, alphas, bits, rows)
        assert_y_close(y[:, rows], ref, name)
        del wb, bits, x


@pytest.mark.parametrize("path", PATHS)
def test_prefill_gate(bd, o, path):
    """Prefill: 4 variants x 4096 tokens (grouped) through a 28672 x 8192 gate
    projection; 48 sampled rows, all 16384 tokens."""
    g = wl.generator(40, DEV)
    N, K, V = 28672, 8192, 4
    wb = wl.base_weights(N, K, g, DEV)
    bits = random_bits(g, N, K, V)
    alphas = torch.tensor([1.0e-3, 0.8e-3, 1.2e-3, 1.1e-3], device=DEV)
    ids = wl.variant_ids_blocks([4096] * V).to(DEV)
    x = wl.activations(ids.numel(), K, g, DEV)
    y = run(bd, path, x, ids, wb, alphas, bits, torch.bfloat16)
    rows = np.sort(np.random.default_rng(41).choice(N, 48, replace=False))
    ref = oracle_y(o, x, ids, wb, alphas, bits, rows)
    assert_y_close(y[:, rows], ref, "prefill gate")


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("M,N,K,V", [(1, 8, 32, 1), (37, 100, 96, 3), (5, 129, 64, 0),
                                     (300, 72, 160, 5), (17, 1000, 512, 64), (37, 200, 128, 3),
                                     (208, 384, 192, 14), (2, 130, 640, 2), (64, 1024, 4096, 14),
                                     (3, 96, 256, 2), (4, 200, 4096, 3)])
def test_ragged_and_edges(bd, o, path, M, N, K, V):
    g = wl.generator(M * 131 + N * 7 + K + V, DEV)
    wb = wl.base_weights(N, K, g, DEV)
    bits = random_bits(g, N, K, V)
    alphas = (torch.rand(V, generator=g, device=DEV) * 2e-3 + 1e-4) if V else torch.zeros(1, device=DEV)
    x = wl.activations(M, K, g, DEV)
    lo = -1
    ids = torch.randint(lo, max(V, 0), (M,), generator=g, device=DEV, dtype=torch.int32) if V else \
        torch.full((M,), -1, dtype=torch.int32, device=DEV)
    y = run(bd, path, x, ids, wb, alphas, bits)
    ref = oracle_y(o, x, ids, wb, alphas[:V] if V else np.zeros(0, np.float32), bits) if V else \
        o.linear(bf16_np(x), ids.cpu().numpy(), bf16_np(wb), np.zeros(0, np.float32), [])
    assert_y_close(y, ref, "edge M=%d N=%d K=%d V=%d" % (M, N, K, V))


@pytest.mark.parametrize("path", PATHS)
def test_invalid_variant_ids(bd, o, path):
    g = wl.generator(50, DEV)
    M, N, K, V = 12, 64, 128, 2
    wb = wl.base_weights(N, K, g, DEV)
    bits = random_bits(g, N, K, V)
    alphas = torch.tensor([1e-3, 2e-3], device=DEV)
    x = wl.activations(M, K, g, DEV)
    ids_h = np.array([0, 1, 5, -1, 1, -7, 0, 2, 1, 0, -2, 1], dtype=np.int32)
    ids = torch.from_numpy(ids_h).to(DEV)
    y = run(bd, path, x, ids, wb, alphas, bits, expect_status=bd.BD_ERR_VARIANT)
    bad = (ids_h < -1) | (ids_h >= V)
    assert np.all(y[bad] == 0.0)
    good = np.nonzero(~bad)[0]
    ref = o.linear(bf16_np(x)[good], ids_h[good], bf16_np(wb), f32_np(alphas),
                   [bits_np(b) for b in bits])
    assert_y_close(y[good], ref, "valid tokens")


@pytest.mark.parametrize("path", PATHS)
def test_many_small_variants_multi_pass(bd, o, path):
    """128 tokens spread two per variant over 64 variants plus base-model and
    invalid tokens: the padded sign segments exceed one tensor-memory pass."""
    g = wl.generator(60, DEV)
    M, N, K, V = 128, 256, 256, 64
    wb = wl.base_weights(N, K, g, DEV)
    bits = random_bits(g, N, K, V)
    alphas = torch.rand(V, generator=g, device=DEV) * 2e-3 + 1e-4
    ids_h = np.repeat(np.arange(V, dtype=np.int32), 2)[:M]
    ids_h[::9] = -1
    rng = np.random.default_rng(61)
    rng.shuffle(ids_h)
    x = wl.activations(M, K, g, DEV)
    ids = torch.from_numpy(ids_h).to(DEV)
    y = run(bd, path, x, ids, wb, alphas, bits)
    ref = oracle_y(o, x, ids, wb, alphas, bits)
    assert_y_close(y, ref, "multi-pass")


def test_empty_batch(bd):
    x = torch.empty((0, 64), dtype=torch.bfloat16, device=DEV)
    ids = torch.empty((0,), dtype=torch.int32, device=DEV)
    wb = torch.zeros((8, 64), dtype=torch.bfloat16, device=DEV)
    y = bd.linear(x, ids, wb, torch.zeros(1, device=DEV), [torch.zeros((8, 2), dtype=torch.int32, device=DEV)])
    assert y.shape == (0, 8)


@pytest.mark.parametrize("M", [1, 3, 16, 77, 128])
def test_single_variant_with_base_and_invalid_tokens(bd, o, M):
    """One variant (V = 1) with base-model tokens and out-of-range ids mixed
    in, on the single-variant kernel (which multiplies the base tile for
    base-model tokens beside the W_eff tile) and the automatic path."""
    g = wl.generator(900 + M, DEV)
    N, K = 384, 1024
    wb = wl.base_weights(N, K, g, DEV)
    bits = random_bits(g, N, K, 1)
    alphas = torch.tensor([1.3e-3], device=DEV)
    x = wl.activations(M, K, g, DEV)
    ids_h = np.zeros(M, dtype=np.int32)
    ids_h[1::3] = -1
    if M > 4:
        ids_h[4::11] = 7
    ids = torch.from_numpy(ids_h).to(DEV)
    bad = (ids_h < -1) | (ids_h >= 1)
    for path in ("decode_weff", "auto"):
        y = run(bd, path, x, ids, wb, alphas, bits, expect_status=bd.BD_ERR_VARIANT if bad.any() else 0)
        assert np.all(y[bad] == 0.0)
        good = np.nonzero(~bad)[0]
        ref = o.linear(bf16_np(x)[good], ids_h[good], bf16_np(wb), f32_np(alphas), [bits_np(b) for b in bits])
        assert_y_close(y[good], ref, "%s M=%d" % (path, M))


@pytest.mark.parametrize("M", [8, 64])
@pytest.mark.parametrize("N,K", [(28672, 8192), (8192, 28672), (8192, 8192)])
def test_single_variant_full_shapes(bd, o, N, K, M):
    """The single-variant kernel on the 70B stack's shapes, where its K split
    comes from the clusters that fit at once (two or more slices per row
    tile), with base-model tokens mixed in; 64 sampled output rows, all
    tokens."""
    g = wl.generator(950 + M + N // 1024, DEV)
    wb = wl.base_weights(N, K, g, DEV)
    bits = random_bits(g, N, K, 1)
    alphas = torch.tensor([8e-4], device=DEV)
    x = wl.activations(M, K, g, DEV)
    ids = torch.zeros(M, dtype=torch.int32, device=DEV)
    ids[::7] = -1
    y = run(bd, "decode_weff", x, ids, wb, alphas, bits, out_dtype=torch.bfloat16)
    rows = np.sort(np.random.default_rng(951).choice(N, 64, replace=False))
    ref = oracle_y(o, x, ids, wb, alphas, bits, rows)
    assert_y_close(y[:, rows], ref, "single variant %dx%d M=%d" % (N, K, M))


@pytest.mark.parametrize("M,N,K,V", [(1, 1000, 128, 1), (2, 777, 4096, 1), (3, 4096, 4096, 3), (5, 300, 1024, 2),
                                     (8, 2048, 4096, 1), (8, 1500, 4096, 5), (4, 1024, 8192, 2), (1, 512, 28672, 1)])
@pytest.mark.parametrize("per_row", [False, True])
def test_small_batch_cuda_cores(bd, o, M, N, K, V, per_row):
    """1 to 8 tokens on the CUDA-core path: ragged row counts, K from 128 to
    28672, one or several variants, base-model tokens and out-of-range ids
    mixed in, per-matrix and per-row scales."""
    g = wl.generator(970 + M * 7 + V + int(per_row), DEV)
    wb = wl.base_weights(N, K, g, DEV)
    bits = random_bits(g, N, K, V)
    x = wl.activations(M, K, g, DEV)
    ids_h = np.arange(M, dtype=np.int32) % V
    if M >= 3:
        ids_h[1] = -1
    if M >= 5:
        ids_h[3] = V + 2
    ids = torch.from_numpy(ids_h).to(DEV)
    bad = (ids_h < -1) | (ids_h >= V)
    if per_row:
        alphas = (2e-4 + 1.8e-3 * torch.rand(V, N, generator=g, device=DEV)).contiguous()
        ws = bd.linear_workspace(M, N, K, V, DEV)
        y = bd.linear_rows(x, ids, wb, alphas, bits, workspace=ws, path="simt")
        assert bd.device_status(ws) == (bd.BD_ERR_VARIANT if bad.any() else 0)
        y = y.float().cpu().numpy().astype(np.float64)
    else:
        alphas = 2e-4 + 1.8e-3 * torch.rand(V, generator=g, device=DEV)
        y = run(bd, "simt", x, ids, wb, alphas, bits, expect_status=bd.BD_ERR_VARIANT if bad.any() else 0)
    assert np.all(y[bad] == 0.0)
    good = np.nonzero(~bad)[0]
    rows = np.arange(N) if N <= 1024 else np.sort(np.random.default_rng(971).choice(N, 256, replace=False))
    ref = o.linear(bf16_np(x)[good], ids_h[good], bf16_np(wb), f32_np(alphas), [bits_np(b) for b in bits],
                   rows=rows, per_row_alpha=per_row)
    assert_y_close(y[good][:, rows], ref, "cuda cores M=%d N=%d K=%d V=%d rows=%s" % (M, N, K, V, per_row))


@pytest.mark.parametrize("N,K,M", [(200, 8192, 128), (1000, 8192, 64), (1366, 16384, 16), (2048, 4096, 128),
                                   (1024, 28672, 32)])
def test_folded_split_reductions(bd, o, N, K, M):
    """The folded kernel's K slices summed over a cluster's shared memory (2 to
    16 slices) or through HBM partials, on ragged row counts (a partial last
    row tile) and deep K: every output row against the oracle."""
    g = wl.generator(990 + M + N // 100, DEV)
    V = 14
    wb = wl.base_weights(N, K, g, DEV)
    bits = random_bits(g, N, K, V)
    alphas = 2e-4 + 1.8e-3 * torch.rand(V, generator=g, device=DEV)
    x = wl.activations(M, K, g, DEV)
    ids = wl.variant_ids_zipf(M, V, 1.1, wl.generator(991)).to(DEV)
    ids[::9] = -1
    y = run(bd, "decode_fold", x, ids, wb, alphas, bits, out_dtype=torch.bfloat16)
    ref = oracle_y(o, x, ids, wb, alphas, bits)
    assert_y_close(y, ref, "folded splits N=%d K=%d M=%d" % (N, K, M))
