"""GPU parity at the edges of the activations' range.

The tensor-core decode kernels feed the sign product sum_k x[t,k] s_v[n,k]
an operand written per token as x[t] 2^s_t split into two e4m3 terms (hi and
lo), 2^s_t a power of two that brings the token's largest |x| into
[128, 256).  These tests aim at where that representation is weakest:
* an all-zero token (its output row must be exactly zero);
* a token with one element 2^12 times its others, so that nearly every
  element lies more than 2^9 below the token's maximum;
* whole tokens scaled to ~1e-30 and ~1e30, and to the ends of the range the
  kernels guarantee (largest |x| from 2^-113 up to the largest bf16);
* a batch mixing all of them with ordinary tokens and the base model.
Each token is held to the y tolerances against its own scale (a large
token's magnitude must not hide a small token's error), and on the decode
paths the sign term alone, y minus the oracle's base product, is held to
1e-2 relative (Frobenius) and 2e-2 (max) per token: a sign operand with
only the hi term (3 mantissa bits) misses that by a factor of about three.
Outputs are f32 so that the sign term is not lost in the rounding of y."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests.gpu_util import Y_FRO_REL, Y_MAX_REL, bf16_np, bits_np, f32_np, load_bd

pytestmark = pytest.mark.gpu
DEV = "cuda"
Y_PATHS = ["simt", "decode_tc", "decode_fold", "prefill_tc", "auto"]
SIGN_PATHS = ["simt", "decode_tc", "decode_fold", "auto"]
SIGN_FRO = 1e-2
SIGN_MAX = 2e-2
# token kinds: (name, how the row is built from a N(0,1) row r)
KINDS = ["normal", "zero", "outlier", "tiny", "huge", "bottom", "top", "unit"]


@pytest.fixture(scope="module")
def bd():
    return load_bd()


@pytest.fixture(scope="module")
def o():
    return oracle.get()


def make_token(kind, r, k0):
    r = r.clone()
    if kind == "zero":
        return torch.zeros_like(r)
    if kind == "outlier":                    # one element 2^12 x the others' scale
        r[k0] = 4096.0
        return r
    scale = {"normal": 1.0, "tiny": 1e-30, "huge": 1e30, "bottom": 4e-33, "top": 1e36}.get(kind)
    if scale is not None:
        return r * scale
    return torch.sign(r) + (r == 0).float()  # "unit": every element +-1 (the split is exact)


def build_batch(kinds, K, g):
    rows = []
    base = torch.randn((len(kinds), K), generator=g, device=DEV, dtype=torch.float32)
    for i, kind in enumerate(kinds):
        rows.append(make_token(kind, base[i], (37 * i + 5) % K))
    return torch.stack(rows).to(torch.bfloat16)


def per_token_check(y, ref, what, max_rel, fro_rel, tokens=None):
    for t in (range(ref.shape[0]) if tokens is None else tokens):
        scale = float(np.max(np.abs(ref[t])))
        if scale == 0.0:
            assert np.all(y[t] == 0.0), "%s token %d: expected an exact zero row" % (what, t)
            continue
        err = float(np.max(np.abs(y[t] - ref[t])))
        fro = float(np.linalg.norm(y[t] - ref[t]) / np.linalg.norm(ref[t]))
        assert np.all(np.isfinite(y[t])), "%s token %d: non-finite" % (what, t)
        assert err <= max_rel * scale, "%s token %d: max err %.3e > %.0e x %.3e" % (what, t, err, max_rel, scale)
        assert fro <= fro_rel, "%s token %d: relative Frobenius %.3e > %.0e" % (what, t, fro, fro_rel)


def run_case(bd, o, path, x, ids, wb, alphas, bits):
    M, K = x.shape
    N = wb.shape[0]
    V = len(bits)
    ws = bd.linear_workspace(M, N, K, V, DEV)
    try:
        y = bd.linear(x, ids, wb, alphas, bits, out_dtype=torch.float32, workspace=ws, path=path)
    except bd.BitDeltaError as e:
        if e.code == bd.BD_ERR_UNSUPPORTED:
            pytest.skip("path %s does not take this shape" % path)
        raise
    st = bd.device_status(ws)
    assert st == 0, bd.status_string(st)
    y = y.cpu().numpy().astype(np.float64)
    xh, idh, wbh = bf16_np(x), ids.cpu().numpy(), bf16_np(wb)
    bh = [bits_np(b) for b in bits]
    ref = o.linear(xh, idh, wbh, f32_np(alphas), bh)
    per_token_check(y, ref, path + " y", Y_MAX_REL, Y_FRO_REL)
    if path in SIGN_PATHS:
        # the sign term of the variants' tokens (base-model tokens have none:
        # y minus the exact base product is only the base product's rounding)
        base = o.linear(xh, idh, wbh, np.zeros(V, np.float32), bh)
        tokens = [t for t in range(M) if idh[t] >= 0]
        per_token_check(y - base, ref - base, path + " sign term", SIGN_MAX, SIGN_FRO, tokens)


def random_bits(g, N, K, V):
    return [torch.randint(-2 ** 31, 2 ** 31, (N, K // 32), generator=g, device=DEV,
                          dtype=torch.int64).to(torch.int32) for _ in range(V)]


@pytest.mark.parametrize("path", Y_PATHS)
@pytest.mark.parametrize("kind", KINDS)
def test_one_kind_per_batch(bd, o, path, kind):
    """16 tokens of one kind over two variants (and the base model)."""
    g = wl.generator(700 + KINDS.index(kind), DEV)
    M, N, K, V = 16, 256, 4096, 2
    wb = wl.base_weights(N, K, g, DEV)
    bits = random_bits(g, N, K, V)
    alphas = torch.tensor([1.0e-3, 2.0e-3], device=DEV)
    x = build_batch([kind] * M, K, g)
    ids = torch.tensor([0, 1] * 7 + [-1, 0], dtype=torch.int32, device=DEV)
    run_case(bd, o, path, x, ids, wb, alphas, bits)


@pytest.mark.parametrize("path", Y_PATHS)
def test_mixed_magnitudes_many_variants(bd, o, path):
    """128 tokens of every kind in one batch, 14 variants with Zipf(1.1) ids
    plus base-model tokens: the folded kernel's shared sign accumulator
    carries tokens of very different scales side by side."""
    g = wl.generator(720, DEV)
    M, N, K, V = 128, 384, 4096, 14
    wb = wl.base_weights(N, K, g, DEV)
    bits = random_bits(g, N, K, V)
    alphas = torch.rand(V, generator=g, device=DEV) * 1.8e-3 + 2e-4
    kinds = [KINDS[i % len(KINDS)] for i in range(M)]
    x = build_batch(kinds, K, g)
    ids = wl.variant_ids_zipf(M, V, 1.1, wl.generator(721))
    ids[::11] = -1
    run_case(bd, o, path, x, ids.to(DEV), wb, alphas, bits)


@pytest.mark.parametrize("kind", KINDS)
def test_one_kind_single_variant(bd, o, kind):
    """The single-variant kernel (bf16 W_eff tiles, the activations used as
    they are) on every token kind, with base-model tokens."""
    g = wl.generator(760 + KINDS.index(kind), DEV)
    M, N, K = 16, 256, 4096
    wb = wl.base_weights(N, K, g, DEV)
    bits = random_bits(g, N, K, 1)
    alphas = torch.tensor([1.5e-3], device=DEV)
    x = build_batch([kind] * M, K, g)
    ids = torch.tensor([0, 0, -1, 0] * 4, dtype=torch.int32, device=DEV)
    run_case(bd, o, "decode_weff", x, ids, wb, alphas, bits)
