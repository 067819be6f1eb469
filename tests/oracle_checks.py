"""Pins for the CPU oracle: checks against facts fixed by the page and by the
mathematics, never against the oracle itself.

Page: "BitDelta: serving 14 Zen models from one GPU cluster" (Hanzo blog).

Each ``check_*`` takes an ``oracle.Oracle`` and raises ``AssertionError`` on a
mismatch.  ``tests/test_oracle_pins.py`` runs them on the real oracle;
``tests/test_oracle_mutants.py`` runs them on copies of the oracle with one
planted mistake each and requires every mutant to fail at least one check.

What pins what:
* packing / bit order / sign(0): an independent packer (numpy ``packbits``,
  little bit order) over all 2^16 sign patterns, and signed zeros;
* alpha = mean|delta|: a hand-computed value, the closed form (all |delta|
  equal), the Laplace expectation E|delta| = b, and least-squares optimality
  of the mean (the scale minimising ||delta - a*sign(delta)||_F);
* the linear: exact integer arithmetic for the closed form, numpy matmul for
  zero delta, all-ones bits, one-hot activations, the linearity split into
  base and sign parts with an independent unpacker, variant id -1;
* sizes printed on the page (tests/golden/page_sizes.json).
"""
from __future__ import annotations

import json
import os

import numpy as np
from fractions import Fraction

HERE = os.path.dirname(os.path.abspath(__file__))


# -- helpers independent of the oracle ------------------------------------

def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float values to bf16 (nearest-even) and return the bit patterns."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f64(u: np.ndarray) -> np.ndarray:
    return (u.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def pack_ref(nonneg: np.ndarray) -> np.ndarray:
    """Independent packer: numpy packbits with little bit order, as u32 words."""
    b = np.packbits(nonneg.astype(np.uint8), axis=1, bitorder="little")
    return np.ascontiguousarray(b).view("<u4")


def unpack_ref(bits: np.ndarray, K: int) -> np.ndarray:
    """Independent unpacker: +1 where the bit is set, -1 elsewhere."""
    u8 = np.ascontiguousarray(bits).view(np.uint8)
    b = np.unpackbits(u8, axis=1, bitorder="little")[:, :K]
    return np.where(b == 1, 1.0, -1.0)


# -- compression pins ------------------------------------------------------

def check_packer_all_sign_patterns(o):
    R = 1 << 16
    c = 2.0 ** -12
    r = np.arange(R, dtype=np.int64)[:, None]
    j = np.arange(16, dtype=np.int64)[None, :]
    lo = np.where((r >> j) & 1, c, -c)            # columns 0..15
    hi = np.where((r >> j) & 1, -c, c)            # columns 16..31, mirrored
    delta = np.concatenate([lo, hi], axis=1)
    delta[::7, 31] = 0.0                          # exact zeros -> bit 1
    rng = np.random.default_rng(1)
    w_base = (rng.integers(-64, 65, size=delta.shape) * 2.0 ** -10).astype(np.float32)
    w_ft = (w_base.astype(np.float64) + delta).astype(np.float32)
    assert np.array_equal(w_ft.astype(np.float64) - w_base.astype(np.float64), delta)
    _, _, bits = o.compress(w_ft, w_base)
    assert np.array_equal(bits, pack_ref(delta >= 0)), "packed bits differ from packbits"


def check_signed_zeros(o):
    w_ft = np.zeros((2, 32), dtype=np.float32)
    w_base = np.zeros((2, 32), dtype=np.float32)
    w_ft[0, :] = -0.0                              # -0 - (+0) = -0
    w_base[1, :] = -0.0                            # +0 - (-0) = +0
    w_ft[0, 5] = -1.0                              # one negative delta
    a64, a32, bits = o.compress(w_ft, w_base)
    assert bits[0, 0] == np.uint32(0xFFFFFFFF ^ (1 << 5)), hex(int(bits[0, 0]))
    assert bits[1, 0] == np.uint32(0xFFFFFFFF)
    assert a64 == 1.0 / 64


def check_hand_alpha(o):
    # row 0: delta = 1..32 * 2^-8, row 1: its negation.
    # sum |delta| = 2 * (32*33/2) * 2^-8 = 4.125; mean over 64 entries:
    # 4.125 / 64 = 0.064453125 exactly.
    d = np.arange(1, 33, dtype=np.float64) * 2.0 ** -8
    w_base = np.full((2, 32), 0.5, dtype=np.float32)
    w_ft = (w_base + np.stack([d, -d])).astype(np.float32)
    a64, a32, bits = o.compress(w_ft, w_base)
    assert a64 == 0.064453125, a64
    assert a32 == np.float32(0.064453125)
    assert bits[0, 0] == np.uint32(0xFFFFFFFF) and bits[1, 0] == 0


def check_bf16_matches_f32_path(o):
    rng = np.random.default_rng(2)
    wb = to_bf16_bits(rng.normal(0, 0.02, size=(64, 256)))
    wf = to_bf16_bits(bf16_bits_to_f64(wb) + rng.laplace(0, 1e-3, size=(64, 256)))
    a64_b, a32_b, bits_b = o.compress(wf, wb)
    a64_f, a32_f, bits_f = o.compress(bf16_bits_to_f64(wf).astype(np.float32),
                                      bf16_bits_to_f64(wb).astype(np.float32))
    assert np.array_equal(bits_b, bits_f)
    assert a64_b == a64_f
    d = bf16_bits_to_f64(wf) - bf16_bits_to_f64(wb)
    assert np.array_equal(bits_b, pack_ref(d >= 0))
    assert abs(a64_b - np.abs(d).mean()) <= 1e-12 * np.abs(d).mean()


def check_closed_form_compress(o):
    rng = np.random.default_rng(3)
    c = 2.0 ** -12
    s = rng.choice([-1.0, 1.0], size=(48, 96))
    w_base = (rng.integers(-64, 65, size=s.shape) * 2.0 ** -10).astype(np.float32)
    w_ft = (w_base.astype(np.float64) + c * s).astype(np.float32)
    a64, a32, bits = o.compress(w_ft, w_base)
    assert a64 == c and a32 == np.float32(c)
    assert np.array_equal(bits, pack_ref(s > 0))


def check_laplace_expectation(o):
    # |delta| ~ Exp(b) when delta ~ Laplace(0, b): E|delta| = b, Var|delta| = b^2,
    # so the sample mean lies within 5 b / sqrt(n) of b.  With a = E|delta|,
    # E(delta - a sign delta)^2 = Var|delta| = b^2 and E delta^2 = 2 b^2, so the
    # relative squared error of the 1-bit code tends to 1/2.
    rng = np.random.default_rng(4)
    b = 1e-3
    N, K = 256, 1024
    n = N * K
    delta = rng.laplace(0.0, b, size=(N, K)).astype(np.float32)
    w_base = np.zeros((N, K), dtype=np.float32)
    a64, a32, bits = o.compress(delta, w_base)
    assert abs(a64 - b) <= 5 * b / np.sqrt(n), (a64, b)
    d = delta.astype(np.float64)
    S = unpack_ref(bits, K)
    rel = np.sum((d - a64 * S) ** 2) / np.sum(d ** 2)
    assert abs(rel - 0.5) < 0.02, rel


def check_alpha_least_squares(o):
    rng = np.random.default_rng(5)
    d = rng.standard_t(3, size=(32, 128)) * 1e-3
    w_base = np.zeros(d.shape, dtype=np.float32)
    w_ft = d.astype(np.float32)
    a64, _, bits = o.compress(w_ft, w_base)
    dd = w_ft.astype(np.float64)
    S = unpack_ref(bits, 128)

    def f(a):
        return float(np.sum((dd - a * S) ** 2))
    assert f(a64) <= f(a64 * (1 + 1e-3)) and f(a64) <= f(a64 * (1 - 1e-3))
    grad = float(np.sum((dd - a64 * S) * S))
    assert abs(grad) <= 1e-9 * float(np.sum(np.abs(dd)))


def check_zero_delta_compress(o):
    rng = np.random.default_rng(6)
    w = to_bf16_bits(rng.normal(0, 0.02, size=(16, 64)))
    a64, a32, bits = o.compress(w, w.copy())
    assert a64 == 0.0 and a32 == 0.0
    assert np.all(bits == np.uint32(0xFFFFFFFF))


def check_rows_alpha(o):
    rng = np.random.default_rng(7)
    wb = rng.normal(0, 0.02, size=(8, 64)).astype(np.float32)
    wf = (wb + rng.laplace(0, 1e-3, size=(8, 64))).astype(np.float32)
    a64, a32, bits = o.compress_rows(wf, wb)
    s64, _, sbits = o.compress(wf, wb)
    assert np.array_equal(bits, sbits)
    d = wf.astype(np.float64) - wb.astype(np.float64)
    assert np.allclose(a64, np.abs(d).mean(axis=1), rtol=1e-13, atol=0)
    assert abs(a64.mean() - s64) <= 1e-13 * s64       # equal row lengths
    one64, _, _ = o.compress_rows(wf[:1], wb[:1])
    r64, _, _ = o.compress(wf[:1], wb[:1])
    assert one64[0] == r64


# -- reconstruction pins ----------------------------------------------------

def check_reconstruct_closed_form(o):
    # W_base on a 2^-10 grid with |W| <= 2^-6, delta = +-2^-12: every W_ft is a
    # bf16 value, so W_eff must equal the bf16 W_ft bit for bit.
    rng = np.random.default_rng(40)
    N, K = 12, 96
    wb = rng.integers(-16, 17, size=(N, K)) * 2.0 ** -10
    s = rng.choice([-1.0, 1.0], size=(N, K))
    wf = wb + s * 2.0 ** -12
    a64, a32, bits = o.compress(wf.astype(np.float32), wb.astype(np.float32))
    assert a64 == 2.0 ** -12
    out = o.reconstruct(to_bf16_bits(wb), a32, bits)
    assert np.array_equal(out, to_bf16_bits(wf))


def check_reconstruct_ties(o):
    # hand-computed roundings around 1.0 (bf16 spacing 2^-7 above, 2^-8 below)
    cases = [  # (W_base bits, alpha, bit, expected bits)
        (0x3F80, 2.0 ** -8, 1, 0x3F80),                 # 1 + 2^-8: tie, to even 1.0
        (0x3F81, 2.0 ** -8, 1, 0x3F82),                 # 1.0078125 + 2^-8: tie, to even
        (0x3F80, 2.0 ** -8 + 2.0 ** -20, 1, 0x3F81),    # just above the tie
        (0x3F80, 2.0 ** -8 - 2.0 ** -20, 1, 0x3F80),    # just below the tie
        (0x3F80, 2.0 ** -8, 0, 0x3F7F),                 # 1 - 2^-8 is a bf16 value
        (0xBF80, 2.0 ** -8, 0, 0xBF80),                 # -1 - 2^-8: tie, to even -1.0
        (0xBF80, 2.0 ** -8 + 2.0 ** -20, 0, 0xBF81),    # beyond the tie, away from zero
    ]
    for wbits, alpha, bit, want in cases:
        wb = np.full((1, 32), wbits, dtype=np.uint16)
        bits = np.full((1, 1), 0xFFFFFFFF if bit else 0, dtype=np.uint32)
        got = o.reconstruct(wb, np.float32(alpha), bits)
        assert np.all(got == want), (hex(wbits), alpha, bit, hex(int(got[0, 0])), hex(want))


def _bf16_nearest_exact(value: Fraction) -> int:
    """Nearest bf16 (ties to even) of an exact rational, by exact arithmetic."""
    if value == 0:
        return 0
    sign = 0x8000 if value < 0 else 0
    mag = -value if value < 0 else value
    e = mag.numerator.bit_length() - mag.denominator.bit_length()
    while Fraction(2) ** e > mag:
        e -= 1
    while Fraction(2) ** (e + 1) <= mag:
        e += 1
    q = round(mag / Fraction(2) ** (e - 7))             # 8 significant bits, half to even
    v = float(q * Fraction(2) ** (e - 7))
    return sign | int(np.float32(v).view(np.uint32) >> 16)


def check_reconstruct_exact_rational(o):
    # random Laplace deltas, per-matrix and per-row scales, against exact
    # rational arithmetic and Python's round-half-even
    rng = np.random.default_rng(41)
    N, K = 3, 64
    wb = to_bf16_bits(rng.normal(0, 0.02, size=(N, K)))
    bits = rng.integers(0, 2 ** 32, size=(N, K // 32), dtype=np.uint64).astype(np.uint32)
    for per_row in (False, True):
        alpha = rng.uniform(1e-4, 3e-3, size=N if per_row else 1).astype(np.float32)
        out = o.reconstruct(wb, alpha, bits, per_row=per_row)
        s = unpack_ref(bits, K)                              # +-1
        for n in range(N):
            a = Fraction(float(alpha[n if per_row else 0]))
            for k in range(K):
                exact = Fraction(float(bf16_bits_to_f64(wb[n, k]))) + a * int(s[n, k])
                assert out[n, k] == _bf16_nearest_exact(exact), (per_row, n, k)


# -- linear pins -------------------------------------------------------------

def _rand_case(rng, M, N, K, V):
    wb = to_bf16_bits(rng.normal(0, 0.02, size=(N, K)))
    x = to_bf16_bits(rng.normal(0, 1.0, size=(M, K)))
    bits = [rng.integers(0, 2 ** 32, size=(N, K // 32), dtype=np.uint64).astype(np.uint32)
            for _ in range(V)]
    alphas = (rng.uniform(2e-4, 2e-3, size=V)).astype(np.float32)
    vid = rng.integers(-1, V, size=M).astype(np.int32)
    return x, vid, wb, alphas, bits


def check_closed_form_linear(o):
    # delta_v = +-c_v exactly, base and activations on dyadic grids: the
    # reconstruction is exact (W_eff == W_ft) and y is an exact integer sum.
    rng = np.random.default_rng(8)
    M, N, K, V = 7, 24, 96, 3
    cs = [2.0 ** -12, 2.0 ** -11, 3 * 2.0 ** -13]
    wb_i = rng.integers(-64, 65, size=(N, K))                 # W_base = wb_i * 2^-10
    wb32 = (wb_i * 2.0 ** -10).astype(np.float32)
    alphas, bits, wft_i = [], [], []
    for c in cs:
        s = rng.choice([-1, 1], size=(N, K))
        wf32 = (wb32.astype(np.float64) + c * s).astype(np.float32)
        a64, a32, b = o.compress(wf32, wb32)
        assert a64 == c
        alphas.append(a32)
        bits.append(b)
        wft_i.append(np.round(wf32.astype(np.float64) * 2 ** 13).astype(np.int64))
    x_i = rng.integers(-8, 9, size=(M, K))                   # x = x_i * 2^-3
    x = to_bf16_bits(x_i * 0.125)
    vid = np.array([0, 1, 2, -1, 2, 0, 1], dtype=np.int32)
    y = o.linear(x, vid, to_bf16_bits(wb32), np.array(alphas, dtype=np.float32), bits)
    for t in range(M):
        v = vid[t]
        w = (wb_i * 8) if v < 0 else wft_i[v]                # units of 2^-13
        exact = (x_i[t][None, :] * w).sum(axis=1) * 2.0 ** -16
        assert np.array_equal(y[t], exact), (t, v)


def check_closed_form_linear_rows(o):
    # per-row scales ("Infrastructure details": one f32 per output dimension):
    # delta_v[n, :] = +-c_{v,n} with c on a dyadic grid, different for every
    # (variant, row); bitdelta's row compression recovers c exactly, the
    # reconstruction with per-row scales is exact (W_eff == W_ft) and y is an
    # exact integer sum.  Catches a wrong (variant, row) index of the scales.
    rng = np.random.default_rng(18)
    M, N, K, V = 6, 20, 64, 3
    wb_i = rng.integers(-64, 65, size=(N, K))                 # W_base = wb_i * 2^-10
    wb32 = (wb_i * 2.0 ** -10).astype(np.float32)
    arows, bits, wft_i = [], [], []
    for v in range(V):
        c = rng.integers(1, 16, size=N) * 2.0 ** -14          # c_{v,n}
        s = rng.choice([-1, 1], size=(N, K))
        wf32 = (wb32.astype(np.float64) + c[:, None] * s).astype(np.float32)
        a64, a32, b = o.compress_rows(wf32, wb32)
        assert np.array_equal(a64, c)
        arows.append(a32)
        bits.append(b)
        wft_i.append(np.round(wf32.astype(np.float64) * 2 ** 14).astype(np.int64))
    x_i = rng.integers(-8, 9, size=(M, K))                   # x = x_i * 2^-3
    x = to_bf16_bits(x_i * 0.125)
    vid = np.array([2, 0, -1, 1, 2, 0], dtype=np.int32)
    y = o.linear(x, vid, to_bf16_bits(wb32), np.stack(arows).astype(np.float32), bits,
                 per_row_alpha=True)
    for t in range(M):
        v = vid[t]
        w = (wb_i * 16) if v < 0 else wft_i[v]               # units of 2^-14
        exact = (x_i[t][None, :] * w).sum(axis=1) * 2.0 ** -17
        assert np.array_equal(y[t], exact), (t, v)


def check_zero_delta_linear(o):
    rng = np.random.default_rng(9)
    M, N, K = 5, 40, 128
    wb = to_bf16_bits(rng.normal(0, 0.02, size=(N, K)))
    x = to_bf16_bits(rng.normal(0, 1, size=(M, K)))
    a64, a32, bits = o.compress(wb, wb.copy())
    y = o.linear(x, np.zeros(M, dtype=np.int32), wb, np.array([a32]), [bits])
    ref = bf16_bits_to_f64(x) @ bf16_bits_to_f64(wb).T
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-13)


def check_all_ones_bits(o):
    rng = np.random.default_rng(10)
    M, N, K, V = 6, 33, 64, 2
    x, vid, wb, alphas, _ = _rand_case(rng, M, N, K, V)
    ones = [np.full((N, K // 32), 0xFFFFFFFF, dtype=np.uint32) for _ in range(V)]
    y = o.linear(x, vid, wb, alphas, ones)
    xf, wf = bf16_bits_to_f64(x), bf16_bits_to_f64(wb)
    for t in range(M):
        a = 0.0 if vid[t] < 0 else float(alphas[vid[t]])
        ref = xf[t] @ wf.T + a * xf[t].sum()
        assert np.allclose(y[t], ref, rtol=1e-12, atol=1e-14)


def check_one_hot_activations(o):
    rng = np.random.default_rng(11)
    N, K, V = 20, 64, 3
    _, _, wb, alphas, bits = _rand_case(rng, 1, N, K, V)
    ks = [0, 5, 31, 32, 63, 17]
    M = len(ks)
    xf = np.zeros((M, K))
    for t, k in enumerate(ks):
        xf[t, k] = 1.0
    vid = np.array([0, 1, 2, -1, 1, 0], dtype=np.int32)
    y = o.linear(to_bf16_bits(xf), vid, wb, alphas, bits)
    wf = bf16_bits_to_f64(wb)
    for t, k in enumerate(ks):
        v = vid[t]
        col = wf[:, k].copy()
        if v >= 0:
            col += float(alphas[v]) * unpack_ref(bits[v], K)[:, k]
        assert np.array_equal(y[t], col), (t, k)


def check_linearity_split(o):
    # y_v - y_base = alpha_v * x S_v^T with S_v from an independent unpacker
    rng = np.random.default_rng(12)
    M, N, K, V = 9, 48, 160, 4
    x, vid, wb, alphas, bits = _rand_case(rng, M, N, K, V)
    y = o.linear(x, vid, wb, alphas, bits)
    yb = o.linear(x, np.full(M, -1, dtype=np.int32), wb, alphas, bits)
    xf = bf16_bits_to_f64(x)
    assert np.allclose(yb, xf @ bf16_bits_to_f64(wb).T, rtol=1e-12, atol=1e-14)
    for t in range(M):
        v = vid[t]
        if v < 0:
            assert np.array_equal(y[t], yb[t])
            continue
        ref = float(alphas[v]) * (xf[t] @ unpack_ref(bits[v], K).T)
        assert np.allclose(y[t] - yb[t], ref, rtol=1e-9, atol=1e-13), t


def check_row_subset(o):
    rng = np.random.default_rng(13)
    x, vid, wb, alphas, bits = _rand_case(rng, 4, 30, 64, 2)
    full = o.linear(x, vid, wb, alphas, bits)
    rows = np.array([29, 0, 7, 7, 15])
    part = o.linear(x, vid, wb, alphas, bits, rows=rows)
    assert np.array_equal(part, full[:, rows])


def check_conceptual_listing(o):
    """The page's conceptual fused_bitdelta_linear restated in torch fp64
    (unpack to +-1, W_eff = W_base + alpha * S, then F.linear)."""
    import torch
    rng = np.random.default_rng(14)
    M, N, K = 3, 17, 96
    x, _, wb, alphas, bits = _rand_case(rng, M, N, K, 1)
    vid = np.zeros(M, dtype=np.int32)
    y = o.linear(x, vid, wb, alphas, bits)
    words = torch.from_numpy(bits[0].astype(np.int64))
    shifts = torch.arange(32, dtype=torch.int64)
    unpacked = ((words[:, :, None] >> shifts) & 1).reshape(N, K).to(torch.float64) * 2 - 1
    w_eff = torch.from_numpy(bf16_bits_to_f64(wb)) + float(alphas[0]) * unpacked
    ref = torch.nn.functional.linear(torch.from_numpy(bf16_bits_to_f64(x)), w_eff).numpy()
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-14)


def check_page_sizes(o):
    with open(os.path.join(HERE, "golden", "page_sizes.json")) as f:
        g = {e["what"].split(",")[0]: e for e in json.load(f)["entries"]}
    e = g["packed sign matrix of a 4096 x 4096 weight"]
    w = np.zeros((e["N"], e["K"]), dtype=np.uint16)
    _, _, bits = o.compress(w, w)
    b8 = bits.view(np.uint8)
    assert b8.shape == (e["packed_rows"], e["packed_cols_bytes"])
    assert bits.nbytes == 2 * 1024 * 1024
    params = g["a 70B-parameter model in BF16"]["params"]
    assert params * 2 / 1e9 == g["a 70B-parameter model in BF16"]["gb"]
    assert params / 8 / 1e9 == g["one BitDelta delta of a 70B model"]["gb"]
    assert 14 * 140 / 1000 == g["14 full copies"]["tb"]
    total = 140 + 14 * 8.75
    assert round(total) in (262, 263) and abs(total - 262) < 1
    assert round(100 * (1 - total / 1960)) == 87
    assert g["storage of a 1-bit sign vs a 32-bit delta entry"]["ratio"] == 1 / 32


ALL_CHECKS = [v for k, v in sorted(globals().items()) if k.startswith("check_")]
