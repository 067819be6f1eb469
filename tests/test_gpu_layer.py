"""GPU: one decoder layer's seven linears chained (bit_delta_compressed_gb300.layer)
with 4 Zipf variants.  Every projection is checked against the CPU oracle on
the input it actually received (sampled rows, all tokens), and the torch glue
(residual adds, SiLU product) against torch on the same tensors."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from bit_delta_compressed_gb300 import layer
from tests.gpu_util import assert_y_close, bf16_np, bits_np, f32_np, load_bd

pytestmark = pytest.mark.gpu
DEV = "cuda"
HIDDEN, KV, FFN = 1024, 256, 2048
SHAPES = {"q": (HIDDEN, HIDDEN), "k": (KV, HIDDEN), "v": (KV, HIDDEN), "o": (HIDDEN, HIDDEN),
          "gate": (FFN, HIDDEN), "up": (FFN, HIDDEN), "down": (HIDDEN, FFN)}


@pytest.fixture(scope="module")
def bd():
    return load_bd()


@pytest.fixture(scope="module")
def o():
    return oracle.get()


@pytest.mark.parametrize("path", ["auto", "decode_tc", "decode_fold"])
def test_chained_layer(bd, o, path):
    g = wl.generator(300, DEV)
    V, M = 4, 32
    ids = wl.variant_ids_zipf(M, V, 1.1, wl.generator(301)).to(DEV)
    lin, bufs = {}, {}
    for name in layer.NAMES:
        N, K = SHAPES[name]
        wb = wl.base_weights(N, K, g, DEV)
        bits = [torch.randint(-2 ** 31, 2 ** 31, (N, K // 32), generator=g, device=DEV,
                              dtype=torch.int64).to(torch.int32) for _ in range(V)]
        alphas = 1e-3 * (1 + torch.rand(V, generator=g, device=DEV))
        lin[name] = {"wb": wb, "alphas": alphas, "bits": bits, "ptrs": bd.bits_pointer_array(bits)}
        bufs[name] = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    ws = bd.linear_workspace(M, FFN, FFN, V, DEV)
    bd.group(ids, V, ws)
    h = wl.activations(M, HIDDEN, g, DEV)
    try:
        h2, parts = layer.chained_layer(bd, lin, h, V, ws, bufs, path=path, keep=True)
    except bd.BitDeltaError as e:
        if e.code == bd.BD_ERR_UNSUPPORTED:
            pytest.skip("path %s does not take this shape" % path)
        raise
    torch.cuda.synchronize()
    assert bd.device_status(ws) == 0
    rng = np.random.default_rng(302)
    ids_np = ids.cpu().numpy()
    for name in layer.NAMES:
        x, y = parts[name]
        N = SHAPES[name][0]
        rows = np.sort(rng.choice(N, 64, replace=False))
        L = lin[name]
        ref = o.linear(bf16_np(x), ids_np, bf16_np(L["wb"]), f32_np(L["alphas"]),
                       [bits_np(b) for b in L["bits"]], rows=rows)
        assert_y_close(y.float().cpu().numpy().astype(np.float64)[:, rows], ref, "%s %s" % (path, name))
    h1 = parts["h1"]
    assert torch.equal(h1, h + parts["o"][1])
    a = parts["down"][0]
    assert torch.equal(a, torch.nn.functional.silu(parts["gate"][1]) * parts["up"][1])
    assert torch.equal(h2, h1 + parts["down"][1])
