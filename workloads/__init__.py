"""Seeded synthetic inputs for the BitDelta hot path (shared by tests and bench).

This module only DRAWS inputs: base weights, fine-tuned weights built from a
synthetic delta, activations and per-token variant ids.  It holds none of the
method's arithmetic (no delta, no scale, no sign packing, no linear); both the
CUDA library and the CPU oracle receive what it produces.

Recipe (the shapes and distributions of the scenario on the web page
"BitDelta: serving 14 Zen models from one GPU cluster": a 70B bf16 base model
with 14 fine-tuned variants whose deltas follow a Laplace(0, b) law, section
"The mathematical foundation"):

* base weights: W_base ~ N(0, 0.02^2), drawn in f32, rounded to bf16 (RNE)
  unless the case keeps f32;
* delta: Laplace(0, b) drawn by the inverse CDF from a uniform variate
  u in (-1/2, 1/2): d = -b * sgn(u) * ln(1 - 2|u|);
* fine-tuned weights: W_ft = W_base + d, computed in f32 and rounded to bf16
  for bf16 cases (what a bf16 fine-tuned checkpoint holds), kept f32 for f32
  cases;
* activations: x ~ N(0, 1) rounded to bf16;
* variant ids: uniform over 0..V-1, or Zipf(s) with P(v = k) proportional to
  (k + 1)^-s, or fixed blocks (prefill: tokens grouped by variant).

Everything is drawn from an explicit ``torch.Generator`` so a (seed, device)
pair reproduces the same tensors.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

# -- shapes of the 70B-class decoder layer (hidden 8192, FFN 28672, 64 query
#    heads and 8 key/value heads of width 128); [d_out, d_in] per linear -----
HIDDEN = 8192
FFN = 28672
KV = 8 * 128
LAYER_LINEARS = (
    ("q", HIDDEN, HIDDEN),
    ("k", KV, HIDDEN),
    ("v", KV, HIDDEN),
    ("o", HIDDEN, HIDDEN),
    ("gate", FFN, HIDDEN),
    ("up", FFN, HIDDEN),
    ("down", HIDDEN, FFN),
)


def generator(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def base_weights(N: int, K: int, gen: torch.Generator, device="cpu",
                 dtype=torch.bfloat16, std: float = 0.02) -> torch.Tensor:
    """W_base ~ N(0, std^2), drawn in f32 then cast (RNE) to ``dtype``."""
    w = torch.randn((N, K), generator=gen, device=device, dtype=torch.float32)
    w.mul_(std)
    return w if dtype == torch.float32 else w.to(dtype)


def laplace(shape, b: float, gen: torch.Generator, device="cpu") -> torch.Tensor:
    """Laplace(0, b) in f32 by the inverse CDF of a uniform variate."""
    u = torch.rand(shape, generator=gen, device=device, dtype=torch.float32)
    u.sub_(0.5)
    # keep 1 - 2|u| away from zero so the logarithm stays finite
    a = u.abs().mul_(2.0).clamp_(max=1.0 - 2.0 ** -24)
    d = torch.log1p(a.neg_())           # ln(1 - 2|u|) <= 0
    d.mul_(-b)
    d.mul_(torch.sign(u))
    return d


def finetuned_weights(w_base: torch.Tensor, b: float, gen: torch.Generator,
                      out_dtype=None, chunk_rows: int = 4096) -> torch.Tensor:
    """W_ft = W_base + Laplace(0, b) in f32, cast to ``out_dtype`` (default:
    w_base's dtype).  Drawn in row chunks to bound the f32 temporaries."""
    out_dtype = out_dtype or w_base.dtype
    N, K = w_base.shape
    out = torch.empty((N, K), dtype=out_dtype, device=w_base.device)
    for r0 in range(0, N, chunk_rows):
        r1 = min(N, r0 + chunk_rows)
        d = laplace((r1 - r0, K), b, gen, device=w_base.device)
        d.add_(w_base[r0:r1].to(torch.float32))
        out[r0:r1].copy_(d)
    return out


def activations(M: int, K: int, gen: torch.Generator, device="cpu") -> torch.Tensor:
    """x ~ N(0, 1) in bf16, [M, K]."""
    return torch.randn((M, K), generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)


def variant_ids_uniform(M: int, V: int, gen: torch.Generator) -> torch.Tensor:
    return torch.randint(0, V, (M,), generator=gen, dtype=torch.int64).to(torch.int32)


def zipf_probs(V: int, s: float) -> torch.Tensor:
    p = torch.tensor([(k + 1) ** (-s) for k in range(V)], dtype=torch.float64)
    return p / p.sum()


def variant_ids_zipf(M: int, V: int, s: float, gen: torch.Generator) -> torch.Tensor:
    """Per-token variant ids with P(v = k) proportional to (k + 1)^-s."""
    return torch.multinomial(zipf_probs(V, s), M, replacement=True, generator=gen).to(torch.int32)


def variant_ids_blocks(counts) -> torch.Tensor:
    """Tokens grouped by variant: counts[v] consecutive tokens of variant v."""
    return torch.cat([torch.full((c,), v, dtype=torch.int32) for v, c in enumerate(counts)])


def scales_uniform(V: int, lo: float, hi: float, gen: torch.Generator) -> list:
    """Per-variant Laplace scales b_v ~ U[lo, hi]."""
    u = torch.rand((V,), generator=gen, dtype=torch.float64)
    return [float(lo + (hi - lo) * t) for t in u]


# -- the five workloads -----------------------------------------------------

@dataclass(frozen=True)
class Workload:
    name: str
    description: str


WORKLOADS = {
    "tiny": Workload("tiny", "f32 256x256, Laplace(0,1e-3) delta, x 4x256, 1 variant, seed 0"),
    "single": Workload("single", "bf16 4096x4096, Laplace(0,5e-4) delta, decode M in {1,8,32,64}, 1 variant"),
    "ffn14": Workload("ffn14", "bf16 14336x4096 up-proj, 14 variants b_v~U[2e-4,2e-3], decode M=64 uniform ids"),
    "stack70b": Workload("stack70b", "20 layers x {q,k,v,o,gate,up,down} of a 70B-shaped decoder "
                                     "(hidden 8192, FFN 28672, kv 1024), 14 variants Laplace(0,1e-3), "
                                     "decode M=128, Zipf(1.1) ids"),
    "prefill": Workload("prefill", "gate/up 28672x8192 bf16, 4 variants x 4096 tokens grouped, "
                                   "Laplace(0,1e-3); compress 14 variants of 28672x8192"),
}


def expected_distinct(M: int, probs) -> float:
    """E[#distinct variants among M i.i.d. draws] = sum_v 1 - (1 - p_v)^M."""
    return float(sum(1.0 - (1.0 - float(p)) ** M for p in probs))


def stack_weight_count(layers: int = 20) -> int:
    return layers * sum(n * k for _, n, k in LAYER_LINEARS)


def log2_ceil(n: int) -> int:
    return int(math.ceil(math.log2(max(1, n))))
