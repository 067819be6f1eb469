"""A decoder layer's seven linears chained as one decode step.

Page: "BitDelta: serving 14 Zen models from one GPU cluster", section
"Serving architecture": every linear of a variant's forward pass runs as the
fused multi-variant linear against the shared base weights.  This module
chains one layer's projections the way a decoder layer feeds them, with the
glue between them in plain torch:

    q, k, v = L_q(h), L_k(h), L_v(h)
    o       = L_o(q)            (q stands in for the attention output: the
                                 attention arithmetic is not part of the method)
    h1      = h + o
    a       = silu(L_gate(h1)) * L_up(h1)
    h2      = h1 + L_down(a)

All tokens of the batch keep their variant through the layer, so the batch is
grouped once (``bd.group``) and every projection runs through
``bd.linear_grouped`` on that grouping.
"""
from __future__ import annotations

NAMES = ("q", "k", "v", "o", "gate", "up", "down")


def chained_layer(bd, lin: dict, h, V: int, ws, bufs: dict, path: str = "auto", keep: bool = False):
    """One layer on the hidden states ``h`` [M, hidden] (bf16).

    ``lin`` maps each name in ``NAMES`` to a dict with ``wb`` (bf16 [N, K]),
    ``alphas`` (f32 [V]) and ``ptrs`` (from ``bd.bits_pointer_array``);
    ``bufs`` maps each name to a preallocated bf16 output [M, N].  The batch
    must already be grouped in ``ws``.  Returns h2, and with ``keep`` also the
    dict of every projection's input and output."""
    import torch

    def proj(name, x):
        L = lin[name]
        bd.linear_grouped(x, L["wb"], L["alphas"], L["ptrs"], V, bufs[name], ws, path=path)
        return bufs[name]

    q = proj("q", h)
    proj("k", h)
    proj("v", h)
    o = proj("o", q)
    h1 = h + o
    g = proj("gate", h1)
    u = proj("up", h1)
    a = torch.nn.functional.silu(g) * u
    d = proj("down", a)
    h2 = h1 + d
    if not keep:
        return h2
    return h2, {"q": (h, q), "k": (h, bufs["k"]), "v": (h, bufs["v"]), "o": (q, o), "h1": h1,
                "gate": (h1, g), "up": (h1, u), "down": (a, d)}
