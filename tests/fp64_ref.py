"""fp64 evaluation of the layer's definition on a set of tokens (test
infrastructure), the anchor that both the CUDA path and the fp32 oracle are
measured against.

For each (token, slot) routed to a local expert e (Chord page, "Two kernel
families" and the layer's definition): g = W13_e[:I] x and u = W13_e[I:] x
accumulated in fp64 (numpy's BLAS, error ~1e-16 relative, far below either
fp32 implementation), h = the correctly rounded bf16(silu(g) * u), y = W2_e h
in fp64, out = sum over the token's local slots of w * y in fp64, not rounded.
The weights are the oracle's dequantised values (oracle.dequant, pinned
exhaustively against exact rational rounding), widened to fp64; bf16 rounding
of h uses pins.rne_bf16 (frexp / rint, independent of oracle.c).

Why it exists: h = bf16(silu(g) * u) is a rounding decision taken on fp32
accumulations.  Any fp32 implementation takes a different decision than the
exact value for a small fraction of h elements, and one flipped element moves
an output by more than 1e-3 * rms(out).  Measured against this evaluation,
the flip fraction of h and the end-to-end tolerance ratio of each
implementation say how far it is from the definition itself, not from another
fp32 implementation with its own summation order.
"""

from __future__ import annotations

import numpy as np

import oracle
import pins
from w4a16_int4_mixture_gb300 import synth


class Fp64Layer:
    """h and out of the definition for the tokens `tokens` of a draw.

    h64[(t, j)]  bf16 bits [I] of the correctly rounded h of token t, slot j
    out64        float64 [len(tokens), H], the unrounded layer output
    """

    def __init__(self, inp: synth.MoEInputs, tokens=None):
        s = inp.shape
        self.tokens = np.arange(s.T) if tokens is None else np.asarray(tokens)
        lid = synth.local_ids(inp)
        row_of = {int(t): i for i, t in enumerate(self.tokens)}
        self.h64 = {}
        self.out64 = np.zeros((len(self.tokens), s.H), dtype=np.float64)
        by_expert = {}
        for t in self.tokens:
            for j in range(s.k):
                e = int(lid[t, j])
                if e >= 0:
                    by_expert.setdefault(e, []).append((int(t), j))
        for e, pairs in sorted(by_expert.items()):
            W13 = oracle.dequant(inp.w13_q[e], inp.w13_s[e], 2 * s.I, s.H).astype(np.float64)
            X = pins.bf16_bits_to_f64(inp.x[[t for t, _ in pairs]])      # [n, H]
            G = X @ W13[:s.I].T
            U = X @ W13[s.I:].T
            del W13
            Hh = pins.rne_bf16(pins.silu64(G) * U)                         # [n, I]
            W2 = oracle.dequant(inp.w2_q[e], inp.w2_s[e], s.H, s.I).astype(np.float64)
            Y = Hh @ W2.T                                                  # [n, H]
            del W2
            bits = pins.f64_to_bf16_bits(Hh)
            for n, (t, j) in enumerate(pairs):
                self.h64[(t, j)] = bits[n]
                self.out64[row_of[t]] += float(inp.topk_weights[t, j]) * Y[n]


def h_flip_stats(h_bits: dict, h64: dict):
    """Fraction of h elements whose bf16 code differs from the correctly
    rounded value, among those the fraction smaller in magnitude, and the
    number of elements compared.  h_bits maps (t, j) to bf16 bits [I] like
    Fp64Layer.h64."""
    keys = [key for key in h64 if key in h_bits]
    if not keys:
        return 0.0, 0.0, 0
    a = np.stack([h_bits[key] for key in keys])
    b = np.stack([h64[key] for key in keys])
    diff = a != b
    n = int(np.count_nonzero(diff))
    if n == 0:
        return 0.0, 0.0, a.size
    av = np.abs(pins.bf16_bits_to_f64(a[diff]))
    bv = np.abs(pins.bf16_bits_to_f64(b[diff]))
    return n / a.size, float(np.mean(av < bv)), a.size


def out_ratio(out_bits, out64) -> float:
    """Worst element of |out - out64| / (1e-2*|out64| + 1e-3*rms(out64))."""
    return pins.tolerance_violation(pins.bf16_bits_to_f64(out_bits), out64)
