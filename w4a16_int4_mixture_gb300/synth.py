"""Seeded synthetic inputs for the W4A16 INT4 MoE expert computation.

This module only draws random inputs.  It holds none of the method's arithmetic
(no dequantisation, no GEMM, no SiLU, no combine): both the CUDA path and the CPU
oracle consume what it produces, and neither depends on the other.

Workloads follow the "Kimi K2.x serving shapes" the Chord W4A16 MoE page
(novita.ai, "vLLM x Novita AI: Chord W4A16 INT4 MoE kernels for Kimi K2.x",
TL;DR and "Measurement") talks about: 384 global experts, hidden 7168,
intermediate 2048, top-8 routing, EP8 (48 local experts) and TP8 (intermediate
sharded to 256) deployments.

Storage conventions (the boundary's input layout):
  * activations: bf16 bit patterns (uint16), row-major [T, H];
  * weight codes: unsigned 4-bit codes, 8 per int32 word along K, element
    c = 8*w + i stored in bits [4i, 4i+4) (low nibble first), row-major
    [E, N, K/8];
  * scales: bf16 bit patterns, one per 32 consecutive input channels,
    row-major [E, N, K/32];
  * routing: global expert ids int32 [T, k], weights float32 [T, k], and an
    optional expert_map int32 [E_global] (local id or -1).

bf16 values are made by truncating float32 samples to their upper 16 bits; the
distribution is what matters here, not the rounding.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


@dataclass
class MoEShape:
    """One workload: sizes plus the routing recipe."""

    name: str
    T: int                 # tokens
    k: int                 # top-k
    E_global: int          # experts the router chooses from
    E_local: int           # experts held on this GPU
    H: int                 # hidden size (gate/up K, down N)
    I: int                 # intermediate size (gate/up N = 2I, down K)
    block_m: int = 16      # padding granularity of the aligned routing
    routing: str = "uniform"   # "uniform" | "softmax_topk" | "zipf"
    zipf_s: float = 1.2
    seed: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def local_first(self) -> int:
        """First global id of the contiguous local expert range (EP shard 0)."""
        return 0


_WORKLOADS = {
    "tiny": dict(name="tiny-E8-k2-T16-H256-I128", T=16, k=2, E_global=8, E_local=8,
                 H=256, I=128, block_m=16, routing="softmax_topk", seed=0),
    "ep8-decode": dict(name="ep8-decode-E48of384-k8-T512-H7168-I2048", T=512, k=8,
                       E_global=384, E_local=48, H=7168, I=2048, seed=1),
    "ep8-prefill": dict(name="ep8-prefill-E48of384-k8-T8192-H7168-I2048", T=8192, k=8,
                        E_global=384, E_local=48, H=7168, I=2048, seed=2),
    "tp8": dict(name="tp8-E384-k8-T2048-H7168-I256", T=2048, k=8,
                E_global=384, E_local=384, H=7168, I=256, seed=3),
    "skewed": dict(name="skewed-zipf1.2-E48-k8-T128-H7168-I2048", T=128, k=8,
                   E_global=48, E_local=48, H=7168, I=2048, routing="zipf",
                   zipf_s=1.2, seed=4),
}
WORKLOADS = tuple(_WORKLOADS)


def workload(key: str, T: int | None = None) -> MoEShape:
    """One of the workloads above by its short name (tiny, ep8-decode,
    ep8-prefill, tp8, skewed), optionally with another token count T."""
    if key not in _WORKLOADS:
        raise ValueError(f"no workload {key!r} (known: {', '.join(WORKLOADS)})")
    s = MoEShape(**_WORKLOADS[key])
    if T is not None and int(T) != s.T:
        if key != "tiny":
            s.name = s.name.replace(f"-T{s.T}-", f"-T{int(T)}-")
        s.T = int(T)
    return s


def _bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 samples -> bf16 bit patterns (upper half of the float32 word)."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    return (a.view(np.uint32) >> 16).astype(np.uint16)


def activations(rng: np.random.Generator, T: int, H: int) -> np.ndarray:
    """x ~ bf16(N(0, 1)), uint16 bits [T, H]."""
    return _bf16_bits(rng.standard_normal((T, H), dtype=np.float32))


def codes_words(rng: np.random.Generator, E: int, N: int, K: int) -> np.ndarray:
    """Uniform 4-bit codes, 8 per int32 word: uniform 32-bit words give i.i.d.
    uniform nibbles.  int32 [E, N, K/8]."""
    assert K % 8 == 0
    return rng.integers(0, 2**32, size=(E, N, K // 8), dtype=np.uint32).view(np.int32)


def scales(rng: np.random.Generator, E: int, N: int, K: int, sigma: float = 0.02) -> np.ndarray:
    """Group-32 scales bf16(|N(0, sigma)|), uint16 bits [E, N, K/32]."""
    assert K % 32 == 0
    s = np.abs(rng.standard_normal((E, N, K // 32), dtype=np.float32)) * np.float32(sigma)
    return _bf16_bits(s)


def mx_scales(rng: np.random.Generator, E: int, N: int, K: int, center: int = 121) -> np.ndarray:
    """MXFP4 block scales: one E8M0 byte per 32 input channels, uniform over
    center-1 .. center+1 (2^-7 .. 2^-5 with the default, so that E2M1 codes
    of magnitude up to 6 give weights of the INT4 draw's size).  uint8
    [E, N, K/32]."""
    assert K % 32 == 0
    return rng.integers(center - 1, center + 2, size=(E, N, K // 32)).astype(np.uint8)


def pack_codes(codes: np.ndarray) -> np.ndarray:
    """Pack explicit 4-bit codes [..., K] (values 0..15) into int32 words [..., K/8]
    in the storage order above.  Used to build structured test inputs."""
    codes = np.asarray(codes, dtype=np.uint32)
    assert codes.shape[-1] % 8 == 0
    assert codes.max(initial=0) < 16
    c = codes.reshape(codes.shape[:-1] + (codes.shape[-1] // 8, 8))
    words = np.zeros(c.shape[:-1], dtype=np.uint32)
    for i in range(8):
        words |= c[..., i] << np.uint32(4 * i)
    return words.view(np.int32)


def const_scales(E: int, N: int, K: int, value_bits: int) -> np.ndarray:
    """Scales all equal to one bf16 bit pattern (e.g. 0x3F80 = 1.0)."""
    return np.full((E, N, K // 32), value_bits, dtype=np.uint16)


def _softmax_rows(z: np.ndarray) -> np.ndarray:
    z = z.astype(np.float64)
    z = z - z.max(axis=1, keepdims=True)
    e = np.exp(z)
    return (e / e.sum(axis=1, keepdims=True)).astype(np.float32)


def routing(rng: np.random.Generator, s: MoEShape):
    """Router output for a workload.

    Returns (topk_ids int32 [T, k] global ids, topk_weights float32 [T, k],
    expert_map int32 [E_global] or None).
      * softmax_topk: logits N(0,1) over all E_global experts, softmax, the k
        largest (ties to the lower id), weights renormalised to sum 1;
      * uniform: k distinct experts uniformly without replacement, weights =
        softmax of k i.i.d. N(0,1) logits;
      * zipf: expert popularity p_e ~ rank(e)^-s with ranks from a seeded
        permutation; k distinct experts per token by Gumbel-top-k; weights as
        for uniform.
    expert_map is given when E_local < E_global: global ids
    [local_first, local_first + E_local) map to 0..E_local-1, the rest to -1.
    """
    T, k, Eg = s.T, s.k, s.E_global
    if s.routing == "softmax_topk":
        logits = rng.standard_normal((T, Eg), dtype=np.float32)
        p = _softmax_rows(logits)
        # stable sort on -p keeps the lower id first among equal probabilities
        order = np.argsort(-p, axis=1, kind="stable")[:, :k]
        ids = order.astype(np.int32)
        w = np.take_along_axis(p, order, axis=1).astype(np.float64)
        w = (w / w.sum(axis=1, keepdims=True)).astype(np.float32)
    elif s.routing == "uniform":
        keys = rng.random((T, Eg))
        ids = np.argsort(keys, axis=1, kind="stable")[:, :k].astype(np.int32)
        w = _softmax_rows(rng.standard_normal((T, k), dtype=np.float32))
    elif s.routing == "zipf":
        rank = rng.permutation(Eg) + 1
        logp = -s.zipf_s * np.log(rank.astype(np.float64))
        g = rng.gumbel(size=(T, Eg))
        ids = np.argsort(-(logp[None, :] + g), axis=1, kind="stable")[:, :k].astype(np.int32)
        w = _softmax_rows(rng.standard_normal((T, k), dtype=np.float32))
    else:
        raise ValueError(s.routing)
    emap = None
    if s.E_local < Eg:
        emap = np.full(Eg, -1, dtype=np.int32)
        emap[s.local_first:s.local_first + s.E_local] = np.arange(s.E_local, dtype=np.int32)
    return np.ascontiguousarray(ids), np.ascontiguousarray(w), emap


@dataclass
class MoEInputs:
    shape: MoEShape
    x: np.ndarray          # uint16 [T, H]
    w13_q: np.ndarray      # int32 [E, 2I, H/8]
    w13_s: np.ndarray      # uint16 [E, 2I, H/32]
    w2_q: np.ndarray       # int32 [E, H, I/8]
    w2_s: np.ndarray       # uint16 [E, H, I/32]
    topk_ids: np.ndarray   # int32 [T, k]
    topk_weights: np.ndarray  # float32 [T, k]
    expert_map: np.ndarray | None


def make_inputs(s: MoEShape, seed: int | None = None, weights: bool = True,
                weight_format: str = "int4") -> MoEInputs:
    """Draw every input of one workload from numpy.random.default_rng(seed).
    weight_format "mxfp4" draws E8M0 scale bytes (mx_scales) instead of bf16
    scales; the codes are uniform 4-bit values either way."""
    rng = np.random.default_rng(s.seed if seed is None else seed)
    E, H, I = s.E_local, s.H, s.I
    if weight_format not in ("int4", "mxfp4"):
        raise ValueError(f"unknown weight format {weight_format!r}")
    draw_scales = scales if weight_format == "int4" else mx_scales
    if weights:
        w13_q = codes_words(rng, E, 2 * I, H)
        w13_s = draw_scales(rng, E, 2 * I, H)
        w2_q = codes_words(rng, E, H, I)
        w2_s = draw_scales(rng, E, H, I)
    else:
        w13_q = w13_s = w2_q = w2_s = None
    x = activations(rng, s.T, H)
    ids, w, emap = routing(rng, s)
    return MoEInputs(s, x, w13_q, w13_s, w2_q, w2_s, ids, w, emap)


def local_ids(inp: MoEInputs) -> np.ndarray:
    """Local expert id per (token, slot), -1 when not held here.  Pure lookup."""
    if inp.expert_map is None:
        ids = inp.topk_ids.copy()
        ids[(ids < 0) | (ids >= inp.shape.E_local)] = -1
        return ids
    return inp.expert_map[inp.topk_ids]


def grouped_contiguous_layout(inp: MoEInputs, align: int = 128):
    """Rows concatenated per local expert (ascending expert, ascending pair id),
    each expert's segment padded to a multiple of `align` rows.

    Returns (a2 uint16 [M, H], m_indices int32 [M] (-1 on padding),
    row_to_pair int32 [M] (-1 on padding))."""
    s = inp.shape
    lid = local_ids(inp).reshape(-1)
    rows_x, m_idx, r2p = [], [], []
    for e in range(s.E_local):
        pairs = np.nonzero(lid == e)[0]
        if len(pairs) == 0:
            continue
        n = len(pairs)
        pad = (-n) % align
        rows_x.append(inp.x[pairs // s.k])
        rows_x.append(np.zeros((pad, s.H), dtype=np.uint16))
        m_idx.append(np.full(n, e, dtype=np.int32))
        m_idx.append(np.full(pad, -1, dtype=np.int32))
        r2p.append(pairs.astype(np.int32))
        r2p.append(np.full(pad, -1, dtype=np.int32))
    if not rows_x:
        return (np.zeros((0, s.H), np.uint16), np.zeros(0, np.int32), np.zeros(0, np.int32))
    return (np.ascontiguousarray(np.concatenate(rows_x)), np.concatenate(m_idx),
            np.concatenate(r2p))


def grouped_masked_layout(inp: MoEInputs, max_m: int | None = None):
    """Fixed row budget per local expert: a3 [E, max_m, H], masked_m int32 [E]
    (valid rows per expert), row_to_pair int32 [E*max_m] (-1 past the count).
    Rows past masked_m are filled with a poison pattern (bf16 NaN bits) so that
    a consumer that reads them shows it."""
    s = inp.shape
    max_m = s.T if max_m is None else max_m
    lid = local_ids(inp).reshape(-1)
    a3 = np.full((s.E_local, max_m, s.H), 0x7FC1, dtype=np.uint16)
    masked_m = np.zeros(s.E_local, dtype=np.int32)
    r2p = np.full(s.E_local * max_m, -1, dtype=np.int32)
    for e in range(s.E_local):
        pairs = np.nonzero(lid == e)[0]
        n = len(pairs)
        assert n <= max_m, "max_m too small for this draw"
        masked_m[e] = n
        a3[e, :n] = inp.x[pairs // s.k]
        r2p[e * max_m:e * max_m + n] = pairs
    return a3, masked_m, r2p
