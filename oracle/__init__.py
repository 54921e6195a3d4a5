"""CPU oracle of the W4A16 INT4 MoE expert computation (test infrastructure).

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline / reference legs
may import this package.  The product path (w4a16_int4_mixture_gb300) never does.

The arithmetic lives in oracle.c (plain C, built with gcc -O2 -ffp-contract=off);
this module builds it and marshals numpy arrays into it.  bf16 values travel as
uint16 bit patterns.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

# planted mistakes (tests only): keep in step with the enum in oracle.c
MUTATIONS = {
    "nibble_high_first": 1,
    "gate_up_swapped": 2,
    "dequant_fma": 3,
    "scale_group": 4,
    "zero_sign": 5,
    "drop_weight": 6,
    "drop_last_slot": 7,
    "align_descending": 8,
    "silu_sign": 9,
    "down_transposed": 10,
    "align_no_pad": 11,
    "code_offset": 12,
    "route_tie_high": 13,
    "route_no_renorm": 14,
    "pack_no_swizzle": 15,
    "pack_tile_rows": 16,
    "mx_scale_bias": 17,
    "mx_no_subnormal": 18,
}
WEIGHT_FORMATS = {"int4": 0, "mxfp4": 1}
_wfmt = 0


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_lib/liboracle.so (gcc, host arch neutral)."""
    os.makedirs(_LIBDIR, exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-fPIC",
           "-shared", "-pthread", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, i32, f32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_void_p
        lib.oracle_set_mutation.argtypes = [i32]
        lib.oracle_get_mutation.restype = i32
        lib.oracle_set_threads.argtypes = [i32]
        lib.oracle_num_threads.restype = i32
        lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f32.restype = f32
        lib.oracle_f32_to_bf16.argtypes = [f32]
        lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
        lib.oracle_silu.argtypes = [f32]
        lib.oracle_silu.restype = f32
        lib.oracle_code.argtypes = [vp, i64, i64, i64]
        lib.oracle_code.restype = i32
        lib.oracle_dequant_one.argtypes = [vp, vp, i64, i64, i64]
        lib.oracle_dequant_one.restype = f32
        lib.oracle_dequant.argtypes = [vp, vp, i64, i64, vp]
        lib.oracle_align_capacity.argtypes = [i64, i64, i64, i64]
        lib.oracle_align_capacity.restype = i64
        lib.oracle_moe_align.argtypes = [vp, i64, i64, i64, vp, i64, i64, vp, vp, vp, i64]
        lib.oracle_moe_align.restype = i32
        lib.oracle_route_topk.argtypes = [vp, i64, i64, i64, i32, vp, vp]
        lib.oracle_prepack.argtypes = [i32, vp, vp, i64, i64, i64, vp]
        lib.oracle_prepack.restype = i32
        lib.oracle_set_weight_format.argtypes = [i32]
        lib.oracle_get_weight_format.restype = i32
        lib.oracle_e2m1.argtypes = [i32]
        lib.oracle_e2m1.restype = ctypes.c_double
        lib.oracle_e8m0.argtypes = [i32]
        lib.oracle_e8m0.restype = ctypes.c_double
        lib.oracle_route_topk.restype = i32
        lib.oracle_expert_mlp.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, vp, vp, vp, vp, vp]
        lib.oracle_expert_mlp.restype = i32
        lib.oracle_moe_indexed.argtypes = [vp, i64, i64, i64, i64, i64, vp, vp, vp, vp, vp,
                                           vp, vp, vp, i64, i64, vp, vp, vp, vp, vp]
        lib.oracle_moe_indexed.restype = i32
        lib.oracle_moe_indexed_down.argtypes = [vp, i64, i64, i64, i64, i64, vp, vp, vp, vp, vp,
                                                vp, i64, i64, vp]
        lib.oracle_moe_indexed_down.restype = i32
        lib.oracle_moe_grouped_down.argtypes = [i32, vp, i64, i64, i64, i64, vp, vp, i64, vp, vp,
                                                vp, vp, i64, i64, vp, vp]
        lib.oracle_moe_grouped_down.restype = i32
        lib.oracle_moe_grouped.argtypes = [i32, vp, i64, i64, i64, i64, vp, vp, i64, vp, vp,
                                           vp, vp, vp, vp, i64, i64, vp, vp, vp, vp]
        lib.oracle_moe_grouped.restype = i32
        _lib = lib
        return lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


class mutation:
    """Context manager planting one mistake in the oracle (tests only)."""

    def __init__(self, name: str):
        self.code = MUTATIONS[name]

    def __enter__(self):
        _load().oracle_set_mutation(self.code)
        return self

    def __exit__(self, *exc):
        _load().oracle_set_mutation(0)
        return False


class weight_format:
    """Context manager: the weight format the oracle reads.  "int4" (the
    default): codes q with bf16 scales, w = (q - 8) * s.  "mxfp4": E2M1 codes
    with one E8M0 scale byte per 32 input channels (uint8 [E, N, K/32] in
    place of the bf16 scales), w = e2m1(q) * 2^(s - 127) (oracle.c, header)."""

    def __init__(self, name: str):
        self.code = WEIGHT_FORMATS[name]

    def __enter__(self):
        global _wfmt
        self.prev = _wfmt
        _wfmt = self.code
        _load().oracle_set_weight_format(self.code)
        return self

    def __exit__(self, *exc):
        global _wfmt
        _wfmt = self.prev
        _load().oracle_set_weight_format(self.prev)
        return False


def _s(a):
    """Scales as the current weight format stores them."""
    return _c(a, np.uint8 if _wfmt == 1 else np.uint16)


def e2m1(q: int) -> float:
    return float(_load().oracle_e2m1(int(q)))


def e8m0(s: int) -> float:
    return float(_load().oracle_e8m0(int(s)))


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (a view, no arithmetic)."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(v: float) -> int:
    return int(_load().oracle_f32_to_bf16(float(v)))


def silu(v: float) -> float:
    return float(_load().oracle_silu(float(v)))


def code(wq: np.ndarray, K: int, n: int, c: int) -> int:
    wq = _c(wq, np.int32)
    return int(_load().oracle_code(_p(wq), K, n, c))


def dequant(wq: np.ndarray, ws: np.ndarray, N: int, K: int) -> np.ndarray:
    """Dequantised [N, K] weight as float32 (every value a bf16 value)."""
    wq = _c(wq, np.int32)
    ws = _s(ws)
    assert wq.size == N * K // 8 and ws.size == N * K // 32
    out = np.empty((N, K), dtype=np.float32)
    _load().oracle_dequant(_p(wq), _p(ws), N, K, _p(out))
    return out


def align_capacity(T: int, k: int, E_local: int, block_m: int) -> int:
    return int(_load().oracle_align_capacity(T, k, E_local, block_m))


def moe_align(topk_ids, E_global, expert_map, E_local, block_m, capacity=None):
    """Returns (sorted_ids [cap], expert_ids [cap/block_m], num_tokens_padded int)."""
    ids = _c(topk_ids, np.int32)
    T, k = ids.shape
    if capacity is None:
        capacity = align_capacity(T, k, E_local, block_m)
    emap = _c(expert_map, np.int32)
    sorted_ids = np.empty(capacity, dtype=np.int32)
    expert_ids = np.empty(capacity // block_m, dtype=np.int32)
    ntp = np.zeros(1, dtype=np.int32)
    rc = _load().oracle_moe_align(_p(ids), T, k, E_global, _p(emap), E_local, block_m,
                                  _p(sorted_ids), _p(expert_ids), _p(ntp), capacity)
    if rc != 0:
        raise ValueError("oracle_moe_align: capacity too small or bad block_m")
    return sorted_ids, expert_ids, int(ntp[0])


def route_topk(logits, k, renormalize=True):
    """Router (oracle.c R14): logits float32 [T, E] -> (topk_ids int32 [T, k],
    topk_weights float32 [T, k])."""
    lg = _c(logits, np.float32)
    T, E = lg.shape
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float32)
    if _load().oracle_route_topk(_p(lg), T, E, k, 1 if renormalize else 0, _p(ids), _p(w)) != 0:
        raise ValueError("oracle_route_topk: bad sizes")
    return ids, w


def prepack(kind, w_q, w_s):
    """Storage order of chord_w4a16_prepack (oracle.c, prepack): kind 1
    (gate/up) or 2 (down), codes int32 [E, N, K/8] and scale bits uint16
    [E, N, K/32] -> the packed bytes (uint8)."""
    if _wfmt != 0:
        raise ValueError("prepack is defined for the INT4 format")
    q = _c(w_q, np.int32)
    sc = _c(w_s, np.uint16)
    E, N, K8 = q.shape
    K = K8 * 8
    out = np.empty(256 + E * (N // 128) * ((K + 255) // 256) * 18432, dtype=np.uint8)
    if _load().oracle_prepack(int(kind), _p(q), _p(sc), E, N, K, _p(out)) != 0:
        raise ValueError("oracle_prepack: bad kind or sizes")
    return out


def expert_mlp(w13_q, w13_s, w2_q, w2_s, e, x_rows):
    """One expert's MLP on explicit bf16 rows [n, H]: returns (g, u, h_bits, y)."""
    x_rows = _c(x_rows, np.uint16)
    n, H = x_rows.shape
    I = w2_q.shape[2] * 8
    w13_q, w13_s, w2_q, w2_s = (_c(w13_q, np.int32), _s(w13_s),
                                _c(w2_q, np.int32), _s(w2_s))
    g = np.empty((n, I), np.float32)
    u = np.empty((n, I), np.float32)
    h = np.empty((n, I), np.uint16)
    y = np.empty((n, H), np.float32)
    rc = _load().oracle_expert_mlp(_p(w13_q), _p(w13_s), _p(w2_q), _p(w2_s), e, H, I, n,
                                   _p(x_rows), _p(g), _p(u), _p(h), _p(y))
    if rc != 0:
        raise MemoryError("oracle_expert_mlp")
    return g, u, h, y


def moe_indexed(x, w13_q, w13_s, w2_q, w2_s, topk_weights, sorted_ids, expert_ids, ntp,
                block_m, k, want_h=False, want_y=False, want_gu=False):
    """Whole layer on the indexed layout.  Returns out bits [T, H] (and h, y,
    and the pre-rounding gate/up values g, u [capacity, I] when asked)."""
    x = _c(x, np.uint16)
    T, H = x.shape
    E = w13_q.shape[0]
    I = w2_q.shape[2] * 8
    w13_q, w13_s, w2_q, w2_s = (_c(w13_q, np.int32), _s(w13_s),
                                _c(w2_q, np.int32), _s(w2_s))
    tw = _c(topk_weights, np.float32)
    sorted_ids = _c(sorted_ids, np.int32)
    expert_ids = _c(expert_ids, np.int32)
    cap = sorted_ids.size
    ntp_a = np.array([ntp], dtype=np.int32)
    out = np.empty((T, H), np.uint16)
    h = np.empty((cap, I), np.uint16) if want_h else None
    y = np.empty((T * k, H), np.float32) if want_y else None
    g = np.empty((cap, I), np.float32) if want_gu else None
    u = np.empty((cap, I), np.float32) if want_gu else None
    rc = _load().oracle_moe_indexed(_p(x), T, H, I, E, k, _p(w13_q), _p(w13_s), _p(w2_q),
                                    _p(w2_s), _p(tw), _p(sorted_ids), _p(expert_ids),
                                    _p(ntp_a), cap, block_m, _p(out), _p(h), _p(y), _p(g), _p(u))
    if rc != 0:
        raise ValueError("oracle_moe_indexed failed")
    if want_gu:
        return out, h, y, g, u
    if want_h or want_y:
        return out, h, y
    return out


def moe_indexed_down(h_rows, w2_q, w2_s, topk_weights, sorted_ids, expert_ids, ntp, block_m,
                     T, k):
    """Down GEMM + combine of the indexed layer on given bf16 rows h_rows
    [capacity, I].  Returns out bits [T, H]."""
    h_rows = _c(h_rows, np.uint16)
    E, H = w2_q.shape[0], w2_q.shape[1]
    I = w2_q.shape[2] * 8
    w2_q, w2_s = _c(w2_q, np.int32), _s(w2_s)
    tw = _c(topk_weights, np.float32)
    sorted_ids = _c(sorted_ids, np.int32)
    expert_ids = _c(expert_ids, np.int32)
    ntp_a = np.array([ntp], dtype=np.int32)
    out = np.empty((T, H), np.uint16)
    rc = _load().oracle_moe_indexed_down(_p(h_rows), T, H, I, E, k, _p(w2_q), _p(w2_s), _p(tw),
                                         _p(sorted_ids), _p(expert_ids), _p(ntp_a),
                                         sorted_ids.size, block_m, _p(out))
    if rc != 0:
        raise ValueError("oracle_moe_indexed_down failed")
    return out


def moe_grouped_down(mode, h_rows, w2_q, w2_s, m_indices=None, masked_m=None, max_m=0,
                     row_to_pair=None, topk_weights=None, T=0, k=0):
    """Down GEMM + outputs of the grouped layer on given rows h_rows [M, I]."""
    m = {"contiguous": 0, "masked": 1}[mode]
    h_rows = _c(h_rows, np.uint16)
    M, I = h_rows.shape
    E, H = w2_q.shape[0], w2_q.shape[1]
    w2_q, w2_s = _c(w2_q, np.int32), _s(w2_s)
    mi, mm = _c(m_indices, np.int32), _c(masked_m, np.int32)
    r2p, tw = _c(row_to_pair, np.int32), _c(topk_weights, np.float32)
    out_rows = np.empty((M, H), np.uint16)
    out_tok = np.empty((T, H), np.uint16) if r2p is not None else None
    rc = _load().oracle_moe_grouped_down(m, _p(h_rows), M, H, I, E, _p(mi), _p(mm), max_m,
                                         _p(w2_q), _p(w2_s), _p(r2p), _p(tw), T, k,
                                         _p(out_rows), _p(out_tok))
    if rc != 0:
        raise ValueError("oracle_moe_grouped_down failed")
    return (out_rows, out_tok) if out_tok is not None else out_rows


def moe_grouped(mode, a, w13_q, w13_s, w2_q, w2_s, m_indices=None, masked_m=None,
                row_to_pair=None, topk_weights=None, T=0, k=0, want_h=False, want_y=False):
    """Whole layer on a grouped layout (mode "contiguous" or "masked").

    contiguous: a [M, H], m_indices [M]; masked: a [E, max_m, H], masked_m [E].
    Returns out_rows bits [M, H] (+ out_tokens [T, H] when row_to_pair given,
    + h [M, I], y [M, H] when asked)."""
    m = {"contiguous": 0, "masked": 1}[mode]
    a = _c(a, np.uint16)
    E = w13_q.shape[0]
    I = w2_q.shape[2] * 8
    if m == 1:
        assert a.ndim == 3
        max_m = a.shape[1]
        a = a.reshape(-1, a.shape[2])
    else:
        max_m = 0
    M, H = a.shape
    w13_q, w13_s, w2_q, w2_s = (_c(w13_q, np.int32), _s(w13_s),
                                _c(w2_q, np.int32), _s(w2_s))
    mi = _c(m_indices, np.int32)
    mm = _c(masked_m, np.int32)
    r2p = _c(row_to_pair, np.int32)
    tw = _c(topk_weights, np.float32)
    out_rows = np.empty((M, H), np.uint16)
    out_tok = np.empty((T, H), np.uint16) if r2p is not None else None
    h = np.empty((M, I), np.uint16) if want_h else None
    y = np.empty((M, H), np.float32) if want_y else None
    rc = _load().oracle_moe_grouped(m, _p(a), M, H, I, E, _p(mi), _p(mm), max_m, _p(w13_q),
                                    _p(w13_s), _p(w2_q), _p(w2_s), _p(r2p), _p(tw), T, k,
                                    _p(out_rows), _p(out_tok), _p(h), _p(y))
    if rc != 0:
        raise ValueError("oracle_moe_grouped failed")
    res = [out_rows]
    if out_tok is not None:
        res.append(out_tok)
    if want_h:
        res.append(h)
    if want_y:
        res.append(y)
    return res[0] if len(res) == 1 else tuple(res)


def run_workload(inp, block_m=None, want_h=False, want_y=False, want_gu=False):
    """Align + indexed layer for a synth.MoEInputs draw."""
    s = inp.shape
    bm = s.block_m if block_m is None else block_m
    sorted_ids, expert_ids, ntp = moe_align(inp.topk_ids, s.E_global, inp.expert_map,
                                            s.E_local, bm)
    res = moe_indexed(inp.x, inp.w13_q, inp.w13_s, inp.w2_q, inp.w2_s, inp.topk_weights,
                      sorted_ids, expert_ids, ntp, bm, s.k, want_h=want_h, want_y=want_y,
                      want_gu=want_gu)
    return (sorted_ids, expert_ids, ntp), res
