"""PyTorch-facing calls of the W4A16 INT4 MoE library.

Thin wrappers over the C ABI (include/chord.h): they check dtypes / devices,
allocate outputs and workspaces with torch (PyTorch only provides device
memory and the current stream) and pass raw pointers to the CUDA library.

Layouts (page: "vLLM x Novita AI: Chord W4A16 INT4 MoE kernels for Kimi
K2.x", sections "Two kernel families", "grouped SM90 kernels", Fig. 3):
  x            bf16 [T, H]
  w13_q        int32 [E, 2I, H/8]  packed 4-bit codes, rows 0..I-1 gate, I..2I-1 up
  w13_s        bf16  [E, 2I, H/32]
  w2_q         int32 [E, H, I/8]
  w2_s         bf16  [E, H, I/32]
  topk_ids     int32 [T, k] global expert ids; topk_weights float32 [T, k]
"""

from __future__ import annotations

import ctypes
from typing import Optional

import torch

from . import _binding as B

ChordError = B.ChordError


def _p(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _req(t: torch.Tensor, name: str, dtypes, dev=None, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype} not in {dtypes}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dev is not None and t.device != dev:
        raise ValueError(f"{name} is on {t.device}, expected {dev}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() not in (ndim if isinstance(ndim, tuple) else (ndim,)):
        raise ValueError(f"{name} must have {ndim} dims")


_BF16 = (torch.bfloat16,)
_I32 = (torch.int32,)
_F32 = (torch.float32,)


class _WorkspacePool:
    """Per-device scratch buffers, grown on demand and reused across calls."""

    def __init__(self):
        self.bufs = {}

    def get(self, device: torch.device, nbytes: int, key: str) -> torch.Tensor:
        k = (device.index, key)
        b = self.bufs.get(k)
        if b is None or b.numel() < nbytes:
            b = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
            self.bufs[k] = b
        return b


_pool = _WorkspacePool()


def lib():
    return B.load()


def moe_align_capacity(T: int, k: int, E_local: int, block_m: int) -> int:
    return int(lib().chord_moe_align_capacity(T, k, E_local, block_m))


def select_block_m(T: int, k: int, E_global: int, E_local: int, H: int, I: int) -> int:
    return int(lib().chord_select_block_m(T, k, E_global, E_local, H, I))


def describe_schedule(T, k, E_global, E_local, H, I, flags=0) -> str:
    buf = ctypes.create_string_buffer(256)
    lib().chord_describe_schedule(T, k, E_global, E_local, H, I, flags, buf, 256)
    return buf.value.decode()


def align_workspace_size(T: int, k: int, E_local: int) -> int:
    return int(lib().chord_moe_align_workspace_size(T, k, E_local))


def moe_align(topk_ids: torch.Tensor, E_global: int, E_local: int, block_m: int = 16,
              expert_map: Optional[torch.Tensor] = None, capacity: Optional[int] = None,
              workspace: Optional[torch.Tensor] = None, out=None):
    """Routing -> (sorted_ids, expert_ids, num_tokens_padded), all device int32."""
    _req(topk_ids, "topk_ids", _I32, ndim=2)
    dev = topk_ids.device
    T, k = topk_ids.shape
    if expert_map is not None:
        _req(expert_map, "expert_map", _I32, dev, 1)
    if capacity is None:
        capacity = moe_align_capacity(T, k, E_local, block_m)
    if out is None:
        sorted_ids = torch.empty(capacity, dtype=torch.int32, device=dev)
        expert_ids = torch.empty(capacity // block_m, dtype=torch.int32, device=dev)
        ntp = torch.empty(1, dtype=torch.int32, device=dev)
    else:
        sorted_ids, expert_ids, ntp = out
    need = align_workspace_size(T, k, E_local)
    ws = workspace if workspace is not None else _pool.get(dev, need, "align")
    st = lib().chord_moe_align(_p(topk_ids), T, k, E_global, _p(expert_map), E_local, block_m,
                               _p(sorted_ids), _p(expert_ids), _p(ntp), capacity, _p(ws),
                               ws.numel(), _stream(dev))
    B.check(st, "chord_moe_align")
    return sorted_ids, expert_ids, ntp


def moe_route_align(logits: torch.Tensor, k: int, E_local: int, block_m: int = 16,
                    expert_map: Optional[torch.Tensor] = None, renormalize: bool = True,
                    capacity: Optional[int] = None, workspace: Optional[torch.Tensor] = None,
                    out=None):
    """Router logits float32 [T, E_global] -> (topk_ids, topk_weights, sorted_ids,
    expert_ids, num_tokens_padded): the k largest logits per token (ties to the
    lower id), softmax weights (renormalised over the k), and their aligned layout."""
    _req(logits, "logits", _F32, ndim=2)
    dev = logits.device
    T, E_global = logits.shape
    if expert_map is not None:
        _req(expert_map, "expert_map", _I32, dev, 1)
    if capacity is None:
        capacity = moe_align_capacity(T, k, E_local, block_m)
    if out is None:
        topk_ids = torch.empty((T, k), dtype=torch.int32, device=dev)
        topk_weights = torch.empty((T, k), dtype=torch.float32, device=dev)
        sorted_ids = torch.empty(capacity, dtype=torch.int32, device=dev)
        expert_ids = torch.empty(capacity // block_m, dtype=torch.int32, device=dev)
        ntp = torch.empty(1, dtype=torch.int32, device=dev)
    else:
        topk_ids, topk_weights, sorted_ids, expert_ids, ntp = out
    need = align_workspace_size(T, k, E_local)
    ws = workspace if workspace is not None else _pool.get(dev, need, "align")
    st = lib().chord_moe_route_align(_p(logits), T, E_global, k, 1 if renormalize else 0,
                                     _p(expert_map), E_local, block_m, _p(topk_ids),
                                     _p(topk_weights), _p(sorted_ids), _p(expert_ids), _p(ntp),
                                     capacity, _p(ws), ws.numel(), _stream(dev))
    B.check(st, "chord_moe_route_align")
    return topk_ids, topk_weights, sorted_ids, expert_ids, ntp


class PackedWeights:
    """One layer's weights after chord_w4a16_prepack (fmt "int4") or
    chord_mxfp4_prepack (fmt "mxfp4"): w13 (kind GATE_UP) and w2 (kind DOWN)
    as uint8 device buffers, with the sizes they were packed for.  Pass it as
    w13_q (with w13_s, w2_q, w2_s None) to the layer calls."""

    def __init__(self, w13: torch.Tensor, w2: torch.Tensor, E: int, H: int, I: int,
                 fmt: str = "int4"):
        if fmt not in ("int4", "mxfp4"):
            raise ValueError(f"unknown weight format {fmt!r}")
        self.w13, self.w2, self.E, self.H, self.I, self.fmt = w13, w2, E, H, I, fmt


def prepack_size(kind: int, E: int, N: int, K: int) -> int:
    return int(lib().chord_w4a16_prepack_size(kind, E, N, K))


def prepack(w_q: torch.Tensor, w_s: torch.Tensor, kind: int, out=None) -> torch.Tensor:
    """One GEMM's codes [E, N, K/8] and scales [E, N, K/32] -> the packed
    uint8 buffer (include/chord.h): bf16 scales give an INT4 pack
    (chord_w4a16_prepack), uint8 E8M0 scale bytes an MXFP4 pack
    (chord_mxfp4_prepack)."""
    _req(w_q, "w_q", _I32, ndim=3)
    dev = w_q.device
    _req(w_s, "w_s", _BF16 + (torch.uint8,), dev, 3)
    mx = w_s.dtype == torch.uint8
    E, N, K8 = w_q.shape
    K = K8 * 8
    if tuple(w_s.shape) != (E, N, K // 32):
        raise ValueError("scales must be [E, N, K/32]")
    need = prepack_size(kind, E, N, K)
    if need == 0:
        B.check(-2, "chord_w4a16_prepack_size")
    if out is None:
        out = torch.empty(need, dtype=torch.uint8, device=dev)
    else:
        _req(out, "out", (torch.uint8,), dev, 1)
    fn = lib().chord_mxfp4_prepack if mx else lib().chord_w4a16_prepack
    st = fn(kind, _p(w_q), _p(w_s), E, N, K, _p(out), out.numel(), _stream(dev))
    B.check(st, "chord_mxfp4_prepack" if mx else "chord_w4a16_prepack")
    return out


def prepack_weights(w13_q, w13_s, w2_q, w2_s) -> PackedWeights:
    """Both GEMMs of a layer -> PackedWeights.  bf16 scales: INT4 weights;
    uint8 scales (E8M0 bytes): MXFP4 weights, whose codes are E2M1 numbers."""
    mx = w13_s.dtype == torch.uint8
    E, H, I = _check_weights(w13_q, w13_s, w2_q, w2_s, w13_q.device, mx)
    return PackedWeights(prepack(w13_q, w13_s, B.PACK_GATE_UP), prepack(w2_q, w2_s, B.PACK_DOWN),
                         E, H, I, "mxfp4" if mx else "int4")


def _weights(w13_q, w13_s, w2_q, w2_s, dev):
    """-> (E, H, I, four pointers, extra flags) for plain or prepacked weights."""
    if isinstance(w13_q, PackedWeights):
        if w13_s is not None or w2_q is not None or w2_s is not None:
            raise ValueError("with PackedWeights, w13_s, w2_q and w2_s must be None")
        pw = w13_q
        need = (prepack_size(B.PACK_GATE_UP, pw.E, 2 * pw.I, pw.H),
                prepack_size(B.PACK_DOWN, pw.E, pw.H, pw.I))
        for n, t, nb in (("packed w13", pw.w13, need[0]), ("packed w2", pw.w2, need[1])):
            _req(t, n, (torch.uint8,), dev, 1)
            # (the device checks the header; a short buffer would be read past its end)
            if t.numel() < nb:
                raise ValueError(f"{n}: {t.numel()} bytes, a pack of these sizes has {nb}")
        flags = B.FLAG_PREPACKED | (B.FLAG_MXFP4 if pw.fmt == "mxfp4" else 0)
        return pw.E, pw.H, pw.I, (_p(pw.w13), None, _p(pw.w2), None), flags
    if w13_s is not None and w13_s.dtype == torch.uint8:
        raise ValueError("MXFP4 weights are used through their packs: prepack_weights() first")
    E, H, I = _check_weights(w13_q, w13_s, w2_q, w2_s, dev)
    return E, H, I, (_p(w13_q), _p(w13_s), _p(w2_q), _p(w2_s)), 0


def _check_weights(w13_q, w13_s, w2_q, w2_s, dev, mx=False):
    sdt = (torch.uint8,) if mx else _BF16
    _req(w13_q, "w13_q", _I32, dev, 3)
    _req(w13_s, "w13_s", sdt, dev, 3)
    _req(w2_q, "w2_q", _I32, dev, 3)
    _req(w2_s, "w2_s", sdt, dev, 3)
    E, N13, H8 = w13_q.shape
    H = H8 * 8
    I = N13 // 2
    if w13_s.shape != (E, 2 * I, H // 32) or w2_q.shape != (E, H, I // 8) or \
            w2_s.shape != (E, H, I // 32):
        raise ValueError("weight shapes are not [E,2I,H/8], [E,2I,H/32], [E,H,I/8], [E,H,I/32]")
    return E, H, I


def moe_workspace_size(T, k, E_global, E_local, H, I, block_m, capacity, flags=0) -> int:
    return int(lib().chord_w4a16_moe_workspace_size(T, k, E_global, E_local, H, I, block_m,
                                                    capacity, flags))


def w4a16_moe_indexed(x, w13_q, w13_s, w2_q, w2_s, topk_weights, sorted_ids, expert_ids,
                      num_tokens_padded, block_m: int, E_global: int, out=None, workspace=None,
                      flags: int = 0, h_out=None):
    """The MoE layer on the moe_align layout; returns out bf16 [T, H].
    h_out (bf16 [capacity, I]) optionally receives the gate/up output."""
    _req(x, "x", _BF16, ndim=2)
    dev = x.device
    E, H, I, wp, wflag = _weights(w13_q, w13_s, w2_q, w2_s, dev)
    flags |= wflag
    T = x.shape[0]
    if x.shape[1] != H:
        raise ValueError("x and weights disagree on H")
    _req(topk_weights, "topk_weights", _F32, dev, 2)
    k = topk_weights.shape[1]
    for n, t in (("sorted_ids", sorted_ids), ("expert_ids", expert_ids),
                 ("num_tokens_padded", num_tokens_padded)):
        _req(t, n, _I32, dev, 1)
    capacity = sorted_ids.numel()
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    else:
        _req(out, "out", _BF16, dev, 2)
    if h_out is not None:
        _req(h_out, "h_out", _BF16, dev, 2)
        if tuple(h_out.shape) != (capacity, I):
            raise ValueError("h_out must be [capacity, I]")
    need = moe_workspace_size(T, k, E_global, E, H, I, block_m, capacity, flags)
    ws = workspace if workspace is not None else _pool.get(dev, need, "layer")
    st = lib().chord_w4a16_moe_indexed(_p(x), T, H, I, E_global, E, k, *wp, _p(topk_weights),
                                       _p(sorted_ids),
                                       _p(expert_ids), _p(num_tokens_padded), capacity, block_m,
                                       _p(ws), ws.numel(), _p(out), _p(h_out), flags,
                                       _stream(dev))
    B.check(st, "chord_w4a16_moe_indexed")
    return out


def grouped_workspace_size(mode, M, H, I, E_local, T=0, k=0, with_tokens=False, expected_m=1):
    return int(lib().chord_w4a16_grouped_workspace_size(mode, M, H, I, E_local, T, k,
                                                        int(with_tokens), expected_m))


def w4a16_moe_grouped(mode: str, a, w13_q, w13_s, w2_q, w2_s, m_indices=None, masked_m=None,
                      expected_m: Optional[int] = None, row_to_pair=None, topk_weights=None,
                      T: int = 0, out_rows=None, out_tokens=None, workspace=None, flags: int = 0,
                      h_out=None):
    """The MoE layer on a grouped layout.

    mode "contiguous": a [M, H] bf16, m_indices int32 [M] (-1 on padding).
    mode "masked":     a [E, max_m, H] bf16, masked_m int32 [E], expected_m int.
    Returns out_rows [M, H] (and out_tokens [T, H] when row_to_pair /
    topk_weights are given)."""
    dev = a.device
    E, H, I, wp, wflag = _weights(w13_q, w13_s, w2_q, w2_s, dev)
    flags |= wflag
    if mode == "contiguous":
        _req(a, "a", _BF16, dev, 2)
        _req(m_indices, "m_indices", _I32, dev, 1)
        M = a.shape[0]
        max_m = 0
        mcode = B.GROUPED_CONTIGUOUS
        exp_m = expected_m or max(1, M // max(E, 1))
    elif mode == "masked":
        _req(a, "a", _BF16, dev, 3)
        _req(masked_m, "masked_m", _I32, dev, 1)
        if expected_m is None or expected_m < 1:
            raise ValueError("masked mode needs a positive expected_m")
        max_m = a.shape[1]
        M = a.shape[0] * max_m
        mcode = B.GROUPED_MASKED
        exp_m = int(expected_m)
    else:
        raise ValueError(f"unknown grouped mode {mode!r}")
    with_tokens = row_to_pair is not None
    k = 0
    if with_tokens:
        _req(row_to_pair, "row_to_pair", _I32, dev, 1)
        _req(topk_weights, "topk_weights", _F32, dev, 2)
        k = topk_weights.shape[1]
        T = topk_weights.shape[0]
        if out_tokens is None:
            out_tokens = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    if out_rows is None:
        out_rows = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
    if h_out is not None:
        _req(h_out, "h_out", _BF16, dev, 2)
        if tuple(h_out.shape) != (M, I):
            raise ValueError("h_out must be [M, I]")
    need = grouped_workspace_size(mcode, M, H, I, E, T, k, with_tokens, exp_m)
    ws = workspace if workspace is not None else _pool.get(dev, need, "grouped")
    st = lib().chord_w4a16_moe_grouped(mcode, _p(a), M, H, I, E, _p(m_indices), _p(masked_m),
                                       max_m, exp_m, *wp,
                                       _p(row_to_pair), _p(topk_weights), T, k, _p(ws),
                                       ws.numel(), _p(out_rows), _p(out_tokens), _p(h_out),
                                       flags, _stream(dev))
    B.check(st, "chord_w4a16_moe_grouped")
    return (out_rows, out_tokens) if with_tokens else out_rows


def w4a16_moe(x, topk_ids, topk_weights, w13_q, w13_s, w2_q, w2_s, E_global: int,
              expert_map=None, block_m: Optional[int] = None, flags: int = 0, out=None):
    """Align + indexed layer in one call (both graph-capturable).  The routing
    layout goes into per-device buffers reused from call to call (like the
    workspaces), so a call allocates nothing once the buffers are large
    enough; calls on different streams of one device share them and must not
    overlap."""
    E, H, I, _, _ = _weights(w13_q, w13_s, w2_q, w2_s, x.device)
    T, k = topk_ids.shape
    bm = block_m or select_block_m(T, k, E_global, E, H, I)
    cap = moe_align_capacity(T, k, E, bm)
    nblk = cap // bm
    nb = 4 * (cap + nblk + 1)
    buf = _pool.get(x.device, nb, "routing")[:nb].view(torch.int32)
    si, ei, ntp = buf[:cap], buf[cap:cap + nblk], buf[cap + nblk:cap + nblk + 1]
    moe_align(topk_ids, E_global, E, bm, expert_map=expert_map, capacity=cap, out=(si, ei, ntp))
    return w4a16_moe_indexed(x, w13_q, w13_s, w2_q, w2_s, topk_weights, si, ei, ntp, bm,
                             E_global, out=out, flags=flags)


def get_device_error(workspace: torch.Tensor, clear: bool = False) -> int:
    """Synchronise and read the device error word of a workspace."""
    bits = ctypes.c_int(0)
    lib().chord_get_device_error(_p(workspace), ctypes.byref(bits), int(clear),
                                 _stream(workspace.device))
    return bits.value


def stage_timing_enable(on: bool = True) -> None:
    B.check(lib().chord_stage_timing_enable(int(on)), "chord_stage_timing_enable")


def stage_timing_read():
    """Summed ms per stage (prepare, gate_up, down, combine) and the call count."""
    ms = (ctypes.c_float * 4)()
    n = ctypes.c_int(0)
    B.check(lib().chord_stage_timing_read(ms, ctypes.byref(n)), "chord_stage_timing_read")
    return [float(v) for v in ms], n.value
