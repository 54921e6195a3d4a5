"""ctypes binding of the C ABI in include/chord.h (argument marshalling only).

Every function here passes device pointers, sizes and the current torch CUDA
stream to the CUDA library; all arithmetic of the path runs in its kernels.
The library must have been built (w4a16_int4_mixture_gb300.build); when it is
missing this module raises instead of falling back to anything else.
"""

from __future__ import annotations

import ctypes
import os
import threading

from . import _build

_lock = threading.Lock()
_lib = None

CHORD_OK = 0
STATUS = {
    0: "ok", -1: "invalid argument", -2: "unsupported shape", -3: "routing capacity too small",
    -4: "layout mode mismatch", -5: "CUDA error", -6: "device wait timed out",
    -7: "invalid routing data", -8: "workspace missing, misaligned or too small",
    -9: "no sm_103a device current",
    -10: "scale outside the supported range",
    -11: "packed weights do not match the call",
}
GROUPED_CONTIGUOUS = 0
GROUPED_MASKED = 1
FLAG_VALIDATE = 1
FLAG_DETERMINISTIC = 2
FLAG_TEST_SKIP_ARRIVE = 4
FLAG_NO_SPLIT_K = 8
FLAG_PREPACKED = 16
FLAG_MXFP4 = 32
PACK_GATE_UP = 1
PACK_DOWN = 2
DEVERR_TIMEOUT = 1
DEVERR_ROUTING = 2
DEVERR_CAPACITY = 4
DEVERR_SCALE_RANGE = 8
DEVERR_PACKED = 16

# every symbol include/chord.h declares, with (restype, argtypes)
_i64, _int, _sz, _vp, _cp = ctypes.c_int64, ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_char_p
SIGNATURES = {
    "chord_status_string": (_cp, [_int]),
    "chord_version": (_int, []),
    "chord_moe_align_capacity": (_i64, [_i64, _int, _int, _int]),
    "chord_select_block_m": (_int, [_i64, _int, _int, _int, _int, _int]),
    "chord_describe_schedule": (_int, [_i64, _int, _int, _int, _int, _int, _int, _cp, _sz]),
    "chord_moe_align_workspace_size": (_sz, [_i64, _int, _int]),
    "chord_w4a16_moe_workspace_size": (_sz, [_i64, _int, _int, _int, _int, _int, _int, _i64, _int]),
    "chord_w4a16_grouped_workspace_size": (_sz, [_int, _i64, _int, _int, _int, _i64, _int, _int,
                                                 _int]),
    "chord_moe_align": (_int, [_vp, _i64, _int, _int, _vp, _int, _int, _vp, _vp, _vp, _i64, _vp,
                               _sz, _vp]),
    "chord_moe_align_noalloc": (_int, [_vp, _i64, _int, _int, _vp, _int, _int, _vp, _vp, _vp,
                                       _i64, _vp]),
    "chord_w4a16_prepack_size": (_sz, [_int, _int, _int, _int]),
    "chord_w4a16_prepack": (_int, [_int, _vp, _vp, _int, _int, _int, _vp, _sz, _vp]),
    "chord_mxfp4_prepack": (_int, [_int, _vp, _vp, _int, _int, _int, _vp, _sz, _vp]),
    "chord_moe_route_align": (_int, [_vp, _i64, _int, _int, _int, _vp, _int, _int, _vp, _vp, _vp,
                                     _vp, _vp, _i64, _vp, _sz, _vp]),
    "chord_w4a16_moe_indexed": (_int, [_vp, _i64, _int, _int, _int, _int, _int, _vp, _vp, _vp,
                                       _vp, _vp, _vp, _vp, _vp, _i64, _int, _vp, _sz, _vp, _vp,
                                       _int, _vp]),
    "chord_w4a16_moe_grouped": (_int, [_int, _vp, _i64, _int, _int, _int, _vp, _vp, _i64, _int,
                                       _vp, _vp, _vp, _vp, _vp, _vp, _i64, _int, _vp, _sz, _vp,
                                       _vp, _vp, _int, _vp]),
    "chord_get_device_error": (_int, [_vp, ctypes.POINTER(ctypes.c_int), _int, _vp]),
    "chord_stage_timing_enable": (_int, [_int]),
    "chord_stage_timing_read": (_int, [ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_int)]),
}


class ChordError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({status})")


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False):
    """Load the CUDA library (optionally building it first).  Raises when it
    is not built: there is no other implementation to fall back to."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if build_if_missing and _build.is_stale():
            _build.build()
        if not os.path.exists(path):
            raise RuntimeError(
                f"CUDA library {path} is not built; run "
                "`python -c 'import __graft_entry__ as g; g.build()'` on a CUDA 13 host")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def check(status: int, where: str) -> None:
    if status != CHORD_OK:
        raise ChordError(status, where)
