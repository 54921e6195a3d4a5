"""chord_moe_align_noalloc: the routing alignment for callers that cannot
allocate device memory or pass a workspace (allocator callbacks, plugins whose
host owns every buffer).  Called through the C ABI and compared with
chord_moe_align, the entry point that takes a workspace: the outputs are
integers, so they must match exactly.  Two calls in a row, with different
routings, check that the shared scratch array carries nothing from one call
into the next.  This file is collected last."""

import ctypes

import numpy as np
import pytest
import torch

from w4a16_int4_mixture_gb300 import synth

pytestmark = pytest.mark.gpu


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def test_noalloc_align_matches_workspace_align():
    import w4a16_int4_mixture_gb300 as chord
    chord.build()
    lib = chord.ops.lib()
    dev = torch.device("cuda:0")
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    draws = [(synth.workload("ep8-decode"), 11), (synth.workload("tp8", T=128), 12)]
    for shape, seed in draws:
        inp = synth.make_inputs(shape, seed=seed, weights=False)
        s = inp.shape
        ids = torch.from_numpy(inp.topk_ids).to(dev)
        emap = None if inp.expert_map is None else torch.from_numpy(inp.expert_map).to(dev)
        cap = chord.moe_align_capacity(s.T, s.k, s.E_local, s.block_m)
        outs = []
        for use_noalloc in (True, False):
            si = torch.full((cap,), -7, dtype=torch.int32, device=dev)
            ei = torch.full((cap // s.block_m,), -7, dtype=torch.int32, device=dev)
            ntp = torch.full((1,), -7, dtype=torch.int32, device=dev)
            if use_noalloc:
                st = lib.chord_moe_align_noalloc(_ptr(ids), s.T, s.k, s.E_global, _ptr(emap),
                                                 s.E_local, s.block_m, _ptr(si), _ptr(ei),
                                                 _ptr(ntp), cap, stream)
            else:
                ws = torch.empty(chord.ops.align_workspace_size(s.T, s.k, s.E_local),
                                 dtype=torch.uint8, device=dev)
                st = lib.chord_moe_align(_ptr(ids), s.T, s.k, s.E_global, _ptr(emap), s.E_local,
                                         s.block_m, _ptr(si), _ptr(ei), _ptr(ntp), cap, _ptr(ws),
                                         ws.numel(), stream)
            assert st == 0, f"status {st}"
            torch.cuda.synchronize()
            outs.append((si.cpu().numpy(), ei.cpu().numpy(), int(ntp.item())))
        (a_si, a_ei, a_n), (b_si, b_ei, b_n) = outs
        assert a_n == b_n and a_n > 0
        assert np.array_equal(a_si, b_si)
        assert np.array_equal(a_ei, b_ei)


def test_noalloc_align_rejects_sizes_beyond_its_scratch():
    import w4a16_int4_mixture_gb300 as chord
    lib = chord.ops.lib()
    fake = ctypes.c_void_p(0x1000)
    # 2^20 tiles of 256 pairs x 8 experts is far beyond the 4 MiB scratch array
    T, k, E = (1 << 28) // 8, 8, 8
    st = lib.chord_moe_align_noalloc(fake, T, k, E, None, E, 16, fake, fake, fake,
                                     chord.moe_align_capacity(T, k, E, 16), None)
    assert st == -2
