"""chord_moe_align_noalloc: the routing alignment for callers that cannot
allocate device memory or pass a workspace (allocator callbacks, plugins whose
host owns every buffer).  Called through the C ABI and compared, bit for bit,
with the oracle's align and with chord_moe_align, the entry point that takes a
workspace: the outputs are integers, so they must match exactly.

The draws cover both forms of the align: small routings (up to 16384 pairs and
512 local experts) run in one CTA that keeps its counts in shared memory;
larger ones run the histogram / scan / scatter kernels, whose per-tile
histogram lives in the library's fixed scratch array.  The calls are issued
back to back on one stream with different routings and read back only at the
end, so a histogram or error word carried from one call into the next would
show.  This file is collected last."""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from w4a16_int4_mixture_gb300 import synth

pytestmark = pytest.mark.gpu


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


# (workload, T, seed): the one-CTA form (up to its limit, 512 x 8 pairs), then
# the three-kernel form at four sizes (just past the limit first)
DRAWS = [("ep8-decode", None, 11), ("tp8", 128, 12), ("tp8", 513, 17),
         ("ep8-decode", 1024, 13), ("ep8-prefill", None, 14), ("tp8", 2048, 15),
         ("ep8-decode", 1024, 16)]


def test_noalloc_align_matches_oracle_and_workspace_align():
    import w4a16_int4_mixture_gb300 as chord
    chord.build()
    lib = chord.ops.lib()
    dev = torch.device("cuda:0")
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    pending = []
    for wl, T, seed in DRAWS:
        inp = synth.make_inputs(synth.workload(wl, T=T), seed=seed, weights=False)
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
            outs.append((si, ei, ntp))
        # keep the inputs alive until the stream has run every call
        pending.append((inp, cap, ids, emap, outs))
    torch.cuda.synchronize()
    for inp, cap, _, _, outs in pending:
        s = inp.shape
        r_si, r_ei, r_n = oracle.moe_align(inp.topk_ids, s.E_global, inp.expert_map, s.E_local,
                                           s.block_m, capacity=cap)
        for (si, ei, ntp), which in zip(outs, ("noalloc", "workspace")):
            assert int(ntp.item()) == r_n > 0, f"{s.name} {which}: num_tokens_padded"
            assert np.array_equal(si.cpu().numpy(), r_si), f"{s.name} {which}: sorted_ids"
            assert np.array_equal(ei.cpu().numpy(), r_ei), f"{s.name} {which}: expert_ids"


def test_noalloc_align_rejects_sizes_beyond_its_scratch():
    import w4a16_int4_mixture_gb300 as chord
    lib = chord.ops.lib()
    # 2^20 tiles of 256 pairs x 8 experts is far beyond the 4 MiB scratch array.
    # Every pointer is NULL: the size check comes first, and if it ever did not,
    # the null-pointer check would refuse the call before anything is launched.
    T, k, E = (1 << 28) // 8, 8, 8
    st = lib.chord_moe_align_noalloc(None, T, k, E, None, E, 16, None, None, None,
                                     chord.moe_align_capacity(T, k, E, 16), None)
    assert st == -2
