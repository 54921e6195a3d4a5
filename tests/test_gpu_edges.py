"""Edges of the supported shapes on the GPU, each checked against the oracle
and the fp64 anchor like the fixed cases: the largest top-k (32, also through
the ordered combine), more local
experts than the align entry point and the masked layout's row compaction take
(1024), a deep reduction (H = 4096) with a six-stage down GEMM (I = 1536), a
hidden size of 128 mod 256, and an empty batch."""

import numpy as np
import pytest
import torch

import oracle
from gpu_util import bf16_to_np, dev_tensor, weights_to
from test_gpu_layer import (DEV, Run, chord, masked_layer_check, run_indexed_full,  # noqa: F401
                            small, verify_indexed)
from w4a16_int4_mixture_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("k", [16, 32])
def test_large_top_k(chord, k):
    inp = small(24, k, 64, 40, 256, 128, 500 + k)
    verify_indexed(inp, run_indexed_full(chord, inp), label=f"top-k {k}")


@pytest.mark.parametrize("T", [24, 300, 2100])
def test_large_top_k_ordered_combine(chord, T):
    """Top-k 32 through the ordered combine (CHORD_FLAG_DETERMINISTIC): a
    token's up to 32 local slots are loaded in batches (eight slots at a time
    up to 256 tokens, two up to 2048, one beyond) and summed in ascending slot
    order, so the three block shapes of the combine each see tokens with more
    slots than one batch; two calls give the same bits."""
    inp = small(T, 32, 64, 40, 256, 128, 520 + T)
    run = run_indexed_full(chord, inp, flags=2)
    tokens = None if T <= 300 else np.sort(np.random.default_rng(T).choice(T, 64, replace=False))
    verify_indexed(inp, run, tokens, label=f"top-k 32 ordered T={T}")
    again = run_indexed_full(chord, inp, flags=2)
    assert np.array_equal(run.out.view(np.uint16), again.out.view(np.uint16)), \
        "the ordered combine must be bit-reproducible"


def test_more_local_experts_than_staged(chord):
    """1500 local experts of 3000, about one routed row each.  The align entry
    point takes at most 1024 local experts; the layer takes any number, so the
    aligned layout comes from the oracle's align here (as it would from a
    caller's own)."""
    inp = small(160, 8, 3000, 1500, 256, 128, 510)
    s = inp.shape
    si, ei, ntp = oracle.moe_align(inp.topk_ids, s.E_global, inp.expert_map, s.E_local, 16)
    x = dev_tensor(inp.x, DEV, True)
    tw = dev_tensor(inp.topk_weights, DEV)
    h = torch.empty((si.size, s.I), dtype=torch.bfloat16, device=DEV)
    out = chord.w4a16_moe_indexed(x, *weights_to(inp, DEV), tw, dev_tensor(si, DEV),
                                  dev_tensor(ei, DEV), dev_tensor(np.array([ntp], np.int32), DEV),
                                  16, s.E_global, flags=1, h_out=h)
    torch.cuda.synchronize()
    run = Run(bf16_to_np(out), bf16_to_np(h), si, ei, int(ntp), 16)
    verify_indexed(inp, run, label="1500 local experts")


def test_more_local_experts_masked(chord):
    """The masked layout with 1100 experts (above the limit of the row
    compaction, so the token boxes read each expert's region in place)."""
    inp = small(20, 2, 1100, 1100, 256, 128, 511, emap=False)
    a3, mm, r2p = synth.grouped_masked_layout(inp)
    masked_layer_check(chord, inp, a3, mm, r2p, weights_to(inp, DEV), "masked, 1100 experts")


@pytest.mark.parametrize("form", ["plain", "packed"])
def test_deep_k(chord, form):
    """H = 4096 (16 gate/up stages of 256) and I = 1536 (six down stages)."""
    inp = small(20, 2, 4, 4, 4096, 1536, 512, emap=False)
    w = weights_to(inp, DEV)
    if form == "packed":
        w = (chord.prepack_weights(*w), None, None, None)
    verify_indexed(inp, run_indexed_full(chord, inp, weights=w), label=f"deep K {form}")


@pytest.mark.parametrize("form", ["plain", "packed", "grouped"])
def test_hidden_size_128_mod_256(chord, form):
    """H = 640 (K of the gate/up GEMM a multiple of 128, not of 256): the
    gate/up GEMM runs the 128-deep stages; packs keep the last block's first
    half."""
    inp = small(48, 4, 8, 8, 640, 256, 514, emap=False)
    w = weights_to(inp, DEV)
    if form == "packed":
        w = (chord.prepack_weights(*w), None, None, None)
    if form == "grouped":
        a3, mm, r2p = synth.grouped_masked_layout(inp)
        masked_layer_check(chord, inp, a3, mm, r2p, w, "H=640 masked")
        return
    verify_indexed(inp, run_indexed_full(chord, inp, weights=w), label=f"H=640 {form}")


def test_empty_batch(chord):
    """T = 0: the call succeeds and touches nothing (the output stays as it was)."""
    s = synth.MoEShape("empty", T=0, k=4, E_global=8, E_local=8, H=256, I=128, seed=513)
    inp = synth.make_inputs(s)
    w = weights_to(inp, DEV)
    x = torch.empty((0, s.H), dtype=torch.bfloat16, device=DEV)
    ids = torch.empty((0, s.k), dtype=torch.int32, device=DEV)
    tw = torch.empty((0, s.k), dtype=torch.float32, device=DEV)
    si, ei, ntp = chord.moe_align(ids, s.E_global, s.E_local, 16)
    out = chord.w4a16_moe_indexed(x, *w, tw, si, ei, ntp, 16, s.E_global, flags=1)
    torch.cuda.synchronize()
    assert tuple(out.shape) == (0, s.H)
    assert int(ntp.item()) == 0
