"""Prepacked weights (chord_w4a16_prepack) on the GPU.

The pack is a byte rearrangement: the GPU's pack must equal the oracle's
(oracle.prepack, written loop by loop from the format in chord.h) byte for
byte, header and scale-range flag included.  The layer on packed weights
does the same arithmetic in the same order as on the plain weights, so with
the ordered combine its outputs are bit-identical to the plain run; they are
also checked against the oracle like every layer test.  A pack that does not
match the call makes the GEMMs compute nothing and report
CHORD_ERR_PACKED (no fault, no wait)."""

import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close_bf16, dev_tensor, weights_to
from test_gpu_layer import (DEV, chord, contiguous_layer_check, masked_layer_check,  # noqa: F401
                            run_indexed_full, small, verify_indexed)
from w4a16_int4_mixture_gb300 import synth

pytestmark = pytest.mark.gpu
ORDERED = 2
ERR_PACKED = -11
ERR_SCALE_RANGE = -10


def _packed(chord, inp):
    w = weights_to(inp, DEV)
    return chord.prepack_weights(*w), w


# (K = 384 and 128: K % 256 == 128, the last block's second half is zeros)
@pytest.mark.parametrize("kind,E,N,K", [(1, 3, 256, 512), (2, 2, 384, 768), (1, 1, 128, 256),
                                        (2, 5, 128, 2048), (2, 3, 256, 384), (1, 2, 256, 128)])
def test_prepack_matches_oracle(chord, kind, E, N, K):
    rng = np.random.default_rng(E * 1000 + N + K + kind)
    w_q = rng.integers(0, 2**32, size=(E, N, K // 8), dtype=np.uint32).view(np.int32)
    w_s = synth.scales(rng, E, N, K)
    if kind == 2:
        w_s[E - 1, N - 1, 3] = 162 << 7  # one scale past 2^35: the flag bit
    got = chord.prepack(dev_tensor(w_q, DEV), dev_tensor(w_s, DEV, True), kind)
    torch.cuda.synchronize()
    ref = oracle.prepack(kind, w_q, w_s)
    g = got.cpu().numpy()
    assert g.size == ref.size == chord.prepack_size(kind, E, N, K)
    assert np.array_equal(g[:256], ref[:256]), f"header {g[:32].view(np.uint32)}"
    bad = np.nonzero(g != ref)[0]
    assert bad.size == 0, f"{bad.size} bytes differ, first at {bad[:8]}"


# (T, k, E_global, E_local, H, I, seed): decode tiles (K stages of 256), a
# prefill-sized expert (the 192-token tile, K stages of 128: half blocks) and
# a K-split last round
CASES = {
    "decode-map": (40, 3, 10, 6, 512, 256, 71),
    "prefill-tile": (700, 2, 3, 3, 256, 256, 72),
    "split-k": (3, 8, 16, 16, 2048, 256, 73),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_layer_on_packed_weights(chord, name):
    T, k, Eg, El, H, I, seed = CASES[name]
    inp = small(T, k, Eg, El, H, I, seed, emap=El < Eg)
    pw, w = _packed(chord, inp)
    a = run_indexed_full(chord, inp, flags=ORDERED, weights=(pw, None, None, None))
    verify_indexed(inp, a, label=f"packed {name}")
    b = run_indexed_full(chord, inp, flags=ORDERED, weights=w)
    assert np.array_equal(a.h[:a.ntp], b.h[:b.ntp]), "packed h differs from the plain run"
    assert np.array_equal(a.out, b.out), "packed output differs from the plain run"
    c = run_indexed_full(chord, inp, weights=(pw, None, None, None))  # fp32 reductions
    verify_indexed(inp, c, label=f"packed {name} reduce")


def test_full_decode_workload_packed(chord):
    s = synth.workload("ep8-decode", T=128)
    inp = synth.make_inputs(s)
    pw, w = _packed(chord, inp)
    a = run_indexed_full(chord, inp, flags=ORDERED, weights=(pw, None, None, None))
    b = run_indexed_full(chord, inp, flags=ORDERED, weights=w)
    assert np.array_equal(a.out, b.out)
    tokens = np.random.default_rng(5).choice(s.T, 24, replace=False)
    verify_indexed(inp, a, tokens, label="EP8 decode T=128 packed (24 sampled tokens)")


def test_grouped_on_packed_weights(chord):
    inp = small(48, 2, 4, 4, 512, 256, 74, emap=False)
    pw, w = _packed(chord, inp)
    rows_p, tok_p = contiguous_layer_check(chord, inp, 16, "contiguous packed",
                                           weights=(pw, None, None, None))
    rows_u, tok_u = contiguous_layer_check(chord, inp, 16, "contiguous plain", weights=w)
    assert_close_bf16(rows_p, rows_u, "contiguous rows: packed vs plain")
    a3, mm, r2p = synth.grouped_masked_layout(inp)
    masked_layer_check(chord, inp, a3, mm, r2p, (pw, None, None, None), "masked packed")


def _status(chord, fn):
    try:
        fn()
    except chord.ChordError as e:
        return e.status
    return 0


def test_mismatched_pack_is_reported(chord):
    inp = small(20, 2, 4, 4, 256, 256, 75, emap=False)
    pw, w = _packed(chord, inp)
    # the gate/up pack given as the down pack (and the reverse): kinds differ.
    # Each goes into a buffer of the size its slot needs, so the host's size
    # check passes and the device's header check decides.
    a = torch.zeros(pw.w13.numel(), dtype=torch.uint8, device=DEV)
    a[:pw.w2.numel()] = pw.w2
    b = pw.w13[:pw.w2.numel()].clone()
    swapped = chord.PackedWeights(a, b, pw.E, pw.H, pw.I)
    st = _status(chord, lambda: run_indexed_full(chord, inp, weights=(swapped, None, None, None)))
    assert st == ERR_PACKED
    # a pack of fewer experts than the call reads, in a buffer of the full size
    # (so that only the header tells)
    inp2 = small(20, 2, 4, 4, 256, 256, 76, emap=False)
    w2 = weights_to(inp2, DEV)
    full = torch.empty_like(pw.w13)
    chord.prepack(w2[0][:2].contiguous(), w2[1][:2].contiguous(), 1, out=full)
    short = chord.PackedWeights(full, pw.w2, pw.E, pw.H, pw.I)
    st = _status(chord, lambda: run_indexed_full(chord, inp, weights=(short, None, None, None)))
    assert st == ERR_PACKED
    # a buffer shorter than a pack of the call's sizes is refused on the host
    cut = chord.PackedWeights(pw.w13[:-16], pw.w2, pw.E, pw.H, pw.I)
    with pytest.raises(ValueError):
        run_indexed_full(chord, inp, weights=(cut, None, None, None))
    # the context is fine afterwards
    verify_indexed(inp, run_indexed_full(chord, inp, weights=(pw, None, None, None)),
                   label="after a mismatched pack")


def test_pack_scale_flag_is_reported(chord):
    inp = small(20, 2, 4, 4, 256, 256, 77, emap=False)
    inp.w2_s = inp.w2_s.copy()
    inp.w2_s[1, 7, 2] = 20 << 7  # 2^-107: below the exact range
    pw, _ = _packed(chord, inp)
    st = _status(chord, lambda: run_indexed_full(chord, inp, weights=(pw, None, None, None)))
    assert st == ERR_SCALE_RANGE
