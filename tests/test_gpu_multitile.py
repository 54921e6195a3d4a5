"""Down GEMM units that hold several weight tiles (a one-stage K: I = 256).

With I = 256 the down GEMM's K is a single stage, and the library lets one
work unit cover up to four 128-row weight tiles that share the unit's token
tile, when the units still give every SM several.  The TP8 workload tests
(test_gpu_layer) run this at their full sizes; these cases add the grouped
entry points and a ragged expert mix, against the oracle.  The last case runs
the 64-row token tile over many units of a long K."""

import numpy as np
import pytest

from gpu_util import weights_to
from test_gpu_layer import (DEV, chord, contiguous_layer_check, masked_layer_check,  # noqa: F401
                            run_indexed_full, small, verify_indexed)
from w4a16_int4_mixture_gb300 import synth

pytestmark = pytest.mark.gpu


def tp8_like(T, k, E, seed):
    # H = 7168 -> 56 down tiles per chunk; ~E * 56 / 4 units of four tiles
    return small(T, k, E, E, 7168, 256, seed, emap=False)


def test_multitile_indexed_ragged(chord):
    # 48 experts, ~2-6 rows each (token tiles of 16 and 32 columns)
    inp = tp8_like(40, 6, 48, 61)
    verify_indexed(inp, run_indexed_full(chord, inp), label="multi-tile indexed")


def test_multitile_masked(chord):
    inp = tp8_like(24, 6, 48, 62)
    a3, mm, r2p = synth.grouped_masked_layout(inp)
    masked_layer_check(chord, inp, a3, mm, r2p, weights_to(inp, DEV), "multi-tile masked")


def test_multitile_contiguous(chord):
    inp = tp8_like(24, 6, 48, 63)
    contiguous_layer_check(chord, inp, 16, "multi-tile contiguous")


def test_multitile_deterministic(chord):
    inp = tp8_like(40, 6, 48, 64)
    a = run_indexed_full(chord, inp, flags=2)
    b = run_indexed_full(chord, inp, flags=2)
    assert np.array_equal(a.out, b.out)


def test_tile64_many_units(chord):
    # 64 experts x ~20 rows (64-row token tile), I = 2048: 32 gate/up tiles and
    # 4 down tiles per chunk, down K in 8 stages
    inp = small(160, 8, 64, 64, 512, 2048, 65, emap=False)
    a = run_indexed_full(chord, inp, flags=2)
    verify_indexed(inp, a, label="64-row tile, many units")
    b = run_indexed_full(chord, inp, flags=2)
    assert np.array_equal(a.out, b.out)


@pytest.mark.parametrize("bm", [16, 32])
def test_indexed_compacted_token_rows(chord, bm):
    # 256 experts x ~2 rows: the layout's padding rows would pass 16 MB, so the
    # gathered token rows are compacted (gate/up token boxes start at each
    # chunk's compacted row); h rows of the padding stay zero
    inp = small(128, 4, 256, 256, 7168, 256, 66 + bm, emap=False)
    run = run_indexed_full(chord, inp, block_m=bm)
    verify_indexed(inp, run, label=f"compacted token rows block_m={bm}")
    pad = np.nonzero(run.si[:run.ntp] >= inp.shape.T * inp.shape.k)[0]
    assert pad.size > 0 and np.all(run.h[pad] == 0)
