"""K-split of the last round of GEMM units on the GPU, against the oracle.

When the units of a GEMM leave at least half of the SMs idle in their last
round, each unit of that round is cut along K into pieces that other CTAs
compute; the last piece to finish adds the partial sums in piece order
(include/chord.h, chord_w4a16_moe_indexed).  The shapes below have few units
and long K, so every unit of the GEMM named in each case is split (for a grid
of ~150 CTAs: rem = units < grid / 2 and K / BK >= 4).  Each case is checked
against the oracle with the split on and off (CHORD_FLAG_NO_SPLIT_K), and the
split result must be bit-identical from run to run."""

import numpy as np
import pytest

from gpu_util import assert_close_bf16, check_h, weights_to
from test_gpu_layer import (DEV, chord, contiguous_layer_check, masked_layer_check,  # noqa: F401
                            run_indexed_full, small, verify_indexed)
from w4a16_int4_mixture_gb300 import synth

pytestmark = pytest.mark.gpu
NO_SPLIT = 8

# (T, k, E, H, I, seed); chunks = experts hit (one chunk each), pieces per
# unit P = min(grid // units, stages // 2), grid ~150
CASES = {
    # gate/up: <= 16 chunks x 4 tiles, K = 2048 in 8 stages of 256 -> P >= 2
    "gate_up": (3, 8, 16, 2048, 256, 51),
    # gate/up: 8 chunks x 4 tiles, K = 2304 in 9 stages -> 4 pieces of 2, 2, 2, 3
    "gate_up-uneven": (1, 8, 16, 2304, 256, 52),
    # down: <= 16 chunks x 2 tiles, K = I = 2048 in 8 stages -> 4 pieces; two
    # epilogue groups
    "down": (3, 8, 16, 256, 2048, 53),
    # both GEMMs, one token: 4 chunks x 16 gate/up tiles (4 stages), 4 chunks x
    # 8 down tiles (4 stages) -> 2 pieces each
    "both": (1, 4, 16, 1024, 1024, 54),
    # prefill tile (BK 128): 4 experts x ~100 rows, 4 tiles, K = 2048 in 16
    # stages; this tile is never split (its pieces' sums cost more than the
    # split saves), so both runs take the whole-unit path
    "prefill-tile": (200, 2, 4, 2048, 256, 55),
}


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("flags", [0, 2], ids=["reduce", "ordered"])
def test_split_matches_oracle_and_unsplit(chord, name, flags):
    T, k, E, H, I, seed = CASES[name]
    inp = small(T, k, E, E, H, I, seed, emap=False)
    a = run_indexed_full(chord, inp, flags=flags)
    verify_indexed(inp, a, label=f"split {name}")
    b = run_indexed_full(chord, inp, flags=flags | NO_SPLIT)
    verify_indexed(inp, b, label=f"unsplit {name}")
    # the two differ only in the fp32 summation order of the accumulators: h
    # within the tolerance and few bf16 rounding flips apart (the outputs are
    # compared through the oracle above, each given its own h)
    check_h(a.h[:a.ntp], b.h[:b.ntp], f"{name}: split vs unsplit h")
    c = run_indexed_full(chord, inp, flags=flags)
    # (rows past num_tokens_padded are not written)
    assert np.array_equal(a.h[:a.ntp], c.h[:c.ntp]), "split gate/up output changed between runs"
    if flags & 2:
        assert np.array_equal(a.out, c.out), "split ordered path is not bit-reproducible"


def test_split_grouped_masked(chord):
    # 4 experts x up to 8 rows: 4 chunks x 16 tiles in both GEMMs (4 stages each) -> 2 pieces
    inp = small(8, 2, 4, 4, 256 * 8, 1024, 56, emap=False)
    a3, mm, r2p = synth.grouped_masked_layout(inp)
    masked_layer_check(chord, inp, a3, mm, r2p, weights_to(inp, DEV), "masked split")


def test_split_grouped_contiguous(chord):
    # 4 experts x up to 6 rows: 4 chunks x 2 down tiles, K = I = 2048 in 8 stages
    inp = small(6, 2, 4, 4, 256, 2048, 57, emap=False)
    rows_a, tok_a = contiguous_layer_check(chord, inp, 16, "contiguous split")
    rows_b, tok_b = contiguous_layer_check(chord, inp, 16, "contiguous unsplit", flags=NO_SPLIT)
    assert_close_bf16(rows_a, rows_b, "contiguous rows: split vs unsplit")
    assert_close_bf16(tok_a, tok_b, "contiguous tokens: split vs unsplit")
