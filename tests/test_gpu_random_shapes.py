"""A seeded sweep of random supported shapes through the layer.

The fixed cases elsewhere pick shapes for the schedule they exercise; this
sweep draws shapes the way a caller might (hidden size a multiple of 128,
intermediate size a multiple of 128, top-k up to 8, any token count, local
experts a subset of the global ones with or without an expert map, any
padding granularity), weights plain INT4, prepacked INT4 or MXFP4, with or
without the ordered combine, and checks each like the fixed cases: the split
check against the oracle and the fp64 anchor of the definition.  A second
draw runs the grouped entry (contiguous layout with a random segment
alignment, masked layout) the same way.  The draws are fixed (seeds 2024 and
2025), so a failing case reproduces by its id."""

import contextlib

import numpy as np
import pytest

import oracle
from test_gpu_layer import (DEV, chord, contiguous_layer_check, masked_layer_check,  # noqa: F401
                            run_indexed_full, small, verify_indexed)
from test_gpu_mxfp4 import mx_small, mx_weights
from gpu_util import weights_to
from w4a16_int4_mixture_gb300 import synth

pytestmark = pytest.mark.gpu


def _draw(n=16, seed=2024):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        H = int(rng.choice([256, 384, 512, 640, 768, 1024]))
        I = int(rng.choice([128, 256, 384, 512]))
        k = int(rng.choice([1, 2, 3, 4, 6, 8]))
        Eg = int(rng.integers(max(k, 2), 40))
        El = int(rng.integers(1, Eg + 1))
        T = int(rng.choice([1, 2, 7, 33, 96, 160, 257]))
        bm = int(rng.choice([1, 4, 16, 32, 64]))
        form = str(rng.choice(["plain", "packed", "mxfp4"]))
        flags = int(rng.choice([0, 2]))  # 2: CHORD_FLAG_DETERMINISTIC
        cases.append((f"r{i}-T{T}-k{k}-E{El}of{Eg}-H{H}-I{I}-bm{bm}-{form}-f{flags}",
                      (T, k, Eg, El, H, I, 3000 + i, bm, form, flags)))
    return cases


CASES = _draw()


@pytest.mark.parametrize("name,args", CASES, ids=[c[0] for c in CASES])
def test_random_shape(chord, name, args):
    T, k, Eg, El, H, I, seed, bm, form, flags = args
    emap = El < Eg
    if form == "mxfp4":
        inp = mx_small(T, k, Eg, El, H, I, seed, emap=emap)
        inp.shape.block_m = bm
        pw = chord.prepack_weights(*mx_weights(inp))
        with oracle.weight_format("mxfp4"):
            run = run_indexed_full(chord, inp, block_m=bm, flags=flags, weights=(pw, None, None, None))
            verify_indexed(inp, run, label=name)
        return
    inp = small(T, k, Eg, El, H, I, seed, bm=bm, emap=emap)
    w = weights_to(inp, DEV)
    if form == "packed":
        w = (chord.prepack_weights(*w), None, None, None)
    run = run_indexed_full(chord, inp, block_m=bm, flags=flags, weights=w)
    verify_indexed(inp, run, label=name)


def _draw_grouped(n=8, seed=2025):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        H = int(rng.choice([256, 384, 512, 768]))
        I = int(rng.choice([128, 256, 384]))
        k = int(rng.choice([1, 2, 4, 8]))
        E = int(rng.integers(max(k, 2), 24))
        T = int(rng.choice([1, 5, 40, 130]))
        mode = "contiguous" if i % 2 == 0 else "masked"
        align = int(rng.choice([16, 64, 128]))
        form = str(rng.choice(["plain", "packed", "mxfp4"]))
        cases.append((f"g{i}-{mode}-T{T}-k{k}-E{E}-H{H}-I{I}-a{align}-{form}",
                      (T, k, E, H, I, 4000 + i, mode, align, form)))
    return cases


GROUPED = _draw_grouped()


@pytest.mark.parametrize("name,args", GROUPED, ids=[c[0] for c in GROUPED])
def test_random_grouped(chord, name, args):
    T, k, E, H, I, seed, mode, align, form = args
    if form == "mxfp4":
        inp = mx_small(T, k, E, E, H, I, seed, emap=False)
        w = (chord.prepack_weights(*mx_weights(inp)), None, None, None)
        fmt = oracle.weight_format("mxfp4")  # the oracle's weight format for this case
    else:
        inp = small(T, k, E, E, H, I, seed, emap=False)
        w = weights_to(inp, DEV)
        if form == "packed":
            w = (chord.prepack_weights(*w), None, None, None)
        fmt = None
    with fmt if fmt is not None else contextlib.nullcontext():
        if mode == "contiguous":
            contiguous_layer_check(chord, inp, align, name, weights=w)
        else:
            a3, mm, r2p = synth.grouped_masked_layout(inp)
            masked_layer_check(chord, inp, a3, mm, r2p, w, name)
