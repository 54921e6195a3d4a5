"""A seeded sweep of random supported shapes through the indexed layer.

The fixed cases elsewhere pick shapes for the schedule they exercise; this
sweep draws shapes the way a caller might (hidden size a multiple of 256,
intermediate size a multiple of 128, top-k up to 8, any token count, local
experts a subset of the global ones with or without an expert map, any
padding granularity), weights plain INT4, prepacked INT4 or MXFP4, with or
without the ordered combine, and checks each like the fixed cases: the split
check against the oracle and the fp64 anchor of the definition.  The draw is
fixed (seed 2024), so a failing case reproduces by its id."""

import numpy as np
import pytest

import oracle
from test_gpu_layer import DEV, chord, run_indexed_full, small, verify_indexed  # noqa: F401
from test_gpu_mxfp4 import mx_small, mx_weights
from gpu_util import weights_to
from w4a16_int4_mixture_gb300 import synth

pytestmark = pytest.mark.gpu


def _draw(n=16, seed=2024):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        H = int(rng.choice([256, 512, 768, 1024]))
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
