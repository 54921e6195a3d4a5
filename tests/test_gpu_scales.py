"""Scale-range contract of the layer calls on the GPU.

The kernels form each weight as bf16((q - 8) * s * 2^-40) and scale the fp32
accumulators back by 2^40, which equals bf16((q - 8) * s) exactly for scales
that are +-0 or of magnitude in [2^-86, 2^35) (include/chord.h).  These tests
drive experts whose scales sit near both ends of that range against the
oracle, and check that CHORD_FLAG_VALIDATE reports scales outside it."""

import numpy as np
import pytest

import oracle
from gpu_util import assert_close_bf16, check_h
from test_gpu_layer import DEV, chord, run_indexed_full, sub_batch  # noqa: F401
from w4a16_int4_mixture_gb300 import synth

pytestmark = pytest.mark.gpu


def pow2_scales(rng, E, N, K, exps):
    """bf16 scales +-2^(exps[e] + u), u uniform in {0..5}, per expert e."""
    u = rng.integers(0, 6, size=(E, N, K // 32))
    sign = np.where(rng.random((E, N, K // 32)) < 0.5, -1.0, 1.0)
    e = np.asarray(exps, dtype=np.int64)[:, None, None] + u
    return synth._bf16_bits((sign * np.ldexp(1.0, e)).astype(np.float32))


def top1_inputs(exps13, exps2, T=160, H=512, I=256, seed=31):
    E = len(exps13)
    s = synth.MoEShape("scale-range", T=T, k=1, E_global=E, E_local=E, H=H, I=I, block_m=16,
                       seed=seed)
    inp = synth.make_inputs(s)
    rng = np.random.default_rng(seed + 1)
    inp.w13_s = pow2_scales(rng, E, 2 * I, H, exps13)
    inp.w2_s = pow2_scales(rng, E, H, I, exps2)
    return inp


def test_scales_near_range_ends_match_oracle(chord):
    # (gate/up exponent, down exponent) per expert: gate/up scales down to
    # 2^-52 (h ~ s^2 stays a normal bf16), down scales from 2^-84 to 2^33.
    exps13 = [-52, -30, 0, 12, 5, -8, 25, 0]
    exps2 = [28, 20, 0, -84, -60, 29, -75, -20]
    inp = top1_inputs(exps13, exps2)
    run = run_indexed_full(chord, inp)
    ids = inp.topk_ids[:, 0]
    # with top-1 routing each token's output comes from one expert: compare the
    # tokens of each expert on their own scale
    for e in range(len(exps13)):
        tok = np.nonzero(ids == e)[0]
        if tok.size == 0:
            continue
        sub = sub_batch(inp, tok)
        (ssi, sei, sntp), (_, sh, _) = oracle.run_workload(sub, block_m=16, want_h=True)
        # GPU h rows of these tokens, in the sub-batch's row order
        pos = {int(p): r for r, p in enumerate(run.si[:run.ntp]) if p < inp.shape.T}
        rows = [pos[int(t)] for t in tok]
        srows = [r for r in range(sntp) if ssi[r] < tok.size]
        order = np.argsort([ssi[r] for r in srows])
        h_gpu = run.h[rows]
        h_ref = sh[np.asarray(srows)[order]]
        check_h(h_gpu, h_ref, f"expert {e} h")
        h_sub = np.zeros_like(sh)
        for i, r in enumerate(np.asarray(srows)[order]):
            h_sub[r] = h_gpu[i]
        down = oracle.moe_indexed_down(h_sub, inp.w2_q, inp.w2_s, sub.topk_weights, ssi, sei,
                                       sntp, 16, tok.size, 1)
        assert_close_bf16(run.out[tok], down, f"expert {e} output given h")


@pytest.mark.parametrize("bad", ["huge", "subnormal", "inf"])
def test_validate_reports_out_of_range_scale(chord, bad):
    inp = top1_inputs([0, 0, 0, 0], [0, 0, 0, 0], T=40)
    bits = {"huge": 0x5100,        # 2^35: first magnitude past the range
            "subnormal": 0x0001,   # smallest positive subnormal
            "inf": 0x7F80}[bad]
    inp.w2_s = inp.w2_s.copy()
    inp.w2_s[2, 5, 1] = bits
    with pytest.raises(chord.ChordError) as ei:
        run_indexed_full(chord, inp)
    assert ei.value.status == -10


def test_validate_accepts_range_bounds_and_zero(chord):
    inp = top1_inputs([0, 0, 0, 0], [0, 0, 0, 0], T=40)
    inp.w13_s = inp.w13_s.copy()
    inp.w13_s[0, 0, 0] = 0x0000     # +0
    inp.w13_s[0, 0, 1] = 0x8000     # -0
    inp.w13_s[1, 3, 2] = 0x1480     # 2^-86, the smallest magnitude in range
    inp.w13_s[2, 7, 3] = 0xD0FF     # -(2^35 - 2^27), the largest magnitude in range
    run_indexed_full(chord, inp)    # validate flag set: must not raise
