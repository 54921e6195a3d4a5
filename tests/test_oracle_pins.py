"""The CPU oracle against what the page and mathematics fix (no GPU)."""

import numpy as np
import pytest

import oracle
import pins


@pytest.mark.parametrize("name", sorted(pins.ALL_PINS))
def test_pin(name):
    ok, detail = pins.ALL_PINS[name]()
    assert ok, detail


@pytest.mark.parametrize("seed,kw", [
    (1, dict(T=9, k=2, Eg=4, El=4, H=96, I=64, bm=8, emap=False)),
    (2, dict(T=5, k=4, Eg=9, El=3, H=32, I=32, bm=1)),
])
def test_brute_force_more_shapes(seed, kw):
    ok, detail = pins.pin_brute_force(seed, **kw)
    assert ok, detail


def test_rne_reference_itself():
    """The independent rounding used by the pins: ties to even, halfway cases,
    subnormals and overflow on hand-picked values."""
    one = 1.0
    ulp1 = 2.0 ** -7               # bf16 spacing just above 1.0
    vals = np.array([one + ulp1 / 2, one + 1.5 * ulp1, one + ulp1 / 2 + 1e-12,
                     2.0 ** -133, 2.0 ** -134, 3 * 2.0 ** -134,
                     float.fromhex("0x1.fep127") + 2.0 ** 119,
                     float.fromhex("0x1.fep127") + 2.0 ** 118, -0.0])
    want = np.array([one, one + 2 * ulp1, one + ulp1, 2.0 ** -133, 0.0, 2 * 2.0 ** -133,
                     np.inf, float.fromhex("0x1.fep127"), -0.0])
    got = pins.rne_bf16(vals)
    assert np.array_equal(got, want)
    assert np.signbit(got[-1])


def test_bf16_bits_roundtrip():
    b = np.arange(0, 65536, 7, dtype=np.uint32).astype(np.uint16)
    f = oracle.bf16_to_f32(b)
    fin = np.isfinite(f)
    back = np.array([oracle.f32_to_bf16(float(v)) for v in f[fin][:2000]], np.uint16)
    assert np.array_equal(back, b[fin][:2000])


def test_downstream_entry_reproduces_the_layer():
    """Down + combine on the oracle's own h reproduces the whole layer bit-exactly
    (indexed and grouped): the split entries are the same arithmetic."""
    inp = pins.small_random_inputs(3)
    s = inp.shape
    (si, ei, ntp), (out, h, _) = oracle.run_workload(inp, want_h=True)
    out2 = oracle.moe_indexed_down(h, inp.w2_q, inp.w2_s, inp.topk_weights, si, ei, ntp,
                                   s.block_m, s.T, s.k)
    assert np.array_equal(out, out2)
    from w4a16_int4_mixture_gb300 import synth
    a3, mm, r2p = synth.grouped_masked_layout(inp)
    rows, toks, hg = oracle.moe_grouped("masked", a3, inp.w13_q, inp.w13_s, inp.w2_q, inp.w2_s,
                                        masked_m=mm, row_to_pair=r2p,
                                        topk_weights=inp.topk_weights, T=s.T, k=s.k,
                                        want_h=True)
    rows2, toks2 = oracle.moe_grouped_down("masked", hg, inp.w2_q, inp.w2_s, masked_m=mm,
                                           max_m=a3.shape[1], row_to_pair=r2p,
                                           topk_weights=inp.topk_weights, T=s.T, k=s.k)
    assert np.array_equal(rows, rows2) and np.array_equal(toks, toks2)
    assert np.array_equal(toks, out)
