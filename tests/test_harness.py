"""The split parity check the GPU tests use, exercised on the CPU with an
oracle-made run standing in for the GPU (it must accept it with zero flips),
and with planted errors in the output or the intermediate (it must reject
those): a large change of one element, a tile of one row far off, and
one-ulp rounding flips in 1.5 % of h (each within the element-wise
tolerance, caught by the flip ceiling and the fp64 anchor)."""

import numpy as np
import pytest

import oracle
import test_gpu_layer as L


def _self_run():
    inp = L.small(40, 3, 10, 6, 512, 256, 1)
    (si, ei, ntp), (out, h, _) = oracle.run_workload(inp, want_h=True)
    return inp, L.Run(out, h, si, ei, ntp, 16)


def test_split_check_accepts_the_oracle_itself():
    inp, run = _self_run()
    assert L.verify_indexed(inp, run, label="self") == 0.0
    assert L.verify_indexed(inp, run, tokens=np.array([3, 7, 11, 0]), label="self-sub") == 0.0


def test_split_check_rejects_a_wrong_output():
    inp, run = _self_run()
    bad = run.out.copy()
    bad[5, 17] ^= 0x0040  # a large change of one element
    with pytest.raises(AssertionError):
        L.verify_indexed(inp, L.Run(bad, run.h, run.si, run.ei, run.ntp, run.bm))


def test_split_check_rejects_a_wrong_intermediate():
    inp, run = _self_run()
    bad = run.h.copy()
    rows = np.nonzero(run.si[:run.ntp] < inp.shape.T * inp.shape.k)[0]
    bad[rows[0], :64] ^= 0x0100  # one tile of one row far off
    with pytest.raises(AssertionError):
        L.verify_indexed(inp, L.Run(run.out, bad, run.si, run.ei, run.ntp, run.bm))


def test_split_check_rejects_many_one_ulp_flips():
    inp, run = _self_run()
    bad = run.h.copy()
    rows = np.nonzero(run.si[:run.ntp] < inp.shape.T * inp.shape.k)[0]
    body = bad[rows]
    rng = np.random.default_rng(0)
    flip = rng.random(body.shape) < 0.015
    flip &= (body & 0x7F80) != 0  # normal numbers: +-1 in the last place stays close
    body[flip] ^= 0x0001
    bad[rows] = body
    with pytest.raises(AssertionError, match="differ|flips"):
        L.verify_indexed(inp, L.Run(run.out, bad, run.si, run.ei, run.ntp, run.bm))
