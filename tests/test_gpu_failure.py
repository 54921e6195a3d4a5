"""Failure detection on the GPU without a fault: a bounded wait that expires.

CHORD_FLAG_TEST_SKIP_ARRIVE makes the gate/up GEMM drop one mbarrier arrival
(first K stage of CTA 0).  The MMA issuer's wait on that barrier is bounded
(2 s); when it expires the CTA records CHORD_DEVERR_TIMEOUT, every role leaves
its loop, copies already issued are drained and TMEM is freed.  The call then
reports CHORD_ERR_TIMEOUT through CHORD_FLAG_VALIDATE, and the same context
keeps producing correct results.  No trap, no fault, no unbounded wait."""

import pytest

from test_gpu_layer import chord, run_indexed_full, verify_indexed  # noqa: F401
from w4a16_int4_mixture_gb300 import synth

pytestmark = pytest.mark.gpu

CHORD_ERR_TIMEOUT = -6


def test_expired_wait_reports_timeout_and_context_survives(chord):
    inp = synth.make_inputs(synth.workload("tiny"))
    with pytest.raises(chord.ChordError) as ei:
        run_indexed_full(chord, inp, flags=chord.ops.B.FLAG_TEST_SKIP_ARRIVE)
    assert ei.value.status == CHORD_ERR_TIMEOUT
    # the next call on the same context is clean and correct
    verify_indexed(inp, run_indexed_full(chord, inp), label="after an expired wait")
