"""Router + align (chord_moe_route_align) on the GPU against the oracle.

The expert ids and the aligned layout are bit-exact: both sides pick the k
largest of the same fp32 logits with ties to the lower id.  The weights use
fp32 exp and sums on the GPU and fp64 in the oracle: within 8 fp32 ulp."""

import zlib

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def chord():
    import w4a16_int4_mixture_gb300 as m
    m.build()
    return m


def _case(T, E, k, El, emap, bm, renorm, ties, seed):
    rng = np.random.default_rng(seed)
    if ties:
        lg = rng.integers(-2, 3, size=(T, E)).astype(np.float32)
    else:
        lg = rng.standard_normal((T, E)).astype(np.float32)
    m = None
    if emap:
        m = np.full(E, -1, np.int32)
        m[rng.permutation(E)[:El]] = np.arange(El, dtype=np.int32)
    return lg, m


CASES = {
    # one CTA (<= 64 tokens, <= 4096 pairs, <= 512 local experts); the router
    # keeps 4, 8, 16 or 32 logits per lane for E <= 128, 256, 512, 1024
    "small-64": (40, 64, 4, 64, False, 16, True, False),
    "tp8-T1": (1, 384, 8, 384, False, 16, True, False),
    "softmax-weights": (64, 96, 6, 96, False, 16, False, False),
    "ties-fused": (50, 40, 8, 40, False, 8, True, True),
    "E256-T16": (16, 256, 8, 256, False, 16, True, False),
    "k32-E1024-fused": (60, 1024, 32, 256, True, 16, True, False),
    # router kernel + the align kernels
    "ep8-decode": (512, 384, 8, 48, True, 16, True, False),
    "tp8-T128": (128, 384, 8, 384, False, 16, True, False),
    "ties": (300, 40, 8, 40, False, 8, True, True),
    "k32-E1024": (100, 1024, 32, 256, True, 16, True, False),
    "E200-T65": (65, 200, 8, 200, False, 16, True, False),
    "tp8-T2048": (2048, 384, 8, 384, False, 16, True, False),
    "many-local": (700, 1000, 8, 600, True, 32, True, True),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_route_align_matches_oracle(chord, name):
    T, E, k, El, emap, bm, renorm, ties = CASES[name]
    lg, m = _case(T, E, k, El, emap, bm, renorm, ties, seed=zlib.crc32(name.encode()) & 0xFFFF)
    tm = None if m is None else torch.from_numpy(m).to(DEV)
    ids, w, si, ei, ntp = chord.moe_route_align(torch.from_numpy(lg).to(DEV), k, El, bm,
                                                expert_map=tm, renormalize=renorm)
    torch.cuda.synchronize()
    rids, rw = oracle.route_topk(lg, k, renorm)
    assert np.array_equal(ids.cpu().numpy(), rids), "expert ids differ"
    gw = w.cpu().numpy().astype(np.float64)
    ulp = np.spacing(rw.astype(np.float32)).astype(np.float64)
    assert np.abs(gw - rw).max() <= 8 * ulp.max(), f"weights off by {np.abs(gw - rw).max()}"
    rsi, rei, rntp = oracle.moe_align(rids, E, m, El, bm)
    assert int(ntp.item()) == rntp
    assert np.array_equal(si.cpu().numpy(), rsi)
    assert np.array_equal(ei.cpu().numpy(), rei)


def test_route_align_equals_align_of_routed_ids(chord):
    """Same layout as chord_moe_align on the router's ids (both forms)."""
    for T in (200, 1500):
        lg, _ = _case(T, 128, 8, 128, False, 16, True, False, seed=T)
        ids, w, si, ei, ntp = chord.moe_route_align(torch.from_numpy(lg).to(DEV), 8, 128, 16)
        si2, ei2, ntp2 = chord.moe_align(ids, 128, 128, 16)
        torch.cuda.synchronize()
        assert torch.equal(si, si2) and torch.equal(ei, ei2) and torch.equal(ntp, ntp2)
