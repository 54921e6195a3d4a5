"""moe_align on the GPU against the oracle: bit-exact over the whole capacity."""

import numpy as np
import pytest
import torch

import oracle
from w4a16_int4_mixture_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def chord():
    import w4a16_int4_mixture_gb300 as m
    m.build()
    return m


def _run(chord, ids, E_global, emap, E_local, bm, capacity=None):
    dev = torch.device("cuda:0")
    tid = torch.from_numpy(np.ascontiguousarray(ids, dtype=np.int32)).to(dev)
    tmap = None if emap is None else torch.from_numpy(np.ascontiguousarray(emap)).to(dev)
    si, ei, ntp = chord.moe_align(tid, E_global, E_local, bm, expert_map=tmap, capacity=capacity)
    torch.cuda.synchronize()
    return si.cpu().numpy(), ei.cpu().numpy(), int(ntp.item())


def _compare(chord, ids, E_global, emap, E_local, bm, capacity=None):
    si, ei, ntp = _run(chord, ids, E_global, emap, E_local, bm, capacity)
    rsi, rei, rntp = oracle.moe_align(ids, E_global, emap, E_local, bm, capacity=capacity)
    assert ntp == rntp
    assert np.array_equal(si, rsi), f"sorted_ids differ at {np.nonzero(si != rsi)[0][:10]}"
    assert np.array_equal(ei, rei), f"expert_ids differ at {np.nonzero(ei != rei)[0][:10]}"


@pytest.mark.parametrize("wl,T", [("tiny", None), ("ep8-decode", None), ("ep8-prefill", None),
                                  ("tp8", 1), ("tp8", 16), ("tp8", 128), ("tp8", 2048),
                                  ("skewed", None)])
def test_align_workloads(chord, wl, T):
    s = synth.workload(wl, T=T)
    inp = synth.make_inputs(s, weights=False)
    _compare(chord, inp.topk_ids, s.E_global, inp.expert_map, s.E_local, s.block_m)


@pytest.mark.parametrize("bm", [1, 4, 8, 16, 32, 64, 128])
def test_align_block_m(chord, bm):
    s = synth.workload("ep8-decode", T=300)
    inp = synth.make_inputs(s, weights=False)
    _compare(chord, inp.topk_ids, s.E_global, inp.expert_map, s.E_local, bm)


def test_align_random_small(chord):
    rng = np.random.default_rng(7)
    for _ in range(25):
        T = int(rng.integers(1, 300))
        k = int(rng.integers(1, 9))
        Eg = int(rng.integers(k, 70))
        El = int(rng.integers(1, Eg + 1))
        emap = np.full(Eg, -1, np.int32)
        emap[rng.permutation(Eg)[:El]] = np.arange(El, dtype=np.int32)
        ids = np.stack([rng.permutation(Eg)[:k] for _ in range(T)]).astype(np.int32)
        bm = int(rng.choice([1, 2, 8, 16, 48]))
        _compare(chord, ids, Eg, emap, El, bm)


@pytest.mark.parametrize("E", [129, 384, 512, 513, 1000])
def test_align_many_local_experts(chord, E):
    # one-CTA form up to 512 local experts and 4096 pairs, three kernels beyond
    rng = np.random.default_rng(E)
    T, k = 300, 8
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    for bm in (1, 16):
        _compare(chord, ids, E, None, E, bm)


def test_align_over_allocated_capacity(chord):
    s = synth.workload("tp8", T=16)
    inp = synth.make_inputs(s, weights=False)
    cap = chord.moe_align_capacity(2048, 8, 384, 16)
    _compare(chord, inp.topk_ids, s.E_global, None, s.E_local, 16, capacity=cap)


def test_align_empty_and_nonlocal(chord):
    _compare(chord, np.zeros((0, 4), np.int32), 8, None, 8, 16)
    emap = np.array([-1, -1, 0, 1], np.int32)
    ids = np.array([[0, 1], [1, 0], [0, 1]], np.int32)
    _compare(chord, ids, 4, emap, 2, 8)


def test_align_many_rows_one_expert(chord):
    # every token to the same experts: long segments
    ids = np.tile(np.array([[5, 1, 2]], np.int32), (3000, 1))
    _compare(chord, ids, 8, None, 8, 16)


def test_align_invalid_ids_are_reported(chord):
    dev = torch.device("cuda:0")
    ids = np.array([[0, 9], [1, -3], [2, 3]], np.int32)
    tid = torch.from_numpy(ids).to(dev)
    ws = torch.zeros(chord.ops.align_workspace_size(3, 2, 4) + 256, dtype=torch.uint8, device=dev)
    si, ei, ntp = chord.moe_align(tid, 4, 4, 4, workspace=ws)
    bits = chord.get_device_error(ws)
    assert bits & 2, "out-of-range ids must set the routing error bit"
    rsi, rei, rntp = oracle.moe_align(ids, 4, None, 4, 4)
    assert np.array_equal(si.cpu().numpy(), rsi) and int(ntp.item()) == rntp


@pytest.mark.parametrize("T,E,spread", [(512, 512, "uniform"), (512, 384, "eight-experts"),
                                        (513, 384, "uniform"), (385, 100, "eight-experts")])
def test_align_one_cta_limit(chord, T, E, spread):
    """Both sides of the one-CTA form's limit (4096 pairs): 512 tokens x 8
    fill its four rounds per warp; with every pair on eight experts a warp's
    count of one expert reaches 16 in a round and an expert's prefix over the
    warps 512; 513 tokens take the three kernels."""
    rng = np.random.default_rng(T + E)
    if spread == "uniform":
        ids = np.stack([rng.permutation(E)[:8] for _ in range(T)]).astype(np.int32)
    else:
        ids = np.stack([rng.permutation(8) for _ in range(T)]).astype(np.int32)
    for bm in (1, 16, 64, 256):
        _compare(chord, ids, E, None, E, bm)
