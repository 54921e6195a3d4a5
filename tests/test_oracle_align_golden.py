"""Hand-derived align example (tests/golden/align_small.json) against the oracle."""

import json
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "align_small.json")


def test_align_hand_example():
    g = json.load(open(GOLDEN))
    ids = np.array(g["topk_ids"], np.int32)
    cap = oracle.align_capacity(g["T"], g["k"], g["E_local"], g["block_m"])
    assert cap == g["capacity"]
    si, ei, ntp = oracle.moe_align(ids, g["E_global"], np.array(g["expert_map"], np.int32),
                                   g["E_local"], g["block_m"])
    assert si.tolist() == g["sorted_ids"]
    assert ei.tolist() == g["expert_ids"]
    assert ntp == g["num_tokens_padded"]


def test_align_capacity_too_small_is_an_error():
    ids = np.array([[0, 1], [1, 0]], np.int32)
    try:
        oracle.moe_align(ids, 2, None, 2, 4, capacity=4)
    except ValueError:
        return
    raise AssertionError("capacity 4 < 8 accepted")


def test_align_no_local_pairs():
    ids = np.array([[3, 2]], np.int32)
    emap = np.array([0, 1, -1, -1], np.int32)
    si, ei, ntp = oracle.moe_align(ids, 4, emap, 2, 4)
    assert ntp == 0 and np.all(si == 2) and np.all(ei == -1)
