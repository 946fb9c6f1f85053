"""The library's placement planner (host code in libmoeroute.so) vs the oracle.

moe_plan_placement runs on the host, so these tests need no GPU: every output
(slots of each expert, slot contents, partition loads) must equal the
oracle's, integer for integer, over random loads and shapes.
"""
import numpy as np
import pytest

import combine_moe_route_06_gb300 as m
import oracle


@pytest.fixture(scope="module")
def lib():
    m.build()
    return m.load_library()


def _same(a, b):
    return (np.array_equal(a["copy_offsets"], b.copy_offsets)
            and np.array_equal(a["copy_slots"], b.copy_slots)
            and np.array_equal(a["slot_expert"], b.slot_expert)
            and np.array_equal(a["part_load"], b.part_load))


@pytest.mark.parametrize("seed", range(6))
def test_planner_matches_oracle(lib, seed):
    rng = np.random.default_rng(seed)
    for trial in range(60):
        P = int(rng.choice([1, 2, 4, 8, 16, 32]))
        L = int(rng.integers(1, 9))
        R = int(rng.integers(0, 5))
        E = P * L
        kind = trial % 3
        if kind == 0:
            load = rng.integers(0, 1000, E)
        elif kind == 1:                                  # Zipf-like, shuffled
            p = (np.arange(E) + 1.0) ** -rng.uniform(0.5, 2.0)
            load = rng.multinomial(E * 50, p / p.sum())
            rng.shuffle(load)
        else:                                            # many equal loads: the tie rules
            load = rng.integers(0, 4, E) * 7
        load = load.astype(np.int64)
        assert _same(oracle.plan_placement(load, P, R), m.moe_plan_placement(load, P, R)), \
            (P, L, R, load.tolist())


def test_planner_hand_example(lib):
    import json
    import os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "placement_hand.json")))
    pl = m.moe_plan_placement(np.array(g["load"], np.int64), g["P"], g["R"])
    assert pl.copy_offsets.tolist() == g["copy_offsets"]
    assert pl.copy_slots.tolist() == g["copy_slots"]
    assert pl.slot_expert.tolist() == g["slot_expert"]
    assert pl.part_load.tolist() == g["part_load"]


@pytest.mark.parametrize("E,P,R", [(10, 4, 1), (64, 8, 200), (8, 0, 1)])
def test_planner_rejects_bad_shapes(lib, E, P, R):
    with pytest.raises((m.MoeError, ZeroDivisionError, ValueError)):
        m.moe_plan_placement(np.ones(E, np.int64), P, R)


def test_planner_rejects_negative_load(lib):
    with pytest.raises(m.MoeError):
        m.moe_plan_placement(np.array([3, -1, 2, 2], np.int64), 2, 1)
