"""The coordinate descent of the tuner ("Iteratively Tuning hipBLASLt TensileLite
Kernels", "The Iteration: Principle and Design"): incumbent in every round,
adoption only on a strict win, held latency never rising, illegal candidates
dropped -- checked on the host with synthetic latency functions."""
import random

import pytest

from shape_driven_tile_gb300.tune import descend


def rounds_over(space):
    """One round per parameter, each opening that parameter's values with the rest pinned."""
    def opener(name, values):
        return name, (lambda held: (dict(held, **{name: v}) for v in values))
    return [opener(n, vs) for n, vs in space.items()]


SPACE = {"a": range(6), "b": range(5), "c": range(4)}
START = {"a": 0, "b": 0, "c": 0}


def test_finds_separable_optimum_and_counts():
    cost = lambda c: 10 + (c["a"] - 3) ** 2 + 2 * (c["b"] - 1) ** 2 + 0.5 * (c["c"] - 2) ** 2
    held, traj = descend(rounds_over(SPACE), START, cost)
    assert held == {"a": 3, "b": 1, "c": 2}
    assert [t["round"] for t in traj] == ["base", "a", "b", "c"]
    assert traj[-1]["us"] == 10
    # every value of the opened parameter, the incumbent's among them (no duplicate)
    assert [t["enumerated"] for t in traj[1:]] == [6, 5, 4]


def test_held_latency_never_rises_under_noise():
    rng = random.Random(7)
    for trial in range(200):
        base = {k: [rng.uniform(1, 100) for _ in v] for k, v in SPACE.items()}
        noisy = lambda c: sum(base[k][c[k]] for k in c) * rng.uniform(0.7, 1.3)
        held, traj = descend(rounds_over(SPACE), START, noisy)
        us = [t["us"] for t in traj]
        assert all(b <= a for a, b in zip(us, us[1:])), us


def test_tie_keeps_incumbent():
    held, traj = descend(rounds_over({"a": range(3)}), {"a": 1}, lambda c: 5.0)
    assert held == {"a": 1} and traj[-1]["us"] == 5.0


def test_incumbent_is_always_a_candidate():
    seen = []

    def measure(c):
        seen.append(dict(c))
        return 1.0 + c["a"]

    # the round opens values that exclude the incumbent's own: it must still be timed
    descend([("a", lambda held: (dict(held, a=v) for v in (4, 5)))], {"a": 2}, measure)
    assert seen.count({"a": 2}) == 2  # once at the start, once inside the round


def test_illegal_candidates_are_dropped():
    legal = lambda c: None if c["a"] % 2 else 10.0 - c["a"]
    held, traj = descend(rounds_over({"a": range(6)}), {"a": 0}, legal)
    assert held == {"a": 4}
    assert traj[1]["enumerated"] == 6 and traj[1]["legal"] == 3


def test_empty_round_holds():
    held, traj = descend([("none", lambda held: iter(()))], {"a": 1}, lambda c: 3.0)
    assert held == {"a": 1} and traj[1]["us"] == 3.0 and traj[1]["enumerated"] == 1


def test_illegal_start_is_rejected():
    with pytest.raises(ValueError):
        descend(rounds_over(SPACE), START, lambda c: None)


def test_p4_shape_list_matches_the_page():
    from shape_driven_tile_gb300.inputs import P4_SHAPES
    # "Experiment Setup": 24 shapes, six probes and eighteen LLM-serving shapes
    assert len(P4_SHAPES) == 24 and len({s[0] for s in P4_SHAPES}) == 24
    probes = {"sqS", "sqL", "tallM", "wideN", "fatK", "thinK"}
    assert probes <= {s[0] for s in P4_SHAPES}
    d = {s[0]: s[1:] for s in P4_SHAPES}
    assert d["d4k_down_pf"] == (4096, 4096, 16384) and d["sn_64_pf"] == (4096, 64, 4096)
    assert d["d4k_ffn_dec"] == (16, 16384, 4096) and d["fatK"] == (1024, 1024, 8192)
    assert all(n % 8 == 0 for _, _, n, _ in P4_SHAPES)  # gemm_ex's only shape rule


def test_passes_shuffle_order_and_keep_best():
    # a device that slows down as it is used: with one fixed order the first candidate
    # would always look fastest; shuffled passes keep each candidate's best time
    clock = [0]
    order_seen = []

    def drifting(c):
        clock[0] += 1
        order_seen.append(c["a"])
        return 10.0 + c["a"] * 0.01 + clock[0] * 0.1

    held, traj = descend([("a", lambda h: (dict(h, a=v) for v in range(4)))], {"a": 3}, drifting, passes=3, seed=1)
    firsts = [order_seen[1 + 4 * p] for p in range(3)]  # first candidate timed in each pass
    assert len(set(firsts)) > 1                         # the order changes between passes
    assert len(order_seen) == 1 + 4 * 3


def test_passes_skip_illegal_after_first_pass():
    calls = []

    def measure(c):
        calls.append(c["a"])
        return None if c["a"] == 1 else 5.0 - c["a"]

    descend([("a", lambda h: (dict(h, a=v) for v in range(3)))], {"a": 0}, measure, passes=3)
    assert calls.count(1) == 1
