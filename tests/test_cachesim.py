"""Pins for the expert-cache policy simulator (CPU only): hand-worked traces for each
policy, the optimality of Belady among demand-loading policies, and the no-eviction
case where every policy only misses first references."""
import numpy as np

from routing_predicted_experts_gb300 import cachesim as CS

# capacity 2; references 1 2 1 3 2 1 (one expert per token)
TR = [[1], [2], [1], [3], [2], [1]]


def test_lru_hand_worked():
    # 1 m, 2 m, 1 h, 3 m (evicts 2), 2 m (evicts 1), 1 m (evicts 3)
    assert CS.lru_hits(TR, 2) == 1


def test_lfu_hand_worked():
    # 1 m, 2 m, 1 h (1 counted twice), 3 m evicts 2 (count 1), 2 m evicts 3 (count 1 < 2), 1 h
    assert CS.lfu_hits(TR, 2) == 2


def test_belady_hand_worked():
    # at 3: 1 is next used at position 5, 2 at 4 -> evict 1; 2 h; 1 m
    assert CS.belady_hits(TR, 2) == 2


def test_static_hand_worked():
    # warm-up of 3 tokens counts 1 twice and 2 once: {1, 2} are held; only 3 misses
    assert CS.static_hits(TR, 2, warmup=3) == 5
    assert CS.static_hits(TR, 1, warmup=3) == 3


def test_pool_rule_never_evicts_the_current_or_previous_set():
    # slots 4, sets of 2: {0,1} {2,3} {4,5}: 4 and 5 must evict 0 and 1 (2, 3 are pinned)
    tr = [[0, 1], [2, 3], [4, 5], [2, 3]]
    assert CS.pool_lru_hits(tr, 4) == 2


def test_belady_bounds_the_online_policies_and_full_capacity():
    rng = np.random.default_rng(3)
    for _ in range(30):
        E = int(rng.integers(4, 20))
        tr = [list(rng.choice(E, size=2, replace=False)) for _ in range(int(rng.integers(5, 40)))]
        c = int(rng.integers(2, E))
        b = CS.belady_hits(tr, c)
        assert b >= CS.lru_hits(tr, c) and b >= CS.lfu_hits(tr, c)
        refs = sum(len(r) for r in tr)
        distinct = len({e for r in tr for e in r})
        for fn in (CS.lru_hits, CS.lfu_hits, CS.belady_hits):
            assert fn(tr, E) == refs - distinct


def test_study_reports_every_policy():
    tr = [np.array(TR), np.array(TR)]
    out = CS.study(tr, E=8, cap=0.25)
    assert out["capacity"] == 2 and out["references"] == 12
    assert abs(out["lru"]["hit_rate"] - 2 / 12) < 1e-12
    assert abs(out["belady"]["misses_per_token"] - (12 - 4) / 6) < 1e-12
