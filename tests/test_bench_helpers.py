"""The bench's byte accounting and cache simulation (CPU only): the algorithmic bytes per
token against the sizes the pages print, and the LRU / Belady hit counts against brute
force on small traces."""
import itertools
import json
import os

import numpy as np

import bench

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "page_numbers.json")


def test_expert_bytes_match_the_printed_sizes():
    g = json.load(open(GOLDEN))
    d, E, F, L = g["d"], g["E"], g["F"], g["layers"]
    # one routed expert: the per-token bytes of a K=1, shared-free, LoRA-free, head-free
    # stack of one layer minus the same with K=0
    one = bench.algorithmic_bytes_per_token(d=d, E=E, F=F, K=1, r=0, L=1, heads=0, routers=0, shared=False)
    zero = bench.algorithmic_bytes_per_token(d=d, E=E, F=F, K=0, r=0, L=1, heads=0, routers=0, shared=False)
    expert = one - zero
    assert abs(expert / 1e6 - g["expert_bytes_MB_printed"]) < 0.01
    assert abs(E * expert / 1e6 - g["layer_expert_bytes_MB_printed"]) < 1.0
    assert abs(L * E * expert / 2**30 - g["stack_expert_bytes_GiB_printed"]) < 0.1
    assert abs(4 * expert / 1e6 - g["k4_layer_expert_bytes_MB_printed"]) < 0.1


def test_bytes_per_token_decomposes():
    """K=8 adds 4 experts per layer to K=4, and each of the 33 heads gathers 2 x 4 more
    one-hot columns of fc1 (bf16, H rows each); each gate adds its own bytes."""
    b4 = bench.algorithmic_bytes_per_token(K=4)
    b8 = bench.algorithmic_bytes_per_token(K=8)
    one = bench.algorithmic_bytes_per_token(K=1, r=0, L=1, heads=0, routers=0, shared=False)
    zero = bench.algorithmic_bytes_per_token(K=0, r=0, L=1, heads=0, routers=0, shared=False)
    assert b8 - b4 == 40 * 4 * (one - zero) + 33 * (2 * 4) * 2 * 1024
    gate = bench.algorithmic_bytes_per_token(routers=9) - b4
    assert gate == 2 * 256 * 2048  # one bf16 [E][d] gate
    assert (b4, b8) == (652839424, 936495616)


def _brute_pool_hits(trace, slots):
    """Hits of the pool's rule written out directly: on a miss with a full pool, evict
    among residents outside the current and previous sets the least recently used."""
    resident, last, hits, prev = set(), {}, 0, set()
    clock = 0
    for t, ids in enumerate(trace):
        pinned = set(ids) | prev
        for e in ids:
            clock += 1
            if e in resident:
                hits += 1
            else:
                if len(resident) >= slots:
                    cand = sorted(r for r in resident if r not in pinned)
                    resident.discard(min(cand, key=lambda r: last[r]))
                resident.add(e)
            last[e] = clock
        prev = set(ids)
    return hits


def test_pool_rule_hit_counts():
    from routing_predicted_experts_gb300 import cachesim as CS
    rng = np.random.default_rng(3)
    for _ in range(20):
        E, K, T, slots = 10, 2, 30, 5
        trace = [list(rng.choice(E, K, replace=False)) for _ in range(T)]
        assert CS.pool_lru_hits(trace, slots) == _brute_pool_hits(trace, slots)
        assert CS.belady_hits(trace, slots) >= CS.lru_hits(trace, slots)
    # a cyclic trace over c + 1 experts: LRU misses every time after warm-up, Belady does not
    trace = [[e] for e in itertools.islice(itertools.cycle(range(4)), 40)]
    assert CS.lru_hits(trace, 3) == 0 and CS.belady_hits(trace, 3) > 0


def test_traffic_record_applies_only_to_the_kernel_it_was_taken_on():
    """The roofline's `traffic` comes from the committed capture's traffic/algorithmic
    ratio, scaled to the workload, and only while the kernel sources hash to the value
    recorded beside it (a changed kernel reports null until it is captured again)."""
    import bench
    import os
    p = os.path.join(bench.ROOT, "profiles", "engine_stack_traffic.txt")
    kv = dict(line.split(":", 1) for line in open(p) if ":" in line and not line.startswith("#"))
    ratio = float(kv["traffic_over_algorithmic"])
    assert 1.0 <= ratio < 1.05  # no re-reads beyond prefetched lines
    if kv["kernel_src_sha"].strip() == bench._kernel_source_hash():
        assert bench._traffic_per_launch(1000000) == round(ratio * 1000000)
    else:
        assert bench._traffic_per_launch(1000000) is None
