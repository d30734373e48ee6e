"""Expert-cache policy simulation over decode routing traces (host side).

"Cacheable by Design?", Appendix E "Cache Simulation": each layer's router trace (a
(T, k) array of expert ids) is replayed through an independent per-layer cache of
capacity c = ceil(cap * E); a reference to an expert that is not resident is a demand
miss and loads it.  Policies:
  LRU     evict the least recently used resident expert;
  LFU     evict the least frequently used one, by cumulative reference counts (ties to
          the least recently used);
  static  hold the c experts most frequently referenced in a warm-up prefix, never
          evict (a miss is served without being cached);
  Belady  evict the resident expert whose next reference lies farthest in the future
          (clairvoyant: the bound no online policy reaches).
The references of a token are replayed in the order the trace lists them.

Readings where the page is silent: the warm-up prefix of the static policy is the first
`warmup` tokens (default a tenth of the trace) and its ties go to the lower id; LFU
counts every reference from the start of the trace; hits and misses are counted over
the whole trace for every policy.  ``pool_lru`` replays the rule the HBM slot pool of
this library applies instead (least recently used, but the experts of the token being
staged and of the previous token are never evicted), so that its counters can be
checked against it.
"""
from __future__ import annotations

import math

import numpy as np


def capacity(cap: float, E: int) -> int:
    """c = ceil(cap * E) slots per layer."""
    return int(math.ceil(cap * E - 1e-12))


def lru_hits(trace, c: int) -> int:
    last: dict[int, int] = {}
    resident: list[int] = []
    hits = clock = 0
    for row in trace:
        for e in map(int, row):
            clock += 1
            if e in resident:
                hits += 1
            else:
                if len(resident) >= c:
                    resident.remove(min(resident, key=lambda r: last[r]))
                resident.append(e)
            last[e] = clock
    return hits


def lfu_hits(trace, c: int) -> int:
    count: dict[int, int] = {}
    last: dict[int, int] = {}
    resident: list[int] = []
    hits = clock = 0
    for row in trace:
        for e in map(int, row):
            clock += 1
            count[e] = count.get(e, 0) + 1
            if e in resident:
                hits += 1
            else:
                if len(resident) >= c:
                    resident.remove(min(resident, key=lambda r: (count[r], last[r])))
                resident.append(e)
            last[e] = clock
    return hits


def static_hits(trace, c: int, warmup: int | None = None) -> int:
    T = len(trace)
    w = max(1, T // 10) if warmup is None else warmup
    counts: dict[int, int] = {}
    for row in trace[:w]:
        for e in map(int, row):
            counts[e] = counts.get(e, 0) + 1
    held = set(sorted(counts, key=lambda e: (-counts[e], e))[:c])
    return sum(1 for row in trace for e in map(int, row) if e in held)


def belady_hits(trace, c: int) -> int:
    flat = [int(e) for row in trace for e in row]
    n = len(flat)
    nxt = [n] * n          # position of the next reference to the same expert
    seen: dict[int, int] = {}
    for p in range(n - 1, -1, -1):
        nxt[p] = seen.get(flat[p], n)
        seen[flat[p]] = p
    resident: dict[int, int] = {}  # expert -> position of its next reference
    hits = 0
    for p, e in enumerate(flat):
        if e in resident:
            hits += 1
        elif len(resident) >= c:
            far = max(resident, key=lambda r: (resident[r], r))
            del resident[far]
        resident[e] = nxt[p]
    return hits


def pool_lru_hits(trace, slots: int) -> int:
    """The slot pool's rule: LRU over the staged sets, never evicting the experts of the
    set being staged or of the previous one (slots >= 2K)."""
    resident: list[int] = []
    stamp: dict[int, int] = {}
    clock = hits = 0
    prev: list[int] = []
    for row in trace:
        ids = [int(e) for e in row]
        pinned = set(ids) | set(prev)
        for e in ids:
            if e in resident:
                hits += 1
            else:
                if len(resident) >= slots:
                    victim = min((r for r in resident if r not in pinned), key=lambda r: stamp[r])
                    resident.remove(victim)
                resident.append(e)
            clock += 1
            stamp[e] = clock
        prev = ids
    return hits


POLICIES = {"lru": lru_hits, "lfu": lfu_hits, "static": static_hits, "belady": belady_hits}


def study(traces, E: int, cap: float) -> dict:
    """Hit rates of every policy over per-layer traces [(T, k) arrays], with
    c = ceil(cap * E); also the misses per token (summed over layers)."""
    c = capacity(cap, E)
    refs = sum(int(np.asarray(tr).size) for tr in traces)
    T = len(traces[0]) if traces else 0
    out = {"capacity": c, "references": refs}
    for name, fn in POLICIES.items():
        hits = sum(fn(tr, c) for tr in traces)
        out[name] = {"hit_rate": hits / max(1, refs), "misses_per_token": (refs - hits) / max(1, T)}
    hits = sum(pool_lru_hits(tr, c) for tr in traces)
    out["pool_lru"] = {"hit_rate": hits / max(1, refs), "misses_per_token": (refs - hits) / max(1, T)}
    return out
