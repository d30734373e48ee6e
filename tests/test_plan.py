"""The CTA work plan of the decode engine (built on the host, no GPU): every row of every
weight a layer streams is assigned to exactly one unit, no CTA holds more units than the
engine supports, and the ordering and placement rules the kernel relies on hold."""
import ctypes

import numpy as np
import pytest

from routing_predicted_experts_gb300 import _lib
from routing_predicted_experts_gb300 import build as BLD

U_EXPERT, U_QROWS, U_LORA_A, U_HEAD, U_LRES, U_ROUTER, U_LORA_B = 1, 2, 3, 4, 5, 6, 7
MAXU = 8
UNIT = np.dtype([("type", "u1"), ("k", "u1"), ("r0", "<u2"), ("r1", "<u2"), ("flags", "<u2")])


def plan(kind, d=2048, E=256, F=512, K=4, H=1024, lr=16, ncta=152):
    BLD.build()
    lib = _lib.lib()
    units = np.zeros(ncta * MAXU, dtype=UNIT)
    counts = np.zeros(ncta, dtype=np.uint8)
    defer = np.zeros(ncta, dtype=np.uint8)
    st = lib.e0_debug_plan(d, E, F, K, H, lr, ncta, kind, ctypes.c_void_p(units.ctypes.data),
                           ctypes.c_void_p(counts.ctypes.data), ctypes.c_void_p(defer.ctypes.data))
    assert st == 0, lib.e0_last_error()
    per_cta = [units[c * MAXU:c * MAXU + int(counts[c])] for c in range(ncta)]
    return per_cta, defer


def covered(per_cta, t):
    rows = []
    for us in per_cta:
        for u in us:
            if u["type"] == t:
                rows.extend(range(int(u["r0"]), int(u["r1"])))
    return sorted(rows)


def check_common(per_cta, d, E, F, K, lr):
    for us in per_cta:
        assert len(us) <= MAXU
        assert all(u["r0"] < u["r1"] for u in us)
    # every expert slab of every routed slot and of the shared expert, once
    slabs = sorted((int(u["k"]), int(u["r0"])) for us in per_cta for u in us if u["type"] == U_EXPERT)
    assert slabs == [(k, s) for k in range(K + 1) for s in range(F // 32)]
    # LoRA base rows and B rows, each exactly once; all ranks of A
    assert covered(per_cta, U_QROWS) == list(range(d))
    assert covered(per_cta, U_LORA_B) == list(range(d))
    a_rows = covered(per_cta, U_LORA_A)
    assert sorted(set(a_rows)) == list(range(lr))
    # B rows on a CTA without a local v wait for the published one: when an A unit keeps
    # v local, nobody publishes it, so every CTA with B rows must then compute its own
    if any(u["flags"] & 1 for us in per_cta for u in us if u["type"] == U_LORA_A):
        for us in per_cta:
            if any(u["type"] == U_LORA_B for u in us):
                assert any(u["type"] == U_LORA_A and u["flags"] & 1 for u in us)
    # a CTA's LoRA A precedes its LoRA B (B reads the v that A computes or publishes)
    for us in per_cta:
        types = [int(u["type"]) for u in us]
        if U_LORA_A in types and U_LORA_B in types:
            assert types.index(U_LORA_A) < types.index(U_LORA_B)
        # expert slabs come last: id-independent work first
        if U_EXPERT in types:
            assert all(t == U_EXPERT for t in types[types.index(U_EXPERT):])


@pytest.mark.parametrize("K", [4, 8])
def test_plan_with_head_covers_every_row(K):
    d, E, F, H, lr = 2048, 256, 512, 1024, 16
    per_cta, defer = plan(0, d, E, F, K, H, lr)
    check_common(per_cta, d, E, F, K, lr)
    assert covered(per_cta, U_HEAD) == list(range(H))
    assert covered(per_cta, U_LRES) == list(range(E))
    for us in per_cta:
        for u in us:
            if u["type"] in (U_HEAD, U_LRES):
                assert u["r1"] - u["r0"] <= 64  # the head buffers hold 64 rows


def test_plan_split_keeps_the_prerouter_off_the_critical_ctas():
    """K = 4 leaves room: prerouter rows only on deferred CTAs, which hold nothing else;
    LoRA base rows in runs of whole 16-row stages of at most an expert slab's bytes (so
    those CTAs finish with the expert CTAs); every A unit that keeps v local holds all
    ranks, and no CTA without such a unit holds B rows (nobody would publish its v)."""
    d, lr = 2048, 16
    per_cta, defer = plan(0, d=d, K=4, lr=lr)
    assert defer.sum() > 0
    for c, us in enumerate(per_cta):
        types = {int(u["type"]) for u in us}
        if defer[c]:
            assert types <= {U_HEAD, U_LRES}
        else:
            assert not types & {U_HEAD, U_LRES}
        for u in us:
            if u["type"] == U_QROWS:
                n = u["r1"] - u["r0"]
                assert n % 16 == 0 and u["r0"] % 16 == 0 and 64 <= n
                assert n * (d // 2 + d // 16) <= 64 * (d // 2 + d // 16) + 20 * d  # <= one expert slab
        local = [u for u in us if u["type"] == U_LORA_A and u["flags"] & 1]
        if U_LORA_B in types:
            assert local and local[0]["r0"] == 0 and local[0]["r1"] == lr
    # the deferred CTAs are the last ones
    first = int(np.argmax(defer))
    assert defer[first:].all() and not defer[:first].any()


def test_plan_without_head_and_router_rows():
    d, E, F, K, lr = 2048, 256, 512, 4, 16
    per_cta, defer = plan(1, d, E, F, K, 1024, lr)
    check_common(per_cta, d, E, F, K, lr)
    assert not defer.any()
    # without a local-v unit every B row waits for a published v: no A unit keeps v local
    assert not any(u["flags"] & 1 for us in per_cta for u in us if u["type"] == U_LORA_A)
    rows, _ = plan(2, d, E, F, K, 1024, lr)
    assert covered(rows, U_ROUTER) == list(range(E))
    # gate rows stay off the CTAs that hold only prerouter work in head layers
    _, defer0 = plan(0, d, E, F, K, 1024, lr)
    for c, us in enumerate(rows):
        if len(us):
            assert not defer0[c]


@pytest.mark.parametrize("K", [4, 8])
def test_plan_after_a_head_layer_stays_off_the_deferred_ctas(K):
    """A layer without a head after one with a head (the last layer of the stack): all of
    its work, every row once, on the CTAs that layers with a head keep on the critical
    path (the deferred CTAs run behind the layers with the prerouter's work)."""
    d, E, F, H, lr = 2048, 256, 512, 1024, 16
    per_cta, defer = plan(3, d, E, F, K, H, lr)
    check_common(per_cta, d, E, F, K, lr)
    assert not defer.any()
    _, defer0 = plan(0, d, E, F, K, H, lr)
    for c, us in enumerate(per_cta):
        if defer0[c]:
            assert len(us) == 0
    if not defer0.any():  # no room for deferred CTAs: the same plan as kind 1
        plain, _ = plan(1, d, E, F, K, H, lr)
        assert [list(map(tuple, us)) for us in plain] == [list(map(tuple, us)) for us in per_cta]


def test_plan_tiny_layer():
    d, E, F, K, H, lr = 256, 16, 128, 4, 64, 4
    for kind in (0, 1):
        per_cta, _ = plan(kind, d, E, F, K, H, lr, ncta=152)
        check_common(per_cta, d, E, F, K, lr)
