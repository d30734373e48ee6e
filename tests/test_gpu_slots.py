"""Bounded expert-slot pool: consistency of the pool's record, its device id -> slot table,
its ready words and the bytes in its slots, including after a staging call whose bundle
copy fails (injected on the host: the copy call reports an error, nothing runs wrong on
the GPU).  The pooled decode stack itself is checked against the oracle in
test_gpu_stack.py (staged from the routing the GPU commits)."""
import numpy as np
import pytest

from routing_predicted_experts_gb300 import synth as S

from _common import dev_array

pytestmark = pytest.mark.gpu


def _pool(slots=8):
    from routing_predicted_experts_gb300 import binding as B, model as M
    sh = S.LayerShape(d=256, E=16, F=128, K=4, H=0, r=0, alpha=1.0, shared=False)
    dm = B.dims(sh.d, sh.E, sh.F, sh.K)
    ly = M.build_layer(7, 0, sh, with_head=False, with_lora=False)
    bundles = B.host_bundles(dm, [ly["routed"]])
    return B, dm, sh, B.SlotPool(dm, 1, slots, bundles), bundles


def _check_consistent(B, dm, pool, bundles, want_tag):
    """Device table == the pool's record; every resident expert's bundle is byte-exact in
    its slot; the ready word holds the last completed staging's tag."""
    import torch
    torch.cuda.synchronize()
    total, offs = B.expert_bundle_layout(dm)
    view = pool.view(0).c()
    rec = pool.resident(0)
    # the table of the tag's parity (a pool keeps one per parity of the token index)
    dev_tab = dev_array(view.slot_of, 2 * dm.E, torch.int16).cpu().numpy().reshape(2, dm.E)[want_tag & 1]
    assert np.array_equal(dev_tab, rec), (dev_tab, rec)
    base = view.gate_up.q - offs[0]
    slots = dev_array(base, view.n * total, torch.uint8).cpu().numpy().reshape(view.n, total)
    host = bundles[0].numpy()
    for e in range(dm.E):
        if rec[e] >= 0:
            assert np.array_equal(slots[rec[e]], host[e]), e
    assert len(set(int(s) for s in rec if s >= 0)) == int((rec >= 0).sum())  # one expert per slot
    assert dev_array(view.ready, 1, torch.int32).cpu().numpy()[0] == want_tag


def test_staging_fills_slots_and_ready_words():
    B, dm, sh, pool, bundles = _pool()
    pool.stage_host([0], [[0, 1, 2, 3]], 0)
    _check_consistent(B, dm, pool, bundles, 0)
    pool.stage_host([0], [[4, 5, 6, 7]], 1)
    pool.stage_host([0], [[8, 9, 10, 11]], 2)   # evicts the least recently used: 0..3
    _check_consistent(B, dm, pool, bundles, 2)
    rec = pool.resident(0)
    assert all(rec[e] >= 0 for e in range(4, 12)) and all(rec[e] < 0 for e in range(4))
    st = pool.stats
    assert (st.hits, st.misses, st.evictions) == (0, 12, 4)
    pool.close()


def test_failed_bundle_copy_leaves_the_pool_consistent():
    """The second bundle copy of a staging call fails: the call returns the copy error,
    only the first miss counts as resident, the device table and the ready word keep
    their previous state, and a retry completes the staging with every slot byte-exact."""
    from routing_predicted_experts_gb300 import _lib
    B, dm, sh, pool, bundles = _pool()
    pool.stage_host([0], [[0, 1, 2, 3]], 0)
    pool.stage_host([0], [[4, 5, 6, 7]], 1)
    _check_consistent(B, dm, pool, bundles, 1)
    before = pool.resident(0).copy()
    pool.fail_copies(1)
    with pytest.raises(_lib.E0Error) as ei:
        pool.stage_host([0], [[8, 9, 10, 11]], 2)
    assert ei.value.status == _lib.E0_ERR_CUDA
    rec = pool.resident(0)
    # 8 took the least recently used unpinned slot (expert 0's); 9..11 were never copied
    assert rec[8] == before[0] and rec[0] < 0 and all(rec[e] < 0 for e in (9, 10, 11))
    import torch
    torch.cuda.synchronize()
    view = pool.view(0).c()
    assert dev_array(view.ready, 1, torch.int32).cpu().numpy()[0] == 1  # the layer was not released
    tabs = dev_array(view.slot_of, 2 * dm.E, torch.int16).cpu().numpy().reshape(2, dm.E)
    assert np.array_equal(tabs[1], before)  # the table tag 1 wrote is untouched
    pool.stage_host([0], [[8, 9, 10, 11]], 2)  # retry
    _check_consistent(B, dm, pool, bundles, 2)
    rec = pool.resident(0)
    assert all(rec[e] >= 0 for e in range(4, 12))
    st = pool.stats
    assert (st.misses, st.hits) == (8 + 1 + 3, 1)
    pool.close()


def test_bad_ids_are_refused_before_any_copy():
    from routing_predicted_experts_gb300 import _lib
    B, dm, sh, pool, bundles = _pool()
    pool.stage_host([0], [[0, 1, 2, 3]], 0)
    before = pool.resident(0).copy()
    with pytest.raises(_lib.E0Error) as ei:
        pool.stage_host([0], [[4, 5, 16, 7]], 1)
    assert ei.value.status == _lib.E0_ERR_INVALID
    assert np.array_equal(pool.resident(0), before)
    _check_consistent(B, dm, pool, bundles, 0)
    pool.close()
