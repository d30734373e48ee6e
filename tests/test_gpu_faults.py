"""Device-side error paths: bounded waits that run out, bad and non-resident expert ids.
Nothing here faults, traps or hangs the GPU: the stall is a wait on a flag that nothing
sets, bounded to 1 ms, and bad ids are rejected before any address is formed."""
import numpy as np
import pytest

from oracle import layer as OL, model_inputs as OM, routing as OR
from routing_predicted_experts_gb300 import synth as S

from _common import bf16_dev, check_protocol, to_dev

pytestmark = pytest.mark.gpu


def _setup(seed=21):
    import torch
    from routing_predicted_experts_gb300 import binding as B, model as M
    sh = S.TINY
    lay = M.build_layer(seed, 0, sh)
    h = OM.hidden(seed, 0, sh.d)
    z = OM.supplied_logits(seed, "cur", sh.E)
    ids, _ = OR.softmax_topk(z, sh.K)
    dm = B.dims(sh.d, sh.E, sh.F, sh.K)
    return sh, lay, h, z, ids, dm


def _run(B, dm, lay, h, z, ids, ws, routed=None):
    import torch
    return B.e0_moe_decode_layer(dm, routed or lay["routed"], lay["shared"], lay["lora"], None, bf16_dev(h)[None],
                                 to_dev(ids, torch.int32)[None], to_dev(z, torch.float32)[None], None, ws)


def test_timeout_sets_status_and_workspace_recovers():
    import torch
    from routing_predicted_experts_gb300 import binding as B
    sh, lay, h, z, ids, dm = _setup()
    ws = B.e0_workspace(dm)
    B.e0_debug_inject_stall(ws, 1_000_000)  # 1 ms wait on a flag nothing sets
    _run(B, dm, lay, h, z, ids, ws)
    st = B.e0_get_device_status(ws)
    assert st & 1, st  # E0_DEV_TIMEOUT
    B.e0_workspace_reset(ws)
    out = _run(B, dm, lay, h, z, ids, ws)
    assert B.e0_get_device_status(ws) == 0
    olay = OM.layer(21, 0, sh, with_head=False)
    ref = OL.layer_step(h, olay, ids, z, None, sh.K)
    check_protocol(out["delta"][0].cpu().numpy(), ref["delta"], "delta after recovery")


def test_bad_and_duplicate_ids_are_skipped():
    from routing_predicted_experts_gb300 import binding as B
    sh, lay, h, z, ids, dm = _setup()
    ws = B.e0_workspace(dm)
    bad = ids.copy()
    bad[1] = sh.E + 5
    bad[3] = bad[0]
    out = _run(B, dm, lay, h, z, bad, ws)
    assert B.e0_get_device_status(ws) & 2  # E0_DEV_BAD_ID
    olay = OM.layer(21, 0, sh, with_head=False)
    ref = OL.layer_step(h, olay, np.array([bad[0], bad[2]]), z, None, 2)
    check_protocol(out["delta"][0].cpu().numpy(), ref["delta"], "delta with skipped ids")


def test_slot_table_indirection_and_non_resident():
    """A pool holding a permuted subset of experts gives the same result as the full
    stack; an id whose slot is -1 is reported and skipped."""
    import torch
    from routing_predicted_experts_gb300 import binding as B
    sh, lay, h, z, ids, dm = _setup()
    r = lay["routed"]
    S_ = 6
    pool_ids = [int(ids[2]), int(ids[0]), 5 if 5 not in ids else 7, int(ids[3]), int(ids[1]), 9 if 9 not in ids else 10]
    gq, gs = 2 * sh.F * sh.d // 8, 2 * sh.F * sh.d // 64
    dq, ds = sh.d * sh.F // 8, sh.d * sh.F // 64

    def take(t, per, lst):
        return torch.cat([t[e * per:(e + 1) * per] for e in lst]).contiguous()
    pool = B.Experts(B.Q4(take(r.gate_up.q, gq, pool_ids), take(r.gate_up.scale, gs, pool_ids),
                          take(r.gate_up.bias, gs, pool_ids)),
                     B.Q4(take(r.down.q, dq, pool_ids), take(r.down.scale, ds, pool_ids),
                          take(r.down.bias, ds, pool_ids)), S_)
    slot_of = np.full(sh.E, -1, np.int16)
    for s, e in enumerate(pool_ids):
        slot_of[e] = s
    pool.slot_of = to_dev(slot_of, torch.int16)
    ws = B.e0_workspace(dm)
    full = _run(B, dm, lay, h, z, ids, ws)
    viap = _run(B, dm, lay, h, z, ids, ws, routed=pool)
    assert B.e0_get_device_status(ws) == 0
    a, b = full["delta"].cpu().numpy(), viap["delta"].cpu().numpy()
    assert np.allclose(a, b, rtol=0, atol=1e-5 * np.abs(a).max())
    slot_of[ids[1]] = -1
    pool.slot_of = to_dev(slot_of, torch.int16)
    miss = _run(B, dm, lay, h, z, ids, ws, routed=pool)
    assert B.e0_get_device_status(ws) & 4  # E0_DEV_NOT_RESIDENT
    olay = OM.layer(21, 0, sh, with_head=False)
    ref = OL.layer_step(h, olay, np.array([ids[0], ids[2], ids[3]]), z, None, 3)
    check_protocol(miss["delta"][0].cpu().numpy(), ref["delta"], "delta without the missing expert")
