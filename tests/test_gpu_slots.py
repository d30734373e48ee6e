"""Bounded expert-slot pool: a decode stack whose prerouted layers read their experts
from a few HBM slots filled from pinned host memory must produce what the fully
resident stack produces, on the same synthetic routing trace (injected through the
logit bias), while the pool misses, evicts and hits as the trace dictates."""
import numpy as np
import pytest

from routing_predicted_experts_gb300 import synth as S

from oracle import bf16 as OB

from _common import bf16_host, check_bf16_protocol

pytestmark = pytest.mark.gpu


def _lru_reference(trace_l, slots, K):
    """Host LRU with the pool's pinning rule (previous and next sets never evicted):
    hits and misses per step, to check the library's counters."""
    resident, stamp, clock = [], {}, 0
    hits = misses = 0
    prev = []
    for ids in trace_l:
        pinned = set(ids) | set(prev)
        for e in ids:
            if e in resident:
                hits += 1
            else:
                misses += 1
                if len(resident) >= slots:
                    victim = min((r for r in resident if r not in pinned), key=lambda r: stamp[r])
                    resident.remove(victim)
                resident.append(e)
            clock += 1
            stamp[e] = clock
        prev = list(ids)
    return hits, misses


@pytest.mark.parametrize("slots", [8, 11])
def test_pooled_stack_matches_resident_stack(slots):
    import torch
    from routing_predicted_experts_gb300 import binding as B, model as M
    sh, seed, L, steps = S.TINY, 5, 6, 12
    owners = {1, 2, 3, 4}
    pre = [1 if (l - 1) in owners else 0 for l in range(L)]
    pooled = [l for l in range(L) if pre[l]]
    dm = B.dims(sh.d, sh.E, sh.F, sh.K)
    layers = [M.build_layer(seed, l, sh, with_head=(l in owners)) for l in range(L)]
    dense = [B.e0_layer_struct(ly["routed"], ly["shared"], ly["lora"], ly["head"], ly["router"]) for ly in layers]
    ref_stack = B.Stack(dm, dense, pre, keepalive=layers)
    bundles = B.host_bundles(dm, [layers[l]["routed"] for l in pooled])
    pool = B.SlotPool(dm, len(pooled), slots, bundles)
    structs = []
    for l, ly in enumerate(layers):
        routed = pool.view(pooled.index(l)) if l in pooled else ly["routed"]
        structs.append(B.e0_layer_struct(routed, ly["shared"], ly["lora"], ly["head"], ly["router"]))
    pool_stack = B.Stack(dm, structs, pre, keepalive=(layers, pool))
    trace = np.stack([S.locality_trace(seed, l, steps + 1, sh.E, sh.K) for l in range(L)], axis=1)  # [t][l][K]
    ws_a, ws_b = ref_stack.workspace(), pool_stack.workspace()
    copy = torch.cuda.Stream()
    comp = torch.cuda.current_stream()
    for t in range(steps):
        bias = np.zeros((2, L, sh.E), dtype=np.float32)
        for l in range(L):
            bias[0, l, trace[t, l]] = 1e4      # own-gate routing at this token
            bias[1, l, trace[t + 1, l]] = 1e4  # what the heads commit for the next token
        bias_d = torch.from_numpy(bias).cuda()
        for i, l in enumerate(pooled):
            pool.stage(i, trace[t, l], copy_stream=copy)
        ev = torch.cuda.Event()
        ev.record(copy)
        comp.wait_event(ev)
        h0 = M.hidden(seed, t, sh.d)
        incr = M.increments(seed, t, L, sh.d)
        outs = []
        for stack, ws in ((ref_stack, ws_a), (pool_stack, ws_b)):
            h_out = torch.empty(sh.d, dtype=torch.int16, device="cuda")
            ids = torch.empty((L, sh.K), dtype=torch.int32, device="cuda")
            stack.step(t, h0, incr, h_out, ws, ids_out=ids, logit_bias=bias_d)
            outs.append((h_out, ids))
        torch.cuda.synchronize()
        assert B.e0_get_device_status(ws_a) == 0 and B.e0_get_device_status(ws_b) == 0
        for (h_out, ids) in outs:
            got = ids.cpu().numpy()
            for l in range(L):
                assert sorted(got[l].tolist()) == sorted(trace[t, l].tolist()), (t, l)
        # same experts and arithmetic; only the order of fp32 reductions may differ
        check_bf16_protocol(bf16_host(outs[1][0]), bf16_host(outs[0][0]), f"h_out t{t}")
        a = OB.bf16_to_f64(bf16_host(outs[0][0]))
        b = OB.bf16_to_f64(bf16_host(outs[1][0]))
        assert np.abs(a - b).max() <= 4 * 2.0 ** -8 * np.abs(a).max(), t
    hits = misses = 0
    for l in pooled:
        h, m = _lru_reference(trace[:steps, l], slots, sh.K)
        hits, misses = hits + h, misses + m
    st = pool.stats
    assert (st.hits, st.misses) == (hits, misses)
    total, _ = B.expert_bundle_layout(dm)
    assert st.h2d_bytes == misses * total
    assert st.evictions > 0
    pool_stack.close()
    pool.close()
