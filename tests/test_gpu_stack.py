"""Decode stack (one launch per token) against the oracle in lock step.

Every checked layer is compared from identical inputs (the GPU's own layer input,
h_trace): the logits it routed by, its ids (exact wherever the decision's gap exceeds
1e-3, otherwise any valid choice, which the oracle then adopts), its combine weights
(1e-5 against the family's weights of the GPU's own logits), its fp32 delta and the
next layer's bf16 input.  Layers routed by a head are checked against the oracle head
evaluated at the previous token on the GPU's inputs.  Small stacks also run the oracle
free from the first hidden state (adopting the GPU's ids only where a decision is
ambiguous) and report the end-to-end drift of h_out.

The same runner covers the routing families (softmax-top-K, sigmoid-group), the routing
sources (head, own gate, route-ahead) and a stack whose head-routed layers read their
experts from a bounded slot pool staged by the routing the GPU committed (the copies of
token t run while launch t is already queued and waiting on the pool's ready words)."""
import numpy as np
import pytest

from oracle import bf16 as OB, layer as OL, model_inputs as OM, routing as OR
from routing_predicted_experts_gb300 import synth as S

from _common import REPORT, bf16_host, check_bf16_protocol, check_protocol, check_route, dev_array

pytestmark = pytest.mark.gpu


def _oracle_sources(route_src):
    return ["head" if s == 1 else ("ahead", -s) if s < 0 else "gate" for s in route_src]


def _lru_reference(staged, slots):
    """Hits and misses of the pool's rule (least recently used; the previous and the
    staged ids are never evicted) on a sequence of staged id lists."""
    resident, stamp, clock, hits, misses, prev = [], {}, 0, 0, 0, []
    for ids in staged:
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


def run_lockstep(seed, sh, L, head_owners, steps, route_src=None, check_layers=None, family=None,
                 pool_slots=None, drift=False, label=""):
    import torch
    from routing_predicted_experts_gb300 import binding as B, model as M
    if route_src is None:
        route_src = [1 if (l - 1) in head_owners else 0 for l in range(L)]
    K, d, E = sh.K, sh.d, sh.E
    layers = [M.build_layer(seed, l, sh, with_head=(l in head_owners)) for l in range(L)]
    pooled = [l for l in range(L) if route_src[l] == 1] if pool_slots else []
    dm = B.dims(d, E, sh.F, K, family)
    pool = None
    if pooled:
        pool = B.SlotPool(dm, len(pooled), pool_slots, B.host_bundles(dm, [layers[l]["routed"] for l in pooled]))
    structs = []
    for l, ly in enumerate(layers):
        routed = pool.view(pooled.index(l)) if l in pooled else ly["routed"]
        structs.append(B.e0_layer_struct(routed, ly["shared"], ly["lora"], ly["head"], ly["router"]))
    stack = B.Stack(dm, structs, route_src, keepalive=(layers, pool))
    ws = stack.workspace()
    comp = torch.cuda.current_stream()
    copy = torch.cuda.Stream() if pool else None
    src = _oracle_sources(route_src)
    olays = {}

    def olay(l):
        if l not in olays:
            olays[l] = OM.layer(seed, l, sh, with_head=(l in head_owners))
        return olays[l]

    routers = [OM.router_weights(seed, l, sh) for l in range(L)]
    # step-0 routing of pooled layers is forced (logit bias) onto known ids, which prime the
    # pool: the first token's routing is not committed by any head
    prime = {l: np.arange(K, dtype=np.int32) + (l % max(1, E // K - 1)) * K for l in pooled}
    # ---- every launch (and, for a pool, the staging of each next token) is queued first,
    # the way a decode loop runs: token t's experts are staged from the ids launch t-1
    # commits, layer by layer, while launch t-1 still runs and launch t waits for them
    box = B.CommitBox(L) if pool else None
    runs = []
    for t in range(steps):
        run = {"h0": M.hidden(seed, t, d), "incr": M.increments(seed, t, L, d),
               "h_out": torch.empty(d, dtype=torch.int16, device="cuda"),
               "ids": torch.empty((L, K), dtype=torch.int32, device="cuda"),
               "w": torch.empty((L, K), dtype=torch.float32, device="cuda"),
               "h_tr": torch.empty((L, d), dtype=torch.int16, device="cuda"),
               "delta": torch.empty((L, d), dtype=torch.float32, device="cuda"),
               "logits": torch.zeros((2, L, E), dtype=torch.float32, device="cuda"),
               "next": torch.empty((L, K), dtype=torch.int32, device="cuda"), "bias": None}
        if pool and t == 0:
            b = np.zeros((2, L, E), dtype=np.float32)
            for l in pooled:
                b[0, l, prime[l]] = 1e4
            run["bias"] = torch.from_numpy(b).cuda()
            pool.stage_host(list(range(len(pooled))), np.stack([prime[l] for l in pooled]), 0, copy_stream=copy)
            ev = torch.cuda.Event()
            ev.record(copy)
            comp.wait_event(ev)  # (t = 0 only; later launches wait on the ready words)
        stack.step(t, run["h0"], run["incr"], run["h_out"], ws, ids_out=run["ids"], w_out=run["w"],
                   h_trace=run["h_tr"], logit_bias=run["bias"], delta=run["delta"], logits=run["logits"],
                   next_ids=run["next"], commit_box=box)
        if pool and t > 0:
            pool.stage_committed(box, list(range(len(pooled))), pooled, t, copy_stream=copy)
        runs.append(run)
    torch.cuda.synchronize()
    assert B.e0_get_device_status(ws) == 0, label
    if pool:
        for i, l in enumerate(pooled):
            view = pool.view(i).c()
            dev_tab = dev_array(view.slot_of, 2 * E, torch.int16).cpu().numpy().reshape(2, E)
            assert np.array_equal(dev_tab[(steps - 1) & 1], pool.resident(i)), (label, l)
            assert dev_array(view.ready, 1, torch.int32).cpu().numpy()[0] == steps - 1
        box.close()

    zhat_prev, ids_prev, prev_next, prev_logits1 = {}, {}, None, None
    ambiguous = decisions = 0
    staged = {l: [prime[l].tolist()] for l in pooled}
    free = {"zhat": {}, "ids": {}}  # the free-running oracle's state (drift)
    for t in range(steps):
        run = runs[t]
        h0, incr, h_out, bias = run["h0"], run["incr"], run["h_out"], run["bias"]
        H, I, W = bf16_host(run["h_tr"]), run["ids"].cpu().numpy(), run["w"].cpu().numpy()
        DL, ZL, NX = run["delta"].cpu().numpy(), run["logits"].cpu().numpy(), run["next"].cpu().numpy()
        inc = bf16_host(incr)
        if pool and t > 0:
            for l in pooled:
                staged[l].append(I[l].tolist())
        bias_np = bias.cpu().numpy() if bias is not None else None
        zhat_now = {}
        xs = {}
        for l in range(L):
            checked = check_layers is None or l in check_layers
            feeds = check_layers is not None and (l + 1) in check_layers and l in head_owners
            if not (checked or feeds):
                continue
            x = OL.rmsnorm(OB.bf16_to_f64(H[l]))
            xs[l] = x
            if not checked:
                # only the head's prediction is needed (it routes the checked layer l + 1 at
                # the next token): evaluated on the GPU's input and routing of layer l
                prev = ids_prev.get(l) if t > 0 else None
                zhat_now[l] = OL.prerouter_logits(x, I[l], prev, olay(l)["head"])
                continue
            headed = src[l] == "head" and t > 0
            if headed:
                z = zhat_prev.get(l - 1)
                zg = prev_logits1[l].astype(np.float64)
            elif isinstance(src[l], tuple):
                j = l - src[l][1]
                z = OL.router_logits(OL.rmsnorm(OB.bf16_to_f64(H[j])), routers[l])
                zg = ZL[0, l].astype(np.float64)
            else:
                z = OL.router_logits(x, routers[l])
                if bias_np is not None:
                    z = z + bias_np[0, l]
                zg = ZL[0, l].astype(np.float64)
            if z is None:
                continue
            gi = I[l].astype(np.int64)
            # the logits the GPU routed by, then its decision and weights
            check_protocol(zg, z, f"{label} logits t{t} l{l}")
            decisions += 1
            if not check_route(gi, z, K, f"{label} ids t{t} l{l}", family):
                ambiguous += 1
            w_ref = OR.route_weights(zg, gi, family)
            assert np.abs(W[l] - w_ref).max() <= 1e-5, (label, t, l, W[l], w_ref)
            if headed:
                assert np.array_equal(I[l], prev_next[l]), (label, t, l)
            prev = ids_prev.get(l) if t > 0 else None
            ref = OL.layer_step(H[l], olay(l), gi, z, prev, K, family, family)
            check_protocol(DL[l], ref["delta"], f"{label} delta t{t} l{l}")
            if ref["next_logits"] is not None and l + 1 < L:
                zhat_now[l] = ref["next_logits"]
                if route_src[l + 1] == 1:
                    check_protocol(ZL[1, l + 1], ref["next_logits"], f"{label} committed logits t{t} l{l + 1}")
                    check_route(NX[l + 1], ref["next_logits"], K, f"{label} next ids t{t} l{l + 1}", family)
            if l + 1 < L:
                nxt = OL.residual_increment(ref["h_out"], inc[l + 1])
                check_bf16_protocol(H[l + 1], nxt, f"{label} h_in t{t} l{l + 1}")
            else:
                check_bf16_protocol(bf16_host(h_out), ref["h_out"], f"{label} h_out t{t}")
        if drift:
            def adopt(l, zz, oids, I=I):
                return I[l] if OR.route_gap(zz, K, family) <= 1e-3 else oids
            fr = OL.stack_token(bf16_host(h0), inc, [olay(l) for l in range(L)], routers, src, K,
                                zhat_prev=free["zhat"], ids_prev=free["ids"], family=family, adopt=adopt)
            free["zhat"] = fr["zhat_next"]
            free["ids"] = {l: rec["ids"] for l, rec in enumerate(fr["layers"])}
            got = OB.bf16_to_f64(bf16_host(h_out))
            ref = OB.bf16_to_f64(fr["h_out"])
            err = np.abs(got - ref)
            REPORT.append(f"{label} step {t}: end-to-end drift over {L} layers: max|err|/max|ref| "
                          f"{err.max() / np.abs(ref).max():.2e}, mean|err|/mean|ref| {err.mean() / np.abs(ref).mean():.2e}")
            check_protocol(got, ref, f"{label} free-running h_out t{t}")
        zhat_prev = zhat_now
        ids_prev = {l: I[l].copy() for l in range(L)}
        prev_next = NX
        prev_logits1 = ZL[1].copy()
    REPORT.append(f"{label}: {decisions} routing decisions checked over {steps} steps, {ambiguous} ambiguous "
                  f"(gap <= 1e-3) adopted from the GPU")
    if pool:
        hits = misses = 0
        for l in pooled:
            h, m = _lru_reference(staged[l], pool_slots)
            hits, misses = hits + h, misses + m
        st = pool.stats
        assert (st.hits, st.misses) == (hits, misses), ((st.hits, st.misses), (hits, misses))
        total, _ = B.expert_bundle_layout(dm)
        assert st.h2d_bytes == misses * total and st.evictions > 0
        REPORT.append(f"{label}: slot pool {pool_slots} slots/layer, {hits} hits, {misses} misses, "
                      f"{st.evictions} evictions")
    stack.close()
    if pool:
        pool.close()
    return ambiguous


def test_tiny_stack_lockstep_with_drift():
    sh = S.TINY
    # heads on layers 1..4 of 6: layers 2..5 route from the previous layer's head
    run_lockstep(seed=11, sh=sh, L=6, head_owners={1, 2, 3, 4}, steps=5, drift=True, label="tiny")


def test_tiny_stack_k1_and_k16():
    for K in (1, 16):
        sh = S.LayerShape(d=256, E=16, F=128, K=K, H=64, r=4, alpha=8.0, shared=True)
        run_lockstep(seed=12 + K, sh=sh, L=3, head_owners={0, 1}, steps=3, drift=True, label=f"tiny K={K}")


@pytest.mark.parametrize("N", [1, 2])
def test_route_ahead_stack(N):
    """Training-free route-ahead: layers >= N rank their own gate on the input N layers
    earlier; the first N route normally.  No heads."""
    sh = S.LayerShape(d=256, E=16, F=128, K=4, H=0, r=4, alpha=8.0, shared=True)
    L = 6
    src = [0 if l < N else -N for l in range(L)]
    run_lockstep(seed=31 + N, sh=sh, L=L, head_owners=set(), steps=3, route_src=src, drift=True,
                 label=f"route-ahead N={N}")


def test_sigmoid_group_stack():
    """The 8B tier's routing family (n = 8 groups, G = 4 kept, s = 2.5, K = 8) through the
    head commit, the own-gate routing and the combine."""
    sh = S.LayerShape(d=256, E=64, F=128, K=8, H=64, r=4, alpha=8.0, shared=True)
    fam = {"kind": "sigmoid_group", "n_group": 8, "topk_group": 4, "scale": 2.5}
    run_lockstep(seed=41, sh=sh, L=5, head_owners={1, 2, 3}, steps=4, family=fam, drift=True,
                 label="sigmoid-group")


@pytest.mark.parametrize("slots", [8, 11])
def test_pooled_stack_staged_from_committed_routing(slots):
    """Head-routed layers read their experts from `slots` HBM slots; from the second
    token on, the ids each launch commits are copied to the host once and drive the
    bundle copies while the next launch is already queued on the ready words."""
    sh = S.LayerShape(d=256, E=16, F=128, K=4, H=64, r=4, alpha=8.0, shared=True)
    run_lockstep(seed=5, sh=sh, L=6, head_owners={1, 2, 3, 4}, steps=10, pool_slots=slots, label=f"pool S={slots}")


@pytest.mark.parametrize("K", [4, 8])
def test_full_size_stack_sampled_layers(K):
    """40 layers of the 35B-class shape, heads on 6..38, K = 4 and 8 (the two work plans:
    prerouter rows on CTAs of their own at K = 4, spread over the expert CTAs at K = 8);
    sampled layers checked over 4 tokens (each prerouted layer consumes three committed
    heads)."""
    sh = S.LAYER35B(K)
    amb = run_lockstep(seed=0, sh=sh, L=S.STACK_LAYERS, head_owners=set(S.HEAD_OWNERS), steps=4,
                       check_layers={0, 6, 7, 8, 20, 39}, label=f"40-layer K={K}")
    assert amb <= 6


def test_repeated_runs_commit_identical_routing():
    """The fp32 accumulators are summed with vector reductions in arrival order, so two
    identical runs may differ in the last bits of h; the routing must still be identical
    wherever the decision's gap (on the GPU's own logits) exceeds 1e-3.  12 layers of the
    35B-class shape (heads on 2..10), K = 4, 3 tokens, two fresh workspaces."""
    import torch
    from routing_predicted_experts_gb300 import binding as B, model as M
    sh, L, steps = S.LAYER35B(4), 12, 3
    owners = set(range(2, 11))
    src = [1 if (l - 1) in owners else 0 for l in range(L)]
    layers = [M.build_layer(3, l, sh, with_head=(l in owners)) for l in range(L)]
    structs = [B.e0_layer_struct(ly["routed"], ly["shared"], ly["lora"], ly["head"], ly["router"]) for ly in layers]
    stack = B.Stack(B.dims(sh.d, sh.E, sh.F, sh.K), structs, src, keepalive=layers)
    outs = []
    for rep in range(2):
        ws = stack.workspace()
        rec = []
        for t in range(steps):
            h0, incr = M.hidden(3, t, sh.d), M.increments(3, t, L, sh.d)
            h_out = torch.empty(sh.d, dtype=torch.int16, device="cuda")
            ids = torch.empty((L, sh.K), dtype=torch.int32, device="cuda")
            zl = torch.zeros((2, L, sh.E), dtype=torch.float32, device="cuda")
            stack.step(t, h0, incr, h_out, ws, ids_out=ids, logits=zl)
            rec.append((h_out, ids, zl))
        torch.cuda.synchronize()
        assert B.e0_get_device_status(ws) == 0
        outs.append([(bf16_host(a), b.cpu().numpy(), c.cpu().numpy()) for a, b, c in rec])
    differing_bits = 0
    for t in range(steps):
        (ha, ia, za), (hb, ib, zb) = outs[0][t], outs[1][t]
        differing_bits += int((ha != hb).sum())
        for l in range(L):
            z = za[0, l] if (t == 0 or not src[l]) else outs[0][t - 1][2][1, l]
            if OR.topk_gap(z.astype(np.float64), sh.K) > 1e-3:
                assert set(ia[l].tolist()) == set(ib[l].tolist()), (t, l)
    REPORT.append(f"repeated runs (12 layers x 3 tokens): routing identical at every clear decision; "
                  f"{differing_bits} of {steps * sh.d} h_out bf16 values differ between the runs")
    stack.close()
