"""Decode stack (one launch per token): lockstep comparison with the oracle, layer by
layer from identical inputs (the GPU's own layer inputs), with routing decisions
checked against the oracle's and adopted only where the top-K gap is ambiguous."""
import numpy as np
import pytest

from oracle import bf16 as OB, layer as OL, model_inputs as OM, routing as OR
from routing_predicted_experts_gb300 import synth as S

from _common import bf16_host, check_bf16_protocol, check_protocol

pytestmark = pytest.mark.gpu


def _build_stack(seed, sh, L, head_owners, device="cuda"):
    from routing_predicted_experts_gb300 import binding as B, model as M
    layers, structs, prerouted = [], [], []
    for l in range(L):
        ly = M.build_layer(seed, l, sh, with_head=(l in head_owners))
        layers.append(ly)
        structs.append(B.e0_layer_struct(ly["routed"], ly["shared"], ly["lora"], ly["head"], ly["router"]))
        prerouted.append(1 if (l - 1) in head_owners else 0)
    stack = B.Stack(B.dims(sh.d, sh.E, sh.F, sh.K), structs, prerouted, keepalive=layers)
    return stack, prerouted


def _run_lockstep(seed, sh, L, head_owners, steps, check_layers=None):
    import torch
    from routing_predicted_experts_gb300 import model as M
    stack, prerouted = _build_stack(seed, sh, L, head_owners)
    ws = stack.workspace()
    K, d = sh.K, sh.d
    zhat_prev = {}      # oracle: head l-1 logits from the previous step
    ids_prev = {}       # GPU ids used at the previous step, per layer
    ambiguous = 0
    for t in range(steps):
        h0 = M.hidden(seed, t, d)
        incr = M.increments(seed, t, L, d)
        h_out = torch.empty(d, dtype=torch.int16, device="cuda")
        ids_t = torch.empty((L, K), dtype=torch.int32, device="cuda")
        w_t = torch.empty((L, K), dtype=torch.float32, device="cuda")
        h_tr = torch.empty((L, d), dtype=torch.int16, device="cuda")
        stack.step(t, h0, incr, h_out, ws, ids_t, w_t, h_tr)
        torch.cuda.synchronize()
        from routing_predicted_experts_gb300 import binding as B
        assert B.e0_get_device_status(ws) == 0
        H = bf16_host(h_tr)
        I = ids_t.cpu().numpy()
        W = w_t.cpu().numpy()
        inc = bf16_host(incr)
        zhat_now = {}
        for l in range(L):
            need = check_layers is None or l in check_layers or (l + 1) in check_layers
            olay = OM.layer(seed, l, sh, with_head=(l in head_owners)) if need else None
            if not need:
                continue
            x = OL.rmsnorm(OB.bf16_to_f64(H[l]))
            if t == 0 or not prerouted[l]:
                z = OL.router_logits(x, OM.router_weights(seed, l, sh))
            else:
                z = zhat_prev.get(l - 1)
            gi = I[l].astype(np.int64)
            if z is not None:
                ref_ids, _ = OR.softmax_topk(z, K)
                gap = OR.topk_gap(z, K)
                if gap > 1e-3:
                    assert list(gi) == list(ref_ids), (t, l, list(gi), list(ref_ids), gap)
                else:
                    ambiguous += 1
                w_ref = OR.renorm_weights(z, gi)
                assert np.abs(W[l] - w_ref).max() <= 2e-3, (t, l)
            prev = ids_prev.get(l) if t > 0 else None
            if z is None:
                continue
            ref = OL.layer_step(H[l], olay, gi, z, prev, K)
            if olay["head"] is not None:
                zhat_now[l] = ref["next_logits"]
            if l + 1 < L:
                nxt = OL.residual_increment(ref["h_out"], inc[l + 1])
                check_bf16_protocol(H[l + 1], nxt, f"h_in step {t} layer {l + 1}")
            else:
                check_bf16_protocol(bf16_host(h_out), ref["h_out"], f"h_out step {t}")
        zhat_prev = zhat_now
        ids_prev = {l: I[l].copy() for l in range(L)}
    stack.close()
    return ambiguous


def test_tiny_stack_lockstep():
    sh = S.TINY
    # heads on layers 1..4 of 6: layers 2..5 route from the previous layer's head
    _run_lockstep(seed=11, sh=sh, L=6, head_owners={1, 2, 3, 4}, steps=4)


def test_tiny_stack_k1_and_k16():
    for K in (1, 16):
        sh = S.LayerShape(d=256, E=16, F=128, K=K, H=64, r=4, alpha=8.0, shared=True)
        _run_lockstep(seed=12 + K, sh=sh, L=3, head_owners={0, 1}, steps=3)


@pytest.mark.parametrize("K", [4, 8])
def test_full_size_stack_sampled_layers(K):
    """40 layers of the 35B-class shape, heads on 6..38, K = 4 and 8 (the two work plans:
    prerouter rows on CTAs of their own at K = 4, spread over the expert CTAs at K = 8);
    sampled layers checked."""
    sh = S.LAYER35B(K)
    amb = _run_lockstep(seed=0, sh=sh, L=S.STACK_LAYERS, head_owners=set(S.HEAD_OWNERS), steps=2,
                        check_layers={0, 6, 7, 8, 20, 39})
    assert amb <= 3
