"""Layer-step, prerouter and LoRA-linear parity: libe0 against the CPU oracle."""
import numpy as np
import pytest

from oracle import bf16 as OB, layer as OL, model_inputs as OM, routing as OR
from routing_predicted_experts_gb300 import synth as S

from _common import bf16_dev, bf16_host, check_bf16_protocol, check_protocol, check_route, check_topk, to_dev

pytestmark = pytest.mark.gpu

CASES = [("tiny", S.TINY, 0), ("35b_k4_s0", S.LAYER35B(4), 0), ("35b_k4_s1", S.LAYER35B(4), 1),
         ("35b_k8_s2", S.LAYER35B(8), 2)]


def _inputs(seed, sh):
    h = OM.hidden(seed, 0, sh.d)
    zc = OM.supplied_logits(seed, "cur", sh.E)
    zp = OM.supplied_logits(seed, "prev", sh.E)
    ids, _ = OR.softmax_topk(zc, sh.K)
    ids_prev, _ = OR.softmax_topk(zp, sh.K)
    return h, zc, ids, ids_prev


@pytest.mark.parametrize("name,sh,seed", CASES, ids=[c[0] for c in CASES])
def test_layer_step_matches_oracle(name, sh, seed):
    import torch
    from routing_predicted_experts_gb300 import binding as B, model as M
    lay = M.build_layer(seed, 0, sh)
    h, zc, ids, ids_prev = _inputs(seed, sh)
    dm = B.dims(sh.d, sh.E, sh.F, sh.K)
    ws = B.e0_workspace(dm)
    out = B.e0_moe_decode_layer(dm, lay["routed"], lay["shared"], lay["lora"], lay["head"], bf16_dev(h)[None],
                                to_dev(ids, torch.int32)[None], to_dev(zc, torch.float32)[None],
                                to_dev(ids_prev, torch.int32)[None], ws)
    torch.cuda.synchronize()
    assert B.e0_get_device_status(ws) == 0
    ref = OL.layer_step(h, OM.layer(seed, 0, sh), ids, zc, ids_prev, sh.K)
    # magnitudes are not vacuous: experts+LoRA move the residual by O(1)
    assert 0.3 < np.std(ref["delta"]) < 5 and 0.3 < np.std(ref["next_logits"]) < 5
    check_protocol(out["delta"][0].cpu().numpy(), ref["delta"], "delta")
    check_bf16_protocol(bf16_host(out["h_out"][0]), ref["h_out"], "h_out")
    zg = out["next_logits"][0].cpu().numpy().astype(np.float64)
    check_protocol(zg, ref["next_logits"], "next_logits")
    check_topk(out["next_ids"][0].cpu().numpy(), ref["next_logits"], sh.K, "next_ids")
    # weights: the renormalised softmax of the GPU's own logits over its ids
    gi = out["next_ids"][0].cpu().numpy()
    assert np.abs(out["next_weights"][0].cpu().numpy() - OR.renorm_weights(zg, gi)).max() <= 1e-5
    assert abs(out["next_weights"][0].cpu().numpy().sum() - 1.0) <= 1e-5


def test_layer_step_multi_token_and_repeat_calls():
    """T = 3 tokens in one call; the workspace keeps working across calls (parity halves)."""
    import torch
    from routing_predicted_experts_gb300 import binding as B, model as M
    sh, seed = S.TINY, 3
    lay = M.build_layer(seed, 0, sh)
    olay = OM.layer(seed, 0, sh)
    T = 3
    H = np.stack([S.normal_bf16(seed, f"hid{t}", (sh.d,)) for t in range(T)])
    Z = np.stack([S.normal_f32(seed, f"z{t}", (sh.E,)) for t in range(T)])
    ids = np.stack([OR.softmax_topk(Z[t], sh.K)[0] for t in range(T)])
    prev = np.roll(ids, 1, axis=0)
    dm = B.dims(sh.d, sh.E, sh.F, sh.K)
    ws = B.e0_workspace(dm)
    for rep in range(3):
        out = B.e0_moe_decode_layer(dm, lay["routed"], lay["shared"], lay["lora"], lay["head"], bf16_dev(H),
                                    to_dev(ids, torch.int32), to_dev(Z, torch.float32), to_dev(prev, torch.int32),
                                    ws)
        torch.cuda.synchronize()
        assert B.e0_get_device_status(ws) == 0
        for t in range(T):
            ref = OL.layer_step(H[t], olay, ids[t], Z[t], prev[t], sh.K)
            check_protocol(out["delta"][t].cpu().numpy(), ref["delta"], f"delta t{t} rep{rep}")
            check_protocol(out["next_logits"][t].cpu().numpy(), ref["next_logits"], f"zhat t{t}")


def test_layer_without_optional_parts_and_zero_lora_b():
    """No head / no shared; LoRA with B = 0 equals LoRA with r = 0 (bit for bit)."""
    import torch
    from routing_predicted_experts_gb300 import binding as B, model as M
    sh, seed = S.TINY, 4
    lay = M.build_layer(seed, 0, sh, with_head=False)
    h, zc, ids, _ = _inputs(seed, sh)
    dm = B.dims(sh.d, sh.E, sh.F, sh.K)
    ws = B.e0_workspace(dm)
    args = (bf16_dev(h)[None], to_dev(ids, torch.int32)[None], to_dev(zc, torch.float32)[None], None, ws)
    lo = lay["lora"]
    lo0 = B.QLora(lo.w, lo.a, torch.zeros_like(lo.bt), lo.out, lo.r, lo.alpha)
    lor = B.QLora(lo.w, None, None, lo.out, 0, lo.alpha)
    o0 = B.e0_moe_decode_layer(dm, lay["routed"], None, lo0, None, *args)
    o1 = B.e0_moe_decode_layer(dm, lay["routed"], None, lor, None, *args)
    o2 = B.e0_moe_decode_layer(dm, lay["routed"], None, None, None, *args)
    torch.cuda.synchronize()
    d0, d1 = o0["delta"].cpu().numpy(), o1["delta"].cpu().numpy()
    assert np.allclose(d0, d1, rtol=0, atol=1e-6 * np.abs(d1).max())
    olay = OM.layer(seed, 0, sh, with_head=False)
    olay["lora"] = None
    ref = OL.layer_step(h, olay, ids, zc, None, sh.K)
    check_protocol(o2["delta"][0].cpu().numpy(), ref["delta"], "delta experts only")


@pytest.mark.parametrize("H", [64, 0])
def test_prerouter_forward_matches_oracle(H):
    import torch
    from routing_predicted_experts_gb300 import binding as B, model as M
    sh = S.LayerShape(d=512, E=64, F=128, K=4, H=H, r=0, alpha=0.0, shared=False)
    seed = 7
    head = M.build_head(seed, 0, sh)
    ohead = OM.head_weights(seed, 0, sh)
    T = 2
    Hh = np.stack([S.normal_bf16(seed, f"ph{t}", (sh.d,)) for t in range(T)])
    cur = np.stack([np.array([3, 9, 17, 40], np.int32), np.array([0, 1, 2, 63], np.int32)])
    prev = np.stack([np.array([5, 9, 33, 62], np.int32), np.array([7, 6, 5, 4], np.int32)])
    bias = np.zeros(sh.E, np.float32)
    bias[11] = 1e4
    dm = B.dims(sh.d, sh.E, 64, sh.K)
    ws = B.e0_workspace(dm)
    logits, ids, w = B.e0_prerouter_forward(head, sh.d, sh.E, sh.K, bf16_dev(Hh), to_dev(cur, torch.int32),
                                            to_dev(prev, torch.int32), ws, logit_bias=to_dev(bias, torch.float32))
    torch.cuda.synchronize()
    assert B.e0_get_device_status(ws) == 0
    for t in range(T):
        x = OL.rmsnorm(OB.bf16_to_f64(Hh[t]))
        z = OL.prerouter_logits(x, cur[t], prev[t], ohead) + bias
        check_protocol(logits[t].cpu().numpy(), z, f"logits t{t}")
        gi = ids[t].cpu().numpy()
        assert gi[0] == 11
        check_topk(gi, z, sh.K, f"ids t{t}")


def test_qlinear_lora_matches_oracle_and_accumulates():
    import torch
    from routing_predicted_experts_gb300 import binding as B, model as M
    sh = S.LayerShape(d=1024, E=8, F=64, K=1, H=0, r=16, alpha=32.0, shared=False, lora_out=512)
    seed = 9
    lo = M.build_lora(seed, 0, sh)
    W, A, Bm, alpha, r = OM.lora_weights(seed, 0, sh)
    T = 2
    X = np.stack([S.normal_bf16(seed, f"qx{t}", (sh.d,)) for t in range(T)])
    Y0 = np.stack([S.normal_bf16(seed, f"qy{t}", (512,)) for t in range(T)])
    ws = B.e0_workspace(B.dims(1024, 8, 64, 1))
    y = bf16_dev(Y0)
    y, yf = B.e0_qlinear_lora(lo, bf16_dev(X), ws, y=y, accumulate=True)
    torch.cuda.synchronize()
    for t in range(T):
        ref = OL.lora_linear(OB.bf16_to_f64(X[t]), W, A, Bm, alpha, r) + OB.bf16_to_f64(Y0[t])
        check_protocol(yf[t].cpu().numpy(), ref, f"y_f32 t{t}")
        check_bf16_protocol(bf16_host(y[t]), OB.f64_to_bf16(ref), f"y t{t}")
    # B == 0 gives exactly the base path (r == 0)
    lo0 = B.QLora(lo.w, lo.a, torch.zeros_like(lo.bt), lo.out, lo.r, lo.alpha)
    lob = B.QLora(lo.w, None, None, lo.out, 0, lo.alpha)
    _, f0 = B.e0_qlinear_lora(lo0, bf16_dev(X), ws)
    _, fb = B.e0_qlinear_lora(lob, bf16_dev(X), ws)
    torch.cuda.synchronize()
    assert np.allclose(f0.cpu().numpy(), fb.cpu().numpy(), rtol=0, atol=1e-6 * fb.abs().max().item())


def test_layer_step_sigmoid_group_routing():
    """Sigmoid-group routing (n = 8, G = 4, s = 2.5, K = 8) in a single layer-step: the
    combine weights of the given ids are s * sigmoid / (sum + 1e-20), and the head's
    prediction is turned into the next layer's ids by the same family, with a selection
    bias that moves the choice but not the weights."""
    import torch
    from routing_predicted_experts_gb300 import binding as B, model as M
    sh = S.LayerShape(d=256, E=64, F=128, K=8, H=64, r=4, alpha=8.0, shared=True)
    seed = 9
    lay = M.build_layer(seed, 0, sh)
    h, zc, _, _ = _inputs(seed, sh)
    bias = S.normal_f32(seed, "sg.bias", (sh.E,), 0.05)
    fam = {"kind": "sigmoid_group", "n_group": 8, "topk_group": 4, "scale": 2.5}
    famb = dict(fam, bias=bias.astype(np.float64))
    ids, _ = OR.route(zc, sh.K, fam)
    prev, _ = OR.route(OM.supplied_logits(seed, "prev", sh.E), sh.K, fam)
    bias_dev = to_dev(bias, torch.float32)
    dm = B.dims(sh.d, sh.E, sh.F, sh.K, fam, score_bias=bias_dev)
    ws = B.e0_workspace(dm)
    out = B.e0_moe_decode_layer(dm, lay["routed"], lay["shared"], lay["lora"], lay["head"], bf16_dev(h)[None],
                                to_dev(ids, torch.int32)[None], to_dev(zc, torch.float32)[None],
                                to_dev(prev, torch.int32)[None], ws)
    torch.cuda.synchronize()
    assert B.e0_get_device_status(ws) == 0
    ref = OL.layer_step(h, OM.layer(seed, 0, sh), ids, zc, prev, sh.K, fam, famb)
    check_protocol(out["delta"][0].cpu().numpy(), ref["delta"], "delta")
    zg = out["next_logits"][0].cpu().numpy().astype(np.float64)
    check_protocol(zg, ref["next_logits"], "next_logits")
    gi = out["next_ids"][0].cpu().numpy()
    check_route(gi, ref["next_logits"], sh.K, "next_ids", famb)
    w = out["next_weights"][0].cpu().numpy()
    assert np.abs(w - OR.route_weights(zg, gi, fam)).max() <= 1e-5
    assert abs(w.sum() - 2.5 * OR.sigmoid(zg[gi]).sum() / (OR.sigmoid(zg[gi]).sum() + 1e-20)) <= 1e-5


@pytest.mark.parametrize("factor", [100.0, 1000.0])
def test_layer_step_with_an_activation_outlier(factor):
    """One hidden element at 100x / 1000x the rms of the rest (real models carry such
    outliers): x is quantised to int16 with one step per 32-element chunk, so the
    outlier costs resolution only within its own chunk and the layer stays at the bar."""
    import torch
    from routing_predicted_experts_gb300 import binding as B, model as M
    sh, seed = S.LAYER35B(4), 0
    lay = M.build_layer(seed, 0, sh)
    h, zc, ids, ids_prev = _inputs(seed, sh)
    h = h.copy()
    h[777] = OB.f64_to_bf16(np.array([factor]))[0]
    h[1500] = OB.f64_to_bf16(np.array([-factor / 3]))[0]
    dm = B.dims(sh.d, sh.E, sh.F, sh.K)
    ws = B.e0_workspace(dm)
    out = B.e0_moe_decode_layer(dm, lay["routed"], lay["shared"], lay["lora"], lay["head"], bf16_dev(h)[None],
                                to_dev(ids, torch.int32)[None], to_dev(zc, torch.float32)[None],
                                to_dev(ids_prev, torch.int32)[None], ws)
    torch.cuda.synchronize()
    assert B.e0_get_device_status(ws) == 0
    ref = OL.layer_step(h, OM.layer(seed, 0, sh), ids, zc, ids_prev, sh.K)
    mx, mn = check_protocol(out["delta"][0].cpu().numpy(), ref["delta"], f"delta, outlier x{factor:g}")
    check_protocol(out["next_logits"][0].cpu().numpy(), ref["next_logits"], f"next_logits, outlier x{factor:g}")
    from _common import REPORT
    REPORT.append(f"35B layer with a {factor:g}x activation outlier: delta max|err|/max|ref| {mx:.2e}, "
                  f"mean|err|/mean|ref| {mn:.2e}")
