"""Pins for the oracle's small helpers and its view of the seeded model (CPU only): the
combine weights of a given id set, the routing-family dispatch, a layer's own gate, bf16
rounding of float64 values, and the int4 weights the oracle draws (each within one
quantisation step of the underlying fp32 draw, in the documented shapes)."""
import numpy as np

from oracle import bf16 as OB, int4 as OI, layer as OL, model_inputs as OM, routing as OR
from routing_predicted_experts_gb300 import synth as S


def test_renorm_weights_hand_worked():
    # softmax over all three, then the picked pair renormalised: e^ln3 : e^ln2 = 3 : 2
    l = np.log(np.array([1.0, 2.0, 3.0]))
    w = OR.renorm_weights(l, np.array([2, 1]))
    assert np.allclose(w, [0.6, 0.4], rtol=0, atol=1e-15)
    # a single id gets weight 1 whatever its logit
    assert OR.renorm_weights(np.array([-50.0, 3.0, 7.0]), np.array([0]))[0] == 1.0


def test_sigmoid_group_weights_hand_worked():
    # sigma(0) = 1/2 for both picks: s * 0.5 / (1 + 1e-20)
    w = OR.sigmoid_group_weights(np.zeros(4), np.array([1, 3]), 2.5)
    assert np.allclose(w, [1.25, 1.25], rtol=0, atol=1e-15)
    # unequal: sigma(ln 3) = 3/4, sigma(-ln 3) = 1/4 -> 2 * (3/4, 1/4) / 1
    w = OR.sigmoid_group_weights(np.array([np.log(3.0), -np.log(3.0)]), np.array([0, 1]), 2.0)
    assert np.allclose(w, [1.5, 0.5], rtol=0, atol=1e-15)


def test_route_dispatches_by_family():
    rng = np.random.default_rng(5)
    l = rng.normal(size=64)
    ids, w = OR.route(l, 4)
    ids2, w2 = OR.softmax_topk(l, 4)
    assert np.array_equal(ids, ids2) and np.array_equal(w, w2)
    fam = {"kind": "sigmoid_group", "n_group": 8, "topk_group": 4, "scale": 2.5}
    ids, w = OR.route(l, 8, fam)
    ids2, w2 = OR.sigmoid_group(l, 8, 8, 4, 2.5, None)
    assert np.array_equal(ids, ids2) and np.array_equal(w, w2)
    assert np.allclose(OR.route_weights(l, ids, fam), OR.sigmoid_group_weights(l, ids, 2.5))


def test_router_logits_hand_worked():
    R = OB.f64_to_bf16(np.array([[1.0, 2.0], [0.5, -1.0]]))  # bf16-exact values
    z = OL.router_logits(np.array([1.0, 1.0]), R)
    assert np.array_equal(z, [3.0, -0.5])
    z = OL.router_logits(np.array([2.0, -3.0]), R)
    assert np.array_equal(z, [-4.0, 4.0])  # a transposed R would give [0.5, 7]


def test_round_to_bf16_f64_ties_to_even():
    u = 2.0 ** -7  # bf16 spacing at 1
    x = np.array([1.0 + u / 2, 1.0 + 3 * u / 2, 1.0 + u / 4, -(1.0 + u / 2), 3.0])
    r = OB.round_to_bf16_f64(x)
    assert np.array_equal(r, [1.0, 1.0 + 2 * u, 1.0, -1.0, 3.0])


def test_model_inputs_shapes_and_quantisation_error():
    sh = S.LayerShape(d=256, E=16, F=128, K=4, H=64, r=4, alpha=8.0, shared=True)
    g, u, dn = OM.expert_weights(3, 0, 5, sh)
    assert g.shape == (sh.F, sh.d) and u.shape == (sh.F, sh.d) and dn.shape == (sh.d, sh.F)
    # each dequantised weight lies within one quantisation step of its fp32 draw
    raw = S.normal_f32(3, S.t_expert(0, 5, "gate"), (sh.F, sh.d), S.W_SIGMA).astype(np.float64)
    grp = raw.reshape(sh.F, sh.d // 64, 64)
    step = (grp.max(axis=2) - grp.min(axis=2)) / 15.0
    err = np.abs(g.reshape(grp.shape) - grp)
    assert np.all(err <= step[..., None] * 1.01 + 1e-12)
    assert np.array_equal(g, OI.quantize_dequantize(raw.astype(np.float32)))
    # the same draw twice (cached), read-only
    assert OM.expert_weights(3, 0, 5, sh)[0] is g and not g.flags.writeable
    s = OM.shared_weights(3, 0, sh)
    assert s is not None and s[2].shape == (sh.d, sh.F)
    W, A, B, alpha, r = OM.lora_weights(3, 0, sh)
    assert W.shape == (sh.lora_rows, sh.d) and A.shape == (sh.r, sh.d) and B.shape == (sh.lora_rows, sh.r)
    assert alpha == sh.alpha and r == sh.r
    hd = OM.head_weights(3, 0, sh)
    assert hd["W1"].shape == (sh.H, sh.d + 2 * sh.E) and hd["W2"].shape == (sh.E, sh.H)
    assert hd["Lres"].shape == (sh.E, sh.d) and hd["b1"].shape == (sh.H,) and hd["b2"].shape == (sh.E,)
    R = OM.router_weights(3, 0, sh)
    assert R.shape == (sh.E, sh.d) and R.dtype == np.uint16
