"""Pins for the oracle's top-K gap, sigmoid-group routing, residual increment and
decode-stack chaining (CPU only).  Each case is worked by hand or reduces to a
definition that a plausible mistake (an off-by-one, a missing mask, h in place of
h_out, a head consumed at the wrong token) would fail."""
import numpy as np
import pytest

from oracle import bf16 as OB, layer as OL, routing as OR


# ---------------------------------------------------------------- top-K gap

def test_topk_gap_closed_form():
    # sorted: 5, 3, 2.5, 1, 0 (given permuted)
    l = np.array([2.5, 0.0, 5.0, 1.0, 3.0])
    assert OR.topk_gap(l, 1) == 2.0          # 5 - 3
    assert OR.topk_gap(l, 2) == 0.5          # 3 - 2.5 (an s[K] - s[K+1] slip gives 1.5)
    assert OR.topk_gap(l, 3) == 1.5          # 2.5 - 1
    assert OR.topk_gap(l, 4) == 1.0          # 1 - 0
    assert OR.topk_gap(l, 5) == float("inf")  # K == E: nothing to confuse
    assert OR.topk_gap(np.array([1.0, 7.0, 7.0, -2.0]), 1) == 0.0  # tie at the boundary


# ---------------------------------------------------------------- sigmoid-group

def _logit(p):
    p = np.asarray(p, dtype=np.float64)
    return np.log(p) - np.log1p(-p)


# eight groups of four experts (E = 32); sigmoid values chosen by hand
_SIG = np.array([
    [0.90, 0.10, 0.08, 0.07],   # g0: top-2 sum 1.00
    [0.60, 0.55, 0.10, 0.05],   # g1: 1.15
    [0.30, 0.30, 0.29, 0.28],   # g2: 0.60
    [0.97, 0.05, 0.02, 0.01],   # g3: 1.02
    [0.50, 0.48, 0.45, 0.40],   # g4: 0.98
    [0.20, 0.20, 0.15, 0.10],   # g5: 0.40
    [0.70, 0.40, 0.35, 0.30],   # g6: 1.10
    [0.85, 0.02, 0.01, 0.01],   # g7: 0.87 (its 0.85 beats most survivors but the group is dropped)
]).reshape(-1)


def test_sigmoid_group_hand_worked_8b_tier_parameters():
    """n = 8 groups, G = 4 kept, s = 2.5, K = 8 (the 8B tier's parameters).
    Group scores rank g1 1.15, g6 1.10, g3 1.02, g0 1.00 | g4 0.98, g7 0.87, g2, g5;
    the top 8 sigmoids of the surviving groups are .97 (12), .90 (0), .70 (24),
    .60 (4), .55 (5), .40 (25), .35 (26), .30 (27), which sum to 4.77."""
    ids, w = OR.sigmoid_group(_logit(_SIG), K=8, n_group=8, topk_group=4, scale=2.5)
    assert list(ids) == [12, 0, 24, 4, 5, 25, 26, 27]
    sel = np.array([0.97, 0.90, 0.70, 0.60, 0.55, 0.40, 0.35, 0.30])
    assert np.allclose(w, 2.5 * sel / (4.77 + 1e-20), rtol=1e-12, atol=0)
    assert abs(w.sum() - 2.5 * 4.77 / (4.77 + 1e-20)) <= 1e-12
    # without the group mask the top 8 would take g7's 0.85 and g4's 0.50
    plain = OR.topk_desc(_SIG, 8)
    assert 28 in plain and 16 in plain and 28 not in ids and 16 not in ids


def test_sigmoid_group_gaps_hand_worked():
    """Group gap: 4th group 1.00 (g0) minus 5th 0.98 (g4); expert gap within the
    survivors: 8th 0.30 minus 9th 0.10."""
    gg, eg = OR.sigmoid_group_gaps(_logit(_SIG), K=8, n_group=8, topk_group=4)
    assert abs(gg - 0.02) < 1e-12 and abs(eg - 0.20) < 1e-12
    fam = {"kind": "sigmoid_group", "n_group": 8, "topk_group": 4, "scale": 2.5}
    assert abs(OR.route_gap(_logit(_SIG), 8, fam) - 0.02) < 1e-12
    assert OR.route_gap(np.array([2.5, 0.0, 5.0, 1.0, 3.0]), 2) == 0.5


def test_sigmoid_group_scores_groups_by_their_top_two():
    """Ranking groups by their single largest sigmoid would keep g7 (0.85) and drop g1
    (0.60): the top-2 sum keeps g1 and drops g7."""
    ids, _ = OR.sigmoid_group(_logit(_SIG), K=4, n_group=8, topk_group=4, scale=1.0)
    kept = {int(e) // 4 for e in ids}
    assert 7 not in kept and 1 in kept


def test_sigmoid_group_invariants_random():
    rng = np.random.default_rng(11)
    for _ in range(50):
        E, n = 64, 8
        G = int(rng.integers(2, 9))
        K = int(rng.integers(1, min(8, G * (E // n)) + 1))
        l = rng.standard_normal(E) * 2
        ids, w = OR.sigmoid_group(l, K, n, G, 2.5)
        sig = 1 / (1 + np.exp(-l))
        gsize = E // n
        gs = np.array([np.sort(sig[g * gsize:(g + 1) * gsize])[-2:].sum() for g in range(n)])
        kept = set(np.argsort(-gs, kind="stable")[:G].tolist())
        assert len(set(ids.tolist())) == K
        assert all(int(e) // gsize in kept for e in ids)
        # no unchosen expert of a kept group beats a chosen one
        cand = [e for e in range(E) if e // gsize in kept and e not in set(ids.tolist())]
        assert not cand or sig[ids].min() >= max(sig[cand])
        assert np.all(np.diff(sig[ids]) <= 0)
        assert abs(w.sum() - 2.5 * sig[ids].sum() / (sig[ids].sum() + 1e-20)) <= 1e-12


def test_sigmoid_group_with_every_group_kept_is_sigmoid_topk():
    rng = np.random.default_rng(12)
    l = rng.standard_normal(32)
    ids, w = OR.sigmoid_group(l, K=6, n_group=4, topk_group=4, scale=1.0)
    assert list(ids) == list(OR.topk_desc(l, 6))     # sigmoid is increasing
    s = 1 / (1 + np.exp(-l[ids]))
    assert np.allclose(w, s / s.sum(), rtol=1e-13)


def test_sigmoid_group_bias_moves_selection_not_weights():
    """The selection bias (the "biased score") changes which experts are picked; the
    weights of the picked ones still use the raw sigmoid."""
    l = _logit(_SIG)
    bias = np.zeros(32)
    bias[28] = 1.0        # g7's 0.85 -> 1.85: g7's group score 1.87 now ranks first
    ids, w = OR.sigmoid_group(l, K=8, n_group=8, topk_group=4, scale=2.5, bias=bias)
    assert ids[0] == 28
    sel = _SIG[ids]
    assert np.allclose(w, 2.5 * sel / (sel.sum() + 1e-20), rtol=1e-12)
    assert np.allclose(OR.route_weights(l, ids, {"kind": "sigmoid_group", "scale": 2.5}), w, rtol=1e-15)


# ---------------------------------------------------------------- residual increment

def _bf(v):
    return OB.f64_to_bf16(np.array(v, dtype=np.float64))


def test_residual_increment_rounds_half_to_even():
    one = _bf([1.0])
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: ties to the even 1.0
    assert OB.bf16_to_f64(OL.residual_increment(one, _bf([2.0 ** -8])))[0] == 1.0
    # 1 + 3 * 2^-8 lies halfway between 1 + 2^-7 (odd) and 1 + 2^-6 (even)
    assert OB.bf16_to_f64(OL.residual_increment(one, _bf([3 * 2.0 ** -8])))[0] == 1.0 + 2.0 ** -6
    assert OB.bf16_to_f64(OL.residual_increment(_bf([-2.0]), _bf([0.5])))[0] == -1.5


# ---------------------------------------------------------------- stack chaining

def _zero_layer(d, F):
    z = (np.zeros((F, d)), np.zeros((F, d)), np.zeros((d, F)))
    return {"expert": lambda e: z, "shared": None, "lora": None, "head": None}


def _router(rows):
    return OB.to_bf16(np.asarray(rows, dtype=np.float32))


def test_stack_chains_h_out_not_h():
    """A layer whose only term is a LoRA base W = 0.9375 I (what int4 g64 stores
    exactly: one nonzero per row gives scale 2^-4 and code 15).  h0 = 1, increments
    0 then 2^-4: layer 0 gives h_out = bf16(1 + 0.9375 * 0.9999995) = 1.9375, layer 1
    reads bf16(1.9375 + 0.0625) = 2 and gives bf16(2 + 0.93749953) = 2.9375.  Chaining
    the layer input h instead of h_out would give 1.0625 and then 2.0."""
    d, F, E, K = 64, 64, 2, 1
    W = 0.9375 * np.eye(d)
    lay = dict(_zero_layer(d, F))
    lay["lora"] = (W, None, None, 2.0, 0)
    routers = [_router(np.zeros((E, d))), _router(np.zeros((E, d)))]
    h0 = _bf(np.ones(d))
    incr = np.stack([_bf(np.zeros(d)), _bf(np.full(d, 0.0625))])
    out = OL.stack_token(h0, incr, [lay, lay], routers, ["gate", "gate"], K)
    assert np.all(OB.bf16_to_f64(out["layers"][0]["h_out"]) == 1.9375)
    assert np.all(OB.bf16_to_f64(out["layers"][1]["h_in"]) == 2.0)
    assert np.all(OB.bf16_to_f64(out["h_out"]) == 2.9375)


def test_stack_consumes_the_head_one_token_later():
    """Layer 1 routes by its own gate at the first token and by head 0's prediction
    (committed at the previous token) afterwards.  Gate 1 prefers expert 0; head 0's
    linear residual prefers expert 1."""
    d, F, E, K = 64, 64, 4, 1
    h0 = _bf(np.ones(d))
    incr = np.stack([_bf(np.zeros(d))] * 2)
    gate = np.zeros((E, d))
    gate[0] = 0.05
    head = {"Lres": _router(np.outer([0, 1, 0, 0], np.ones(d)) * 0.05), "b2": None, "W1": None, "b1": None,
            "W2": None}
    l0 = dict(_zero_layer(d, F))
    l0["head"] = head
    layers = [l0, _zero_layer(d, F)]
    routers = [_router(gate), _router(gate)]
    t0 = OL.stack_token(h0, incr, layers, routers, ["gate", "head"], K)
    assert list(t0["layers"][1]["ids"]) == [0]                   # first token: own gate
    assert list(OR.topk_desc(t0["zhat_next"][1], 1)) == [1]      # head 0 predicts expert 1
    t1 = OL.stack_token(h0, incr, layers, routers, ["gate", "head"], K, zhat_prev=t0["zhat_next"])
    assert list(t1["layers"][1]["ids"]) == [1]                   # next token: the prediction
    assert np.array_equal(t1["layers"][1]["logits"], t0["zhat_next"][1])


def test_stack_route_ahead_uses_the_earlier_hidden_state():
    """Route-ahead N = 1: layer 1 ranks its own gate on layer 0's input.  h0 = e0 and
    layer 1's increment adds 4 e1, so the gate (row 0 reads e0, row 1 reads e1) picks
    expert 0 on x_0 and expert 1 on x_1."""
    d, F, E, K = 64, 64, 2, 1
    h0 = np.zeros(d)
    h0[0] = 1.0
    inc1 = np.zeros(d)
    inc1[1] = 4.0
    incr = np.stack([_bf(np.zeros(d)), _bf(inc1)])
    gate = np.zeros((E, d))
    gate[0, 0] = 1.0
    gate[1, 1] = 1.0
    layers = [_zero_layer(d, F), _zero_layer(d, F)]
    routers = [_router(gate), _router(gate)]
    own = OL.stack_token(_bf(h0), incr, layers, routers, ["gate", "gate"], K)
    ahead = OL.stack_token(_bf(h0), incr, layers, routers, ["gate", ("ahead", 1)], K)
    assert list(own["layers"][1]["ids"]) == [1]
    assert list(ahead["layers"][1]["ids"]) == [0]
    x0 = OL.rmsnorm(OB.bf16_to_f64(_bf(h0)))
    assert np.allclose(ahead["layers"][1]["logits"], OB.bf16_to_f64(_router(gate)) @ x0, rtol=0, atol=0)
    # nothing lies N layers before layer 0: it routes by its own gate
    first = OL.stack_token(_bf(h0), incr, layers, routers, [("ahead", 1), ("ahead", 1)], K)
    assert list(first["layers"][0]["ids"]) == [0]


def test_zero_network_stack_is_the_bf16_chain_of_increments():
    d, F, E, K, L = 64, 64, 2, 1, 3
    h0 = _bf(np.ones(d))
    incr = np.stack([_bf(np.full(d, 2.0 ** -8))] * L)
    out = OL.stack_token(h0, incr, [_zero_layer(d, F)] * L, [_router(np.zeros((E, d)))] * L, ["gate"] * L, K)
    # every 1 + 2^-8 ties back to 1.0; the exact sum would be 1 + 3 * 2^-8
    assert np.all(OB.bf16_to_f64(out["h_out"]) == 1.0)
