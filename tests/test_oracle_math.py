"""Pins for the oracle's routing, head, expert, LoRA and layer-step maths (CPU only)."""
import itertools
import math
import os

import numpy as np
import pytest

from oracle import bf16, int4, layer as OL, routing as OR

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _table(name):
    rows = []
    for line in open(os.path.join(GOLD, name)):
        if line.strip() and not line.startswith("#"):
            rows.append(tuple(float(v) for v in line.split()))
    return rows


# ---------------------------------------------------------------- routing

def test_softmax_topk_closed_form():
    ids, w = OR.softmax_topk(np.log(np.array([1.0, 2.0, 3.0, 4.0])), 2)
    assert list(ids) == [3, 2]
    assert np.allclose(w, [4 / 7, 3 / 7], rtol=0, atol=1e-15)


def test_topk_ties_go_to_lower_index_and_k1_weight_is_one():
    ids, w = OR.softmax_topk(np.array([0.5, 2.0, 2.0, -1.0, 2.0]), 2)
    assert list(ids) == [1, 2]
    ids, w = OR.softmax_topk(np.array([0.1, 0.7, 0.3]), 1)
    assert list(ids) == [1] and w[0] == 1.0


def test_topk_ranks_logits_that_underflow_in_softmax():
    # exp(-1e4) underflows to 0 in fp64: the ranking must still follow the logits
    l = np.array([0.3, -0.2, 0.9, 1e4, 0.1])
    ids, w = OR.softmax_topk(l, 3)
    assert list(ids) == [3, 2, 0]
    assert w[0] == 1.0 and w[1] == 0.0


def test_routing_brute_force_tiny():
    rng = np.random.default_rng(5)
    for _ in range(20):
        l = rng.standard_normal(16)
        ids, w = OR.softmax_topk(l, 4)
        best = max(itertools.combinations(range(16), 4), key=lambda c: sum(l[list(c)]))
        assert set(ids) == set(best)
        assert abs(w.sum() - 1.0) <= 1e-12
        # selected-only softmax is the same distribution
        e = np.exp(l[ids] - l[ids].max())
        assert np.allclose(w, e / e.sum(), rtol=1e-13, atol=0)
        assert np.all(np.diff(l[ids]) <= 0)


# ---------------------------------------------------------------- activations

def test_gelu_erf_against_printed_normal_cdf():
    for u, phi in _table("normal_cdf_table.txt"):
        assert abs(OL.gelu_erf(np.array([u]))[0] - u * phi) <= abs(u) * 6e-6 + 1e-12


def test_silu_against_printed_logistic():
    for u, sig in _table("silu_values.txt"):
        assert abs(OL.silu(np.array([u]))[0] - u * sig) <= abs(u) * 6e-7 + 1e-12


def test_rmsnorm_closed_form():
    h = np.full(64, -3.0)
    x = OL.rmsnorm(h)
    assert np.allclose(x, -3.0 / math.sqrt(9.0 + OL.RMS_EPS), rtol=1e-15)
    h = np.random.default_rng(6).standard_normal(256) * 5
    assert abs(np.mean(OL.rmsnorm(h) ** 2) - 1.0) < 1e-6


# ---------------------------------------------------------------- head

def _head(rng, d=32, E=8, H=16):
    def bfr(*shape):
        return bf16.to_bf16((rng.standard_normal(shape) * 0.1).astype(np.float32))
    return {"W1": bfr(H, d + 2 * E), "b1": bfr(H), "W2": bfr(E, H), "b2": bfr(E), "Lres": bfr(E, d)}


def test_head_one_hot_blocks_add_single_columns():
    rng = np.random.default_rng(7)
    d, E, H = 32, 8, 16
    hd = _head(rng, d, E, H)
    x = rng.standard_normal(d)
    W1 = bf16.bf16_to_f64(hd["W1"])
    b1 = bf16.bf16_to_f64(hd["b1"])

    def pre(cur, prev):
        feat = np.concatenate([x, OL.onehot(cur, E), OL.onehot(prev, E)])
        return W1 @ feat + b1

    base = pre(None, None)
    assert np.allclose(base, W1[:, :d] @ x + b1, rtol=1e-14, atol=1e-14)
    assert np.allclose(pre([3], None) - base, W1[:, d + 3], rtol=0, atol=1e-14)
    assert np.allclose(pre(None, [5]) - base, W1[:, d + E + 5], rtol=0, atol=1e-14)
    # the head itself uses that pre-activation
    z = OL.prerouter_logits(x, [3], [5], hd)
    expect = bf16.bf16_to_f64(hd["W2"]) @ OL.gelu_erf(pre([3], [5])) + bf16.bf16_to_f64(hd["b2"]) \
        + bf16.bf16_to_f64(hd["Lres"]) @ x
    assert np.allclose(z, expect, rtol=1e-14, atol=1e-14)


def test_head_zero_mlp_is_linear_residual():
    rng = np.random.default_rng(8)
    hd = _head(rng)
    hd["W1"] = np.zeros_like(hd["W1"])
    hd["W2"] = np.zeros_like(hd["W2"])
    x = rng.standard_normal(32)
    z = OL.prerouter_logits(x, [1, 2], [3, 4], hd)
    assert np.allclose(z, bf16.bf16_to_f64(hd["Lres"]) @ x + bf16.bf16_to_f64(hd["b2"]), rtol=1e-15)


# ---------------------------------------------------------------- expert / LoRA

def test_expert_against_scalar_loops():
    rng = np.random.default_rng(9)
    d, F = 64, 64
    Wg, Wu = (int4.quantize_dequantize(rng.standard_normal((F, d)).astype(np.float32) * 0.1) for _ in range(2))
    Wd = int4.quantize_dequantize(rng.standard_normal((d, F)).astype(np.float32) * 0.1)
    x = rng.standard_normal(d)
    a = []
    for f in range(F):
        g = sum(Wg[f, c] * x[c] for c in range(d))
        u = sum(Wu[f, c] * x[c] for c in range(d))
        a.append(g / (1.0 + math.exp(-g)) * u)
    y = [sum(Wd[i, f] * a[f] for f in range(F)) for i in range(d)]
    assert np.allclose(OL.expert(x, Wg, Wu, Wd), y, rtol=1e-12, atol=1e-12)


def test_lora_b_zero_is_base_and_unmerged_equals_merged():
    rng = np.random.default_rng(10)
    d, r, alpha = 128, 8, 16.0
    W = int4.quantize_dequantize((rng.standard_normal((d, d)) * 0.02).astype(np.float32))
    A = bf16.to_bf16((rng.standard_normal((r, d)) * 0.02).astype(np.float32))
    B = bf16.to_bf16((rng.standard_normal((d, r)) * 0.02).astype(np.float32))
    x = rng.standard_normal(d)
    assert np.array_equal(OL.lora_linear(x, W, A, np.zeros_like(B), alpha, r), W @ x)
    assert np.array_equal(OL.lora_linear(x, W, A, B, alpha, 0), W @ x)
    merged = W + (alpha / r) * bf16.bf16_to_f64(B) @ bf16.bf16_to_f64(A)
    assert np.allclose(OL.lora_linear(x, W, A, B, alpha, r), merged @ x, rtol=1e-12, atol=1e-12)


def test_merge_and_requantize_erases_most_of_a_small_delta():
    # "The Other Half of the Memory Wall" §3.3: deltas of RMS ~1e-3 sit below the 4-bit
    # group step, so merging and requantising keeps little of them; unmerged keeps all.
    rng = np.random.default_rng(11)
    d, r = 256, 16
    W0 = (rng.standard_normal((d, d)) * 0.02).astype(np.float32)
    q, s, b = int4.pack(W0)
    Wb = int4.dequantize(q, s, b)
    A = rng.standard_normal((r, d)) * 0.0112
    B = rng.standard_normal((d, r)) * 0.0112
    delta = 2.0 * B @ A
    assert 0.5e-3 < np.sqrt(np.mean(delta ** 2)) < 2e-3
    Wm = int4.quantize_dequantize((Wb + delta).astype(np.float32))
    x = rng.standard_normal(d)
    U, M, Bs = (Wb + delta) @ x, Wm @ x, Wb @ x
    retention = 1 - np.linalg.norm(U - M) / np.linalg.norm(U - Bs)
    weight_ret = np.sum((Wm - Wb) * delta) / np.sum(delta ** 2)
    assert retention < 0.5 and weight_ret < 0.5


# ---------------------------------------------------------------- layer-step

def _tiny_layer(rng, d=64, E=8, F=64, H=16, r=4, shared=True, zero=False):
    def q4(rows, cols):
        w = (rng.standard_normal((rows, cols)) * 0.05).astype(np.float32)
        return int4.quantize_dequantize(np.zeros_like(w) if zero else w)
    experts = {e: (q4(F, d), q4(F, d), q4(d, F)) for e in range(E)}
    bfr = (lambda *s: bf16.to_bf16(np.zeros(s, np.float32) if zero else (rng.standard_normal(s) * 0.05).astype(np.float32)))
    return {"expert": lambda e: experts[e],
            "shared": (q4(F, d), q4(F, d), q4(d, F)) if shared else None,
            "lora": (q4(d, d), bfr(r, d), bfr(d, r), 2.0 * r, r),
            "head": {"W1": bfr(H, d + 2 * E), "b1": bfr(H), "W2": bfr(E, H), "b2": bfr(E), "Lres": bfr(E, d)}}


def test_k_equals_e_is_dense_soft_moe():
    rng = np.random.default_rng(12)
    E = 8
    lay = _tiny_layer(rng, E=E)
    lay["lora"] = None
    lay["shared"] = None
    h = bf16.to_bf16(rng.standard_normal(64).astype(np.float32))
    l = rng.standard_normal(E)
    ids, _ = OR.softmax_topk(l, E)
    out = OL.layer_step(h, lay, ids, l, None, E)
    x = OL.rmsnorm(bf16.bf16_to_f64(h))
    p = np.exp(l - l.max())
    p /= p.sum()
    dense = np.zeros(64)
    for e in range(E):
        Wg, Wu, Wd = lay["expert"](e)
        a = np.array([Wg[f] @ x for f in range(64)])
        u = np.array([Wu[f] @ x for f in range(64)])
        dense += p[e] * (Wd @ (a / (1 + np.exp(-a)) * u))
    assert np.allclose(out["delta"], dense, rtol=1e-12, atol=1e-13)


def test_zero_weight_network_is_identity():
    rng = np.random.default_rng(13)
    lay = _tiny_layer(rng, zero=True)
    h = bf16.to_bf16(rng.standard_normal(64).astype(np.float32))
    out = OL.layer_step(h, lay, [0, 1], np.zeros(8), [2, 3], 2)
    assert np.array_equal(out["h_out"], h)
    assert np.all(out["delta"] == 0)
    assert np.all(out["next_logits"] == 0)
    assert list(out["next_ids"]) == [0, 1]


def test_prefill_equals_per_token_decode():
    rng = np.random.default_rng(14)
    lay = _tiny_layer(rng)
    T, K = 3, 2
    H = bf16.to_bf16(rng.standard_normal((T, 64)).astype(np.float32))
    L = rng.standard_normal((T, 8))
    outs = OL.prefill_chunk(H, lay, L, K)
    for t in range(T):
        ids, _ = OR.softmax_topk(L[t], K)
        lay2 = dict(lay)
        lay2["head"] = None
        ref = OL.layer_step(H[t], lay2, ids, L[t])
        assert np.array_equal(outs[t]["h_out"], ref["h_out"])


def test_layer_weights_and_output_rounding():
    rng = np.random.default_rng(15)
    lay = _tiny_layer(rng)
    h = bf16.to_bf16(rng.standard_normal(64).astype(np.float32))
    l = rng.standard_normal(8)
    ids = np.array([6, 2, 3])
    out = OL.layer_step(h, lay, ids, l, [1, 2, 3], 3)
    e = np.exp(l[ids])
    assert np.allclose(out["weights"], e / e.sum(), rtol=1e-14)
    assert np.array_equal(out["h_out"], bf16.f64_to_bf16(bf16.bf16_to_f64(h) + out["delta"]))
