"""Layer-step maths for the oracle (test infrastructure only).

Everything is float64.  bf16 inputs are widened exactly; int4 weights arrive
dequantised (see ``oracle.int4``).  Sources, by page title and section:

* "The Other Half of the Memory Wall" §3.1 "Math contract": an expert computes
  down(silu(gate(x)) * up(x)).
* §3.2 "Motivation"/"Head": the head of layer N reads layer N's post-attention norm
  output; fc1 -> erf-GELU -> fc2 plus a linear residual path; input feature =
  [hidden ; one-hot of the experts this layer routed to at this token ; one-hot of
  those at the previous token] (dimension d + 2E).
* §3.2 "Prediction-as-routing" and Appendix A: routing weights are the softmax of
  the logits, restricted to the K selected experts and renormalised.
* §3.3: the recovery LoRA is served unmerged, y = W_int4(x) + (alpha/r) * B(A(x)).

Readings (the pages do not say):
* x = RMSNorm(h) = h / sqrt(mean(h^2) + 1e-6) with unit gain is the "post-attention
  norm output" that the head, the router, the experts and the LoRA linear consume;
  the layer adds its output to the residual h (pre-norm block).
* the one-hot blocks are binary K-hot vectors; an absent previous step is all zero.
* the shared expert is added without a gate; the LoRA linear's output is added to
  the residual stream as well.
* h_out is the bf16 rounding (nearest even) of h + delta.
"""
import math

import numpy as np

from .bf16 import bf16_to_f64, f64_to_bf16
from .routing import route, route_weights

RMS_EPS = 1e-6


def rmsnorm(h: np.ndarray) -> np.ndarray:
    h = np.asarray(h, dtype=np.float64)
    return h / math.sqrt(float(np.mean(h * h)) + RMS_EPS)


def silu(u: np.ndarray) -> np.ndarray:
    u = np.asarray(u, dtype=np.float64)
    return u / (1.0 + np.exp(-u))


_erf = np.frompyfunc(math.erf, 1, 1)


def gelu_erf(u: np.ndarray) -> np.ndarray:
    """Exact (erf) GELU: 0.5 * u * (1 + erf(u / sqrt(2)))."""
    u = np.asarray(u, dtype=np.float64)
    return 0.5 * u * (1.0 + _erf(u / math.sqrt(2.0)).astype(np.float64))


def router_logits(x: np.ndarray, R_bf16: np.ndarray) -> np.ndarray:
    """A layer's own gate: z = R x with R bf16 [E][d]."""
    return bf16_to_f64(R_bf16) @ np.asarray(x, dtype=np.float64)


def onehot(ids, E: int) -> np.ndarray:
    v = np.zeros(E, dtype=np.float64)
    if ids is not None:
        for e in np.asarray(ids).reshape(-1):
            v[int(e)] = 1.0
    return v


def prerouter_logits(x: np.ndarray, ids_cur, ids_prev, head: dict) -> np.ndarray:
    """Cross-token prerouter head: predicted next-layer logits for the next token.

    head: W1 bf16 [H][d+2E], b1 bf16 [H] or None, W2 bf16 [E][H], b2 bf16 [E] or None,
    Lres bf16 [E][d].  H == 0 (no W1/W2) leaves only the linear residual path.
    """
    Lres = bf16_to_f64(head["Lres"])
    E, d = Lres.shape
    zhat = Lres @ x
    if head.get("W1") is not None:
        feat = np.concatenate([x, onehot(ids_cur, E), onehot(ids_prev, E)])
        W1 = bf16_to_f64(head["W1"])
        assert W1.shape[1] == d + 2 * E
        u = W1 @ feat
        if head.get("b1") is not None:
            u = u + bf16_to_f64(head["b1"])
        p = gelu_erf(u)
        zhat = zhat + bf16_to_f64(head["W2"]) @ p
    if head.get("b2") is not None:
        zhat = zhat + bf16_to_f64(head["b2"])
    return zhat


def expert(x: np.ndarray, Wg: np.ndarray, Wu: np.ndarray, Wd: np.ndarray) -> np.ndarray:
    """down(silu(gate(x)) * up(x)) with dequantised fp64 weights."""
    return Wd @ (silu(Wg @ x) * (Wu @ x))


def lora_linear(x: np.ndarray, W: np.ndarray, A_bf16, B_bf16, alpha: float, r: int) -> np.ndarray:
    """Unmerged recovery LoRA: W x + (alpha/r) B (A x); B None or r == 0 -> base only."""
    y = W @ x
    if B_bf16 is None or r == 0:
        return y
    A = bf16_to_f64(A_bf16)
    B = bf16_to_f64(B_bf16)
    return y + (alpha / r) * (B @ (A @ x))


def layer_step(h_bf16, layer: dict, ids, logits, ids_prev=None, K: int | None = None, family=None,
               next_family=None):
    """One MoE decode layer-step for one token.

    layer: {"expert": callable e -> (Wg, Wu, Wd) fp64, "shared": (Wg, Wu, Wd) or None,
            "lora": (W, A_bf16, B_bf16, alpha, r) or None, "head": dict or None}
    ids/logits: this layer's committed routing; the combine weights are those of the
    routing family (``family``, see ``oracle.routing.route``; None = the renormalised
    softmax of ``logits`` over ``ids``).  The head's prediction for the next layer is
    turned into ids by ``next_family`` (the next layer's routing family).
    Returns dict(x, delta, h_out (bf16 bits), weights, next_logits, next_ids).
    """
    h = bf16_to_f64(h_bf16)
    x = rmsnorm(h)
    ids = np.asarray(ids, dtype=np.int64)
    w = route_weights(logits, ids, family)
    delta = np.zeros_like(x)
    for k, e in enumerate(ids):
        Wg, Wu, Wd = layer["expert"](int(e))
        delta += w[k] * expert(x, Wg, Wu, Wd)
    if layer.get("shared") is not None:
        delta += expert(x, *layer["shared"])
    if layer.get("lora") is not None:
        delta += lora_linear(x, *layer["lora"])
    out = {"x": x, "delta": delta, "h_out": f64_to_bf16(h + delta), "weights": w,
           "next_logits": None, "next_ids": None}
    if layer.get("head") is not None:
        zhat = prerouter_logits(x, ids, ids_prev, layer["head"])
        out["next_logits"] = zhat
        out["next_ids"], _ = route(zhat, K if K is not None else ids.size, next_family)
    return out


def prefill_chunk(H_bf16: np.ndarray, layer: dict, logits: np.ndarray, K: int, family=None):
    """T tokens through one layer, routed by the given logits (no prerouter)."""
    T = H_bf16.shape[0]
    outs = []
    for t in range(T):
        ids, _ = route(logits[t], K, family)
        lay = dict(layer)
        lay["head"] = None
        outs.append(layer_step(H_bf16[t], lay, ids, logits[t], None, K, family))
    return outs


def residual_increment(h_out_bf16, delta_bf16):
    """Attention stand-in between layers: h_next = bf16(h_out + Delta)."""
    return f64_to_bf16(bf16_to_f64(h_out_bf16) + bf16_to_f64(delta_bf16))


def stack_token(h0_bf16, incr_bf16, layers, routers, sources, K: int, zhat_prev=None, ids_prev=None,
                family=None, adopt=None):
    """One decode token through a stack of layer-steps.

    Sources: "The Other Half of the Memory Wall" §3.2 "Two consumption profiles" and
    "Prediction-as-routing" (the head owned by layer l-1 predicts layer l's routing at
    the next token, and that prediction is the routing); the route-ahead notes
    (BigMoeOnEdge, "Route-ahead": layer l routes by its own gate applied to the hidden
    state N layers earlier in the same forward pass; layers with nothing N layers
    before them route normally).

    h0_bf16: bf16 [d], the token's hidden state entering the stack; incr_bf16: bf16
    [L][d], the per-layer residual increments standing in for attention: layer l's
    input is h_l = bf16(h_out_{l-1} + incr_l), with h_out_{-1} = h0.
    layers[l]: a layer dict as ``layer_step`` takes; routers[l]: bf16 [E][d] gate.
    sources[l]: "gate" (own gate on x_l), "head" (the logits head l-1 committed at the
    previous token; falls back to the gate when ``zhat_prev`` has none, i.e. at the
    first token) or ("ahead", N) (gate_l applied to x_{l-N} of this token).
    zhat_prev: {l: logits committed for layer l at the previous token}.
    ids_prev: {l: ids layer l used at the previous token} (the heads' second one-hot).
    adopt(l, logits, ids) -> ids lets a lockstep caller substitute ids where the
    choice is ambiguous; None keeps the oracle's.
    Returns dict(h_out, layers=[per-layer dicts of layer_step plus h_in, logits, ids],
    zhat_next={l: logits committed for layer l at the next token}).
    """
    zhat_prev = zhat_prev or {}
    ids_prev = ids_prev or {}
    L = len(layers)
    xs, recs, zhat_next = [], [], {}
    h_prev_out = h0_bf16
    for l in range(L):
        h = residual_increment(h_prev_out, incr_bf16[l])
        x = rmsnorm(bf16_to_f64(h))
        xs.append(x)
        src = sources[l]
        if src == "head" and l in zhat_prev:
            z = zhat_prev[l]
        elif isinstance(src, tuple) and src[0] == "ahead" and l - src[1] >= 0:
            z = router_logits(xs[l - src[1]], routers[l])
        else:
            z = router_logits(x, routers[l])
        ids, _ = route(z, K, family)
        if adopt is not None:
            ids = np.asarray(adopt(l, z, ids), dtype=np.int64)
        rec = layer_step(h, layers[l], ids, z, ids_prev.get(l), K, family, family)
        rec.update(h_in=h, logits=z, ids=np.asarray(ids, dtype=np.int64))
        recs.append(rec)
        if rec["next_logits"] is not None and l + 1 < L:
            zhat_next[l + 1] = rec["next_logits"]
        h_prev_out = rec["h_out"]
    return {"h_out": h_prev_out, "layers": recs, "zhat_next": zhat_next}
