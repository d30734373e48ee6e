"""Routing functions of the oracle (test infrastructure only).

Source: "The Other Half of the Memory Wall", Appendix A "Routing Math":
* "Softmax-topk (K, renormalize)": g = softmax(l), inds = top-k(g, K),
  w = g[inds] / sum_inds g;
* "Sigmoid-group (K, G of n groups, scale s)": sigma = sigmoid(l); a group's score is
  the sum of its two largest sigmoids; the top G groups survive and the others are
  masked to -inf; inds = top-k of sigma within the survivors; w = s * sigma[inds] /
  (sum sigma[inds] + 1e-20);
and §3.2 "Prediction-as-routing" (the committed prediction goes through the same math).

Readings where the page is silent: ties between equal scores go to the lower expert
(or group) index, and the K selected ids are listed in descending score order.  The
groups of sigmoid-group routing are n contiguous blocks of E/n experts.  The page
says selection uses "the biased score" but prints no bias term; the reading kept
here is the one its DeepSeek-style citation describes: an optional per-expert bias
is added to sigma for the group scores and the top-k only, and the weights use the
raw sigma.  With no bias (the default) the formula is exactly the printed one.
"""
import numpy as np


def softmax(l: np.ndarray) -> np.ndarray:
    l = np.asarray(l, dtype=np.float64)
    m = l.max()
    e = np.exp(l - m)
    return e / e.sum()


def topk_desc(scores: np.ndarray, K: int) -> np.ndarray:
    """Indices of the K largest scores, largest first, equal scores by lower index."""
    order = np.argsort(-np.asarray(scores, dtype=np.float64), kind="stable")
    return order[:K].astype(np.int32)


def softmax_topk(l: np.ndarray, K: int):
    """Returns (ids int32[K], w float64[K]) as Appendix A writes it.

    softmax is strictly increasing, so top-k of g = softmax(l) is top-k of l in exact
    arithmetic; the ranking is taken on l itself because in floating point exp()
    underflows far below the maximum logit and would turn distinct scores into ties.
    The weights are g[inds] / sum(g[inds]) from the full softmax, as written.
    """
    g = softmax(l)
    inds = topk_desc(l, K)
    sel = g[inds]
    return inds, sel / sel.sum()


def renorm_weights(l: np.ndarray, ids: np.ndarray) -> np.ndarray:
    """Combine weights for a given committed id set: softmax over all E, pick, renormalise."""
    g = softmax(l)
    sel = g[np.asarray(ids, dtype=np.int64)]
    return sel / sel.sum()


def topk_gap(l: np.ndarray, K: int) -> float:
    """Gap between the K-th and (K+1)-th largest logits (inf when K == E)."""
    s = np.sort(np.asarray(l, dtype=np.float64))[::-1]
    if K >= s.size:
        return float("inf")
    return float(s[K - 1] - s[K])


def sigmoid(l: np.ndarray) -> np.ndarray:
    l = np.asarray(l, dtype=np.float64)
    return 1.0 / (1.0 + np.exp(-l))


def sigmoid_group(l: np.ndarray, K: int, n_group: int, topk_group: int, scale: float, bias=None):
    """Sigmoid-group routing as Appendix A writes it; returns (ids int32[K], w float64[K])."""
    sig = sigmoid(l)
    E = sig.size
    assert E % n_group == 0 and E // n_group >= 2 and topk_group * (E // n_group) >= K
    score = sig + (0.0 if bias is None else np.asarray(bias, dtype=np.float64))
    gsize = E // n_group
    group_score = np.empty(n_group)
    for g in range(n_group):
        block = np.sort(score[g * gsize:(g + 1) * gsize])[::-1]
        group_score[g] = block[0] + block[1]          # sum of the group's top-2
    keep = topk_desc(group_score, topk_group)        # the top G groups survive
    masked = np.full(E, -np.inf)
    for g in keep:
        masked[g * gsize:(g + 1) * gsize] = score[g * gsize:(g + 1) * gsize]
    ids = topk_desc(masked, K)
    sel = sig[ids]
    return ids, scale * sel / (sel.sum() + 1e-20)


def sigmoid_group_weights(l: np.ndarray, ids: np.ndarray, scale: float) -> np.ndarray:
    """Combine weights of sigmoid-group routing for a given committed id set."""
    sel = sigmoid(l)[np.asarray(ids, dtype=np.int64)]
    return scale * sel / (sel.sum() + 1e-20)


def route(l: np.ndarray, K: int, family=None):
    """(ids, w) of the routing family: None = softmax-top-k, else a dict with
    kind "sigmoid_group", n_group, topk_group, scale and an optional bias."""
    if family is None:
        return softmax_topk(l, K)
    assert family["kind"] == "sigmoid_group"
    return sigmoid_group(l, K, family["n_group"], family["topk_group"], family["scale"], family.get("bias"))


def route_weights(l: np.ndarray, ids: np.ndarray, family=None) -> np.ndarray:
    """Combine weights of a committed id set under the routing family."""
    if family is None:
        return renorm_weights(l, ids)
    return sigmoid_group_weights(l, ids, family["scale"])


def sigmoid_group_gaps(l: np.ndarray, K: int, n_group: int, topk_group: int, bias=None):
    """(group gap, expert gap) of a sigmoid-group decision: the topk_group-th minus the
    next group score (inf when every group survives) and, within the surviving groups,
    the K-th minus the (K+1)-th score (inf when they hold exactly K experts).  A decision
    is unambiguous when both exceed the tolerance."""
    score = sigmoid(l) + (0.0 if bias is None else np.asarray(bias, dtype=np.float64))
    E = score.size
    gsize = E // n_group
    gs = np.array([np.sort(score[g * gsize:(g + 1) * gsize])[::-1][:2].sum() for g in range(n_group)])
    ggap = topk_gap(gs, topk_group)
    keep = topk_desc(gs, topk_group)
    surv = np.concatenate([score[g * gsize:(g + 1) * gsize] for g in keep])
    return ggap, topk_gap(surv, K)


def route_gap(l: np.ndarray, K: int, family=None) -> float:
    """The smallest score gap a routing decision of the family rests on."""
    if family is None:
        return topk_gap(l, K)
    return min(sigmoid_group_gaps(l, K, family["n_group"], family["topk_group"], family.get("bias")))
