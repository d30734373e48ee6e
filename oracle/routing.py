"""Softmax-top-k routing with renormalisation (test infrastructure only).

Source: "The Other Half of the Memory Wall", Appendix A "Softmax-topk (K,
renormalize)": g = softmax(l), inds = top-k(g, K), w = g[inds] / sum_inds g; and §3.2
"Prediction-as-routing" (the committed prediction goes through the same math).

Readings where the page is silent: ties between equal scores go to the lower expert
index, and the K selected ids are listed in descending score order.
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
