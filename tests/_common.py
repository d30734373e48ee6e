"""Shared helpers for the GPU parity tests (CPU oracle on one side, libe0 on the other)."""
import numpy as np

# lines for the end-of-run summary (tests/conftest.py prints them): ambiguous routing
# decisions the oracle adopted, end-to-end drift, bytes per token
REPORT = []

from oracle import bf16 as OB


def to_dev(a, dtype):
    import torch
    return torch.from_numpy(np.array(a, copy=True)).to(dtype).cuda()


def bf16_dev(bits):
    import torch
    return to_dev(np.asarray(bits, dtype=np.uint16).view(np.int16), torch.int16)


def bf16_host(t):
    return t.cpu().numpy().view(np.uint16)


def check_protocol(got, ref, name, max_rel=1e-2, mean_rel=1e-3):
    """max|err| <= 1e-2 * max|ref| and mean|err| <= 1e-3 * mean|ref| (the parity bar)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), name
    err = np.abs(got - ref)
    assert err.max() <= max_rel * np.abs(ref).max(), (name, err.max(), np.abs(ref).max())
    assert err.mean() <= mean_rel * np.abs(ref).mean(), (name, err.mean(), np.abs(ref).mean())
    return err.max() / max(np.abs(ref).max(), 1e-30), err.mean() / max(np.abs(ref).mean(), 1e-30)


def check_bf16_protocol(got_bits, ref_bits, name):
    return check_protocol(OB.bf16_to_f64(got_bits), OB.bf16_to_f64(ref_bits), name)


def check_topk(got_ids, ref_logits, K, name, gap_tol=1e-3):
    """Routing parity for one token.

    Where the oracle's K-th/(K+1)-th logit gap exceeds gap_tol the chosen SET must be
    the oracle's, listed in descending logit order (two chosen ids whose logits lie
    within gap_tol may come in either order).  Otherwise several sets are correct:
    every chosen logit must lie within gap_tol of the K-th largest, and every id whose
    logit exceeds the K-th largest by more than gap_tol must be chosen.  Returns True
    when the decision was unambiguous."""
    from oracle import routing as OR
    ref_logits = np.asarray(ref_logits, dtype=np.float64)
    ref_ids, _ = OR.softmax_topk(ref_logits, K)
    gap = OR.topk_gap(ref_logits, K)
    got = np.asarray(got_ids).astype(np.int64)
    assert got.shape == (K,) and np.all((got >= 0) & (got < ref_logits.size)), (name, list(got))
    assert len(set(got.tolist())) == K, (name, list(got))
    zg = ref_logits[got]
    assert np.all(np.diff(zg) <= gap_tol), (name, list(got), "not in descending order")
    if gap > gap_tol:
        assert set(got.tolist()) == set(ref_ids.tolist()), (name, list(got), list(ref_ids), gap)
        return True
    kth = np.sort(ref_logits)[::-1][K - 1]
    assert np.all(zg >= kth - gap_tol), (name, list(got))
    must = set(np.nonzero(ref_logits > kth + gap_tol)[0].tolist())
    assert must <= set(got.tolist()), (name, list(got), sorted(must))
    return False


def check_route(got_ids, ref_logits, K, name, family=None, gap_tol=1e-3):
    """check_topk for either routing family.  Sigmoid-group: where both of the decision's
    gaps exceed gap_tol the chosen set must be the oracle's; otherwise every chosen id
    must lie in a group within gap_tol of the last surviving group's score and score
    within gap_tol of the K-th score of those groups.  Returns True when unambiguous."""
    if family is None:
        return check_topk(got_ids, ref_logits, K, name, gap_tol)
    from oracle import routing as OR
    z = np.asarray(ref_logits, dtype=np.float64)
    got = np.asarray(got_ids).astype(np.int64)
    assert got.shape == (K,) and len(set(got.tolist())) == K and np.all((got >= 0) & (got < z.size)), (name, got)
    ref_ids, _ = OR.route(z, K, family)
    if OR.route_gap(z, K, family) > gap_tol:
        assert set(got.tolist()) == set(ref_ids.tolist()), (name, list(got), list(ref_ids))
        return True
    score = OR.sigmoid(z) + (0.0 if family.get("bias") is None else np.asarray(family["bias"]))
    n, G = family["n_group"], family["topk_group"]
    gsize = z.size // n
    gs = np.array([np.sort(score[g * gsize:(g + 1) * gsize])[::-1][:2].sum() for g in range(n)])
    gth = np.sort(gs)[::-1][G - 1]
    ok_groups = [g for g in range(n) if gs[g] >= gth - gap_tol]
    assert all(int(e) // gsize in ok_groups for e in got), (name, list(got))
    pool = np.concatenate([score[g * gsize:(g + 1) * gsize] for g in ok_groups])
    kth = np.sort(pool)[::-1][K - 1]
    assert np.all(score[got] >= kth - gap_tol), (name, list(got))
    return False


class DevView:
    """A device array given by raw pointer, readable by torch.as_tensor (tests only)."""

    def __init__(self, ptr, n, typestr):
        self.__cuda_array_interface__ = {"shape": (n,), "typestr": typestr, "data": (int(ptr), False),
                                         "version": 2}


def dev_array(ptr, n, dtype):
    import torch
    typestr = {torch.int16: "<i2", torch.int32: "<i4", torch.uint32: "<u4", torch.uint8: "|u1"}[dtype]
    return torch.as_tensor(DevView(ptr, n, typestr), device="cuda")
