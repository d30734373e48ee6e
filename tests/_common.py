"""Shared helpers for the GPU parity tests (CPU oracle on one side, libe0 on the other)."""
import numpy as np

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
    """Ids must equal the oracle's top-K wherever the K-th/(K+1)-th gap exceeds gap_tol;
    otherwise every chosen logit must be within gap_tol of the K-th largest."""
    from oracle import routing as OR
    ref_ids, _ = OR.softmax_topk(ref_logits, K)
    gap = OR.topk_gap(ref_logits, K)
    got = np.asarray(got_ids).astype(np.int64)
    if gap > gap_tol:
        assert list(got) == list(ref_ids), (name, list(got), list(ref_ids), gap)
        return True
    kth = np.sort(ref_logits)[::-1][K - 1]
    assert len(set(got)) == K and np.all(ref_logits[got] >= kth - gap_tol), name
    return False
