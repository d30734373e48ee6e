"""Prefill chunk (T tokens through one layer on the tcgen05 tensor cores) against the
CPU oracle: routing by top-K of each token's logits, the grouped int4 experts, the
shared expert, the LoRA linear and the residual add."""
import numpy as np
import pytest

from oracle import layer as OL, model_inputs as OM, routing as OR
from routing_predicted_experts_gb300 import synth as S

from _common import bf16_dev, bf16_host, check_bf16_protocol, check_protocol, check_topk, to_dev

pytestmark = pytest.mark.gpu


def _run(sh, seed, T, logits, sample=None, with_shared=True, with_lora=True):
    import torch
    from routing_predicted_experts_gb300 import binding as B, model as M
    lay = M.build_layer(seed, 0, sh, with_head=False)
    H = np.stack([S.normal_bf16(seed, f"pf.h{t}", (sh.d,)) for t in range(T)])
    dm = B.dims(sh.d, sh.E, sh.F, sh.K)
    lora = lay["lora"] if with_lora else None
    ws = B.e0_prefill_workspace(dm, T, lora.out if lora else 0)
    out = B.e0_moe_prefill_layer(dm, lay["routed"], lay["shared"] if with_shared else None, lora, bf16_dev(H),
                                 to_dev(logits, torch.float32), ws)
    torch.cuda.synchronize()
    assert B.e0_get_device_status(ws) == 0
    ids = out["ids"].cpu().numpy()
    w = out["weights"].cpu().numpy()
    # routing: every token, against the oracle's top-K and renormalised softmax
    for t in range(T):
        check_topk(ids[t], logits[t].astype(np.float64), sh.K, f"ids t{t}")
        assert np.abs(w[t] - OR.renorm_weights(logits[t].astype(np.float64), ids[t])).max() <= 1e-5
    olay = dict(OM.layer(seed, 0, sh))
    olay["head"] = None
    if not with_shared:
        olay["shared"] = None
    if not with_lora:
        olay["lora"] = None
    toks = range(T) if sample is None else sample
    got_d, ref_d, got_h, ref_h = [], [], [], []
    for t in toks:
        ref = OL.layer_step(H[t], olay, ids[t], logits[t].astype(np.float64), None, sh.K)
        got_d.append(out["delta"][t].cpu().numpy())
        ref_d.append(ref["delta"])
        got_h.append(bf16_host(out["h_out"][t]))
        ref_h.append(ref["h_out"])
    check_protocol(np.stack(got_d), np.stack(ref_d), "delta")
    check_bf16_protocol(np.stack(got_h), np.stack(ref_h), "h_out")
    return out, ids


def test_prefill_tiny_every_token():
    sh, seed, T = S.TINY, 0, 64
    _run(sh, seed, T, S.zipf_gumbel_logits(seed, T, sh.E))


def test_prefill_ragged_tiles_and_one_hot_expert():
    """T = 129 tokens all routed to the same K experts: three 64-row token tiles per
    expert, the last holding one row; the other experts get no rows."""
    sh, seed, T = S.TINY, 1, 129
    z = S.zipf_gumbel_logits(seed, T, sh.E)
    z[:, :sh.K] += 100.0
    _, ids = _run(sh, seed, T, z)
    assert set(ids.ravel().tolist()) == set(range(sh.K))


def test_prefill_single_token_without_shared_or_lora():
    sh, seed = S.TINY, 2
    _run(sh, seed, 1, S.zipf_gumbel_logits(seed, 1, sh.E), with_shared=False, with_lora=False)


def test_prefill_35b_class_k8_t512_sampled():
    """The prefill workload: T = 512, K = 8, Zipf(1.1)-Gumbel logits (skewed expert
    counts); routing checked for every token, outputs for a sample of tokens."""
    sh, seed, T = S.LAYER35B(8), 0, 512
    z = S.zipf_gumbel_logits(seed, T, sh.E)
    out, ids = _run(sh, seed, T, z, sample=[0, 1, 77, 255, 256, 400, 511])
    counts = np.bincount(ids.ravel(), minlength=sh.E)
    assert counts.max() > 128  # the most popular expert spans more than one row tile
    assert np.all(np.isfinite(out["delta"].cpu().numpy()))
