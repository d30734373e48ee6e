"""Prefill chunk (T tokens through one layer on the tcgen05 tensor cores) against the
CPU oracle: routing by top-K of each token's logits, the grouped int4 experts, the
shared expert, the LoRA linear and the residual add."""
import numpy as np
import pytest

from oracle import layer as OL, model_inputs as OM, routing as OR
from routing_predicted_experts_gb300 import synth as S

from _common import bf16_dev, bf16_host, check_bf16_protocol, check_protocol, check_route, to_dev

pytestmark = pytest.mark.gpu


def _run(sh, seed, T, logits, sample=None, with_shared=True, with_lora=True, family=None):
    import torch
    from routing_predicted_experts_gb300 import binding as B, model as M
    lay = M.build_layer(seed, 0, sh, with_head=False)
    H = np.stack([S.normal_bf16(seed, f"pf.h{t}", (sh.d,)) for t in range(T)])
    dm = B.dims(sh.d, sh.E, sh.F, sh.K, family)
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
        check_route(ids[t], logits[t].astype(np.float64), sh.K, f"ids t{t}", family)
        assert np.abs(w[t] - OR.route_weights(logits[t].astype(np.float64), ids[t], family)).max() <= 1e-5
    olay = dict(OM.layer(seed, 0, sh))
    olay["head"] = None
    if not with_shared:
        olay["shared"] = None
    if not with_lora:
        olay["lora"] = None
    toks = range(T) if sample is None else sample
    got_d, ref_d, got_h, ref_h = [], [], [], []
    for t in toks:
        ref = OL.layer_step(H[t], olay, ids[t], logits[t].astype(np.float64), None, sh.K, family)
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


def test_prefill_sigmoid_group_routing():
    """The 8B tier's routing family (n = 8, G = 4, s = 2.5, K = 8) in prefill."""
    sh = S.LayerShape(d=256, E=64, F=128, K=8, H=0, r=4, alpha=8.0, shared=True)
    fam = {"kind": "sigmoid_group", "n_group": 8, "topk_group": 4, "scale": 2.5}
    T = 40
    _run(sh, 3, T, S.zipf_gumbel_logits(3, T, sh.E), family=fam)


def test_prefill_35b_class_k8_t512_every_token():
    """The prefill workload: T = 512, K = 8, Zipf(1.1)-Gumbel logits (skewed expert
    counts: the most popular expert spans several 64-row tiles, the tail experts hold 1
    to 5 rows); routing and outputs checked for every token."""
    sh, seed, T = S.LAYER35B(8), 0, 512
    z = S.zipf_gumbel_logits(seed, T, sh.E)
    out, ids = _run(sh, seed, T, z)
    counts = np.bincount(ids.ravel(), minlength=sh.E)
    assert counts.max() > 128  # the most popular expert spans more than one row tile
    assert ((counts > 0) & (counts < 8)).sum() > 0  # and some experts hold only a few rows
