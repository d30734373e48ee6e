"""Several decode tokens in one layer-step call (T = 2..16): every weight is read once
for all the tokens (grouped tensor-core experts, multi-token head).  Each token's delta,
h_out, head logits, committed ids and weights against the oracle's single-token
layer-step on the same inputs; the bytes a call reads per token are reported."""
import numpy as np
import pytest

from oracle import layer as OL, model_inputs as OM, routing as OR
from routing_predicted_experts_gb300 import synth as S

from _common import REPORT, bf16_dev, bf16_host, check_bf16_protocol, check_protocol, check_route, to_dev

pytestmark = pytest.mark.gpu


def _bytes_per_token(sh, ids, H):
    """Weight bytes a T-token call reads, per token: every distinct routed expert once,
    the shared expert, the LoRA linear and the head once."""
    q4 = lambda rows, cols: rows * cols // 2 + rows * (cols // 64) * 4
    expert = q4(2 * sh.F, sh.d) + q4(sh.d, sh.F)
    lora = q4(sh.d, sh.d) + 2 * sh.r * sh.d * 2
    head = 2 * H * sh.d + 2 * H + 2 * sh.E * H + 2 * sh.E + 2 * sh.E * sh.d
    T = ids.shape[0]
    onehot = 2 * 2 * H * len(set(ids.ravel().tolist()))
    total = len(set(ids.ravel().tolist())) * expert + expert + lora + head + onehot
    return total / T


def _run(sh, seed, T, family=None, label=""):
    import torch
    from routing_predicted_experts_gb300 import binding as B, model as M
    lay = M.build_layer(seed, 0, sh)
    olay = OM.layer(seed, 0, sh)
    H = np.stack([S.normal_bf16(seed, f"mt.h{t}", (sh.d,)) for t in range(T)])
    Z = np.stack([S.normal_f32(seed, f"mt.z{t}", (sh.E,)) for t in range(T)]).astype(np.float64)
    Zp = np.stack([S.normal_f32(seed, f"mt.zp{t}", (sh.E,)) for t in range(T)]).astype(np.float64)
    ids = np.stack([OR.route(Z[t], sh.K, family)[0] for t in range(T)]).astype(np.int32)
    prev = np.stack([OR.route(Zp[t], sh.K, family)[0] for t in range(T)]).astype(np.int32)
    dm = B.dims(sh.d, sh.E, sh.F, sh.K, family)
    ws = B.e0_decode_workspace(dm, T, lay["lora"].out, sh.H)
    out = B.e0_moe_decode_layer(dm, lay["routed"], lay["shared"], lay["lora"], lay["head"], bf16_dev(H),
                                to_dev(ids, torch.int32), to_dev(Z.astype(np.float32), torch.float32),
                                to_dev(prev, torch.int32), ws)
    torch.cuda.synchronize()
    assert B.e0_get_device_status(ws) == 0
    got_d, ref_d, got_h, ref_h = [], [], [], []
    for t in range(T):
        ref = OL.layer_step(H[t], olay, ids[t], Z[t].astype(np.float32).astype(np.float64), prev[t], sh.K, family,
                            family)
        got_d.append(out["delta"][t].cpu().numpy())
        ref_d.append(ref["delta"])
        got_h.append(bf16_host(out["h_out"][t]))
        ref_h.append(ref["h_out"])
        zg = out["next_logits"][t].cpu().numpy().astype(np.float64)
        check_protocol(zg, ref["next_logits"], f"{label} next_logits t{t}")
        gi = out["next_ids"][t].cpu().numpy()
        check_route(gi, ref["next_logits"], sh.K, f"{label} next_ids t{t}", family)
        assert np.abs(out["next_weights"][t].cpu().numpy() - OR.route_weights(zg, gi, family)).max() <= 1e-5
    check_protocol(np.stack(got_d), np.stack(ref_d), f"{label} delta")
    check_bf16_protocol(np.stack(got_h), np.stack(ref_h), f"{label} h_out")
    return ids


@pytest.mark.parametrize("T", [2, 8, 16])
def test_multi_token_35b_layer(T):
    sh = S.LAYER35B(4)
    ids = _run(sh, 0, T, label=f"35B T={T}")
    REPORT.append(f"multi-token decode, 35B-class layer K=4, T={T}: {len(set(ids.ravel().tolist()))} distinct "
                  f"experts, {_bytes_per_token(sh, ids, sh.H) / 1e6:.2f} MB of weights read per token "
                  f"(T=1: {_bytes_per_token(sh, ids[:1], sh.H) / 1e6:.2f} MB)")


def test_multi_token_tiny_odd_count_sigmoid_group():
    sh = S.LayerShape(d=256, E=64, F=128, K=8, H=64, r=4, alpha=8.0, shared=True)
    fam = {"kind": "sigmoid_group", "n_group": 8, "topk_group": 4, "scale": 2.5}
    _run(sh, 4, 5, fam, label="tiny sigmoid-group T=5")


def test_multi_token_prerouter_forward():
    import torch
    from routing_predicted_experts_gb300 import binding as B, model as M
    sh, seed, T = S.LAYER35B(8), 1, 7
    lay = M.build_layer(seed, 0, sh)
    hd = OM.head_weights(seed, 0, sh)
    H = np.stack([S.normal_bf16(seed, f"pf.h{t}", (sh.d,)) for t in range(T)])
    cur = np.stack([OR.softmax_topk(S.normal_f32(seed, f"c{t}", (sh.E,)), sh.K)[0] for t in range(T)])
    prev = np.stack([OR.softmax_topk(S.normal_f32(seed, f"p{t}", (sh.E,)), sh.K)[0] for t in range(T)])
    dm = B.dims(sh.d, sh.E, sh.F, sh.K)
    ws = B.e0_decode_workspace(dm, T, 0, sh.H)
    z, ids, w = B.e0_prerouter_forward(lay["head"], sh.d, sh.E, sh.K, bf16_dev(H), to_dev(cur, torch.int32),
                                       to_dev(prev, torch.int32), ws)
    torch.cuda.synchronize()
    assert B.e0_get_device_status(ws) == 0
    for t in range(T):
        x = OL.rmsnorm(OB_bf16(H[t]))
        ref = OL.prerouter_logits(x, cur[t], prev[t], hd)
        zg = z[t].cpu().numpy().astype(np.float64)
        check_protocol(zg, ref, f"head logits t{t}")
        check_route(ids[t].cpu().numpy(), ref, sh.K, f"head ids t{t}")
        assert np.abs(w[t].cpu().numpy() - OR.renorm_weights(zg, ids[t].cpu().numpy())).max() <= 1e-5


def OB_bf16(bits):
    from oracle import bf16 as OB
    return OB.bf16_to_f64(bits)
