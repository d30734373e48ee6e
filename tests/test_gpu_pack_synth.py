"""GPU packer and GPU generator against their CPU definitions (bit-exact)."""
import numpy as np
import pytest

from oracle import int4 as OI
from routing_predicted_experts_gb300 import synth as S

pytestmark = pytest.mark.gpu


def test_gpu_generator_matches_numpy_bit_exact():
    import torch
    from routing_predicted_experts_gb300 import binding as B
    for name, sigma, n, off in [("L3.E7.gate", 0.02, 100_003, 0), ("hidden.s0", 1.0, 4096, 17),
                                ("x", 0.5, 1000, 123_456)]:
        g = torch.empty(n, dtype=torch.float32, device="cuda")
        B.e0_synth_normal(g, 5, S.stream_id(name), off, sigma)
        ref = S.normal_f32(5, name, (n,), sigma, offset=off)
        assert np.array_equal(g.cpu().numpy().view(np.uint32), ref.view(np.uint32)), name
        gb = torch.empty(n, dtype=torch.int16, device="cuda")
        B.e0_synth_normal(gb, 5, S.stream_id(name), off, sigma)
        assert np.array_equal(gb.cpu().numpy().view(np.uint16), S.bf16_bits(ref)), name


@pytest.mark.parametrize("rows,cols,batch", [(32, 256, 1), (48, 2048, 2), (16, 64, 3), (1024, 512, 1)])
def test_gpu_pack_matches_oracle(rows, cols, batch):
    import torch
    from routing_predicted_experts_gb300 import binding as B, _lib
    rng = np.random.default_rng(rows + cols)
    w = (rng.standard_normal((batch, rows, cols)) * 0.02).astype(np.float32)
    # edge cases: constant group, huge dynamic range, exact-code group, negative-only group
    w[0, 0, :64] = 0.25
    w[0, 1, :64] = np.linspace(-1e-30, 3e3, 64, dtype=np.float32)
    w[0, 2, :64] = (-0.75 + 0.0625 * (np.arange(64) % 16)).astype(np.float32)
    w[-1, -1, -64:] = -np.abs(w[-1, -1, -64:]) - 1.0
    gw = torch.from_numpy(w).cuda()
    for layout in (_lib.E0_LAYOUT_ROWS, _lib.E0_LAYOUT_COLSLAB):
        out = B.e0_pack_int4(gw, layout)
        q = out.q.cpu().numpy().view(np.uint32)
        s = out.scale.cpu().numpy().view(np.uint16)
        b = out.bias.cpu().numpy().view(np.uint16)
        for bt in range(batch):
            rq, rs, rb = OI.pack(w[bt])
            if layout == _lib.E0_LAYOUT_COLSLAB:
                rq, rs, rb = OI.to_column_slab(rq, rs, rb)
            nq, ns = rq.size, rs.size
            assert np.array_equal(q[bt * nq:(bt + 1) * nq], rq.ravel()), (layout, bt)
            assert np.array_equal(s[bt * ns:(bt + 1) * ns], rs.ravel()), (layout, bt)
            assert np.array_equal(b[bt * ns:(bt + 1) * ns], rb.ravel()), (layout, bt)
