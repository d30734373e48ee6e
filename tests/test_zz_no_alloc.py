"""The allocation-free layer-step entry point against the regular one.

e0_moe_decode_layer_noalloc exists for callers that cannot allocate device memory
(for example a host callback that must not enter the CUDA allocator, or a plugin
whose host framework owns all allocations): it keeps its workspace in a fixed array
inside the library.  This file is collected last so that a run stopping at the first
failure has already run every other test; it also passes on its own.
"""
import ctypes as C

import numpy as np
import pytest

from oracle import model_inputs as OM, routing as OR
from routing_predicted_experts_gb300 import synth as S

from _common import bf16_dev, check_protocol, to_dev

pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_entry_point_twice():
    import torch
    from routing_predicted_experts_gb300 import _lib, binding as B, model as M
    sh, seed = S.TINY, 5
    lay = M.build_layer(seed, 0, sh)
    dm = B.dims(sh.d, sh.E, sh.F, sh.K)
    h = bf16_dev(OM.hidden(seed, 0, sh.d))[None]
    z = OM.supplied_logits(seed, "cur", sh.E)
    ids = to_dev(OR.softmax_topk(z, sh.K)[0], torch.int32)[None]
    prev = to_dev(OR.softmax_topk(OM.supplied_logits(seed, "prev", sh.E), sh.K)[0], torch.int32)[None]
    zl = to_dev(z, torch.float32)[None]
    ws = B.e0_workspace(dm)
    ref = B.e0_moe_decode_layer(dm, lay["routed"], lay["shared"], lay["lora"], lay["head"], h, ids, zl, prev, ws)
    torch.cuda.synchronize()
    lib = _lib.lib()
    r, lo, hd = lay["routed"].c(), lay["lora"].c(), lay["head"].c()
    p = B._p
    for call in range(2):
        h_out = torch.empty((1, sh.d), dtype=torch.int16, device="cuda")
        delta = torch.empty((1, sh.d), dtype=torch.float32, device="cuda")
        nl = torch.empty((1, sh.E), dtype=torch.float32, device="cuda")
        ni = torch.empty((1, sh.K), dtype=torch.int32, device="cuda")
        nw = torch.empty((1, sh.K), dtype=torch.float32, device="cuda")
        st = lib.e0_moe_decode_layer_noalloc(C.byref(dm), C.byref(r), None, C.byref(lo), C.byref(hd), p(h), p(ids),
                                             p(zl), p(prev), p(h_out), p(delta), p(nl), p(ni), p(nw),
                                             B._stream())
        assert st == 0, lib.e0_last_error()
        torch.cuda.synchronize()
        check_protocol(delta.cpu().numpy(), ref["delta"].cpu().numpy(), f"delta call {call}")
        check_protocol(nl.cpu().numpy(), ref["next_logits"].cpu().numpy(), f"next_logits call {call}")
        ho = h_out.cpu().numpy().view(np.uint16)
        hr = ref["h_out"].cpu().numpy().view(np.uint16)
        from oracle import bf16 as OB
        check_protocol(OB.bf16_to_f64(ho), OB.bf16_to_f64(hr), f"h_out call {call}")


def test_noalloc_checks_arguments_before_queueing_anything():
    """Every valid dims fits the built-in scratch (its workspace grows only with E, and
    E = 1024 still fits); unsupported dims and missing pointers are refused with the
    shape / invalid-argument status before anything is queued on the stream."""
    import torch  # noqa: F401
    from routing_predicted_experts_gb300 import _lib, binding as B
    lib = _lib.lib()
    dm = B.dims(2048, 1024, 512, 4)
    assert lib.e0_workspace_size(C.byref(dm), 1) <= 128 * 1024
    bad = B.dims(300, 256, 512, 4)
    st = lib.e0_moe_decode_layer_noalloc(C.byref(bad), None, None, None, None, None, None, None, None, None, None,
                                         None, None, None, None)
    assert st == _lib.E0_ERR_SHAPE, st
    st = lib.e0_moe_decode_layer_noalloc(C.byref(dm), None, None, None, None, None, None, None, None, None, None,
                                         None, None, None, None)
    assert st == _lib.E0_ERR_INVALID, st
