"""The C ABI library builds, loads and exports every function include/e0.h declares (CPU only)."""
import os
import re

from routing_predicted_experts_gb300 import _lib
from routing_predicted_experts_gb300 import build as B

HDR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "e0.h")


def declared_functions():
    text = open(HDR).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(e0_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ["e0_pack_int4", "e0_prerouter_forward", "e0_moe_decode_layer", "e0_qlinear_lora",
                     "e0_stack_create", "e0_stack_step", "e0_last_error", "e0_get_device_status"]:
        assert required in names


def test_library_exports_every_declared_symbol():
    B.build()
    lib = _lib.lib()
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert set(_lib.PROTOTYPES) <= set(declared_functions())


def test_host_side_argument_errors_without_gpu():
    lib = _lib.lib()
    # NULL arguments are rejected before any CUDA call
    st = lib.e0_pack_int4(None, 1, 1, 64, 64, 0, None, None, None, None)
    assert st == -1 and b"null" in lib.e0_last_error().lower()
    dm = _lib.e0_dims(300, 256, 512, 4)
    assert lib.e0_workspace_size(None, 1) == 0
    st = lib.e0_moe_decode_layer(dm, None, None, None, None, None, None, None, None, 1, None, None, None, None,
                                 None, None, 0, None)
    assert st == -2  # d = 300 unsupported


def test_routing_family_parameters_are_checked_without_gpu():
    lib = _lib.lib()
    bad_groups = _lib.e0_dims(256, 64, 128, 8, _lib.E0_ROUTE_SIGMOID_GROUP, 7, 4, 2.5, None)  # 7 does not divide 64
    st = lib.e0_moe_decode_layer(bad_groups, None, None, None, None, None, None, None, None, 1, None, None, None, None,
                                 None, None, 0, None)
    assert st == _lib.E0_ERR_SHAPE
    too_few = _lib.e0_dims(256, 64, 128, 8, _lib.E0_ROUTE_SIGMOID_GROUP, 8, 0, 2.5, None)  # no group kept
    assert lib.e0_moe_decode_layer(too_few, None, None, None, None, None, None, None, None, 1, None, None, None, None,
                                   None, None, 0, None) == _lib.E0_ERR_SHAPE
    unknown = _lib.e0_dims(256, 64, 128, 8, 5, 0, 0, 0.0, None)
    assert lib.e0_moe_decode_layer(unknown, None, None, None, None, None, None, None, None, 1, None, None, None, None,
                                   None, None, 0, None) == _lib.E0_ERR_UNSUPPORTED


def test_misaligned_prefill_weights_are_refused_without_gpu():
    """The grouped path copies codes and reads scales with vector accesses: int4 arrays that
    are not 16-byte aligned come back as an argument error before any CUDA call."""
    lib = _lib.lib()
    dm = _lib.e0_dims(256, 16, 128, 4)
    base = 1 << 20  # never dereferenced: the call returns at the argument checks

    def q4(off):
        return _lib.e0_q4(base + off, base + 4096 + off, base + 8192 + off)

    good = _lib.e0_experts(q4(0), q4(0), 16, None, 0, None)
    bad = _lib.e0_experts(_lib.e0_q4(base, base + 4098, base + 8192), q4(0), 16, None, 0, None)
    def call(experts, ws_bytes):
        # h_in, logits, T, h_out, delta, ids_out, weights_out, workspace, bytes, stream
        return lib.e0_moe_prefill_layer(dm, experts, None, None, base, base, 4, base, None, None, None, base, ws_bytes,
                                        None)

    assert call(bad, 1 << 30) == _lib.E0_ERR_INVALID
    assert b"aligned" in lib.e0_last_error()
    # with aligned weights the checks go on to the workspace size (none given here)
    assert call(good, 0) == -5  # E0_ERR_NOMEM
