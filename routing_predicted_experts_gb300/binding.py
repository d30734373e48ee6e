"""Thin Python binding over libe0 (argument marshalling only; every step runs in the
library's CUDA kernels).  Names follow the C ABI in include/e0.h.

Tensors are torch tensors on the current CUDA device; bf16 data is carried in
``torch.int16``/``torch.bfloat16`` tensors and passed as raw bit patterns.  All calls
are enqueued on ``torch.cuda.current_stream()`` unless a stream is given.
"""
from __future__ import annotations

import ctypes as C
from dataclasses import dataclass
from typing import Optional

import torch

from . import _lib as L
from ._lib import check, lib


def _p(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _event(ev) -> Optional[int]:
    """cudaEvent_t of a torch.cuda.Event (None -> NULL); the event must have been recorded."""
    if ev is None:
        return None
    return int(ev.cuda_event)


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


# ------------------------------------------------------------------ data holders
@dataclass
class Q4:
    q: torch.Tensor       # int32 words
    scale: torch.Tensor   # bf16 bits (int16)
    bias: torch.Tensor

    def c(self) -> L.e0_q4:
        return L.e0_q4(_p(self.q), _p(self.scale), _p(self.bias))


@dataclass
class Experts:
    gate_up: Q4           # row layout [n][2F][d], rows interleaved gate/up
    down: Q4              # column-slab layout [n][d][F]
    n: int
    slot_of: Optional[torch.Tensor] = None   # int16 [E]
    stride: int = 0                           # bytes between stored experts (slot bundles); 0 = dense

    def c(self) -> L.e0_experts:
        return L.e0_experts(self.gate_up.c(), self.down.c(), self.n, _p(self.slot_of), self.stride)


@dataclass
class QLora:
    w: Q4                 # row layout [out][in]
    a: Optional[torch.Tensor]   # bf16 [r][in]
    bt: Optional[torch.Tensor]  # bf16 [r][out]
    out: int
    r: int
    alpha: float

    def c(self) -> L.e0_qlora:
        return L.e0_qlora(self.w.c(), _p(self.a), _p(self.bt), self.out, self.r, self.alpha)


@dataclass
class Prerouter:
    H: int
    w1h: Optional[torch.Tensor]
    w1c_t: Optional[torch.Tensor]
    w1p_t: Optional[torch.Tensor]
    b1: Optional[torch.Tensor]
    w2t: Optional[torch.Tensor]
    b2: Optional[torch.Tensor]
    lres: torch.Tensor

    def c(self) -> L.e0_prerouter:
        return L.e0_prerouter(self.H, _p(self.w1h), _p(self.w1c_t), _p(self.w1p_t), _p(self.b1), _p(self.w2t),
                              _p(self.b2), _p(self.lres))


def dims(d: int, E: int, F: int, K: int, family: Optional[dict] = None,
         score_bias: Optional[torch.Tensor] = None) -> L.e0_dims:
    """Layer dimensions and routing family: None = softmax-top-K, or a dict
    {"kind": "sigmoid_group", "n_group", "topk_group", "scale"}; score_bias (device fp32
    [E], sigmoid-group only) is the selection bias of the routing a single-layer call
    chooses."""
    dm = L.e0_dims(d, E, F, K)
    if family is not None:
        assert family["kind"] == "sigmoid_group"
        dm.route = L.E0_ROUTE_SIGMOID_GROUP
        dm.n_group = int(family["n_group"])
        dm.topk_group = int(family["topk_group"])
        dm.route_scale = float(family["scale"])
        dm.score_bias = _p(score_bias)
        dm._keepalive = score_bias  # the struct holds only the address
    return dm


# ------------------------------------------------------------------ calls
def e0_pack_int4(w: torch.Tensor, layout: int = L.E0_LAYOUT_ROWS, out: Optional[Q4] = None, stream=None) -> Q4:
    """fp32 [batch][rows][cols] (or [rows][cols]) -> packed int4 in the given layout.

    ``out`` (optional) receives the result in caller-provided flat tensors."""
    if w.dim() == 2:
        w = w.unsqueeze(0)
    assert w.dtype == torch.float32
    b, rows, cols = w.shape
    if out is None:
        q = torch.empty(b * rows * cols // 8, dtype=torch.int32, device=w.device)
        s = torch.empty(b * rows * cols // 64, dtype=torch.int16, device=w.device)
        out = Q4(q, s, torch.empty_like(s))
    assert out.q.numel() == b * rows * cols // 8 and out.scale.numel() == b * rows * cols // 64
    check(lib().e0_pack_int4(_p(w.contiguous()), b, rows, cols, 64, layout, _p(out.q), _p(out.scale),
                             _p(out.bias), _stream(stream)))
    return out


def e0_decode_workspace(dm: L.e0_dims, T: int, lora_out: int = 0, H: int = 0, device=None) -> torch.Tensor:
    """Zeroed workspace of e0_moe_decode_layer / e0_prerouter_forward for T tokens."""
    n = lib().e0_decode_workspace_size(C.byref(dm), T, lora_out, H)
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def e0_workspace(dm: L.e0_dims, layers: int = 1, device=None) -> torch.Tensor:
    n = lib().e0_workspace_size(C.byref(dm), layers)
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def e0_workspace_reset(ws: torch.Tensor, stream=None) -> None:
    check(lib().e0_workspace_reset(_p(ws), ws.numel(), _stream(stream)))


def e0_get_device_status(ws: torch.Tensor, stream=None) -> int:
    v = L.u32(0)
    check(lib().e0_get_device_status(_p(ws), C.byref(v), _stream(stream)))
    return int(v.value)


def e0_debug_inject_stall(ws: torch.Tensor, limit_ns: int, stream=None) -> None:
    check(lib().e0_debug_inject_stall(_p(ws), limit_ns, _stream(stream)))


def e0_synth_normal(out: torch.Tensor, seed: int, stream_id: int, offset: int = 0, sigma: float = 1.0,
                    stream=None) -> torch.Tensor:
    bf = 1 if out.dtype in (torch.int16, torch.bfloat16) else 0
    if not bf:
        assert out.dtype == torch.float32
    check(lib().e0_synth_normal(_p(out), out.numel(), seed, stream_id, offset, sigma, bf, _stream(stream)))
    return out


def e0_moe_decode_layer(dm: L.e0_dims, routed: Experts, shared: Optional[Experts], lora: Optional[QLora],
                        head: Optional[Prerouter], h_in: torch.Tensor, ids: torch.Tensor, logits: torch.Tensor,
                        ids_prev: Optional[torch.Tensor], ws: torch.Tensor, want_delta: bool = True, stream=None):
    """Returns dict(h_out, delta, next_logits, next_ids, next_weights) for T = h_in.shape[0] tokens."""
    T = h_in.shape[0] if h_in.dim() == 2 else 1
    dev = h_in.device
    h_out = torch.empty((T, dm.d), dtype=torch.int16, device=dev)
    delta = torch.empty((T, dm.d), dtype=torch.float32, device=dev) if want_delta else None
    nl = ni = nw = None
    if head is not None:
        nl = torch.empty((T, dm.E), dtype=torch.float32, device=dev)
        ni = torch.empty((T, dm.K), dtype=torch.int32, device=dev)
        nw = torch.empty((T, dm.K), dtype=torch.float32, device=dev)
    r, s_, l_, h_ = routed.c(), (shared.c() if shared else None), (lora.c() if lora else None), \
        (head.c() if head else None)
    check(lib().e0_moe_decode_layer(C.byref(dm), C.byref(r), C.byref(s_) if s_ else None,
                                    C.byref(l_) if l_ else None, C.byref(h_) if h_ else None, _p(h_in), _p(ids),
                                    _p(logits), _p(ids_prev), T, _p(h_out), _p(delta), _p(nl), _p(ni), _p(nw),
                                    _p(ws), ws.numel(), _stream(stream)))
    return {"h_out": h_out, "delta": delta, "next_logits": nl, "next_ids": ni, "next_weights": nw}


def e0_prefill_workspace(dm: L.e0_dims, T: int, lora_out: int = 0, device=None) -> torch.Tensor:
    n = lib().e0_prefill_workspace_size(C.byref(dm), T, lora_out)
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def e0_moe_prefill_layer(dm: L.e0_dims, routed: Experts, shared: Optional[Experts], lora: Optional[QLora],
                         h_in: torch.Tensor, logits: torch.Tensor, ws: torch.Tensor, want_delta: bool = True,
                         stream=None):
    """T tokens (h_in bf16 bits [T][d], logits fp32 [T][E]) through one layer on the tensor cores.
    Returns dict(h_out, delta, ids, weights)."""
    T = h_in.shape[0]
    dev = h_in.device
    h_out = torch.empty((T, dm.d), dtype=torch.int16, device=dev)
    delta = torch.empty((T, dm.d), dtype=torch.float32, device=dev) if want_delta else None
    ids = torch.empty((T, dm.K), dtype=torch.int32, device=dev)
    w = torch.empty((T, dm.K), dtype=torch.float32, device=dev)
    r, s_, l_ = routed.c(), (shared.c() if shared else None), (lora.c() if lora else None)
    check(lib().e0_moe_prefill_layer(C.byref(dm), C.byref(r), C.byref(s_) if s_ else None,
                                     C.byref(l_) if l_ else None, _p(h_in), _p(logits), T, _p(h_out), _p(delta),
                                     _p(ids), _p(w), _p(ws), ws.numel(), _stream(stream)))
    return {"h_out": h_out, "delta": delta, "ids": ids, "weights": w}


def e0_prerouter_forward(head: Prerouter, d: int, E: int, K: int, h: torch.Tensor, ids_cur, ids_prev,
                         ws: torch.Tensor, logit_bias=None, stream=None):
    T = h.shape[0] if h.dim() == 2 else 1
    dev = h.device
    logits = torch.empty((T, E), dtype=torch.float32, device=dev)
    ids = torch.empty((T, K), dtype=torch.int32, device=dev)
    w = torch.empty((T, K), dtype=torch.float32, device=dev)
    hc = head.c()
    check(lib().e0_prerouter_forward(C.byref(hc), d, E, _p(h), _p(ids_cur), _p(ids_prev), T, K, _p(logit_bias),
                                     _p(logits), _p(ids), _p(w), _p(ws), ws.numel(), _stream(stream)))
    return logits, ids, w


def e0_qlinear_lora(lora: QLora, x: torch.Tensor, ws: torch.Tensor, y: Optional[torch.Tensor] = None,
                    accumulate: bool = False, want_f32: bool = True, stream=None):
    T = x.shape[0] if x.dim() == 2 else 1
    inn = x.shape[-1]
    if y is None:
        y = torch.zeros((T, lora.out), dtype=torch.int16, device=x.device)
    yf = torch.empty((T, lora.out), dtype=torch.float32, device=x.device) if want_f32 else None
    lc = lora.c()
    check(lib().e0_qlinear_lora(C.byref(lc), inn, _p(x), T, 1 if accumulate else 0, _p(y), _p(yf), _p(ws),
                                ws.numel(), _stream(stream)))
    return y, yf


class Stack:
    """Owns an e0_stack (layer descriptors + work plan on the device)."""

    def __init__(self, dm: L.e0_dims, layers: list, route_src: list[int], keepalive=None):
        """route_src[l]: 1 routed by head l-1 (after the first token), 0 own gate, -N
        route-ahead by N layers."""
        self.dm = dm
        self.L = len(layers)
        arr = (L.e0_layer * self.L)()
        for i, ly in enumerate(layers):
            arr[i] = ly
        pre = (C.c_int8 * self.L)(*route_src)
        h = C.c_void_p()
        check(lib().e0_stack_create(C.byref(h), C.byref(dm), arr, self.L, C.cast(pre, C.c_void_p)))
        self.handle = h
        self.keepalive = keepalive

    def workspace(self, device=None) -> torch.Tensor:
        n = lib().e0_stack_workspace_size(self.handle)
        return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")

    def step(self, step: int, h0: torch.Tensor, incr: torch.Tensor, h_out: torch.Tensor, ws: torch.Tensor,
             ids_out=None, w_out=None, h_trace=None, stream=None, logit_bias=None, delta=None, logits=None,
             next_ids=None, commit_box=None) -> None:
        """One token; the optional outputs are e0_stack_outputs' (ids, weights, h_trace,
        delta, logits [2][L][E], next_ids, commit_box: a CommitBox)."""
        outs = None
        if any(t is not None for t in (ids_out, w_out, h_trace, delta, logits, next_ids, commit_box)):
            outs = L.e0_stack_outputs(_p(ids_out), _p(w_out), _p(h_trace), _p(delta), _p(logits), _p(next_ids),
                                      commit_box.device if commit_box is not None else None)
        check(lib().e0_stack_step(self.handle, step, _p(h0), _p(incr), _p(h_out),
                                  C.byref(outs) if outs is not None else None, _p(logit_bias), _p(ws), ws.numel(),
                                  _stream(stream)))

    def close(self):
        if self.handle:
            lib().e0_stack_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def e0_layer_struct(routed: Experts, shared: Optional[Experts], lora: Optional[QLora], head: Optional[Prerouter],
                    router: torch.Tensor, score_bias: Optional[torch.Tensor] = None) -> L.e0_layer:
    ly = L.e0_layer()
    ly.score_bias = _p(score_bias)
    ly.routed = routed.c()
    if shared is not None:
        ly.shared = shared.c()
    if lora is not None:
        ly.lora = lora.c()
    if head is not None:
        ly.head = head.c()
    ly.router = _p(router)
    return ly


# ------------------------------------------------------------------ slot pool
def expert_bundle_layout(dm: L.e0_dims):
    """(bundle bytes, offsets of the six tensors) of one expert bundle."""
    offs = (C.c_size_t * 6)()
    total = lib().e0_expert_bundle_bytes(C.byref(dm), C.cast(offs, C.c_void_p))
    return int(total), [int(o) for o in offs]


def host_bundles(dm: L.e0_dims, stacks: list, pin: bool = True) -> torch.Tensor:
    """Pinned host bundles [len(stacks)][E][bundle] from dense device expert stacks (n == E)."""
    total, offs = expert_bundle_layout(dm)
    E = dm.E
    hb = torch.zeros((len(stacks), E, total), dtype=torch.uint8, pin_memory=pin)
    for l, ex in enumerate(stacks):
        parts = [ex.gate_up.q, ex.gate_up.scale, ex.gate_up.bias, ex.down.q, ex.down.scale, ex.down.bias]
        for off, t in zip(offs, parts):
            src = t.contiguous().view(torch.uint8).reshape(E, -1)
            hb[l, :, off:off + src.shape[1]].copy_(src.cpu())
    return hb


class _RawExperts:
    def __init__(self, st: L.e0_experts):
        self.st = st

    def c(self) -> L.e0_experts:
        return self.st


class SlotPool:
    """Owns an e0_slot_pool: per layer, `slots` HBM bundle slots over pinned host bundles."""

    def __init__(self, dm: L.e0_dims, layers: int, slots: int, bundles: torch.Tensor):
        total, _ = expert_bundle_layout(dm)
        assert bundles.is_pinned() and bundles.numel() == layers * dm.E * total
        h = C.c_void_p()
        check(lib().e0_slot_pool_create(C.byref(h), C.byref(dm), layers, slots, C.c_void_p(bundles.data_ptr()),
                                        total))
        self.handle = h
        self.bundles = bundles
        self.E = dm.E
        self.K = dm.K
        self.stats = L.e0_stage_stats()

    def view(self, layer: int) -> _RawExperts:
        ex = L.e0_experts()
        check(lib().e0_slot_pool_view(self.handle, layer, C.byref(ex)))
        return _RawExperts(ex)

    def stage_host(self, layers, ids, tag: int, copy_stream=None, after=None) -> None:
        """Stage HOST ids [len(layers)][K] into the given pool layers, then write `tag`
        into their ready words (priming, or a routing the host knows)."""
        import numpy as np
        lay = np.ascontiguousarray(np.asarray(layers, dtype=np.int32))
        arr = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
        check(lib().e0_stage_slots_host(self.handle, C.c_void_p(lay.ctypes.data), len(lay),
                                        C.c_void_p(arr.ctypes.data), arr.shape[-1], tag & 0xFFFFFFFF,
                                        _stream(copy_stream), _event(after), C.byref(self.stats)))

    def stage(self, layers, next_ids: torch.Tensor, rows, tag: int, copy_stream=None, after=None) -> None:
        """Stage the DEVICE ids a stack launch committed (next_ids int32 [*][K]; row rows[i]
        for pool layer layers[i]) after event `after`, then write `tag` into the ready
        words.  Blocks the calling thread until the ids have reached the host."""
        import numpy as np
        lay = np.ascontiguousarray(np.asarray(layers, dtype=np.int32))
        rw = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
        assert next_ids.dtype == torch.int32 and next_ids.is_cuda
        check(lib().e0_stage_slots(self.handle, C.c_void_p(lay.ctypes.data), len(lay), _p(next_ids),
                                   C.c_void_p(rw.ctypes.data), next_ids.shape[-1], tag & 0xFFFFFFFF,
                                   _stream(copy_stream), _event(after), C.byref(self.stats)))

    def stage_committed(self, box: "CommitBox", layers, rows, tag: int, copy_stream=None,
                        timeout_ns: int = 2_000_000_000) -> None:
        """Stage token `tag` from the commit box as the running launch commits each layer
        (rows[i]: the stack layer of pool layer layers[i]); returns when every layer's
        copies are queued."""
        import numpy as np
        lay = np.ascontiguousarray(np.asarray(layers, dtype=np.int32))
        rw = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
        check(lib().e0_stage_slots_committed(self.handle, box.handle, C.c_void_p(lay.ctypes.data),
                                             C.c_void_p(rw.ctypes.data), len(lay), self.K, tag & 0xFFFFFFFF,
                                             _stream(copy_stream), timeout_ns, C.byref(self.stats)))

    def resident(self, layer: int):
        """The pool's own id -> slot table of a layer (int16 [E], -1 = absent)."""
        import numpy as np
        out = np.empty(self.E, dtype=np.int16)
        check(lib().e0_slot_pool_resident(self.handle, layer, C.c_void_p(out.ctypes.data)))
        return out

    def fail_copies(self, n: int) -> None:
        """Tests: make the (n+1)-th bundle copy from now fail as a failed copy call would."""
        check(lib().e0_debug_fail_copies(self.handle, n))

    def close(self):
        if self.handle:
            lib().e0_slot_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class CommitBox:
    """Owns an e0_commit_box: pinned host-mapped memory a stack launch writes each
    head-routed layer's committed ids into as soon as its head is done."""

    def __init__(self, layers: int):
        h = C.c_void_p()
        check(lib().e0_commit_box_create(C.byref(h), layers))
        self.handle = h
        self.device = lib().e0_commit_box_device(h)

    def close(self):
        if self.handle:
            lib().e0_commit_box_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
