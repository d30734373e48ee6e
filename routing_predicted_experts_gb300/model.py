"""Synthetic model weights built on the GPU: seeded draws (e0_synth_normal) packed
with e0_pack_int4 into the layouts the engine streams.

Tensor names and shapes come from ``synth`` so the oracle can draw the same values
on the host.  bf16 tensors are held as int16 bit patterns.
"""
from __future__ import annotations

import torch

from . import synth as S
from ._lib import E0_LAYOUT_COLSLAB, E0_LAYOUT_ROWS
from .binding import Experts, Prerouter, Q4, QLora, e0_pack_int4, e0_synth_normal


def draw(shape, seed: int, name: str, sigma: float, bf16: bool = False, device="cuda") -> torch.Tensor:
    out = torch.empty(shape, dtype=torch.int16 if bf16 else torch.float32, device=device)
    e0_synth_normal(out, seed, S.stream_id(name), 0, sigma)
    return out


def _q4_empty(n: int, rows: int, cols: int, device) -> Q4:
    q = torch.empty(n * rows * cols // 8, dtype=torch.int32, device=device)
    s = torch.empty(n * rows * cols // 64, dtype=torch.int16, device=device)
    return Q4(q, s, torch.empty_like(s))


def _view(q4: Q4, lo: int, hi: int, rows: int, cols: int) -> Q4:
    """Experts lo..hi of a flat stacked Q4 (both layouts keep experts contiguous)."""
    wq, ws = rows * cols // 8, rows * cols // 64
    return Q4(q4.q[lo * wq: hi * wq], q4.scale[lo * ws: hi * ws], q4.bias[lo * ws: hi * ws])


def build_experts(seed: int, names, n: int, F: int, d: int, device="cuda", chunk: int = 16) -> Experts:
    """names(e, which) -> tensor name.  gate_up rows interleaved (2j gate, 2j+1 up)."""
    gu = _q4_empty(n, 2 * F, d, device)
    dn = _q4_empty(n, d, F, device)
    for e0 in range(0, n, chunk):
        m = min(chunk, n - e0)
        w = torch.empty((m, F, 2, d), dtype=torch.float32, device=device)
        wd = torch.empty((m, d, F), dtype=torch.float32, device=device)
        for j in range(m):
            e = e0 + j
            w[j, :, 0, :] = draw((F, d), seed, names(e, "gate"), S.W_SIGMA, device=device)
            w[j, :, 1, :] = draw((F, d), seed, names(e, "up"), S.W_SIGMA, device=device)
            wd[j] = draw((d, F), seed, names(e, "down"), S.W_SIGMA, device=device)
        e0_pack_int4(w.view(m, 2 * F, d), E0_LAYOUT_ROWS, out=_view(gu, e0, e0 + m, 2 * F, d))
        e0_pack_int4(wd, E0_LAYOUT_COLSLAB, out=_view(dn, e0, e0 + m, d, F))
        del w, wd
    return Experts(gu, dn, n)


def build_lora(seed: int, layer: int, sh: S.LayerShape, device="cuda") -> QLora:
    rows = sh.lora_rows
    W = draw((rows, sh.d), seed, S.t_lora(layer, "W"), S.W_SIGMA, device=device)
    w = e0_pack_int4(W, E0_LAYOUT_ROWS)
    if sh.r == 0:
        return QLora(w, None, None, rows, 0, sh.alpha)
    A = draw((sh.r, sh.d), seed, S.t_lora(layer, "A"), S.W_SIGMA, bf16=True, device=device)
    B = draw((rows, sh.r), seed, S.t_lora(layer, "B"), S.W_SIGMA, bf16=True, device=device)
    return QLora(w, A, B.t().contiguous(), rows, sh.r, sh.alpha)


def build_head(seed: int, layer: int, sh: S.LayerShape, device="cuda") -> Prerouter:
    d, E, H = sh.d, sh.E, sh.H
    lres = draw((E, d), seed, S.t_head(layer, "Lres"), S.W_SIGMA, bf16=True, device=device)
    b2 = draw((E,), seed, S.t_head(layer, "b2"), S.W_SIGMA, bf16=True, device=device)
    if H == 0:
        return Prerouter(0, None, None, None, None, None, b2, lres)
    W1 = draw((H, d + 2 * E), seed, S.t_head(layer, "W1"), S.W_SIGMA, bf16=True, device=device)
    b1 = draw((H,), seed, S.t_head(layer, "b1"), S.W_SIGMA, bf16=True, device=device)
    W2 = draw((E, H), seed, S.t_head(layer, "W2"), S.W_SIGMA, bf16=True, device=device)
    return Prerouter(H, W1[:, :d].contiguous(), W1[:, d:d + E].t().contiguous(),
                     W1[:, d + E:].t().contiguous(), b1, W2.t().contiguous(), b2, lres)


def build_layer(seed: int, layer: int, sh: S.LayerShape, with_head: bool = True, with_lora: bool = True,
                device="cuda") -> dict:
    routed = build_experts(seed, lambda e, w: S.t_expert(layer, e, w), sh.E, sh.F, sh.d, device)
    shared = build_experts(seed, lambda e, w: S.t_shared(layer, w), 1, sh.F, sh.d, device) if sh.shared else None
    return {
        "routed": routed,
        "shared": shared,
        "lora": build_lora(seed, layer, sh, device) if with_lora else None,
        "head": build_head(seed, layer, sh, device) if with_head else None,
        "router": draw((sh.E, sh.d), seed, S.t_router(layer), S.W_SIGMA, bf16=True, device=device),
    }


def hidden(seed: int, step: int, d: int, device="cuda") -> torch.Tensor:
    return draw((d,), seed, S.t_hidden(step), S.H_SIGMA, bf16=True, device=device)


def increments(seed: int, step: int, L: int, d: int, device="cuda") -> torch.Tensor:
    out = torch.empty((L, d), dtype=torch.int16, device=device)
    for l in range(L):
        e0_synth_normal(out[l], seed, S.stream_id(S.t_increment(step, l)), 0, S.H_SIGMA)
    return out
