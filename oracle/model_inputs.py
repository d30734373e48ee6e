"""Oracle-side view of the seeded synthetic model (test infrastructure only).

Draws the same fp32 / bf16 tensors as the CUDA side from
``routing_predicted_experts_gb300.synth`` (the shared generator module, which holds
no layer arithmetic) and quantises the int4 ones with the oracle's own packer.
Generated tensors are cached per (seed, name).
"""
from functools import lru_cache

import numpy as np

from routing_predicted_experts_gb300 import synth as S

from . import int4


@lru_cache(maxsize=None)
def _f32(seed: int, name: str, shape: tuple, sigma: float) -> np.ndarray:
    a = S.normal_f32(seed, name, shape, sigma)
    a.setflags(write=False)
    return a


@lru_cache(maxsize=None)
def _bf16(seed: int, name: str, shape: tuple, sigma: float) -> np.ndarray:
    a = S.bf16_bits(_f32(seed, name, shape, sigma))
    a.setflags(write=False)
    return a


@lru_cache(maxsize=None)
def _dq(seed: int, name: str, shape: tuple) -> np.ndarray:
    w = int4.quantize_dequantize(_f32(seed, name, shape, S.W_SIGMA))
    w.setflags(write=False)
    return w


def expert_weights(seed: int, layer: int, e: int, sh: S.LayerShape):
    return (_dq(seed, S.t_expert(layer, e, "gate"), (sh.F, sh.d)),
            _dq(seed, S.t_expert(layer, e, "up"), (sh.F, sh.d)),
            _dq(seed, S.t_expert(layer, e, "down"), (sh.d, sh.F)))


def shared_weights(seed: int, layer: int, sh: S.LayerShape):
    if not sh.shared:
        return None
    return (_dq(seed, S.t_shared(layer, "gate"), (sh.F, sh.d)),
            _dq(seed, S.t_shared(layer, "up"), (sh.F, sh.d)),
            _dq(seed, S.t_shared(layer, "down"), (sh.d, sh.F)))


def lora_weights(seed: int, layer: int, sh: S.LayerShape):
    W = _dq(seed, S.t_lora(layer, "W"), (sh.lora_rows, sh.d))
    if sh.r == 0:
        return (W, None, None, sh.alpha, 0)
    A = _bf16(seed, S.t_lora(layer, "A"), (sh.r, sh.d), S.W_SIGMA)
    B = _bf16(seed, S.t_lora(layer, "B"), (sh.lora_rows, sh.r), S.W_SIGMA)
    return (W, A, B, sh.alpha, sh.r)


def head_weights(seed: int, layer: int, sh: S.LayerShape):
    hd = {"Lres": _bf16(seed, S.t_head(layer, "Lres"), (sh.E, sh.d), S.W_SIGMA),
          "b2": _bf16(seed, S.t_head(layer, "b2"), (sh.E,), S.W_SIGMA),
          "W1": None, "b1": None, "W2": None}
    if sh.H > 0:
        hd["W1"] = _bf16(seed, S.t_head(layer, "W1"), (sh.H, sh.d + 2 * sh.E), S.W_SIGMA)
        hd["b1"] = _bf16(seed, S.t_head(layer, "b1"), (sh.H,), S.W_SIGMA)
        hd["W2"] = _bf16(seed, S.t_head(layer, "W2"), (sh.E, sh.H), S.W_SIGMA)
    return hd


def router_weights(seed: int, layer: int, sh: S.LayerShape) -> np.ndarray:
    return _bf16(seed, S.t_router(layer), (sh.E, sh.d), S.W_SIGMA)


def layer(seed: int, layer_idx: int, sh: S.LayerShape, with_head: bool = True,
          with_lora: bool = True) -> dict:
    return {
        "expert": lambda e: expert_weights(seed, layer_idx, e, sh),
        "shared": shared_weights(seed, layer_idx, sh),
        "lora": lora_weights(seed, layer_idx, sh) if with_lora else None,
        "head": head_weights(seed, layer_idx, sh) if with_head else None,
    }


def hidden(seed: int, step: int, d: int) -> np.ndarray:
    return _bf16(seed, S.t_hidden(step), (d,), S.H_SIGMA)


def increment(seed: int, step: int, layer_idx: int, d: int) -> np.ndarray:
    return _bf16(seed, S.t_increment(step, layer_idx), (d,), S.H_SIGMA)


def supplied_logits(seed: int, which: str, E: int) -> np.ndarray:
    return _f32(seed, S.t_logits(which), (E,), S.H_SIGMA)
