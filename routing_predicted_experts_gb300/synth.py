"""Seeded synthetic inputs shared by the CUDA path, the oracle, the tests and the bench.

This module draws numbers and nothing else: it holds none of the layer-step
arithmetic (no quantisation, routing, expert or head math).  Both sides of every
parity test receive the same arrays from here.

Generator ("e0synth", counter based, so any slice of any tensor can be produced on
its own and the CUDA generator kernel reproduces it bit for bit):

* ``mix(z)`` is the SplitMix64 finaliser: ``z ^= z>>30; z *= 0xBF58476D1CE4E5B9;
  z ^= z>>27; z *= 0x94D049BB133111EB; z ^= z>>31`` (all arithmetic mod 2**64).
* a tensor is named by ``(seed, stream)``; ``stream`` is the CRC-32 of the tensor's
  name.  ``base = mix(seed*G + stream*H + 1)`` with ``G = 0x9E3779B97F4A7C15`` and
  ``H = 0xD1B54A32D192ED03``.
* draw ``n`` of the tensor is ``mix(base + (n+1)*G)``.
* a 24-bit uniform integer is ``draw >> 40``.
* element ``i`` of an approximately normal tensor with standard deviation ``sigma``
  is the Irwin-Hall sum of twelve uniforms: ``S = sum_{k<12} u24(12*i + k)``,
  ``v = fp32( (fp64(S - 6*2**24) * sigma) * 2**-24 )``.  Only exact integer work,
  one correctly rounded fp64 product, an exact power-of-two scale and one fp32
  rounding are involved, so numpy and CUDA produce identical bits.  The values
  have mean 0, standard deviation ``sigma`` and are bounded by ``6*sigma``.

Host-only draws (routing logits of the prefill workload, decode traces of the
slot-pool workload) use ``uniform_f64`` and ordinary numpy maths; those arrays are
generated once on the host and handed to both sides.
"""
from __future__ import annotations

import zlib

import numpy as np

_G = np.uint64(0x9E3779B97F4A7C15)
_H = np.uint64(0xD1B54A32D192ED03)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def stream_id(name: str) -> int:
    """CRC-32 of a tensor name, the ``stream`` half of its generator key."""
    return zlib.crc32(name.encode("utf-8")) & 0xFFFFFFFF


def _mix(z: np.ndarray) -> np.ndarray:
    z = z.astype(np.uint64, copy=True)
    with np.errstate(over="ignore"):
        z ^= z >> np.uint64(30)
        z *= _M1
        z ^= z >> np.uint64(27)
        z *= _M2
        z ^= z >> np.uint64(31)
    return z


def _base(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        s = np.array([seed], dtype=np.uint64) * _G + np.array([stream], dtype=np.uint64) * _H + np.uint64(1)
    return _mix(s)[0]


def draws_u64(seed: int, stream: int, index: np.ndarray) -> np.ndarray:
    """Raw 64-bit draws number ``index`` (uint64 array) of tensor ``(seed, stream)``."""
    base = _base(seed, stream)
    with np.errstate(over="ignore"):
        z = base + (index.astype(np.uint64) + np.uint64(1)) * _G
    return _mix(z)


def normal_f32(seed: int, name: str, shape, sigma: float = 1.0, offset: int = 0) -> np.ndarray:
    """Approximately N(0, sigma^2) fp32 tensor; element i uses draws 12*(offset+i)..+11.

    Computed in chunks of elements (all twelve draws of a chunk at once, in place) so
    that the temporaries stay in cache; the arithmetic is the module's definition."""
    n = int(np.prod(shape)) if len(shape) else 1
    base = _base(seed, stream_id(name))
    out = np.empty(n, dtype=np.float32)
    k = np.arange(12, dtype=np.uint64)
    chunk = 4096
    with np.errstate(over="ignore"):
        for c0 in range(0, n, chunk):
            c1 = min(n, c0 + chunk)
            i = np.arange(c0, c1, dtype=np.uint64) + np.uint64(offset)
            z = i[:, None] * np.uint64(12) + k[None, :] + np.uint64(1)   # draw index + 1
            z *= _G
            z += base
            t = z >> np.uint64(30)
            z ^= t
            z *= _M1
            np.right_shift(z, np.uint64(27), out=t)
            z ^= t
            z *= _M2
            np.right_shift(z, np.uint64(31), out=t)
            z ^= t
            z >>= np.uint64(40)                                         # 24-bit uniforms
            s = z.sum(axis=1).astype(np.int64)
            v = ((s - 6 * (1 << 24)).astype(np.float64) * np.float64(sigma)) * np.float64(2.0 ** -24)
            out[c0:c1] = v.astype(np.float32)
    return out.reshape(shape)


def uniform_f64(seed: int, name: str, shape) -> np.ndarray:
    """Uniform fp64 in [0, 1) with 53 random bits per element (host-only draws)."""
    n = int(np.prod(shape)) if len(shape) else 1
    d = draws_u64(seed, stream_id(name), np.arange(n, dtype=np.uint64))
    return ((d >> np.uint64(11)).astype(np.float64) * 2.0 ** -53).reshape(shape)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bfloat16 (round-to-nearest-even) and return the 16-bit patterns.

    Used only to hand bf16 inputs to both sides; the oracle has its own conversion.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def normal_bf16(seed: int, name: str, shape, sigma: float = 1.0, offset: int = 0) -> np.ndarray:
    return bf16_bits(normal_f32(seed, name, shape, sigma, offset))


# --------------------------------------------------------------------------------------
# Workload-specific host draws
# --------------------------------------------------------------------------------------

def zipf_gumbel_logits(seed: int, T: int, E: int, s: float = 1.1) -> np.ndarray:
    """Routing logits for a prefill chunk with skewed expert popularity.

    ``z[t][e] = log p_{pi(e)} + Gumbel(0,1)`` with ``p`` a Zipf(s) law over ranks
    1..E and ``pi`` a seeded permutation.  Taking the top-K of these logits is sampling
    K experts without replacement in proportion to ``p`` (the Gumbel-top-k trick), so
    per-expert token counts come out skewed like a real popularity law.
    """
    ranks = np.arange(1, E + 1, dtype=np.float64)
    p = ranks ** (-s)
    p /= p.sum()
    perm = np.argsort(uniform_f64(seed, "prefill.perm", (E,)), kind="stable")
    logp = np.empty(E)
    logp[perm] = np.log(p)
    u = uniform_f64(seed, "prefill.gumbel", (T, E))
    u = np.clip(u, 2.0 ** -53, 1.0 - 2.0 ** -53)
    g = -np.log(-np.log(u))
    return (logp[None, :] + g).astype(np.float32)


def popularity_for_coverage(E: int, top_frac: float = 0.525, traffic: float = 0.95) -> float:
    """Zipf exponent s such that the top ``top_frac`` of E experts carry ``traffic`` of picks."""
    k = int(round(top_frac * E))
    lo, hi = 0.0, 8.0
    for _ in range(80):
        mid = 0.5 * (lo + hi)
        p = np.arange(1, E + 1, dtype=np.float64) ** (-mid)
        share = p[:k].sum() / p.sum()
        if share < traffic:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def locality_trace(seed: int, layer: int, steps: int, E: int, K: int,
                   keep_p: float = 0.25, top_frac: float = 0.525, traffic: float = 0.95) -> np.ndarray:
    """Decode routing trace ``ids[steps][K]`` for one layer of the slot-pool workload.

    Popularity is a Zipf law over a seeded permutation, with the exponent chosen so the
    top ``top_frac`` of experts carry ``traffic`` of the picks.  Each step keeps each id of
    the previous step with probability ``keep_p`` (adjacent-token overlap) and fills the
    remaining slots in proportion to popularity, excluding ids already chosen.
    """
    s = popularity_for_coverage(E, top_frac, traffic)
    p = np.arange(1, E + 1, dtype=np.float64) ** (-s)
    perm = np.argsort(uniform_f64(seed, f"trace.L{layer}.perm", (E,)), kind="stable")
    pop = np.empty(E)
    pop[perm] = p / p.sum()
    u_keep = uniform_f64(seed, f"trace.L{layer}.keep", (steps, K))
    u_pick = uniform_f64(seed, f"trace.L{layer}.pick", (steps, K))
    out = np.zeros((steps, K), dtype=np.int32)
    prev: list[int] = []
    for t in range(steps):
        cur = [e for j, e in enumerate(prev) if u_keep[t, j] < keep_p]
        w = pop.copy()
        w[prev] = 0.0  # fill from experts not used at the previous step
        w[cur] = 0.0
        j = 0
        while len(cur) < K:
            c = np.cumsum(w)
            e = int(np.searchsorted(c, u_pick[t, j] * c[-1], side="right"))
            e = min(e, E - 1)
            while w[e] == 0.0:  # numerical edge: step to the next available expert
                e = (e + 1) % E
            cur.append(e)
            w[e] = 0.0
            j = (j + 1) % K
        out[t] = np.array(cur[:K], dtype=np.int32)
        prev = list(out[t])
    return out


# --------------------------------------------------------------------------------------
# Workload shapes and tensor names (shared definition of the inputs; no arithmetic)
# --------------------------------------------------------------------------------------

from dataclasses import dataclass  # noqa: E402

W_SIGMA = 0.02      # every weight tensor: N(0, 0.02)
H_SIGMA = 1.0       # hidden states, residual increments and supplied logits: N(0, 1)


@dataclass(frozen=True)
class LayerShape:
    d: int          # hidden width
    E: int          # routed experts
    F: int          # expert SwiGLU width
    K: int          # experts per token
    H: int          # prerouter head hidden width (0 = no MLP, linear residual only)
    r: int          # LoRA rank (0 = no LoRA)
    alpha: float    # LoRA alpha
    shared: bool    # one shared expert of width F
    lora_out: int = 0   # LoRA linear output width (0 -> d)

    @property
    def lora_rows(self) -> int:
        return self.lora_out or self.d


# Tiny single layer (correctness): d=256, E=16, F=128, K=4, head 64, LoRA r=4 alpha=8.
TINY = LayerShape(d=256, E=16, F=128, K=4, H=64, r=4, alpha=8.0, shared=False)
# 35B-A3B-class layer: d=2048, E=256, F=512, head 1024, shared F=512, LoRA r=16 alpha=32.
def LAYER35B(K: int = 4) -> LayerShape:
    return LayerShape(d=2048, E=256, F=512, K=K, H=1024, r=16, alpha=32.0, shared=True)


STACK_LAYERS = 40
HEAD_OWNERS = range(6, 39)        # heads on layers 6..38 (33 heads)
PREROUTED = range(7, 39)          # layers 7..38 route from the previous layer's head


def t_expert(layer: int, e: int, which: str) -> str:
    return f"L{layer}.E{e}.{which}"          # which: gate [F][d], up [F][d], down [d][F]


def t_shared(layer: int, which: str) -> str:
    return f"L{layer}.S.{which}"


def t_lora(layer: int, which: str) -> str:
    return f"L{layer}.lora.{which}"          # W [out][d] fp32->int4, A [r][d], B [out][r]


def t_head(layer: int, which: str) -> str:
    return f"L{layer}.head.{which}"          # W1 [H][d+2E], b1 [H], W2 [E][H], b2 [E], Lres [E][d]


def t_router(layer: int) -> str:
    return f"L{layer}.router"                # R [E][d]


def t_hidden(step: int) -> str:
    return f"hidden.s{step}"


def t_increment(step: int, layer: int) -> str:
    return f"incr.s{step}.L{layer}"


def t_logits(which: str) -> str:
    return f"logits.{which}"
