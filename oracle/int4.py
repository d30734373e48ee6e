"""int4 affine group-64 quantisation for the oracle (test infrastructure only).

Source: "The Other Half of the Memory Wall", §3.1 "Problem" (experts stored int4) and
"Executor paths" (every projection carries its weights with their scales and biases);
§2 "Quantization" (int4 affine group-64).  The pages name the format but not its
rounding rules; the reading used here (also the CUDA packer's contract):

* a group is 64 consecutive weights along the input (column) dimension of W[out][in];
* lo = min, hi = max of the group in fp32;
* scale s = bf16_rne((hi - lo) / 15) and bias b = bf16_rne(lo), both rounded to
  bf16 *before* the codes are chosen;
* code q = clamp(rint_half_even((w - b) / s), 0, 15) in fp32 IEEE arithmetic,
  and q = 0 for every weight of a group whose s is 0;
* dequantised weight = s * q + b.

Byte layout ("row" layout): q is uint32 [rows][cols/8], element j of a row lives in
word j // 8 at bits 4*(j % 8) .. 4*(j % 8)+3; scale and bias are bf16 [rows][cols/64].

"column-slab" layout (same codes, different byte order; used for projections that
are consumed 32 input columns at a time): q is uint32 [cols/32][rows][4], holding
words 4c .. 4c+3 of every row in slab c; scale and bias are bf16 [cols/64][rows].
"""
import numpy as np

from .bf16 import to_bf16, bf16_to_f32, bf16_to_f64

GROUP = 64


def quantize_groups(w: np.ndarray):
    """fp32 W[rows][cols] -> (codes uint8 [rows][cols], scale bf16 [rows][g], bias bf16 [rows][g])."""
    w = np.asarray(w, dtype=np.float32)
    rows, cols = w.shape
    assert cols % GROUP == 0
    g = w.reshape(rows, cols // GROUP, GROUP)
    lo = g.min(axis=2)
    hi = g.max(axis=2)
    s32 = (hi - lo) / np.float32(15.0)          # fp32 subtract and divide
    s = to_bf16(s32)
    b = to_bf16(lo)
    sf = bf16_to_f32(s)[:, :, None]
    bf = bf16_to_f32(b)[:, :, None]
    zero = sf == 0
    safe = np.where(zero, np.float32(1.0), sf).astype(np.float32)
    t = (g - bf) / safe                          # fp32 subtract and divide
    q = np.clip(np.rint(t), 0, 15)
    q = np.where(zero, 0, q).astype(np.uint8)
    return q.reshape(rows, cols), s, b


def pack_codes(codes: np.ndarray) -> np.ndarray:
    """uint8 codes [rows][cols] -> uint32 words [rows][cols/8], element j at bits 4*(j%8)."""
    rows, cols = codes.shape
    c = codes.astype(np.uint32).reshape(rows, cols // 8, 8)
    words = np.zeros((rows, cols // 8), dtype=np.uint32)
    for j in range(8):
        words |= c[:, :, j] << np.uint32(4 * j)
    return words


def unpack_codes(words: np.ndarray) -> np.ndarray:
    """uint32 words [rows][cols/8] -> uint8 codes [rows][cols]."""
    rows, nw = words.shape
    out = np.zeros((rows, nw, 8), dtype=np.uint8)
    for j in range(8):
        out[:, :, j] = ((words >> np.uint32(4 * j)) & np.uint32(0xF)).astype(np.uint8)
    return out.reshape(rows, nw * 8)


def pack(w: np.ndarray):
    """fp32 W[rows][cols] -> (q uint32 [rows][cols/8], scale uint16 [rows][cols/64], bias uint16)."""
    codes, s, b = quantize_groups(w)
    return pack_codes(codes), s, b


def to_column_slab(q: np.ndarray, s: np.ndarray, b: np.ndarray):
    """Row layout -> column-slab layout (a pure re-ordering of the same bytes)."""
    rows, nw = q.shape
    slabs = nw // 4
    q_cs = np.empty((slabs, rows, 4), dtype=np.uint32)
    for c in range(slabs):
        q_cs[c] = q[:, 4 * c: 4 * c + 4]
    return q_cs, np.ascontiguousarray(s.T), np.ascontiguousarray(b.T)


def dequantize(q: np.ndarray, s: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Row layout -> float64 W_hat[rows][cols] = s * q + b (exact in fp64)."""
    codes = unpack_codes(q).astype(np.float64)
    rows, cols = codes.shape
    sf = np.repeat(bf16_to_f64(s), GROUP, axis=1)
    bf = np.repeat(bf16_to_f64(b), GROUP, axis=1)
    assert sf.shape == (rows, cols)
    return sf * codes + bf


def quantize_dequantize(w: np.ndarray) -> np.ndarray:
    return dequantize(*pack(w))
