"""Elementary operations of the decode step, float64 unless stated.

Test infrastructure (see the package docstring).  Parity pins for every
function live in tests/test_oracle_pins.py.
"""
from __future__ import annotations

import numpy as np


# --------------------------------------------------------------------------
# Number formats
# --------------------------------------------------------------------------

def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns -> float32 (exact: bf16 is the top half of fp32)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns -> float64 (exact)."""
    return bf16_bits_to_f32(bits).astype(np.float64)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 (ties to even), as float64.

    Written from the format: keep the sign, 8 exponent bits and 7 fraction
    bits.  x is first rounded to float32 (ties to even), whose spacing is a
    divisor of bf16's, then the low 16 bits of the float32 are rounded away
    with ties to even.  Finite inputs only.
    """
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return bf16_bits_to_f64(u.astype(np.uint16))


def _e4m3_value(code: int) -> float:
    """Value of one float8_e4m3fn code (OCP 8-bit floating point, E4M3).

    Bit 7 sign, bits 6..3 exponent with bias 7, bits 2..0 mantissa.  Exponent
    field 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN; there are no
    infinities, so the largest finite magnitude is 1.75 * 2^8 = 448.
    """
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** (1 - 7)
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


E4M3_TABLE = np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """float8_e4m3fn codes (uint8) -> float64 values."""
    return E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


# Non-negative finite codes 0..126 have strictly increasing values.
_POS_VALUES = E4M3_TABLE[:127]


def e4m3_encode_rne(x: np.ndarray) -> np.ndarray:
    """float -> float8_e4m3fn code, round to nearest, ties to even code.

    Inputs must be finite with |x| <= 448 (the quantiser clamps first).
    Nearest of the two neighbouring representable values wins; on an exact
    tie the code with a zero mantissa LSB (the even code) wins.  -0.0 keeps
    its sign bit.
    """
    x = np.asarray(x, dtype=np.float64)
    if np.any(~np.isfinite(x)) or np.any(np.abs(x) > 448.0):
        raise ValueError("e4m3_encode_rne: input outside [-448, 448]")
    a = np.abs(x)
    hi = np.searchsorted(_POS_VALUES, a, side="left")      # first value >= a
    hi = np.minimum(hi, 126)
    lo = np.maximum(hi - 1, 0)
    v_hi = _POS_VALUES[hi]
    v_lo = _POS_VALUES[lo]
    d_hi = v_hi - a
    d_lo = a - v_lo
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(a == v_hi, hi, np.where(pick_hi, hi, lo)).astype(np.uint8)
    sign = np.signbit(x)
    return (code | np.where(sign, 0x80, 0).astype(np.uint8)).astype(np.uint8)


def fp8_quantize_rows(w_bits: np.ndarray):
    """Per-row symmetric FP8 quantisation of one [out][in] bf16 weight.

    drbaph s2-pro-fp8 model card, "Quantization Details": every output row
    gets its own float32 scale, weights become float8_e4m3fn.  Reading of the
    scale (the card's formula did not survive extraction): scale = amax/448
    with amax = max |w| over the row, in float32 (IEEE division); a zero row
    gets scale 1.  q = e4m3_RNE(clamp(w / scale, -448, 448)) with w / scale a
    float32 division.  Returns (codes uint8 [out][in], scale float32 [out]).
    """
    w = bf16_bits_to_f32(w_bits)
    amax = np.max(np.abs(w), axis=1).astype(np.float32)
    scale = (amax / np.float32(448.0)).astype(np.float32)
    scale = np.where(amax == 0, np.float32(1.0), scale).astype(np.float32)
    ratio = (w / scale[:, None]).astype(np.float32)
    ratio = np.clip(ratio, np.float32(-448.0), np.float32(448.0))
    return e4m3_encode_rne(ratio), scale


def fp8_dequant_rows(codes: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """Dequantised weight = float32(scale[row] * e4m3 value), as float64.

    The product of a float32 and an e4m3 value rounded once to float32, the
    way a dequantise-to-float module computes it.
    """
    v = e4m3_decode(codes).astype(np.float32)
    return (np.asarray(scale, np.float32)[:, None] * v).astype(np.float32).astype(np.float64)


def _e2m1_value(code: int) -> float:
    """Value of one FP4 E2M1 code (OCP Microscaling formats, FP4 E2M1).

    Bit 3 sign, bits 2..1 exponent with bias 1, bit 0 mantissa.  Exponent
    field 0 is subnormal (m/2 * 2^0); there are no infinities or NaNs, so the
    magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4, 6.
    """
    s = -1.0 if code & 0x8 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        return s * (m / 2.0)
    return s * (1.0 + m / 2.0) * 2.0 ** (e - 1)


E2M1_TABLE = np.array([_e2m1_value(c) for c in range(16)], dtype=np.float64)
_E2M1_POS = E2M1_TABLE[:8]


def e2m1_decode(codes: np.ndarray) -> np.ndarray:
    """FP4 E2M1 codes (0..15) -> float64 values."""
    return E2M1_TABLE[np.asarray(codes, dtype=np.uint8) & 0xF]


def e2m1_encode_rne(x: np.ndarray) -> np.ndarray:
    """float -> FP4 E2M1 code, round to nearest, ties to the even code
    (mantissa bit 0); inputs finite with |x| <= 6 (the quantiser clamps)."""
    x = np.asarray(x, dtype=np.float64)
    if np.any(~np.isfinite(x)) or np.any(np.abs(x) > 6.0):
        raise ValueError("e2m1_encode_rne: input outside [-6, 6]")
    a = np.abs(x)
    hi = np.minimum(np.searchsorted(_E2M1_POS, a, side="left"), 7)
    lo = np.maximum(hi - 1, 0)
    d_hi = _E2M1_POS[hi] - a
    d_lo = a - _E2M1_POS[lo]
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(a == _E2M1_POS[hi], hi, np.where(pick_hi, hi, lo)).astype(np.uint8)
    return (code | np.where(np.signbit(x), 0x8, 0).astype(np.uint8)).astype(np.uint8)


def nvfp4_quantize_rows(w_bits: np.ndarray):
    """Block-scaled 4-bit quantisation of one [out][in] bf16 weight.

    The tuna-fish README lists nvfp4 among its weight formats (intro list,
    "Support int8/fp8/int4/nvfp4 quantization"; memory table) without the
    details.  Reading, after NVIDIA's NVFP4 layout: FP4 E2M1 elements, one
    E4M3 scale per 16 consecutive elements of a row, and a float32 scale per
    output row (where NVFP4 keeps one per tensor; per row follows the fp8
    model card).  All in float32, in this order:
      s_row = amax(row) / (6 * 448)            (1 for an all-zero row)
      s_b   = e4m3_RNE(min(amax(block) / f32(6 * s_row), 448))
      code  = e2m1_RNE(clamp(w / f32(value(s_b) * s_row), -6, 6))   (0 if s_b = 0)
    Returns (codes uint8 [out][in/16][16] (one code per byte), block scales
    uint8 [out][in/16], row scales float32 [out]).
    """
    w = bf16_bits_to_f32(w_bits)
    rows, cols = w.shape
    blocks = w.reshape(rows, cols // 16, 16)
    F = np.float32
    amax = np.max(np.abs(w), axis=1).astype(F)
    s_row = np.where(amax == 0, F(1.0), (amax / F(6.0 * 448.0)).astype(F)).astype(F)
    denom = (F(6.0) * s_row).astype(F)
    bs = (np.max(np.abs(blocks), axis=2).astype(F) / denom[:, None]).astype(F)
    bs = np.minimum(bs, F(448.0))
    sb = e4m3_encode_rne(bs)
    d = (e4m3_decode(sb).astype(F) * s_row[:, None]).astype(F)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = (blocks / d[:, :, None]).astype(F)
    q = np.where(d[:, :, None] == 0, F(0.0), q)
    q = np.clip(q, F(-6.0), F(6.0))
    return e2m1_encode_rne(q), sb, s_row


def nvfp4_dequant_rows(codes: np.ndarray, sb: np.ndarray, s_row: np.ndarray) -> np.ndarray:
    """Dequantised weight = float32(e2m1 * e4m3(s_b) * s_row) as float64 [out][in]
    (e2m1 * e4m3 is exact, so the one rounding is the row scale's)."""
    v = e2m1_decode(codes) * e4m3_decode(sb)[:, :, None]
    out = (v.astype(np.float32) * np.asarray(s_row, np.float32)[:, None, None]).astype(np.float32)
    return out.reshape(codes.shape[0], -1).astype(np.float64)


# --------------------------------------------------------------------------
# Transformer pieces
# --------------------------------------------------------------------------

def linear(w: np.ndarray, x: np.ndarray) -> np.ndarray:
    """nn.Linear without bias: weight [out][in], y[..., o] = sum_i w[o, i] x[..., i]."""
    return x @ w.T


def rmsnorm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm: x / sqrt(mean(x^2) + eps) * w over the last axis.

    Reading: the pages name only "layer norms"; the Llama-style pre-norm
    RMSNorm with weight w (not 1 + w) is taken, eps 1e-6.
    """
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * w


def rope_angles(pos: int, head_dim: int, theta: float) -> np.ndarray:
    """Rotation angles pos * theta^(-2i/D), i = 0 .. D/2-1, in float64."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    inv_freq = theta ** (-2.0 * i / head_dim)
    return pos * inv_freq


def apply_rope(v: np.ndarray, pos: int, theta: float) -> np.ndarray:
    """Rotary position embedding of head vectors v[..., D] at position pos.

    The "Fish Speech" tour lists rotary embeddings in the decoder.  Reading:
    half-split pairs (i, i + D/2) rotated by angle pos * theta^(-2i/D):
      v'[i]       = v[i] cos - v[i + D/2] sin
      v'[i + D/2] = v[i + D/2] cos + v[i] sin
    """
    D = v.shape[-1]
    a = rope_angles(pos, D, theta)
    c, s = np.cos(a), np.sin(a)
    x1 = v[..., : D // 2]
    x2 = v[..., D // 2:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def attention_row(q: np.ndarray, K: np.ndarray, V: np.ndarray, n_valid: int) -> np.ndarray:
    """Grouped-query attention of one query row over cached keys 0..n_valid-1.

    q [Hq][D]; K, V [Hkv][T][D] (positions beyond n_valid are ignored).
    Query head h reads kv head h // (Hq / Hkv); scores scaled by 1/sqrt(D);
    softmax with max subtraction.  Returns o [Hq][D].
    """
    Hq, D = q.shape
    Hkv = K.shape[0]
    group = Hq // Hkv
    out = np.empty((Hq, D), dtype=np.float64)
    for h in range(Hq):
        g = h // group
        s = K[g, :n_valid] @ q[h] / np.sqrt(D)
        p = np.exp(s - np.max(s))
        out[h] = (p / np.sum(p)) @ V[g, :n_valid]
    return out


def causal_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, positions) -> np.ndarray:
    """attention_row for a block of query rows at once (the prompt pass).

    q [R][Hq][D], row r at position positions[r]; K, V [Hkv][T][D].  Row r
    attends to keys 0..positions[r], exactly as attention_row(q[r], K, V,
    positions[r] + 1): the same scores, scale, max subtraction and grouping,
    with the keys a row may not see masked out of its softmax.  Returns
    o [R][Hq][D].
    """
    R, Hq, D = q.shape
    Hkv = K.shape[0]
    group = Hq // Hkv
    pos = np.asarray(positions, dtype=np.int64)
    n = int(pos.max()) + 1
    visible = np.arange(n)[None, :] <= pos[:, None]          # [R][n]
    out = np.empty((R, Hq, D), dtype=np.float64)
    for h in range(Hq):
        g = h // group
        s = q[:, h, :] @ K[g, :n].T / np.sqrt(D)             # [R][n]
        s = np.where(visible, s, -np.inf)
        p = np.exp(s - np.max(s, axis=1, keepdims=True))
        out[:, h, :] = (p / np.sum(p, axis=1, keepdims=True)) @ V[g, :n]
    return out


def silu(z: np.ndarray) -> np.ndarray:
    """SiLU: z / (1 + exp(-z)) (the gate of the SwiGLU MLP)."""
    return z / (1.0 + np.exp(-z))
