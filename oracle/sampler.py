"""Codebook-id selection: greedy argmax and seeded top-k sampling.

Test infrastructure (see the package docstring).

The "Fish Speech" tour ("Why You Need This") names top-k sampling in the
generation loop; the long-context workload samples with top-k = 30 from a
seeded Philox stream.  The pages give no formula, so the selection rule below
is this project's reading, written so that a GPU and a CPU can reach the same
index bit for bit:

  * selection runs on float32 logits;
  * candidates are ordered by (logit descending, index ascending) and the
    first k are kept;
  * weights p_i = exp32(d_i) with d_i = (z_i - z_max) / temperature in float32,
    where exp32 is the routine below (no fused multiply-add anywhere);
  * S = sum of p_i in candidate order, c_i the running sums, all float32;
  * u = (w0 >> 8) * 2^-24 with w0 the first word of
    Philox4x32-10(counter = (frame, codebook, sequence, 0), key = seed);
  * the pick is the first candidate with u * S < c_i, else the last one;
  * optional nucleus (top_p) and repetition window: see topk_sample and
    apply_repetition_penalty.
"""
from __future__ import annotations

import numpy as np

F32 = np.float32

# --------------------------------------------------------------------------
# Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy
# as 1, 2, 3", SC'11): 10 rounds of a multiply-xor bijection keyed by a Weyl
# sequence.
# --------------------------------------------------------------------------
_PHILOX_M0 = 0xD2511F53
_PHILOX_M1 = 0xCD9E8D57
_PHILOX_W0 = 0x9E3779B9   # golden ratio
_PHILOX_W1 = 0xBB67AE85   # sqrt(3) - 1
_MASK32 = 0xFFFFFFFF


def philox4x32_10(counter, key):
    """Philox4x32 with 10 rounds.  counter: 4 uint32, key: 2 uint32."""
    c0, c1, c2, c3 = (int(v) & _MASK32 for v in counter)
    k0, k1 = (int(v) & _MASK32 for v in key)
    for rnd in range(10):
        if rnd:
            k0 = (k0 + _PHILOX_W0) & _MASK32
            k1 = (k1 + _PHILOX_W1) & _MASK32
        p0 = _PHILOX_M0 * c0
        p1 = _PHILOX_M1 * c2
        hi0, lo0 = p0 >> 32, p0 & _MASK32
        hi1, lo1 = p1 >> 32, p1 & _MASK32
        c0, c1, c2, c3 = (hi1 ^ c1 ^ k0), lo1, (hi0 ^ c3 ^ k1), lo0
    return (c0, c1, c2, c3)


def uniform24(word: int) -> np.float32:
    """Top 24 bits of a 32-bit word as a float32 in [0, 1): (w >> 8) * 2^-24."""
    return F32((int(word) & _MASK32) >> 8) * F32(2.0 ** -24)


# --------------------------------------------------------------------------
# exp32: exp for float32 arguments, written out so that any IEEE float32
# machine evaluates it bit for bit the same way (each step a single rounded
# float32 multiply or add; no fused multiply-add).
#   1. x < -80 returns 0 (every result kept is a normal float32).
#   2. Cody-Waite reduction: n = rint(x * log2(e)), r = (x - n*ln2_hi) - n*ln2_lo
#      with ln2_hi = ln 2 cut to its leading 12 significand bits (n * ln2_hi
#      is exact for |n| < 2^12) and ln2_lo = float32(ln 2 - ln2_hi).
#   3. p = Taylor polynomial of degree 7 in Horner form, coefficients
#      float32(1/k!) (|r| <= ln2/2 keeps the truncation error below 1e-8).
#   4. result = p * 2^n, an exact power-of-two scaling.
# --------------------------------------------------------------------------
LOG2E_F32 = F32(1.4426950408889634)
LN2_HI_F32 = F32(0.693145751953125)          # 0x3F317200
LN2_LO_F32 = F32(0.6931471805599453 - 0.693145751953125)
_EXP_COEF = [F32(1.0 / float(np.prod(np.arange(1, k + 1)))) for k in range(8)]


def exp_f32(x) -> np.float32:
    x = F32(x)
    if x < F32(-80.0):
        return F32(0.0)
    n = np.rint(F32(x * LOG2E_F32))                 # ties to even
    r = F32(x - F32(n * LN2_HI_F32))
    r = F32(r - F32(n * LN2_LO_F32))
    p = _EXP_COEF[7]
    for k in range(6, -1, -1):
        p = F32(F32(p * r) + _EXP_COEF[k])
    return F32(np.ldexp(p, int(n)))


# --------------------------------------------------------------------------
# Selection
# --------------------------------------------------------------------------

def argmax_lowest(z) -> int:
    """Greedy pick: index of the largest logit, lowest index on ties.

    NaN logits are an error.
    """
    z = np.asarray(z)
    if np.any(np.isnan(z)):
        raise ValueError("NaN logit")
    m = np.max(z)
    return int(np.flatnonzero(z == m)[0])


def topk_candidates(z32: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest float32 logits, ordered by (logit desc, index asc)."""
    z32 = np.asarray(z32, dtype=np.float32)
    order = np.lexsort((np.arange(z32.size), -z32.astype(np.float64)))
    return order[: min(k, z32.size)]


def apply_repetition_penalty(z32: np.ndarray, recent, penalty: float) -> np.ndarray:
    """Repetition window ("Fish Speech" tour, "Why You Need This": the
    generation loop has repetition windows; the pages give no formula).

    Reading: every id in `recent` (the ids this codebook fed back in the
    previous W frames of the sequence; each id counts once) has its float32
    logit divided by `penalty` when it is positive and multiplied by it
    otherwise (the CTRL-style penalty), one IEEE float32 operation each.
    penalty 1 leaves the logits unchanged.  Returns a new float32 array.
    """
    z = np.array(z32, dtype=np.float32, copy=True)
    r = F32(penalty)
    for i in sorted(set(int(v) for v in recent if 0 <= int(v) < z.size)):
        z[i] = F32(z[i] / r) if z[i] > F32(0.0) else F32(z[i] * r)
    return z


def topk_sample(z32: np.ndarray, k: int, seed: int, frame: int, codebook: int,
                sequence: int = 0, temperature: float = 1.0, top_p: float = 1.0):
    """Seeded top-k draw from float32 logits (rule in the module docstring),
    optionally restricted to a nucleus ("Fish Speech" tour: top-p sampling).

    Nucleus reading: with top_p < 1, keep the shortest prefix of the ordered
    candidates whose running weight sum c_i reaches top_p * S (float32
    product), i.e. up to the first i with c_i >= top_p * S, and draw within it
    with S' = c_i in place of S.  top_p >= 1 keeps every candidate.

    Returns (index, details) where details holds the candidate list, the
    float32 weights, cumulative sums, S, the kept count n and its sum S', u
    and t, for robustness checks.
    """
    z32 = np.asarray(z32, dtype=np.float32)
    if np.any(np.isnan(z32)):
        raise ValueError("NaN logit")
    cand = topk_candidates(z32, k)
    zmax = z32[cand[0]]
    temp = F32(temperature)
    p = []
    for i in cand:
        d = F32(z32[i] - zmax)
        if temp != F32(1.0):
            d = F32(d / temp)
        p.append(exp_f32(d))
    c = []
    acc = F32(0.0)
    for v in p:
        acc = F32(acc + v)
        c.append(acc)
    S = acc
    n = len(cand)
    if F32(top_p) < F32(1.0):
        tp = F32(F32(top_p) * S)
        for i, ci in enumerate(c):
            if ci >= tp:
                n = i + 1
                break
    Sk = c[n - 1]
    key = (seed & _MASK32, (seed >> 32) & _MASK32)
    w0 = philox4x32_10((frame, codebook, sequence, 0), key)[0]
    u = uniform24(w0)
    t = F32(u * Sk)
    pick = n - 1
    for j in range(n):
        if t < c[j]:
            pick = j
            break
    return int(cand[pick]), dict(cand=cand, p=np.array(p, np.float32),
                                 c=np.array(c, np.float32), S=S, n=n, Sk=Sk, u=u, t=t,
                                 pick=pick)
