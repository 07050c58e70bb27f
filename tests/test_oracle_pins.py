"""Pins of the CPU oracle against things other than itself.

Each test checks one oracle function against a library routine, a closed
form, an invariant, brute force on tiny inputs, a published known-answer
vector, or numbers the source pages print.  A dropped term, a wrong sign, a
wrong index or a transposed operand in the oracle fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import model as om
from synth import TINY, FULL, make_weights, make_prompt, make_logits, f32_to_bf16_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------- formats

def test_bf16_decode_matches_torch():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 1 << 16, size=100000, dtype=np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]            # finite only
    t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert np.array_equal(oracle.bf16_bits_to_f32(bits), t)


def test_round_to_bf16_matches_torch_cast():
    rng = np.random.default_rng(12)
    x = np.concatenate([rng.standard_normal(200000) * 10.0 ** rng.integers(-6, 6, 200000),
                        [0.0, -0.0, 1.0, 1.00390625, 1.01171875, 3.0e38]])
    ref = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    assert np.array_equal(oracle.round_to_bf16(x), ref)


def test_bf16_rounding_of_inputs_matches_torch():
    x = np.random.default_rng(2).standard_normal(100000).astype(np.float32) * 0.02
    ours = f32_to_bf16_bits(x)
    theirs = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, theirs)


def test_e4m3_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    ours = oracle.e4m3_decode(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert set(np.flatnonzero(nan)) == {0x7F, 0xFF}
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.nanmax(ours) == 448.0 and ours[0x7E] == 448.0
    assert ours[0x01] == 2.0 ** -9          # smallest subnormal
    assert ours[0x08] == 2.0 ** -6          # smallest normal


def test_e4m3_bit_placement_identity():
    """An e4m3 code s.eeee.mmm placed as float32 bits (s << 31) | (eeeemmm << 20)
    is the code's value times 2^-120 exactly, subnormal codes included (both
    formats put the hidden bit in the same place once the exponent bias
    difference, 127 - 7 = 120, is taken out)."""
    codes = np.arange(256, dtype=np.uint32)
    bits = ((codes & 0x80) << 24) | ((codes & 0x7F) << 20)
    placed = bits.astype(np.uint32).view(np.float32).astype(np.float64) * 2.0 ** 120
    ref = oracle.e4m3_decode(codes.astype(np.uint8))
    ok = ~np.isnan(ref)
    assert np.array_equal(placed[ok], ref[ok])
    assert np.all(np.isfinite(placed))       # the NaN codes become finite: decode must mask them


def test_e4m3_encode_matches_torch_cast_including_ties():
    vals = oracle.e4m3_decode(np.arange(127, dtype=np.uint8))
    mids = (vals[1:] + vals[:-1]) / 2                     # exact ties
    rng = np.random.default_rng(3)
    rnd = rng.uniform(-448, 448, 200000)
    small = rng.standard_normal(50000) * 0.01
    x = np.concatenate([vals, -vals, mids, -mids, rnd, small]).astype(np.float32)
    ours = oracle.e4m3_encode_rne(x)
    theirs = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, theirs)


def test_fp8_row_quantiser_bounds_and_definition():
    rng = np.random.default_rng(4)
    w = f32_to_bf16_bits(rng.standard_normal((64, 300)).astype(np.float32) * 0.02)
    w[5] = 0                                           # an all-zero row
    codes, scale = oracle.fp8_quantize_rows(w)
    wf = oracle.bf16_bits_to_f32(w).astype(np.float64)
    assert scale.dtype == np.float32 and scale[5] == 1.0 and not codes[5].any()
    amax = np.max(np.abs(wf), axis=1)
    nz = amax > 0
    # scale is the float32 quotient amax / 448
    assert np.array_equal(scale[nz], (amax[nz].astype(np.float32) / np.float32(448)))
    # the largest magnitude of each row lands on +-448
    v = oracle.e4m3_decode(codes)
    assert np.all(np.max(np.abs(v[nz]), axis=1) == 448.0)
    # half a unit in the last place: 2^-4 relative for normals, 2^-10 * scale below
    deq = oracle.fp8_dequant_rows(codes, scale)
    bound = np.maximum(np.abs(wf) * 2.0 ** -4, scale[:, None].astype(np.float64) * 2.0 ** -10)
    assert np.all(np.abs(deq - wf) <= bound * (1 + 1e-6) + 1e-30)
    # dequant is the float32 product scale * value
    assert np.array_equal(deq, (scale[:, None] * v.astype(np.float32)).astype(np.float32).astype(np.float64))


# ----------------------------------------------------------------- pieces

def test_e2m1_codes_equal_their_e4m3_rebiasing_under_torch():
    """FP4 E2M1 (bias 1) and FP8 E4M3 (bias 7) share the IEEE layout, so a
    normal e2m1 code (s, e, m) is the e4m3 code (s, e + 6, m << 2) and the
    subnormal 0.5 is 2^-1 = e4m3 (s, 6, 0); torch's float8_e4m3fn decodes
    those e4m3 codes, pinning every e2m1 value."""
    for c in range(16):
        s_, e, m = c >> 3, (c >> 1) & 3, c & 1
        if e == 0:
            e8 = (s_ << 7) | ((6 << 3) if m else 0)
        else:
            e8 = (s_ << 7) | ((e + 6) << 3) | (m << 2)
        want = torch.tensor([e8], dtype=torch.uint8).view(torch.float8_e4m3fn).float().item()
        assert oracle.e2m1_decode(np.array([c]))[0] == want, c


def test_e2m1_encode_round_trip_and_ties():
    codes = np.arange(16, dtype=np.uint8)
    vals = oracle.e2m1_decode(codes)
    back = oracle.e2m1_encode_rne(vals)
    assert np.array_equal(oracle.e2m1_decode(back), vals)          # -0 and +0 alike
    # midpoints go to the neighbour with an even code (mantissa bit 0)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    assert oracle.e2m1_decode(oracle.e2m1_encode_rne(mids)).tolist() == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]
    assert oracle.e2m1_decode(oracle.e2m1_encode_rne(-mids)).tolist() == [-0.0, -1.0, -1.0, -2.0, -2.0,
                                                                        -4.0, -4.0]
    # off the midpoints: the nearest value
    x = np.linspace(-6, 6, 2001)
    got = oracle.e2m1_decode(oracle.e2m1_encode_rne(x))
    dist = np.abs(oracle.e2m1_decode(np.arange(16))[None, :] - x[:, None]).min(axis=1)
    assert np.allclose(np.abs(got - x), dist)


def test_nvfp4_quantiser_bounds_and_structure():
    rng = np.random.default_rng(4)
    w = f32_to_bf16_bits(rng.standard_normal((24, 256)).astype(np.float32) * 0.02)
    w[0] = 0                                            # all-zero row
    w[1, :16] = 0                                       # all-zero block
    w[2, 5] = f32_to_bf16_bits(np.array([3.0], np.float32))[0]   # an outlier
    codes, sb, sr = oracle.nvfp4_quantize_rows(w)
    wf = oracle.bf16_bits_to_f64(w)
    deq = oracle.nvfp4_dequant_rows(codes, sb, sr)
    assert sr[0] == 1.0 and not codes[0].any() and not sb[0].any()
    assert not sb[1, 0] and not codes[1, 0].any()
    # the row scale maps the row maximum to 6 * 448
    amax = np.abs(oracle.bf16_bits_to_f32(w[2:])).max(axis=1)
    assert np.array_equal(sr[2:], (amax / np.float32(2688.0)).astype(np.float32))
    # every element within one e2m1 step of its block (value(s_b) * s_row)
    step = oracle.e4m3_decode(sb) * sr[:, None].astype(np.float64)
    err = np.abs(deq - wf).reshape(24, 16, 16)
    assert np.all(err <= step[:, :, None] * (1 + 1e-6) + 1e-30)
    # a normal block scale puts the block's largest element at +-6
    mags = (codes & 7).reshape(24, 16, 16)
    bmax = np.abs(wf.reshape(24, 16, 16)).argmax(axis=2)
    normal = oracle.e4m3_decode(sb) >= 2.0 ** -6
    top = np.take_along_axis(mags, bmax[:, :, None], axis=2)[:, :, 0]
    assert np.all(top[normal] == 7)


def test_linear_matches_torch_nonsquare():
    rng = np.random.default_rng(5)
    w = rng.standard_normal((7, 13))
    x = rng.standard_normal((3, 13))
    ref = F.linear(torch.from_numpy(x), torch.from_numpy(w)).numpy()
    assert np.allclose(oracle.linear(w, x), ref, rtol=1e-13, atol=1e-13)


def test_rmsnorm_closed_form_and_torch():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((5, 256)) * 3.0
    eps = 1e-6
    y = oracle.rmsnorm(x, np.ones(256), eps)
    ms = np.mean(x * x, axis=-1)
    rms_y = np.sqrt(np.mean(y * y, axis=-1))
    assert np.allclose(rms_y, 1.0 / np.sqrt(1.0 + eps / ms), rtol=1e-12)
    w = rng.standard_normal(256)
    ref = F.rms_norm(torch.from_numpy(x), (256,), torch.from_numpy(w), eps).numpy()
    assert np.allclose(oracle.rmsnorm(x, w, eps), ref, rtol=1e-12, atol=1e-12)


def test_rope_closed_forms_and_invariants():
    # D = 2: one pair, inverse frequency 1, rotation by `pos` radians
    for pos in (0, 1, 5):
        v = oracle.apply_rope(np.array([1.0, 0.0]), pos, 1e6)
        assert np.allclose(v, [math.cos(pos), math.sin(pos)], atol=1e-15)
    # D = 4, theta = 100: pairs (0, 2) at rate 1 and (1, 3) at rate 100^-1/2
    v = oracle.apply_rope(np.array([0.0, 1.0, 0.0, 0.0]), 3, 100.0)
    assert np.allclose(v, [0.0, math.cos(0.3), 0.0, math.sin(0.3)], atol=1e-15)
    rng = np.random.default_rng(7)
    q = rng.standard_normal(128)
    k = rng.standard_normal(128)
    assert np.array_equal(oracle.apply_rope(q, 0, 1e6), q)
    for p in (1, 17, 1023):
        assert abs(np.linalg.norm(oracle.apply_rope(q, p, 1e6)) / np.linalg.norm(q) - 1) < 1e-12
    # <R(q, m), R(k, n)> depends on m - n only
    d1 = oracle.apply_rope(q, 40, 1e6) @ oracle.apply_rope(k, 33, 1e6)
    d2 = oracle.apply_rope(q, 907, 1e6) @ oracle.apply_rope(k, 900, 1e6)
    assert abs(d1 - d2) < 1e-9


def _rope_complex(x, pos, theta):
    """Independent restatement of half-split RoPE as a complex multiply."""
    D = x.shape[-1]
    z = torch.complex(x[..., : D // 2], x[..., D // 2:])
    inv = theta ** (-2.0 * torch.arange(D // 2, dtype=torch.float64) / D)
    ang = pos[:, None].to(torch.float64) * inv[None, :]
    rot = torch.polar(torch.ones_like(ang), ang)
    shape = [1] * (x.dim() - 2) + list(rot.shape)
    z = z * rot.view(*shape) if x.dim() == 2 else z * rot[:, None, :]
    return torch.cat([z.real, z.imag], dim=-1)


def test_rope_matches_complex_restatement():
    rng = np.random.default_rng(8)
    x = rng.standard_normal((9, 3, 64))
    pos = torch.arange(9) * 7 + 2
    ref = _rope_complex(torch.from_numpy(x), pos, 1e6).numpy()
    ours = np.stack([oracle.apply_rope(x[i], int(pos[i]), 1e6) for i in range(9)])
    assert np.allclose(ours, ref, rtol=1e-12, atol=1e-12)


def test_attention_brute_force_and_sdpa():
    rng = np.random.default_rng(9)
    Hq, Hkv, T, D = 4, 2, 6, 8
    q = rng.standard_normal((Hq, D))
    K = rng.standard_normal((Hkv, T, D))
    V = rng.standard_normal((Hkv, T, D))
    n = 4
    out = oracle.attention_row(q, K, V, n)
    for h in range(Hq):
        g = h // (Hq // Hkv)
        s = [sum(q[h, d] * K[g, t, d] for d in range(D)) / math.sqrt(D) for t in range(n)]
        e = [math.exp(v) for v in s]
        tot = sum(e)
        ref = [sum(e[t] / tot * V[g, t, d] for t in range(n)) for d in range(D)]
        assert np.allclose(out[h], ref, rtol=1e-12, atol=1e-12)
    # keys beyond n_valid are ignored
    K2, V2 = K.copy(), V.copy()
    K2[:, n:] = 1e3
    V2[:, n:] = -1e3
    assert np.array_equal(oracle.attention_row(q, K2, V2, n), out)
    # torch SDPA with grouped-query heads
    sd = F.scaled_dot_product_attention(
        torch.from_numpy(q)[None, :, None, :], torch.from_numpy(K[:, :n])[None],
        torch.from_numpy(V[:, :n])[None], enable_gqa=True).numpy()[0, :, 0]
    assert np.allclose(out, sd, rtol=1e-12, atol=1e-12)
    # Hkv == Hq reduces to multi-head attention
    Kf = np.repeat(K, 2, axis=0)
    Vf = np.repeat(V, 2, axis=0)
    assert np.allclose(oracle.attention_row(q, Kf, Vf, n), out, rtol=1e-14, atol=1e-14)


def test_causal_attention_block_matches_sdpa_and_rows():
    """The prompt pass's block attention: torch SDPA with an explicit causal
    mask over grouped-query heads, and row by row the single-row routine."""
    rng = np.random.default_rng(21)
    Hq, Hkv, T, D = 8, 2, 12, 16
    pos = [2, 3, 4, 5, 6, 7, 8]
    q = rng.standard_normal((len(pos), Hq, D))
    K = rng.standard_normal((Hkv, T, D))
    V = rng.standard_normal((Hkv, T, D))
    out = oracle.causal_attention(q, K, V, pos)
    n = max(pos) + 1
    mask = torch.from_numpy(np.arange(n)[None, :] <= np.array(pos)[:, None])
    sd = F.scaled_dot_product_attention(
        torch.from_numpy(q).transpose(0, 1)[None], torch.from_numpy(K[:, :n])[None],
        torch.from_numpy(V[:, :n])[None], attn_mask=mask, enable_gqa=True).numpy()[0]
    assert np.allclose(out, sd.transpose(1, 0, 2), rtol=1e-12, atol=1e-12)
    for r, p in enumerate(pos):
        assert np.allclose(out[r], oracle.attention_row(q[r], K, V, p + 1), rtol=1e-13, atol=1e-13)
    # keys past a row's position never matter
    K2, V2 = K.copy(), V.copy()
    K2[:, n:] = 1e3
    V2[:, n:] = -1e3
    assert np.array_equal(oracle.causal_attention(q, K2, V2, pos), out)


def test_silu_matches_torch():
    z = np.linspace(-30, 30, 1001)
    assert np.allclose(oracle.silu(z), F.silu(torch.from_numpy(z)).numpy(), rtol=1e-14, atol=1e-14)


# ----------------------------------------------------------------- sampler

def test_philox_known_answers():
    for v in _golden("philox4x32_10_kat.json")["vectors"]:
        ctr = [int(s, 16) for s in v["ctr"]]
        key = [int(s, 16) for s in v["key"]]
        assert list(oracle.philox4x32_10(ctr, key)) == [int(s, 16) for s in v["out"]]


def test_exp32_within_two_ulp_and_cutoff():
    xs = np.concatenate([np.linspace(-80, 0, 40001), [-0.0, -1e-30, -79.99999]]).astype(np.float32)
    e = np.array([oracle.exp_f32(x) for x in xs], dtype=np.float32)
    ref = np.exp(xs.astype(np.float64))
    ulp = np.abs(e.astype(np.float64) - ref) / np.spacing(np.abs(e))
    assert ulp.max() <= 2.0
    assert oracle.exp_f32(np.float32(0.0)) == 1.0
    assert oracle.exp_f32(np.float32(-80.5)) == 0.0


def test_uniform24_range():
    assert oracle.uniform24(0) == 0.0
    assert oracle.uniform24(0xFFFFFFFF) == np.float32(1 - 2.0 ** -24)
    assert oracle.uniform24(0x80000000) == 0.5


def test_argmax_lowest_index_on_ties():
    z = np.array([1.0, 3.0, -2.0, 3.0, 3.0], np.float32)
    assert oracle.argmax_lowest(z) == 1
    with pytest.raises(ValueError):
        oracle.argmax_lowest(np.array([0.0, np.nan], np.float32))


def test_topk_candidates_order():
    z = np.array([0.5, 2.0, 2.0, -1.0, 2.0, 0.5], np.float32)
    assert list(oracle.topk_candidates(z, 4)) == [1, 2, 4, 0]


def test_topk_one_is_argmax():
    Z = make_logits(50, 256, seed=3, ties=True)
    for i, z in enumerate(Z):
        idx, _ = oracle.topk_sample(z, 1, seed=11, frame=i, codebook=i % 10)
        assert idx == oracle.argmax_lowest(z)


def test_topk_frequencies_follow_truncated_softmax():
    z = make_logits(1, 64, seed=5, scale=1.5)[0]
    k = 8
    cand = oracle.topk_candidates(z, k)
    p = np.exp(z[cand].astype(np.float64) - z[cand[0]])
    p /= p.sum()
    n = 6000
    counts = np.zeros(k)
    pos = {int(c): i for i, c in enumerate(cand)}
    for t in range(n):
        idx, _ = oracle.topk_sample(z, k, seed=1234, frame=t, codebook=3)
        counts[pos[idx]] += 1
    chi2 = np.sum((counts - n * p) ** 2 / (n * p))
    assert chi2 < 30.0          # 7 degrees of freedom: p-value ~ 1e-4


def test_topk_temperature_frequencies_follow_tempered_softmax():
    """At temperature T the draw frequencies over the top-k candidates follow
    softmax(z / T): a slip such as multiplying by T, or dividing before the
    max subtraction in a way that changes the weights, moves them off it."""
    z = make_logits(1, 64, seed=6, scale=1.0)[0]
    k, temp = 6, 0.7
    cand = oracle.topk_candidates(z, k)
    zc = z[cand].astype(np.float64)
    p = np.exp((zc - zc[0]) / temp)
    p /= p.sum()
    # the untempered weights differ enough for the test to tell them apart
    p1 = np.exp(zc - zc[0])
    p1 /= p1.sum()
    n = 6000
    assert np.sum((n * p1 - n * p) ** 2 / (n * p)) > 60.0
    counts = np.zeros(k)
    pos = {int(c): i for i, c in enumerate(cand)}
    for t in range(n):
        idx, det = oracle.topk_sample(z, k, seed=99, frame=t, codebook=5, temperature=temp)
        counts[pos[idx]] += 1
    chi2 = np.sum((counts - n * p) ** 2 / (n * p))
    assert chi2 < 26.0          # 5 degrees of freedom: p-value ~ 1e-4
    # the weights themselves: exp32 of the tempered differences, largest first
    _, det = oracle.topk_sample(z, k, seed=99, frame=0, codebook=5, temperature=temp)
    assert det["p"][0] == 1.0
    assert np.allclose(det["p"], np.exp((zc - zc[0]) / temp), rtol=1e-6)


def test_topp_frequencies_follow_the_renormalised_nucleus():
    """top-p: draws follow softmax over the shortest ordered prefix of the
    top-k candidates whose probability reaches top_p, renormalised."""
    z = make_logits(1, 64, seed=8, scale=1.2)[0]
    k, top_p = 12, 0.6
    cand = oracle.topk_candidates(z, k)
    w = np.exp(z[cand].astype(np.float64) - z[cand[0]])
    cum = np.cumsum(w) / w.sum()
    n = int(np.argmax(cum >= top_p)) + 1          # shortest prefix reaching top_p
    assert 1 < n < k
    p = w[:n] / w[:n].sum()
    N = 6000
    counts = np.zeros(n)
    pos = {int(c): i for i, c in enumerate(cand)}
    for t in range(N):
        idx, det = oracle.topk_sample(z, k, seed=7, frame=t, codebook=2, top_p=top_p)
        assert det["n"] == n
        counts[pos[idx]] += 1                     # never outside the nucleus
    chi2 = np.sum((counts - N * p) ** 2 / (N * p))
    assert chi2 < 10.0 + 3.0 * n                  # ~p = 1e-4 for n - 1 degrees of freedom


def test_topp_limits():
    Z = make_logits(40, 128, seed=9, scale=1.0)
    for t, z in enumerate(Z):
        # a tiny nucleus is the first candidate: the argmax
        idx, _ = oracle.topk_sample(z, 30, seed=3, frame=t, codebook=1, top_p=1e-6)
        assert idx == oracle.argmax_lowest(z)
        # top_p = 1 keeps every candidate: the plain top-k draw
        a, _ = oracle.topk_sample(z, 30, seed=3, frame=t, codebook=1, top_p=1.0)
        b, _ = oracle.topk_sample(z, 30, seed=3, frame=t, codebook=1)
        assert a == b


def test_repetition_penalty_closed_form():
    z = np.array([2.0, -1.5, 0.0, 3.0, -0.25, 1.0], np.float32)
    out = oracle.apply_repetition_penalty(z, [0, 1, 1, 2, 4, 99, -3], 2.0)
    # positive logits divided, the rest multiplied; each id once; others untouched
    assert out.tolist() == [1.0, -3.0, 0.0, 3.0, -0.5, 1.0]
    assert np.array_equal(oracle.apply_repetition_penalty(z, [0, 3, 5], 1.0), z)
    assert np.array_equal(oracle.apply_repetition_penalty(z, [], 5.0), z)
    assert z.tolist() == [2.0, -1.5, 0.0, 3.0, -0.25, 1.0]   # input untouched


def test_repetition_window_blocks_recent_ids_in_the_model():
    """With a huge penalty and greedy selection, no codebook repeats an id it
    fed back within the last W frames (every codebook has a positive logit
    outside the window); without the window the same run does repeat."""
    d = TINY
    w = make_weights(d, seed=12)
    prompt = make_prompt(d, 8, seed=13)
    W = 3

    def run(sampling):
        o = oracle.DualAROracle(d, w)
        fr = [o.prefill(prompt, sampling)[0][0]]
        for _ in range(9):
            fr.append(o.decode_frame(sampling)[0][0])
        return np.array(fr)

    plain = run(None)
    pen = run({"top_k": 0, "rep_window": W, "rep_penalty": 1e6})
    assert any(plain[t, j] in plain[max(0, t - W):t, j] for t in range(1, 10) for j in range(10))
    for t in range(1, 10):
        for j in range(10):
            assert pen[t, j] not in pen[max(0, t - W):t, j], (t, j)
    # the window holds the ids fed back: under teacher forcing, the forced ones
    forced = np.array([[[5] * 10]] * 10, np.int32)            # always feed id 5
    o = oracle.DualAROracle(d, w)
    f0, _ = o.prefill(prompt, {"rep_window": W, "rep_penalty": 1e6}, forced=forced[0])
    for t in range(1, 10):
        f, _ = o.decode_frame({"rep_window": W, "rep_penalty": 1e6}, forced=forced[t])
        assert (f[0] != 5).all()                                # 5 sits in every window


# ----------------------------------------------------------------- load formula

def test_load_formula_page_numbers():
    g = _golden("load_formula.json")
    total = om.load_formula(g["slow_params_wo_emb"], g["fast_params_wo_emb"], g["batch"],
                            g["slow_layers"], g["fast_layers"], g["c_kv"], g["max_length"])
    assert total == g["decode_params_load"]
    assert round(total * 2 / 2 ** 30, 2) == g["bf16_gb_per_step"]
    per_it = total * 2 / 2 ** 30
    for row in g["speedtest_bf16"]:
        assert abs(row["it_s"] * per_it - row["gb_s"]) <= 0.05 * per_it + 0.05
    for row in g["prefill128_decode896"] + g["dingzhen_prefill163"]:
        gib = total * row["bytes_per_elem"] / 2 ** 30
        assert abs(row["decode_tok_s"] * gib - row["gb_s"]) <= 0.05 * gib + 0.05


def test_fidelity_options_reproduce_the_page_counts_through_the_tensor_list():
    """The tensors the options add: with slow q/k norms the slow decoder's
    tensor list (linears, norms, final norm, the 4096-row semantic slice)
    falls short of the tuna-fish slowAR count by one hidden-size vector; the
    fast decoder with a 1024-row head and no q/k norm is the fastAR count."""
    g = _golden("load_formula.json")
    d = FULL.replace(qk_norm=True, codebook_size=1024)
    from synth import tensor_specs
    specs = tensor_specs(d)
    slow = sum(int(np.prod(sh)) for n, sh, _ in specs if n.startswith("slow."))
    assert slow + d.semantic_vocab * d.hidden + d.hidden == g["slow_params_wo_emb"]
    fast = sum(int(np.prod(sh)) for n, sh, _ in specs if n.startswith("fast.") and n != "fast.cb_embed")
    assert fast == g["fast_params_wo_emb"]


def test_layer_shapes_reproduce_page_param_counts():
    g = _golden("load_formula.json")
    # fastAR with a 1024-row head reproduces the inference count exactly,
    # with a codebook-size (4096) head the training-estimation count
    assert om.decoder_params(FULL, 4, 1024) == g["fast_params_wo_emb"]
    assert om.decoder_params(FULL, 4, 4096) == g["training_estimation"]["fast_wo_emb_params"]
    # slowAR: 36 layers + final norm + 4096-row head, plus per-head q/k norms
    # and one more hidden-size vector, is the page's count
    assert om.decoder_params(FULL, 36, 4096, qk_norm=True) + FULL.hidden == g["slow_params_wo_emb"]
    assert len(om.linear_names(FULL)) == 201


# ----------------------------------------------------------------- whole model

def _torch_decoder(prefix, x, W, d):
    """Full-sequence causal restatement of one decoder with torch library ops."""
    S = x.shape[0]
    pos = torch.arange(S)
    a = F.rms_norm(x, (d.hidden,), W[f"{prefix}.attn_norm"], d.rms_eps)
    qkv = F.linear(a, W[f"{prefix}.wqkv"])
    q = qkv[:, : d.q_dim].view(S, d.n_heads, d.head_dim)
    k = qkv[:, d.q_dim: d.q_dim + d.kv_dim].view(S, d.n_kv_heads, d.head_dim)
    v = qkv[:, d.q_dim + d.kv_dim:].view(S, d.n_kv_heads, d.head_dim)
    if f"{prefix}.q_norm" in W:   # per-head RMSNorm of q and k before RoPE
        q = F.rms_norm(q, (d.head_dim,), W[f"{prefix}.q_norm"], d.rms_eps)
        k = F.rms_norm(k, (d.head_dim,), W[f"{prefix}.k_norm"], d.rms_eps)
    q = _rope_complex(q, pos, d.rope_theta)
    # the static KV cache holds bfloat16 values
    k = _rope_complex(k, pos, d.rope_theta).to(torch.bfloat16).double()
    v = v.to(torch.bfloat16).double()
    o = F.scaled_dot_product_attention(q.transpose(0, 1)[None], k.transpose(0, 1)[None],
                                       v.transpose(0, 1)[None], is_causal=True,
                                       enable_gqa=True)[0].transpose(0, 1).reshape(S, -1)
    x = x + F.linear(o, W[f"{prefix}.wo"])
    m = F.rms_norm(x, (d.hidden,), W[f"{prefix}.ffn_norm"], d.rms_eps)
    return x + F.linear(F.silu(F.linear(m, W[f"{prefix}.w1"])) * F.linear(m, W[f"{prefix}.w3"]),
                        W[f"{prefix}.w2"])


def _torch_weights(w):
    return {k: torch.from_numpy(oracle.bf16_bits_to_f64(v)) for k, v in w.items()}


def _recompute_frames(d, w, prompt, frames):
    """Logits of every frame by full recompute of both decoders (no KV cache).

    Slow sequence: the prompt, then the tied-embedding rows sem_base + c0 of
    frames 0..N-2.  Fast sequence of frame t: [h_t, cb_0[c0], ..., cb_8[c8]].
    """
    W = _torch_weights(w)
    ids = list(prompt) + [d.sem_base + int(f[0]) for f in frames[:-1]]
    x = W["text_embed"][torch.tensor(ids)]
    if "slow.cb_embed" in W:   # decoded positions add the previous frame's codes 1..9
        P = len(prompt)
        for t, f in enumerate(frames[:-1]):
            for j in range(1, d.n_codebooks):
                x[P + t] = x[P + t] + W["slow.cb_embed"][j - 1, int(f[j])]
    for i in range(d.slow_layers):
        x = _torch_decoder(f"slow.{i}", x, W, d)
    P = len(prompt)
    out = []
    for t, f in enumerate(frames):
        h = F.rms_norm(x[P - 1 + t], (d.hidden,), W["slow.norm"], d.rms_eps)
        z0 = F.linear(h, W["text_embed"][d.sem_base:])
        rows = [h] + [W["fast.cb_embed"][j, int(f[j])] for j in range(d.n_codebooks - 1)]
        y = torch.stack(rows)
        for i in range(d.fast_layers):
            y = _torch_decoder(f"fast.{i}", y, W, d)
        zf = F.linear(F.rms_norm(y[1:], (d.hidden,), W["fast.norm"], d.rms_eps), W["fast.head"])
        out.append((z0.numpy(), zf.numpy()))
    return out


@pytest.mark.parametrize("dims", [TINY, TINY.replace(n_kv_heads=4, hidden=192, ffn=320,
                                                     text_vocab=300, semantic_vocab=40,
                                                     codebook_size=48, head_dim=32),
                                  TINY.replace(qk_norm=True, qk_norm_fast=True, slow_cb_sum=True),
                                  TINY.replace(qk_norm=True, codebook_size=16)])
def test_cached_decode_equals_full_recompute(dims):
    w = make_weights(dims, seed=3)
    o = oracle.DualAROracle(dims, w)
    prompt = make_prompt(dims, 11, seed=4)
    f0, z0 = o.prefill(prompt)
    frames, logits = [f0[0]], [z0[0]]
    for _ in range(5):
        f, z = o.decode_frame()
        frames.append(f[0])
        logits.append(z[0])
    ref = _recompute_frames(dims, w, prompt[0], frames)
    for t in range(len(frames)):
        zs, zf = ref[t]
        assert np.allclose(logits[t][0, : dims.semantic_vocab], zs, rtol=1e-9, atol=1e-11)
        assert np.allclose(logits[t][1:, : dims.codebook_size], zf, rtol=1e-9, atol=1e-11)
        # greedy ids are the argmax of the restated logits
        assert frames[t][0] == oracle.argmax_lowest(zs.astype(np.float32))
        for j in range(1, dims.n_codebooks):
            assert frames[t][j] == oracle.argmax_lowest(zf[j - 1].astype(np.float32))


def test_teacher_forcing_drives_inputs_not_outputs():
    w = make_weights(TINY, seed=5)
    prompt = make_prompt(TINY, 8, seed=6)
    forced = np.random.default_rng(0).integers(0, 64, size=(4, 1, 10)).astype(np.int32)
    o = oracle.DualAROracle(TINY, w)
    frames = []
    f, _ = o.prefill(prompt, forced=forced[0])
    frames.append(f[0])
    zs = []
    for t in range(1, 4):
        f, z = o.decode_frame(forced=forced[t])
        frames.append(f[0])
        zs.append(z[0])
    # the recompute over the forced trajectory gives the same logits
    ref = _recompute_frames(TINY, w, prompt[0], [fr[0] for fr in forced])
    for t in range(1, 4):
        assert np.allclose(zs[t - 1][0, :64], ref[t][0], rtol=1e-9, atol=1e-11)
        assert np.allclose(zs[t - 1][1:, :64], ref[t][1], rtol=1e-9, atol=1e-11)


def test_fast_step_one_two_rows_equal_two_single_rows():
    d = TINY
    w = make_weights(d, seed=8)
    o = oracle.DualAROracle(d, w)
    rng = np.random.default_rng(1)
    rows = rng.standard_normal((2, d.hidden))
    K = np.zeros((d.n_kv_heads, 10, d.head_dim))
    V = np.zeros_like(K)
    both = o._layer("fast.0", rows, [0, 1], K, V)
    K2 = np.zeros_like(K)
    V2 = np.zeros_like(K)
    a = o._layer("fast.0", rows[:1], [0], K2, V2)
    b = o._layer("fast.0", rows[1:], [1], K2, V2)
    assert np.allclose(both, np.concatenate([a, b]), rtol=1e-13, atol=1e-13)
    # cached keys and values are bf16 values
    assert np.array_equal(K2[:, :2], oracle.round_to_bf16(K2[:, :2]))
    assert np.array_equal(V2[:, :2], oracle.round_to_bf16(V2[:, :2]))


def test_fp8_model_uses_dequantised_weights():
    d = TINY
    w = make_weights(d, seed=9)
    o8 = oracle.DualAROracle(d, w, weight_format="fp8")
    codes, scale = oracle.fp8_quantize_rows(w["slow.0.w2"])
    assert np.array_equal(o8.W("slow.0.w2"), oracle.fp8_dequant_rows(codes, scale))
    # embeddings and norms stay bf16
    assert np.array_equal(o8.embed_row("text_embed", 3), oracle.bf16_bits_to_f64(w["text_embed"][3]))
    f8, z8 = o8.prefill(make_prompt(d, 8))
    ob = oracle.DualAROracle(d, w)
    fb, zb = ob.prefill(make_prompt(d, 8))
    # codebook 0 depends on the prompt only (later codebooks follow the ids)
    rel = np.linalg.norm(z8[0, 0] - zb[0, 0]) / np.linalg.norm(zb[0, 0])
    assert 1e-4 < rel < 0.1          # close to bf16, but not identical


def test_kv_capacity_and_prompt_bounds():
    d = TINY.replace(max_seq_len=10)
    o = oracle.DualAROracle(d, make_weights(d, seed=1))
    o.prefill(make_prompt(d, 9))
    o.decode_frame()              # position 9 = T - 1
    with pytest.raises(ValueError):
        o.decode_frame()
    with pytest.raises(ValueError):
        o.prefill(make_prompt(d, 11))


def test_tiny_golden_frames_reproduce():
    """Regression pin: the stored tiny-model frames (written by
    tests/golden/make_tiny_golden.py from the oracle) still come out."""
    g = _golden("tiny_frames.json")
    o = oracle.DualAROracle(TINY, make_weights(TINY, 0))
    f, z = o.prefill(make_prompt(TINY, 16, seed=0))
    frames, sums = [f[0].tolist()], [float(np.sum(z))]
    for _ in range(8):
        f, z = o.decode_frame()
        frames.append(f[0].tolist())
        sums.append(float(np.sum(z)))
    assert frames == g["greedy_frames"]
    assert np.allclose(sums, g["greedy_logit_sums"], rtol=1e-9)


def test_batched_oracle_is_independent_sequences():
    """R17: a batch of B sequences computes what B single-sequence runs
    compute; under top-k sampling, sequence b draws with Philox counter word
    3 = b (so the draws differ between otherwise equal sequences)."""
    d = TINY
    w = make_weights(d, seed=12)
    prompts = make_prompt(d, 7, seed=30, batch=3)
    ob = oracle.DualAROracle(d, w, batch=3)
    fb, zb = ob.prefill(prompts)
    frames_b, logits_b = [fb], [zb]
    for _ in range(3):
        f, z = ob.decode_frame()
        frames_b.append(f)
        logits_b.append(z)
    for b in range(3):
        o1 = oracle.DualAROracle(d, w)
        f, z = o1.prefill(prompts[b:b + 1])
        assert np.array_equal(f[0], frames_b[0][b]) and np.array_equal(z[0], logits_b[0][b])
        for t in range(1, 4):
            f, z = o1.decode_frame()
            assert np.array_equal(f[0], frames_b[t][b]) and np.array_equal(z[0], logits_b[t][b])

    # top-k: two copies of one prompt have identical logits, and each draw is
    # the sampler's pick for its own sequence index
    s = {"top_k": 8, "seed": 77}
    same = np.repeat(prompts[:1], 2, axis=0)
    ot = oracle.DualAROracle(d, w, batch=2)
    ft, zt = ot.prefill(same, s)
    assert np.array_equal(zt[0][0], zt[1][0])            # codebook-0 logits: same prompt
    for b in range(2):
        z32 = zt[b][0, : d.semantic_vocab].astype(np.float32)
        pick, _ = oracle.topk_sample(z32, 8, 77, 0, 0, b)
        assert ft[b][0] == pick
    draws = [oracle.topk_sample(zt[0][0, : d.semantic_vocab].astype(np.float32), 8, 77, 0, 0, b)[0]
             for b in range(16)]
    assert len(set(draws)) > 1                            # the sequence index reaches the draw
