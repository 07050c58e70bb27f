"""GPU parity of batched decode: B independent sequences in lockstep, every
linear layer one skinny tensor-core GEMM over the B activation rows.

The oracle runs each sequence on its own (no batching in its arithmetic);
the gates are those of single-sequence decode: logits relative L2 <= 1e-2
(bf16) / 2e-2 (fp8) for every sequence, codebook and frame under teacher
forcing, ids equal wherever the oracle's margin allows.
"""
import numpy as np
import pytest
import torch

import oracle
from dual_ar_decode_gb300 import Decoder, TfError, op_gemm_skinny
from synth import FULL, TINY, make_prompt, make_weights, f32_to_bf16_bits

from gpu_helpers import BF16_TOL, FP8_TOL, ContinuousForced, TeacherForced, rel_l2, vocab_of

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def dev_u16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV)


# ------------------------------------------------------------------ op

@pytest.mark.parametrize("M,N,K", [(1, 256, 256), (3, 200, 200), (16, 6144, 2560),
                                   (32, 19456, 2560), (17, 2560, 9728), (64, 4096, 2560),
                                   (2, 64, 256), (33, 2560, 4096), (16, 130, 72)])
def test_skinny_gemm_matches_oracle(M, N, K):
    """Split-K swap-AB tcgen05 GEMM against A @ W^T in float64, including
    ragged weight tiles (N % 128) and ragged K slices (K % 64)."""
    rng = np.random.default_rng(M * 13 + N + K)
    A = rng.standard_normal((M, K)).astype(np.float32)
    Wb = f32_to_bf16_bits(rng.standard_normal((N, K)).astype(np.float32) * 0.02)
    Ad = torch.from_numpy(A).to(DEV)
    Wd = dev_u16(Wb)
    C = torch.full((M, N), np.nan, dtype=torch.float32, device=DEV)
    op_gemm_skinny(Ad.data_ptr(), Wd.data_ptr(), M, N, K, C.data_ptr())
    ref = oracle.linear(oracle.bf16_bits_to_f64(Wb), A.astype(np.float64))
    got = C.cpu().numpy().astype(np.float64)
    rms = np.sqrt(np.mean(ref ** 2))
    assert np.isfinite(got).all()
    # as the prompt GEMM: bf16 hi + lo parts carry A to ~2^-17 relative, fp32
    # accumulation in TMEM and over the K splits adds about as much again
    assert np.max(np.abs(got - ref)) <= 2e-4 * rms
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= 5e-5


@pytest.mark.parametrize("M,N,K,all_codes", [(16, 6144, 2560, False), (32, 19456, 2560, False),
                                             (17, 2560, 9728, False), (3, 200, 208, False),
                                             (64, 4096, 2560, False), (16, 300, 512, True)])
def test_skinny_gemm_fp8_matches_oracle(M, N, K, all_codes):
    """The e4m3 skinny GEMM (codes converted to bf16 in shared memory, row
    scale in the epilogue) against A @ dequant(W)^T in float64, with the
    oracle's own quantiser (or every finite code, with random row scales)."""
    from dual_ar_decode_gb300 import op_gemm_skinny_fp8
    rng = np.random.default_rng(M * 7 + N + K)
    A = rng.standard_normal((M, K)).astype(np.float32)
    if all_codes:
        codes = (np.arange(N * K) % 256).astype(np.uint8).reshape(N, K)
        codes[(codes & 0x7F) == 0x7F] = 0          # NaN codes are refused at load
        scale = rng.uniform(0.5, 2.0, N).astype(np.float32) / 448.0
    else:
        codes, scale = oracle.fp8_quantize_rows(
            f32_to_bf16_bits(rng.standard_normal((N, K)).astype(np.float32) * 0.02))
    Ad = torch.from_numpy(A).to(DEV)
    Wd = torch.from_numpy(np.ascontiguousarray(codes)).to(DEV)
    Sd = torch.from_numpy(np.asarray(scale, np.float32)).to(DEV)
    C = torch.full((M, N), np.nan, dtype=torch.float32, device=DEV)
    op_gemm_skinny_fp8(Ad.data_ptr(), Wd.data_ptr(), Sd.data_ptr(), M, N, K, C.data_ptr())
    ref = oracle.linear(oracle.fp8_dequant_rows(codes, scale), A.astype(np.float64))
    got = C.cpu().numpy().astype(np.float64)
    rms = np.sqrt(np.mean(ref ** 2))
    assert np.isfinite(got).all()
    # the bf16 values of the codes are exact; hi + lo activations and fp32
    # accumulation as in the bf16 case, the row scale one more rounding
    assert np.max(np.abs(got - ref)) <= 2e-4 * rms
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= 5e-5


@pytest.mark.parametrize("M,N,K,all_codes", [(16, 6144, 2560, False), (32, 19456, 2560, False),
                                             (17, 2560, 9728, False), (3, 200, 256, False),
                                             (64, 4096, 2560, False), (16, 130, 512, True)])
def test_skinny_gemm_nvfp4_matches_oracle(M, N, K, all_codes):
    """The 4-bit skinny GEMM (e2m1 codes times e4m3 block scales decoded to
    bf16 in shared memory, row scale in the epilogue) against A @ dequant(W)^T
    in float64, with the oracle's quantiser, or every code under a range of
    block scales (2^-9 .. 448) with random row scales."""
    from dual_ar_decode_gb300 import op_gemm_skinny_nvfp4
    from gpu_helpers import nvfp4_pack
    rng = np.random.default_rng(M * 11 + N + K)
    A = rng.standard_normal((M, K)).astype(np.float32)
    if all_codes:
        codes = (np.arange(N * K) % 16).astype(np.uint8).reshape(N, K // 16, 16)
        sb = np.array([0x01, 0x20, 0x38, 0x40, 0x55, 0x7E], np.uint8)[np.arange(N * (K // 16)) % 6]
        sb = sb.reshape(N, K // 16)
        sr = rng.uniform(0.5, 2.0, N).astype(np.float32) / 2688.0
    else:
        codes, sb, sr = oracle.nvfp4_quantize_rows(
            f32_to_bf16_bits(rng.standard_normal((N, K)).astype(np.float32) * 0.02))
    Ad = torch.from_numpy(A).to(DEV)
    Wd = torch.from_numpy(nvfp4_pack(codes, sb)).to(DEV)
    Sd = torch.from_numpy(np.asarray(sr, np.float32)).to(DEV)
    C = torch.full((M, N), np.nan, dtype=torch.float32, device=DEV)
    op_gemm_skinny_nvfp4(Ad.data_ptr(), Wd.data_ptr(), Sd.data_ptr(), M, N, K, C.data_ptr())
    ref = oracle.linear(oracle.nvfp4_dequant_rows(codes, sb, sr), A.astype(np.float64))
    got = C.cpu().numpy().astype(np.float64)
    rms = np.sqrt(np.mean(ref ** 2))
    assert np.isfinite(got).all()
    # exact bf16 weights (e2m1 x e4m3 has <= 6 significant bits); hi + lo
    # activations and fp32 accumulation as in the bf16 case; the row scale
    # applied once where the oracle rounds each weight
    assert np.max(np.abs(got - ref)) <= 2e-4 * rms
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= 5e-5


def test_skinny_gemm_is_deterministic_and_rejects_bad_shapes():
    rng = np.random.default_rng(3)
    M, N, K = 16, 2560, 9728
    Ad = torch.from_numpy(rng.standard_normal((M, K)).astype(np.float32)).to(DEV)
    Wd = dev_u16(f32_to_bf16_bits(rng.standard_normal((N, K)).astype(np.float32) * 0.02))
    outs = []
    for _ in range(3):
        C = torch.empty((M, N), dtype=torch.float32, device=DEV)
        op_gemm_skinny(Ad.data_ptr(), Wd.data_ptr(), M, N, K, C.data_ptr())
        outs.append(C.cpu().numpy())
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2])
    C = torch.empty((65, N), dtype=torch.float32, device=DEV)
    with pytest.raises(TfError, match="INVAL"):      # more than 64 rows
        op_gemm_skinny(Ad.data_ptr(), Wd.data_ptr(), 65, N, K, C.data_ptr())
    with pytest.raises(TfError, match="INVAL"):      # odd N
        op_gemm_skinny(Ad.data_ptr(), Wd.data_ptr(), M, N - 1, K, C.data_ptr())


# ------------------------------------------------------------------ model

TINY_ODD = TINY.replace(hidden=192, ffn=320, n_heads=4, n_kv_heads=4, head_dim=64,
                        text_vocab=300, semantic_vocab=40, codebook_size=48, max_seq_len=40)
TINY_G8 = TINY.replace(hidden=256, ffn=512, n_heads=8, n_kv_heads=1, head_dim=128,
                       max_seq_len=64)


TINY_OPTS = TINY.replace(qk_norm=True, qk_norm_fast=True, slow_cb_sum=True, codebook_size=32)


@pytest.mark.parametrize("dims,fmt,tol,B,P", [(TINY, "bf16", BF16_TOL, 3, 16),
                                              (TINY, "fp8", FP8_TOL, 2, 16),
                                              (TINY_ODD, "bf16", BF16_TOL, 5, 12),
                                              (TINY_G8, "bf16", BF16_TOL, 4, 40),
                                              (TINY, "bf16", BF16_TOL, 32, 8),
                                              (TINY_OPTS, "bf16", BF16_TOL, 3, 40),
                                              (TINY, "nvfp4", FP8_TOL, 4, 16)])
def test_tiny_batched_teacher_forced(dims, fmt, tol, B, P):
    """B sequences with their own prompts; P = 40 reaches the split
    attention path (more than 32 keys) with one ticket per row."""
    tf = TeacherForced(dims, fmt, seed=0, batch=B)
    tf.prefill(make_prompt(dims, P, seed=10, batch=B))
    for _ in range(5):
        tf.decode()
    worst, compared, skipped = tf.check(tol)
    assert compared > 0.5 * (compared + skipped)
    tf.dec.close()


@pytest.mark.parametrize("k", [30, 4])
def test_tiny_batched_topk_teacher_forced(k):
    """Sampling draws per sequence: Philox counter (frame, codebook, sequence)."""
    s = {"top_k": k, "seed": 99}
    tf = TeacherForced(TINY, "bf16", seed=0, batch=4)
    tf.prefill(make_prompt(TINY, 16, seed=3, batch=4), s)
    for _ in range(4):
        tf.decode(s)
    worst, compared, skipped = tf.check(BF16_TOL, s)
    assert compared >= 20
    tf.dec.close()


def test_batched_decode_frames_equal_single_calls_and_deterministic():
    w = make_weights(TINY, seed=5)
    prompt = make_prompt(TINY, 12, seed=5, batch=5)
    runs = []
    for mode in ("single", "batched", "batched"):
        dec = Decoder(TINY, "bf16", max_batch=8)
        dec.load_weights(w)
        f0, _ = dec.prefill(prompt)
        if mode == "single":
            fr = np.stack([dec.decode_frame()[0] for _ in range(6)])
        else:
            fr = dec.decode_frames(6)
        assert fr.shape == (6, 5, 10)
        runs.append(np.concatenate([f0[None], fr]))
        dec.close()
    assert np.array_equal(runs[0], runs[1]) and np.array_equal(runs[1], runs[2])


def test_batch_size_changes_and_errors():
    """Prefills of different B on one context; B beyond max_batch and a bad
    forced row are refused without changing the state."""
    d = TINY
    w = make_weights(d, seed=6)
    dec = Decoder(d, "bf16", max_batch=4)
    dec.load_weights(w)
    with pytest.raises(TfError, match="INVAL"):
        dec.prefill(make_prompt(d, 4, batch=5))
    f3, _ = dec.prefill(make_prompt(d, 6, seed=1, batch=3))
    assert f3.shape == (3, 10)
    bad = np.zeros((3, 10), np.int32)
    bad[2, 4] = d.codebook_size
    with pytest.raises(TfError, match="INVAL"):
        dec.decode_frame(forced=bad)
    g3, _ = dec.decode_frame()
    assert g3.shape == (3, 10)
    # back to one sequence (the batch-1 kernels) and again to four
    ref1 = oracle.DualAROracle(d, w)
    rf, rz = ref1.prefill(make_prompt(d, 6, seed=2))
    gf, gz = dec.prefill(make_prompt(d, 6, seed=2), forced=rf, logits=True)
    for j in range(10):
        V = vocab_of(d, j)
        assert rel_l2(gz[0, j, :V], rz[0, j, :V]) <= BF16_TOL
    f4, _ = dec.prefill(make_prompt(d, 6, seed=3, batch=4))
    assert dec.decode_frames(3).shape == (3, 4, 10)
    dec.close()


# ------------------------------------------------------------------ continuous batching

def _continuous_schedule(cf, d, sampling=None):
    """Joins, decodes and releases with prompts of different lengths; the
    first phase has slot 0 alone (the batch-1 kernels), later ones the
    batched kernels with idle slots inside the batch."""
    P = lambda n, seed: make_prompt(d, n, seed=seed)[0]
    cf.join(0, P(10, 1))
    for _ in range(3):
        cf.decode(sampling)
    cf.join(2, P(5, 2))                      # slot 1 idle inside the batch
    for _ in range(3):
        cf.decode(sampling)
    cf.leave(0)
    cf.join(1, P(40, 3))                     # more than one 32-position page
    for _ in range(3):
        cf.decode(sampling)
    cf.join(0, P(1, 4))                      # a one-id prompt: no prompt pass
    cf.leave(2)
    for _ in range(2):
        cf.decode(sampling)


@pytest.mark.parametrize("dims,fmt,tol,paged", [(TINY, "bf16", BF16_TOL, False),
                                                (TINY, "bf16", BF16_TOL, True),
                                                (TINY_OPTS, "bf16", BF16_TOL, True),
                                                (TINY, "fp8", FP8_TOL, True)])
def test_continuous_batching_ragged_prompts(dims, fmt, tol, paged):
    """Sequences join and leave slots while others decode, each at its own
    position, with dense or paged KV caches; every sequence matches its own
    oracle run."""
    w = make_weights(dims, seed=31)
    dec = Decoder(dims, fmt, max_batch=4, paged=paged)
    dec.load_weights(w)
    cf = ContinuousForced(dims, dec, w, fmt)
    _continuous_schedule(cf, dims)
    worst, compared, skipped = cf.check(tol)
    assert compared > 0.5 * (compared + skipped)
    dec.close()


def test_continuous_batching_topk_uses_the_slot_as_sequence():
    s = {"top_k": 4, "seed": 5}
    w = make_weights(TINY, seed=32)
    dec = Decoder(TINY, "bf16", max_batch=4, paged=True)
    dec.load_weights(w)
    cf = ContinuousForced(TINY, dec, w)
    _continuous_schedule(cf, TINY, s)
    worst, compared, skipped = cf.check(BF16_TOL, s)
    assert compared >= 40
    dec.close()


@pytest.mark.parametrize("paged", [False, True])
def test_lockstep_batch_on_paged_caches(paged):
    tf = TeacherForced(TINY, "bf16", seed=0, batch=3,
                       dec=Decoder(TINY, "bf16", max_batch=3, paged=paged))
    tf.dec.load_weights(tf.w)
    tf.prefill(make_prompt(TINY, 37, seed=10, batch=3))
    for _ in range(4):
        tf.decode()
    worst, compared, skipped = tf.check(BF16_TOL)
    assert compared > 0.5 * (compared + skipped)
    tf.dec.close()


def test_paged_kv_matches_dense_bit_for_bit_in_the_batched_step():
    """The batched step reads and writes the paged caches through the block
    table in the same order as the dense caches: with the same forced ids the
    logits agree bit for bit (prompt pass and batched step both use the
    row-streaming attention)."""
    w = make_weights(TINY, seed=34)
    prompts = make_prompt(TINY, 45, seed=11, batch=3)     # 2 pages, a ragged third
    decs = [Decoder(TINY, "bf16", max_batch=3, paged=pg) for pg in (False, True)]
    forced = np.random.default_rng(3).integers(0, TINY.codebook_size, (6, 3, 10)).astype(np.int32)
    outs = []
    for dec in decs:
        dec.load_weights(w)
        f0, z0 = dec.prefill(prompts, forced=forced[0], logits=True)
        zs = [z0]
        for t in range(1, 6):
            zs.append(dec.decode_frame(forced=forced[t], logits=True)[1])
        outs.append(np.stack(zs))
        dec.close()
    assert np.isfinite(outs[0]).all()
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))


def test_continuous_batching_errors():
    d = TINY.replace(max_seq_len=24)
    w = make_weights(d, seed=33)
    dec = Decoder(d, "bf16", max_batch=2, paged=True)
    dec.load_weights(w)
    with pytest.raises(TfError, match="INVAL"):
        dec.prefill_seq(2, make_prompt(d, 4)[0])                 # no such slot
    with pytest.raises(TfError, match="INVAL"):
        dec.prefill_seq(0, np.array([0, d.text_vocab], np.int32))  # id out of range
    with pytest.raises(TfError, match="STATE"):
        dec.decode_frame()                                        # nothing active
    dec.prefill_seq(1, make_prompt(d, 22, seed=1)[0])             # positions 0..21
    dec.decode_frame()                                            # frame 0 at 21
    dec.decode_frame()                                            # frame 1 at 22
    dec.decode_frame()                                            # frame 2 at 23
    with pytest.raises(TfError, match="CAPACITY"):
        dec.decode_frame()
    dec.release_seq(1)
    dec.prefill_seq(0, make_prompt(d, 3, seed=2)[0])              # the pages came back
    f, _ = dec.decode_frame()
    assert f.shape == (1, 10) and (f >= 0).all()
    dec.close()


# ------------------------------------------------------------------ full size

def test_full_size_batched16_sampled_sequences():
    """Full-size model, 16 sequences, KV length 4096 (the batched benchmark's
    context), prompts of 64 tokens (more than 32 keys: split attention),
    2 decode frames.  The oracle runs sequences 0 and 15 on their own; the
    other sequences are teacher-forced with fixed ids."""
    d = FULL.replace(max_seq_len=4096)
    B, P = 16, 64
    w = make_weights(d, seed=0)
    prompts = make_prompt(d, P, seed=20, batch=B)
    checked = (0, 15)
    refs = {b: oracle.DualAROracle(d, w) for b in checked}
    dec = Decoder(d, "bf16", max_batch=B)
    dec.load_weights(w)
    forced = np.zeros((B, 10), np.int32)
    ref_out = {}
    for b in checked:
        ref_out[b] = refs[b].prefill(prompts[b:b + 1])
        forced[b] = ref_out[b][0][0]
    gf, gz = dec.prefill(prompts, forced=forced, logits=True)
    results = [(ref_out, gf, gz)]
    for _ in range(2):
        ref_out = {b: refs[b].decode_frame() for b in checked}
        for b in checked:
            forced[b] = ref_out[b][0][0]
        gf, gz = dec.decode_frame(forced=forced, logits=True)
        results.append((ref_out, gf, gz))
    compared = 0
    for t, (ro, gf, gz) in enumerate(results):
        for b in checked:
            rf, rz = ro[b][0][0], ro[b][1][0]
            for j in range(10):
                V = vocab_of(d, j)
                e = rel_l2(gz[b, j, :V], rz[j, :V])
                assert e <= BF16_TOL, (t, b, j, e)
                s = np.sort(rz[j, :V])
                if s[-1] - s[-2] > 5e-2:
                    compared += 1
                    assert gf[b, j] == rf[j], (t, b, j)
    assert compared >= 30
    dec.close()


def test_full_size_continuous_batching_paged():
    """Full-size bf16 with paged caches: sequences with 37-, 130- and 513-id
    prompts join four slots at different times (split attention over many
    pages); two of them are checked against their own oracle runs, the
    third is teacher-forced with its oracle too but only for 1 frame."""
    d = FULL.replace(max_seq_len=1024)
    w = make_weights(d, seed=0)
    dec = Decoder(d, "bf16", max_batch=4, paged=True)
    dec.load_weights(w)
    cf = ContinuousForced(d, dec, w)
    cf.join(3, make_prompt(d, 513, seed=41)[0])
    cf.decode()
    cf.join(0, make_prompt(d, 37, seed=42)[0])
    cf.decode()
    cf.leave(3)
    cf.join(1, make_prompt(d, 130, seed=43)[0])
    cf.decode()
    worst, compared, skipped = cf.check(BF16_TOL)
    assert compared >= 20
    dec.close()
