"""Shared helpers of the GPU parity tests (teacher-forced comparison)."""
import numpy as np

import oracle
from dual_ar_decode_gb300 import Decoder
from synth import make_prompt, make_weights

BF16_TOL = 1e-2      # logits relative L2, bf16 weights
FP8_TOL = 2e-2       # logits relative L2, fp8 per-row weights
MARGIN = 5e-2        # ids must agree where the oracle's top-1 - top-2 gap exceeds this


def vocab_of(d, j):
    return d.semantic_vocab if j == 0 else d.codebook_size


def rel_l2(g, o):
    return float(np.linalg.norm(g - o) / np.linalg.norm(o))


def margin(z):
    s = np.sort(np.asarray(z, np.float64))
    return s[-1] - s[-2]


def topk_robust(z, k, tol_abs, seed, frame, codebook, sequence=0, temperature=1.0):
    """True when the top-k draw from logits z cannot change under logit
    perturbations of size tol_abs: the k-th / (k+1)-th gap is wide, the
    picked candidate cannot trade places with a neighbour in the (logit
    desc, index asc) order, and the draw u*S sits away from every running-sum
    boundary by more than the relative change such a perturbation can make
    to the weights."""
    z32 = np.asarray(z, np.float32)
    s = np.sort(z32.astype(np.float64))[::-1]
    if len(s) > k and (s[k - 1] - s[k]) <= 4 * tol_abs:
        return False
    _, det = oracle.topk_sample(z32, k, seed, frame, codebook, sequence, temperature)
    zc = z32[det["cand"]].astype(np.float64)
    i = det["pick"]
    for nb in (i - 1, i + 1):
        if 0 <= nb < len(zc) and abs(zc[i] - zc[nb]) <= 4 * tol_abs:
            return False
    rel = 4 * tol_abs / temperature
    gaps = np.abs(det["c"].astype(np.float64) - float(det["t"]))
    return bool(np.min(gaps) > rel * float(det["S"]))


class TeacherForced:
    """Runs the oracle free (greedy or sampled) and the GPU with the
    oracle's ids forced, frame by frame, keeping both sides' logits; with
    batch > 1, B independent sequences decode in lockstep on both sides."""

    def __init__(self, dims, fmt="bf16", seed=0, weights=None, dec=None, batch=1):
        self.d = dims
        self.batch = batch
        self.w = weights if weights is not None else make_weights(dims, seed)
        self.ref = oracle.DualAROracle(dims, self.w, fmt, batch=batch)
        self.dec = dec if dec is not None else Decoder(dims, fmt, max_batch=batch)
        if dec is None:
            self.dec.load_weights(self.w)
        self.frames = []   # (frame t, sequence b, oracle ids, oracle logits, gpu ids, gpu logits)
        self.t = 0

    def _keep(self, rf, rz, gf, gz):
        for b in range(self.batch):
            self.frames.append((self.t, b, rf[b], rz[b], gf[b], gz[b]))
        self.t += 1

    def prefill(self, prompt, sampling=None):
        rf, rz = self.ref.prefill(prompt, sampling)
        gf, gz = self.dec.prefill(prompt, sampling, forced=rf, logits=True)
        self.t = 0
        self._keep(rf, rz, gf, gz)
        return rf, rz, gf, gz

    def decode(self, sampling=None):
        rf, rz = self.ref.decode_frame(sampling)
        gf, gz = self.dec.decode_frame(sampling, forced=rf, logits=True)
        self._keep(rf, rz, gf, gz)
        return rf, rz, gf, gz

    def check(self, tol, sampling=None):
        """Asserts the parity gates on every frame of every sequence; returns
        (worst rel-L2, ids compared, ids skipped)."""
        worst, compared, skipped = 0.0, 0, 0
        k = int(sampling.get("top_k", 0)) if sampling else 0
        for t, b, rf, rz, gf, gz in self.frames:
            for j in range(self.d.n_codebooks):
                V = vocab_of(self.d, j)
                o, g = rz[j, :V], gz[j, :V]
                e = rel_l2(g, o)
                worst = max(worst, e)
                assert e <= tol, f"frame {t} sequence {b} codebook {j}: rel-L2 {e:.3e} > {tol}"
                # size of the perturbation actually present in this vector
                # (itself bounded by the rel-L2 gate above)
                pert = 2.0 * float(np.max(np.abs(g.astype(np.float64) - o))) + 1e-6
                if k <= 1:
                    robust = margin(o) > MARGIN
                else:
                    robust = topk_robust(o, k, pert, int(sampling.get("seed", 0)), t, j,
                                         b, float(sampling.get("temperature", 1.0)))
                if robust:
                    compared += 1
                    assert gf[j] == rf[j], f"frame {t} sequence {b} codebook {j}: id {gf[j]} != {rf[j]}"
                else:
                    skipped += 1
                    # the rest must still be valid: a near-tied argmax, or a
                    # member of the oracle's candidate set
                    if k <= 1:
                        assert o[gf[j]] >= np.max(o) - MARGIN, (t, b, j, gf[j])
                    else:
                        cand = oracle.topk_candidates(o.astype(np.float32), k + 2)
                        assert gf[j] in set(int(c) for c in cand), (t, b, j, gf[j])
        return worst, compared, skipped
