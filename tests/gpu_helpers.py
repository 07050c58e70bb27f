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


def topk_delta(o, tol):
    """A-priori per-logit perturbation for the top-k robustness test: three
    times the RMS error that the relative-L2 gate tol allows (3 tol rms(o)),
    from the oracle's logits only."""
    o = np.asarray(o, np.float64)
    return 3.0 * tol * float(np.sqrt(np.mean(o * o)))


def margin(z):
    s = np.sort(np.asarray(z, np.float64))
    return s[-1] - s[-2]


def topk_robust(z, k, delta, seed, frame, codebook, sequence=0, temperature=1.0, top_p=1.0):
    """True when the oracle's top-k draw from logits z stays the same under
    any change of every logit by at most delta (an a-priori bound taken from
    the oracle's logits and the parity tolerance, never from the GPU's).

    Such a change can only (a) swap candidates whose logits lie within
    2*delta, and (b) scale every weight exp((z_i - z_max) / T) by a factor
    within exp(+-2*delta/T), which moves each normalised running sum r_i =
    c_i / S to at most r e^a / (r e^a + (1 - r) e^-a) and at least
    r e^-a / (r e^-a + (1 - r) e^a), a = 2*delta/T.  The pick i (the first
    candidate with u < r_i) is stable when the picked candidate cannot trade
    places with a neighbour, cannot be displaced from the set when it is the
    last candidate, and u keeps clear of the moved r_{i-1} and r_i.  With a
    nucleus (top_p < 1) the cut must also stay where it is (the moved
    r_{n-1} stays >= top_p and r_{n-2} below it), and the draw is judged on
    the sums normalised by the nucleus' own sum."""
    z32 = np.asarray(z, np.float32)
    _, det = oracle.topk_sample(z32, k, seed, frame, codebook, sequence, temperature, top_p)
    zc = z32[det["cand"]].astype(np.float64)
    i = det["pick"]
    for nb in (i - 1, i + 1):
        if 0 <= nb < len(zc) and abs(zc[i] - zc[nb]) <= 2 * delta:
            return False
    if i == len(zc) - 1 and len(z32) > len(zc):
        nxt = np.sort(z32.astype(np.float64))[::-1][len(zc)]
        if zc[i] - nxt <= 2 * delta:
            return False
    a = 2 * delta / temperature
    up = lambda x: x * np.exp(a) / (x * np.exp(a) + (1 - x) * np.exp(-a))
    dn = lambda x: x * np.exp(-a) / (x * np.exp(-a) + (1 - x) * np.exp(a))
    eps = 1e-6   # float32 rounding of the running sums and of u * S
    n = int(det["n"])
    if n < len(zc):   # a nucleus cut: it must not move
        rS = det["c"].astype(np.float64) / float(det["S"])
        if dn(rS[n - 1]) < top_p + eps or (n >= 2 and up(rS[n - 2]) > top_p - eps):
            return False
    r = det["c"][:n].astype(np.float64) / float(det["Sk"])
    u = float(det["u"])
    lo_ok = i == 0 or u > up(r[i - 1]) + eps
    hi_ok = i == n - 1 or u < dn(r[i]) - eps
    return bool(lo_ok and hi_ok)


class TeacherForced:
    """Runs the oracle free (greedy or sampled) and the GPU with the
    oracle's ids forced, frame by frame, keeping both sides' logits; with
    batch > 1, B independent sequences decode in lockstep on both sides."""

    def __init__(self, dims, fmt="bf16", seed=0, weights=None, dec=None, batch=1, fp8_codes=None):
        self.d = dims
        self.batch = batch
        self.w = weights if weights is not None else make_weights(dims, seed)
        self.ref = oracle.DualAROracle(dims, self.w, fmt, batch=batch, fp8_codes=fp8_codes)
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
        (worst rel-L2, ids compared, ids skipped).  With a repetition window
        the selection input is the oracle's logits after the penalty over the
        ids fed back (under teacher forcing, the oracle's own picks) in the
        previous rep_window frames; a penalty r scales a logit's change by at
        most max(1, r), so the bounds scale with it."""
        worst, compared, skipped = 0.0, 0, 0
        s = sampling or {}
        k = int(s.get("top_k", 0))
        W = int(s.get("rep_window", 0))
        r = float(s.get("rep_penalty", 1.0))
        amp = max(1.0, r) if W else 1.0
        fed = {}    # (sequence, frame) -> oracle ids fed back
        for t, b, rf, rz, gf, gz in self.frames:
            fed[(b, t)] = rf
        for t, b, rf, rz, gf, gz in self.frames:
            for j in range(self.d.n_codebooks):
                V = vocab_of(self.d, j)
                o, g = rz[j, :V], gz[j, :V]
                e = rel_l2(g, o)
                worst = max(worst, e)
                assert e <= tol, f"frame {t} sequence {b} codebook {j}: rel-L2 {e:.3e} > {tol}"
                if W:
                    recent = [fed[(b, u)][j] for u in range(max(0, t - W), t)]
                    o = oracle.apply_repetition_penalty(o.astype(np.float32), recent, r)
                if k <= 1:
                    robust = margin(o) > MARGIN * amp
                else:
                    # per-logit change the gate allows if the error were
                    # spread like noise at the tolerance: 3 * tol * rms
                    delta = topk_delta(rz[j, :V], tol) * amp
                    robust = topk_robust(o, k, delta, int(s.get("seed", 0)), t, j,
                                         b, float(s.get("temperature", 1.0)),
                                         float(s.get("top_p", 1.0)))
                if robust:
                    compared += 1
                    assert gf[j] == rf[j], f"frame {t} sequence {b} codebook {j}: id {gf[j]} != {rf[j]}"
                else:
                    skipped += 1
                    # the rest must still be valid: a near-tied argmax, or a
                    # member of the oracle's candidate set
                    if k <= 1:
                        assert o[gf[j]] >= np.max(o) - MARGIN * amp, (t, b, j, gf[j])
                    else:
                        cand = oracle.topk_candidates(o.astype(np.float32), k + 2)
                        assert gf[j] in set(int(c) for c in cand), (t, b, j, gf[j])
        return worst, compared, skipped


class ContinuousForced:
    """Continuous batching under teacher forcing: sequences join slots of one
    decoder (tf_prefill_seq) and leave them (tf_release_seq) while the others
    decode; every sequence is also run by its own oracle (Philox sequence word
    = its slot).  A sequence's frame 0 is the decode call right after it
    joined.  Records (slot, frame t, oracle ids, oracle logits, gpu ids, gpu
    logits) for check(); idle slots must read -1."""

    def __init__(self, dims, dec, weights, fmt="bf16"):
        self.d, self.dec, self.w, self.fmt = dims, dec, weights, fmt
        self.seqs = {}      # slot -> [oracle, prompt, frames decoded]
        self.frames = []
        self.idle_ok = True

    def join(self, slot, prompt):
        self.dec.prefill_seq(slot, prompt)
        self.seqs[slot] = [oracle.DualAROracle(self.d, self.w, self.fmt, seq_offset=slot),
                           np.asarray(prompt, np.int32)[None], 0]

    def leave(self, slot):
        self.dec.release_seq(slot)
        del self.seqs[slot]

    def decode(self, sampling=None):
        B = self.dec.batch
        forced = np.zeros((B, self.d.n_codebooks), np.int32)
        want = {}
        for slot, st in self.seqs.items():
            o, prompt, t = st
            rf, rz = (o.prefill(prompt, sampling) if t == 0 else o.decode_frame(sampling))
            forced[slot] = rf[0]
            want[slot] = (t, rf[0], rz[0])
            st[2] = t + 1
        gf, gz = self.dec.decode_frame(sampling, forced=forced, logits=True)
        for slot in range(B):
            if slot in want:
                t, rf, rz = want[slot]
                self.frames.append((t, slot, rf, rz, gf[slot], gz[slot]))
            else:
                self.idle_ok &= bool((gf[slot] == -1).all())

    def check(self, tol, sampling=None):
        """The gates of TeacherForced.check on every recorded (slot, frame)."""
        assert self.idle_ok, "an idle slot did not read -1"
        tf = TeacherForced.__new__(TeacherForced)
        tf.d = self.d
        tf.frames = [(t, slot, rf, rz, gf, gz) for t, slot, rf, rz, gf, gz in self.frames]
        return TeacherForced.check(tf, tol, sampling)


def nvfp4_pack(codes, sb):
    """Oracle codes [rows][blocks][16] and block scales -> the stored rows:
    two codes per byte (even element in the low nibble), then the scales."""
    c = codes.reshape(codes.shape[0], -1)
    return np.concatenate([(c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8), sb], axis=1)
