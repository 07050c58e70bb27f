"""The Dual-AR decode step, restated plainly in float64.

Test infrastructure (see the package docstring).

Structure (fish-s2-pro-mlx-local-deploy README, architecture paragraph; tuna-fish
README, "Inference estimation"): a slow decoder runs along time, one token per
frame, and predicts codebook 0 (the semantic codebook); then a fast decoder
runs along depth and predicts residual codebooks 1..9 one after another, each
conditioned on the previous ones.  A frame is the 10 codebook ids.  Both
decoders keep a static KV cache; the fast one has 10 slots and starts empty
every frame (its KV term in the load formula is 2*1*4*1024*10 per step).

Readings taken where the pages are open (each is tested):
  R1  shapes as in the workload table: no q/k-norm, fused wqkv, SwiGLU w1 (gate),
      w3 (up), w2 (down); fast head has codebook_size rows.
  R2  slow input of a decoded frame is the tied text embedding row
      sem_base + c0 of the previous frame (sem_base = text_vocab - semantic_vocab);
      the semantic head is the slice [sem_base, text_vocab) of that embedding
      (tuna-fish README, "training estimation": "slowAR tied emb").
  R3  the fast decoder's first input is the slow hidden state after the final
      RMSNorm (the vector the semantic head reads).
  R5  fast step 1 processes two rows under one weight pass: position 0 = h,
      position 1 = codebook-0 embedding of c0; only position 1's logits are used.
      Step j >= 2 processes the codebook-(j-1) embedding of c_{j-1} at position j.
      9 fast weight passes per frame, as the load formula counts.
  R14 prefill of P tokens fills positions 0..P-1 and emits frame 0 from the
      last row; decode call t feeds c0 of frame t-1 at position P + t - 1.
  R16 the static KV cache holds bfloat16 values: the tuna-fish load formula
      counts every KV element at 2 bytes ("bfloat16 memory"), so keys (after
      RoPE) and values are rounded to bf16 when they are written to the cache;
      everything else stays float64.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from .numerics import (bf16_bits_to_f64, round_to_bf16, fp8_quantize_rows, fp8_dequant_rows,
                       nvfp4_quantize_rows, nvfp4_dequant_rows,
                       rmsnorm, apply_rope, attention_row, causal_attention, silu, linear)
from .sampler import argmax_lowest, apply_repetition_penalty, topk_sample

LINEAR_SUFFIXES = ("wqkv", "wo", "w1", "w3", "w2")


def linear_names(dims):
    """Names of all nn.Linear weights (the fp8 model card's 201 at full size)."""
    names = []
    for part, n in (("slow", dims.slow_layers), ("fast", dims.fast_layers)):
        for i in range(n):
            names += [f"{part}.{i}.{s}" for s in LINEAR_SUFFIXES]
    names.append("fast.head")
    return names


def load_formula(slow_params_wo_emb: int, fast_params_wo_emb: int, batch: int,
                 slow_layers: int, fast_layers: int, c_kv: int, max_length: int,
                 fast_steps: int = 9, fast_kv_len: int = 10) -> int:
    """Elements loaded per decode step, tuna-fish README "Inference estimation":

    (slow params w/o emb + fast params w/o emb * 9)
      + (2*B*L_slow*C*T  +  2*1*L_fast*C*10*9)
    i.e. the weights of one slow pass and nine fast passes plus the full static
    KV buffers.  The page evaluates it to 7,377,351,168 at B=1, T=1024.
    """
    weights = slow_params_wo_emb + fast_params_wo_emb * fast_steps
    kv = 2 * batch * slow_layers * c_kv * max_length \
        + 2 * 1 * fast_layers * c_kv * fast_kv_len * fast_steps
    return weights + kv


def decoder_params(dims, layers: int, head_rows: int, qk_norm: bool = False) -> int:
    """Parameters of a decoder without its input embedding: layers (fused wqkv,
    wo, w1, w3, w2 and two RMSNorm weights, optionally a per-head-dim q/k norm),
    the final norm and an output head of head_rows x hidden."""
    H, F = dims.hidden, dims.ffn
    per_layer = H * dims.qkv_dim + dims.q_dim * H + 3 * H * F + 2 * H
    if qk_norm:
        per_layer += 2 * dims.head_dim
    return layers * per_layer + H + head_rows * H


class DualAROracle:
    """Slow + fast decoder with static KV caches, float64 activations.

    weights: name -> bf16 bit patterns (uint16), shapes as synth.tensor_specs.
    weight_format: "bf16", or "fp8" to quantise every linear weight per row
    (fp8_quantize_rows) and use the dequantised values; embeddings and norms
    stay bf16 (drbaph s2-pro-fp8 model card, "Quantization Details"); or
    "nvfp4" for the block-scaled 4-bit format (nvfp4_quantize_rows).
    batch: number of independent sequences.
    seq_offset: added to the sequence index in the sampling counter (a
    sequence run on its own that sits in batch slot seq_offset elsewhere).
    fp8_codes: optional name -> (codes, scale) of fp8_quantize_rows already
    computed for these weights (the quantisation is then not repeated).
    """

    def __init__(self, dims, weights: dict, weight_format: str = "bf16",
                 batch: int = 1, cache_f64: bool | None = None, fp8_codes: dict | None = None,
                 seq_offset: int = 0):
        self.d = dims
        self.seq_offset = seq_offset   # sequence b draws with Philox sequence word b + seq_offset
        self.raw = weights
        self.fmt = weight_format
        self.batch = batch
        total = sum(int(np.prod(v.shape)) for v in weights.values())
        # float64 copies are kept for small models; for large ones only the
        # fast decoder's (used 9 times per frame) are kept, the rest are
        # converted from bf16 on each use.
        self.cache_f64 = (total < 100_000_000) if cache_f64 is None else cache_f64
        self.cache_fast = total >= 100_000_000
        self._cache = {}
        self.fp8 = {}
        if weight_format in ("fp8", "nvfp4"):
            names = linear_names(dims)
            quant = fp8_quantize_rows if weight_format == "fp8" else nvfp4_quantize_rows
            if fp8_codes is not None:
                self.fp8 = {n: fp8_codes[n] for n in names}
            else:   # one tensor per task; NumPy releases the GIL in its loops
                with ThreadPoolExecutor(min(32, os.cpu_count() or 1)) as ex:
                    self.fp8 = dict(zip(names, ex.map(lambda n: quant(weights[n]), names)))
        elif weight_format != "bf16":
            raise ValueError(weight_format)
        self.reset()

    # ---- weights -------------------------------------------------------
    def W(self, name: str) -> np.ndarray:
        if name in self._cache:
            return self._cache[name]
        if name in self.fp8:
            w = (fp8_dequant_rows if self.fmt == "fp8" else nvfp4_dequant_rows)(*self.fp8[name])
        else:
            w = bf16_bits_to_f64(self.raw[name])
        if self.cache_f64 or (self.cache_fast and name.startswith("fast.")):
            self._cache[name] = w
        return w

    def embed_row(self, name: str, *index) -> np.ndarray:
        return bf16_bits_to_f64(self.raw[name][index])

    # ---- state ---------------------------------------------------------
    def reset(self):
        d = self.d
        shape = (d.slow_layers, d.n_kv_heads, d.max_seq_len, d.head_dim)
        self.Ks = [np.zeros(shape) for _ in range(self.batch)]
        self.Vs = [np.zeros(shape) for _ in range(self.batch)]
        self.pos = [0] * self.batch
        self.feedback_c0 = [None] * self.batch
        self.fed_hist = [[] for _ in range(self.batch)]   # ids fed back, per frame
        self.frame_index = 0

    # ---- one decoder layer over a block of rows -------------------------
    def _layer(self, prefix, x, positions, K, V):
        """Pre-norm decoder layer over rows x [M][H] at the given positions.

        Every row's key/value is written into K, V [Hkv][T][D] at its
        position before attention (rounded to bf16, R16), and row r attends
        to positions 0..positions[r] (causal); rows are in increasing
        position order.
        """
        d = self.d
        a = rmsnorm(x, bf16_bits_to_f64(self.raw[f"{prefix}.attn_norm"]), d.rms_eps)
        qkv = linear(self.W(f"{prefix}.wqkv"), a)
        q = qkv[:, : d.q_dim].reshape(-1, d.n_heads, d.head_dim)
        k = qkv[:, d.q_dim: d.q_dim + d.kv_dim].reshape(-1, d.n_kv_heads, d.head_dim)
        v = qkv[:, d.q_dim + d.kv_dim:].reshape(-1, d.n_kv_heads, d.head_dim)
        if f"{prefix}.q_norm" in self.raw:
            # Option: per-head q/k RMSNorm before RoPE.  The tuna-fish README's
            # slowAR count ("Inference estimation", params w/o emb) holds
            # 2 x head_dim more parameters per layer than the linears and
            # norms, the size of a q and a k norm weight; read as RMSNorm over
            # each head's head_dim values with those weights (eps as elsewhere).
            q = rmsnorm(q, bf16_bits_to_f64(self.raw[f"{prefix}.q_norm"]), d.rms_eps)
            k = rmsnorm(k, bf16_bits_to_f64(self.raw[f"{prefix}.k_norm"]), d.rms_eps)
        for r, p in enumerate(positions):
            K[:, p] = round_to_bf16(apply_rope(k[r], p, d.rope_theta))
            V[:, p] = round_to_bf16(v[r])
        qr = np.stack([apply_rope(q[r], p, d.rope_theta) for r, p in enumerate(positions)])
        if len(positions) == 1:
            o = attention_row(qr[0], K, V, positions[0] + 1).reshape(1, -1)
        else:
            o = causal_attention(qr, K, V, positions).reshape(len(positions), -1)
        x = x + linear(self.W(f"{prefix}.wo"), o)
        m = rmsnorm(x, bf16_bits_to_f64(self.raw[f"{prefix}.ffn_norm"]), d.rms_eps)
        g = linear(self.W(f"{prefix}.w1"), m)
        u = linear(self.W(f"{prefix}.w3"), m)
        return x + linear(self.W(f"{prefix}.w2"), silu(g) * u)

    # ---- slow decoder ---------------------------------------------------
    def _slow(self, b, x, positions):
        for i in range(self.d.slow_layers):
            x = self._layer(f"slow.{i}", x, positions, self.Ks[b][i], self.Vs[b][i])
        return x

    def _semantic_logits(self, h):
        """Tied semantic head: rows [sem_base, text_vocab) of the text embedding."""
        d = self.d
        E = bf16_bits_to_f64(self.raw["text_embed"][d.sem_base: d.text_vocab])
        return linear(E, h)

    # ---- fast decoder ---------------------------------------------------
    def _fast_frame(self, h, c0_in, select):
        """Residual codebooks 1..n_codebooks-1 (R3, R5).

        h: post-norm slow hidden [H]; c0_in: codebook-0 id fed to the fast
        decoder; select(j, z) -> (chosen id, id fed to step j+1).
        Returns (ids 1..9 chosen, logits [9][codebook_size]).
        """
        d = self.d
        T = d.n_codebooks
        Kf = [np.zeros((d.n_kv_heads, T, d.head_dim)) for _ in range(d.fast_layers)]
        Vf = [np.zeros((d.n_kv_heads, T, d.head_dim)) for _ in range(d.fast_layers)]
        head = self.W("fast.head")
        fnorm = bf16_bits_to_f64(self.raw["fast.norm"])
        ids, logits = [], []
        prev = c0_in
        for j in range(1, d.n_codebooks):
            e = self.embed_row("fast.cb_embed", j - 1, prev)
            if j == 1:
                x, positions = np.stack([h, e]), [0, 1]
            else:
                x, positions = e[None, :], [j]
            for i in range(d.fast_layers):
                x = self._layer(f"fast.{i}", x, positions, Kf[i], Vf[i])
            z = linear(head, rmsnorm(x[-1], fnorm, d.rms_eps))
            chosen, fed = select(j, z)
            ids.append(chosen)
            logits.append(z)
            prev = fed
        return ids, np.stack(logits)

    # ---- selection --------------------------------------------------------
    def _selector(self, b, sampling, forced_row):
        s = sampling or {}
        top_k = int(s.get("top_k", 0))
        seed = int(s.get("seed", 0))
        temp = float(s.get("temperature", 1.0))
        top_p = float(s.get("top_p", 1.0))
        window = int(s.get("rep_window", 0))
        penalty = float(s.get("rep_penalty", 1.0))
        frame = self.frame_index
        past = self.fed_hist[b][max(0, len(self.fed_hist[b]) - window):] if window > 0 else []
        fed_now = {}

        def select(j, z):
            z32 = z.astype(np.float32)
            if window > 0:
                z32 = apply_repetition_penalty(z32, [f[j] for f in past], penalty)
            if top_k > 1:
                chosen, _ = topk_sample(z32, top_k, seed, frame, j, b + self.seq_offset, temp, top_p)
            else:
                chosen = argmax_lowest(z32)
            fed = chosen if forced_row is None else int(forced_row[j])
            fed_now[j] = fed
            return chosen, fed
        select.fed = fed_now
        return select

    def _frame_tail(self, b, x_last, sampling, forced_row):
        """Final norm + semantic head + c0 + fast loop, from the last slow row."""
        d = self.d
        select = self._selector(b, sampling, forced_row)
        h = rmsnorm(x_last, bf16_bits_to_f64(self.raw["slow.norm"]), d.rms_eps)
        z0 = self._semantic_logits(h)
        c0, c0_fed = select(0, z0)
        ids, zf = self._fast_frame(h, c0_fed, select)
        self.feedback_c0[b] = c0_fed
        self.fed_hist[b].append([select.fed[j] for j in range(d.n_codebooks)])
        logits = np.zeros((d.n_codebooks, max(d.semantic_vocab, d.codebook_size)))
        logits[0, : d.semantic_vocab] = z0
        logits[1:, : d.codebook_size] = zf
        return [c0] + ids, logits

    # ---- public calls -----------------------------------------------------
    def prefill(self, tokens, sampling=None, forced=None):
        """Prompt ids int [B][P] -> (frame 0 ids [B][10], logits [B][10][V]).

        Resets every sequence to position 0 first.
        """
        tokens = np.asarray(tokens)
        self.reset()
        d = self.d
        P = tokens.shape[1]
        if P < 1 or P > d.max_seq_len:
            raise ValueError("prompt length out of range")
        frames, logits = [], []
        for b in range(self.batch):
            x = np.stack([self.embed_row("text_embed", int(t)) for t in tokens[b]])
            x = self._slow(b, x, list(range(P)))
            self.pos[b] = P
            f, z = self._frame_tail(b, x[-1], sampling,
                                    None if forced is None else forced[b])
            frames.append(f)
            logits.append(z)
        self.frame_index += 1
        return np.array(frames, dtype=np.int32), np.stack(logits)

    def decode_frame(self, sampling=None, forced=None):
        """One decode call: feed each sequence's last c0, emit the next frame."""
        d = self.d
        frames, logits = [], []
        for b in range(self.batch):
            p = self.pos[b]
            if p >= d.max_seq_len:
                raise ValueError("KV capacity reached")
            x = self.embed_row("text_embed", d.sem_base + int(self.feedback_c0[b]))[None, :]
            if "slow.cb_embed" in self.raw:
                # Option: the slow input also sums the embeddings of the previous
                # frame's residual codes 1..9 (codebook j-1's table holds code c_j),
                # read from the Dual-AR description: the slow AR sees each past
                # frame, and a frame is all 10 codes.
                for j in range(1, d.n_codebooks):
                    x = x + self.embed_row("slow.cb_embed", j - 1, int(self.fed_hist[b][-1][j]))[None, :]
            x = self._slow(b, x, [p])
            self.pos[b] = p + 1
            f, z = self._frame_tail(b, x[-1], sampling,
                                    None if forced is None else forced[b])
            frames.append(f)
            logits.append(z)
        self.frame_index += 1
        return np.array(frames, dtype=np.int32), np.stack(logits)
