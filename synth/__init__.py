"""Seeded synthetic inputs for the Dual-AR decode step.

This module is shared by the CPU oracle tests and the CUDA path's tests and
bench.  It holds model *shapes* and seeded *inputs* only: random-init weights,
prompt token ids and random logits.  None of the decode arithmetic lives here.

Recipe (the same for every workload):
  * Every tensor is drawn in a fixed name order.  Tensor number ``i`` of model
    seed ``s`` uses ``numpy.random.Generator(PCG64(SeedSequence([s, i])))`` and
    ``standard_normal(float32) * std`` (std 0.02), then is rounded to bfloat16
    (round to nearest even) and kept as its raw 16-bit pattern.
  * RMSNorm weights are 1.0 (bf16 0x3F80) and still consume their index;
    the optional per-head q/k norm weights are 1 + 0.1 N(0, 1).
  * Prompt ids of sequence ``b`` are ``Generator(PCG64(seed + b))``
    ``.integers(0, text_vocab)``.

The shapes follow the S2-Pro-shaped Dual-AR model of the tuna-fish README
("Inference estimation": slowAR 36 layers, fastAR 4 layers, C_kv 1024) and a
tiny model of the same structure for fast tests.
"""
from __future__ import annotations

import dataclasses
from concurrent.futures import ThreadPoolExecutor

import numpy as np

BF16_ONE = 0x3F80

__all__ = [
    "ModelDims", "TINY", "FULL", "Workload", "WORKLOADS", "tensor_specs",
    "make_weights", "make_prompt", "make_logits", "f32_to_bf16_bits",
]


@dataclasses.dataclass(frozen=True)
class ModelDims:
    """Shape of one Dual-AR model (slowAR along time + fastAR along depth)."""
    slow_layers: int
    fast_layers: int
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    text_vocab: int
    semantic_vocab: int      # rows of the tied text embedding used as slow head
    codebook_size: int       # size of each residual codebook (fast head rows)
    n_codebooks: int = 10
    max_seq_len: int = 1024
    rms_eps: float = 1e-6
    rope_theta: float = 1e6
    # Model-fidelity options (off in every benchmark workload):
    qk_norm: bool = False        # per-head RMSNorm of q and k before RoPE (slow decoder)
    qk_norm_fast: bool = False   # the same in the fast decoder
    slow_cb_sum: bool = False    # slow input adds the previous frame's codebook 1..9 embeddings

    @property
    def q_dim(self) -> int:
        return self.n_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    @property
    def qkv_dim(self) -> int:
        return self.q_dim + 2 * self.kv_dim

    @property
    def sem_base(self) -> int:
        """First text-vocab row of the semantic slice of the tied embedding."""
        return self.text_vocab - self.semantic_vocab

    def replace(self, **kw) -> "ModelDims":
        return dataclasses.replace(self, **kw)


# 2+2 layers, hidden 256, 4 q / 2 kv heads of 64, ffn 768, vocab 512,
# semantic head 64, 10 codebooks of 64.  Static KV length 64.
TINY = ModelDims(slow_layers=2, fast_layers=2, hidden=256, n_heads=4,
                 n_kv_heads=2, head_dim=64, ffn=768, text_vocab=512,
                 semantic_vocab=64, codebook_size=64, max_seq_len=64)

# S2-Pro-shaped: 36 slow + 4 fast layers, hidden 2560, 32 q / 8 kv heads of
# 128 (C_kv = 1024), ffn 9728, text vocab 151936, semantic head 4096,
# codebooks of 4096.  Static KV length 1024.
FULL = ModelDims(slow_layers=36, fast_layers=4, hidden=2560, n_heads=32,
                 n_kv_heads=8, head_dim=128, ffn=9728, text_vocab=151936,
                 semantic_vocab=4096, codebook_size=4096, max_seq_len=1024)


@dataclasses.dataclass(frozen=True)
class Workload:
    """A named decode workload: model, weight format and schedule."""
    name: str
    dims: ModelDims
    weight_dtype: str          # "bf16", "fp8" (e4m3 + per-row fp32 scale) or "nvfp4"
                               # (e2m1 + e4m3 per 16 elements + per-row fp32 scale)
    batch: int
    prefill: int
    decode: int
    top_k: int = 0             # 0 = greedy argmax
    seed: int = 0


WORKLOADS = {
    "tiny": Workload("tiny bf16 2+2 layers, prefill 16 + decode 8", TINY,
                     "bf16", 1, 16, 8),
    "full_bf16": Workload("full-size bf16, prefill 128 + decode 896 (T=1024)",
                          FULL, "bf16", 1, 128, 896),
    "full_fp8": Workload("full-size fp8 per-row, prefill 128 + decode 896 (T=1024)",
                         FULL, "fp8", 1, 128, 896),
    "full_nvfp4": Workload("full-size 4-bit block-scaled, prefill 128 + decode 896 (T=1024)",
                           FULL, "nvfp4", 1, 128, 896),
    "full_prefill_heavy": Workload(
        "full-size bf16, prefill 1024 + decode 64 (T=2048)",
        FULL.replace(max_seq_len=2048), "bf16", 1, 1024, 64),
    "full_batched16": Workload(
        "full-size bf16, batch 16, prefill 512 + decode 512 (T=4096)",
        FULL.replace(max_seq_len=4096), "bf16", 16, 512, 512),
    "full_fp8_batched16": Workload(
        "full-size fp8 per-row, batch 16, prefill 512 + decode 512 (T=4096)",
        FULL.replace(max_seq_len=4096), "fp8", 16, 512, 512),
    "full_nvfp4_batched16": Workload(
        "full-size 4-bit block-scaled, batch 16, prefill 512 + decode 512 (T=4096)",
        FULL.replace(max_seq_len=4096), "nvfp4", 16, 512, 512),
    "full_fp8_long_topk": Workload(
        "full-size fp8 per-row, prefill 3072 + decode 1024 (T=4096), top-k 30",
        FULL.replace(max_seq_len=4096), "fp8", 1, 3072, 1024, top_k=30),
}


def tensor_specs(d: ModelDims):
    """(name, shape, kind) in the fixed generation order.

    kind is "linear" (an nn.Linear weight, [out][in]), "embed", "norm" or
    "qknorm" (the optional per-head q/k RMSNorm weights, [head_dim]).
    Linear weights: wqkv [q_dim + 2 kv_dim][hidden] (rows: q heads, k heads,
    v heads), wo [hidden][q_dim], w1 (gate) and w3 (up) [ffn][hidden],
    w2 (down) [hidden][ffn], fast.head [codebook_size][hidden].
    """
    H = d.hidden
    specs = [("text_embed", (d.text_vocab, H), "embed")]

    def layer(prefix, qk):
        out = [
            (f"{prefix}.attn_norm", (H,), "norm"),
            (f"{prefix}.wqkv", (d.qkv_dim, H), "linear"),
            (f"{prefix}.wo", (H, d.q_dim), "linear"),
            (f"{prefix}.ffn_norm", (H,), "norm"),
            (f"{prefix}.w1", (d.ffn, H), "linear"),
            (f"{prefix}.w3", (d.ffn, H), "linear"),
            (f"{prefix}.w2", (H, d.ffn), "linear"),
        ]
        if qk:
            out += [(f"{prefix}.q_norm", (d.head_dim,), "qknorm"),
                    (f"{prefix}.k_norm", (d.head_dim,), "qknorm")]
        return out

    for i in range(d.slow_layers):
        specs += layer(f"slow.{i}", d.qk_norm)
    specs.append(("slow.norm", (H,), "norm"))
    for i in range(d.fast_layers):
        specs += layer(f"fast.{i}", d.qk_norm_fast)
    specs.append(("fast.norm", (H,), "norm"))
    specs.append(("fast.head", (d.codebook_size, H), "linear"))
    # table j-1 embeds the id fed at fast step j: c0 (semantic) at step 1,
    # c_{j-1} after; with a semantic vocabulary larger than the codebooks the
    # tables are as tall as the larger of the two
    specs.append(("fast.cb_embed", (d.n_codebooks - 1, max(d.semantic_vocab, d.codebook_size), H),
                  "embed"))
    if d.slow_cb_sum:
        specs.append(("slow.cb_embed", (d.n_codebooks - 1, d.codebook_size, H), "embed"))
    return specs


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); return uint16 bits.

    Only used on finite synthetic values.
    """
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = (u >> np.uint32(16)) & np.uint32(1)
    r += np.uint32(0x7FFF)
    r += u
    r >>= np.uint32(16)
    return r.astype(np.uint16)


def _draw(seed: int, idx: int, shape, std: float) -> np.ndarray:
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, idx])))
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    step = 1 << 24
    for s in range(0, n, step):
        e = min(n, s + step)
        x = g.standard_normal(e - s, dtype=np.float32)
        x *= np.float32(std)
        out[s:e] = f32_to_bf16_bits(x)
    return out.reshape(shape)


def make_weights(d: ModelDims, seed: int = 0, std: float = 0.02,
                 threads: int = 0) -> dict:
    """All model tensors as bf16 bit patterns (numpy uint16), keyed by name."""
    specs = tensor_specs(d)
    out = {}

    def one(item):
        idx, (name, shape, kind) = item
        if kind == "norm":
            return name, np.full(shape, BF16_ONE, dtype=np.uint16)
        if kind == "qknorm":   # 1 + N(0, 0.1): not all ones, so their indexing shows
            g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, idx])))
            w = 1.0 + 0.1 * g.standard_normal(shape, dtype=np.float32)
            return name, f32_to_bf16_bits(w.astype(np.float32))
        return name, _draw(seed, idx, shape, std)

    n_thr = threads or min(32, max(1, __import__("os").cpu_count() or 1))
    with ThreadPoolExecutor(n_thr) as ex:
        for name, arr in ex.map(one, enumerate(specs)):
            out[name] = arr
    return out


def make_prompt(d: ModelDims, length: int, seed: int = 0, batch: int = 1) -> np.ndarray:
    """Prompt token ids, int32 [batch][length], uniform in [0, text_vocab)."""
    rows = []
    for b in range(batch):
        g = np.random.Generator(np.random.PCG64(seed + b))
        rows.append(g.integers(0, d.text_vocab, size=length, dtype=np.int64))
    return np.stack(rows).astype(np.int32)


def make_logits(n: int, vocab: int, seed: int = 0, scale: float = 1.0,
                ties: bool = False) -> np.ndarray:
    """float32 [n][vocab] logits ~ N(0, scale); with ties, values are coarsely
    quantised so that equal logits occur often."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 7])))
    z = g.standard_normal((n, vocab), dtype=np.float32) * np.float32(scale)
    if ties:
        z = np.round(z * 4.0).astype(np.float32) / np.float32(4.0)
    return z
