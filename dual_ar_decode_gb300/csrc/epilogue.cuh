// Epilogue helpers shared by the decode GEMV and the prompt GEMM.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace tf {

// Sequence of activation row m: rows are grouped by sequence (p.rps rows
// each) from sequence seq_base, or all belong to sequence seq_base.
__device__ __forceinline__ int row_seq(const GemvParams& p, int m) {
  return p.seq_base + (p.rps > 0 ? m / p.rps : 0);
}

// Position of activation row m: its sequence's position plus its index among
// the sequence's rows, or pos_fixed plus the row index.
__device__ __forceinline__ int row_pos(const GemvParams& p, int m) {
  return (p.pos_ptr ? __ldg(p.pos_ptr + row_seq(p, m)) : p.pos_fixed) + (p.rps > 0 ? m % p.rps : m);
}

// Element offset of the cached K (or V) row of (sequence, KV head g,
// position): dense caches [sequence][Hkv][T][D], or pages
// [page][Hkv][kKvPage][D] found in the block table.
__device__ __forceinline__ size_t kv_index(const int32_t* tbl, int npp, int hkv, int T, int64_t kv_seq,
                                           int seq, int g, int pos, int D) {
  if (tbl) {
    const int page = __ldg(tbl + (size_t)seq * npp + pos / kKvPage);
    return (((size_t)page * hkv + g) * kKvPage + pos % kKvPage) * D;
  }
  return (size_t)seq * (size_t)kv_seq + ((size_t)g * T + pos) * D;
}

__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }

// Dot product of one 16-byte weight chunk with the matching activations.
template <int WT, int EPC>
__device__ __forceinline__ float chunk_dot(const uint4 w, const float* a) {
  float s = 0.f;
  if constexpr (WT == 0) {
    const uint32_t v[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      s = fmaf(bf16_lo(v[i]), a[2 * i], s);
      s = fmaf(bf16_hi(v[i]), a[2 * i + 1], s);
    }
  } else {
    const uint32_t v[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 lo = e4m3x2_to_f32x2(static_cast<uint16_t>(v[i] & 0xFFFFu));
      float2 hi = e4m3x2_to_f32x2(static_cast<uint16_t>(v[i] >> 16));
      s = fmaf(lo.x, a[4 * i], s);
      s = fmaf(lo.y, a[4 * i + 1], s);
      s = fmaf(hi.x, a[4 * i + 2], s);
      s = fmaf(hi.y, a[4 * i + 3], s);
    }
  }
  return s;
}

__device__ __forceinline__ unsigned long long pack_key(float v, int idx) {
  if (v == 0.f) v = 0.f;  // -0 and +0 tie, as equal floats do
  return (static_cast<unsigned long long>(float_order_key(v)) << 32) |
         static_cast<unsigned long long>(0xFFFFFFFFu - static_cast<uint32_t>(idx));
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    unsigned long long w = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    v = w > v ? w : v;
  }
  return v;
}

// Pair epilogue for RoPE-ordered q/k rows and plain v rows, given row m's
// position and the (cos, sin) of this pair at that position (unused for v).
__device__ __forceinline__ void epi_qkv_pair_at(const GemvParams& p, int m, int pair, float v0,
                                                float v1, int pos, float2 cs) {
  const int half = p.head_dim >> 1;
  if (pos < 0 || pos >= p.T) {
    atomicOr(p.err, ERR_BAD_POS);
    return;
  }
  const int qp = p.q_dim >> 1, kp = p.kv_dim >> 1;
  if (pair < qp + kp && p.qk_raw) {  // q/k norm follows in k_qknorm
    float* r = p.qk_raw + (size_t)m * (p.q_dim + p.kv_dim) + 2 * (size_t)pair;
    r[0] = v0;
    r[1] = v1;
    return;
  }
  if (pair < qp + kp) {
    const bool isq = pair < qp;
    const int pr = isq ? pair : pair - qp;
    const int h = pr / half, i = pr - h * half;
    const float r0 = v0 * cs.x - v1 * cs.y;
    const float r1 = v1 * cs.x + v0 * cs.y;
    if (isq) {
      float* q = p.qout + (size_t)m * p.q_dim + h * p.head_dim;
      q[i] = r0;
      q[i + half] = r1;
    } else {
      uint16_t* k = p.Kc + kv_index(p.kv_tbl, p.kv_npp, p.kv_dim / p.head_dim, p.T, p.kv_seq,
                                    row_seq(p, m), h, pos, p.head_dim);
      k[i] = f32_to_bf16(r0);
      k[i + half] = f32_to_bf16(r1);
    }
  } else {
    const int d0 = 2 * (pair - qp - kp);
    const int g = d0 / p.head_dim, d = d0 - g * p.head_dim;
    uint16_t* v = p.Vc + kv_index(p.kv_tbl, p.kv_npp, p.kv_dim / p.head_dim, p.T, p.kv_seq, row_seq(p, m),
                                  g, pos, p.head_dim) + d;
    v[0] = f32_to_bf16(v0);
    v[1] = f32_to_bf16(v1);
  }
}

// (cos, sin) of a q/k pair at a position; (1, 0) for v pairs and positions
// outside the table (the caller reports those).
__device__ __forceinline__ float2 qkv_pair_rope(const GemvParams& p, int pair, int pos) {
  const int half = p.head_dim >> 1;
  const int qp = p.q_dim >> 1, kp = p.kv_dim >> 1;
  if (pair >= qp + kp || pos < 0 || pos >= p.T) return make_float2(1.f, 0.f);
  const int pr = pair < qp ? pair : pair - qp;
  return __ldg(&p.rope[(size_t)pos * half + (pr % half)]);
}

// Pair epilogue for RoPE-ordered q/k rows and plain v rows.
__device__ __forceinline__ void epi_qkv_pair(const GemvParams& p, int m, int pair, float v0,
                                             float v1) {
  const int pos = row_pos(p, m);
  epi_qkv_pair_at(p, m, pair, v0, v1, pos, qkv_pair_rope(p, pair, pos));
}

// SwiGLU output u = silu(gate) * up of row m, column i: fp32, or bf16 hi / lo
// parts when the next GEMM reads it from the tensor cores.
__device__ __forceinline__ void epi_swiglu(const GemvParams& p, int m, int i, float g, float u) {
  const float v = silu(g) * u;
  const size_t o = (size_t)m * p.ldo + i;
  if (p.out_hi) {
    const uint16_t h = f32_to_bf16(v);
    p.out_hi[o] = h;
    p.out_lo[o] = f32_to_bf16(v - bf16_to_f32(h));
  } else {
    p.out[o] = v;
  }
}

}  // namespace tf
