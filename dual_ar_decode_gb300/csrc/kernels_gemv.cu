// Weight-streaming GEMV for batch-1 decode (sm_103a).
//
// Every linear layer of the decode step is a matrix-vector product whose
// cost is reading the weight once from HBM (tuna-fish README, "Inference
// estimation": the decode step loads every parameter once per step).  The
// kernel is built around that:
//   * one CTA per SM; CTA c owns a contiguous, balanced range of rows, which
//     is one contiguous block of the row-major weight;
//   * a producer warp streams that block into a ring of shared-memory stages
//     with bulk copies on the TMA engine (cp.async.bulk + mbarrier
//     transaction counts), L2 evict-first; it starts before the previous
//     kernel finishes (programmatic dependent launch) because weights never
//     depend on activations;
//   * 8 consumer warps hold the activation slice they need in registers
//     (thread t owns 16-byte chunks t, t+256, ... of every row) and reduce
//     each row with warp shuffles; per-warp row sums meet in shared memory
//     in a fixed order, so results are bitwise deterministic;
//   * fused prologue (RMSNorm) and epilogues (residual add, SwiGLU, RoPE +
//     KV-cache append, logits + grid-wide argmax).
// FP8 weights (e4m3 with a float32 scale per row, drbaph s2-pro-fp8 model
// card, "Quantization Details") are decoded in registers and the row scale is
// applied once to the finished dot product.
#include <cuda_fp16.h>

#include <algorithm>
#include <cstdlib>

#include "common.cuh"
#include "device_once.h"
#include "epilogue.cuh"
#include "kernels.h"

namespace tf {

namespace {

constexpr int kMaxConsumerWarps = 16;
constexpr int kRowBatch = 128;  // rows reduced per epilogue round
#ifndef TF_GEMV_STAGE_BYTES
#define TF_GEMV_STAGE_BYTES (40 * 1024)
#endif
constexpr int kStageTarget = TF_GEMV_STAGE_BYTES;  // bytes of whole rows per stage
constexpr int kRingPerSm = 160 * 1024;  // ring bytes per SM, split over its CTAs
#ifndef TF_GEMV_QUAD
#define TF_GEMV_QUAD 1
#endif
// Narrow rows (few consumer warps per CTA) run four CTAs per SM, so that an
// SM still has about 20 consumer warps to hide the reduction latencies.
constexpr int kQuadMaxThreads = TF_GEMV_QUAD ? 192 : 0;

__device__ __forceinline__ void consumer_sync(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

// d = a * b + c on a pair of floats (one packed FMA, each lane rounded once).
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  uint64_t A, B, C, D;
  A = *reinterpret_cast<uint64_t*>(&a);
  B = *reinterpret_cast<uint64_t*>(&b);
  C = *reinterpret_cast<uint64_t*>(&c);
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(D) : "l"(A), "l"(B), "l"(C));
  return *reinterpret_cast<float2*>(&D);
}

// How e4m3 weight codes become numbers in the fp8 GEMV (compile-time):
//   0  cvt.rn.f16x2.e4m3x2, then f16 -> f32, packed f32 FMA (fp32 activations);
//   1  bit placement into f32: code s.eeee.mmm placed as float32 bits
//      s << 31 | eeeemmm << 20 is the code's value times 2^-120 exactly
//      (subnormal codes included); activations carry 2^60 and the row scale
//      the other 2^60, so products stay in float32's normal range;
//   2  bit placement into f16: the same code placed as f16 bits
//      s << 15 | eeeemmm << 7 is its value times 2^-8 exactly (f16 has 5
//      exponent bits, bias 15); f16 activations (more precise than the bf16
//      activations of the fp8 model card), mixed f16 x f16 + f32 FMA;
//   3  cvt.rn.f16x2.e4m3x2 (exact), f16 activations, mixed FMA.
#ifndef TF_FP8_PATH
#define TF_FP8_PATH 3
#endif
constexpr int kFp8Path = TF_FP8_PATH;
// Power of two the finished fp8 dot product is multiplied by, besides the row scale.
constexpr float kFp8Rescale = kFp8Path == 1 ? 1.152921504606846976e18f   // 2^60
                            : kFp8Path == 2 ? 256.0f : 1.0f;
// Power of two the fp8 activations are multiplied by before the dot product.
constexpr float kFp8ActScale = kFp8Path == 1 ? 1.152921504606846976e18f : 1.0f;
constexpr bool kFp8HalfAct = kFp8Path == 2 || kFp8Path == 3;   // activations as packed f16 pairs

// Weight storage per format (WT): 0 bf16, 1 e4m3 codes, 2 block-scaled 4-bit
// (a row is K/2 bytes of e2m1 codes, two per byte with the even element in
// the low nibble, then K/16 bytes of e4m3 block scales, one per 16 elements).
// A consumer chunk is EPC consecutive elements: 16 bytes of bf16 or e4m3, or
// one 16-element block of e2m1 (8 code bytes and its scale byte).
__host__ __device__ constexpr int row_bytes(int wt, int K) {
  return wt == 0 ? 2 * K : wt == 1 ? K : K / 2 + K / 16;
}
__host__ __device__ constexpr int chunk_elems(int wt) { return wt == 0 ? 8 : 16; }

// d = a * b + c with a, b the two f16 halves selected by the template and c float.
__device__ __forceinline__ float fma_h(uint32_t w2, uint32_t a2, float c, int half) {
  float d;
  if (half == 0)
    asm("{.reg .b16 wl, wh, al, ah; mov.b32 {wl, wh}, %1; mov.b32 {al, ah}, %2;"
        " fma.rn.f32.f16 %0, wl, al, %3;}" : "=f"(d) : "r"(w2), "r"(a2), "f"(c));
  else
    asm("{.reg .b16 wl, wh, al, ah; mov.b32 {wl, wh}, %1; mov.b32 {al, ah}, %2;"
        " fma.rn.f32.f16 %0, wh, ah, %3;}" : "=f"(d) : "r"(w2), "r"(a2), "f"(c));
  return d;
}

// Accumulates one 16-byte weight chunk times its activations into acc
// (two interleaved partial sums).  For fp8 with half activations, a[] holds
// the packed f16 pairs (as float bit patterns) in the order the decode below
// pairs the codes.
template <int WT, int EPC>
__device__ __forceinline__ float2 chunk_fma(const uint4 w, const float* a, float2 acc) {
  const uint32_t v[4] = {w.x, w.y, w.z, w.w};
  if constexpr (WT == 0) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      acc = fma2(make_float2(bf16_lo(v[i]), bf16_hi(v[i])), make_float2(a[2 * i], a[2 * i + 1]), acc);
  } else if constexpr (kFp8Path == 0) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 lo = e4m3x2_to_f32x2(static_cast<uint16_t>(v[i] & 0xFFFFu));
      const float2 hi = e4m3x2_to_f32x2(static_cast<uint16_t>(v[i] >> 16));
      acc = fma2(lo, make_float2(a[4 * i], a[4 * i + 1]), acc);
      acc = fma2(hi, make_float2(a[4 * i + 2], a[4 * i + 3]), acc);
    }
  } else if constexpr (kFp8Path == 1) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      // byte b of v at bits 31..24 (zeros below), then (x >>arith 4) & 0x87F00000
      float f[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        uint32_t x;
        asm("prmt.b32 %0, %1, 0, %2;" : "=r"(x) : "r"(v[i]), "r"(0x0444u | (static_cast<uint32_t>(b) << 12)));
        f[b] = __uint_as_float(static_cast<uint32_t>(static_cast<int32_t>(x) >> 4) & 0x87F00000u);
      }
      acc = fma2(make_float2(f[0], f[1]), make_float2(a[4 * i], a[4 * i + 1]), acc);
      acc = fma2(make_float2(f[2], f[3]), make_float2(a[4 * i + 2], a[4 * i + 3]), acc);
    }
  } else if constexpr (kFp8Path == 2) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      // lanes (b0, b2) and (b1, b3) of v as f16 bit patterns
      const uint32_t t = v[i] << 8;
      const uint32_t p02 = (t & 0x80008000u) | ((t >> 1) & 0x3F803F80u);
      const uint32_t p13 = (v[i] & 0x80008000u) | ((v[i] >> 1) & 0x3F803F80u);
      const uint32_t a02 = __float_as_uint(a[2 * i]), a13 = __float_as_uint(a[2 * i + 1]);
      acc.x = fma_h(p02, a02, acc.x, 0);
      acc.y = fma_h(p13, a13, acc.y, 0);
      acc.x = fma_h(p02, a02, acc.x, 1);
      acc.y = fma_h(p13, a13, acc.y, 1);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t h01, h23;
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h01) : "h"(static_cast<uint16_t>(v[i] & 0xFFFFu)));
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h23) : "h"(static_cast<uint16_t>(v[i] >> 16)));
      const uint32_t a01 = __float_as_uint(a[2 * i]), a23 = __float_as_uint(a[2 * i + 1]);
      acc.x = fma_h(h01, a01, acc.x, 0);
      acc.y = fma_h(h01, a01, acc.y, 1);
      acc.x = fma_h(h23, a23, acc.x, 0);
      acc.y = fma_h(h23, a23, acc.y, 1);
    }
  }
  return acc;
}

// One 16-element block of e2m1 codes (w: 8 bytes, element 2i in the low
// nibble of byte i) with its e4m3 block scale sb: the codes are converted
// exactly to f16 pairs, multiplied by the f16 activation pairs a[0..7] with
// float32 accumulation, and the block sum is scaled by the block scale
// (placed as float32 bits: value x 2^-120, times 2^120, both exact; block
// scales are never negative) before it joins acc.
__device__ __forceinline__ float e2m1_block_fma(const uint2 w, uint32_t sb, const float* a, float acc) {
  const uint32_t v[2] = {w.x, w.y};
  float s0 = 0.f, s1 = 0.f;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    uint32_t h[4];  // the word's four code pairs as f16 pairs
    asm("{.reg .b8 b0, b1, b2, b3; mov.b32 {b0, b1, b2, b3}, %4;"
        " cvt.rn.f16x2.e2m1x2 %0, b0; cvt.rn.f16x2.e2m1x2 %1, b1;"
        " cvt.rn.f16x2.e2m1x2 %2, b2; cvt.rn.f16x2.e2m1x2 %3, b3;}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3]) : "r"(v[i]));
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint32_t ap = __float_as_uint(a[4 * i + b]);
      s0 = fma_h(h[b], ap, s0, 0);
      s1 = fma_h(h[b], ap, s1, 1);
    }
  }
  const float scale = __uint_as_float((sb & 0x7Fu) << 20) * 1.329227995784915873e36f;  // 2^120
  return fmaf(s0 + s1, scale, acc);
}

// f16 bits of x, round to nearest even (finite activations).
__device__ __forceinline__ uint32_t f16_bits(float x) {
  return static_cast<uint32_t>(__half_as_ushort(__float2half_rn(x)));
}

// Rewrites one chunk's EPC fp32 activations for the fp8 decode in use: the
// 2^60 pre-scale (bit placement into f32), or packed f16 pairs in a[0..7] in
// the pairing chunk_fma expects (f16 paths).
template <int WT, int EPC>
__device__ __forceinline__ void fp8_prepare(float* a) {
  if constexpr (WT == 1 && kFp8Path == 1) {
#pragma unroll
    for (int e = 0; e < EPC; ++e) a[e] *= kFp8ActScale;
  } else if constexpr ((WT == 1 && kFp8HalfAct) || WT == 2) {
    float pk[EPC / 2];
#pragma unroll
    for (int i = 0; i < EPC / 4; ++i) {
      if constexpr (WT == 1 && kFp8Path == 2) {   // (a0, a2), (a1, a3) of each 4 codes
        pk[2 * i] = __uint_as_float(f16_bits(a[4 * i]) | (f16_bits(a[4 * i + 2]) << 16));
        pk[2 * i + 1] = __uint_as_float(f16_bits(a[4 * i + 1]) | (f16_bits(a[4 * i + 3]) << 16));
      } else {                         // (a0, a1), (a2, a3)
        pk[2 * i] = __uint_as_float(f16_bits(a[4 * i]) | (f16_bits(a[4 * i + 1]) << 16));
        pk[2 * i + 1] = __uint_as_float(f16_bits(a[4 * i + 2]) | (f16_bits(a[4 * i + 3]) << 16));
      }
    }
#pragma unroll
    for (int i = 0; i < EPC / 2; ++i) a[i] = pk[i];
  }
}

// Sums V values over the 32 lanes of a warp with a transposing butterfly:
// log2(V) halving exchanges, then 5 - log2(V) plain ones.  Afterwards lane l
// holds the warp total of value l >> (5 - log2 V).
template <int V>
__device__ __forceinline__ float warp_reduce_many(float (&v)[V], int lane) {
  int n = V;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    if (n > 1) {
      const bool up = lane & off;
      const int h = n >> 1;
#pragma unroll
      for (int k = 0; k < V / 2; ++k) {
        if (k < h) {
          const float send = up ? v[k] : v[k + h];
          const float keep = up ? v[k + h] : v[k];
          v[k] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, off);
        }
      }
      n = h;
    } else {
      v[0] += __shfl_xor_sync(0xFFFFFFFFu, v[0], off);
    }
  }
  return v[0];
}

template <int WT, int M, int J>
__global__ void __launch_bounds__(kMaxConsumerWarps * 32 + 32, 1) k_gemv(const GemvParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int EPC = chunk_elems(WT);  // elements per chunk
  constexpr int R = M == 1 ? 8 : 4;     // rows reduced together
  constexpr int V = R * M;              // values per butterfly (8)
  constexpr int LOGV = 3;
  const int NT = static_cast<int>(blockDim.x) - 32;  // consumer threads
  const int NW = NT >> 5;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, c = blockIdx.x;
  const int u0 = (int)((long long)p.units * c / G);
  const int u1 = (int)((long long)p.units * (c + 1) / G);
  const int r0 = u0 * p.unit;
  const int nrows = (u1 - u0) * p.unit;
  const uint32_t rowbytes = static_cast<uint32_t>(row_bytes(WT, p.K));
  const int nch = p.K / EPC;

  uint8_t* ring = smem;
  float* red = reinterpret_cast<float*>(smem + (size_t)p.nst * p.stb);  // [kRowBatch][NW][M]
  uint64_t* full = reinterpret_cast<uint64_t*>(red + kRowBatch * kMaxConsumerWarps * M);
  uint64_t* empty = full + p.nst;
  float* misc = reinterpret_cast<float*>(empty + p.nst);  // [16][M]
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(misc + kMaxConsumerWarps * M);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(keys + kMaxConsumerWarps);

  pdl_launch_dependents();
  if (tid == 0) {
    for (int s = 0; s < p.nst; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NW);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == NW) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int s = 0;
      for (int b0 = 0; b0 < nrows && !*abort_flag; b0 += kRowBatch) {
        const int nb = min(kRowBatch, nrows - b0);
        for (int i0 = 0; i0 < nb; i0 += p.rs) {
          const int n = min(p.rs, nb - i0);
          const int slot = s % p.nst;
          if (s >= p.nst && !mbar_wait(&empty[slot], ((s / p.nst) & 1) ^ 1, p.err)) {
            *abort_flag = 1;
            break;
          }
          const uint32_t bytes = static_cast<uint32_t>(n) * rowbytes;
          mbar_arrive_expect_tx(&full[slot], bytes);
          const bool skip = p.test_skip_copy && c == 0 && b0 + i0 + n >= nrows;  // failure test
          if (!skip)
            bulk_g2s(ring + (size_t)slot * p.stb, p.W + (size_t)(r0 + b0 + i0) * rowbytes, bytes,
                     &full[slot], pol);
          ++s;
        }
      }
      // Hint L2 with the start of the next GEMV's matching row block.
      if (p.pf_w && !*abort_flag) {
        for (int cn = c; cn < p.pf_grid; cn += G) {
          const int v0 = (int)((long long)p.pf_units * cn / p.pf_grid);
          const int v1 = (int)((long long)p.pf_units * (cn + 1) / p.pf_grid);
          const size_t start = (size_t)v0 * p.pf_unit * p.pf_rowbytes;
          size_t len = (size_t)(v1 - v0) * p.pf_unit * p.pf_rowbytes;
          if (len > (size_t)p.pf_bytes) len = (size_t)p.pf_bytes;
          for (size_t o = 0; o + 16 <= len; o += 32768) {
            const uint32_t n = static_cast<uint32_t>(std::min<size_t>(32768, len - o) & ~size_t(15));
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.pf_w + start + o), "r"(n)
                         : "memory");
          }
        }
      }
      // Hint L2 with this CTA's share of the cached K and V rows the
      // attention after this QKV GEMV reads (they do not depend on it).
      if (p.kv_pf && !*abort_flag) {
        const int pos = row_pos(p, 0);
        if (pos >= 32 && pos <= p.T) {
          const int hkv = p.kv_dim / p.head_dim;
          const size_t region = (size_t)pos * p.head_dim * 2;  // one head's cached rows, bytes
          const size_t total = 2 * (size_t)hkv * region;
          const size_t b0 = (total * c / G) & ~size_t(255);
          const size_t b1 = c + 1 == G ? total : (total * (c + 1) / G) & ~size_t(255);
          const size_t seq_off = (size_t)row_seq(p, 0) * (size_t)p.kv_seq;
          for (size_t b = b0; b < b1;) {
            const size_t r = b / region, off = b - r * region;
            const size_t n = std::min(b1 - b, region - off);
            const uint16_t* head = (r < (size_t)hkv ? p.Kc : p.Vc) + seq_off +
                                   (r % hkv) * (size_t)p.T * p.head_dim;
            const uint8_t* src = reinterpret_cast<const uint8_t*>(head) + off;
            for (size_t o = 0; o < n; o += 32768) {
              const uint32_t len = static_cast<uint32_t>(std::min<size_t>(32768, n - o));
              asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src + o), "r"(len) : "memory");
            }
            b += n;
          }
        }
      }
      // Drain: the last (up to nst) issued copies may still be in flight.
      for (int t = max(0, s - p.nst); t < s; ++t)
        mbar_wait(&full[t % p.nst], (t / p.nst) & 1, p.err);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  pdl_wait();  // activations come from the previous kernel

  float a[M][J][EPC];
#pragma unroll
  for (int m = 0; m < M; ++m) {
    const float* xm = p.x + (size_t)m * p.ldx;
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int ch = tid + j * NT;
      if (ch < nch) {
        const float4* src = reinterpret_cast<const float4*>(xm + ch * EPC);
#pragma unroll
        for (int q = 0; q < EPC / 4; ++q) {
          const float4 v = src[q];
          a[m][j][4 * q] = v.x;
          a[m][j][4 * q + 1] = v.y;
          a[m][j][4 * q + 2] = v.z;
          a[m][j][4 * q + 3] = v.w;
        }
      } else {
#pragma unroll
        for (int e = 0; e < EPC; ++e) a[m][j][e] = 0.f;
      }
    }
  }
  // Everything else the consumers will read from global memory is loaded
  // now, in one round trip with the activations: the RMSNorm weight of their
  // chunks, and the epilogue inputs of their first row (residual, or the
  // position and RoPE factors of a q/k pair).
  // (The RMSNorm inputs are hidden-size rows, J <= 2; wider variants keep
  // their registers for the activations.)
  constexpr int NWU = WT ? 2 : 1;  // 16-byte norm-weight pieces per chunk
  constexpr bool kNwRegs = J <= 2;
  uint4 nwc[kNwRegs ? J : 1][NWU];
  if (kNwRegs && p.pro == PRO_NORM) {
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int ch = tid + j * NT;
#pragma unroll
      for (int u = 0; u < NWU; ++u)
        nwc[j][u] = ch < nch ? __ldg(reinterpret_cast<const uint4*>(p.nw + ch * EPC) + u)
                             : make_uint4(0u, 0u, 0u, 0u);
    }
  }
  const int nb0 = min(kRowBatch, nrows);
  float xr0[M];
  float2 cs0[M];
  int pos0[M];
#pragma unroll
  for (int m = 0; m < M; ++m) {
    xr0[m] = 0.f;
    cs0[m] = make_float2(1.f, 0.f);
    pos0[m] = 0;
  }
  if (p.epi == EPI_QKV && tid < (nb0 >> 1)) {
    const int pair = (r0 >> 1) + tid;
#pragma unroll
    for (int m = 0; m < M; ++m) {
      pos0[m] = row_pos(p, m);
      cs0[m] = qkv_pair_rope(p, pair, pos0[m]);
    }
  } else if (p.epi == EPI_RESID && tid < nb0) {
#pragma unroll
    for (int m = 0; m < M; ++m) xr0[m] = p.out[(size_t)m * p.ldo + r0 + tid];
  }
  if (p.pro == PRO_NORM) {
#pragma unroll
    for (int m = 0; m < M; ++m) {
      float ss = 0.f;
#pragma unroll
      for (int j = 0; j < J; ++j)
#pragma unroll
        for (int e = 0; e < EPC; ++e) ss = fmaf(a[m][j][e], a[m][j][e], ss);
      ss = warp_sum(ss);
      if (lane == 0) misc[warp * M + m] = ss;
    }
    consumer_sync(NT);
#pragma unroll
    for (int m = 0; m < M; ++m) {
      float ss = 0.f;
      for (int w = 0; w < NW; ++w) ss += misc[w * M + m];
      const float rstd = 1.0f / sqrtf(ss / static_cast<float>(p.K) + p.eps);
#pragma unroll
      for (int j = 0; j < J; ++j) {
        if constexpr (kNwRegs) {
          const uint32_t* wv = reinterpret_cast<const uint32_t*>(&nwc[j][0]);
#pragma unroll
          for (int e = 0; e < EPC; e += 2) {
            a[m][j][e] = a[m][j][e] * rstd * bf16_lo(wv[e >> 1]);
            a[m][j][e + 1] = a[m][j][e + 1] * rstd * bf16_hi(wv[e >> 1]);
          }
        } else {
          const int ch = tid + j * NT;
          if (ch < nch) {
#pragma unroll
            for (int e = 0; e < EPC; ++e)
              a[m][j][e] = a[m][j][e] * rstd * bf16_to_f32(__ldg(&p.nw[ch * EPC + e]));
          }
        }
      }
    }
  }

  if constexpr (WT >= 1) {
#pragma unroll
    for (int m = 0; m < M; ++m)
#pragma unroll
      for (int j = 0; j < J; ++j) fp8_prepare<WT, EPC>(a[m][j]);
  }

  unsigned long long best = 0ull;  // EPI_LOGITS: best (value, lowest index) key seen
  int s = 0;
  for (int b0 = 0; b0 < nrows; b0 += kRowBatch) {
    const int nb = min(kRowBatch, nrows - b0);
    for (int i0 = 0; i0 < nb; i0 += p.rs) {
      const int n = min(p.rs, nb - i0);
      const int slot = s % p.nst;
      if (!*abort_flag && !mbar_wait(&full[slot], (s / p.nst) & 1, p.err)) *abort_flag = 1;
      const uint8_t* st = ring + (size_t)slot * p.stb;
      for (int i = 0; i < n; i += R) {
        float v[V];
#pragma unroll
        for (int r = 0; r < R; ++r) {
          float2 acc[M];
#pragma unroll
          for (int m = 0; m < M; ++m) acc[m] = make_float2(0.f, 0.f);
          if (i + r < n) {
            const uint8_t* rowp = st + (size_t)(i + r) * rowbytes;
#pragma unroll
            for (int j = 0; j < J; ++j) {
              const int ch = tid + j * NT;
              if (ch < nch) {
                if constexpr (WT == 2) {
                  const uint2 w = reinterpret_cast<const uint2*>(rowp)[ch];
                  const uint32_t sb = rowp[(p.K >> 1) + ch];
#pragma unroll
                  for (int m = 0; m < M; ++m) acc[m].x = e2m1_block_fma(w, sb, a[m][j], acc[m].x);
                } else {
                  const uint4 w = reinterpret_cast<const uint4*>(rowp)[ch];
#pragma unroll
                  for (int m = 0; m < M; ++m) acc[m] = chunk_fma<WT, EPC>(w, a[m][j], acc[m]);
                }
              }
            }
          }
#pragma unroll
          for (int m = 0; m < M; ++m) v[r * M + m] = acc[m].x + acc[m].y;
        }
        const float tot = warp_reduce_many<V>(v, lane);
        if ((lane & ((32 >> LOGV) - 1)) == 0) {
          const int idx = lane >> (5 - LOGV);
          const int r = idx / M, m = idx - r * M;
          if (i + r < n) red[((i0 + i + r) * NW + warp) * M + m] = tot;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
      ++s;
    }
    consumer_sync(NT);

    // ---------------------------------------------------------- epilogue
    if (p.unit == 2) {
      for (int pi = tid; pi < (nb >> 1); pi += NT) {
        const int rg = r0 + b0 + 2 * pi;
#pragma unroll
        for (int m = 0; m < M; ++m) {
          float v0 = 0.f, v1 = 0.f;
          for (int w = 0; w < NW; ++w) {
            v0 += red[((2 * pi) * NW + w) * M + m];
            v1 += red[((2 * pi + 1) * NW + w) * M + m];
          }
          if (p.scale) {
            v0 *= __ldg(&p.scale[rg]) * (WT == 1 ? kFp8Rescale : 1.0f);
            v1 *= __ldg(&p.scale[rg + 1]) * (WT == 1 ? kFp8Rescale : 1.0f);
          }
          if (p.epi == EPI_SWIGLU) {
            epi_swiglu(p, m, rg >> 1, v0, v1);
          } else if (b0 == 0 && pi == tid) {  // EPI_QKV, inputs loaded up front
            epi_qkv_pair_at(p, m, rg >> 1, v0, v1, pos0[m], cs0[m]);
          } else {
            epi_qkv_pair(p, m, rg >> 1, v0, v1);
          }
        }
      }
    } else {
      for (int ri = tid; ri < nb; ri += NT) {
        const int rg = r0 + b0 + ri;
#pragma unroll
        for (int m = 0; m < M; ++m) {
          float v = 0.f;
          for (int w = 0; w < NW; ++w) v += red[(ri * NW + w) * M + m];
          if (p.scale) v *= __ldg(&p.scale[rg]) * (WT == 1 ? kFp8Rescale : 1.0f);
          float* o = p.out + (size_t)m * p.ldo + rg;
          if (p.epi == EPI_RESID) {
            *o = ((b0 == 0 && ri == tid) ? xr0[m] : *o) + v;
          } else {
            *o = v;
            if (p.epi == EPI_LOGITS) {
              if (v != v) atomicOr(p.err, ERR_NAN);
              const unsigned long long k = pack_key(v, rg);
              best = k > best ? k : best;
            }
          }
        }
      }
    }
    consumer_sync(NT);
  }

  if (p.epi == EPI_LOGITS && p.select) {
    best = warp_max_u64(best);
    if (lane == 0) keys[warp] = best;
    consumer_sync(NT);
    if (tid == 0) {
      unsigned long long b = 0ull;
      for (int w = 0; w < NW; ++w) b = keys[w] > b ? keys[w] : b;
      if (b) atomicMax(p.best, b);
      __threadfence();
      const uint32_t t = atomicAdd(p.ticket, 1u);
      if (t == static_cast<uint32_t>(G) - 1u) {
        __threadfence();
        const unsigned long long fin = atomicExch(p.best, 0ull);
        const int idx = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(fin & 0xFFFFFFFFull));
        *p.sel = idx;
        *p.fb = (p.forced_on && *p.forced_on) ? *p.forced : idx;
        *p.ticket = 0u;
      }
    }
  }
}

template <int WT, int M, int J>
cudaError_t launch_t(const GemvParams& p, int nt, int grid, bool pdl, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(nt + 32);
  cfg.dynamicSmemBytes = gemv_smem_bytes(p, M);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_gemv<WT, M, J>, p);
}

template <int WT, int M>
cudaError_t launch_j(const GemvParams& p, int J, int nt, int grid, bool pdl, cudaStream_t s) {
  switch (J) {
    case 1: return launch_t<WT, M, 1>(p, nt, grid, pdl, s);
    case 2: return launch_t<WT, M, 2>(p, nt, grid, pdl, s);
    case 3: return launch_t<WT, M, 3>(p, nt, grid, pdl, s);
    case 4: return launch_t<WT, M, 4>(p, nt, grid, pdl, s);
    case 5: return launch_t<WT, M, 5>(p, nt, grid, pdl, s);
    default: return cudaErrorInvalidValue;
  }
}

template <typename K>
cudaError_t set_smem(K kernel) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  if (e) return e;
  // Every decode kernel asks for the full shared-memory carveout, so that a
  // CTA of the next kernel (launched early by PDL) can share the SM.
  return cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                              cudaSharedmemCarveoutMaxShared);
}

template <int WT, int M>
cudaError_t set_attr_m() {
  cudaError_t e;
  if ((e = set_smem(k_gemv<WT, M, 1>))) return e;
  if ((e = set_smem(k_gemv<WT, M, 2>))) return e;
  if ((e = set_smem(k_gemv<WT, M, 3>))) return e;
  if ((e = set_smem(k_gemv<WT, M, 4>))) return e;
  return set_smem(k_gemv<WT, M, 5>);
}

}  // namespace

size_t gemv_smem_bytes(const GemvParams& p, int M) {
  size_t b = (size_t)p.nst * p.stb;
  b += (size_t)kRowBatch * kMaxConsumerWarps * M * sizeof(float);
  b += 2 * (size_t)p.nst * sizeof(uint64_t);
  b += (size_t)kMaxConsumerWarps * M * sizeof(float) + kMaxConsumerWarps * sizeof(unsigned long long) + 16;
  return b;
}

namespace {

template <int WT, int M>
const void* kernel_j(int J) {
  switch (J) {
    case 1: return (const void*)k_gemv<WT, M, 1>;
    case 2: return (const void*)k_gemv<WT, M, 2>;
    case 3: return (const void*)k_gemv<WT, M, 3>;
    case 4: return (const void*)k_gemv<WT, M, 4>;
    default: return (const void*)k_gemv<WT, M, 5>;
  }
}

const void* kernel_for(int wt, int M, int J) {
  if (wt == 0) return M == 1 ? kernel_j<0, 1>(J) : kernel_j<0, 2>(J);
  if (wt == 1) return M == 1 ? kernel_j<1, 1>(J) : kernel_j<1, 2>(J);
  return M == 1 ? kernel_j<2, 1>(J) : kernel_j<2, 2>(J);
}

void set_ring(GemvParams& p, int rowbytes, int ring) {
  const int target = std::min(kStageTarget, ring / 2);
  p.rs = rowbytes >= target ? 1 : target / rowbytes;
  p.stb = ((p.rs * rowbytes + 127) / 128) * 128;
  p.nst = std::max(2, std::min(16, ring / p.stb));
}

}  // namespace

int gemv_grid(const GemvParams& p, int num_sms) {
  return std::min(num_sms * p.ctas_per_sm, p.units);
}

// Splits of a row's chunks over consumer threads, most even first (multiples
// of 32 threads, at most 5 chunks each); the plan takes the first split that
// lets two CTAs share an SM (registers and shared memory), else the most even
// one with a single CTA: with only one CTA's consumer warps per SM the row
// reductions are latency-bound.
void gemv_plan(GemvParams& p, int wt, int num_sms, int M) {
  (void)num_sms;
  p.unit = (p.epi == EPI_SWIGLU || p.epi == EPI_QKV) ? 2 : 1;
  p.units = p.N / p.unit;
  const int rowbytes = row_bytes(wt, p.K);
  const int nch = p.K / chunk_elems(wt);
  struct Split {
    int nt, J;
    double eff;
  };
  Split cand[kMaxConsumerWarps];
  int nc = 0;
  for (int w = 1; w <= kMaxConsumerWarps; ++w) {
    const int nt = 32 * w, J = (nch + nt - 1) / nt;
    if (J > 5) continue;
    cand[nc++] = {nt, J, static_cast<double>(nch) / (static_cast<double>(nt) * J)};
  }
  std::stable_sort(cand, cand + nc, [](const Split& a, const Split& b) {
    if (a.eff > b.eff + 1e-9) return true;
    if (b.eff > a.eff + 1e-9) return false;
    return std::abs(a.nt - 320) < std::abs(b.nt - 320);
  });
  for (int i = 0; i < nc; ++i) {
    if (cand[i].eff < 0.9) break;  // not worth a second CTA
    for (int ctas = 4; ctas >= 2; ctas -= 2) {
      if (ctas == 4 && cand[i].nt + 32 > kQuadMaxThreads) continue;
      set_ring(p, rowbytes, kRingPerSm / ctas);
      int n = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
              &n, kernel_for(wt, M, cand[i].J), cand[i].nt + 32, gemv_smem_bytes(p, M)) ==
              cudaSuccess &&
          n >= ctas) {
        p.ctas_per_sm = ctas;
        p.nt = cand[i].nt;
        p.J = cand[i].J;
        return;
      }
      (void)cudaGetLastError();
    }
  }
  p.ctas_per_sm = 1;
  p.nt = nc ? cand[0].nt : 32;
  p.J = nc ? cand[0].J : 5;
  set_ring(p, rowbytes, kRingPerSm);
}

cudaError_t launch_gemv(const GemvParams& p, int wt, int M, int grid, bool pdl, cudaStream_t s) {
  const int J = p.J, nt = p.nt;
  if (J < 1 || J > 5 || M < 1 || M > 2) return cudaErrorInvalidValue;
  if (wt == 0) return M == 1 ? launch_j<0, 1>(p, J, nt, grid, pdl, s) : launch_j<0, 2>(p, J, nt, grid, pdl, s);
  if (wt == 1) return M == 1 ? launch_j<1, 1>(p, J, nt, grid, pdl, s) : launch_j<1, 2>(p, J, nt, grid, pdl, s);
  return M == 1 ? launch_j<2, 1>(p, J, nt, grid, pdl, s) : launch_j<2, 2>(p, J, nt, grid, pdl, s);
}

cudaError_t gemv_set_attributes() {
  static DeviceOnce once;
  return device_once(once, [] {
    cudaError_t e;
    if ((e = set_attr_m<0, 1>())) return e;
    if ((e = set_attr_m<0, 2>())) return e;
    if ((e = set_attr_m<1, 1>())) return e;
    if ((e = set_attr_m<1, 2>())) return e;
    if ((e = set_attr_m<2, 1>())) return e;
    return set_attr_m<2, 2>();
  });
}

}  // namespace tf
