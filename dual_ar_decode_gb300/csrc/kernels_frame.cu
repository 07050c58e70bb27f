// Persistent decode-frame kernel (sm_103a).
//
// One cooperative launch runs whole decode frames (tuna-fish README,
// "Inference estimation": a decode step is one slowAR token plus nine fastAR
// passes, bound by streaming every weight once).  The frame is a program of
// ops (GEMV with fused prologue/epilogue, attention, selection, bookkeeping)
// separated by grid barriers.  Each CTA (one per SM) has
//   * a producer warp that walks the program and streams the CTA's row slice
//     of every GEMV weight, op after op and frame after frame, into a ring
//     of shared-memory slots with bulk copies (TMA engine, mbarrier
//     transaction counts, L2 evict-first).  It never waits for activations,
//     only for free slots, so HBM keeps streaming while the consumers sit in
//     a grid barrier;
//   * ten consumer warps that execute the ops: GEMV rows against activations
//     held in registers (row sums by a transposing warp butterfly, per-warp
//     sums combined in a fixed order, so results are deterministic), the
//     split-key GQA attention, and the selection.
// Grid barriers are a monotonic counter in global memory (release add /
// acquire poll); every wait is bounded by %globaltimer and raises an error
// bit instead of hanging.  Activations written by other CTAs are read with
// L2-coherent loads (ld.global.cg).
#include <cuda_fp16.h>

#include <algorithm>

#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.h"

namespace tf {

namespace {

constexpr int kCW = kFrameConsumerWarps;
constexpr int kCT = kCW * 32;
constexpr int kThreads = kCT + 32;
constexpr int kRowBatch = 128;

__device__ __forceinline__ void csync() { asm volatile("bar.sync 1, %0;" ::"n"(kCT) : "memory"); }

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_add(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  uint64_t A = *reinterpret_cast<uint64_t*>(&a), B = *reinterpret_cast<uint64_t*>(&b),
           C = *reinterpret_cast<uint64_t*>(&c), D;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(D) : "l"(A), "l"(B), "l"(C));
  return *reinterpret_cast<float2*>(&D);
}

template <int WT>
__device__ __forceinline__ float2 chunk_fma(const uint4 w, const float* a, float2 acc) {
  const uint32_t v[4] = {w.x, w.y, w.z, w.w};
  if constexpr (WT == 0) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      acc = fma2(make_float2(bf16_lo(v[i]), bf16_hi(v[i])), make_float2(a[2 * i], a[2 * i + 1]), acc);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 lo = e4m3x2_to_f32x2(static_cast<uint16_t>(v[i] & 0xFFFFu));
      const float2 hi = e4m3x2_to_f32x2(static_cast<uint16_t>(v[i] >> 16));
      acc = fma2(lo, make_float2(a[4 * i], a[4 * i + 1]), acc);
      acc = fma2(hi, make_float2(a[4 * i + 2], a[4 * i + 3]), acc);
    }
  }
  return acc;
}

// Transposing butterfly: after it, lane l holds the warp total of value
// l >> (5 - log2 V).
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

struct Shared {
  uint8_t* ring;
  uint8_t* un;            // union scratch (GEMV reduction / attention merge / select)
  uint64_t* full;
  uint64_t* empty;
  float* misc;            // [16][2]
  unsigned long long* keys;  // [16]
  volatile uint32_t* abort_flag;
  int slots;
};

__device__ __forceinline__ void op_rows(const FrameOp& op, int c, int G, int* r0, int* nrows) {
  const int units = op.N / op.unit;
  const int u0 = (int)((long long)units * c / G);
  const int u1 = (int)((long long)units * (c + 1) / G);
  *r0 = u0 * op.unit;
  *nrows = (u1 - u0) * op.unit;
}

__device__ __forceinline__ int op_pos(const FrameParams& P, const FrameOp& op, int m) {
  return (op.use_pos ? *reinterpret_cast<volatile int32_t*>(P.pos) : op.pos_fixed) + m;
}

// RoPE-pair / V-pair epilogue of the fused QKV op.
__device__ __forceinline__ void qkv_pair(const FrameParams& P, const FrameOp& op, int m, int pair,
                                         float v0, float v1) {
  const int half = P.D >> 1;
  const int pos = op_pos(P, op, m);
  if (pos < 0 || pos >= P.T) {
    atomicOr(P.err, ERR_BAD_POS);
    return;
  }
  const int qp = P.q_dim >> 1, kp = P.kv_dim >> 1;
  if (pair < qp + kp) {
    const bool isq = pair < qp;
    const int pr = isq ? pair : pair - qp;
    const int h = pr / half, i = pr - h * half;
    const float2 cs = __ldg(&P.rope[(size_t)pos * half + i]);
    const float r0 = v0 * cs.x - v1 * cs.y;
    const float r1 = v1 * cs.x + v0 * cs.y;
    if (isq) {
      float* q = op.out + (size_t)m * P.q_dim + h * P.D;
      q[i] = r0;
      q[i + half] = r1;
    } else {
      uint16_t* k = op.Kc + ((size_t)h * P.T + pos) * P.D;
      k[i] = f32_to_bf16(r0);
      k[i + half] = f32_to_bf16(r1);
    }
  } else {
    const int d0 = 2 * (pair - qp - kp);
    const int g = d0 / P.D, d = d0 - g * P.D;
    uint16_t* v = op.Vc + ((size_t)g * P.T + pos) * P.D + d;
    v[0] = f32_to_bf16(v0);
    v[1] = f32_to_bf16(v1);
  }
}

// ------------------------------------------------------------------ GEMV op
// JM = chunks per consumer thread, a compile-time count so that the hot loop
// carries no predicated-off chunk slots.
template <int WT, int M, int JM>
__device__ __noinline__ void gemv_op(const FrameParams& P, const FrameOp& op, Shared& S, int& s_ctr) {
  constexpr int EPC = WT ? 16 : 8;
  constexpr int R = M == 1 ? 8 : 4;
  constexpr int V = R * M;  // 8 values per butterfly
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x;
  int r0, nrows;
  op_rows(op, blockIdx.x, G, &r0, &nrows);
  const uint32_t rowbytes = static_cast<uint32_t>(op.K) * (WT ? 1u : 2u);
  const int nch = static_cast<int>(rowbytes >> 4);
  const int nt = op.nt;
  const bool active = tid < nt;

  // ---- activation rows into registers
  float a[M][JM][EPC];
#pragma unroll
  for (int m = 0; m < M; ++m)
#pragma unroll
    for (int j = 0; j < JM; ++j)
#pragma unroll
      for (int e = 0; e < EPC; ++e) a[m][j][e] = 0.f;

  int id = 0;
  if (op.src != SRC_X) {
    id = *reinterpret_cast<const volatile int32_t*>(op.id_ptr);
    if (id < 0 || id >= op.table_rows) {
      if (tid == 0) atomicOr(P.err, ERR_BAD_ID);
      id = 0;
    }
  }
#pragma unroll
  for (int m = 0; m < M; ++m) {
#pragma unroll
    for (int j = 0; j < JM; ++j) {
      const int ch = tid + j * nt;
      if (!active || ch >= nch) continue;
      const bool from_table = (op.src == SRC_EMBED && m == 0) || (op.src == SRC_FAST1 && m == 1);
      if (from_table) {
        const uint16_t* row = op.table + (size_t)(op.row_base + id) * op.K + ch * EPC;
#pragma unroll
        for (int q = 0; q < EPC / 8; ++q) {
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(row) + q);
          const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            a[m][j][8 * q + 2 * i] = bf16_lo(u[i]);
            a[m][j][8 * q + 2 * i + 1] = bf16_hi(u[i]);
          }
        }
      } else {
        const float* xm = (op.src == SRC_FAST1) ? op.xs : op.x + (size_t)m * op.ldx;
        const float4* src = reinterpret_cast<const float4*>(xm + ch * EPC);
#pragma unroll
        for (int q = 0; q < EPC / 4; ++q) {
          const float4 v = __ldcg(src + q);
          a[m][j][4 * q] = v.x;
          a[m][j][4 * q + 1] = v.y;
          a[m][j][4 * q + 2] = v.z;
          a[m][j][4 * q + 3] = v.w;
        }
      }
    }
  }
  auto block_sumsq = [&](int m_only, float* out_ss) {
    // sum of squares of row(s); m_only < 0: all rows
#pragma unroll
    for (int m = 0; m < M; ++m) {
      float ss = 0.f;
      if (m_only < 0 || m_only == m) {
#pragma unroll
        for (int j = 0; j < JM; ++j)
#pragma unroll
          for (int e = 0; e < EPC; ++e) ss = fmaf(a[m][j][e], a[m][j][e], ss);
      }
      ss = warp_sum(ss);
      if (lane == 0) S.misc[warp * 2 + m] = ss;
    }
    csync();
#pragma unroll
    for (int m = 0; m < M; ++m) {
      float t = 0.f;
      for (int w = 0; w < kCW; ++w) t += S.misc[w * 2 + m];
      out_ss[m] = t;
    }
    csync();
  };
  if (op.src == SRC_FAST1) {
    // row 0 = RMSNorm(slow residual) * final-norm weight (the semantic head's input)
    float ss[M];
    block_sumsq(0, ss);
    const float rstd = 1.0f / sqrtf(ss[0] / static_cast<float>(op.K) + P.eps);
#pragma unroll
    for (int j = 0; j < JM; ++j) {
      const int ch = tid + j * nt;
      if (!active || ch >= nch) continue;
#pragma unroll
      for (int e = 0; e < EPC; ++e)
        a[0][j][e] = a[0][j][e] * rstd * bf16_to_f32(__ldg(&op.nw_src[ch * EPC + e]));
    }
  }
  if (op.src != SRC_X && blockIdx.x == 0) {
    // CTA 0 publishes the built rows as the residual of the pass.
#pragma unroll
    for (int m = 0; m < M; ++m)
#pragma unroll
      for (int j = 0; j < JM; ++j) {
        const int ch = tid + j * nt;
        if (!active || ch >= nch) continue;
#pragma unroll
        for (int e = 0; e < EPC; ++e) op.xres[(size_t)m * op.K + ch * EPC + e] = a[m][j][e];
      }
  }
  if (op.pro == PRO_NORM) {
    float ss[M];
    block_sumsq(-1, ss);
#pragma unroll
    for (int m = 0; m < M; ++m) {
      const float rstd = 1.0f / sqrtf(ss[m] / static_cast<float>(op.K) + P.eps);
#pragma unroll
      for (int j = 0; j < JM; ++j) {
        const int ch = tid + j * nt;
        if (!active || ch >= nch) continue;
#pragma unroll
        for (int e = 0; e < EPC; ++e)
          a[m][j][e] = a[m][j][e] * rstd * bf16_to_f32(__ldg(&op.nw[ch * EPC + e]));
      }
    }
  }

  // ---- stream the CTA's rows
  float* red = reinterpret_cast<float*>(S.un);  // [kRowBatch][kCW][M]
  unsigned long long best = 0ull;
  for (int b0 = 0; b0 < nrows; b0 += kRowBatch) {
    const int nb = min(kRowBatch, nrows - b0);
    for (int i0 = 0; i0 < nb; i0 += op.rs) {
      const int n = min(op.rs, nb - i0);
      const int slot = s_ctr % S.slots;
      if (!*S.abort_flag && !mbar_wait(&S.full[slot], (s_ctr / S.slots) & 1, P.err)) *S.abort_flag = 1;
      const uint8_t* st = S.ring + (size_t)slot * P.stage;
      for (int i = 0; i < n; i += R) {
        float v[V];
#pragma unroll
        for (int r = 0; r < R; ++r) {
          float2 acc[M];
#pragma unroll
          for (int m = 0; m < M; ++m) acc[m] = make_float2(0.f, 0.f);
          if (i + r < n && active) {
            const uint4* row = reinterpret_cast<const uint4*>(st + (size_t)(i + r) * rowbytes);
#pragma unroll
            for (int j = 0; j < JM; ++j) {
              const int ch = tid + j * nt;
              if (ch < nch) {
                const uint4 w = row[ch];
#pragma unroll
                for (int m = 0; m < M; ++m) acc[m] = chunk_fma<WT>(w, a[m][j], acc[m]);
              }
            }
          }
#pragma unroll
          for (int m = 0; m < M; ++m) v[r * M + m] = acc[m].x + acc[m].y;
        }
        const float tot = warp_reduce_many<V>(v, lane);
        if ((lane & 3) == 0) {  // V == 8: lane >> 2 selects the value
          const int idx = lane >> 2;
          const int r = idx / M, m = idx - r * M;
          if (i + r < n) red[((i0 + i + r) * kCW + warp) * M + m] = tot;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[slot]);
      ++s_ctr;
    }
    csync();
    // ---- epilogue
    if (op.unit == 2) {
      for (int pi = tid; pi < (nb >> 1); pi += kCT) {
        const int rg = r0 + b0 + 2 * pi;
#pragma unroll
        for (int m = 0; m < M; ++m) {
          float v0 = 0.f, v1 = 0.f;
#pragma unroll
          for (int w = 0; w < kCW; ++w) {
            v0 += red[((2 * pi) * kCW + w) * M + m];
            v1 += red[((2 * pi + 1) * kCW + w) * M + m];
          }
          if (op.scale) {
            v0 *= __ldg(&op.scale[rg]);
            v1 *= __ldg(&op.scale[rg + 1]);
          }
          if (op.epi == EPI_SWIGLU) op.out[(size_t)m * op.ldo + (rg >> 1)] = silu(v0) * v1;
          else qkv_pair(P, op, m, rg >> 1, v0, v1);
        }
      }
    } else {
      for (int ri = tid; ri < nb; ri += kCT) {
        const int rg = r0 + b0 + ri;
#pragma unroll
        for (int m = 0; m < M; ++m) {
          float v = 0.f;
#pragma unroll
          for (int w = 0; w < kCW; ++w) v += red[(ri * kCW + w) * M + m];
          if (op.scale) v *= __ldg(&op.scale[rg]);
          float* o = op.out + (size_t)m * op.ldo + rg;
          if (op.epi == EPI_RESID) {
            *o = __ldcg(o) + v;
          } else {
            *o = v;
            if (op.epi == EPI_LOGITS) {
              if (v != v) atomicOr(P.err, ERR_NAN);
              const unsigned long long k = pack_key(v, rg);
              best = k > best ? k : best;
            }
          }
        }
      }
    }
    csync();
  }
  if (op.epi == EPI_LOGITS && op.select) {
    best = warp_max_u64(best);
    if (lane == 0) S.keys[warp] = best;
    csync();
    if (tid == 0) {
      unsigned long long b = 0ull;
      for (int w = 0; w < kCW; ++w) b = S.keys[w] > b ? S.keys[w] : b;
      if (b) atomicMax(&P.best[op.cb], b);
      __threadfence();
      const uint32_t t = atomicAdd(&P.ticket[op.cb], 1u);
      if (t == static_cast<uint32_t>(G) - 1u) {
        __threadfence();
        const unsigned long long fin = atomicExch(&P.best[op.cb], 0ull);
        const int idx = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(fin & 0xFFFFFFFFull));
        P.sel[op.cb] = idx;
        P.fb[op.cb] = (*P.forced_on) ? P.forced[op.cb] : idx;
        P.ticket[op.cb] = 0u;
      }
    }
  }
}

template <int WT, int M>
__device__ __forceinline__ void gemv_dispatch_j(const FrameParams& P, const FrameOp& op, Shared& S,
                                                int& s_ctr) {
  if constexpr (WT == 0) {
    switch (op.J) {
      case 1: gemv_op<0, M, 1>(P, op, S, s_ctr); break;
      case 2: gemv_op<0, M, 2>(P, op, S, s_ctr); break;
      case 3: gemv_op<0, M, 3>(P, op, S, s_ctr); break;
      case 4: gemv_op<0, M, 4>(P, op, S, s_ctr); break;
      default: gemv_op<0, M, 5>(P, op, S, s_ctr); break;
    }
  } else {
    switch (op.J) {
      case 1: gemv_op<1, M, 1>(P, op, S, s_ctr); break;
      case 2: gemv_op<1, M, 2>(P, op, S, s_ctr); break;
      default: gemv_op<1, M, 3>(P, op, S, s_ctr); break;
    }
  }
}

__device__ __noinline__ void gemv_dispatch(const FrameParams& P, const FrameOp& op, Shared& S,
                                           int& s_ctr) {
  if (op.wt == 0) {
    if (op.M == 1) gemv_dispatch_j<0, 1>(P, op, S, s_ctr);
    else gemv_dispatch_j<0, 2>(P, op, S, s_ctr);
  } else {
    if (op.M == 1) gemv_dispatch_j<1, 1>(P, op, S, s_ctr);
    else gemv_dispatch_j<1, 2>(P, op, S, s_ctr);
  }
}

// ------------------------------------------------------------------ attention op
template <int D, int G>
__device__ void attn_op(const FrameParams& P, const FrameOp& op, Shared& S) {
  constexpr int DL = D / 32;
  constexpr int kUnroll = 4;
  constexpr int kMinKeys = 32;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  float* sm_m = reinterpret_cast<float*>(S.un);   // [kCW][G]
  float* sm_l = sm_m + kCW * G;                   // [kCW][G]
  float* sm_acc = sm_l + kCW * G;                 // [kCW][G][D]
  float* sm_f = sm_acc + kCW * G * D;             // [G][D+2]
  uint32_t* sm_last = reinterpret_cast<uint32_t*>(sm_f + G * (D + 2));
  const int units = P.Hkv * op.S * op.M;
  for (int u = blockIdx.x; u < units; u += gridDim.x) {
    const int s = u % op.S;
    const int g = (u / op.S) % P.Hkv;
    const int m = u / (op.S * P.Hkv);
    const int pos = op_pos(P, op, m);
    if (pos < 0 || pos >= P.T) {
      if (tid == 0 && s == 0 && g == 0) atomicOr(P.err, ERR_BAD_POS);
      continue;
    }
    const int n = pos + 1;
    const int L = max((n + op.S - 1) / op.S, kMinKeys);
    const int sact = (n + L - 1) / L;
    if (s >= sact) continue;
    const int k0 = s * L, k1 = min(n, k0 + L);
    const float scale = rsqrtf(static_cast<float>(D));
    float q[G][DL];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float* qh = op.q + (size_t)m * P.Hq * D + (size_t)(g * G + h) * D + lane * DL;
#pragma unroll
      for (int d = 0; d < DL; ++d) q[h][d] = __ldcg(qh + d) * scale;
    }
    float mx[G], l[G], acc[G][DL];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      mx[h] = -INFINITY;
      l[h] = 0.f;
#pragma unroll
      for (int d = 0; d < DL; ++d) acc[h][d] = 0.f;
    }
    const uint16_t* Kg = op.Kc + (size_t)g * P.T * D + lane * DL;
    const uint16_t* Vg = op.Vc + (size_t)g * P.T * D + lane * DL;
    for (int t0 = k0 + warp * kUnroll; t0 < k1; t0 += kCW * kUnroll) {
      uint32_t kr[kUnroll][DL / 2], vr[kUnroll][DL / 2];
#pragma unroll
      for (int uu = 0; uu < kUnroll; ++uu) {
        const int t = t0 + uu;
        if (t < k1) {
          if constexpr (DL == 4) {
            const uint2 kk = __ldcg(reinterpret_cast<const uint2*>(Kg + (size_t)t * D));
            const uint2 vv = __ldcg(reinterpret_cast<const uint2*>(Vg + (size_t)t * D));
            kr[uu][0] = kk.x;
            kr[uu][1] = kk.y;
            vr[uu][0] = vv.x;
            vr[uu][1] = vv.y;
          } else {
            kr[uu][0] = __ldcg(reinterpret_cast<const uint32_t*>(Kg + (size_t)t * D));
            vr[uu][0] = __ldcg(reinterpret_cast<const uint32_t*>(Vg + (size_t)t * D));
          }
        }
      }
#pragma unroll
      for (int uu = 0; uu < kUnroll; ++uu) {
        if (t0 + uu >= k1) break;
        float kf[DL], vf[DL];
#pragma unroll
        for (int i = 0; i < DL / 2; ++i) {
          kf[2 * i] = bf16_lo(kr[uu][i]);
          kf[2 * i + 1] = bf16_hi(kr[uu][i]);
          vf[2 * i] = bf16_lo(vr[uu][i]);
          vf[2 * i + 1] = bf16_hi(vr[uu][i]);
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float sc = 0.f;
#pragma unroll
          for (int d = 0; d < DL; ++d) sc = fmaf(q[h][d], kf[d], sc);
          sc = warp_sum(sc);
          const float mn = fmaxf(mx[h], sc);
          const float corr = expf(mx[h] - mn);
          const float pr = expf(sc - mn);
          l[h] = l[h] * corr + pr;
#pragma unroll
          for (int d = 0; d < DL; ++d) acc[h][d] = fmaf(acc[h][d], corr, pr * vf[d]);
          mx[h] = mn;
        }
      }
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
      if (lane == 0) {
        sm_m[warp * G + h] = mx[h];
        sm_l[warp * G + h] = l[h];
      }
#pragma unroll
      for (int d = 0; d < DL; ++d) sm_acc[(warp * G + h) * D + lane * DL + d] = acc[h][d];
    }
    csync();
    for (int e = tid; e < G * D; e += kCT) {
      const int h = e / D, d = e - h * D;
      float Mx = -INFINITY;
      for (int w = 0; w < kCW; ++w) Mx = fmaxf(Mx, sm_m[w * G + h]);
      float Ls = 0.f, A = 0.f;
      for (int w = 0; w < kCW; ++w) {
        if (sm_m[w * G + h] == -INFINITY) continue;
        const float f = expf(sm_m[w * G + h] - Mx);
        Ls += sm_l[w * G + h] * f;
        A += sm_acc[(w * G + h) * D + d] * f;
      }
      sm_f[h * (D + 2) + d] = A;
      if (d == 0) {
        sm_f[h * (D + 2) + D] = Mx;
        sm_f[h * (D + 2) + D + 1] = Ls;
      }
    }
    csync();
    if (sact == 1) {
      for (int e = tid; e < G * D; e += kCT) {
        const int h = e / D, d = e - h * D;
        op.o[(size_t)m * P.Hq * D + (size_t)(g * G + h) * D + d] = sm_f[h * (D + 2) + d] / sm_f[h * (D + 2) + D + 1];
      }
      csync();
      continue;
    }
    for (int e = tid; e < G * (D + 2); e += kCT) {
      const int h = e / (D + 2), d = e - h * (D + 2);
      P.part[(((size_t)m * P.Hq + g * G + h) * op.S + s) * (D + 2) + d] = sm_f[h * (D + 2) + d];
    }
    __threadfence();
    csync();
    if (tid == 0) {
      const uint32_t t = atomicAdd(&P.counters[m * P.Hkv + g], 1u);
      *sm_last = (t == static_cast<uint32_t>(sact) - 1u);
    }
    csync();
    if (*sm_last) {
      __threadfence();
      for (int e = tid; e < G * D; e += kCT) {
        const int h = e / D, d = e - h * D;
        const float* ph = P.part + (((size_t)m * P.Hq + g * G + h) * op.S) * (D + 2);
        float Mx = -INFINITY;
        for (int j = 0; j < sact; ++j) Mx = fmaxf(Mx, __ldcg(ph + (size_t)j * (D + 2) + D));
        float Ls = 0.f, A = 0.f;
        for (int j = 0; j < sact; ++j) {
          const float f = expf(__ldcg(ph + (size_t)j * (D + 2) + D) - Mx);
          Ls += __ldcg(ph + (size_t)j * (D + 2) + D + 1) * f;
          A += __ldcg(ph + (size_t)j * (D + 2) + d) * f;
        }
        op.o[(size_t)m * P.Hq * D + (size_t)(g * G + h) * D + d] = A / Ls;
      }
      if (tid == 0) P.counters[m * P.Hkv + g] = 0u;
    }
    csync();
  }
}

template <int D>
__device__ void attn_dispatch_g(const FrameParams& P, const FrameOp& op, Shared& S) {
  switch (P.Hq / P.Hkv) {
    case 1: attn_op<D, 1>(P, op, S); break;
    case 2: attn_op<D, 2>(P, op, S); break;
    case 4: attn_op<D, 4>(P, op, S); break;
    default: attn_op<D, 8>(P, op, S); break;
  }
}

// ------------------------------------------------------------------ select op
// Exact top-k draw (or argmax) over one logits row by the consumer threads of
// CTA 0; the same rule as the standalone selection kernel.
__device__ __forceinline__ float exp32(float x) {
  if (x < -80.0f) return 0.0f;
  const float kLog2e = __uint_as_float(0x3fb8aa3bu);
  const float kLn2Hi = __uint_as_float(0x3f317200u);
  const float kLn2Lo = __uint_as_float(0x35bfbe8eu);
  const float c[8] = {__uint_as_float(0x3f800000u), __uint_as_float(0x3f800000u),
                      __uint_as_float(0x3f000000u), __uint_as_float(0x3e2aaaabu),
                      __uint_as_float(0x3d2aaaabu), __uint_as_float(0x3c088889u),
                      __uint_as_float(0x3ab60b61u), __uint_as_float(0x39500d01u)};
  const float n = rintf(__fmul_rn(x, kLog2e));
  float r = __fsub_rn(x, __fmul_rn(n, kLn2Hi));
  r = __fsub_rn(r, __fmul_rn(n, kLn2Lo));
  float p = c[7];
#pragma unroll
  for (int k = 6; k >= 0; --k) p = __fadd_rn(__fmul_rn(p, r), c[k]);
  return ldexpf(p, static_cast<int>(n));
}

__device__ __forceinline__ uint32_t philox_w0(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                              uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t hi0 = __umulhi(0xD2511F53u, c0), lo0 = 0xD2511F53u * c0;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c2), lo1 = 0xCD9E8D57u * c2;
    const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
  }
  return c0;
}

__device__ __forceinline__ uint32_t sel_key(float z) {
  if (z == 0.f) z = 0.f;
  return float_order_key(z);
}

__device__ void select_op(const FrameParams& P, const FrameOp& op, Shared& S) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = op.vocab;
  const int k = min(P.top_k, V);
  uint32_t* keys = reinterpret_cast<uint32_t*>(S.un);  // [V]
  uint32_t* hist = keys + V;                            // [256]
  int* cand_idx = reinterpret_cast<int*>(hist + 256);   // [k]
  uint32_t* cand_key = reinterpret_cast<uint32_t*>(cand_idx + k);
  int* sort_idx = reinterpret_cast<int*>(cand_key + k);
  float* sort_z = reinterpret_cast<float*>(sort_idx + k);
  float* wts = sort_z + k;
  uint32_t* sc = reinterpret_cast<uint32_t*>(wts + k);  // prefix, remaining, ncand
  const float* z = op.logits;
  bool nan = false;
  for (int i = tid; i < V; i += kCT) {
    const float v = __ldcg(z + i);
    nan |= (v != v);
    keys[i] = sel_key(v);
  }
  if (nan) atomicOr(P.err, ERR_NAN);
  if (tid == 0) {
    sc[0] = 0u;
    sc[1] = static_cast<uint32_t>(k);
    sc[2] = 0u;
  }
  uint32_t mask = 0u;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += kCT) hist[i] = 0u;
    csync();
    const uint32_t prefix = sc[0];
    for (int i = tid; i < V; i += kCT)
      if ((keys[i] & mask) == prefix) atomicAdd(&hist[(keys[i] >> shift) & 0xFFu], 1u);
    csync();
    if (tid == 0) {
      uint32_t rem = sc[1], cum = 0u;
      int b = 255;
      for (; b > 0; --b) {
        if (cum + hist[b] >= rem) break;
        cum += hist[b];
      }
      sc[1] = rem - cum;
      sc[0] = prefix | (static_cast<uint32_t>(b) << shift);
    }
    mask |= 0xFFu << shift;
    csync();
  }
  const uint32_t T = sc[0];
  const uint32_t need_eq = sc[1];
  for (int i = tid; i < V; i += kCT) {
    if (keys[i] > T) {
      const uint32_t slot = atomicAdd(&sc[2], 1u);
      cand_idx[slot] = i;
      cand_key[slot] = keys[i];
    }
  }
  csync();
  if (warp == 0) {
    uint32_t taken = 0u;
    for (int base = 0; base < V && taken < need_eq; base += 32) {
      const int i = base + lane;
      const bool eq = i < V && keys[i] == T;
      const uint32_t bal = __ballot_sync(0xFFFFFFFFu, eq);
      const uint32_t before = __popc(bal & ((1u << lane) - 1u));
      if (eq && taken + before < need_eq) {
        const uint32_t slot = sc[2] + taken + before;
        cand_idx[slot] = i;
        cand_key[slot] = T;
      }
      taken += __popc(bal);
    }
  }
  csync();
  for (int c = tid; c < k; c += kCT) {
    const uint32_t ki = cand_key[c];
    const int ii = cand_idx[c];
    int r = 0;
    for (int j = 0; j < k; ++j) {
      const uint32_t kj = cand_key[j];
      r += (kj > ki) || (kj == ki && cand_idx[j] < ii);
    }
    sort_idx[r] = ii;
    sort_z[r] = __ldcg(z + ii);
  }
  csync();
  for (int c = tid; c < k; c += kCT) {
    float d = __fsub_rn(sort_z[c], sort_z[0]);
    if (P.temperature != 1.0f) d = __fdiv_rn(d, P.temperature);
    wts[c] = exp32(d);
  }
  csync();
  if (tid == 0) {
    float Ssum = 0.f;
    for (int j = 0; j < k; ++j) Ssum = __fadd_rn(Ssum, wts[j]);
    const int frame = *reinterpret_cast<volatile int32_t*>(P.frame_index);
    const uint32_t w0 = philox_w0(static_cast<uint32_t>(frame), static_cast<uint32_t>(op.cb), 0u, 0u,
                                  P.key0, P.key1);
    const float u = __fmul_rn(static_cast<float>(w0 >> 8), 5.9604644775390625e-8f);
    const float t = __fmul_rn(u, Ssum);
    int pk = k - 1;
    float cum = 0.f;
    for (int j = 0; j < k; ++j) {
      cum = __fadd_rn(cum, wts[j]);
      if (t < cum) {
        pk = j;
        break;
      }
    }
    const int pick = sort_idx[pk];
    P.sel[op.cb] = pick;
    P.fb[op.cb] = (*P.forced_on) ? P.forced[op.cb] : pick;
  }
}

// ------------------------------------------------------------------ kernel
__global__ void __launch_bounds__(kThreads, kFrameCtasPerSm) k_frame(const FrameParams P) {
  extern __shared__ __align__(128) uint8_t smem[];
  Shared S;
  S.slots = P.slots;
  S.ring = smem;
  S.un = smem + (size_t)P.slots * P.stage;
  S.full = reinterpret_cast<uint64_t*>(S.un + P.un_bytes);
  S.empty = S.full + P.slots;
  S.misc = reinterpret_cast<float*>(S.empty + P.slots);
  S.keys = reinterpret_cast<unsigned long long*>(S.misc + 32);
  S.abort_flag = reinterpret_cast<volatile uint32_t*>(S.keys + 16);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x;
  if (tid == 0) {
    for (int i = 0; i < P.slots; ++i) {
      mbar_init(&S.full[i], 1);
      mbar_init(&S.empty[i], kCW);
    }
    *S.abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kCW) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int s = 0;
      for (int f = 0; f < P.n_frames && !*S.abort_flag; ++f) {
        for (int i = 0; i < P.n_ops && !*S.abort_flag; ++i) {
          const FrameOp& op = P.ops[i];
          if (op.kind != OPK_GEMV) continue;
          int r0, nrows;
          op_rows(op, blockIdx.x, G, &r0, &nrows);
          const uint32_t rowbytes = static_cast<uint32_t>(op.K) * (op.wt ? 1u : 2u);
          for (int b0 = 0; b0 < nrows; b0 += kRowBatch) {
            const int nb = min(kRowBatch, nrows - b0);
            for (int i0 = 0; i0 < nb; i0 += op.rs) {
              const int n = min(op.rs, nb - i0);
              const int slot = s % P.slots;
              if (s >= P.slots && !mbar_wait(&S.empty[slot], ((s / P.slots) & 1) ^ 1, P.err)) {
                *S.abort_flag = 1;
                break;
              }
              const uint32_t bytes = static_cast<uint32_t>(n) * rowbytes;
              mbar_arrive_expect_tx(&S.full[slot], bytes);
              bulk_g2s(S.ring + (size_t)slot * P.stage, op.W + (size_t)(r0 + b0 + i0) * rowbytes,
                       bytes, &S.full[slot], pol);
              ++s;
            }
            if (*S.abort_flag) break;
          }
        }
      }
      for (int t = max(0, s - P.slots); t < s; ++t)
        mbar_wait(&S.full[t % P.slots], (t / P.slots) & 1, P.err);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  int s_ctr = 0;
  for (int f = 0; f < P.n_frames; ++f) {
    for (int i = 0; i < P.n_ops; ++i) {
      const FrameOp& op = P.ops[i];
      const uint32_t gi = static_cast<uint32_t>(f) * P.n_ops + i;
      const int trace_slot = (P.trace && f == 0 && tid == 0)
                                 ? (blockIdx.x == 0 ? 0 : (blockIdx.x == G - 1 ? 1 : -1))
                                 : -1;
      if (trace_slot >= 0) P.trace[(i * 2 + trace_slot) * 3 + 0] = globaltimer_ns();
      // grid barrier: every CTA has finished ops 0 .. gi-1
      if (gi > 0) {
        if (tid == 0 && !*S.abort_flag) {
          const uint32_t target = gi * static_cast<uint32_t>(G);
          if (ld_acquire(P.gbar) < target) {
            const uint64_t t0 = globaltimer_ns();
            while (ld_acquire(P.gbar) < target) {
              if (globaltimer_ns() - t0 > kWaitBudgetNs) {
                atomicOr(P.err, ERR_TIMEOUT);
                *S.abort_flag = 1;
                break;
              }
            }
          }
          __threadfence();
        }
        csync();
      }
      if (trace_slot >= 0) P.trace[(i * 2 + trace_slot) * 3 + 1] = globaltimer_ns();
      switch (op.kind) {
        case OPK_GEMV:
          gemv_dispatch(P, op, S, s_ctr);
          break;
        case OPK_ATTN:
          if (P.D == 128) attn_dispatch_g<128>(P, op, S);
          else attn_dispatch_g<64>(P, op, S);
          break;
        case OPK_SELECT:
          if (blockIdx.x == 0) select_op(P, op, S);
          break;
        default:  // OPK_END
          if (blockIdx.x == 0 && tid == 0) {
            *P.pos += op.advance;
            *P.frame_index += 1;
            if (P.hist) {
              const int h = *P.hist_idx;
              if (h < P.hist_cap) {
                for (int c = 0; c < P.ncb; ++c) P.hist[(size_t)h * P.ncb + c] = P.sel[c];
                *P.hist_idx = h + 1;
              }
            }
          }
          break;
      }
      csync();
      if (trace_slot >= 0) P.trace[(i * 2 + trace_slot) * 3 + 2] = globaltimer_ns();
      if (tid == 0) {
        __threadfence();
        red_release_add(P.gbar, 1u);
      }
    }
  }
}

}  // namespace

bool frame_plan_gemv(FrameOp& op, int stage) {
  const int eb = op.wt ? 1 : 2;
  const int rowbytes = op.K * eb;
  if (rowbytes % 16 || rowbytes > stage) return false;
  const int nch = rowbytes / 16;
  // Most even split of the row's chunks over at most kCT threads (multiples
  // of 32), at most 5 (bf16) or 3 (fp8) chunks per thread; ties go to more
  // threads.
  const int jmax = op.wt ? 3 : 5;
  double best = -1.0;
  op.J = 0;
  for (int w = kCW; w >= 1; --w) {
    const int nt = 32 * w, J = (nch + nt - 1) / nt;
    if (J > jmax) continue;
    const double eff = static_cast<double>(nch) / (static_cast<double>(nt) * J);
    if (eff > best + 1e-9) {
      best = eff;
      op.J = J;
      op.nt = nt;
    }
  }
  if (op.J == 0) return false;
  op.rs = std::max(1, stage / rowbytes);
  op.rs = std::min(op.rs, kRowBatch);
  op.unit = (op.epi == EPI_SWIGLU || op.epi == EPI_QKV) ? 2 : 1;
  return op.N % op.unit == 0;
}

int frame_union_bytes(int G, int D, int max_vocab) {
  const int red = kRowBatch * kCW * 2 * 4;
  const int attn = (2 * kCW * G + kCW * G * D + G * (D + 2)) * 4 + 16;
  const int sel = (max_vocab + 256 + 6 * 256 + 8) * 4;
  return ((std::max({red, attn, sel}) + 127) / 128) * 128;
}

size_t frame_smem_bytes(int slots, int stage, int un_bytes) {
  return (size_t)slots * stage + un_bytes + 2 * (size_t)slots * 8 + 32 * 4 + 16 * 8 + 16;
}

cudaError_t frame_set_attributes() {
  cudaError_t e = cudaFuncSetAttribute(k_frame, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  if (e) return e;
  return cudaFuncSetAttribute(k_frame, cudaFuncAttributePreferredSharedMemoryCarveout,
                              cudaSharedmemCarveoutMaxShared);
}

cudaError_t launch_frame(const FrameParams& p, int grid, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = frame_smem_bytes(p.slots, p.stage, p.un_bytes);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_frame, p);
}

}  // namespace tf
