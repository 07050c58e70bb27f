// Grouped-query decode attention over the static KV cache (sm_103a).
//
// "Fish Speech" tour, "Why You Need This": the decoder uses rotary embeddings
// and grouped-query attention; the tuna-fish README ("Inference estimation")
// keeps a static KV cache of max_length positions per layer.  One query row
// at position p attends to keys 0..p of its KV head (query head h reads KV
// head h / (Hq/Hkv)), scaled by 1/sqrt(D), softmax over the keys.
//
// Flash-decode split: grid (S, Hkv, M).  CTA (s, g, m) takes a contiguous
// slice of the key range and all Hq/Hkv query heads that share KV head g, so
// every K/V row is read from HBM once per layer.  Each warp walks keys with
// lanes across the head dimension (one coalesced 8-byte load per lane per
// row, four rows in flight), keeps an online softmax per head, and the warps
// merge in shared memory.  The last CTA of each (g, m) to finish (ticket on
// a global counter) merges the S partials in split order, so the result is
// deterministic, and re-arms the counter.
#include "common.cuh"
#include "kernels.h"

namespace tf {

namespace {

constexpr int kWarps = 8;
constexpr int kUnroll = 4;
constexpr int kMinKeys = 32;

template <int D, int G>
__global__ void __launch_bounds__(kWarps * 32) k_attn(const AttnParams p) {
  constexpr int DL = D / 32;  // dims per lane
  const int s = blockIdx.x, g = blockIdx.y, m = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  __shared__ float sm_m[kWarps][G], sm_l[kWarps][G];
  __shared__ float sm_acc[kWarps][G][D];
  __shared__ float sm_f[G][D + 2];
  __shared__ uint32_t sm_last;

  pdl_launch_dependents();
  pdl_wait();
  const int pos = (p.pos_ptr ? p.pos_ptr[0] : p.pos_fixed) + m;
  if (pos < 0 || pos >= p.T) {
    if (tid == 0 && s == 0) atomicOr(p.err, ERR_BAD_POS);
    return;
  }
  const int n = pos + 1;
  // At least kMinKeys keys per split: short contexts use fewer CTAs.
  const int L = max((n + p.S - 1) / p.S, kMinKeys);
  const int sact = (n + L - 1) / L;
  if (s >= sact) return;
  const int k0 = s * L, k1 = min(n, k0 + L);

  // Queries of the G heads of this group, pre-scaled by 1/sqrt(D).
  const float scale = rsqrtf(static_cast<float>(D));
  float q[G][DL];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const float* qh = p.q + (size_t)m * p.Hq * D + (size_t)(g * G + h) * D + lane * DL;
#pragma unroll
    for (int d = 0; d < DL; ++d) q[h][d] = qh[d] * scale;
  }

  float mx[G], l[G], acc[G][DL];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    mx[h] = -INFINITY;
    l[h] = 0.f;
#pragma unroll
    for (int d = 0; d < DL; ++d) acc[h][d] = 0.f;
  }

  const uint16_t* Kg = p.Kc + (size_t)g * p.T * D + lane * DL;
  const uint16_t* Vg = p.Vc + (size_t)g * p.T * D + lane * DL;
  for (int t0 = k0 + warp * kUnroll; t0 < k1; t0 += kWarps * kUnroll) {
    // Load up to kUnroll rows of K and V (DL bf16 per lane).
    uint32_t kr[kUnroll][DL / 2], vr[kUnroll][DL / 2];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int t = t0 + u;
      if (t < k1) {
        if constexpr (DL == 4) {
          const uint2 kk = *reinterpret_cast<const uint2*>(Kg + (size_t)t * D);
          const uint2 vv = *reinterpret_cast<const uint2*>(Vg + (size_t)t * D);
          kr[u][0] = kk.x; kr[u][1] = kk.y;
          vr[u][0] = vv.x; vr[u][1] = vv.y;
        } else {
          kr[u][0] = *reinterpret_cast<const uint32_t*>(Kg + (size_t)t * D);
          vr[u][0] = *reinterpret_cast<const uint32_t*>(Vg + (size_t)t * D);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (t0 + u >= k1) break;
      float kf[DL], vf[DL];
#pragma unroll
      for (int i = 0; i < DL / 2; ++i) {
        kf[2 * i] = bf16_lo(kr[u][i]);
        kf[2 * i + 1] = bf16_hi(kr[u][i]);
        vf[2 * i] = bf16_lo(vr[u][i]);
        vf[2 * i + 1] = bf16_hi(vr[u][i]);
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

  // Merge the warps of this CTA.
#pragma unroll
  for (int h = 0; h < G; ++h) {
    if (lane == 0) {
      sm_m[warp][h] = mx[h];
      sm_l[warp][h] = l[h];
    }
#pragma unroll
    for (int d = 0; d < DL; ++d) sm_acc[warp][h][lane * DL + d] = acc[h][d];
  }
  __syncthreads();
  for (int e = tid; e < G * D; e += kWarps * 32) {
    const int h = e / D, d = e - h * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w][h]);
    float Ls = 0.f, A = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      if (sm_m[w][h] == -INFINITY) continue;  // warp saw no keys
      const float f = expf(sm_m[w][h] - M);
      Ls += sm_l[w][h] * f;
      A += sm_acc[w][h][d] * f;
    }
    sm_f[h][d] = A;
    if (d == 0) {
      sm_f[h][D] = M;
      sm_f[h][D + 1] = Ls;
    }
  }
  __syncthreads();

  if (sact == 1) {
    for (int e = tid; e < G * D; e += kWarps * 32) {
      const int h = e / D, d = e - h * D;
      p.out[(size_t)m * p.Hq * D + (size_t)(g * G + h) * D + d] = sm_f[h][d] / sm_f[h][D + 1];
    }
    return;
  }

  // Publish this split's partial and take a ticket.
  for (int e = tid; e < G * (D + 2); e += kWarps * 32) {
    const int h = e / (D + 2), d = e - h * (D + 2);
    p.part[(((size_t)m * p.Hq + g * G + h) * p.S + s) * (D + 2) + d] = sm_f[h][d];
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const uint32_t t = atomicAdd(&p.counters[m * p.Hkv + g], 1u);
    sm_last = (t == static_cast<uint32_t>(sact) - 1u);
  }
  __syncthreads();
  if (!sm_last) return;
  __threadfence();
  for (int e = tid; e < G * D; e += kWarps * 32) {
    const int h = e / D, d = e - h * D;
    const float* ph = p.part + (((size_t)m * p.Hq + g * G + h) * p.S) * (D + 2);
    float M = -INFINITY;
    for (int j = 0; j < sact; ++j) M = fmaxf(M, __ldcg(ph + (size_t)j * (D + 2) + D));
    float Ls = 0.f, A = 0.f;
    for (int j = 0; j < sact; ++j) {
      const float f = expf(__ldcg(ph + (size_t)j * (D + 2) + D) - M);
      Ls += __ldcg(ph + (size_t)j * (D + 2) + D + 1) * f;
      A += __ldcg(ph + (size_t)j * (D + 2) + d) * f;
    }
    p.out[(size_t)m * p.Hq * D + (size_t)(g * G + h) * D + d] = A / Ls;
  }
  if (tid == 0) p.counters[m * p.Hkv + g] = 0u;
}

template <int D, int G>
cudaError_t launch_dg(const AttnParams& p, int M, bool pdl, cudaStream_t s) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k_attn<D, G>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         cudaSharedmemCarveoutMaxShared);
    if (e) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.S, p.Hkv, M);
  cfg.blockDim = dim3(kWarps * 32);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_attn<D, G>, p);
}

template <int D>
cudaError_t launch_d(const AttnParams& p, int M, bool pdl, cudaStream_t s) {
  switch (p.Hq / p.Hkv) {
    case 1: return launch_dg<D, 1>(p, M, pdl, s);
    case 2: return launch_dg<D, 2>(p, M, pdl, s);
    case 4: return launch_dg<D, 4>(p, M, pdl, s);
    case 8: return launch_dg<D, 8>(p, M, pdl, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_attention(const AttnParams& p, int M, bool pdl, cudaStream_t s) {
  if (p.Hq % p.Hkv) return cudaErrorInvalidValue;
  if (p.D == 128) return launch_d<128>(p, M, pdl, s);
  if (p.D == 64) return launch_d<64>(p, M, pdl, s);
  return cudaErrorInvalidValue;
}

}  // namespace tf
