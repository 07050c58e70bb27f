// Grouped-query decode attention over the static KV cache (sm_103a).
//
// "Fish Speech" tour, "Why You Need This": the decoder uses rotary embeddings
// and grouped-query attention; the tuna-fish README ("Inference estimation")
// keeps a static KV cache of max_length positions per layer.  One query row
// at position p attends to keys 0..p of its KV head (query head h reads KV
// head h / (Hq/Hkv)), scaled by 1/sqrt(D), softmax over the keys.
//
// Flash-decode split: grid (S, Hkv, M).  CTA (s, g, m) takes a contiguous
// slice of row m's key range and all Hq/Hkv query heads that share KV head g,
// so every K/V row is read from HBM once per layer.  The slice's K and V rows
// are contiguous in the cache ([Hkv][T][D] per sequence), so the CTA stages
// them into shared memory with bulk copies, 64 keys at a time, two chunks in
// flight; scores, an online softmax per head and the weighted sum of V run
// out of shared memory.  With more than one slice, each CTA publishes its
// (max, sum, weighted V) and takes a ticket; the last CTA of each (g, m)
// merges the slices in slice order (deterministic) and re-arms the counter.
// Every dependent global round trip costs on this two-die part, so the kernel
// issues each group of loads at once: the K/V chunks, then all slices'
// (max, sum) pairs, then their weighted V in batches.
#include <mutex>

#include "../../include/tf.h"
#include "common.cuh"
#include "device_once.h"
#include "kernels.h"

namespace tf {

namespace {

constexpr int kThreads = 256;
constexpr int kChunk = 64;      // keys per staged chunk
constexpr int kMinKeys = 32;    // keys per slice at least
constexpr int kMaxSlices = 64;  // slices a combine can hold

// Output element i of row data: fp32, or bf16 hi / lo parts for a GEMM that
// reads its activations from the tensor cores.
__device__ __forceinline__ void store_out(const AttnParams& p, size_t i, float v) {
  if (p.out_hi) {
    const uint16_t h = f32_to_bf16(v);
    p.out_hi[i] = h;
    p.out_lo[i] = f32_to_bf16(v - bf16_to_f32(h));
  } else {
    p.out[i] = v;
  }
}

__device__ __forceinline__ uint32_t ticket_acq_rel(uint32_t* t) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(t) : "memory");
  return old;
}

__device__ __forceinline__ void bulk_g2s_plain(void* dst, const void* src, uint32_t bytes,
                                               uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

template <int D, int G>
struct AttnSmem {
  static constexpr int kRow = D * 2;                          // bytes of one K or V row
  static constexpr int kBuf = kChunk * kRow;                  // one K (or V) chunk
  static constexpr size_t kOffQ = 4 * (size_t)kBuf;           // K0 V0 K1 V1, then q
  static constexpr size_t kOffSc = kOffQ + (size_t)G * D * 4;  // scores [G][kChunk]
  static constexpr size_t kOffStat = kOffSc + (size_t)G * kChunk * 4;  // max, sum, rescale [G]
  static constexpr size_t kOffBar = (kOffStat + 3 * G * 4 + 15) / 16 * 16;
  static constexpr size_t kBytes = kOffBar + 2 * 8 + 16;
  static_assert(4 * (size_t)kBuf >= 2 * (size_t)G * kMaxSlices * 4 + G * 4,
                "the combine's statistics reuse the K/V buffers");
};

template <int D, int G>
__global__ void __launch_bounds__(kThreads) k_attn(const AttnParams p) {
  using SL = AttnSmem<D, G>;
  constexpr int DL = D / 32;                                 // dims per lane (score step)
  constexpr int NP = (G * D + kThreads - 1) / kThreads;      // (head, dim) outputs per thread
  extern __shared__ __align__(128) uint8_t sm[];
  uint16_t* kv = reinterpret_cast<uint16_t*>(sm);
  float* q_s = reinterpret_cast<float*>(sm + SL::kOffQ);
  float* sc = reinterpret_cast<float*>(sm + SL::kOffSc);
  float* m_run = reinterpret_cast<float*>(sm + SL::kOffStat);
  float* l_run = m_run + G;
  float* corr = l_run + G;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + SL::kOffBar);
  volatile uint32_t* flag = reinterpret_cast<volatile uint32_t*>(bar + 2);

  const int s = blockIdx.x, g = blockIdx.y, m = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  pdl_launch_dependents();
  pdl_wait();
  // Row m is row m % rps of sequence seq_base + m / rps (rps = 0: every row
  // belongs to sequence seq_base).
  const int seq = p.seq_base + (p.rps > 0 ? m / p.rps : 0);
  const int pos = (p.pos_ptr ? p.pos_ptr[seq] : p.pos_fixed) + (p.rps > 0 ? m % p.rps : m);
  if (pos < 0 || pos >= p.T) {
    if (tid == 0 && s == 0) atomicOr(p.err, ERR_BAD_POS);
    return;
  }
  const int n = pos + 1;
  // At least kMinKeys keys per slice: short contexts use fewer CTAs.  Paged
  // caches: slices start on page boundaries, so a 64-key chunk is two pages.
  int L = max((n + p.S - 1) / p.S, kMinKeys);
  if (p.kv_tbl) L = (L + kKvPage - 1) / kKvPage * kKvPage;
  const int sact = (n + L - 1) / L;
  if (s >= sact) return;
  const int k0 = s * L, nk = min(n, k0 + L) - k0;
  const int nch = (nk + kChunk - 1) / kChunk;
  const size_t kvo = (size_t)seq * (size_t)p.kv_seq;
  const uint16_t* Kg = p.Kc + kvo + ((size_t)g * p.T + k0) * D;
  const uint16_t* Vg = p.Vc + kvo + ((size_t)g * p.T + k0) * D;

  auto issue = [&](int ch) {  // one thread: chunk ch of K and V into buffer ch & 1
    const int b = ch & 1;
    const int rows = min(kChunk, nk - ch * kChunk);
    const uint32_t bytes = static_cast<uint32_t>(rows * SL::kRow);
    mbar_arrive_expect_tx(&bar[b], 2 * bytes);
    uint16_t* kd = kv + (size_t)(2 * b) * kChunk * D;
    uint16_t* vd = kv + (size_t)(2 * b + 1) * kChunk * D;
    if (p.kv_tbl) {  // one copy per page run of the chunk
      for (int r0 = 0; r0 < rows; r0 += kKvPage) {
        const int kpos = k0 + ch * kChunk + r0;
        const int page = p.kv_tbl[(size_t)seq * p.kv_npp + kpos / kKvPage];
        const size_t src = (((size_t)page * p.Hkv + g) * kKvPage) * D;
        const uint32_t rb = static_cast<uint32_t>(min(kKvPage, rows - r0) * SL::kRow);
        bulk_g2s_plain(kd + (size_t)r0 * D, p.Kc + src, rb, &bar[b]);
        bulk_g2s_plain(vd + (size_t)r0 * D, p.Vc + src, rb, &bar[b]);
      }
    } else {
      bulk_g2s_plain(kd, Kg + (size_t)ch * kChunk * D, bytes, &bar[b]);
      bulk_g2s_plain(vd, Vg + (size_t)ch * kChunk * D, bytes, &bar[b]);
    }
  };
  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbar_init();
    *flag = 0u;
    issue(0);
    if (nch > 1) issue(1);
  }
  // Queries of the G heads of this group, pre-scaled by 1/sqrt(D).
  const float scale = rsqrtf(static_cast<float>(D));
  for (int e = tid; e < G * D; e += kThreads) {
    const int h = e / D, d = e - h * D;
    q_s[e] = p.q[(size_t)m * p.Hq * D + (size_t)(g * G + h) * D + d] * scale;
  }
  if (tid < G) {
    m_run[tid] = -INFINITY;
    l_run[tid] = 0.f;
  }
  __syncthreads();

  float acc[NP];
#pragma unroll
  for (int i = 0; i < NP; ++i) acc[i] = 0.f;
  for (int ch = 0; ch < nch; ++ch) {
    const int b = ch & 1;
    const int rows = min(kChunk, nk - ch * kChunk);
    const bool got = mbar_wait(&bar[b], (ch >> 1) & 1, p.err);
    if (__syncthreads_or(got ? 0 : 1)) {
      // Expired (reported): before the CTA gives up, let the copies still in
      // flight into its shared memory land (chunks ch .. ch + 1), each wait
      // bounded again, so none of them writes into a later CTA's memory.
      if (tid == 0)
        for (int c2 = ch; c2 < min(nch, ch + 2); ++c2)
          if (!mbar_wait(&bar[c2 & 1], (c2 >> 1) & 1, p.err)) break;
      return;
    }
    const uint16_t* Ks = kv + (size_t)(2 * b) * kChunk * D;
    const uint16_t* Vs = Ks + (size_t)kChunk * D;
    // scores: warp w takes keys w, w + 8, ...; lanes across the head dimension
    for (int t = warp; t < rows; t += kThreads / 32) {
      float kf[DL];
      if constexpr (DL == 4) {
        const uint2 kk = *reinterpret_cast<const uint2*>(Ks + (size_t)t * D + lane * DL);
        kf[0] = bf16_lo(kk.x);
        kf[1] = bf16_hi(kk.x);
        kf[2] = bf16_lo(kk.y);
        kf[3] = bf16_hi(kk.y);
      } else {
        const uint32_t kk = *reinterpret_cast<const uint32_t*>(Ks + (size_t)t * D + lane * DL);
        kf[0] = bf16_lo(kk);
        kf[1] = bf16_hi(kk);
      }
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float d = 0.f;
#pragma unroll
        for (int i = 0; i < DL; ++i) d = fmaf(q_s[h * D + lane * DL + i], kf[i], d);
        d = warp_sum(d);
        if (lane == 0) sc[h * kChunk + t] = d;
      }
    }
    __syncthreads();
    // online softmax: warp h updates head h's running max and sum
    if (warp < G) {
      const int h = warp;
      float mx = -INFINITY;
      for (int t = lane; t < rows; t += 32) mx = fmaxf(mx, sc[h * kChunk + t]);
      mx = warp_max(mx);
      const float mo = m_run[h];
      const float mn = fmaxf(mo, mx);
      float sum = 0.f;
      for (int t = lane; t < rows; t += 32) {
        const float e = expf(sc[h * kChunk + t] - mn);
        sc[h * kChunk + t] = e;
        sum += e;
      }
      sum = warp_sum(sum);
      if (lane == 0) {
        const float cr = expf(mo - mn);
        corr[h] = cr;
        l_run[h] = l_run[h] * cr + sum;
        m_run[h] = mn;
      }
    }
    __syncthreads();
    // weighted V: thread owns (head, dim) outputs
#pragma unroll
    for (int i = 0; i < NP; ++i) {
      const int e = tid + i * kThreads;
      if (e < G * D) {
        const int h = e / D, d = e - h * D;
        const float* ph = sc + h * kChunk;
        float a = acc[i] * corr[h];
        for (int t = 0; t < rows; ++t) a = fmaf(ph[t], bf16_to_f32(Vs[(size_t)t * D + d]), a);
        acc[i] = a;
      }
    }
    __syncthreads();  // buffer b is free again
    if (tid == 0 && ch + 2 < nch) issue(ch + 2);
  }

  if (sact == 1) {
#pragma unroll
    for (int i = 0; i < NP; ++i) {
      const int e = tid + i * kThreads;
      if (e < G * D) {
        const int h = e / D, d = e - h * D;
        store_out(p, (size_t)m * p.Hq * D + (size_t)(g * G + h) * D + d, acc[i] / l_run[h]);
      }
    }
    return;
  }

  // Publish this slice: part[m][head][slice][D + 2] = (weighted V, max, sum).
  float* pb = p.part + ((size_t)m * p.Hq + (size_t)g * G) * p.S * (D + 2);
#pragma unroll
  for (int i = 0; i < NP; ++i) {
    const int e = tid + i * kThreads;
    if (e < G * D) {
      const int h = e / D, d = e - h * D;
      __stcg(pb + ((size_t)h * p.S + s) * (D + 2) + d, acc[i]);
    }
  }
  if (tid < G) {
    __stcg(pb + ((size_t)tid * p.S + s) * (D + 2) + D, m_run[tid]);
    __stcg(pb + ((size_t)tid * p.S + s) * (D + 2) + D + 1, l_run[tid]);
  }
  __syncthreads();
  if (tid == 0) {
    const uint32_t t = ticket_acq_rel(&p.counters[m * p.Hkv + g]);
    *flag = (t == static_cast<uint32_t>(sact) - 1u) ? 1u : 0u;
  }
  __syncthreads();
  if (!*flag) return;

  // Merge (last CTA): every slice's (max, sum) at once, then the slices'
  // weights exp(max_j - max) and the total sum per head, then the weighted
  // V of all slices in batches of independent loads.
  float* wj = reinterpret_cast<float*>(kv);  // [G][sact]: max, then weight
  float* lj = wj + G * kMaxSlices;           // [G][sact]: sums
  float* lt = lj + G * kMaxSlices;           // [G]: total
  for (int e = tid; e < G * sact; e += kThreads) {
    const int h = e / sact, j = e - h * sact;
    wj[h * kMaxSlices + j] = __ldcg(pb + ((size_t)h * p.S + j) * (D + 2) + D);
    lj[h * kMaxSlices + j] = __ldcg(pb + ((size_t)h * p.S + j) * (D + 2) + D + 1);
  }
  __syncthreads();
  if (warp < G) {
    const int h = warp;
    float M = -INFINITY;
    for (int j = lane; j < sact; j += 32) M = fmaxf(M, wj[h * kMaxSlices + j]);
    M = warp_max(M);
    __syncwarp();
    for (int j = lane; j < sact; j += 32) wj[h * kMaxSlices + j] = expf(wj[h * kMaxSlices + j] - M);
    __syncwarp();
    if (lane == 0) {  // total in slice order
      float Ls = 0.f;
      for (int j = 0; j < sact; ++j) Ls += lj[h * kMaxSlices + j] * wj[h * kMaxSlices + j];
      lt[h] = Ls;
    }
  }
  __syncthreads();
  constexpr int kB = 16;  // independent loads in flight per thread
#pragma unroll
  for (int i = 0; i < NP; ++i) {
    const int e = tid + i * kThreads;
    if (e < G * D) {
      const int h = e / D, d = e - h * D;
      const float* ph = pb + (size_t)h * p.S * (D + 2) + d;
      float A = 0.f;
      for (int j0 = 0; j0 < sact; j0 += kB) {
        float v[kB];
#pragma unroll
        for (int u = 0; u < kB; ++u) v[u] = (j0 + u < sact) ? __ldcg(ph + (size_t)(j0 + u) * (D + 2)) : 0.f;
#pragma unroll
        for (int u = 0; u < kB; ++u)
          if (j0 + u < sact) A = fmaf(v[u], wj[h * kMaxSlices + j0 + u], A);
      }
      store_out(p, (size_t)m * p.Hq * D + (size_t)(g * G + h) * D + d, A / lt[h]);
    }
  }
  if (tid == 0) p.counters[m * p.Hkv + g] = 0u;
}

template <int D, int G>
cudaError_t launch_dg(const AttnParams& p, int M, bool pdl, cudaStream_t s) {
  using SL = AttnSmem<D, G>;
  static DeviceOnce once;
  cudaError_t ea = device_once(once, [] {
    return cudaFuncSetAttribute(k_attn<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(SL::kBytes));
  });
  if (ea) return ea;
  if (p.S < 1 || p.S > kMaxSlices || M < 1) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.S, p.Hkv, M);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = SL::kBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_attn<D, G>, p);
}

// ------------------------------------------------------------------------
// Prompt rows: one query row per prompt position, one key slice per row
// (P rows already spread the work).  Each warp streams its keys straight from
// the cache, four rows in flight, with lanes across the head dimension and an
// online softmax per head in registers; the warps merge in shared memory.  For
// long key ranges this beats the staged decode kernel, whose chunk barriers
// and shared-memory footprint only pay off when a CTA's slice is short.
constexpr int kRowWarps = 8;
constexpr int kRowUnroll = 4;
#ifndef TF_ROWS_MINB
#define TF_ROWS_MINB 2
#endif

// TF_ROWS_MINB CTAs of 8 warps fit one SM (registers capped to match); the
// eight-head groups keep more registers.
template <int D, int G>
__global__ void __launch_bounds__(kRowWarps * 32, G >= 8 ? 2 : TF_ROWS_MINB) k_attn_rows(const AttnParams p) {
  constexpr int DL = D / 32;  // dims per lane
  const int s = blockIdx.x, g = blockIdx.y, m = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  __shared__ float sm_m[kRowWarps][G], sm_l[kRowWarps][G];
  __shared__ float sm_acc[kRowWarps][G][D];
  __shared__ float sm_f[G][D + 2];
  __shared__ uint32_t sm_last;

  pdl_launch_dependents();
  pdl_wait();
  // Row m is row m % rps of sequence seq_base + m / rps (rps = 0: every row
  // belongs to sequence seq_base).
  const int seq = p.seq_base + (p.rps > 0 ? m / p.rps : 0);
  const int pos = (p.pos_ptr ? p.pos_ptr[seq] : p.pos_fixed) + (p.rps > 0 ? m % p.rps : m);
  const size_t kvo = (size_t)seq * (size_t)p.kv_seq;
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

  const uint16_t* Kg = p.Kc + lane * DL;
  const uint16_t* Vg = p.Vc + lane * DL;
  // element offset of key t's row in the caches: dense, or through the block table
  auto key_off = [&](int t) -> size_t {
    if (!p.kv_tbl) return kvo + ((size_t)g * p.T + t) * D;
    const int page = __ldg(p.kv_tbl + (size_t)seq * p.kv_npp + t / kKvPage);
    return (((size_t)page * p.Hkv + g) * kKvPage + t % kKvPage) * D;
  };
  // Up to kRowUnroll rows of K and V (DL bf16 per lane) from key t0 on.
  auto load_rows = [&](int t0, uint32_t (&kr)[kRowUnroll][DL / 2], uint32_t (&vr)[kRowUnroll][DL / 2]) {
#pragma unroll
    for (int u = 0; u < kRowUnroll; ++u) {
      const int t = t0 + u;
      if (t < k1) {
        const size_t o = key_off(t);
        if constexpr (DL == 4) {
          const uint2 kk = *reinterpret_cast<const uint2*>(Kg + o);
          const uint2 vv = *reinterpret_cast<const uint2*>(Vg + o);
          kr[u][0] = kk.x; kr[u][1] = kk.y;
          vr[u][0] = vv.x; vr[u][1] = vv.y;
        } else {
          kr[u][0] = *reinterpret_cast<const uint32_t*>(Kg + o);
          vr[u][0] = *reinterpret_cast<const uint32_t*>(Vg + o);
        }
      }
    }
  };
  // The next group of rows is loaded before the current one is used, so two
  // groups per warp are in flight.
  uint32_t kn[kRowUnroll][DL / 2], vn[kRowUnroll][DL / 2];
  int t0 = k0 + warp * kRowUnroll;
  if (t0 < k1) load_rows(t0, kn, vn);
  for (; t0 < k1; t0 += kRowWarps * kRowUnroll) {
    uint32_t kr[kRowUnroll][DL / 2], vr[kRowUnroll][DL / 2];
#pragma unroll
    for (int u = 0; u < kRowUnroll; ++u)
#pragma unroll
      for (int i = 0; i < DL / 2; ++i) {
        kr[u][i] = kn[u][i];
        vr[u][i] = vn[u][i];
      }
    if (t0 + kRowWarps * kRowUnroll < k1) load_rows(t0 + kRowWarps * kRowUnroll, kn, vn);
#pragma unroll
    for (int u = 0; u < kRowUnroll; ++u) {
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
  for (int e = tid; e < G * D; e += kRowWarps * 32) {
    const int h = e / D, d = e - h * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kRowWarps; ++w) M = fmaxf(M, sm_m[w][h]);
    float Ls = 0.f, A = 0.f;
#pragma unroll
    for (int w = 0; w < kRowWarps; ++w) {
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
    for (int e = tid; e < G * D; e += kRowWarps * 32) {
      const int h = e / D, d = e - h * D;
      store_out(p, (size_t)m * p.Hq * D + (size_t)(g * G + h) * D + d, sm_f[h][d] / sm_f[h][D + 1]);
    }
    return;
  }

  // Publish this split's partial and take a ticket.
  for (int e = tid; e < G * (D + 2); e += kRowWarps * 32) {
    const int h = e / (D + 2), d = e - h * (D + 2);
    p.part[(((size_t)m * p.Hq + g * G + h) * p.S + s) * (D + 2) + d] = sm_f[h][d];
  }
  __syncthreads();
  if (tid == 0) {
    const uint32_t t = ticket_acq_rel(&p.counters[m * p.Hkv + g]);
    sm_last = (t == static_cast<uint32_t>(sact) - 1u);
  }
  __syncthreads();
  if (!sm_last) return;
  for (int e = tid; e < G * D; e += kRowWarps * 32) {
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
    store_out(p, (size_t)m * p.Hq * D + (size_t)(g * G + h) * D + d, A / Ls);
  }
  if (tid == 0) p.counters[m * p.Hkv + g] = 0u;
}

template <int D, int G>
cudaError_t launch_rows_dg(const AttnParams& p, int M, bool pdl, cudaStream_t s) {
  static DeviceOnce once;
  cudaError_t ea = device_once(once, [] {
    return cudaFuncSetAttribute(k_attn_rows<D, G>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                cudaSharedmemCarveoutMaxShared);
  });
  if (ea) return ea;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.S, p.Hkv, M);
  cfg.blockDim = dim3(kRowWarps * 32);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_attn_rows<D, G>, p);
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

template <int D>
cudaError_t launch_rows_d(const AttnParams& p, int M, bool pdl, cudaStream_t s) {
  switch (p.Hq / p.Hkv) {
    case 1: return launch_rows_dg<D, 1>(p, M, pdl, s);
    case 2: return launch_rows_dg<D, 2>(p, M, pdl, s);
    case 4: return launch_rows_dg<D, 4>(p, M, pdl, s);
    case 8: return launch_rows_dg<D, 8>(p, M, pdl, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_attention_rows(const AttnParams& p, int M, bool pdl, cudaStream_t s) {
  if (p.Hq % p.Hkv) return cudaErrorInvalidValue;
  if (p.D == 128) return launch_rows_d<128>(p, M, pdl, s);
  if (p.D == 64) return launch_rows_d<64>(p, M, pdl, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_attention(const AttnParams& p, int M, bool pdl, cudaStream_t s) {
  if (p.Hq % p.Hkv) return cudaErrorInvalidValue;
  if (p.D == 128) return launch_d<128>(p, M, pdl, s);
  if (p.D == 64) return launch_d<64>(p, M, pdl, s);
  return cudaErrorInvalidValue;
}

// ------------------------------------------------------------------------
// Allocation-free attention entry point.
//
// Some callers cannot allocate device memory at the time they run attention:
// code inside an allocator-free real-time loop, a host that has handed all
// device memory to its own pool, or a plugin that must not touch the global
// CUDA allocator.  tf_op_attention_noalloc runs the same kernel as
// tf_op_attention but takes its scratch (split partials, tickets, error word)
// from a fixed array compiled into this library instead of cudaMalloc.
//
// The array lives in device memory on every GPU that loads the library,
// until the process exits.  Host code cannot use the array's name as a
// device address (on the host it only stands for the symbol), so the device
// address is looked up once per device (and again in a new context on it)
// with cudaGetSymbolAddress, with that device current, on the first call
// there; that first call should happen before any stream capture.  All calls
// share the one array and it keeps what the last call left: tickets and the
// error word are cleared on every call, and calls that overlap on the GPU
// (different streams, or different host threads) race on it.
constexpr size_t kNoAllocPartFloats = 512 * 1024;  // 2 MiB of split partials
constexpr size_t kNoAllocTickets = 1024;
constexpr size_t kNoAllocBytes = kNoAllocPartFloats * 4 + kNoAllocTickets * 4 + 256;
static __device__ __align__(256) unsigned char g_attn_noalloc_scratch[kNoAllocBytes];

namespace {
// Device address of the scratch array on the current device, looked up with
// that device current and kept per device together with the id of the
// context it belongs to: a new context on the device (after cudaDeviceReset)
// looks it up again.
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};
uint64_t g_noalloc_ctx[kMaxDevices] = {};

void* noalloc_scratch(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  const uint64_t ctx = current_context_id();
  if (!g_noalloc_ptr[dev] || ctx == 0 || ctx != g_noalloc_ctx[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_attn_noalloc_scratch) != cudaSuccess) {
      (void)cudaGetLastError();
      return nullptr;
    }
    g_noalloc_ptr[dev] = ptr;
    g_noalloc_ctx[dev] = current_context_id();
  }
  return g_noalloc_ptr[dev];
}
}  // namespace

}  // namespace tf

extern "C" tf_status tf_op_attention_noalloc(const float* q, const uint16_t* K, const uint16_t* V,
                                             int32_t T, int32_t Hq, int32_t Hkv, int32_t D,
                                             int32_t rows, int32_t pos0, int32_t splits, float* out,
                                             void* stream) {
  using namespace tf;
  if (!q || !K || !V || !out || T < 1 || Hq < 1 || Hkv < 1 || rows < 1 || pos0 < 0 ||
      (int64_t)pos0 + rows > T || splits < 1 || splits > 64 || rows > 65535)
    return TF_E_INVAL;
  if ((D != 64 && D != 128) || Hq % Hkv) return TF_E_INVAL;
  const int g = Hq / Hkv;
  if (g != 1 && g != 2 && g != 4 && g != 8) return TF_E_INVAL;
  // Sizes beyond the fixed scratch are refused.
  if ((size_t)rows * Hq * splits * (D + 2) > kNoAllocPartFloats ||
      (size_t)rows * Hkv > kNoAllocTickets)
    return TF_E_INVAL;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return TF_E_CUDA;
  unsigned char* base = static_cast<unsigned char*>(noalloc_scratch(dev));
  if (!base) return TF_E_CUDA;
  float* part = reinterpret_cast<float*>(base);
  uint32_t* cnt = reinterpret_cast<uint32_t*>(base + kNoAllocPartFloats * 4);
  uint32_t* err = cnt + kNoAllocTickets;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(cnt, 0, (size_t)rows * Hkv * 4, s) != cudaSuccess ||
      cudaMemsetAsync(err, 0, 4, s) != cudaSuccess)
    return TF_E_CUDA;
  AttnParams a = {};
  a.q = q;
  a.Kc = K;
  a.Vc = V;
  a.T = T;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.D = D;
  a.pos_fixed = pos0;
  a.S = splits;
  a.part = part;
  a.counters = cnt;
  a.out = out;
  a.err = err;
  if (launch_attention(a, rows, false, s) != cudaSuccess) return TF_E_CUDA;
  uint32_t e = 0;
  if (cudaMemcpyAsync(&e, err, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return TF_E_CUDA;
  if (e & ERR_TIMEOUT) return TF_E_TIMEOUT;
  return e ? TF_E_INVAL : TF_OK;
}
