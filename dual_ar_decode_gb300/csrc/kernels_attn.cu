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
#include <mutex>

#include "../../include/tf.h"
#include "common.cuh"
#include "kernels.h"

namespace tf {

namespace {

constexpr int kWarps = 8;
constexpr int kUnroll = 4;
constexpr int kMinKeys = 32;

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
  // Row m is row m % rps of sequence m / rps (rps = 0: one sequence).
  const int pos = (p.pos_ptr ? p.pos_ptr[0] : p.pos_fixed) + (p.rps > 0 ? m % p.rps : m);
  const size_t kvo = p.rps > 0 ? static_cast<size_t>(m / p.rps) * static_cast<size_t>(p.kv_seq) : 0;
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

  const uint16_t* Kg = p.Kc + kvo + (size_t)g * p.T * D + lane * DL;
  const uint16_t* Vg = p.Vc + kvo + (size_t)g * p.T * D + lane * DL;
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
      store_out(p, (size_t)m * p.Hq * D + (size_t)(g * G + h) * D + d, sm_f[h][d] / sm_f[h][D + 1]);
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
    store_out(p, (size_t)m * p.Hq * D + (size_t)(g * G + h) * D + d, A / Ls);
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
// address is looked up once per device with cudaGetSymbolAddress, with that
// device current, on the first call on it; that first call should happen
// before any stream capture.  All calls share the one array and it keeps
// what the last call left: tickets and the error word are cleared on every
// call, and calls that overlap on the GPU (different streams, or different
// host threads) race on it.
constexpr size_t kNoAllocPartFloats = 512 * 1024;  // 2 MiB of split partials
constexpr size_t kNoAllocTickets = 1024;
constexpr size_t kNoAllocBytes = kNoAllocPartFloats * 4 + kNoAllocTickets * 4 + 256;
static __device__ __align__(256) unsigned char g_attn_noalloc_scratch[kNoAllocBytes];

namespace {
constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kNoAllocMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once).
void* noalloc_scratch(int dev) {
  if (dev < 0 || dev >= kNoAllocMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_attn_noalloc_scratch) != cudaSuccess) {
      (void)cudaGetLastError();
      return nullptr;
    }
    g_noalloc_ptr[dev] = ptr;
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
  return e ? TF_E_INVAL : TF_OK;
}
