// Small kernels of the decode path (sm_103a): input-row building, frame
// bookkeeping, codebook-id selection (argmax / exact top-k with a Philox
// draw), weight re-layout and per-row FP8 quantisation, and the prompt
// (prefill) row GEMM on CUDA cores.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <algorithm>

#include "common.cuh"
#include "device_once.h"
#include "epilogue.cuh"
#include "kernels.h"

namespace tf {

namespace {

cudaLaunchConfig_t make_cfg(dim3 grid, dim3 block, size_t smem, bool pdl, cudaStream_t s,
                            cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cfg;
}

__device__ __forceinline__ float block_sum_256(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += red[w];
  return t;
}

// ------------------------------------------------------------------ build
// Row m of a decoder pass's input as the skinny GEMM reads it: x * nw_next
// as bf16 parts and the row's sum of squares (deferred RMSNorm).
__device__ void build_norm_out(const BuildParams& p, int m, const float* xo, float* red) {
  float ss = 0.f;
  for (int k = threadIdx.x; k < p.H; k += blockDim.x) {
    const float v = xo[k];
    ss = fmaf(v, v, ss);
    const float a = v * bf16_to_f32(p.nw_next[k]);
    const uint16_t h = f32_to_bf16(a);
    p.nx_hi[(size_t)m * p.H + k] = h;
    p.nx_lo[(size_t)m * p.H + k] = f32_to_bf16(a - bf16_to_f32(h));
  }
  ss = block_sum_256(ss, red);
  if (threadIdx.x == 0) p.ssq_out[m] = ss;
}

// Rows that start a decoder pass (see BuildMode).  fp32 residual rows; one
// CTA per row.
__global__ void __launch_bounds__(256) k_build(const BuildParams p) {
  __shared__ float red[32];
  pdl_launch_dependents();
  pdl_wait();
  const int tid = threadIdx.x;
  const int m = blockIdx.x;
  float* xo = p.x + (size_t)m * p.H;
  int id;
  if (p.mode == BUILD_FAST1) {
    const int b = m >> 1;
    if ((m & 1) == 0) {
      // h = RMSNorm(slow residual) * w_final: the vector the semantic head reads.
      const float* xs = p.xs + (size_t)b * p.H;
      float ss = 0.f;
      for (int k = tid; k < p.H; k += blockDim.x) ss = fmaf(xs[k], xs[k], ss);
      ss = block_sum_256(ss, red);
      const float rstd = 1.0f / sqrtf(ss / static_cast<float>(p.H) + p.eps);
      for (int k = tid; k < p.H; k += blockDim.x) xo[k] = xs[k] * rstd * bf16_to_f32(p.nw[k]);
      if (p.nx_hi) {
        __syncthreads();
        build_norm_out(p, m, xo, red);
      }
      return;
    }
    id = p.ids[(size_t)b * p.id_stride];
  } else if (p.mode == BUILD_TOKENS) {
    id = p.ids[m];
  } else {
    id = p.ids[(size_t)m * p.id_stride];
  }
  const int pend = (p.mode == BUILD_SLOW && p.pending) ? p.pending[m] : -1;
  if (pend >= 0) {  // the sequence's last prompt id, a text token
    const uint16_t* row = p.table + (size_t)(pend < p.text_rows ? pend : 0) * p.H;
    if (pend >= p.text_rows && tid == 0) atomicOr(p.err, ERR_BAD_ID);
    for (int k = tid; k < p.H; k += blockDim.x) xo[k] = bf16_to_f32(row[k]);
    if (p.nx_hi) build_norm_out(p, m, xo, red);
    return;
  }
  if (id < 0 || id >= p.table_rows) {
    if (tid == 0) atomicOr(p.err, ERR_BAD_ID);
    id = 0;
  }
  const uint16_t* row = p.table + (size_t)(p.row_base + id) * p.H;
  if (p.mode == BUILD_SLOW && p.cb_sum) {
    // the previous frame's codes 1..ncb-1 add their rows, in codebook order
    int cid[16];
    for (int j = 1; j < p.ncb; ++j) {
      int v = p.ids[(size_t)m * p.id_stride + j];
      if (v < 0 || v >= p.cb_rows) {
        if (tid == 0) atomicOr(p.err, ERR_BAD_ID);
        v = 0;
      }
      cid[j] = v;
    }
    for (int k = tid; k < p.H; k += blockDim.x) {
      float acc = bf16_to_f32(row[k]);
      for (int j = 1; j < p.ncb; ++j)
        acc += bf16_to_f32(p.cb_sum[((size_t)(j - 1) * p.cb_rows + cid[j]) * p.H + k]);
      xo[k] = acc;
    }
  } else {
    for (int k = tid; k < p.H; k += blockDim.x) xo[k] = bf16_to_f32(row[k]);
  }
  if (p.nx_hi) build_norm_out(p, m, xo, red);
}

// ------------------------------------------------------------------ q/k norm
// One CTA per (head of q or k, row), one thread per RoPE pair (i, i + D/2):
// RMSNorm over the head's D raw values with the head-dim weight, then the
// rotation at the row's position; q to qout, k (bf16) to the row's KV cache.
__global__ void __launch_bounds__(64) k_qknorm(const GemvParams p) {
  __shared__ float red[2];
  pdl_launch_dependents();
  pdl_wait();
  const int half = p.head_dim >> 1, i = threadIdx.x;
  const int hq = p.q_dim / p.head_dim;
  const int h = blockIdx.x, m = blockIdx.y;
  const bool isq = h < hq;
  const int hh = isq ? h : h - hq;
  const size_t pair = (size_t)(isq ? 0 : p.q_dim >> 1) + (size_t)hh * half + i;
  const float* r = p.qk_raw + (size_t)m * (p.q_dim + p.kv_dim) + 2 * pair;
  const float v0 = r[0], v1 = r[1];
  float ss = warp_sum(fmaf(v0, v0, v1 * v1));
  if ((i & 31) == 0) red[i >> 5] = ss;
  __syncthreads();
  ss = half > 32 ? red[0] + red[1] : red[0];
  const float rstd = 1.0f / sqrtf(ss / static_cast<float>(p.head_dim) + p.eps);
  const uint16_t* w = isq ? p.q_norm : p.k_norm;
  const float a = v0 * rstd * bf16_to_f32(w[i]);
  const float b = v1 * rstd * bf16_to_f32(w[i + half]);
  const int pos = row_pos(p, m);
  if (pos < 0 || pos >= p.T) {
    if (i == 0) atomicOr(p.err, ERR_BAD_POS);
    return;
  }
  const float2 cs = __ldg(&p.rope[(size_t)pos * half + i]);
  const float r0 = a * cs.x - b * cs.y;
  const float r1 = b * cs.x + a * cs.y;
  if (isq) {
    float* q = p.qout + (size_t)m * p.q_dim + (size_t)hh * p.head_dim;
    q[i] = r0;
    q[i + half] = r1;
  } else {
    uint16_t* k = p.Kc + kv_index(p.kv_tbl, p.kv_npp, p.kv_dim / p.head_dim, p.T, p.kv_seq, row_seq(p, m),
                                  hh, pos, p.head_dim);
    k[i] = f32_to_bf16(r0);
    k[i + half] = f32_to_bf16(r1);
  }
}

// ------------------------------------------------------------------ frame end
__global__ void k_frame_end(const FrameEndParams p) {
  pdl_launch_dependents();
  pdl_wait();
  if (threadIdx.x == 0) {
    for (int b = 0; b < p.nseq; ++b) {
      if (p.active && !p.active[b]) continue;  // an idle slot stays where it is
      if (p.fb_ring) {  // the ids fed back this frame, for later repetition windows
        const int slot = p.frame_index[b] % kRepRing;
        for (int c = 0; c < p.ncb; ++c)
          p.fb_ring[((size_t)b * kRepRing + slot) * kRepIds + c] = p.fb[(size_t)b * p.sel_stride + c];
      }
      p.pos[b] += p.advance;
      p.frame_index[b] += 1;
      if (p.pending) p.pending[b] = -1;
    }
    if (p.hist) {
      const int i = *p.hist_idx;
      if (i < p.hist_cap) {
        for (int b = 0; b < p.nseq; ++b)
          for (int c = 0; c < p.ncb; ++c)
            p.hist[((size_t)i * p.nseq + b) * p.ncb + c] = p.sel[(size_t)b * p.sel_stride + c];
        *p.hist_idx = i + 1;
      }
    }
  }
}

// ------------------------------------------------------------------ select
// exp32 and Philox4x32-10 exactly as the selection rule defines them (each
// step one IEEE float32 operation with round-to-nearest; no contraction).
// Constants: log2(e), ln2 split Cody-Waite style into a 12-significant-bit
// head and a float32 tail, and float32(1/k!) for k = 0..7.
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

constexpr int kSelThreads = 1024;
constexpr int kSelMaxVocab = 8192;
constexpr int kSelMaxK = 256;

__device__ __forceinline__ uint32_t sel_key(float z) {
  if (z == 0.f) z = 0.f;  // -0 and +0 are equal logits
  return float_order_key(z);
}

// One CTA per row of logits.  Exact top-k: a 4-pass radix select finds the
// k-th largest value; candidates are the larger values plus the lowest-index
// copies of that value; a rank count orders them by (value desc, index asc);
// weights, running sums and the draw follow the selection rule.
__global__ void __launch_bounds__(kSelThreads) k_select(const SelectParams p) {
  __shared__ uint32_t keys[kSelMaxVocab];
  __shared__ uint32_t hist[256];
  __shared__ unsigned long long wbest[kSelThreads / 32];
  __shared__ uint32_t s_prefix, s_remaining, s_ncand;
  __shared__ int cand_idx[kSelMaxK];
  __shared__ uint32_t cand_key[kSelMaxK];
  __shared__ int sort_idx[kSelMaxK];
  __shared__ float sort_z[kSelMaxK];
  __shared__ float wts[kSelMaxK];
  __shared__ uint32_t rep_bits[kSelMaxVocab / 32];   // ids of the repetition window

  pdl_launch_dependents();
  pdl_wait();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = blockIdx.x;
  const float* z = p.logits + (size_t)row * p.ld;
  const int V = p.vocab;
  const uint32_t cb = static_cast<uint32_t>(p.seq_rows ? p.codebook0 : p.codebook0 + row);
  const uint32_t sq = static_cast<uint32_t>(p.seq_rows ? p.sequence + row : p.sequence);
  const int frame = p.frame_ptr ? p.frame_ptr[sq] : p.frame;

  // Repetition window: the ids this codebook fed back in the previous
  // rep_window frames of the sequence (or the explicit list), as a bitmap.
  const bool rep = (p.recent && p.n_recent > 0) || (p.fb_ring && p.rep_window > 0);
  if (rep) {
    for (int w = tid; w < kSelMaxVocab / 32; w += kSelThreads) rep_bits[w] = 0u;
    __syncthreads();
    int id = -1;
    if (p.recent) {
      if (tid < p.n_recent) id = p.recent[(size_t)row * p.n_recent + tid];
    } else if (tid < p.rep_window && frame - 1 - tid >= 0) {
      const int t = frame - 1 - tid;  // one of the previous rep_window frames
      id = p.fb_ring[((size_t)sq * kRepRing + t % kRepRing) * kRepIds + cb];
    }
    if (id >= 0 && id < V) atomicOr(&rep_bits[id >> 5], 1u << (id & 31));
    __syncthreads();
  }
  // logit i as the selection sees it (repetition penalty applied)
  auto zsel = [&](int i) {
    float v = z[i];
    if (rep && ((rep_bits[i >> 5] >> (i & 31)) & 1u))
      v = v > 0.f ? __fdiv_rn(v, p.rep_penalty) : __fmul_rn(v, p.rep_penalty);
    return v;
  };

  bool nan = false;
  unsigned long long best = 0ull;
  for (int i = tid; i < V; i += kSelThreads) {
    const float v = zsel(i);
    nan |= (v != v);
    keys[i] = sel_key(v);
    const unsigned long long k = pack_key(v, i);
    best = k > best ? k : best;
  }
  if (nan) atomicOr(p.err, ERR_NAN);
  int pick;
  if (p.top_k <= 1) {
    best = warp_max_u64(best);
    if (lane == 0) wbest[warp] = best;
    __syncthreads();
    if (tid == 0) {
      unsigned long long b = 0ull;
      for (int w = 0; w < kSelThreads / 32; ++w) b = wbest[w] > b ? wbest[w] : b;
      s_prefix = 0xFFFFFFFFu - static_cast<uint32_t>(b & 0xFFFFFFFFull);
    }
    __syncthreads();
    pick = static_cast<int>(s_prefix);
  } else {
    const int k = min(p.top_k, V);
    if (tid == 0) {
      s_prefix = 0u;
      s_remaining = static_cast<uint32_t>(k);
      s_ncand = 0u;
    }
    uint32_t mask = 0u;
    for (int shift = 24; shift >= 0; shift -= 8) {
      if (tid < 256) hist[tid] = 0u;
      __syncthreads();
      const uint32_t prefix = s_prefix;
      for (int i = tid; i < V; i += kSelThreads)
        if ((keys[i] & mask) == prefix) atomicAdd(&hist[(keys[i] >> shift) & 0xFFu], 1u);
      __syncthreads();
      if (tid == 0) {
        uint32_t rem = s_remaining, cum = 0u;
        int b = 255;
        for (; b > 0; --b) {
          if (cum + hist[b] >= rem) break;
          cum += hist[b];
        }
        s_remaining = rem - cum;
        s_prefix = prefix | (static_cast<uint32_t>(b) << shift);
      }
      mask |= 0xFFu << shift;
      __syncthreads();
    }
    const uint32_t T = s_prefix;       // k-th largest key
    const uint32_t need_eq = s_remaining;  // copies of T to take, lowest index first
    for (int i = tid; i < V; i += kSelThreads) {
      if (keys[i] > T) {
        const uint32_t slot = atomicAdd(&s_ncand, 1u);
        cand_idx[slot] = i;
        cand_key[slot] = keys[i];
      }
    }
    __syncthreads();
    if (warp == 0) {
      uint32_t taken = 0u;
      for (int base = 0; base < V && taken < need_eq; base += 32) {
        const int i = base + lane;
        const bool eq = i < V && keys[i] == T;
        const uint32_t bal = __ballot_sync(0xFFFFFFFFu, eq);
        const uint32_t before = __popc(bal & ((1u << lane) - 1u));
        if (eq && taken + before < need_eq) {
          const uint32_t slot = s_ncand + taken + before;
          cand_idx[slot] = i;
          cand_key[slot] = T;
        }
        taken += __popc(bal);
      }
    }
    __syncthreads();
    // Rank: order by (key desc, index asc).
    if (tid < k) {
      const uint32_t ki = cand_key[tid];
      const int ii = cand_idx[tid];
      int r = 0;
      for (int j = 0; j < k; ++j) {
        const uint32_t kj = cand_key[j];
        r += (kj > ki) || (kj == ki && cand_idx[j] < ii);
      }
      sort_idx[r] = ii;
      sort_z[r] = zsel(ii);
    }
    __syncthreads();
    if (tid < k) {
      float d = __fsub_rn(sort_z[tid], sort_z[0]);
      if (p.temperature != 1.0f) d = __fdiv_rn(d, p.temperature);
      wts[tid] = exp32(d);
    }
    __syncthreads();
    if (tid == 0) {
      float S = 0.f;
      for (int j = 0; j < k; ++j) S = __fadd_rn(S, wts[j]);
      // nucleus: the shortest prefix whose running sum reaches top_p * S
      int nk = k;
      float Sk = S;
      if (p.top_p < 1.0f) {
        const float tp = __fmul_rn(p.top_p, S);
        float acc = 0.f;
        for (int j = 0; j < k; ++j) {
          acc = __fadd_rn(acc, wts[j]);
          if (acc >= tp) {
            nk = j + 1;
            Sk = acc;
            break;
          }
        }
      }
      const uint32_t w0 = philox_w0(static_cast<uint32_t>(frame), cb, sq, 0u, p.key0, p.key1);
      const float u = __fmul_rn(static_cast<float>(w0 >> 8), 5.9604644775390625e-8f);  // 2^-24
      const float t = __fmul_rn(u, Sk);
      int pk = nk - 1;
      float cum = 0.f;
      for (int j = 0; j < nk; ++j) {
        cum = __fadd_rn(cum, wts[j]);
        if (t < cum) {
          pk = j;
          break;
        }
      }
      s_prefix = static_cast<uint32_t>(sort_idx[pk]);
    }
    __syncthreads();
    pick = static_cast<int>(s_prefix);
  }
  if (tid == 0) {
    const size_t slot = p.seq_rows ? (size_t)row * p.id_stride : (size_t)row;
    p.sel[slot] = pick;
    if (p.fb) p.fb[slot] = (p.forced_on && *p.forced_on) ? p.forced[slot] : pick;
  }
}

// ------------------------------------------------------------------ pack
__device__ __forceinline__ int64_t map_row(const PackParams& p, int64_t s) {
  if (p.map == MAP_GATE) return 2 * s;
  if (p.map == MAP_UP) return 2 * s + 1;
  if (p.map == MAP_QKV && s < p.q_dim + p.kv_dim) {
    const int64_t base = s < p.q_dim ? 0 : p.q_dim;
    const int64_t r = s - base;
    const int hd = p.head_dim, half = hd >> 1;
    const int64_t h = r / hd, d = r - h * hd;
    const int64_t i = d % half, hi = d / half;
    return base + 2 * (h * half + i) + hi;
  }
  return s;
}

// e2m1 code (0..15) of a float32 in [-6, 6], round to nearest with ties to
// the even code: the magnitude code counts the midpoints 0.25, 0.75, 1.25,
// 1.75, 2.5, 3.5, 5 that |q| passes, a tie going to the even neighbour.
__device__ __forceinline__ uint32_t e2m1_rne(float q) {
  const float a = fabsf(q);
  const uint32_t m = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) +
                     (a >= 3.5f) + (a > 5.0f);
  return m | ((__float_as_uint(q) >> 31) << 3);
}

// Block-scaled 4-bit row (the tuna-fish README's nvfp4 weight format, read
// after NVIDIA's NVFP4 layout with a per-row float32 scale): s_row =
// amax / (6 * 448) (1 for a zero row); per 16-element block s_b =
// e4m3_RNE(min(amax_block / (6 * s_row), 448)); code = e2m1_RNE(clamp(w /
// (value(s_b) * s_row), +-6)), 0 where s_b is 0; every step one float32
// operation in that order.  dst row: K/2 code bytes, then K/16 scale bytes.
__device__ void nvfp4_row(const PackParams& p, int64_t s, int64_t d, float* red) {
  const int tid = threadIdx.x;
  const uint16_t* w = reinterpret_cast<const uint16_t*>(p.src) + s * p.cols;
  float amax = 0.f;
  for (int64_t i = tid; i < p.cols; i += blockDim.x) amax = fmaxf(amax, fabsf(bf16_to_f32(w[i])));
  amax = warp_max(amax);
  __syncthreads();
  if ((tid & 31) == 0) red[tid >> 5] = amax;
  __syncthreads();
  amax = 0.f;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) amax = fmaxf(amax, red[i]);
  const float s_row = amax == 0.f ? 1.0f : __fdiv_rn(amax, 2688.0f);
  const float denom = __fmul_rn(6.0f, s_row);
  uint8_t* out = p.dst + d * (p.cols / 2 + p.cols / 16);
  for (int64_t b = tid; b < p.cols / 16; b += blockDim.x) {
    float v[16];
    float bm = 0.f;
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      v[e] = bf16_to_f32(w[b * 16 + e]);
      bm = fmaxf(bm, fabsf(v[e]));
    }
    const float bs = fminf(__fdiv_rn(bm, denom), 448.0f);
    const uint8_t sb = static_cast<uint8_t>(
        __nv_cvt_float2_to_fp8x2(make_float2(bs, 0.f), __NV_SATFINITE, __NV_E4M3) & 0xFF);
    const float sbv = e4m3x2_to_f32x2(sb).x;
    const float dd = __fmul_rn(sbv, s_row);
    uint32_t packed[2] = {0u, 0u};
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      float q = dd == 0.f ? 0.f : __fdiv_rn(v[e], dd);
      q = fminf(fmaxf(q, -6.0f), 6.0f);
      packed[e >> 3] |= e2m1_rne(q) << (4 * (e & 7));
    }
    reinterpret_cast<uint2*>(out)[b] = make_uint2(packed[0], packed[1]);
    out[p.cols / 2 + b] = sb;
  }
  if (tid == 0) p.dst_scale[d] = s_row;
}

// One CTA per source row.  mode 0: copy bf16; mode 1: quantise bf16 -> e4m3
// with a per-row scale; mode 2: copy e4m3 codes and their scale.
__global__ void __launch_bounds__(256) k_pack(const PackParams p) {
  __shared__ float red[32];
  const int64_t s = blockIdx.x;
  const int64_t d = map_row(p, s);
  const int tid = threadIdx.x;
  if (p.mode == 0) {
    const uint4* src = reinterpret_cast<const uint4*>(p.src + s * p.cols * 2);
    uint4* dst = reinterpret_cast<uint4*>(p.dst + d * p.cols * 2);
    for (int64_t i = tid; i < p.cols / 8; i += blockDim.x) dst[i] = src[i];
    return;
  }
  if (p.mode == 2) {
    // Codes handed over as they are: NaN codes (S.1111.111) are refused, since
    // the GEMV's decode reads every code as a finite number.
    const uint4* src = reinterpret_cast<const uint4*>(p.src + s * p.cols);
    uint4* dst = reinterpret_cast<uint4*>(p.dst + d * p.cols);
    uint32_t nan = 0;
    for (int64_t i = tid; i < p.cols / 16; i += blockDim.x) {
      const uint4 v = src[i];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) nan |= ((w[k] & 0x7F7F7F7Fu) + 0x01010101u) & 0x80808080u;
      dst[i] = v;
    }
    if (nan && p.err) atomicOr(p.err, ERR_BAD_CODE);
    if (tid == 0) p.dst_scale[d] = p.src_scale[s];
    return;
  }
  if (p.mode == 4) {
    nvfp4_row(p, s, d, red);
    return;
  }
  // Per-row symmetric FP8 (drbaph s2-pro-fp8 model card, "Quantization
  // Details"): scale = amax / 448 (IEEE float32 division), 1 for a zero row;
  // code = e4m3 round-to-nearest-even of clamp(w / scale, -448, 448).
  const uint16_t* w = reinterpret_cast<const uint16_t*>(p.src) + s * p.cols;
  float amax = 0.f;
  for (int64_t i = tid; i < p.cols; i += blockDim.x) amax = fmaxf(amax, fabsf(bf16_to_f32(w[i])));
  amax = warp_max(amax);
  __syncthreads();
  if ((tid & 31) == 0) red[tid >> 5] = amax;
  __syncthreads();
  amax = 0.f;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) amax = fmaxf(amax, red[i]);
  const float scale = amax == 0.f ? 1.0f : __fdiv_rn(amax, 448.0f);
  uint8_t* q = p.dst + d * p.cols;
  for (int64_t i = 2 * tid; i < p.cols; i += 2 * blockDim.x) {
    float r0 = __fdiv_rn(bf16_to_f32(w[i]), scale);
    float r1 = __fdiv_rn(bf16_to_f32(w[i + 1]), scale);
    r0 = fminf(fmaxf(r0, -448.0f), 448.0f);
    r1 = fminf(fmaxf(r1, -448.0f), 448.0f);
    // __nv_cvt_float2_to_fp8x2: .x -> low byte, .y -> high byte.
    const __nv_fp8x2_storage_t v = __nv_cvt_float2_to_fp8x2(make_float2(r0, r1), __NV_SATFINITE, __NV_E4M3);
    *reinterpret_cast<__nv_fp8x2_storage_t*>(q + i) = v;
  }
  if (tid == 0) p.dst_scale[d] = scale;
}

// ------------------------------------------------------------------ prefill
__global__ void __launch_bounds__(256) k_rmsnorm_rows(const float* x, const uint16_t* w, float* a,
                                                      int H, float eps) {
  __shared__ float red[32];
  const int m = blockIdx.x;
  const float* xm = x + (size_t)m * H;
  float ss = 0.f;
  for (int k = threadIdx.x; k < H; k += blockDim.x) ss = fmaf(xm[k], xm[k], ss);
  ss = block_sum_256(ss, red);
  const float rstd = 1.0f / sqrtf(ss / static_cast<float>(H) + eps);
  for (int k = threadIdx.x; k < H; k += blockDim.x)
    a[(size_t)m * H + k] = xm[k] * rstd * bf16_to_f32(w[k]);
}

// RMSNorm rows straight into the bf16 hi / lo parts a tensor-core prompt GEMM
// reads: a = x * rstd * w (per element the same float operations as
// k_rmsnorm_rows), hi = bf16(a), lo = bf16(a - hi); one CTA per row.  Rows of
// a multiple of 4 elements move as 16-byte loads and 8-byte stores.
__device__ __forceinline__ uint32_t split_pair(float a0, float a1, uint32_t* lo) {
  const uint16_t h0 = f32_to_bf16(a0), h1 = f32_to_bf16(a1);
  const uint16_t l0 = f32_to_bf16(a0 - bf16_to_f32(h0)), l1 = f32_to_bf16(a1 - bf16_to_f32(h1));
  *lo = static_cast<uint32_t>(l0) | (static_cast<uint32_t>(l1) << 16);
  return static_cast<uint32_t>(h0) | (static_cast<uint32_t>(h1) << 16);
}

__global__ void __launch_bounds__(256) k_rmsnorm_split(const float* x, const uint16_t* w,
                                                       uint16_t* hi, uint16_t* lo, int H, float eps) {
  __shared__ float red[32];
  const int m = blockIdx.x;
  const float* xm = x + (size_t)m * H;
  const bool v4 = (H & 3) == 0;
  float ss = 0.f;
  if (v4) {
    const float4* x4 = reinterpret_cast<const float4*>(xm);
    for (int k = threadIdx.x; k < (H >> 2); k += blockDim.x) {
      const float4 v = x4[k];
      ss = fmaf(v.x, v.x, ss);
      ss = fmaf(v.y, v.y, ss);
      ss = fmaf(v.z, v.z, ss);
      ss = fmaf(v.w, v.w, ss);
    }
  } else {
    for (int k = threadIdx.x; k < H; k += blockDim.x) ss = fmaf(xm[k], xm[k], ss);
  }
  ss = block_sum_256(ss, red);
  const float rstd = 1.0f / sqrtf(ss / static_cast<float>(H) + eps);
  if (v4) {
    const float4* x4 = reinterpret_cast<const float4*>(xm);
    const uint2* w4 = reinterpret_cast<const uint2*>(w);
    uint2* h4 = reinterpret_cast<uint2*>(hi + (size_t)m * H);
    uint2* l4 = reinterpret_cast<uint2*>(lo + (size_t)m * H);
    for (int k = threadIdx.x; k < (H >> 2); k += blockDim.x) {
      const float4 v = x4[k];
      const uint2 wk = w4[k];
      uint2 hv, lv;
      hv.x = split_pair(v.x * rstd * bf16_lo(wk.x), v.y * rstd * bf16_hi(wk.x), &lv.x);
      hv.y = split_pair(v.z * rstd * bf16_lo(wk.y), v.w * rstd * bf16_hi(wk.y), &lv.y);
      h4[k] = hv;
      l4[k] = lv;
    }
  } else {
    for (int k = threadIdx.x; k < H; k += blockDim.x) {
      const float a = xm[k] * rstd * bf16_to_f32(w[k]);
      const uint16_t h = f32_to_bf16(a);
      hi[(size_t)m * H + k] = h;
      lo[(size_t)m * H + k] = f32_to_bf16(a - bf16_to_f32(h));
    }
  }
}

// Rows for a skinny GEMM with a deferred RMSNorm: x[m] * w as bf16 hi / lo
// parts and the row's sum of squares; one CTA per row.
__global__ void __launch_bounds__(256) k_rows_prep(const float* x, int ldx, int K,
                                                   const uint16_t* w, uint16_t* hi, uint16_t* lo,
                                                   float* ssq) {
  __shared__ float red[32];
  pdl_launch_dependents();
  pdl_wait();
  const int m = blockIdx.x;
  const float* xm = x + (size_t)m * ldx;
  float ss = 0.f;
  for (int k = threadIdx.x; k < K; k += blockDim.x) {
    const float v = xm[k];
    ss = fmaf(v, v, ss);
    const float a = w ? v * bf16_to_f32(w[k]) : v;
    const uint16_t h = f32_to_bf16(a);
    hi[(size_t)m * K + k] = h;
    lo[(size_t)m * K + k] = f32_to_bf16(a - bf16_to_f32(h));
  }
  ss = block_sum_256(ss, red);
  if (ssq && threadIdx.x == 0) ssq[m] = ss;
}

// C[m][n] = sum_k A[m][k] W[n][k], 64x64 tile per CTA, 4x4 per thread,
// k-steps of 32 through shared memory; epilogue as the decode GEMV's.
template <int WT>
__global__ void __launch_bounds__(256) k_gemm_rows(const GemvParams p, int M) {
  constexpr int BM = 64, BN = 64, BK = 32;
  __shared__ __align__(16) float As[BK][BM + 4];
  __shared__ __align__(16) float Ws[BK][BN + 4];
  const int tid = threadIdx.x;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  const int tm = tid >> 4, tn = tid & 15;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < p.K; k0 += BK) {
    // A tile: 64 x 32 fp32 (8 per thread)
    for (int e = tid; e < BM * BK; e += 256) {
      const int r = e / BK, c = e - r * BK;
      const int m = m0 + r;
      As[c][r] = m < M ? p.x[(size_t)m * p.ldx + k0 + c] : 0.f;
    }
    // W tile: 64 rows x 32 cols
    if (WT == 0) {
      const int r = tid >> 2, q = tid & 3;  // 4 chunks of 8 per row
      const int n = n0 + r;
      float v[8] = {};
      if (n < p.N) {
        const uint4 w = *reinterpret_cast<const uint4*>(p.W + ((size_t)n * p.K + k0 + q * 8) * 2);
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
        for (int i = 0; i < 4; ++i) {
          v[2 * i] = bf16_lo(u[i]);
          v[2 * i + 1] = bf16_hi(u[i]);
        }
      }
      for (int i = 0; i < 8; ++i) Ws[q * 8 + i][r] = v[i];
    } else if (tid < 128) {
      const int r = tid >> 1, q = tid & 1;  // 2 chunks of 16 per row
      const int n = n0 + r;
      float v[16] = {};
      if (n < p.N) {
        const uint4 w = *reinterpret_cast<const uint4*>(p.W + (size_t)n * p.K + k0 + q * 16);
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
        for (int i = 0; i < 4; ++i) {
          const float2 lo = e4m3x2_to_f32x2(static_cast<uint16_t>(u[i] & 0xFFFFu));
          const float2 hi = e4m3x2_to_f32x2(static_cast<uint16_t>(u[i] >> 16));
          v[4 * i] = lo.x;
          v[4 * i + 1] = lo.y;
          v[4 * i + 2] = hi.x;
          v[4 * i + 3] = hi.y;
        }
      }
      for (int i = 0; i < 16; ++i) Ws[q * 16 + i][r] = v[i];
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < BK; ++kk) {
      const float4 av = *reinterpret_cast<const float4*>(&As[kk][tm * 4]);
      const float4 wv = *reinterpret_cast<const float4*>(&Ws[kk][tn * 4]);
      const float a4[4] = {av.x, av.y, av.z, av.w};
      const float w4[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a4[i], w4[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + tm * 4 + i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; j += 2) {
      const int n = n0 + tn * 4 + j;
      if (n >= p.N) continue;
      float v0 = acc[i][j], v1 = acc[i][j + 1];
      if (p.scale) {
        v0 *= p.scale[n];
        v1 *= p.scale[n + 1];
      }
      if (p.epi == EPI_QKV) {
        epi_qkv_pair(p, m, n >> 1, v0, v1);
      } else if (p.epi == EPI_SWIGLU) {
        epi_swiglu(p, m, n >> 1, v0, v1);
      } else if (p.epi == EPI_RESID) {
        p.out[(size_t)m * p.ldo + n] += v0;
        p.out[(size_t)m * p.ldo + n + 1] += v1;
      } else {
        p.out[(size_t)m * p.ldo + n] = v0;
        p.out[(size_t)m * p.ldo + n + 1] = v1;
      }
    }
  }
}

}  // namespace

// Full shared-memory carveout for the small decode kernels too (see the
// GEMV): kernels with equal carveouts can share an SM under PDL.
template <typename K>
cudaError_t carveout(DeviceOnce& once, K kernel) {
  return device_once(once, [kernel] {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                cudaSharedmemCarveoutMaxShared);
  });
}

cudaError_t launch_build(const BuildParams& p, bool pdl, cudaStream_t s) {
  static DeviceOnce once;
  if (cudaError_t e = carveout(once, k_build)) return e;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(p.M), dim3(256), 0, pdl, s, attr);
  return cudaLaunchKernelEx(&cfg, k_build, p);
}

cudaError_t launch_qknorm(const GemvParams& p, int M, bool pdl, cudaStream_t s) {
  if (p.head_dim != 64 && p.head_dim != 128) return cudaErrorInvalidValue;
  static DeviceOnce once;
  if (cudaError_t e = carveout(once, k_qknorm)) return e;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3((p.q_dim + p.kv_dim) / p.head_dim, M), dim3(p.head_dim / 2),
                                    0, pdl, s, attr);
  return cudaLaunchKernelEx(&cfg, k_qknorm, p);
}

cudaError_t launch_frame_end(const FrameEndParams& p, bool pdl, cudaStream_t s) {
  static DeviceOnce once;
  if (cudaError_t e = carveout(once, k_frame_end)) return e;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(1), dim3(32), 0, pdl, s, attr);
  return cudaLaunchKernelEx(&cfg, k_frame_end, p);
}

cudaError_t launch_select(const SelectParams& p, bool pdl, cudaStream_t s) {
  if (p.vocab < 1 || p.vocab > kSelMaxVocab || p.top_k > kSelMaxK || p.n < 1 ||
      p.rep_window > kRepRing || p.n_recent > kSelThreads)
    return cudaErrorInvalidValue;
  static DeviceOnce once;
  if (cudaError_t e = carveout(once, k_select)) return e;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(p.n), dim3(kSelThreads), 0, pdl, s, attr);
  return cudaLaunchKernelEx(&cfg, k_select, p);
}

// Block-scaled 4-bit rows -> bf16 bits of e2m1 x block scale (exact: at
// most 2 + 4 significant bits, within bf16's range), one thread per block.
__global__ void k_nvfp4_to_bf16(const uint8_t* q, uint16_t* out, int N, int K) {
  const int nb = K / 16;
  const int rb = K / 2 + K / 16;
  for (size_t t = (size_t)blockIdx.x * blockDim.x + threadIdx.x; t < (size_t)N * nb;
       t += (size_t)gridDim.x * blockDim.x) {
    const size_t r = t / nb, b = t - r * nb;
    const uint8_t* row = q + r * rb;
    const uint2 w = reinterpret_cast<const uint2*>(row)[b];
    const float sbv = e4m3x2_to_f32x2(row[K / 2 + b]).x;
    const uint32_t v[2] = {w.x, w.y};
    uint16_t* o = out + r * K + b * 16;
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const uint32_t c = (v[e >> 3] >> (4 * (e & 7))) & 0xFu;
      const uint32_t mag = c & 7u;
      // e2m1 value: exponent field 0 -> m / 2, else (1 + m / 2) * 2^(e - 1)
      const float val = (mag < 2u) ? 0.5f * static_cast<float>(mag)
                                   : ldexpf(1.0f + 0.5f * static_cast<float>(mag & 1u),
                                            static_cast<int>(mag >> 1) - 1);
      o[e] = f32_to_bf16((c & 8u) ? -(val * sbv) : val * sbv);
    }
  }
}

cudaError_t launch_nvfp4_to_bf16(const uint8_t* q, uint16_t* out, int N, int K, cudaStream_t s) {
  const size_t n = (size_t)N * (K / 16);
  const int grid = static_cast<int>(std::min<size_t>((n + 255) / 256, 8192));
  k_nvfp4_to_bf16<<<grid, 256, 0, s>>>(q, out, N, K);
  return cudaGetLastError();
}

cudaError_t launch_pack(const PackParams& p, cudaStream_t s) {
  if (p.rows <= 0) return cudaSuccess;
  k_pack<<<static_cast<unsigned>(p.rows), 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm_rows(const float* x, const uint16_t* w, float* a, int M, int H,
                                float eps, cudaStream_t s) {
  k_rmsnorm_rows<<<M, 256, 0, s>>>(x, w, a, H, eps);
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm_split(const float* x, const uint16_t* w, uint16_t* hi, uint16_t* lo,
                                 int M, int H, float eps, cudaStream_t s) {
  if (M < 1) return cudaSuccess;
  k_rmsnorm_split<<<M, 256, 0, s>>>(x, w, hi, lo, H, eps);
  return cudaGetLastError();
}

cudaError_t launch_rows_prep(const float* x, int ldx, int M, int K, const uint16_t* w,
                             uint16_t* hi, uint16_t* lo, float* ssq, bool pdl, cudaStream_t s) {
  if (M < 1) return cudaSuccess;
  static DeviceOnce once;
  if (cudaError_t e = carveout(once, k_rows_prep)) return e;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(M), dim3(256), 0, pdl, s, attr);
  return cudaLaunchKernelEx(&cfg, k_rows_prep, x, ldx, K, w, hi, lo, ssq);
}

cudaError_t launch_gemm_rows(const GemvParams& p, int wt, int M, cudaStream_t s) {
  if (p.K % 32) return cudaErrorInvalidValue;
  dim3 grid((p.N + 63) / 64, (M + 63) / 64);
  if (wt == 0) k_gemm_rows<0><<<grid, 256, 0, s>>>(p, M);
  else k_gemm_rows<1><<<grid, 256, 0, s>>>(p, M);
  return cudaGetLastError();
}

}  // namespace tf
