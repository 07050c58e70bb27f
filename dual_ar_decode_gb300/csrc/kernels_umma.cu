// Tensor-core (tcgen05 / TMEM) GEMM for the prompt (sm_103a).
//
// Prefill runs every prompt token through the slow decoder (tuna-fish README,
// "Inference speedtest": prefill is reported separately in tokens/s); its
// linear layers are dense contractions C[m][n] = sum_k A[m][k] W[n][k] with
// m over prompt tokens, so they belong on the 5th-generation tensor cores:
//   * the work is split into units (a 128-row x GBN-column output tile,
//     GBN = 128 or 256, and a slice of K); warp 0 streams 64-wide K slices
//     of the activation tile and the weight tile into a 3- or 4-stage
//     shared-memory ring with TMA tensor copies (128-byte swizzle),
//     completion counted on mbarriers;
//   * warp 1 owns the TMEM accumulator(s) (fp32, GBN columns each) and
//     issues tcgen05.mma kind::f16 (bf16 x bf16 -> fp32), four K=16 steps
//     per slice; tcgen05.commit frees a stage once the MMAs reading it are
//     done, and marks a unit's accumulator full after its last slice;
//   * the activations enter as two bf16 parts (hi = bf16(a), lo = bf16(a -
//     hi)) multiplied by the same weight slice, so the products keep about 16
//     significant bits of the fp32 activations instead of 8;
//   * warps 2-5 wait for a full accumulator, read it with tcgen05.ld (each
//     warp its 32-lane quarter, one row per thread), hand it back, and run
//     the decode path's fused epilogues (RoPE + KV append, residual add,
//     SwiGLU, store);
//   * with bf16 weights one CTA per SM works through all units, and two
//     accumulators alternate: one unit's epilogue runs while the MMAs of the
//     next fill the other, and the producer runs ahead across units;
//   * few tiles (short prompts, or the 2560-wide O and down projections)
//     would leave most SMs idle, so K is split until the units fill whole
//     waves: each split stores its partial tile and takes a ticket, and the
//     tile's last split adds the partials in split order (deterministic)
//     before the epilogue.
// Every wait is bounded; the TMEM columns are always released.
//
// Batched decode (several sequences in lockstep, one row each per step) turns
// every decode GEMV into a skinny GEMM with M = 16..64 rows: k_umma_skinny
// swaps the operands (weight rows on the MMA's 128-row side, activation rows
// on its N side) and splits K so that the grid covers the GPU; see there.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "device_once.h"
#include "epilogue.cuh"
#include "kernels.h"

namespace tf {

namespace {

constexpr int BM = 128, BN = 128, BK = 64;
#ifndef TF_GEMM_PERSISTENT
#define TF_GEMM_PERSISTENT 1  // bf16 prompt GEMM: one CTA per SM over all units
#endif
constexpr int kTileA = BM * BK * 2;             // 16 KB (one bf16 part)
constexpr int kThreads = 6 * 32;

// Prompt GEMM tile shapes: 128 prompt rows x GBN weight rows.  256-wide tiles
// (where N allows) halve the activation bytes each weight byte needs, and
// their MMAs are twice as wide.
// WT = 1 / 2: e4m3 or 4-bit weights (128-wide tiles), staged as they are
// behind the bf16 tile and converted into it by the epilogue warps.
template <int GBN, int WT = 0>
struct GemmCfg {
  static constexpr int kTileW = GBN * BK * 2;              // 16 or 32 KB
  static constexpr int kTileWq = WT == 1 ? GBN * BK : WT == 2 ? GBN * 48 : 0;
  static constexpr int kStageBytes = 2 * kTileA + kTileW + kTileWq;  // A hi, A lo, W (, W staged)
  static constexpr int kStages = (GBN == 256 || WT) ? 3 : 4;
  // kind::f16, fp32 accumulate, bf16 A and B, both K-major, M = 128, N = GBN.
  static constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(GBN >> 3) << 17) |
                                     ((uint32_t)(BM >> 4) << 24);
  static constexpr size_t kSmem = 1024 + (size_t)kStages * kStageBytes + (3 * kStages + 5) * 8 + 64;
  static_assert(kStageBytes % 1024 == 0, "stages keep the 1024-byte swizzle alignment");
};

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Shared-memory matrix descriptor: K-major operand tile in the 128-byte
// swizzle layout that TMA writes (8-row groups of 128-byte rows, 1024 bytes
// apart).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr >> 4) & 0x3FFFu);  // start address
  d |= static_cast<uint64_t>(1) << 16;                // leading offset (unused here)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;        // stride between 8-row groups
  d |= static_cast<uint64_t>(1) << 46;                // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                // 128-byte swizzle
  return d;
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void epi_bar_sync() {
  asm volatile("bar.sync 1, 128;" ::: "memory");  // the four epilogue warps
}

// Ticket of a split-K tile: the add releases this CTA's partial (stored by
// the four epilogue warps before the barrier that precedes it) and acquires
// the partials of the CTAs that came earlier.
__device__ __forceinline__ uint32_t ticket_acq_rel(uint32_t* t) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(t) : "memory");
  return old;
}

// Epilogue of 16 consecutive output columns n..n+15 of prompt row m (n a
// multiple of 16), with vector loads and stores: the row's columns are
// contiguous in every output, so each chunk costs a few wide accesses
// instead of one dependent round trip per element.  xr: the residual of
// the same columns (EPI_RESID), loaded ahead by the caller.
__device__ __forceinline__ void store4(float* dst, const float* v) {
  *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
}

__device__ __forceinline__ uint4 pack_bf16x8(const float* v) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    w[i] = static_cast<uint32_t>(f32_to_bf16(v[2 * i])) |
           (static_cast<uint32_t>(f32_to_bf16(v[2 * i + 1])) << 16);
  return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ void gemm_epi_chunk(const GemvParams& p, int m, int n, float (&v)[16],
                                               const float (&xr)[16]) {
  if (p.scale) {
#pragma unroll
    for (int i = 0; i < 16; i += 4) {
      const float4 sc = __ldg(reinterpret_cast<const float4*>(p.scale + n + i));
      v[i] *= sc.x;
      v[i + 1] *= sc.y;
      v[i + 2] *= sc.z;
      v[i + 3] *= sc.w;
    }
  }
  if (p.epi == EPI_RESID) {
    float* o = p.out + (size_t)m * p.ldo + n;
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = xr[i] + v[i];
#pragma unroll
    for (int i = 0; i < 16; i += 4) store4(o + i, v + i);
  } else if (p.epi == EPI_SWIGLU) {
    float u[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) u[i] = silu(v[2 * i]) * v[2 * i + 1];
    const size_t o = (size_t)m * p.ldo + (n >> 1);
    if (p.out_hi) {
      float hv[8], lv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        hv[i] = bf16_to_f32(f32_to_bf16(u[i]));
        lv[i] = u[i] - hv[i];
      }
      *reinterpret_cast<uint4*>(p.out_hi + o) = pack_bf16x8(hv);
      *reinterpret_cast<uint4*>(p.out_lo + o) = pack_bf16x8(lv);
    } else {
      store4(p.out + o, u);
      store4(p.out + o + 4, u + 4);
    }
  } else if (p.epi == EPI_QKV) {
    const int pos = row_pos(p, m);
    if (pos < 0 || pos >= p.T) {
      atomicOr(p.err, ERR_BAD_POS);
      return;
    }
    const int half = p.head_dim >> 1;
    const int qp = p.q_dim >> 1, kp = p.kv_dim >> 1;
    const int pair = n >> 1;  // the chunk's 8 pairs lie in one head
    if (pair < qp + kp && p.qk_raw) {  // q/k norm follows in k_qknorm
      float* r = p.qk_raw + (size_t)m * (p.q_dim + p.kv_dim) + n;
#pragma unroll
      for (int i = 0; i < 16; i += 4) store4(r + i, v + i);
      return;
    }
    if (pair < qp + kp) {
      const bool isq = pair < qp;
      const int pr = isq ? pair : pair - qp;
      const int h = pr / half, i0 = pr - h * half;
      const float4* rp = reinterpret_cast<const float4*>(p.rope + (size_t)pos * half + i0);
      float r0[8], r1[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float4 cs = __ldg(rp + j);  // (cos, sin) of pairs 2j and 2j + 1
        const float a0 = v[4 * j], b0 = v[4 * j + 1], a1 = v[4 * j + 2], b1 = v[4 * j + 3];
        r0[2 * j] = a0 * cs.x - b0 * cs.y;
        r1[2 * j] = b0 * cs.x + a0 * cs.y;
        r0[2 * j + 1] = a1 * cs.z - b1 * cs.w;
        r1[2 * j + 1] = b1 * cs.z + a1 * cs.w;
      }
      if (isq) {
        float* q = p.qout + (size_t)m * p.q_dim + h * p.head_dim + i0;
        store4(q, r0);
        store4(q + 4, r0 + 4);
        store4(q + half, r1);
        store4(q + half + 4, r1 + 4);
      } else {
        uint16_t* k = p.Kc + kv_index(p.kv_tbl, p.kv_npp, p.kv_dim / p.head_dim, p.T, p.kv_seq,
                                      row_seq(p, m), h, pos, p.head_dim) + i0;
        *reinterpret_cast<uint4*>(k) = pack_bf16x8(r0);
        *reinterpret_cast<uint4*>(k + half) = pack_bf16x8(r1);
      }
    } else {
      const int d0 = 2 * (pair - qp - kp);
      const int g = d0 / p.head_dim, d = d0 - g * p.head_dim;
      uint16_t* vv = p.Vc + kv_index(p.kv_tbl, p.kv_npp, p.kv_dim / p.head_dim, p.T, p.kv_seq,
                                     row_seq(p, m), g, pos, p.head_dim) + d;
      *reinterpret_cast<uint4*>(vv) = pack_bf16x8(v);
      *reinterpret_cast<uint4*>(vv + 8) = pack_bf16x8(v + 8);
    }
  } else {
    float* o = p.out + (size_t)m * p.ldo + n;
#pragma unroll
    for (int i = 0; i < 16; i += 4) store4(o + i, v + i);
  }
}

// 8 e4m3 codes (two words) -> 8 bf16 (four words), exactly.
__device__ __forceinline__ void e4m3x8_to_bf16x8(uint32_t a, uint32_t b, uint32_t* o) {
  const uint32_t w[2] = {a, b};
#pragma unroll
  for (int i = 0; i < 2; ++i) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint16_t pr = static_cast<uint16_t>(w[i] >> (16 * h));
      uint32_t h2;
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(pr));
      const __half2 hv = *reinterpret_cast<__half2*>(&h2);
      const float2 f = __half22float2(hv);
      uint32_t d;
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(f.y), "f"(f.x));
      o[2 * i + h] = d;
    }
  }
}

// 16 4-bit codes (w: 8 bytes, element 2i in the low nibble of byte i) times
// their block scale (e4m3 bits sb) -> 16 bf16 (eight words), exactly: an
// e2m1 value times an e4m3 value has at most 6 significant bits.
__device__ __forceinline__ void e2m1x16_to_bf16(const uint2 w, uint32_t sb, uint32_t* o) {
  const float sc = __uint_as_float((sb & 0x7Fu) << 20) * 1.329227995784915873e36f;  // e4m3 by bit placement, x 2^120
  const uint32_t v[2] = {w.x, w.y};
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    uint32_t h[4];
    asm("{.reg .b8 b0, b1, b2, b3; mov.b32 {b0, b1, b2, b3}, %4;"
        " cvt.rn.f16x2.e2m1x2 %0, b0; cvt.rn.f16x2.e2m1x2 %1, b1;"
        " cvt.rn.f16x2.e2m1x2 %2, b2; cvt.rn.f16x2.e2m1x2 %3, b3;}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3]) : "r"(v[i]));
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[b]));
      uint32_t d;
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(f.y * sc), "f"(f.x * sc));
      o[4 * i + b] = d;
    }
  }
}

// One quantised weight slice (128 rows x 64 elements) at q -> bf16 in the
// 128-byte swizzle layout at w (row r at r * 128, 16-byte chunk c at
// c ^ (r & 7)), by the 128 threads et: four lanes per row, so that the reads
// of q are contiguous across a warp.  WT = 1: e4m3 rows of 64 bytes.
// WT = 2: 4-bit rows of 32 bytes, then the slice's 16-byte scale boxes (the
// scales of slices kb & ~3 .. kb | 3).
template <int WT>
__device__ __forceinline__ void dequant_slice(const uint8_t* q, uint8_t* w, int kb, int et) {
  const int lane = et & 31, q4 = lane & 3;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int r = (et >> 5) * 32 + k * 8 + (lane >> 2);
    uint32_t o[8];
    if constexpr (WT == 2) {
      const uint2 c = *reinterpret_cast<const uint2*>(q + r * 32 + q4 * 8);
      e2m1x16_to_bf16(c, q[128 * 32 + r * 16 + (kb & 3) * 4 + q4], o);
    } else {
      const uint4 c = *reinterpret_cast<const uint4*>(q + r * BK + q4 * 16);
      e4m3x8_to_bf16x8(c.x, c.y, o);
      e4m3x8_to_bf16x8(c.z, c.w, o + 4);
    }
    uint8_t* row = w + r * 128;
    *reinterpret_cast<uint4*>(row + (((2 * q4) ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<uint4*>(row + (((2 * q4 + 1) ^ (r & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

template <int GBN, int WT>
__global__ void __launch_bounds__(kThreads, 1)
    k_umma_gemm(const __grid_constant__ CUtensorMap map_ahi,
                const __grid_constant__ CUtensorMap map_alo,
                const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_s,
                const GemvParams p, int M, int S, float* part, uint32_t* tickets) {
  using G = GemmCfg<GBN, WT>;
  constexpr int BN = GBN, kStages = G::kStages, kStageBytes = G::kStageBytes;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment for the swizzled tiles
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* conv = empty + kStages;      // WT: the stage's bf16 weight tile is written
  uint64_t* acc_full = conv + kStages;   // [2] accumulator b holds a finished unit
  uint64_t* acc_empty = acc_full + 2;    // [2] accumulator b was read out
  uint64_t* drain = acc_empty + 2;       // the MMA warp's last MMAs are done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  volatile uint32_t* consumed = tmem_slot + 2;  // K slices the MMA warp took
  volatile uint32_t* okv = tmem_slot + 4;       // [4] epilogue warps' wait outcomes
  volatile uint32_t* last_flag = tmem_slot + 8;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Work units: (128-row tile, GBN-column tile, K split), row tiles fastest.
  // CTA c takes units c, c + gridDim.x, ...; with more units than CTAs the
  // two accumulators alternate, so one unit's epilogue overlaps the next
  // unit's MMAs and the producer runs ahead across units.
  const int mt = (M + BM - 1) / BM, nt = p.N / BN;
  const int tiles = mt * nt, units = tiles * S;
  const int nkt = p.K / BK;
  const bool two = static_cast<int>(gridDim.x) < units;
  const uint32_t tcols = two ? 2u * BN : static_cast<uint32_t>(BN);
  struct Unit {
    int m0, n0, split, tile, kb0, nk;
  };
  auto unit = [&](int u) {
    Unit w;
    const int mi = u % mt, rest = u / mt;
    const int ni = rest % nt;
    w.split = rest / nt;
    w.m0 = mi * BM;
    w.n0 = ni * BN;
    w.tile = mi * nt + ni;
    w.kb0 = static_cast<int>((int64_t)w.split * nkt / S);
    w.nk = static_cast<int>((int64_t)(w.split + 1) * nkt / S) - w.kb0;
    return w;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&conv[s], 128);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    *consumed = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(tcols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int kc = 0, issued = 0;  // K slices over all of this CTA's units
      for (int u = blockIdx.x; u < units && !*abort_flag; u += gridDim.x) {
        const Unit w = unit(u);
        for (int k = 0; k < w.nk; ++k, ++kc) {
          const int s = kc % kStages;
          if (kc >= kStages && !mbar_wait(&empty[s], ((kc / kStages) & 1) ^ 1, p.err)) {
            *abort_flag = 1;
            break;
          }
          uint8_t* st = smem + s * kStageBytes;
          const int kx = (w.kb0 + k) * BK;
          mbar_arrive_expect_tx(&full[s], WT ? 2 * kTileA + G::kTileWq : kStageBytes);
          tma_load_2d(st, &map_ahi, kx, w.m0, &full[s]);
          tma_load_2d(st + kTileA, &map_alo, kx, w.m0, &full[s]);
          uint8_t* wq = st + 2 * kTileA + G::kTileW;  // quantised staging
          if constexpr (WT == 2) {
            tma_load_2d(wq, &map_w, (w.kb0 + k) * 32, w.n0, &full[s]);
            tma_load_2d(wq + 128 * 32, &map_s, p.K / 2 + ((w.kb0 + k) >> 2) * 16, w.n0, &full[s]);
          } else if constexpr (WT == 1) {
            tma_load_2d(wq, &map_w, kx, w.n0, &full[s]);
          } else {
            tma_load_2d(st + 2 * kTileA, &map_w, kx, w.n0, &full[s]);
          }
          issued = kc + 1;
        }
      }
      // After an abort, let the copies still in flight land before the CTA
      // leaves (bounded).
      if (*abort_flag)
        for (int k = static_cast<int>(*consumed); k < issued; ++k)
          if (!mbar_wait(&full[k % kStages], (k / kStages) & 1, p.err)) break;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int kc = 0, li = 0;
      for (int u = blockIdx.x; u < units; u += gridDim.x, ++li) {
        const Unit w = unit(u);
        const int b = two ? (li & 1) : 0;
        bool ok = !*abort_flag;
        // accumulator b is free once the epilogue has read out unit li - 2
        if (ok && two && li >= 2 && !mbar_wait(&acc_empty[b], ((li >> 1) & 1) ^ 1, p.err)) ok = false;
        if (ok) {
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          const uint32_t acc = tmem + static_cast<uint32_t>(b * BN);
          for (int k = 0; k < w.nk; ++k, ++kc) {
            const int s = kc % kStages;
            if (*abort_flag || !mbar_wait(&full[s], (kc / kStages) & 1, p.err) ||
                (WT && !mbar_wait(&conv[s], (kc / kStages) & 1, p.err))) {
              ok = false;
              break;
            }
            *consumed = static_cast<uint32_t>(kc + 1);
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint32_t st = smem_u32(smem + s * kStageBytes);
#pragma unroll
            for (int part = 0; part < 2; ++part) {
              const uint32_t a_base = st + part * kTileA;
              const uint32_t w_base = st + 2 * kTileA;
#pragma unroll
              for (int kk = 0; kk < BK / 16; ++kk) {
                mma_bf16(acc, smem_desc_sw128(a_base + kk * 32), smem_desc_sw128(w_base + kk * 32), G::kIdesc,
                         (k > 0 || part > 0 || kk > 0) ? 1u : 0u);
              }
            }
            mma_commit(&empty[s]);  // frees the stage when these MMAs are done
          }
        }
        if (!ok) *abort_flag = 1;
        mma_commit(&acc_full[b]);  // unit complete (or abandoned)
        if (!ok) break;
      }
      // no MMA of this thread is in flight when the TMEM is released
      mma_commit(drain);
      mbar_wait(drain, 0, p.err);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;
    const size_t tile_stride = (size_t)tiles * (BM * BN);
    [[maybe_unused]] int kc = 0;  // K slices converted (staged weights)
    int li = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++li) {
      const Unit w = unit(u);
      const int b = two ? (li & 1) : 0;
      if constexpr (WT != 0) {
        // First the weight conversion of every slice: stage s's staged codes
        // into its bf16 tile (the MMA of its previous slice is done: the
        // producer reloaded the stage only after it).
        const int et = threadIdx.x - 64;
        for (int k = 0; k < w.nk; ++k, ++kc) {
          const int s = kc % kStages;
          uint8_t* st = smem + s * kStageBytes;
          if (!*abort_flag && mbar_wait(&full[s], (kc / kStages) & 1, p.err))
            dequant_slice<WT>(st + 2 * kTileA + G::kTileW, st + 2 * kTileA, w.kb0 + k, et);
          else
            *abort_flag = 1;
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          mbar_arrive(&conv[s]);
        }
      }
      const int m = w.m0 + row;
      // the first chunk's residual is loaded while the MMAs run
      const bool resid = p.epi == EPI_RESID && m < M;
      const float* xrow = p.out + (size_t)m * p.ldo + w.n0;
      float xr[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) xr[i] = 0.f;
      if (resid) {
#pragma unroll
        for (int i = 0; i < 16; i += 4) {
          const float4 t = *reinterpret_cast<const float4*>(xrow + i);
          xr[i] = t.x;
          xr[i + 1] = t.y;
          xr[i + 2] = t.z;
          xr[i + 3] = t.w;
        }
      }
      const bool wok =
          __all_sync(0xFFFFFFFFu, mbar_wait(&acc_full[b], (li >> 1) & 1, p.err) ? 1 : 0) && !*abort_flag;
      if (lane == 0) okv[q] = wok ? 1u : 0u;
      epi_bar_sync();
      const bool ok = okv[0] && okv[1] && okv[2] && okv[3];  // uniform over the four warps
      if (!ok) break;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint32_t acc = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(b * BN);
      bool run = true;
      if (S > 1) {
        // this split's partial tile [128 rows][BN columns], then a ticket
        float* mine = part + w.split * tile_stride + (size_t)w.tile * (BM * BN) + (size_t)row * BN;
#pragma unroll 1
        for (int c = 0; c < BN; c += 16) {
          float v[16];
          tmem_ld16(acc + c, v);
#pragma unroll
          for (int i = 0; i < 16; i += 4)
            __stcg(reinterpret_cast<float4*>(mine + c + i), make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]));
        }
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        mbar_arrive(&acc_empty[b]);  // the accumulator is free for unit li + 2
        epi_bar_sync();
        if (threadIdx.x == 64) {
          const uint32_t t = ticket_acq_rel(&tickets[w.tile]);
          *last_flag = (t == static_cast<uint32_t>(S) - 1u) ? 1u : 0u;
        }
        epi_bar_sync();
        run = *last_flag != 0;
      }
      if (run) {
#pragma unroll 1
        for (int c = 0; c < BN; c += 16) {
          float v[16];
          if (S > 1) {
            // the splits' partials, added in split order
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = 0.f;
            const float* src = part + (size_t)w.tile * (BM * BN) + (size_t)row * BN + c;
            for (int j = 0; j < S; ++j, src += tile_stride) {
#pragma unroll
              for (int i = 0; i < 16; i += 4) {
                const float4 t = __ldcg(reinterpret_cast<const float4*>(src + i));
                v[i] += t.x;
                v[i + 1] += t.y;
                v[i + 2] += t.z;
                v[i + 3] += t.w;
              }
            }
          } else {
            tmem_ld16(acc + c, v);
          }
          if (m >= M) continue;
          float xc[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) xc[i] = xr[i];
          if (resid && c + 16 < BN) {  // the next chunk's residual, ahead of this chunk's stores
#pragma unroll
            for (int i = 0; i < 16; i += 4) {
              const float4 t = *reinterpret_cast<const float4*>(xrow + c + 16 + i);
              xr[i] = t.x;
              xr[i + 1] = t.y;
              xr[i + 2] = t.z;
              xr[i + 3] = t.w;
            }
          }
          gemm_epi_chunk(p, m, w.n0 + c, v, xc);
        }
        if (S > 1 && threadIdx.x == 64) tickets[w.tile] = 0u;
      }
      if (S == 1) {
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        mbar_arrive(&acc_empty[b]);
      }
      epi_bar_sync();  // okv and last_flag are written again for the next unit
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 1) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(tcols) : "memory");
  }
}

__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map, int x, int y,
                                                 uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void bulk_g2s_plain(void* dst, const void* src, uint32_t bytes,
                                               uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}


// ---------------------------------------------------------------- skinny GEMM
// D[n][m] = sum_k W[n][k] a[m][k] for one 128-row weight tile and one slice of
// K per CTA (grid: weight tiles x K splits).  Warp 0 streams 64-wide K slices
// of the weight tile and of the activation rows (hi and lo parts) into a
// 4-stage ring; warp 1 issues tcgen05.mma with the weight slice as the
// 128-row A operand and the NB activation rows as the N = NB operand, so one
// accumulator column per activation row; warps 2-5 read their TMEM lane
// quarter (one weight row per thread, NB values).  With more than one split
// each CTA stores its partial [128][NB] and takes a ticket; the last CTA of
// the tile adds the partials in split order (deterministic) and runs the
// epilogue.  Rows n >= N and k >= K come in as zeros (TMA out-of-bounds fill).
#ifndef TF_SKINNY_STAGES
#define TF_SKINNY_STAGES 4
#endif
#ifndef TF_SKINNY_CTAS_PER_SM
#define TF_SKINNY_CTAS_PER_SM 2
#endif
#ifndef TF_SKINNY_PREFETCH
#define TF_SKINNY_PREFETCH 8   // weight slices requested into L2 ahead of the ring
#endif
constexpr int kSkPrefetch = TF_SKINNY_PREFETCH;

// Fire-and-forget request of one weight box into L2.
__device__ __forceinline__ void tma_prefetch_l2(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
constexpr int kSkStages = TF_SKINNY_STAGES;
#ifndef TF_SKINNY_F8_BSLOTS
#define TF_SKINNY_F8_BSLOTS 3   // e4m3 weights: bf16 slots the converters fill
#endif
#ifndef TF_SKINNY_F8_SLOTS
#define TF_SKINNY_F8_SLOTS 3    // e4m3 weights: e4m3 + activation slots in flight
#endif
constexpr int kSkThreads = 6 * 32;

// WT = 0: bf16 weights.  WT = 1: e4m3 weights (fp32 row scale applied in the
// epilogue), so that HBM only carries the e4m3 bytes: the producer streams
// each e4m3 slice (8 KB) with its activation parts into a deep ring; the
// four epilogue warps convert the slice (one row per thread, exactly: every
// e4m3 value is a bf16 value) into a slot of a shallow ring of bf16 slices,
// and the MMA reads the bf16 slot and the activation parts where they
// landed.  Two CTAs per SM for up to 32 rows.
template <int NB, int WT>
struct Skinny {
  static constexpr int kStages = WT ? TF_SKINNY_F8_BSLOTS : kSkStages;  // WT = 0: weight + activation stages;
                                                      // WT = 1: bf16 weight slots
  static constexpr int kW = 128 * BK * 2;            // weight slice (bf16), 16 KB
  static constexpr int kA = NB * BK * 2;             // one activation part
  // one quantised slice: e4m3 codes (128 x 64 B), or 4-bit codes (128 x 32 B)
  // followed by the 16-byte scale box that holds its block scales (128 x 16 B)
  static constexpr int kW8 = WT == 2 ? 128 * 32 + 128 * 16 : 128 * BK;
  static constexpr int kF8 = WT ? TF_SKINNY_F8_SLOTS : 0;  // e4m3 + activation slots
  static constexpr int kF8Slot = kW8 + 2 * kA;
  static constexpr int kStage = WT ? kW : kW + 2 * kA;
  static constexpr size_t kRing = (size_t)kStages * kStage + (size_t)kF8 * kF8Slot;
  static constexpr uint32_t kCols = NB < 32 ? 32u : static_cast<uint32_t>(NB);
  // kind::f16, fp32 accumulate, bf16 A and B, both K-major, M = 128, N = NB.
  static constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) |
                                     ((uint32_t)(NB >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
  static constexpr size_t kSmem =
      1024 + kRing + (3 * kStages + 2 * kF8 + 2) * 8 + 64 + (64 + 4 * NB) * 4;
  // one split's partial of a tile: [NB][128] fp32
  static constexpr uint32_t kChunk = NB * 128 * 4;
  static constexpr int kChunksPerRound = static_cast<int>(kRing / kChunk);
};

// WT = 2: 4-bit rows (K/2 code bytes, then K/16 e4m3 block-scale bytes):
// map_w takes 32-byte code boxes, map_s the 16-byte scale boxes (4 slices'
// scales each); the row scale is applied in the epilogue.
template <int NB, int WT>
__global__ void __launch_bounds__(kSkThreads, NB <= 32 ? TF_SKINNY_CTAS_PER_SM : 1)
    k_umma_skinny(const __grid_constant__ CUtensorMap map_w,
                  const __grid_constant__ CUtensorMap map_ahi,
                  const __grid_constant__ CUtensorMap map_alo, const __grid_constant__ CUtensorMap map_s,
                  const GemvParams p, int M, int S, float* part, uint32_t* tickets) {
  using C = Skinny<NB, WT>;
  constexpr int kSkStages = C::kStages;
  static_assert(C::kStage % 1024 == 0, "stages must keep the 1024-byte swizzle alignment");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* f8 = smem + kSkStages * C::kStage;   // WT = 1: [kF8][e4m3 128 x 64 B | A hi | A lo]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kRing);
  uint64_t* empty = full + kSkStages;
  uint64_t* conv = empty + kSkStages;     // WT = 1: the slot's bf16 slice is written
  uint64_t* f8full = conv + kSkStages;    // WT = 1: an e4m3 slice landed
  uint64_t* f8empty = f8full + C::kF8;    // WT = 1: the MMA is done with a slot
  uint64_t* done = f8empty + C::kF8;
  uint64_t* red = done + 1;   // split partials staged into the (idle) ring
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(red + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  volatile uint32_t* last_flag = tmem_slot + 2;
  volatile uint32_t* consumed = tmem_slot + 3;   // k slices the MMA warp took
  volatile uint32_t* okv = tmem_slot + 4;        // [4] epilogue warps' wait outcomes
  volatile uint32_t* red_fail = tmem_slot + 8;   // a staging wait expired
  float* rstd_s = reinterpret_cast<float*>(tmem_slot + 16);  // [64] row rstd
  float* red_s = rstd_s + 64;                               // [4][NB] sums of squares

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x, split = blockIdx.y;
  const int n0 = tile * 128;
  const int nk = (p.K + BK - 1) / BK;
  const int kb0 = static_cast<int>((int64_t)split * nk / S);
  const int kb1 = static_cast<int>((int64_t)(split + 1) * nk / S);
  const int nkb = kb1 - kb0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kSkStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&conv[s], 128);
    }
    for (int s = 0; s < C::kF8; ++s) {
      mbar_init(&f8full[s], 1);
      mbar_init(&f8empty[s], 1);
    }
    mbar_init(done, 1);
    mbar_init(red, 1);
    *abort_flag = 0;
    *consumed = 0;
    *red_fail = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(C::kCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      prefetch_tensormap(&map_w);
      if constexpr (WT >= 1) {
        prefetch_tensormap(&map_ahi);
        prefetch_tensormap(&map_alo);
        if (WT == 2) prefetch_tensormap(&map_s);
        // e4m3 slices into their ring; the converters load the activations.
        int issued = 0;
        for (int i = 0; i < nkb; ++i) {
          const int s8 = i % C::kF8;
          if (i >= C::kF8 && !mbar_wait(&f8empty[s8], ((i / C::kF8) & 1) ^ 1, p.err)) {
            *abort_flag = 1;
            break;
          }
          if (*abort_flag) break;
          uint8_t* sl = f8 + s8 * C::kF8Slot;
          mbar_arrive_expect_tx(&f8full[s8], C::kF8Slot);
          if constexpr (WT == 2) {
            tma_load_2d_hint(sl, &map_w, (kb0 + i) * 32, n0, &f8full[s8], pol);
            tma_load_2d_hint(sl + 128 * 32, &map_s, p.K / 2 + ((kb0 + i) >> 2) * 16, n0, &f8full[s8], pol);
          } else {
            tma_load_2d_hint(sl, &map_w, (kb0 + i) * BK, n0, &f8full[s8], pol);
          }
          if (i == (nkb < C::kF8 ? nkb : C::kF8) - 1 || i >= C::kF8) {
            // the activation parts come from the previous kernel: the first
            // ring's worth of weight slices is issued before waiting for it
            if (i == (nkb < C::kF8 ? nkb : C::kF8) - 1) {
              pdl_wait();
              for (int j = 0; j < i; ++j) {
                uint8_t* sj = f8 + j * C::kF8Slot;
                tma_load_2d(sj + C::kW8, &map_ahi, (kb0 + j) * BK, 0, &f8full[j]);
                tma_load_2d(sj + C::kW8 + C::kA, &map_alo, (kb0 + j) * BK, 0, &f8full[j]);
              }
            }
            tma_load_2d(sl + C::kW8, &map_ahi, (kb0 + i) * BK, 0, &f8full[s8]);
            tma_load_2d(sl + C::kW8 + C::kA, &map_alo, (kb0 + i) * BK, 0, &f8full[s8]);
          }
          issued = i + 1;
          // L2 requests kSkPrefetch slices beyond the ring's
          constexpr int kx = WT == 2 ? 32 : BK;  // x extent of one slice's codes
          if (i == 0)
            for (int j = C::kF8; j < nkb && j < C::kF8 + kSkPrefetch; ++j)
              tma_prefetch_l2(&map_w, (kb0 + j) * kx, n0);
          else if (i >= C::kF8 && i + kSkPrefetch < nkb)
            tma_prefetch_l2(&map_w, (kb0 + i + kSkPrefetch) * kx, n0);
        }
        // the last fills still in flight land before the CTA leaves (bounded)
        for (int i = issued > C::kF8 ? issued - C::kF8 : 0; i < issued; ++i)
          if (!mbar_wait(&f8full[i % C::kF8], (i / C::kF8) & 1, p.err)) break;
      } else {
      prefetch_tensormap(&map_ahi);
      prefetch_tensormap(&map_alo);
      // The weights do not depend on the previous kernel: fill the ring with
      // weight slices and ask L2 for the next kSkPrefetch slices, then wait
      // for the activations' producer.  The L2 requests keep HBM busy while
      // this kernel waits and while the ring drains; the ring's loads then
      // mostly hit L2.
      const int pre = nkb < kSkStages ? nkb : kSkStages;
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(&full[i], C::kStage);
        tma_load_2d_hint(smem + i * C::kStage, &map_w, (kb0 + i) * BK, n0, &full[i], pol);
      }
      for (int i = pre; i < nkb && i < pre + kSkPrefetch; ++i)
        tma_prefetch_l2(&map_w, (kb0 + i) * BK, n0);
      pdl_wait();
      for (int i = 0; i < pre; ++i) {
        uint8_t* st = smem + i * C::kStage;
        tma_load_2d(st + C::kW, &map_ahi, (kb0 + i) * BK, 0, &full[i]);
        tma_load_2d(st + C::kW + C::kA, &map_alo, (kb0 + i) * BK, 0, &full[i]);
      }
      int issued = pre;
      for (int i = pre; i < nkb; ++i) {
        const int s = i % kSkStages;
        if (!mbar_wait(&empty[s], ((i / kSkStages) & 1) ^ 1, p.err)) {
          *abort_flag = 1;
          break;
        }
        uint8_t* st = smem + s * C::kStage;
        mbar_arrive_expect_tx(&full[s], C::kStage);
        tma_load_2d_hint(st, &map_w, (kb0 + i) * BK, n0, &full[s], pol);
        tma_load_2d(st + C::kW, &map_ahi, (kb0 + i) * BK, 0, &full[s]);
        tma_load_2d(st + C::kW + C::kA, &map_alo, (kb0 + i) * BK, 0, &full[s]);
        issued = i + 1;
        if (i + kSkPrefetch < nkb) tma_prefetch_l2(&map_w, (kb0 + i + kSkPrefetch) * BK, n0);
      }
      // After an abort, let the copies still in flight land before the CTA
      // leaves (bounded).
      const int from = static_cast<int>(*consumed);
      if (*abort_flag)
        for (int i = from; i < issued; ++i)
          if (!mbar_wait(&full[i % kSkStages], (i / kSkStages) & 1, p.err)) break;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      for (int i = 0; i < nkb; ++i) {
        const int s = i % kSkStages;
        const int s8 = WT ? i % C::kF8 : 0;
        if (*abort_flag ||
            (WT ? (!mbar_wait(&conv[s], (i / kSkStages) & 1, p.err) ||
                   !mbar_wait(&f8full[s8], (i / C::kF8) & 1, p.err))
                : !mbar_wait(&full[s], (i / kSkStages) & 1, p.err))) {
          *abort_flag = 1;
          break;
        }
        *consumed = static_cast<uint32_t>(i + 1);
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t st = smem_u32(smem + s * C::kStage);
        // activation parts: behind the weights (WT = 0) or in the e4m3 slot
        const uint32_t at = WT ? smem_u32(f8 + s8 * C::kF8Slot + C::kW8) : st + C::kW;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
#pragma unroll
          for (int prt = 0; prt < 2; ++prt) {
            const uint64_t wd = smem_desc_sw128(st + kk * 32);
            const uint64_t ad = smem_desc_sw128(at + prt * C::kA + kk * 32);
            const uint32_t acc = (i > 0 || kk > 0 || prt > 0) ? 1u : 0u;
            asm volatile(
                "{\n\t.reg .pred q;\n\t"
                "setp.ne.b32 q, %4, 0;\n\t"
                "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, q;\n\t}" ::"r"(tmem),
                "l"(wd), "l"(ad), "r"(C::kIdesc), "r"(acc)
                : "memory");
          }
        }
        mma_commit(&empty[s]);
        if constexpr (WT >= 1) mma_commit(&f8empty[s8]);
      }
      mma_commit(done);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int et = threadIdx.x - 64;  // 0..127 over the four epilogue warps
    if constexpr (WT >= 1) {
      // Slot sb of the bf16 ring takes slice i once the MMA is done with it:
      // the e4m3 slice is converted into the 128-byte swizzle layout
      // (16-byte chunk c of row r at c ^ (r & 7)).
      for (int i = 0; i < nkb; ++i) {
        const int sb = i % kSkStages, s8 = i % C::kF8;
        bool ok = !*abort_flag;
        if (ok && i >= kSkStages) ok = mbar_wait(&empty[sb], ((i / kSkStages) & 1) ^ 1, p.err);
        if (ok) ok = mbar_wait(&f8full[s8], (i / C::kF8) & 1, p.err);
        if (ok) {
          dequant_slice<WT>(f8 + s8 * C::kF8Slot, smem + sb * C::kStage, kb0 + i, et);
        } else {
          *abort_flag = 1;
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive(&conv[sb]);
      }
    }
    pdl_wait();
    const int q = warp & 3;
    const int nl = q * 32 + lane;     // weight row within the tile (TMEM lane)
    const int n = n0 + nl;
    // Everything the epilogue reads from global memory is loaded while the
    // weights stream (the loads would otherwise queue behind its stores):
    // the row rstd of a deferred RMSNorm, the residual, the RoPE factors.
    if (p.ssq_in && et < M) {
      const int r = p.in_rps > 1 ? et * p.in_rps + p.in_rps - 1 : et;
      float ss = 0.f;
      for (int t = 0; t < p.ssq_n; ++t) ss += p.ssq_in[t * kSsqRows + r];
      rstd_s[et] = 1.0f / sqrtf(ss / static_cast<float>(p.K) + p.eps);
    }
    float xr[NB];                          // residual rows (EPI_RESID)
    float2 cs_t = make_float2(1.f, 0.f);   // RoPE (cos, sin) of this thread's pair (EPI_QKV)
    int pos0 = 0;
    if (p.epi == EPI_RESID) {
#pragma unroll
      for (int c = 0; c < NB; ++c)
        xr[c] = (c < M && n < p.N) ? p.out[(size_t)c * p.ldo + n] : 0.f;
    } else if (p.epi == EPI_QKV) {
      // pair (et & 63) of the tile, rows of parity et >> 6: with one or two
      // rows per sequence they all sit at one position
      pos0 = p.pos_ptr ? *p.pos_ptr : p.pos_fixed;
      if ((p.rps == 1 || p.rps == 2) && (!p.pos_ptr || p.pos_uniform))
        cs_t = qkv_pair_rope(p, (n0 >> 1) + (et & 63), pos0 + (p.rps == 2 ? (et >> 6) : 0));
    }
    const bool wok = __all_sync(0xFFFFFFFFu, mbar_wait(done, 0, p.err) ? 1 : 0) && !*abort_flag;
    if (lane == 0) okv[q] = wok ? 1u : 0u;
    epi_bar_sync();  // publishes rstd_s and every warp's wait outcome
    const bool ok = okv[0] && okv[1] && okv[2] && okv[3];
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    float v[NB];
#pragma unroll
    for (int c = 0; c < NB; ++c) v[c] = 0.f;
    if (ok) {
#pragma unroll
      for (int c = 0; c < NB; c += 16) {
        float t[16];
        tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + c, t);
#pragma unroll
        for (int i = 0; i < 16; ++i) v[c + i] = t[i];
      }
    }
    bool run = ok;  // CTA-uniform from here on
    if (S > 1) {
      // this split's partial of the tile, [NB][128] (coalesced per row c)
      float* mine = part + ((size_t)split * gridDim.x + tile) * (NB * 128);
      if (ok) {
#pragma unroll
        for (int c = 0; c < NB; ++c) __stcg(mine + c * 128 + nl, v[c]);
      }
      epi_bar_sync();
      if (et == 0) {
        const uint32_t t = ticket_acq_rel(&tickets[tile]);
        *last_flag = (t == static_cast<uint32_t>(S) - 1u) ? 1u : 0u;
      }
      epi_bar_sync();
      run = ok && *last_flag != 0;
      if (run) {
        // The last CTA of the tile stages all splits' partials into its ring
        // (idle now: every MMA has completed) with bulk copies, one round
        // trip per kChunksPerRound splits, and adds them in split order.
        const float* st = reinterpret_cast<const float*>(smem);
#pragma unroll
        for (int c = 0; c < NB; ++c) v[c] = 0.f;
        int round = 0;
        for (int j0 = 0; j0 < S; j0 += C::kChunksPerRound, ++round) {
          const int nr = (S - j0) < C::kChunksPerRound ? (S - j0) : C::kChunksPerRound;
          if (*red_fail) break;  // CTA-uniform (read after a barrier)
          if (et == 0) {
            // the partials were written through the generic proxy
            asm volatile("fence.proxy.async.global;" ::: "memory");
            mbar_arrive_expect_tx(red, nr * C::kChunk);
            for (int r = 0; r < nr; ++r)
              bulk_g2s_plain(smem + r * C::kChunk,
                             part + ((size_t)(j0 + r) * gridDim.x + tile) * (NB * 128), C::kChunk, red);
          }
          if (mbar_wait(red, round & 1, p.err)) {
            for (int r = 0; r < nr; ++r) {
#pragma unroll
              for (int c = 0; c < NB; ++c) v[c] += st[(r * NB + c) * 128 + nl];
            }
          } else {
            *red_fail = 1;
          }
          epi_bar_sync();  // the ring is refilled by the next round
        }
        if (et == 0) tickets[tile] = 0u;
      }
    }
    if (run) {
      const float sc = (p.scale && n < p.N) ? __ldg(&p.scale[n]) : 1.0f;
#pragma unroll
      for (int c = 0; c < NB; ++c)
        v[c] *= p.ssq_in ? (c < M ? sc * rstd_s[c] : 0.f) : sc;
      if (p.epi == EPI_QKV || p.epi == EPI_SWIGLU) {
        // The tile's results go through shared memory (the ring is idle) so
        // that the pair epilogue runs as one short loop: its code stays in
        // the instruction cache instead of being fetched once per row.
        // Thread et takes pair pl of the tile for the rows of parity par.
        float* vs = reinterpret_cast<float*>(smem);
#pragma unroll
        for (int c = 0; c < NB; ++c) vs[c * 128 + nl] = v[c];
        epi_bar_sync();
        const int pl = et & 63, par = et >> 6;
        const int pair = (n0 >> 1) + pl;
        if (2 * pair < p.N) {
#pragma unroll 1
          for (int c = par; c < M; c += 2) {
            const float v0 = vs[c * 128 + 2 * pl], v1 = vs[c * 128 + 2 * pl + 1];
            if (p.epi == EPI_QKV) {
              // with one position for every sequence, parity fixes a row's position
              const bool pre = (p.rps == 1 || p.rps == 2) && (!p.pos_ptr || p.pos_uniform);
              const int pos = pre ? pos0 + (p.rps > 0 ? c % p.rps : c) : row_pos(p, c);
              epi_qkv_pair_at(p, c, pair, v0, v1, pos, pre ? cs_t : qkv_pair_rope(p, pair, pos));
            } else {
              epi_swiglu(p, c, pair, v0, v1);
            }
          }
        }
      } else {
        // store / residual add; with nw_next also the consumer's input
        // (x * nw_next as bf16 parts) and this tile's sums of x^2 per row
        const bool nx = p.nx_hi != nullptr;
        const float wn = (nx && n < p.N) ? bf16_to_f32(p.nw_next[n]) : 0.f;
#pragma unroll
        for (int c = 0; c < NB; ++c) {
          float xn = 0.f;
          if (c < M && n < p.N) {
            xn = p.epi == EPI_RESID ? xr[c] + v[c] : v[c];
            p.out[(size_t)c * p.ldo + n] = xn;
            if (nx) {
              const float a = xn * wn;
              const uint16_t h = f32_to_bf16(a);
              p.nx_hi[(size_t)c * p.ldo + n] = h;
              p.nx_lo[(size_t)c * p.ldo + n] = f32_to_bf16(a - bf16_to_f32(h));
            }
          }
          v[c] = xn * xn;
        }
        if (nx) {
#pragma unroll
          for (int c = 0; c < NB; ++c) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v[c] += __shfl_xor_sync(0xFFFFFFFFu, v[c], o);
          }
          if (lane == 0) {
#pragma unroll
            for (int c = 0; c < NB; ++c) red_s[q * NB + c] = v[c];
          }
          epi_bar_sync();
          if (et < M)
            p.ssq_out[tile * kSsqRows + et] =
                ((red_s[et] + red_s[NB + et]) + red_s[2 * NB + et]) + red_s[3 * NB + et];
        }
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 1) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(C::kCols)
                 : "memory");
  }
}

// ---------------------------------------------------------------- prompt attention
// Causal attention of prompt rows on the tensor cores ("Fish Speech" tour,
// "Why You Need This": grouped-query attention; the tuna-fish README's
// prefill tokens/s).  One CTA per (block of 128 query rows, query head,
// sequence); the keys 0..pos of every row are visited in tiles of 128:
//   * warp 0 loads the block's queries once (bf16 hi and lo parts), the K
//     tiles of the head's KV group into two stages and the V tiles into one
//     (TMA, 128-byte swizzle; paged caches: one box per 32-position page);
//   * warp 1 issues S = Q K^T (hi and lo parts, fp32 in TMEM columns 0..127)
//     and, once the probabilities are in shared memory, O += P V (hi and lo
//     parts of P; TMEM columns 128..; V is read in its cache layout, an
//     MN-major operand);
//   * warps 2-5 own one query row each (its TMEM lane): they read the row's
//     128 scores, apply the 1/sqrt(D) scale and the causal mask, keep the
//     running maximum m and sum l, and write p = 2^(s - m) as bf16 hi and lo
//     parts (about 16 significant bits, like the activations of the prompt
//     GEMMs).  O is rescaled (read, scaled, written back in TMEM) only when
//     the maximum grows by more than 2^8, so p <= 256 and nothing overflows;
//     the same m scales l, so the result is exact up to rounding.
// V rows past the block's last key are zeroed in shared memory before the
// product (the cache holds stale rows there; their p is 0, but 0 x NaN is
// not).  Bounded waits; TMEM always released.
template <int D>
struct PAttn {
  static constexpr int kBoxes = D / 64;            // 64-column boxes per row
  static constexpr int kQ = 128 * D * 2;           // one query part, bytes
  static constexpr int kKV = 128 * D * 2;          // one K or V tile
  static constexpr int kP = 128 * 128 * 2;         // one part of the probabilities
  static constexpr size_t kOffK = 2 * (size_t)kQ;  // [2 stages]
  static constexpr size_t kOffV = kOffK + 2 * (size_t)kKV;
  static constexpr size_t kOffP = kOffV + kKV;     // [hi, lo]
  static constexpr size_t kOffBar = kOffP + 2 * (size_t)kP;
  static constexpr size_t kSmem = 1024 + kOffBar + 128;
  static constexpr uint32_t kCols = 256;           // S: 0..127, O: 128..
  // kind::f16, fp32 accumulate, bf16 operands, M = 128.  S: B (keys x D)
  // K-major, N = 128.  O: B (keys x D) MN-major (bit 16), N = D.
  static constexpr uint32_t kIdescS =
      (1u << 4) | (1u << 7) | (1u << 10) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
  static constexpr uint32_t kIdescO = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) |
                                      ((uint32_t)(D >> 3) << 17) | ((128u >> 4) << 24);
};

// Descriptor of an MN-major operand in the 128-byte swizzle layout TMA
// writes for [rows = K][64 elements along N] boxes: 8-row groups 1024 bytes
// apart (stride), 64-element column blocks `lbo` bytes apart (leading).
__device__ __forceinline__ uint64_t smem_desc_sw128_mn(uint32_t addr, uint32_t lbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Two floats -> two bf16 (round to nearest even) in one word, the first in
// the low half (the hardware conversion; inputs here are finite).
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// 2^x with the SFU's approximate base-2 exponential (relative error about
// 2^-22; 2^-inf = 0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}


template <int D>
__global__ void __launch_bounds__(192, 1)
    k_umma_attn(const __grid_constant__ CUtensorMap map_qhi, const __grid_constant__ CUtensorMap map_qlo,
                const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                const PromptAttnArgs a) {
  using C = PAttn<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sq = smem;                    // [hi, lo][boxes][128 rows][128 B]
  uint8_t* sk = smem + C::kOffK;         // [stage][boxes][128 rows][128 B]
  uint8_t* sv = smem + C::kOffV;         // [boxes][128 rows][128 B]
  uint8_t* sp = smem + C::kOffP;         // [hi, lo][2 key halves][128 rows][128 B]
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* q_full = bar;
  uint64_t* k_full = bar + 1;            // [2]
  uint64_t* k_empty = bar + 3;           // [2]
  uint64_t* v_full = bar + 5;
  uint64_t* v_empty = bar + 6;
  uint64_t* s_full = bar + 7;
  uint64_t* p_full = bar + 8;
  uint64_t* o_full = bar + 9;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 10);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  volatile uint32_t* issued_k = tmem_slot + 2;
  volatile uint32_t* issued_v = tmem_slot + 3;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nblk = (a.P + 127) / 128;
  const int blk = nblk - 1 - static_cast<int>(blockIdx.x);   // longest rows first
  const int h = blockIdx.y;
  const int g = h / (a.Hq / a.Hkv);
  const int seq = a.seq + static_cast<int>(blockIdx.z);       // this sequence's slot
  const int qbase = static_cast<int>(blockIdx.z) * a.P;       // its first row in q and out
  const int q0 = blk * 128;                                  // first query row
  const int rows = min(128, a.P - q0);
  const int last_key = a.pos0 + q0 + rows - 1;               // the block's last key
  const int nt = last_key / 128 + 1;                         // key tiles

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    mbar_init(v_full, 1);
    mbar_init(v_empty, 1);
    mbar_init(s_full, 1);
    mbar_init(p_full, 128);
    mbar_init(o_full, 1);
    *abort_flag = 0;
    *issued_k = 0;
    *issued_v = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(C::kCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_s = tmem, tmem_o = tmem + 128;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tensormap(&map_qhi);
      prefetch_tensormap(&map_qlo);
      prefetch_tensormap(&map_k);
      prefetch_tensormap(&map_v);
      mbar_arrive_expect_tx(q_full, 2 * C::kQ);
      for (int b = 0; b < C::kBoxes; ++b) {
        tma_load_2d(sq + b * 16384, &map_qhi, h * D + b * 64, qbase + q0, q_full);
        tma_load_2d(sq + C::kQ + b * 16384, &map_qlo, h * D + b * 64, qbase + q0, q_full);
      }
      // one tile of K or V rows (128 keys from kbase) into dst
      auto load_tile = [&](const CUtensorMap* map, uint8_t* dst, int kbase, uint64_t* b_) {
        if (a.kv_tbl) {
          for (int pg = 0; pg < 128 / kKvPage; ++pg) {
            const int pi = kbase / kKvPage + pg;
            const int page = pi < a.kv_npp ? __ldg(a.kv_tbl + (size_t)seq * a.kv_npp + pi) : 0;
            const int y = (page * a.Hkv + g) * kKvPage;
            for (int b = 0; b < C::kBoxes; ++b)
              tma_load_2d(dst + b * 16384 + pg * (kKvPage * 128), map, b * 64, y, b_);
          }
        } else {
          for (int b = 0; b < C::kBoxes; ++b)
            tma_load_2d(dst + b * 16384, map, b * 64, (seq * a.Hkv + g) * a.T + kbase, b_);
        }
      };
      for (int j = 0; j < nt; ++j) {
        const int st = j & 1;
        if (j >= 2 && !mbar_wait(&k_empty[st], ((j >> 1) - 1) & 1, a.err)) {
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(&k_full[st], C::kKV);
        load_tile(&map_k, sk + (size_t)st * C::kKV, j * 128, &k_full[st]);
        *issued_k = static_cast<uint32_t>(j + 1);
        if (j >= 1 && !mbar_wait(v_empty, (j - 1) & 1, a.err)) {
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(v_full, C::kKV);
        load_tile(&map_v, sv, j * 128, v_full);
        *issued_v = static_cast<uint32_t>(j + 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = mbar_wait(q_full, 0, a.err);
      const uint32_t qb = smem_u32(sq);
      const uint32_t pb = smem_u32(sp);
      const uint32_t vb = smem_u32(sv);
      for (int j = 0; ok && j < nt; ++j) {
        const int st = j & 1;
        if (*abort_flag || !mbar_wait(&k_full[st], (j >> 1) & 1, a.err)) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t kb = smem_u32(sk + (size_t)st * C::kKV);
#pragma unroll
        for (int prt = 0; prt < 2; ++prt)
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_f16(tmem_s, smem_desc_sw128(qb + prt * C::kQ + off), smem_desc_sw128(kb + off),
                    C::kIdescS, (prt > 0 || kk > 0) ? 1u : 0u);
          }
        mma_commit(&k_empty[st]);
        mma_commit(s_full);
        if (!mbar_wait(p_full, j & 1, a.err) || !mbar_wait(v_full, j & 1, a.err)) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll
        for (int prt = 0; prt < 2; ++prt)
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t aoff = prt * C::kP + (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_f16(tmem_o, smem_desc_sw128(pb + aoff), smem_desc_sw128_mn(vb + kk * 2048, 16384),
                    C::kIdescO, (j > 0 || prt > 0 || kk > 0) ? 1u : 0u);
          }
        mma_commit(v_empty);
        mma_commit(o_full);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax rows
    const int qw = warp & 3;
    const int r = qw * 32 + lane;                 // query row in the block (TMEM lane)
    const int qpos = a.pos0 + q0 + r;
    const uint32_t lane_base = static_cast<uint32_t>(qw * 32) << 16;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      // waits are made warp-uniform: tcgen05.ld is a warp-collective
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(s_full, j & 1, a.err) ? 1 : 0)) {
        ok = false;
        break;
      }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      float s[128];
#pragma unroll
      for (int c = 0; c < 128; c += 16) {
        float t[16];
        tmem_ld16(tmem_s + lane_base + c, t);
#pragma unroll
        for (int i = 0; i < 16; ++i) s[c + i] = t[i];
      }
      const int kbase = j * 128;
      float mx = -INFINITY;
      if (kbase + 127 <= a.pos0 + q0) {  // a tile below the block's diagonal: no mask
#pragma unroll
        for (int i = 0; i < 128; ++i) mx = fmaxf(mx, s[i]);
      } else {
#pragma unroll
        for (int i = 0; i < 128; ++i) {
          s[i] = (kbase + i <= qpos) ? s[i] : -INFINITY;
          mx = fmaxf(mx, s[i]);
        }
      }
      mx *= a.scale_log2;  // the scale is positive: max(s) * c = max(s * c)
      // The previous product must be done before O is rescaled or the
      // probability tiles are overwritten.
      if (j > 0) {
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(o_full, (j - 1) & 1, a.err) ? 1 : 0)) {
          ok = false;
          break;
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      }
      // A new reference maximum (always on tile 0).  The rescale of O is
      // decided per warp: tcgen05.ld / st are warp-collective, so every lane
      // takes part (alpha = 1 for rows that keep their maximum).
      const bool grow = mx > m_used + 8.0f;
      const float alpha = grow ? ex2_approx(m_used - mx) : 1.0f;
      if (grow) {
        l *= alpha;
        m_used = mx;
      }
      if (j > 0 && __any_sync(0xFFFFFFFFu, grow)) {
#pragma unroll 1
        for (int c = 0; c < D; c += 16) {
          float t[16];
          tmem_ld16(tmem_o + lane_base + c, t);
#pragma unroll
          for (int i = 0; i < 16; ++i) t[i] *= alpha;
          tmem_st16(tmem_o + lane_base + c, t);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      }
      // p = 2^(s - m) as bf16 hi and lo parts, the row's 128 keys in two
      // 64-key halves of the 128-byte swizzle layout (16-byte chunk c of row
      // r at c ^ (r & 7))
      // p = 2^(s * c - m): one FMA and one ex2 per key (masked keys: 2^-inf = 0)
      const float nm = -m_used;
#pragma unroll
      for (int i = 0; i < 128; ++i) {
        s[i] = ex2_approx(fmaf(s[i], a.scale_log2, nm));
        l += s[i];
      }
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint8_t* rowp = sp + half * 16384 + r * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t wh[4], wl[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float p0 = s[half * 64 + c * 8 + 2 * e];
            const float p1 = s[half * 64 + c * 8 + 2 * e + 1];
            wh[e] = bf16x2_rn(p0, p1);
            wl[e] = bf16x2_rn(p0 - __uint_as_float(wh[e] << 16), p1 - __uint_as_float(wh[e] & 0xFFFF0000u));
          }
          const int cs = (c ^ (r & 7)) << 4;
          *reinterpret_cast<uint4*>(rowp + cs) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
          *reinterpret_cast<uint4*>(rowp + C::kP + cs) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
        }
      }
      if (j == nt - 1 && kbase + r > last_key) {
        // V rows past the block's last key: zero (this thread's row r of the
        // tile, every column box), after the tile has landed
        if (!mbar_wait(v_full, j & 1, a.err)) {
          ok = false;
        } else {
          uint8_t* vrow = sv + r * 128;
#pragma unroll
          for (int b = 0; b < C::kBoxes; ++b)
#pragma unroll
            for (int c = 0; c < 8; ++c)
              *reinterpret_cast<uint4*>(vrow + b * 16384 + c * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      ok = __all_sync(0xFFFFFFFFu, ok ? 1 : 0) != 0;
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      mbar_arrive(p_full);
      if (!ok) break;
    }
    if (ok && __all_sync(0xFFFFFFFFu, mbar_wait(o_full, (nt - 1) & 1, a.err) ? 1 : 0)) {
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const float inv = 1.0f / l;
      const int m = q0 + r;
      const size_t o = (size_t)(qbase + m) * a.Hq * D + (size_t)h * D;
#pragma unroll 1
      for (int c = 0; c < D; c += 16) {
        float t[16];
        tmem_ld16(tmem_o + lane_base + c, t);
        if (m < a.P) {
#pragma unroll
          for (int i = 0; i < 16; ++i) t[i] *= inv;
          if (a.out_hi) {
            float hv[16], lv[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              hv[i] = bf16_to_f32(f32_to_bf16(t[i]));
              lv[i] = t[i] - hv[i];
            }
            *reinterpret_cast<uint4*>(a.out_hi + o + c) = pack_bf16x8(hv);
            *reinterpret_cast<uint4*>(a.out_hi + o + c + 8) = pack_bf16x8(hv + 8);
            *reinterpret_cast<uint4*>(a.out_lo + o + c) = pack_bf16x8(lv);
            *reinterpret_cast<uint4*>(a.out_lo + o + c + 8) = pack_bf16x8(lv + 8);
          } else {
#pragma unroll
            for (int i = 0; i < 16; i += 4) store4(a.out + o + c + i, t + i);
          }
        }
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0 && lane == 0) {
    // Copies still in flight (a tile abandoned after an expired wait) land
    // before the CTA leaves: the last fill of each buffer, bounded.
    const int nk = static_cast<int>(*issued_k), nv = static_cast<int>(*issued_v);
    for (int j = nk > 2 ? nk - 2 : 0; j < nk; ++j)
      if (!mbar_wait(&k_full[j & 1], (j >> 1) & 1, a.err)) break;
    if (nv > 0) mbar_wait(v_full, (nv - 1) & 1, a.err);
    mbar_wait(q_full, 0, a.err);
  }
  if (warp == 1) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(C::kCols)
                 : "memory");
  }
}

// e4m3 codes -> bf16 bits of the same values (exact: every e4m3 value is a
// bf16 value); the per-row scale is applied later, in the GEMM epilogue.
__global__ void k_e4m3_to_bf16(const uint8_t* q, uint16_t* out, size_t n2) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n2;
       i += (size_t)gridDim.x * blockDim.x) {
    const uint16_t v = reinterpret_cast<const uint16_t*>(q)[i];
    const float2 f = e4m3x2_to_f32x2(v);
    reinterpret_cast<uint32_t*>(out)[i] =
        static_cast<uint32_t>(f32_to_bf16(f.x)) | (static_cast<uint32_t>(f32_to_bf16(f.y)) << 16);
  }
}

// Splits fp32 rows into bf16 hi and lo parts: hi = bf16(a), lo = bf16(a - hi).
__global__ void k_split_bf16(const float* a, uint16_t* hi, uint16_t* lo, size_t n) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    const float x = a[i];
    const uint16_t h = f32_to_bf16(x);
    hi[i] = h;
    lo[i] = f32_to_bf16(x - bf16_to_f32(h));
  }
}

// The same, four elements per step: 16-byte loads, 8-byte stores.
__global__ void k_split_bf16_x4(const float4* a, uint2* hi, uint2* lo, size_t n4) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += (size_t)gridDim.x * blockDim.x) {
    const float4 x = a[i];
    const float v[4] = {x.x, x.y, x.z, x.w};
    uint32_t h[2], l[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const uint16_t h0 = f32_to_bf16(v[2 * j]), h1 = f32_to_bf16(v[2 * j + 1]);
      const uint16_t l0 = f32_to_bf16(v[2 * j] - bf16_to_f32(h0));
      const uint16_t l1 = f32_to_bf16(v[2 * j + 1] - bf16_to_f32(h1));
      h[j] = static_cast<uint32_t>(h0) | (static_cast<uint32_t>(h1) << 16);
      l[j] = static_cast<uint32_t>(l0) | (static_cast<uint32_t>(l1) << 16);
    }
    hi[i] = make_uint2(h[0], h[1]);
    lo[i] = make_uint2(l[0], l[1]);
  }
}

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
  static EncodeTiled fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(f);
    else
      (void)cudaGetLastError();
  });
  return fn;
}

// bf16 [rows][cols] with rows `ld` elements apart (0: cols), box of 64
// columns x box_rows rows, 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
              uint64_t ld = 0) {
  EncodeTiled fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {(ld ? ld : cols) * 2};
  const cuuint32_t box[2] = {BK, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// uint8 [rows][cols] (e4m3 codes, or 4-bit rows), box of box_cols bytes x
// box_rows rows, no swizzle.
bool make_map_u8(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                 uint32_t box_cols = BK) {
  EncodeTiled fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NB, int WT>
cudaError_t launch_skinny_nb(const GemvParams& p, const CUtensorMap& mw, const CUtensorMap& mhi,
                             const CUtensorMap& mlo, const CUtensorMap& ms, int M, int S, float* part,
                             uint32_t* tickets, bool pdl, cudaStream_t s) {
  static DeviceOnce once;
  cudaError_t ea = device_once(once, [] {
    return cudaFuncSetAttribute(k_umma_skinny<NB, WT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)Skinny<NB, WT>::kSmem);
  });
  if (ea) return ea;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((p.N + 127) / 128, S);
  cfg.blockDim = dim3(kSkThreads);
  cfg.dynamicSmemBytes = Skinny<NB, WT>::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_umma_skinny<NB, WT>, mw, mhi, mlo, ms, p, M, S, part, tickets);
}

int skinny_nb(int M) { return M <= 16 ? 16 : M <= 32 ? 32 : 64; }

}  // namespace

int skinny_splits(int N, int K, int num_sms) {
  const int tiles = (N + 127) / 128, nk = (K + BK - 1) / BK;
  const int target = TF_SKINNY_CTAS_PER_SM * num_sms;
  int S = (target + tiles / 2) / tiles;
  return std::max(1, std::min(S, nk));
}

size_t skinny_part_floats(int N, int K, int M, int num_sms) {
  const int S = skinny_splits(N, K, num_sms);
  return S > 1 ? (size_t)S * ((N + 127) / 128) * 128 * skinny_nb(M) : 0;
}

cudaError_t launch_gemm_skinny(const GemvParams& p, int wt, const uint16_t* a_hi, const uint16_t* a_lo,
                               int M, float* part, uint32_t* tickets, int num_sms, bool pdl,
                               cudaStream_t s) {
  if (M < 1 || M > 64 || p.N < 2 || (p.N & 1) || p.K < 8 || (p.K % 8) || wt < 0 || wt > 2 ||
      (wt == 1 && p.K % 16) || (wt == 2 && p.K % 256))
    return cudaErrorInvalidValue;
  const int NB = skinny_nb(M);
  // activation row m is row m * in_rps + in_rps - 1 of the parts
  const int rs = p.in_rps > 1 ? p.in_rps : 1;
  const size_t a0 = (size_t)(rs - 1) * p.K;
  CUtensorMap mw, mhi, mlo, ms;
  const uint64_t qrow = (uint64_t)p.K / 2 + (uint64_t)p.K / 16;  // bytes of one 4-bit row
  bool ok = wt == 2 ? (make_map_u8(&mw, p.W, p.N, qrow, 128, 32) && make_map_u8(&ms, p.W, p.N, qrow, 128, 16))
          : wt == 1 ? make_map_u8(&mw, p.W, p.N, p.K, 128)
                    : make_map(&mw, p.W, p.N, p.K, 128);
  if (wt != 2) ms = mw;  // unused
  if (!ok || !make_map(&mhi, a_hi + a0, M, p.K, NB, (size_t)rs * p.K) ||
      !make_map(&mlo, a_lo + a0, M, p.K, NB, (size_t)rs * p.K))
    return cudaErrorInvalidValue;
  const int S = skinny_splits(p.N, p.K, num_sms);
  if (S > 1 && (!part || !tickets)) return cudaErrorInvalidValue;
#define TF_SKINNY_CASE(WTV)                                                                            \
  switch (NB) {                                                                                        \
    case 16: return launch_skinny_nb<16, WTV>(p, mw, mhi, mlo, ms, M, S, part, tickets, pdl, s);      \
    case 32: return launch_skinny_nb<32, WTV>(p, mw, mhi, mlo, ms, M, S, part, tickets, pdl, s);      \
    default: return launch_skinny_nb<64, WTV>(p, mw, mhi, mlo, ms, M, S, part, tickets, pdl, s);      \
  }
  if (wt == 2) TF_SKINNY_CASE(2)
  if (wt == 1) TF_SKINNY_CASE(1)
  TF_SKINNY_CASE(0)
#undef TF_SKINNY_CASE
}

template <int D>
cudaError_t launch_prompt_attn_d(const CUtensorMap& mqh, const CUtensorMap& mql, const CUtensorMap& mk,
                                 const CUtensorMap& mv, const PromptAttnArgs& a, cudaStream_t s) {
  static DeviceOnce once;
  cudaError_t ea = device_once(once, [] {
    return cudaFuncSetAttribute(k_umma_attn<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)PAttn<D>::kSmem);
  });
  if (ea) return ea;
  const dim3 grid((a.P + 127) / 128, a.Hq, a.nseq);
  k_umma_attn<D><<<grid, 192, PAttn<D>::kSmem, s>>>(mqh, mql, mk, mv, a);
  return cudaGetLastError();
}

bool prompt_attention_tc_supported(int D, int Hq, int Hkv) {
  return (D == 64 || D == 128) && Hkv > 0 && Hq % Hkv == 0 && encode_fn() != nullptr;
}

cudaError_t launch_prompt_attention_tc(const uint16_t* q_hi, const uint16_t* q_lo, const uint16_t* Kc,
                                       const uint16_t* Vc, int64_t kv_rows, int D,
                                       const PromptAttnArgs& a, cudaStream_t s) {
  if (!prompt_attention_tc_supported(D, a.Hq, a.Hkv) || a.P < 1 || a.nseq < 1 || a.pos0 < 0 ||
      a.pos0 + a.P > a.T)
    return cudaErrorInvalidValue;
  const uint32_t box = a.kv_tbl ? static_cast<uint32_t>(kKvPage) : 128u;
  CUtensorMap mqh, mql, mk, mv;
  const uint64_t qrows = (uint64_t)a.P * a.nseq;
  if (!make_map(&mqh, q_hi, qrows, (uint64_t)a.Hq * D, 128) || !make_map(&mql, q_lo, qrows, (uint64_t)a.Hq * D, 128) ||
      !make_map(&mk, Kc, kv_rows, D, box) || !make_map(&mv, Vc, kv_rows, D, box))
    return cudaErrorInvalidValue;
  return D == 64 ? launch_prompt_attn_d<64>(mqh, mql, mk, mv, a, s)
                 : launch_prompt_attn_d<128>(mqh, mql, mk, mv, a, s);
}

bool gemm_tc_supported(int N, int K) { return N % BN == 0 && K % BK == 0 && encode_fn() != nullptr; }

// Weight rows per tile: 256 for prompts above 512 rows where N allows (at
// 512 rows the 256-wide tiles were slower: 216 -> 233 ms for 16 x 512 ids).  Short prompts
// have few tiles and split K many ways; 256-wide partials would make the
// last CTA's reduce the bottleneck (measured: 128 ids 8.7 -> 14.7 ms).
int gemm_tc_bn(int M, int N) { return (N % 256 == 0 && M > 512) ? 256 : 128; }

// K splits of a prompt GEMM: the fewest that fill at least 80% of the last
// wave of CTAs (one CTA per SM), keeping >= 4 K slices per split; else the
// best fill found.
int gemm_tc_splits(int M, int N, int K, int num_sms, int wt) {
  const int tiles = ((M + BM - 1) / BM) * (N / (wt ? 128 : gemm_tc_bn(M, N)));
  const int smax = std::max(1, std::min(16, (K / BK) / 4));
  int best = 1;
  double best_fill = 0.0;
  for (int S = 1; S <= smax; ++S) {
    const long ctas = (long)tiles * S;
    const long waves = (ctas + num_sms - 1) / num_sms;
    const double fill = (double)ctas / ((double)waves * num_sms);
    if (fill >= 0.8) return S;
    if (fill > best_fill + 1e-9) {
      best_fill = fill;
      best = S;
    }
  }
  return best;
}

size_t gemm_tc_part_floats(int M, int N, int K, int num_sms) {
  const int S = std::max(gemm_tc_splits(M, N, K, num_sms, 0), gemm_tc_splits(M, N, K, num_sms, 1));
  return S > 1 ? (size_t)S * ((M + BM - 1) / BM) * (size_t)N * BM : 0;
}

size_t gemm_tc_smem_bytes() { return GemmCfg<256>::kSmem; }

cudaError_t launch_split_bf16(const float* a, uint16_t* hi, uint16_t* lo, size_t n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const bool v4 = n % 4 == 0 && reinterpret_cast<uintptr_t>(a) % 16 == 0 &&
                  reinterpret_cast<uintptr_t>(hi) % 8 == 0 && reinterpret_cast<uintptr_t>(lo) % 8 == 0;
  if (v4) {
    const int grid = static_cast<int>(std::min<size_t>((n / 4 + 255) / 256, 4096));
    k_split_bf16_x4<<<grid, 256, 0, s>>>(reinterpret_cast<const float4*>(a), reinterpret_cast<uint2*>(hi),
                                         reinterpret_cast<uint2*>(lo), n / 4);
  } else {
    const int grid = static_cast<int>(std::min<size_t>((n + 255) / 256, 4096));
    k_split_bf16<<<grid, 256, 0, s>>>(a, hi, lo, n);
  }
  return cudaGetLastError();
}

cudaError_t launch_e4m3_to_bf16(const uint8_t* q, uint16_t* out, size_t n, cudaStream_t s) {
  const int grid = static_cast<int>(std::min<size_t>((n / 2 + 255) / 256, 8192));
  k_e4m3_to_bf16<<<grid, 256, 0, s>>>(q, out, n / 2);
  return cudaGetLastError();
}

template <int GBN, int WT>
cudaError_t launch_gemm_tc_bn(const CUtensorMap& ma_hi, const CUtensorMap& ma_lo, const CUtensorMap& mw,
                              const CUtensorMap& ms, const GemvParams& p, int M, int S, float* part,
                              uint32_t* tickets, int num_sms, cudaStream_t s) {
  static DeviceOnce once;
  cudaError_t ea = device_once(once, [] {
    return cudaFuncSetAttribute(k_umma_gemm<GBN, WT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)GemmCfg<GBN, WT>::kSmem);
  });
  if (ea) return ea;
  // bf16 weights: one CTA per SM working through the units (two TMEM
  // accumulators); staged quantised weights: one CTA per unit, because their
  // epilogue warps are also the converters of the unit's weight slices.
  const int units = ((M + BM - 1) / BM) * (p.N / GBN) * S;
  const int grid = (WT == 0 && TF_GEMM_PERSISTENT) ? std::min(units, std::max(1, num_sms)) : units;
  k_umma_gemm<GBN, WT><<<grid, kThreads, GemmCfg<GBN, WT>::kSmem, s>>>(ma_hi, ma_lo, mw, ms, p, M, S, part,
                                                                       tickets);
  return cudaGetLastError();
}

cudaError_t launch_gemm_tc(const GemvParams& p, int wt, const uint16_t* a_hi, const uint16_t* a_lo, int M,
                           float* part, uint32_t* tickets, int num_sms, cudaStream_t s) {
  if (!gemm_tc_supported(p.N, p.K) || M < 1 || wt < 0 || wt > 2 || (wt == 2 && p.K % 256))
    return cudaErrorInvalidValue;
  const int bn = wt ? 128 : gemm_tc_bn(M, p.N);
  CUtensorMap ma_hi, ma_lo, mw, ms;
  const uint64_t qrow = (uint64_t)p.K / 2 + (uint64_t)p.K / 16;  // bytes of one 4-bit row
  const bool okw = wt == 2 ? (make_map_u8(&mw, p.W, p.N, qrow, 128, 32) && make_map_u8(&ms, p.W, p.N, qrow, 128, 16))
                 : wt == 1 ? make_map_u8(&mw, p.W, p.N, p.K, 128)
                           : make_map(&mw, p.W, p.N, p.K, bn);
  if (wt != 2) ms = mw;  // unused
  if (!okw || !make_map(&ma_hi, a_hi, M, p.K, BM) || !make_map(&ma_lo, a_lo, M, p.K, BM))
    return cudaErrorInvalidValue;
  const int S = gemm_tc_splits(M, p.N, p.K, num_sms, wt);
  if (S > 1 && (!part || !tickets)) return cudaErrorInvalidValue;
  if (wt == 2) return launch_gemm_tc_bn<128, 2>(ma_hi, ma_lo, mw, ms, p, M, S, part, tickets, num_sms, s);
  if (wt == 1) return launch_gemm_tc_bn<128, 1>(ma_hi, ma_lo, mw, ms, p, M, S, part, tickets, num_sms, s);
  return bn == 256 ? launch_gemm_tc_bn<256, 0>(ma_hi, ma_lo, mw, ms, p, M, S, part, tickets, num_sms, s)
                   : launch_gemm_tc_bn<128, 0>(ma_hi, ma_lo, mw, ms, p, M, S, part, tickets, num_sms, s);
}

}  // namespace tf
