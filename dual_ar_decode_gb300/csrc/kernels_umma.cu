// Tensor-core (tcgen05 / TMEM) GEMM for the prompt (sm_103a).
//
// Prefill runs every prompt token through the slow decoder (tuna-fish README,
// "Inference speedtest": prefill is reported separately in tokens/s); its
// linear layers are dense contractions C[m][n] = sum_k A[m][k] W[n][k] with
// m over prompt tokens, so they belong on the 5th-generation tensor cores:
//   * one CTA per 128 x 128 output tile; warp 0 streams 64-wide K slices of
//     the activation tile and the weight tile into a 4-stage shared-memory
//     ring with TMA tensor copies (128-byte swizzle), completion counted on
//     mbarriers;
//   * warp 1 owns 128 TMEM columns (the fp32 accumulator) and issues
//     tcgen05.mma kind::f16 (bf16 x bf16 -> fp32), four K=16 steps per slice;
//     tcgen05.commit frees a stage once the MMAs reading it are done;
//   * the activations enter as two bf16 parts (hi = bf16(a), lo = bf16(a -
//     hi)) multiplied by the same weight slice, so the products keep about 16
//     significant bits of the fp32 activations instead of 8;
//   * warps 2-5 wait for the final commit, read the accumulator with
//     tcgen05.ld (each warp its 32-lane quarter, one row per thread) and run
//     the decode path's fused epilogues (RoPE + KV append, residual add,
//     SwiGLU, store).
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
constexpr int kStages = 4;
constexpr int kTileA = BM * BK * 2;             // 16 KB (one bf16 part)
constexpr int kTileW = BN * BK * 2;             // 16 KB
constexpr int kStageBytes = 2 * kTileA + kTileW;  // A hi, A lo, W
constexpr int kThreads = 6 * 32;
constexpr uint32_t kTmemCols = 128;

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

// Instruction descriptor, kind::f16: fp32 accumulate, bf16 A and B, both
// K-major, M = 128, N = BN.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                            ((uint32_t)(BM >> 4) << 24);

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
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

__global__ void __launch_bounds__(kThreads, 1)
    k_umma_gemm(const __grid_constant__ CUtensorMap map_ahi,
                const __grid_constant__ CUtensorMap map_alo,
                const __grid_constant__ CUtensorMap map_w, const GemvParams p, int M) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment for the swizzled tiles
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* done = empty + kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  volatile uint32_t* consumed = tmem_slot + 2;  // K slices the MMA warp took

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * BM, n0 = blockIdx.y * BN;
  const int nk = p.K / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    *consumed = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kTmemCols)
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
      int issued = 0;
      for (int k = 0; k < nk; ++k) {
        const int s = k % kStages;
        if (k >= kStages && !mbar_wait(&empty[s], ((k / kStages) & 1) ^ 1, p.err)) {
          *abort_flag = 1;
          break;
        }
        uint8_t* st = smem + s * kStageBytes;
        mbar_arrive_expect_tx(&full[s], kStageBytes);
        tma_load_2d(st, &map_ahi, k * BK, m0, &full[s]);
        tma_load_2d(st + kTileA, &map_alo, k * BK, m0, &full[s]);
        tma_load_2d(st + 2 * kTileA, &map_w, k * BK, n0, &full[s]);
        issued = k + 1;
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
      for (int k = 0; k < nk; ++k) {
        const int s = k % kStages;
        if (*abort_flag || !mbar_wait(&full[s], (k / kStages) & 1, p.err)) {
          *abort_flag = 1;
          break;
        }
        *consumed = static_cast<uint32_t>(k + 1);
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t st = smem_u32(smem + s * kStageBytes);
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          const uint32_t a_base = st + part * kTileA;
          const uint32_t w_base = st + 2 * kTileA;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            mma_bf16(tmem, smem_desc_sw128(a_base + kk * 32), smem_desc_sw128(w_base + kk * 32),
                     (k > 0 || part > 0 || kk > 0) ? 1u : 0u);
          }
        }
        mma_commit(&empty[s]);  // frees the stage when these MMAs are done
      }
      mma_commit(done);         // accumulator complete (or abandoned)
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;       // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;
    const int m = m0 + row;
    const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(done, 0, p.err) ? 1 : 0) && !*abort_flag;
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (ok) {
#pragma unroll 1
      for (int c = 0; c < BN; c += 16) {
        float v[16];
        tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + c, v);
        if (m >= M) continue;
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
          const int n = n0 + c + i;
          float v0 = v[i], v1 = v[i + 1];
          if (p.scale) {
            v0 *= __ldg(&p.scale[n]);
            v1 *= __ldg(&p.scale[n + 1]);
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
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 1) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
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

__device__ __forceinline__ void epi_bar_sync() {
  asm volatile("bar.sync 1, 128;" ::: "memory");  // the four epilogue warps
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
constexpr int kSkThreads = 6 * 32;

// Ticket of a split-K tile: the add releases this CTA's partial (stored by
// the four epilogue warps before the barrier that precedes it) and acquires
// the partials of the CTAs that came earlier.
__device__ __forceinline__ uint32_t ticket_acq_rel(uint32_t* t) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(t) : "memory");
  return old;
}

template <int NB>
struct Skinny {
  static constexpr int kW = 128 * BK * 2;            // weight slice, 16 KB
  static constexpr int kA = NB * BK * 2;             // one activation part
  static constexpr int kStage = kW + 2 * kA;
  static constexpr uint32_t kCols = NB < 32 ? 32u : static_cast<uint32_t>(NB);
  // kind::f16, fp32 accumulate, bf16 A and B, both K-major, M = 128, N = NB.
  static constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) |
                                     ((uint32_t)(NB >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
  static constexpr size_t kSmem =
      1024 + (size_t)kSkStages * kStage + (2 * kSkStages + 2) * 8 + 64 + (64 + 4 * NB) * 4;
  // one split's partial of a tile: [NB][128] fp32
  static constexpr uint32_t kChunk = NB * 128 * 4;
  static constexpr int kChunksPerRound = (kSkStages * kStage) / kChunk;
};

template <int NB>
__global__ void __launch_bounds__(kSkThreads, NB <= 32 ? TF_SKINNY_CTAS_PER_SM : 1)
    k_umma_skinny(const __grid_constant__ CUtensorMap map_w,
                  const __grid_constant__ CUtensorMap map_ahi,
                  const __grid_constant__ CUtensorMap map_alo, const GemvParams p, int M, int S,
                  float* part, uint32_t* tickets) {
  using C = Skinny<NB>;
  static_assert(C::kStage % 1024 == 0, "stages must keep the 1024-byte swizzle alignment");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kSkStages * C::kStage);
  uint64_t* empty = full + kSkStages;
  uint64_t* done = empty + kSkStages;
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
  const size_t Np = (size_t)gridDim.x * 128;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kSkStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
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
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      for (int i = 0; i < nkb; ++i) {
        const int s = i % kSkStages;
        if (*abort_flag || !mbar_wait(&full[s], (i / kSkStages) & 1, p.err)) {
          *abort_flag = 1;
          break;
        }
        *consumed = static_cast<uint32_t>(i + 1);
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t st = smem_u32(smem + s * C::kStage);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
#pragma unroll
          for (int prt = 0; prt < 2; ++prt) {
            const uint64_t wd = smem_desc_sw128(st + kk * 32);
            const uint64_t ad = smem_desc_sw128(st + C::kW + prt * C::kA + kk * 32);
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
      }
      mma_commit(done);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    pdl_wait();
    const int q = warp & 3;
    const int et = threadIdx.x - 64;  // 0..127 over the four epilogue warps
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

template <int NB>
cudaError_t launch_skinny_nb(const GemvParams& p, const CUtensorMap& mw, const CUtensorMap& mhi,
                             const CUtensorMap& mlo, int M, int S, float* part, uint32_t* tickets,
                             bool pdl, cudaStream_t s) {
  static DeviceOnce once;
  cudaError_t ea = device_once(once, [] {
    return cudaFuncSetAttribute(k_umma_skinny<NB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)Skinny<NB>::kSmem);
  });
  if (ea) return ea;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((p.N + 127) / 128, S);
  cfg.blockDim = dim3(kSkThreads);
  cfg.dynamicSmemBytes = Skinny<NB>::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_umma_skinny<NB>, mw, mhi, mlo, p, M, S, part, tickets);
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

cudaError_t launch_gemm_skinny(const GemvParams& p, const uint16_t* a_hi, const uint16_t* a_lo,
                               int M, float* part, uint32_t* tickets, int num_sms, bool pdl,
                               cudaStream_t s) {
  if (M < 1 || M > 64 || p.N < 2 || (p.N & 1) || p.K < 8 || (p.K % 8)) return cudaErrorInvalidValue;
  const int NB = skinny_nb(M);
  // activation row m is row m * in_rps + in_rps - 1 of the parts
  const int rs = p.in_rps > 1 ? p.in_rps : 1;
  const size_t a0 = (size_t)(rs - 1) * p.K;
  CUtensorMap mw, mhi, mlo;
  if (!make_map(&mw, p.W, p.N, p.K, 128) || !make_map(&mhi, a_hi + a0, M, p.K, NB, (size_t)rs * p.K) ||
      !make_map(&mlo, a_lo + a0, M, p.K, NB, (size_t)rs * p.K))
    return cudaErrorInvalidValue;
  const int S = skinny_splits(p.N, p.K, num_sms);
  if (S > 1 && (!part || !tickets)) return cudaErrorInvalidValue;
  switch (NB) {
    case 16: return launch_skinny_nb<16>(p, mw, mhi, mlo, M, S, part, tickets, pdl, s);
    case 32: return launch_skinny_nb<32>(p, mw, mhi, mlo, M, S, part, tickets, pdl, s);
    default: return launch_skinny_nb<64>(p, mw, mhi, mlo, M, S, part, tickets, pdl, s);
  }
}

bool gemm_tc_supported(int N, int K) { return N % BN == 0 && K % BK == 0 && encode_fn() != nullptr; }

size_t gemm_tc_smem_bytes() { return 1024 + kStages * kStageBytes + (2 * kStages + 1) * 8 + 16; }

cudaError_t launch_split_bf16(const float* a, uint16_t* hi, uint16_t* lo, size_t n, cudaStream_t s) {
  const int grid = static_cast<int>(std::min<size_t>((n + 255) / 256, 4096));
  k_split_bf16<<<grid, 256, 0, s>>>(a, hi, lo, n);
  return cudaGetLastError();
}

cudaError_t launch_e4m3_to_bf16(const uint8_t* q, uint16_t* out, size_t n, cudaStream_t s) {
  const int grid = static_cast<int>(std::min<size_t>((n / 2 + 255) / 256, 8192));
  k_e4m3_to_bf16<<<grid, 256, 0, s>>>(q, out, n / 2);
  return cudaGetLastError();
}

cudaError_t launch_gemm_tc(const GemvParams& p, const uint16_t* a_hi, const uint16_t* a_lo, int M,
                           cudaStream_t s) {
  static DeviceOnce once;
  cudaError_t ea = device_once(once, [] {
    return cudaFuncSetAttribute(k_umma_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)gemm_tc_smem_bytes());
  });
  if (ea) return ea;
  if (!gemm_tc_supported(p.N, p.K) || M < 1) return cudaErrorInvalidValue;
  CUtensorMap ma_hi, ma_lo, mw;
  if (!make_map(&ma_hi, a_hi, M, p.K, BM) || !make_map(&ma_lo, a_lo, M, p.K, BM) ||
      !make_map(&mw, p.W, p.N, p.K, BN))
    return cudaErrorInvalidValue;
  dim3 grid((M + BM - 1) / BM, p.N / BN);
  k_umma_gemm<<<grid, kThreads, gemm_tc_smem_bytes(), s>>>(ma_hi, ma_lo, mw, p, M);
  return cudaGetLastError();
}

}  // namespace tf
