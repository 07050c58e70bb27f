// C ABI of the Dual-AR decode library: context, weights, prefill and the
// decode frame (declared in include/tf.h).
//
// One decode frame (fish-s2-pro-mlx-local-deploy README, architecture
// paragraph; tuna-fish README, "Inference estimation"):
//   slow:  x = text_embed[sem_base + c0(prev)]; 36 x layer; semantic head
//          (tied text-embedding slice) -> c0
//   fast:  step 1 rows [RMSNorm(x_slow), cb_embed[0][c0]] at positions 0, 1;
//          step j = 2..9 row cb_embed[j-1][c_{j-1}] at position j;
//          4 x layer each; fast head -> c_j
//   layer: QKV GEMV (RMSNorm prologue, RoPE + KV append epilogue) ->
//          attention -> O GEMV (+residual) -> gate/up GEMV (RMSNorm prologue,
//          SwiGLU epilogue) -> down GEMV (+residual)
// The whole frame is captured once as a CUDA graph whose kernels are chained
// with programmatic dependent launch, and replayed per decode call; all
// frame-varying state (position, fed-back ids, forced ids, frame index)
// lives in device memory.
//
// A batch of B sequences (lockstep, prompts of one length) runs the same
// frame with each linear layer as one skinny tensor-core GEMM over the B rows
// (the weights stream once per step for all sequences), per-sequence KV
// caches, attention and selection; the RMSNorm in front of a GEMM is deferred
// into it (RMSNorm(x) * w = rstd * (x * w), rstd applied in the epilogue).
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "../../include/tf.h"
#include "kernels.h"

using namespace tf;

namespace {

constexpr int kAlign = 256;
constexpr int kMaxBatch = 32;  // sequences per context (fast step 1: 2 rows each <= 64)
constexpr int kIdStride = 16;  // id slots per sequence in the device state
static_assert(kIdStride == kRepIds, "the repetition ring keeps one frame's id slots");
#ifndef TF_BATCH_ATTN_CTAS
#define TF_BATCH_ATTN_CTAS 2
#endif
constexpr int kBatchAttnCtasPerSm = TF_BATCH_ATTN_CTAS;  // batched attention grid density
#ifndef TF_BATCH_ATTN_STREAM
#define TF_BATCH_ATTN_STREAM 1
#endif
// Batched attention kernel: 1 = streaming (keys straight from the cache, small
// shared-memory footprint), 0 = staged (key chunks bulk-copied to shared memory).
constexpr bool kBatchAttnStream = TF_BATCH_ATTN_STREAM != 0;
#ifndef TF_SKINNY_FP8
#define TF_SKINNY_FP8 1
#endif
// Batched steps read e4m3 weights directly (converted in the GEMM's shared
// memory) instead of through a bf16 copy of each linear.
constexpr bool kSkinnyFp8 = TF_SKINNY_FP8 != 0;
thread_local std::string g_create_error;
// Failure test: the n-th following device allocation is refused (0: off).
std::atomic<int> g_fail_alloc{0};

struct Lin {
  uint8_t* w = nullptr;
  float* s = nullptr;  // per-row scales (fp8, 4-bit)
  int N = 0, K = 0;
  int wt = 0;          // storage: 0 bf16, 1 e4m3 codes, 2 block-scaled 4-bit rows
};

// Bytes of one stored row of K weights in format wt (4-bit rows: K/2 code
// bytes, then K/16 block-scale bytes).
size_t lin_row_bytes(int wt, size_t K) { return wt == 0 ? 2 * K : wt == 1 ? K : K / 2 + K / 16; }

struct Layer {
  Lin qkv, o, w13, w2;
  uint16_t* attn_norm = nullptr;
  uint16_t* ffn_norm = nullptr;
  uint16_t* q_norm = nullptr;  // per-head q/k RMSNorm weights [D] (TF_FLAG_QK_NORM*)
  uint16_t* k_norm = nullptr;
  bool paged = false;          // K/V are page pools addressed through the block table
  uint16_t* K = nullptr;  // [Hkv][T][D]
  uint16_t* V = nullptr;
};

// Device-resident frame state, per sequence slot: the next slow position,
// the frames emitted since the sequence started, whether the slot decodes,
// and a prompt id still to feed (a sequence that joined with
// tf_prefill_seq); sequence b's ids sit at [b * kIdStride + codebook].
struct DevState {
  int32_t pos[kMaxBatch];
  int32_t frame_index[kMaxBatch];
  int32_t active[kMaxBatch];
  int32_t pending[kMaxBatch];
  int32_t forced_on;
  int32_t hist_idx;
  uint32_t err;
  uint32_t samp[3];       // Philox key low, high; temperature bits
  int32_t forced[kMaxBatch * kIdStride];
  int32_t sel[kMaxBatch * kIdStride];
  int32_t fb[kMaxBatch * kIdStride];
  unsigned long long best[16];   // fused argmax of the batch-1 heads
  uint32_t ticket[16];
};

}  // namespace

struct tf_ctx {
  tf_config cfg{};
  int device = 0;
  int num_sms = 0;
  int wt = 0;        // linear weight format: 0 bf16, 1 fp8 per row, 2 block-scaled 4-bit
  bool fp8 = false;  // quantised linears (wt != 0): a float32 scale per row
  cudaStream_t own_stream = nullptr;
  cudaStream_t stream = nullptr;
  std::string err;
  bool poisoned = false;

  // sizes
  int H = 0, Q = 0, KV = 0, QKV = 0, F = 0, D = 0, Hq = 0, Hkv = 0, T = 0;
  int Vt = 0, Vs = 0, Vc = 0, NCB = 0, Vmax = 0, sem_base = 0;

  // device memory
  std::vector<void*> allocs;
  size_t device_bytes = 0;
  size_t weight_bytes = 0;
  uint8_t* wbuf = nullptr;
  std::vector<Layer> slow, fast;
  uint16_t* text_embed = nullptr;
  uint16_t* slow_norm = nullptr;
  uint16_t* fast_norm = nullptr;
  Lin fast_head;
  Lin sem;                    // semantic head: the tied text-embedding slice (bf16)
  uint16_t* cb_embed = nullptr;  // [NCB-1][Vmax][H]
  uint16_t* slow_cb = nullptr;   // [NCB-1][Vc][H] (TF_FLAG_SLOW_CB_SUM)
  float* qk_raw = nullptr;       // raw q/k pairs of a QKV GEMM (q/k norm options)
  std::vector<std::string> loaded;
  float2* rope = nullptr;
  uint8_t* staging = nullptr;
  size_t staging_bytes = 0;
  float* staging_scale = nullptr;

  float *xs = nullptr, *xf = nullptr, *qbuf = nullptr, *obuf = nullptr, *ubuf = nullptr;
  float* logits = nullptr;
  float* part = nullptr;
  uint32_t* counters = nullptr;
  float *px = nullptr, *pa = nullptr, *pq = nullptr, *po = nullptr, *pu = nullptr;
  int32_t* tokens = nullptr;
  uint16_t *a_hi = nullptr, *a_lo = nullptr;  // prompt GEMM inputs as bf16 hi / lo parts
  uint16_t *u_hi = nullptr, *u_lo = nullptr;  // the SwiGLU output as parts (down GEMM input)
  float* g_part = nullptr;                    // prompt GEMM split-K partials
  uint32_t* g_tickets = nullptr;              // one per output tile
  size_t g_part_floats = 0, g_tiles = 0;
  uint16_t* wconv = nullptr;  // fp8 weight converted to bf16 for one tensor-core GEMM
  bool prefill_tc = false;
  bool attn_tc = false;        // prompt attention on the tensor cores
  // batched decode
  int Bmax = 1;               // sequences the context holds
  int Bc = 1;                 // sequences of the current prefill
  int64_t kv_seq = 0;         // elements between two sequences' KV caches
  uint16_t* bh[2] = {nullptr, nullptr};  // skinny-GEMM activations, bf16 hi parts [64][Kmax]
  uint16_t* bl[2] = {nullptr, nullptr};  // and lo parts (two sets, alternating)
  float* sk_part = nullptr;   // split-K partials
  float* ssq = nullptr;       // deferred RMSNorm: partial sums of squares [tile][kSsqRows]
  uint32_t* sk_tickets = nullptr;
  int graph_B = 1;            // slots the captured graphs were built for
  int32_t* hist = nullptr;
  int32_t* fb_ring = nullptr;  // [Bmax][kRepRing][kRepIds] fed-back ids (repetition window)
  DevState* st = nullptr;
  int S_slow = 1;

  // host mirrors of the per-slot state (DevState) and the batch shape
  int32_t pos_host[kMaxBatch] = {};
  int32_t frame_host[kMaxBatch] = {};
  int32_t active_host[kMaxBatch] = {};
  int32_t pending_host[kMaxBatch] = {};
  bool prefilled = false;
  bool uniform = true;        // every slot at one position (lockstep batch)
  bool graph_uniform = true;  // the captured graphs' assumption
  // paged KV caches (TF_FLAG_PAGED_KV): block table [Bmax][npp] on the
  // device and its host mirror, free pages, each slot's pages in order
  bool paged = false;
  int npp = 0;
  int32_t* kv_tbl = nullptr;
  std::vector<int32_t> tbl_host;
  std::vector<int32_t> free_pages;
  std::vector<int32_t> seq_pages[kMaxBatch];

  cudaGraphExec_t graph[2] = {nullptr, nullptr};  // [0] greedy, [1] top-k
  bool inject_armed = false;  // failure test: next decode frame skips one copy
  bool inject_skip = false;   //   (consumed by the first GEMV enqueued)
  int graph_nodes = 0;
  tf_sampling graph_samp{};

};

namespace {

tf_status fail(tf_ctx* c, tf_status s, const std::string& msg) {
  c->err = msg;
  return s;
}

tf_status cuda_fail(tf_ctx* c, cudaError_t e, const char* where) {
  c->err = std::string(where) + ": " + cudaGetErrorString(e);
  c->poisoned = true;
  return TF_E_CUDA;
}

#define CK(expr)                                          \
  do {                                                    \
    cudaError_t e_ = (expr);                              \
    if (e_ != cudaSuccess) return cuda_fail(c, e_, #expr); \
  } while (0)

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

tf_status dev_alloc(tf_ctx* c, void** p, size_t bytes) {
  if (g_fail_alloc.load() > 0 && g_fail_alloc.fetch_sub(1) == 1) {
    *p = nullptr;
    return fail(c, TF_E_NOMEM, "device allocation of " + std::to_string(bytes) +
                                   " bytes refused (failure test)");
  }
  cudaError_t e = cudaMalloc(p, bytes);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    *p = nullptr;
    return fail(c, TF_E_NOMEM, "cudaMalloc of " + std::to_string(bytes) + " bytes failed");
  }
  c->allocs.push_back(*p);
  c->device_bytes += bytes;
  return TF_OK;
}

template <typename T>
tf_status dev_alloc_t(tf_ctx* c, T** p, size_t count) {
  return dev_alloc(c, reinterpret_cast<void**>(p), align_up(count * sizeof(T)));
}

bool valid_config(const tf_config* cfg, std::string* why) {
  auto bad = [&](const char* m) {
    *why = m;
    return false;
  };
  if (!cfg) return bad("cfg is NULL");
  if (cfg->slow_layers < 1 || cfg->fast_layers < 1) return bad("layers must be >= 1");
  if (cfg->head_dim != 64 && cfg->head_dim != 128) return bad("head_dim must be 64 or 128");
  if (cfg->n_kv_heads < 1 || cfg->n_heads < cfg->n_kv_heads || cfg->n_heads % cfg->n_kv_heads)
    return bad("n_heads must be a multiple of n_kv_heads");
  const int g = cfg->n_heads / cfg->n_kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8) return bad("n_heads / n_kv_heads must be 1, 2, 4 or 8");
  if (cfg->hidden < 16 || cfg->hidden % 32) return bad("hidden must be a positive multiple of 32");
  if (cfg->ffn < 16 || cfg->ffn % 32) return bad("ffn must be a positive multiple of 32");
  if ((cfg->n_heads * cfg->head_dim) % 32) return bad("n_heads*head_dim must be a multiple of 32");
  // GEMV activations live in registers: K * bytes / 16 chunks over 256 threads <= 5 each.
  const int eb = cfg->weight_dtype == TF_WEIGHT_BF16 ? 2 : 1;
  const int kmax = std::max(std::max(cfg->hidden, cfg->ffn), cfg->n_heads * cfg->head_dim);
  if (kmax * eb / 16 > 5 * 256) return bad("hidden/ffn too large for the decode GEMV");
  if (cfg->hidden > 16384) return bad("hidden too large");
  if (cfg->n_codebooks != 10) return bad("n_codebooks must be 10");
  if (cfg->semantic_vocab < 1 || cfg->semantic_vocab > cfg->text_vocab)
    return bad("semantic_vocab must be in [1, text_vocab]");
  if (cfg->semantic_vocab > 8192 || cfg->codebook_size > 8192 || cfg->codebook_size < 1)
    return bad("semantic_vocab and codebook_size must be in [1, 8192]");
  if (cfg->max_seq_len < 10 || cfg->max_seq_len > 65536) return bad("max_seq_len must be in [10, 65536]");
  if (cfg->max_batch < 1 || cfg->max_batch > kMaxBatch) return bad("max_batch must be in [1, 32]");
  if (!(cfg->rms_eps > 0.f) || !(cfg->rope_theta > 1.f)) return bad("rms_eps > 0 and rope_theta > 1 required");
  if (cfg->weight_dtype != TF_WEIGHT_BF16 && cfg->weight_dtype != TF_WEIGHT_FP8 &&
      cfg->weight_dtype != TF_WEIGHT_NVFP4)
    return bad("weight_dtype must be TF_WEIGHT_BF16, TF_WEIGHT_FP8 or TF_WEIGHT_NVFP4");
  if (cfg->weight_dtype == TF_WEIGHT_NVFP4 &&
      (cfg->hidden % 256 || cfg->ffn % 256 || (cfg->n_heads * cfg->head_dim) % 256))
    return bad("4-bit weights need hidden, ffn and n_heads*head_dim multiples of 256");
  if (cfg->flags & ~(TF_FLAG_QK_NORM | TF_FLAG_QK_NORM_FAST | TF_FLAG_SLOW_CB_SUM | TF_FLAG_PAGED_KV))
    return bad("unknown flags");
  return true;
}

tf_status check_kernel_errors(tf_ctx* c) {
  uint32_t e = 0;
  CK(cudaMemcpyAsync(&e, &c->st->err, sizeof(e), cudaMemcpyDeviceToHost, c->stream));
  CK(cudaStreamSynchronize(c->stream));
  if (!e) return TF_OK;
  if (e & ERR_TIMEOUT) {
    c->poisoned = true;
    return fail(c, TF_E_TIMEOUT, "a bounded device wait expired");
  }
  CK(cudaMemsetAsync(&c->st->err, 0, sizeof(uint32_t), c->stream));
  CK(cudaStreamSynchronize(c->stream));
  if (e & ERR_NAN) return fail(c, TF_E_NUMERIC, "NaN logit met during selection");
  c->poisoned = true;
  return fail(c, TF_E_STATE, "device reported an id or position out of range");
}

// Uploads the host mirrors of the per-slot state (positions, frame indices,
// active flags, pending prompt ids) to DevState.
tf_status upload_slots(tf_ctx* c) {
  CK(cudaMemcpyAsync(c->st->pos, c->pos_host, sizeof(c->pos_host), cudaMemcpyHostToDevice, c->stream));
  CK(cudaMemcpyAsync(c->st->frame_index, c->frame_host, sizeof(c->frame_host), cudaMemcpyHostToDevice,
                     c->stream));
  CK(cudaMemcpyAsync(c->st->active, c->active_host, sizeof(c->active_host), cudaMemcpyHostToDevice,
                     c->stream));
  CK(cudaMemcpyAsync(c->st->pending, c->pending_host, sizeof(c->pending_host), cudaMemcpyHostToDevice,
                     c->stream));
  return TF_OK;
}

// Paged caches: gives slot `slot` pages for positions 0..last (in order,
// from the free list) and uploads its block-table row if it changed.
tf_status ensure_pages(tf_ctx* c, int slot, int last) {
  if (!c->paged) return TF_OK;
  std::vector<int32_t>& mine = c->seq_pages[slot];
  const size_t need = (size_t)last / kKvPage + 1;
  if (mine.size() >= need) return TF_OK;
  while (mine.size() < need) {
    if (c->free_pages.empty()) return fail(c, TF_E_CAPACITY, "no free KV page");
    const int32_t pg = c->free_pages.back();
    c->free_pages.pop_back();
    c->tbl_host[(size_t)slot * c->npp + mine.size()] = pg;
    mine.push_back(pg);
  }
  CK(cudaMemcpyAsync(c->kv_tbl + (size_t)slot * c->npp, c->tbl_host.data() + (size_t)slot * c->npp,
                     sizeof(int32_t) * c->npp, cudaMemcpyHostToDevice, c->stream));
  return TF_OK;
}

// Frees slot `slot`: its pages go back to the free list (its block-table row
// points at the scratch page 0 again) and its state is cleared on the host.
tf_status release_slot(tf_ctx* c, int slot) {
  c->active_host[slot] = 0;
  c->pos_host[slot] = 0;
  c->frame_host[slot] = 0;
  c->pending_host[slot] = -1;
  if (!c->paged) return TF_OK;
  std::vector<int32_t>& mine = c->seq_pages[slot];
  if (mine.empty()) return TF_OK;
  for (size_t i = mine.size(); i-- > 0;) c->free_pages.push_back(mine[i]);
  mine.clear();
  std::fill(c->tbl_host.begin() + (size_t)slot * c->npp, c->tbl_host.begin() + (size_t)(slot + 1) * c->npp, 0);
  CK(cudaMemcpyAsync(c->kv_tbl + (size_t)slot * c->npp, c->tbl_host.data() + (size_t)slot * c->npp,
                     sizeof(int32_t) * c->npp, cudaMemcpyHostToDevice, c->stream));
  return TF_OK;
}

// Slots a decode step runs: up to the last active one.
int slots_in_use(const tf_ctx* c) {
  int n = 0;
  for (int b = 0; b < c->Bmax; ++b)
    if (c->active_host[b]) n = b + 1;
  return n;
}

// Sampling that needs the selection kernel (a draw or a repetition window);
// plain greedy decoding takes the argmax inside the head GEMVs.
bool uses_select(const tf_sampling* s) { return s->top_k > 0 || s->rep_window > 0; }

// ------------------------------------------------------------------ launches
#ifndef TF_GEMV_PREFETCH_BYTES
#define TF_GEMV_PREFETCH_BYTES (32 * 1024)
#endif
constexpr int kGemvPrefetch = TF_GEMV_PREFETCH_BYTES;  // per CTA, into L2, across a boundary
#ifndef TF_KV_PREFETCH
#define TF_KV_PREFETCH 1
#endif
constexpr bool kKvPrefetch = TF_KV_PREFETCH;  // QKV GEMVs hint L2 with the cached K / V rows

// The GEMV that follows in the stream (its weight is prefetched into L2).
struct NextGemv {
  const Lin* L = nullptr;
  int epi = EPI_STORE;
  int M = 1;
};

cudaError_t gemv(tf_ctx* c, const Lin& L, int pro, const float* x, const uint16_t* nw, int epi,
                 float* out, int ldo, int M, bool pdl, const Layer* layer = nullptr,
                 const int32_t* pos_ptr = nullptr, int pos_fixed = 0, int cb = -1,
                 bool select = false, const NextGemv& next = NextGemv()) {
  GemvParams p = {};
  p.W = L.w;
  p.scale = L.s;
  p.N = L.N;
  p.K = L.K;
  p.pro = pro;
  p.x = x;
  p.ldx = L.K;
  p.nw = nw;
  p.eps = c->cfg.rms_eps;
  p.epi = epi;
  p.out = out;
  p.ldo = ldo;
  p.q_dim = c->Q;
  p.kv_dim = c->KV;
  p.head_dim = c->D;
  p.qout = c->qbuf;
  if (layer) {
    p.Kc = layer->K;
    p.Vc = layer->V;
    if (layer->q_norm && epi == EPI_QKV) p.qk_raw = c->qk_raw;
    if (layer->paged) {
      p.kv_tbl = c->kv_tbl;
      p.kv_npp = c->npp;
    }
    p.kv_pf = kKvPrefetch && epi == EPI_QKV && M == 1 && !layer->paged;
  }
  p.kv_seq = c->kv_seq;
  p.T = c->T;
  p.pos_ptr = pos_ptr;
  p.pos_fixed = pos_fixed;
  p.rope = c->rope;
  p.err = &c->st->err;
  if (cb >= 0) {
    p.select = select ? 1 : 0;
    p.best = &c->st->best[cb];
    p.ticket = &c->st->ticket[cb];
    p.sel = &c->st->sel[cb];
    p.fb = &c->st->fb[cb];
    p.forced = &c->st->forced[cb];
    p.forced_on = &c->st->forced_on;
  }
  if (c->inject_skip) {
    p.test_skip_copy = 1;
    c->inject_skip = false;
  }
  gemv_plan(p, L.wt, c->num_sms, M);
  const int grid = gemv_grid(p, c->num_sms);
  if (next.L && kGemvPrefetch > 0) {
    GemvParams q = {};
    q.N = next.L->N;
    q.K = next.L->K;
    q.epi = next.epi;
    gemv_plan(q, next.L->wt, c->num_sms, next.M);
    p.pf_w = next.L->w;
    p.pf_units = q.units;
    p.pf_unit = q.unit;
    p.pf_rowbytes = static_cast<int32_t>(lin_row_bytes(next.L->wt, q.K));
    p.pf_grid = gemv_grid(q, c->num_sms);
    p.pf_bytes = kGemvPrefetch;
  }
  return launch_gemv(p, L.wt, M, grid, pdl, c->stream);
}

// The q/k norm option: finish the q and k a QKV GEMM left raw (rows at
// pos_ptr / pos_fixed, rps rows per sequence from sequence seq_base, the
// caches of `L`).
cudaError_t qknorm(tf_ctx* c, const Layer& L, int M, const int32_t* pos_ptr, int pos_fixed, int rps,
                   int seq_base, float* qout, bool pdl) {
  GemvParams p = {};
  p.q_dim = c->Q;
  p.kv_dim = c->KV;
  p.head_dim = c->D;
  p.qk_raw = c->qk_raw;
  p.q_norm = L.q_norm;
  p.k_norm = L.k_norm;
  p.eps = c->cfg.rms_eps;
  p.qout = qout;
  p.Kc = L.K;
  p.Vc = L.V;
  if (L.paged) {
    p.kv_tbl = c->kv_tbl;
    p.kv_npp = c->npp;
  }
  p.T = c->T;
  p.pos_ptr = pos_ptr;
  p.pos_fixed = pos_fixed;
  p.rps = rps;
  p.seq_base = seq_base;
  p.kv_seq = c->kv_seq;
  p.rope = c->rope;
  p.err = &c->st->err;
  return launch_qknorm(p, M, pdl, c->stream);
}

cudaError_t layer_decode(tf_ctx* c, const Layer& L, float* x, int M, const int32_t* pos_ptr,
                         int pos_fixed, int S, bool pdl_first, const NextGemv& after) {
  cudaError_t e;
  if ((e = gemv(c, L.qkv, PRO_NORM, x, L.attn_norm, EPI_QKV, nullptr, 0, M, pdl_first, &L, pos_ptr,
                pos_fixed, -1, false, NextGemv{&L.o, EPI_RESID, M})))
    return e;
  if (L.q_norm && (e = qknorm(c, L, M, pos_ptr, pos_fixed, 0, 0, c->qbuf, true))) return e;
  AttnParams a = {};
  a.q = c->qbuf;
  a.Kc = L.K;
  a.Vc = L.V;
  a.T = c->T;
  a.Hq = c->Hq;
  a.Hkv = c->Hkv;
  a.D = c->D;
  a.pos_ptr = pos_ptr;
  a.pos_fixed = pos_fixed;
  a.kv_seq = c->kv_seq;
  if (L.paged) {
    a.kv_tbl = c->kv_tbl;
    a.kv_npp = c->npp;
  }
  a.S = S;
  a.part = c->part;
  a.counters = c->counters;
  a.out = c->obuf;
  a.err = &c->st->err;
  if ((e = launch_attention(a, M, true, c->stream))) return e;
  if ((e = gemv(c, L.o, PRO_PLAIN, c->obuf, nullptr, EPI_RESID, x, c->H, M, true, nullptr, nullptr,
                0, -1, false, NextGemv{&L.w13, EPI_SWIGLU, M})))
    return e;
  if ((e = gemv(c, L.w13, PRO_NORM, x, L.ffn_norm, EPI_SWIGLU, c->ubuf, c->F, M, true, nullptr,
                nullptr, 0, -1, false, NextGemv{&L.w2, EPI_RESID, M})))
    return e;
  return gemv(c, L.w2, PRO_PLAIN, c->ubuf, nullptr, EPI_RESID, x, c->H, M, true, nullptr, nullptr, 0,
              -1, false, after);
}

cudaError_t enqueue_select(tf_ctx* c, int cb, const tf_sampling* s) {
  SelectParams q = {};
  q.logits = c->logits + (size_t)cb * c->Vmax;
  q.ld = c->Vmax;
  q.vocab = cb == 0 ? c->Vs : c->Vc;
  q.n = 1;
  q.top_k = s->top_k;
  q.temperature = s->temperature;
  q.key0 = static_cast<uint32_t>(s->seed & 0xFFFFFFFFull);
  q.key1 = static_cast<uint32_t>(s->seed >> 32);
  q.top_p = s->top_p;
  q.rep_penalty = s->rep_penalty;
  q.rep_window = s->rep_window;
  q.fb_ring = c->fb_ring;
  q.frame_ptr = c->st->frame_index;
  q.codebook0 = cb;
  q.sequence = 0;
  q.sel = &c->st->sel[cb];
  q.fb = &c->st->fb[cb];
  q.forced = &c->st->forced[cb];
  q.forced_on = &c->st->forced_on;
  q.err = &c->st->err;
  return launch_select(q, true, c->stream);
}

// Semantic head + fast loop + bookkeeping, from the slow residual xs.
cudaError_t enqueue_tail(tf_ctx* c, const tf_sampling* s, int advance, bool pdl_first) {
  cudaError_t e;
  const bool topk = uses_select(s);  // otherwise the head GEMVs take the argmax themselves
  const int Lf = static_cast<int>(c->fast.size());
  if ((e = gemv(c, c->sem, PRO_NORM, c->xs, c->slow_norm, EPI_LOGITS, c->logits, 0, 1, pdl_first,
                nullptr, nullptr, 0, 0, !topk, NextGemv{&c->fast[0].qkv, EPI_QKV, 2})))
    return e;
  if (topk && (e = enqueue_select(c, 0, s))) return e;
  for (int j = 1; j < c->NCB; ++j) {
    BuildParams b = {};
    b.mode = j == 1 ? BUILD_FAST1 : BUILD_FASTJ;
    b.j = j;
    b.H = c->H;
    b.M = j == 1 ? 2 : 1;
    b.table = c->cb_embed + (size_t)(j - 1) * c->Vmax * c->H;
    b.table_rows = j == 1 ? c->Vs : c->Vc;  // step 1 feeds code 0
    b.row_base = 0;
    b.ids = &c->st->fb[j - 1];
    b.xs = c->xs;
    b.nw = c->slow_norm;
    b.eps = c->cfg.rms_eps;
    b.x = c->xf;
    b.err = &c->st->err;
    if ((e = launch_build(b, true, c->stream))) return e;
    const int M = b.M;
    for (int i = 0; i < Lf; ++i) {
      const NextGemv after = i + 1 < Lf ? NextGemv{&c->fast[i + 1].qkv, EPI_QKV, M}
                                        : NextGemv{&c->fast_head, EPI_LOGITS, 1};
      if ((e = layer_decode(c, c->fast[i], c->xf, M, nullptr, j == 1 ? 0 : j, 1, true, after)))
        return e;
    }
    // after the last head: the next frame's first slow GEMV
    const NextGemv after_head = j + 1 < c->NCB ? NextGemv{&c->fast[0].qkv, EPI_QKV, 1}
                                               : NextGemv{&c->slow[0].qkv, EPI_QKV, 1};
    if ((e = gemv(c, c->fast_head, PRO_NORM, c->xf + (size_t)(M - 1) * c->H, c->fast_norm,
                  EPI_LOGITS, c->logits + (size_t)j * c->Vmax, 0, 1, true, nullptr, nullptr, 0, j,
                  !topk, after_head)))
      return e;
    if (topk && (e = enqueue_select(c, j, s))) return e;
  }
  FrameEndParams f = {};
  f.pos = c->st->pos;
  f.advance = advance;
  f.frame_index = c->st->frame_index;
  f.active = c->st->active;
  f.pending = c->st->pending;
  f.sel = c->st->sel;
  f.sel_stride = kIdStride;
  f.nseq = 1;
  f.ncb = c->NCB;
  f.hist = c->hist;
  f.hist_idx = &c->st->hist_idx;
  f.hist_cap = c->T;
  f.fb = c->st->fb;
  f.fb_ring = c->fb_ring;
  return launch_frame_end(f, true, c->stream);
}

// ------------------------------------------------------------ batched decode
// B > 1 sequences in lockstep: every linear layer is one skinny tensor-core
// GEMM over the B (fast step 1: 2B) activation rows, which enter as bf16
// hi / lo parts; attention, selection and the input rows work per sequence.

// Options of one skinny GEMM of the batched step.
struct SkOpt {
  const Layer* layer = nullptr;  // EPI_QKV: the layer's KV caches
  int rps = 0;                   // rows per sequence (positions, caches)
  const int32_t* pos_ptr = nullptr;
  int pos_fixed = 0;
  int out_set = -1;              // EPI_SWIGLU: the result as parts of this set
  int ssq_n = 0;                 // input rows carry a deferred RMSNorm with ssq_n
  int in_rps = 1;                //   partial sums each; row m reads row m*in_rps+in_rps-1
  const uint16_t* nw_next = nullptr;  // EPI_RESID: emit x * nw_next as parts of set 0
};

// Tiles of 128 columns over the hidden size: the partial sums of squares a
// residual GEMM leaves per row.
int hidden_tiles(const tf_ctx* c) { return (c->H + 127) / 128; }

// out = epi(W * a) for the M activation rows held in part set `set`.
cudaError_t skinny(tf_ctx* c, const Lin& L, int set, int M, int epi, float* out, int ldo,
                   const SkOpt& o = SkOpt()) {
  GemvParams p = {};
  p.W = L.w;
  p.scale = L.s;
  p.N = L.N;
  p.K = L.K;
  p.epi = epi;
  p.out = out;
  p.ldo = ldo;
  if (o.out_set >= 0) {
    p.out_hi = c->bh[o.out_set];
    p.out_lo = c->bl[o.out_set];
  }
  p.q_dim = c->Q;
  p.kv_dim = c->KV;
  p.head_dim = c->D;
  p.qout = c->qbuf;
  if (o.layer) {
    p.Kc = o.layer->K;
    p.Vc = o.layer->V;
    if (o.layer->q_norm && epi == EPI_QKV) p.qk_raw = c->qk_raw;
    if (o.layer->paged) {
      p.kv_tbl = c->kv_tbl;
      p.kv_npp = c->npp;
    }
  }
  p.pos_uniform = c->uniform ? 1 : 0;
  p.T = c->T;
  p.pos_ptr = o.pos_ptr;
  p.pos_fixed = o.pos_fixed;
  p.rps = o.rps;
  p.kv_seq = c->kv_seq;
  p.rope = c->rope;
  p.eps = c->cfg.rms_eps;
  p.err = &c->st->err;
  if (o.ssq_n > 0) {
    p.ssq_in = c->ssq;
    p.ssq_n = o.ssq_n;
    p.in_rps = o.in_rps;
  }
  if (o.nw_next) {
    p.nw_next = o.nw_next;
    p.nx_hi = c->bh[0];
    p.nx_lo = c->bl[0];
    p.ssq_out = c->ssq;
  }
  // The GEMM streams its weight slices before it waits for the previous
  // kernel (programmatic dependent launch), which is only right for weights
  // no kernel writes: a converted fp8 weight is launched without the overlap.
  // e4m3 and 4-bit weights are converted to bf16 inside the GEMM (shared
  // memory only).
  bool pdl = true;
  int wt = 0;
  if (L.wt == TF_WEIGHT_FP8 && kSkinnyFp8) {
    wt = 1;
  } else if (L.wt == TF_WEIGHT_NVFP4 && kSkinnyFp8 && L.K % 256 == 0) {
    wt = 2;
  } else if (L.s) {  // exact bf16 copy of the values; the row scale stays in p.scale
    if (cudaError_t e = L.wt == 2 ? launch_nvfp4_to_bf16(L.w, c->wconv, L.N, L.K, c->stream)
                                  : launch_e4m3_to_bf16(L.w, c->wconv, (size_t)L.N * L.K, c->stream))
      return e;
    p.W = reinterpret_cast<const uint8_t*>(c->wconv);
    pdl = false;
  }
  return launch_gemm_skinny(p, wt, c->bh[set], c->bl[set], M, c->sk_part, c->sk_tickets, c->num_sms,
                            pdl, c->stream);
}

// One decoder layer over M rows (rps rows per sequence) of the residual x.
// In: part set 0 = x * attn_norm with ssq_in partial sums of squares per row.
// Out: x updated; part set 0 = x * nw_after with hidden_tiles() sums per row.
cudaError_t layer_batched(tf_ctx* c, const Layer& L, float* x, int M, int rps,
                          const int32_t* pos_ptr, int pos_fixed, int S, int ssq_in,
                          const uint16_t* nw_after) {
  cudaError_t e;
  SkOpt q;
  q.layer = &L;
  q.rps = rps;
  q.pos_ptr = pos_ptr;
  q.pos_fixed = pos_fixed;
  q.ssq_n = ssq_in;
  if ((e = skinny(c, L.qkv, 0, M, EPI_QKV, nullptr, 0, q))) return e;
  if (L.q_norm && (e = qknorm(c, L, M, pos_ptr, pos_fixed, rps, 0, c->qbuf, true))) return e;
  AttnParams a = {};
  a.q = c->qbuf;
  a.Kc = L.K;
  a.Vc = L.V;
  a.T = c->T;
  a.Hq = c->Hq;
  a.Hkv = c->Hkv;
  a.D = c->D;
  a.pos_ptr = pos_ptr;
  a.pos_fixed = pos_fixed;
  a.rps = rps;
  a.kv_seq = c->kv_seq;
  if (L.paged) {
    a.kv_tbl = c->kv_tbl;
    a.kv_npp = c->npp;
  }
  a.S = S;
  a.part = c->part;
  a.counters = c->counters;
  a.out = c->obuf;
  a.out_hi = c->bh[1];
  a.out_lo = c->bl[1];
  a.err = &c->st->err;
  if ((e = (kBatchAttnStream ? launch_attention_rows : launch_attention)(a, M, true, c->stream)))
    return e;
  SkOpt oo;
  oo.nw_next = L.ffn_norm;
  if ((e = skinny(c, L.o, 1, M, EPI_RESID, x, c->H, oo))) return e;
  SkOpt og;
  og.out_set = 1;
  og.ssq_n = hidden_tiles(c);
  if ((e = skinny(c, L.w13, 0, M, EPI_SWIGLU, nullptr, c->F, og))) return e;
  SkOpt od;
  od.nw_next = nw_after;
  return skinny(c, L.w2, 1, M, EPI_RESID, x, c->H, od);
}

cudaError_t select_batched(tf_ctx* c, int cb, int B, const tf_sampling* s) {
  SelectParams q = {};
  q.logits = c->logits + (size_t)cb * c->Vmax;
  q.ld = c->NCB * c->Vmax;
  q.vocab = cb == 0 ? c->Vs : c->Vc;
  q.n = B;
  q.top_k = s->top_k;
  q.temperature = s->temperature;
  q.key0 = static_cast<uint32_t>(s->seed & 0xFFFFFFFFull);
  q.key1 = static_cast<uint32_t>(s->seed >> 32);
  q.top_p = s->top_p;
  q.rep_penalty = s->rep_penalty;
  q.rep_window = s->rep_window;
  q.fb_ring = c->fb_ring;
  q.frame_ptr = c->st->frame_index;
  q.codebook0 = cb;
  q.sequence = 0;
  q.seq_rows = 1;
  q.id_stride = kIdStride;
  q.sel = c->st->sel + cb;
  q.fb = c->st->fb + cb;
  q.forced = c->st->forced + cb;
  q.forced_on = &c->st->forced_on;
  q.err = &c->st->err;
  return launch_select(q, true, c->stream);
}

// Semantic heads, fast loop and bookkeeping for B sequences whose final slow
// residuals are xs[0..B).
// `prep`: xs comes from the prompt pass (not from a residual GEMM that
// already left xs * slow_norm in part set 0).
cudaError_t enqueue_tail_batched(tf_ctx* c, const tf_sampling* s, int B, int advance, bool prep) {
  cudaError_t e;
  const int ldl = c->NCB * c->Vmax;
  Lin sem;
  sem.w = reinterpret_cast<uint8_t*>(c->text_embed + (size_t)c->sem_base * c->H);
  sem.N = c->Vs;
  sem.K = c->H;
  SkOpt hs;
  hs.ssq_n = prep ? 1 : hidden_tiles(c);
  if (prep &&
      (e = launch_rows_prep(c->xs, c->H, B, c->H, c->slow_norm, c->bh[0], c->bl[0], c->ssq, true,
                            c->stream)))
    return e;
  if ((e = skinny(c, sem, 0, B, EPI_STORE, c->logits, ldl, hs))) return e;
  if ((e = select_batched(c, 0, B, s))) return e;
  const int Lf = static_cast<int>(c->fast.size());
  for (int j = 1; j < c->NCB; ++j) {
    const int rps = j == 1 ? 2 : 1;
    const int M = rps * B;
    BuildParams b = {};
    b.mode = j == 1 ? BUILD_FAST1 : BUILD_FASTJ;
    b.j = j;
    b.H = c->H;
    b.M = M;
    b.table = c->cb_embed + (size_t)(j - 1) * c->Vmax * c->H;
    b.table_rows = j == 1 ? c->Vs : c->Vc;  // step 1 feeds code 0
    b.row_base = 0;
    b.ids = c->st->fb + (j - 1);
    b.id_stride = kIdStride;
    b.xs = c->xs;
    b.nw = c->slow_norm;
    b.eps = c->cfg.rms_eps;
    b.x = c->xf;
    b.err = &c->st->err;
    b.nw_next = c->fast[0].attn_norm;
    b.nx_hi = c->bh[0];
    b.nx_lo = c->bl[0];
    b.ssq_out = c->ssq;
    if ((e = launch_build(b, true, c->stream))) return e;
    for (int i = 0; i < Lf; ++i)
      if ((e = layer_batched(c, c->fast[i], c->xf, M, rps, nullptr, j == 1 ? 0 : j, 1,
                             i == 0 ? 1 : hidden_tiles(c),
                             i + 1 < Lf ? c->fast[i + 1].attn_norm : c->fast_norm)))
        return e;
    // the head reads each sequence's last row
    SkOpt hf;
    hf.ssq_n = hidden_tiles(c);
    hf.in_rps = rps;
    if ((e = skinny(c, c->fast_head, 0, B, EPI_STORE, c->logits + (size_t)j * c->Vmax, ldl, hf)))
      return e;
    if ((e = select_batched(c, j, B, s))) return e;
  }
  FrameEndParams f = {};
  f.pos = c->st->pos;
  f.advance = advance;
  f.frame_index = c->st->frame_index;
  f.active = c->st->active;
  f.pending = c->st->pending;
  f.sel = c->st->sel;
  f.sel_stride = kIdStride;
  f.nseq = B;
  f.ncb = c->NCB;
  f.hist = c->hist;
  f.hist_idx = &c->st->hist_idx;
  f.hist_cap = c->T;
  f.fb = c->st->fb;
  f.fb_ring = c->fb_ring;
  return launch_frame_end(f, true, c->stream);
}

cudaError_t enqueue_decode_batched(tf_ctx* c, const tf_sampling* s, int B) {
  cudaError_t e;
  BuildParams b = {};
  b.mode = BUILD_SLOW;
  b.H = c->H;
  b.M = B;
  b.table = c->text_embed;
  b.table_rows = c->Vs;
  b.row_base = c->sem_base;
  b.ids = c->st->fb;
  b.id_stride = kIdStride;
  b.cb_sum = c->slow_cb;
  b.cb_rows = c->Vc;
  b.ncb = c->NCB;
  b.pending = c->st->pending;
  b.text_rows = c->Vt;
  b.x = c->xs;
  b.err = &c->st->err;
  b.nw_next = c->slow[0].attn_norm;
  b.nx_hi = c->bh[0];
  b.nx_lo = c->bl[0];
  b.ssq_out = c->ssq;
  if ((e = launch_build(b, false, c->stream))) return e;
  // Key-range splits: B * Hkv (row, KV head) pairs already spread the work,
  // so split each range only as far as a few CTAs per SM.
  const int S = std::max(1, std::min(c->S_slow, kBatchAttnCtasPerSm * c->num_sms / (B * c->Hkv)));
  const int Ls = static_cast<int>(c->slow.size());
  for (int i = 0; i < Ls; ++i)
    if ((e = layer_batched(c, c->slow[i], c->xs, B, 1, c->st->pos, 0, S,
                           i == 0 ? 1 : hidden_tiles(c),
                           i + 1 < Ls ? c->slow[i + 1].attn_norm : c->slow_norm)))
      return e;
  return enqueue_tail_batched(c, s, B, 1, false);
}

cudaError_t enqueue_decode_frame(tf_ctx* c, const tf_sampling* s) {
  if (c->Bc > 1) return enqueue_decode_batched(c, s, c->Bc);
  cudaError_t e;
  BuildParams b = {};
  b.mode = BUILD_SLOW;
  b.H = c->H;
  b.M = 1;
  b.table = c->text_embed;
  b.table_rows = c->Vs;
  b.row_base = c->sem_base;
  b.ids = &c->st->fb[0];
  b.cb_sum = c->slow_cb;
  b.cb_rows = c->Vc;
  b.ncb = c->NCB;
  b.pending = c->st->pending;
  b.text_rows = c->Vt;
  b.x = c->xs;
  b.err = &c->st->err;
  if ((e = launch_build(b, false, c->stream))) return e;
  const int Ls = static_cast<int>(c->slow.size());
  for (int i = 0; i < Ls; ++i) {
    const NextGemv after = i + 1 < Ls ? NextGemv{&c->slow[i + 1].qkv, EPI_QKV, 1}
                                      : NextGemv{&c->sem, EPI_LOGITS, 1};
    if ((e = layer_decode(c, c->slow[i], c->xs, 1, c->st->pos, 0, c->S_slow, true, after)))
      return e;
  }
  return enqueue_tail(c, s, 1, true);
}

// Prompt pass of nseq sequences with P ids each (nseq * P <= T rows): the ids
// at tokens_dev (device, [nseq][P]) at positions 0..P-1 through the slow
// decoder into slots slot .. slot + nseq - 1 (tensor-core GEMMs over all the
// rows with the decode path's epilogues, causal attention per sequence); each
// sequence's last row's residual goes to xs[its slot].
cudaError_t prompt_pass(tf_ctx* c, int slot, int nseq, const int32_t* tokens_dev, int P) {
  cudaError_t e;
  const int rows = nseq * P;
  BuildParams b = {};
  b.mode = BUILD_TOKENS;
  b.H = c->H;
  b.M = rows;
  b.table = c->text_embed;
  b.table_rows = c->Vt;
  b.ids = tokens_dev;
  b.x = c->px;
  b.err = &c->st->err;
  if ((e = launch_build(b, false, c->stream))) return e;
  // Tensor-core GEMMs take their input as bf16 hi / lo parts: written by the
  // fused RMSNorm, by the SwiGLU epilogue, or split from the attention output.
  // The CUDA-core fallback takes fp32 rows (e4m3 rows as they are; 4-bit rows
  // go through a bf16 copy).
  const bool tc = c->prefill_tc;
  const int wt = c->wt == TF_WEIGHT_FP8 ? 1 : 0;
  auto gemm = [&](const Lin& L, const float* A, const uint16_t* hi, const uint16_t* lo, int epi,
                  float* out, int ldo, const Layer* layer) {
    GemvParams p = {};
    p.W = L.w;
    p.scale = L.s;
    p.N = L.N;
    p.K = L.K;
    p.x = A;
    p.ldx = L.K;
    p.epi = epi;
    p.out = out;
    p.ldo = ldo;
    p.q_dim = c->Q;
    p.kv_dim = c->KV;
    p.head_dim = c->D;
    p.qout = c->pq;
    if (layer) {
      p.Kc = layer->K;
      p.Vc = layer->V;
      p.seq_base = slot;
      p.rps = P;  // row m: sequence slot + m / P at position m % P
      p.kv_seq = c->kv_seq;
      if (layer->paged) {
        p.kv_tbl = c->kv_tbl;
        p.kv_npp = c->npp;
      }
      if (layer->q_norm) p.qk_raw = c->qk_raw;
    }
    if (epi == EPI_SWIGLU && tc) {  // the down GEMM's input parts, no fp32 rows
      p.out_hi = c->u_hi;
      p.out_lo = c->u_lo;
    }
    p.T = c->T;
    p.pos_fixed = 0;
    p.rope = c->rope;
    p.err = &c->st->err;
    cudaError_t e2;
    if (tc) {
      // Short prompts: e4m3 and 4-bit weights stream as they are and are
      // converted in the GEMM's shared memory.  Longer prompts (more than
      // four row tiles, each converting the weight again) take one exact
      // bf16 copy per linear and the 256-wide bf16 tiles (measured: 3072
      // fp8 ids 60.0 ms this way, 75.6 ms converting in the GEMM).  The row
      // scale stays in p.scale either way.
      const bool q_in_gemm = rows <= 512;
      const int gwt = !q_in_gemm ? 0 : c->wt == TF_WEIGHT_FP8 ? 1
                      : (c->wt == TF_WEIGHT_NVFP4 && L.K % 256 == 0) ? 2 : 0;
      if (c->wt == TF_WEIGHT_NVFP4 && gwt == 0) {  // exact bf16 copy of e2m1 x block scale
        if ((e2 = launch_nvfp4_to_bf16(L.w, c->wconv, L.N, L.K, c->stream))) return e2;
        p.W = reinterpret_cast<const uint8_t*>(c->wconv);
      } else if (c->wt == TF_WEIGHT_FP8 && gwt == 0) {  // exact bf16 copy of the e4m3 values
        if ((e2 = launch_e4m3_to_bf16(L.w, c->wconv, (size_t)L.N * L.K, c->stream))) return e2;
        p.W = reinterpret_cast<const uint8_t*>(c->wconv);
      }
      return launch_gemm_tc(p, gwt, hi, lo, rows, c->g_part, c->g_tickets, c->num_sms, c->stream);
    }
    if (c->wt == TF_WEIGHT_NVFP4) {  // exact bf16 copy of e2m1 x block scale; row scale in p.scale
      if ((e2 = launch_nvfp4_to_bf16(L.w, c->wconv, L.N, L.K, c->stream))) return e2;
      p.W = reinterpret_cast<const uint8_t*>(c->wconv);
    }
    return launch_gemm_rows(p, wt, rows, c->stream);
  };
  auto norm = [&](const uint16_t* w) {
    return tc ? launch_rmsnorm_split(c->px, w, c->a_hi, c->a_lo, rows, c->H, c->cfg.rms_eps, c->stream)
              : launch_rmsnorm_rows(c->px, w, c->pa, rows, c->H, c->cfg.rms_eps, c->stream);
  };
  for (const Layer& L : c->slow) {
    if ((e = norm(L.attn_norm))) return e;
    if ((e = gemm(L.qkv, c->pa, c->a_hi, c->a_lo, EPI_QKV, nullptr, 0, &L))) return e;
    if (L.q_norm && (e = qknorm(c, L, rows, nullptr, 0, P, slot, c->pq, false))) return e;
    AttnParams a = {};
    a.q = c->pq;
    a.Kc = L.K;
    a.Vc = L.V;
    a.T = c->T;
    a.Hq = c->Hq;
    a.Hkv = c->Hkv;
    a.D = c->D;
    a.pos_fixed = 0;
    a.rps = P;
    a.seq_base = slot;
    a.kv_seq = c->kv_seq;
    if (L.paged) {
      a.kv_tbl = c->kv_tbl;
      a.kv_npp = c->npp;
    }
    a.S = 1;
    a.part = c->part;
    a.counters = c->counters;
    a.out = c->po;
    if (tc) {  // the O GEMM's input parts
      a.out_hi = c->a_hi;
      a.out_lo = c->a_lo;
    }
    a.err = &c->st->err;
    if (c->attn_tc) {
      // tensor-core causal attention; the queries as bf16 parts in the
      // (idle) SwiGLU part buffers
      if ((e = launch_split_bf16(c->pq, c->u_hi, c->u_lo, (size_t)rows * c->Q, c->stream))) return e;
      PromptAttnArgs t = {};
      t.P = P;
      t.nseq = nseq;
      t.pos0 = 0;
      t.Hq = c->Hq;
      t.Hkv = c->Hkv;
      t.T = c->T;
      t.seq = slot;
      t.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt((double)c->D));
      t.out = c->po;
      t.out_hi = a.out_hi;
      t.out_lo = a.out_lo;
      t.err = &c->st->err;
      int64_t kv_rows = (int64_t)c->Bmax * c->Hkv * c->T;  // every slot's dense cache
      if (L.paged) {
        t.kv_tbl = c->kv_tbl;
        t.kv_npp = c->npp;
        kv_rows = (int64_t)(c->Bmax * c->npp + 1) * c->Hkv * kKvPage;
      }
      if ((e = launch_prompt_attention_tc(c->u_hi, c->u_lo, L.K, L.V, kv_rows, c->D, t, c->stream))) return e;
    } else if ((e = launch_attention_rows(a, rows, false, c->stream))) {
      return e;
    }
    if ((e = gemm(L.o, c->po, c->a_hi, c->a_lo, EPI_RESID, c->px, c->H, nullptr))) return e;
    if ((e = norm(L.ffn_norm))) return e;
    if ((e = gemm(L.w13, c->pa, c->a_hi, c->a_lo, EPI_SWIGLU, c->pu, c->F, nullptr))) return e;
    if ((e = gemm(L.w2, c->pu, c->u_hi, c->u_lo, EPI_RESID, c->px, c->H, nullptr))) return e;
  }
  return cudaMemcpy2DAsync(c->xs + (size_t)slot * c->H, sizeof(float) * c->H, c->px + (size_t)(P - 1) * c->H,
                           sizeof(float) * c->H * P, sizeof(float) * c->H, nseq, cudaMemcpyDeviceToDevice,
                           c->stream);
}

bool same_sampling(const tf_sampling& a, const tf_sampling& b) {
  return a.top_k == b.top_k && a.temperature == b.temperature && a.seed == b.seed &&
         a.top_p == b.top_p && a.rep_penalty == b.rep_penalty && a.rep_window == b.rep_window;
}

tf_status get_graph(tf_ctx* c, const tf_sampling* s, cudaGraphExec_t* out) {
  if (c->graph_B != c->Bc || c->graph_uniform != c->uniform) {  // graphs are per batch shape
    for (auto& g : c->graph)
      if (g) {
        cudaGraphExecDestroy(g);
        g = nullptr;
      }
    c->graph_B = c->Bc;
    c->graph_uniform = c->uniform;
  }
  const int gi = uses_select(s) ? 1 : 0;
  if (c->graph[gi] && (gi == 0 || same_sampling(c->graph_samp, *s))) {
    *out = c->graph[gi];
    return TF_OK;
  }
  if (c->graph[gi]) {
    cudaGraphExecDestroy(c->graph[gi]);
    c->graph[gi] = nullptr;
  }
  cudaGraph_t g = nullptr;
  CK(cudaStreamBeginCapture(c->stream, cudaStreamCaptureModeThreadLocal));
  cudaError_t e = enqueue_decode_frame(c, s);
  cudaError_t e2 = cudaStreamEndCapture(c->stream, &g);
  if (e != cudaSuccess) {
    if (g) cudaGraphDestroy(g);
    return cuda_fail(c, e, "capture of the decode frame");
  }
  if (e2 != cudaSuccess) return cuda_fail(c, e2, "cudaStreamEndCapture");
  size_t n = 0;
  cudaGraphGetNodes(g, nullptr, &n);
  c->graph_nodes = static_cast<int>(n);
  cudaError_t e3 = cudaGraphInstantiate(&c->graph[gi], g, 0);
  cudaGraphDestroy(g);
  if (e3 != cudaSuccess) return cuda_fail(c, e3, "cudaGraphInstantiate");
  if (gi == 1) c->graph_samp = *s;
  *out = c->graph[gi];
  return TF_OK;
}

tf_status check_sampling(tf_ctx* c, const tf_sampling* s, tf_sampling* out) {
  tf_sampling d = {0, 1.0f, 0, 1.0f, 1.0f, 0};
  if (s) d = *s;
  if (d.top_k < 0 || d.top_k > 256) return fail(c, TF_E_INVAL, "top_k must be in [0, 256]");
  if (!(d.temperature > 0.f) || !std::isfinite(d.temperature))
    return fail(c, TF_E_INVAL, "temperature must be finite and > 0");
  if (d.top_p == 0.f) d.top_p = 1.0f;  // unset
  if (!(d.top_p > 0.f && d.top_p <= 1.0f)) return fail(c, TF_E_INVAL, "top_p must be in (0, 1]");
  if (d.rep_penalty == 0.f) d.rep_penalty = 1.0f;  // unset
  if (!(d.rep_penalty > 0.f) || !std::isfinite(d.rep_penalty))
    return fail(c, TF_E_INVAL, "rep_penalty must be finite and > 0");
  if (d.rep_window < 0 || d.rep_window > kRepRing)
    return fail(c, TF_E_INVAL, "rep_window must be in [0, 64]");
  if (d.rep_window == 0 || d.rep_penalty == 1.0f) {  // no window
    d.rep_window = 0;
    d.rep_penalty = 1.0f;
  }
  if (d.top_k == 1) d.top_k = 0;  // one candidate: the argmax
  if (d.top_k == 0) {
    d.temperature = 1.0f;
    d.seed = 0;
    d.top_p = 1.0f;
  }
  *out = d;
  return TF_OK;
}

// forced: NULL or host [B][NCB]; checked before anything is copied.
tf_status set_forced(tf_ctx* c, const int32_t* forced, int B) {
  int32_t on = forced ? 1 : 0;
  if (forced) {
    std::vector<int32_t> slots((size_t)B * kIdStride, 0);
    for (int b = 0; b < B; ++b)
      for (int j = 0; j < c->NCB; ++j) {
        const int lim = j == 0 ? c->Vs : c->Vc;
        const int32_t v = forced[(size_t)b * c->NCB + j];
        if (v < 0 || v >= lim)
          return fail(c, TF_E_INVAL, "forced id out of range at sequence " + std::to_string(b) +
                                         ", codebook " + std::to_string(j));
        slots[(size_t)b * kIdStride + j] = v;
      }
    CK(cudaMemcpyAsync(c->st->forced, slots.data(), sizeof(int32_t) * slots.size(),
                       cudaMemcpyHostToDevice, c->stream));
    CK(cudaStreamSynchronize(c->stream));  // `slots` is a host temporary
  }
  CK(cudaMemcpyAsync(&c->st->forced_on, &on, sizeof(on), cudaMemcpyHostToDevice, c->stream));
  return TF_OK;
}

// frame: host [B][NCB]; logits: NULL or host [B][NCB][Vmax].
tf_status read_frame(tf_ctx* c, int32_t* frame, float* logits, int B) {
  std::vector<int32_t> slots((size_t)B * kIdStride);
  CK(cudaMemcpyAsync(slots.data(), c->st->sel, sizeof(int32_t) * slots.size(),
                     cudaMemcpyDeviceToHost, c->stream));
  if (logits)
    CK(cudaMemcpyAsync(logits, c->logits, sizeof(float) * B * c->NCB * c->Vmax,
                       cudaMemcpyDeviceToHost, c->stream));
  tf_status r = check_kernel_errors(c);  // synchronises the stream
  if (frame)
    for (int b = 0; b < B; ++b)
      for (int j = 0; j < c->NCB; ++j)
        frame[(size_t)b * c->NCB + j] = c->active_host[b] ? slots[(size_t)b * kIdStride + j] : -1;
  return r;
}

bool all_loaded(tf_ctx* c, std::string* missing);

}  // namespace

// =================================================================== C ABI
extern "C" {

tf_status tf_create(const tf_config* cfg, int device, tf_ctx** out) {
  if (!out) {
    g_create_error = "out is NULL";
    return TF_E_INVAL;
  }
  *out = nullptr;
  std::string why;
  if (!valid_config(cfg, &why)) {
    g_create_error = why;
    return TF_E_INVAL;
  }
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) {
    (void)cudaGetLastError();
    g_create_error = "no such CUDA device";
    return TF_E_INVAL;
  }
  tf_ctx* c = new (std::nothrow) tf_ctx();
  if (!c) {
    g_create_error = "host allocation failed";
    return TF_E_NOMEM;
  }
  c->cfg = *cfg;
  c->device = device;
  auto bail = [&](tf_status s) {
    g_create_error = c->err;
    tf_destroy(c);
    return s;
  };
  if (cudaSetDevice(device) != cudaSuccess) {
    c->err = "cudaSetDevice failed";
    return bail(TF_E_CUDA);
  }
  cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, device);
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device);
  if (major * 10 + minor != 103) {
    c->err = "this library is built for sm_103 (GB300); device is sm_" + std::to_string(major * 10 + minor);
    return bail(TF_E_INVAL);
  }
  if (cudaStreamCreateWithFlags(&c->own_stream, cudaStreamNonBlocking) != cudaSuccess) {
    c->err = "cudaStreamCreate failed";
    return bail(TF_E_CUDA);
  }
  c->stream = c->own_stream;
  if (gemv_set_attributes() != cudaSuccess) {
    c->err = "cudaFuncSetAttribute failed";
    return bail(TF_E_CUDA);
  }

  c->wt = cfg->weight_dtype;
  c->fp8 = c->wt != TF_WEIGHT_BF16;
  c->Bmax = cfg->max_batch;
  c->H = cfg->hidden;
  c->D = cfg->head_dim;
  c->Hq = cfg->n_heads;
  c->Hkv = cfg->n_kv_heads;
  c->Q = c->Hq * c->D;
  c->KV = c->Hkv * c->D;
  c->QKV = c->Q + 2 * c->KV;
  c->F = cfg->ffn;
  c->T = cfg->max_seq_len;
  c->Vt = cfg->text_vocab;
  c->Vs = cfg->semantic_vocab;
  c->Vc = cfg->codebook_size;
  c->NCB = cfg->n_codebooks;
  c->Vmax = std::max(c->Vs, c->Vc);
  c->sem_base = c->Vt - c->Vs;
  c->S_slow = std::max(1, std::min(64, 2 * c->num_sms / c->Hkv));

  // ---- weights: one allocation
  const size_t H = c->H;
  auto lin_bytes = [&](size_t n, size_t k) {
    return align_up(n * lin_row_bytes(c->wt, k)) + (c->fp8 ? align_up(n * sizeof(float)) : 0);
  };
  const size_t layer_bytes = lin_bytes(c->QKV, H) + lin_bytes(H, c->Q) + lin_bytes(2 * c->F, H) +
                             lin_bytes(H, c->F) + 2 * align_up(H * 2);
  const bool qk_slow = cfg->flags & TF_FLAG_QK_NORM, qk_fast = cfg->flags & TF_FLAG_QK_NORM_FAST;
  const bool cb_sum = cfg->flags & TF_FLAG_SLOW_CB_SUM;
  const size_t qk_bytes = 2 * align_up((size_t)c->D * 2);
  size_t wtotal = align_up((size_t)c->Vt * H * 2) + (cfg->slow_layers + cfg->fast_layers) * layer_bytes +
                  2 * align_up(H * 2) + lin_bytes(c->Vc, H) +
                  align_up((size_t)(c->NCB - 1) * c->Vmax * H * 2) +
                  (qk_slow ? cfg->slow_layers * qk_bytes : 0) + (qk_fast ? cfg->fast_layers * qk_bytes : 0) +
                  (cb_sum ? align_up((size_t)(c->NCB - 1) * c->Vc * H * 2) : 0);
  if (dev_alloc(c, reinterpret_cast<void**>(&c->wbuf), wtotal) != TF_OK) return bail(TF_E_NOMEM);
  c->weight_bytes = wtotal;
  uint8_t* cur = c->wbuf;
  auto take = [&](size_t bytes) {
    uint8_t* p = cur;
    cur += align_up(bytes);
    return p;
  };
  auto make_lin = [&](int n, int k) {
    Lin L;
    L.N = n;
    L.K = k;
    L.w = take((size_t)n * lin_row_bytes(c->wt, k));
    L.wt = c->wt;
    if (c->fp8) L.s = reinterpret_cast<float*>(take((size_t)n * sizeof(float)));
    return L;
  };
  c->text_embed = reinterpret_cast<uint16_t*>(take((size_t)c->Vt * H * 2));
  auto make_layers = [&](std::vector<Layer>& v, int n, bool qk) {
    v.resize(n);
    for (Layer& L : v) {
      L.qkv = make_lin(c->QKV, c->H);
      L.o = make_lin(c->H, c->Q);
      L.w13 = make_lin(2 * c->F, c->H);
      L.w2 = make_lin(c->H, c->F);
      L.attn_norm = reinterpret_cast<uint16_t*>(take(H * 2));
      L.ffn_norm = reinterpret_cast<uint16_t*>(take(H * 2));
      if (qk) {
        L.q_norm = reinterpret_cast<uint16_t*>(take((size_t)c->D * 2));
        L.k_norm = reinterpret_cast<uint16_t*>(take((size_t)c->D * 2));
      }
    }
  };
  make_layers(c->slow, cfg->slow_layers, qk_slow);
  make_layers(c->fast, cfg->fast_layers, qk_fast);
  c->slow_norm = reinterpret_cast<uint16_t*>(take(H * 2));
  c->fast_norm = reinterpret_cast<uint16_t*>(take(H * 2));
  c->fast_head = make_lin(c->Vc, c->H);
  c->cb_embed = reinterpret_cast<uint16_t*>(take((size_t)(c->NCB - 1) * c->Vmax * H * 2));
  if (cb_sum) c->slow_cb = reinterpret_cast<uint16_t*>(take((size_t)(c->NCB - 1) * c->Vc * H * 2));
  c->sem.w = reinterpret_cast<uint8_t*>(c->text_embed + (size_t)c->sem_base * H);
  c->sem.N = c->Vs;
  c->sem.K = c->H;

  // ---- KV caches: [sequence][Hkv][T][D] per layer, or (paged) page pools
  // [page][Hkv][kKvPage][D] with one page per kKvPage positions of every
  // slot plus the scratch page 0, addressed through a block table
  const size_t kv_elems = (size_t)c->Hkv * c->T * c->D;
  c->kv_seq = static_cast<int64_t>(kv_elems);
  const size_t B = c->Bmax;
  c->paged = cfg->flags & TF_FLAG_PAGED_KV;
  c->npp = (c->T + kKvPage - 1) / kKvPage;
  const size_t n_pages = B * c->npp + 1;
  const size_t slow_kv = c->paged ? n_pages * c->Hkv * kKvPage * c->D : B * kv_elems;
  for (Layer& L : c->slow) {
    L.paged = c->paged;
    if (dev_alloc_t(c, &L.K, slow_kv) || dev_alloc_t(c, &L.V, slow_kv)) return bail(TF_E_NOMEM);
  }
  if (c->paged) {
    if (dev_alloc_t(c, &c->kv_tbl, B * c->npp)) return bail(TF_E_NOMEM);
    c->tbl_host.assign(B * c->npp, 0);
    for (size_t pg = n_pages - 1; pg >= 1; --pg) c->free_pages.push_back(static_cast<int32_t>(pg));
  }
  const size_t fkv = B * kv_elems;  // fast uses positions 0..9 of a T-slot cache
  for (Layer& L : c->fast) {
    if (dev_alloc_t(c, &L.K, fkv) || dev_alloc_t(c, &L.V, fkv)) return bail(TF_E_NOMEM);
  }

  // ---- staging for weight loads (largest linear tensor, bf16)
  size_t st = std::max({(size_t)c->QKV * H, (size_t)H * c->Q, (size_t)c->F * H, (size_t)c->Vc * H}) * 2;
  c->staging_bytes = st;
  if (dev_alloc(c, reinterpret_cast<void**>(&c->staging), st)) return bail(TF_E_NOMEM);
  if (dev_alloc_t(c, &c->staging_scale, std::max({c->QKV, c->H, c->F, c->Vc}))) return bail(TF_E_NOMEM);

  // ---- activations and state
  const int T = c->T;
  if (dev_alloc_t(c, &c->xs, B * H) || dev_alloc_t(c, &c->xf, 2 * B * H) ||
      dev_alloc_t(c, &c->qbuf, 2 * B * c->Q) || dev_alloc_t(c, &c->obuf, 2 * B * c->Q) ||
      dev_alloc_t(c, &c->ubuf, 2 * B * c->F) ||
      dev_alloc_t(c, &c->logits, B * c->NCB * c->Vmax) ||
      dev_alloc_t(c, &c->part, std::max<size_t>(2, B) * c->Hq * c->S_slow * (c->D + 2)) ||
      dev_alloc_t(c, &c->counters, 2 * B * c->Hkv) ||
      dev_alloc_t(c, &c->px, (size_t)T * H) || dev_alloc_t(c, &c->pa, (size_t)T * H) ||
      dev_alloc_t(c, &c->pq, (size_t)T * c->Q) || dev_alloc_t(c, &c->po, (size_t)T * c->Q) ||
      dev_alloc_t(c, &c->pu, (size_t)T * c->F) || dev_alloc_t(c, &c->tokens, (size_t)T * B) ||
      dev_alloc_t(c, &c->hist, (size_t)T * B * c->NCB) || dev_alloc_t(c, &c->st, 1) ||
      dev_alloc_t(c, &c->fb_ring, B * kRepRing * kRepIds) ||
      dev_alloc_t(c, &c->rope, (size_t)T * (c->D / 2)))
    return bail(TF_E_NOMEM);
  if ((qk_slow || qk_fast) &&
      dev_alloc_t(c, &c->qk_raw, (size_t)std::max<int>(T, 2 * (int)B) * (c->Q + c->KV)))
    return bail(TF_E_NOMEM);
  // Tensor-core prompt GEMMs for bf16 weights whenever every shape tiles.
  c->prefill_tc = gemm_tc_supported(c->QKV, c->H) && gemm_tc_supported(c->H, c->Q) &&
                  gemm_tc_supported(2 * c->F, c->H) && gemm_tc_supported(c->H, c->F);
  if (c->prefill_tc) {
    // split-K scratch for the largest partial set of any prompt length
    const int shapes[4][2] = {{c->QKV, c->H}, {c->H, c->Q}, {2 * c->F, c->H}, {c->H, c->F}};
    for (int m = 128; m < T + 128; m += 128)
      for (auto& sh : shapes) {
        const int M = std::min(m, T);
        c->g_part_floats = std::max(c->g_part_floats, gemm_tc_part_floats(M, sh[0], sh[1], c->num_sms));
        if (std::max(gemm_tc_splits(M, sh[0], sh[1], c->num_sms, 0), gemm_tc_splits(M, sh[0], sh[1], c->num_sms, 1)) > 1)
          c->g_tiles = std::max(c->g_tiles, (size_t)((M + 127) / 128) * (sh[0] / 128));
      }
    c->attn_tc = prompt_attention_tc_supported(c->D, c->Hq, c->Hkv) && c->F >= c->Q;
    if (dev_alloc_t(c, &c->a_hi, (size_t)T * std::max(c->H, c->Q)) ||
        dev_alloc_t(c, &c->a_lo, (size_t)T * std::max(c->H, c->Q)) ||
        dev_alloc_t(c, &c->u_hi, (size_t)T * c->F) || dev_alloc_t(c, &c->u_lo, (size_t)T * c->F) ||
        dev_alloc_t(c, &c->g_part, std::max<size_t>(c->g_part_floats, 4)) ||
        dev_alloc_t(c, &c->g_tickets, std::max<size_t>(c->g_tiles, 1)) ||
        cudaMemset(c->g_tickets, 0, std::max<size_t>(c->g_tiles, 1) * 4))
      return bail(TF_E_NOMEM);
  }
  if (c->fp8 && (c->prefill_tc || B > 1 || c->wt == TF_WEIGHT_NVFP4) &&
      dev_alloc_t(c, &c->wconv,
                  std::max({(size_t)c->QKV * H, (size_t)H * c->Q, (size_t)2 * c->F * H,
                            (size_t)H * c->F, (size_t)c->Vc * H})))
    return bail(TF_E_NOMEM);
  // Batched decode: skinny-GEMM activation parts and split-K scratch.
  if (B > 1) {
    const size_t kmax = std::max({c->H, c->Q, c->F});
    size_t part = 0;
    const int shapes[6][2] = {{c->QKV, c->H}, {c->H, c->Q}, {2 * c->F, c->H},
                              {c->H, c->F}, {c->Vs, c->H}, {c->Vc, c->H}};
    for (auto& sh : shapes)
      part = std::max(part, skinny_part_floats(sh[0], sh[1], 2 * c->Bmax, c->num_sms));
    for (int i = 0; i < 2; ++i)
      if (dev_alloc_t(c, &c->bh[i], 2 * B * kmax) || dev_alloc_t(c, &c->bl[i], 2 * B * kmax))
        return bail(TF_E_NOMEM);
    if (dev_alloc_t(c, &c->sk_part, std::max<size_t>(part, 64)) ||
        dev_alloc_t(c, &c->ssq, (size_t)((c->H + 127) / 128 + 1) * kSsqRows) ||
        dev_alloc_t(c, &c->sk_tickets, 1024) || cudaMemset(c->sk_tickets, 0, 1024 * 4)) {
      if (c->err.empty()) c->err = "batched decode buffers";
      return bail(TF_E_NOMEM);
    }
  }

  // RoPE table: angle pos * theta^(-2i/D) evaluated in double, stored as float.
  {
    std::vector<float2> tab((size_t)T * (c->D / 2));
    for (int p = 0; p < T; ++p)
      for (int i = 0; i < c->D / 2; ++i) {
        const double inv = std::pow((double)cfg->rope_theta, -2.0 * i / c->D);
        const double a = p * inv;
        tab[(size_t)p * (c->D / 2) + i] = make_float2((float)std::cos(a), (float)std::sin(a));
      }
    if (cudaMemcpy(c->rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice)) {
      c->err = "rope table upload failed";
      return bail(TF_E_CUDA);
    }
  }
  if (cudaMemset(c->st, 0, sizeof(DevState)) || cudaMemset(c->counters, 0, 2 * B * c->Hkv * 4) ||
      (c->kv_tbl && cudaMemset(c->kv_tbl, 0, B * c->npp * 4))) {
    c->err = "state init failed";
    return bail(TF_E_CUDA);
  }
  for (int b = 0; b < kMaxBatch; ++b) c->pending_host[b] = -1;
  if (upload_slots(c) != TF_OK) return bail(TF_E_CUDA);
  for (const Layer& L : c->fast) {
    cudaMemset(L.K, 0, fkv * 2);
    cudaMemset(L.V, 0, fkv * 2);
  }
  if (cudaDeviceSynchronize() != cudaSuccess) {
    c->err = "device sync failed";
    return bail(TF_E_CUDA);
  }
  *out = c;
  return TF_OK;
}

void tf_destroy(tf_ctx* c) {
  if (!c) return;
  for (auto& g : c->graph)
    if (g) cudaGraphExecDestroy(g);
  if (c->own_stream) cudaStreamSynchronize(c->own_stream);
  for (void* p : c->allocs) cudaFree(p);
  if (c->own_stream) cudaStreamDestroy(c->own_stream);
  delete c;
}

const char* tf_last_error(const tf_ctx* c) {
  if (!c) return g_create_error.c_str();
  return c->err.c_str();
}

tf_status tf_set_stream(tf_ctx* c, void* stream) {
  if (!c) return TF_E_INVAL;
  if (c->poisoned) return fail(c, TF_E_STATE, "context poisoned by an earlier error");
  CK(cudaStreamSynchronize(c->stream));
  c->stream = stream ? static_cast<cudaStream_t>(stream) : c->own_stream;
  return TF_OK;
}

void* tf_get_stream(const tf_ctx* c) { return c ? static_cast<void*>(c->stream) : nullptr; }

tf_status tf_get_info(const tf_ctx* c, tf_info* info) {
  if (!c || !info) return TF_E_INVAL;
  info->position = c->pos_host[0];
  info->frame_index = c->frame_host[0];
  info->num_sms = c->num_sms;
  info->graph_nodes = c->graph_nodes;
  info->weight_bytes = static_cast<int64_t>(c->weight_bytes);
  const int w = c->wt;
  int64_t lin = (int64_t)(c->QKV * lin_row_bytes(w, c->H) + c->H * lin_row_bytes(w, c->Q) +
                          2LL * c->F * lin_row_bytes(w, c->H) + c->H * lin_row_bytes(w, c->F));
  int64_t norms = 2LL * c->H * 2;
  int64_t slow = c->slow.size() * (lin + norms) + (int64_t)c->Vs * c->H * 2 + c->H * 2 + c->H * 2;
  int64_t fast = c->fast.size() * (lin + norms) + (int64_t)(c->Vc * lin_row_bytes(w, c->H)) + c->H * 2 +
                 c->H * 2;
  if (c->fp8) {
    slow += c->slow.size() * (int64_t)(c->QKV + c->H + 2 * c->F + c->H) * 4;
    fast += c->fast.size() * (int64_t)(c->QKV + c->H + 2 * c->F + c->H) * 4 + (int64_t)c->Vc * 4;
  }
  info->frame_weight_bytes = slow + (c->NCB - 1) * fast;
  info->device_bytes = static_cast<int64_t>(c->device_bytes);
  return TF_OK;
}

tf_status tf_load_weights(tf_ctx* c, const tf_tensor* t, int32_t n) {
  if (!c || (!t && n) || n < 0) return TF_E_INVAL;
  if (c->poisoned) return fail(c, TF_E_STATE, "context poisoned by an earlier error");
  CK(cudaSetDevice(c->device));
  for (int32_t i = 0; i < n; ++i) {
    const tf_tensor& x = t[i];
    if (!x.name || !x.data) return fail(c, TF_E_INVAL, "tensor without name or data");
    const std::string name = x.name;
    auto shape_is = [&](std::initializer_list<int64_t> s) {
      if (x.ndim != (int)s.size()) return false;
      int k = 0;
      for (int64_t v : s)
        if (x.shape[k++] != v) return false;
      return true;
    };
    auto bad_shape = [&]() { return fail(c, TF_E_INVAL, "wrong shape for " + name); };
    auto copy_raw = [&](void* dst, size_t bytes) -> tf_status {
      if (x.dtype != TF_DTYPE_BF16) return fail(c, TF_E_INVAL, name + " must be bf16");
      CK(cudaMemcpyAsync(dst, x.data, bytes, cudaMemcpyDefault, c->stream));
      return TF_OK;
    };
    auto load_lin = [&](Lin& L, int rows, int cols, int map, size_t dst_row0) -> tf_status {
      if (!shape_is({rows, cols})) return bad_shape();
      PackParams p = {};
      p.rows = rows;
      p.cols = cols;
      p.map = map;
      p.q_dim = c->Q;
      p.kv_dim = c->KV;
      p.head_dim = c->D;
      p.src = c->staging;
      p.dst = L.w + dst_row0 * lin_row_bytes(c->wt, cols);
      p.dst_scale = L.s ? L.s + dst_row0 : nullptr;
      if (x.dtype == TF_DTYPE_BF16) {
        CK(cudaMemcpyAsync(c->staging, x.data, (size_t)rows * cols * 2, cudaMemcpyDefault, c->stream));
        p.mode = c->wt == TF_WEIGHT_NVFP4 ? 4 : c->fp8 ? 1 : 0;
      } else if (x.dtype == TF_DTYPE_FP8_E4M3) {
        if (c->wt != TF_WEIGHT_FP8) return fail(c, TF_E_INVAL, name + ": fp8 tensor in a non-fp8 context");
        if (!x.row_scale) return fail(c, TF_E_INVAL, name + ": fp8 tensor without row_scale");
        CK(cudaMemcpyAsync(c->staging, x.data, (size_t)rows * cols, cudaMemcpyDefault, c->stream));
        CK(cudaMemcpyAsync(c->staging_scale, x.row_scale, (size_t)rows * 4, cudaMemcpyDefault, c->stream));
        p.src_scale = c->staging_scale;
        p.mode = 2;
        p.err = &c->st->err;
      } else {
        return fail(c, TF_E_INVAL, name + ": unknown dtype");
      }
      CK(launch_pack(p, c->stream));
      if (p.mode == 2) {
        uint32_t e = 0;
        CK(cudaMemcpyAsync(&e, &c->st->err, sizeof(e), cudaMemcpyDeviceToHost, c->stream));
        CK(cudaStreamSynchronize(c->stream));
        if (e & ERR_BAD_CODE) {
          CK(cudaMemsetAsync(&c->st->err, 0, sizeof(uint32_t), c->stream));
          CK(cudaStreamSynchronize(c->stream));
          return fail(c, TF_E_INVAL, name + ": e4m3 NaN code (0x7F or 0xFF) in the weight");
        }
      }
      return TF_OK;
    };
    tf_status s = TF_OK;
    const size_t H = c->H;
    int li = -1;
    char part[16] = {0}, field[32] = {0};
    if (name == "text_embed") {
      s = shape_is({c->Vt, c->H}) ? copy_raw(c->text_embed, (size_t)c->Vt * H * 2) : bad_shape();
    } else if (name == "slow.norm" || name == "fast.norm") {
      s = shape_is({c->H}) ? copy_raw(name[0] == 's' ? c->slow_norm : c->fast_norm, H * 2) : bad_shape();
    } else if (name == "fast.head") {
      s = load_lin(c->fast_head, c->Vc, c->H, MAP_IDENTITY, 0);
    } else if (name == "fast.cb_embed") {
      s = shape_is({c->NCB - 1, c->Vmax, c->H})
              ? copy_raw(c->cb_embed, (size_t)(c->NCB - 1) * c->Vmax * H * 2)
              : bad_shape();
    } else if (name == "slow.cb_embed" && c->slow_cb) {
      s = shape_is({c->NCB - 1, c->Vc, c->H}) ? copy_raw(c->slow_cb, (size_t)(c->NCB - 1) * c->Vc * H * 2)
                                              : bad_shape();
    } else if (std::sscanf(name.c_str(), "%15[a-z].%d.%31s", part, &li, field) == 3 &&
               (std::string(part) == "slow" || std::string(part) == "fast")) {
      std::vector<Layer>& v = std::string(part) == "slow" ? c->slow : c->fast;
      if (li < 0 || li >= (int)v.size()) return fail(c, TF_E_INVAL, "layer index out of range: " + name);
      Layer& L = v[li];
      const std::string f = field;
      if (f == "attn_norm" || f == "ffn_norm") {
        s = shape_is({c->H}) ? copy_raw(f[0] == 'a' ? L.attn_norm : L.ffn_norm, H * 2) : bad_shape();
      } else if ((f == "q_norm" || f == "k_norm") && L.q_norm) {
        s = shape_is({c->D}) ? copy_raw(f[0] == 'q' ? L.q_norm : L.k_norm, (size_t)c->D * 2) : bad_shape();
      } else if (f == "wqkv") {
        s = load_lin(L.qkv, c->QKV, c->H, MAP_QKV, 0);
      } else if (f == "wo") {
        s = load_lin(L.o, c->H, c->Q, MAP_IDENTITY, 0);
      } else if (f == "w1") {
        s = load_lin(L.w13, c->F, c->H, MAP_GATE, 0);
      } else if (f == "w3") {
        s = load_lin(L.w13, c->F, c->H, MAP_UP, 0);
      } else if (f == "w2") {
        s = load_lin(L.w2, c->H, c->F, MAP_IDENTITY, 0);
      } else {
        return fail(c, TF_E_INVAL, "unknown tensor " + name);
      }
    } else {
      return fail(c, TF_E_INVAL, "unknown tensor " + name);
    }
    if (s != TF_OK) return s;
    // The staging buffer is reused by the next tensor.
    CK(cudaStreamSynchronize(c->stream));
    bool seen = false;
    for (auto& l : c->loaded) seen |= (l == name);
    if (!seen) c->loaded.push_back(name);
  }
  CK(cudaStreamSynchronize(c->stream));
  return TF_OK;
}

}  // extern "C"

namespace {
bool all_loaded(tf_ctx* c, std::string* missing) {
  size_t need = 1 + 7 * (c->slow.size() + c->fast.size()) + 4;
  if (c->cfg.flags & TF_FLAG_QK_NORM) need += 2 * c->slow.size();
  if (c->cfg.flags & TF_FLAG_QK_NORM_FAST) need += 2 * c->fast.size();
  if (c->cfg.flags & TF_FLAG_SLOW_CB_SUM) need += 1;
  if (c->loaded.size() >= need) return true;
  *missing = std::to_string(need - c->loaded.size()) + " tensor(s) not loaded";
  return false;
}
}  // namespace

extern "C" {

tf_status tf_prefill(tf_ctx* c, const int32_t* tokens, int32_t B, int32_t P,
                     const tf_sampling* sampling, const int32_t* forced, int32_t* frame0,
                     float* logits) {
  if (!c) return TF_E_INVAL;
  if (c->poisoned) return fail(c, TF_E_STATE, "context poisoned by an earlier error");
  if (!tokens || !frame0) return fail(c, TF_E_INVAL, "tokens and frame0 are required");
  if (B < 1 || B > c->Bmax) return fail(c, TF_E_INVAL, "B must be in [1, max_batch]");
  if (P < 1 || P > c->T) return fail(c, TF_E_INVAL, "P must be in [1, max_seq_len]");
  std::string missing;
  if (!all_loaded(c, &missing)) return fail(c, TF_E_STATE, missing);
  for (int64_t i = 0; i < (int64_t)B * P; ++i)
    if (tokens[i] < 0 || tokens[i] >= c->Vt) return fail(c, TF_E_INVAL, "prompt id out of range");
  tf_sampling s;
  tf_status r = check_sampling(c, sampling, &s);
  if (r) return r;
  CK(cudaSetDevice(c->device));
  if ((r = set_forced(c, forced, B))) return r;
  // every slot starts over: B sequences at position P, the others idle
  for (int b = 0; b < c->Bmax; ++b)
    if ((r = release_slot(c, b))) return r;
  for (int b = 0; b < B; ++b) {
    if ((r = ensure_pages(c, b, P - 1))) return r;
    c->pos_host[b] = P;
    c->active_host[b] = 1;
  }
  if ((r = upload_slots(c))) return r;
  CK(cudaMemcpyAsync(c->tokens, tokens, sizeof(int32_t) * B * P, cudaMemcpyHostToDevice, c->stream));
  const int32_t zero = 0;
  CK(cudaMemcpyAsync(&c->st->hist_idx, &zero, 4, cudaMemcpyHostToDevice, c->stream));
  CK(cudaStreamSynchronize(c->stream));  // the host copies above read host memory
  c->Bc = B;
  c->uniform = true;
  c->prefilled = false;
  // as many prompts per pass as the T-row prompt buffers hold
  const int per_pass = std::max(1, c->T / P);
  for (int sb = 0; sb < B; sb += per_pass)
    CK(prompt_pass(c, sb, std::min(per_pass, B - sb), c->tokens + (size_t)sb * P, P));
  if (B > 1) {
    CK(enqueue_tail_batched(c, &s, B, 0, true));
  } else {
    CK(enqueue_tail(c, &s, 0, false));
  }
  for (int b = 0; b < B; ++b) c->frame_host[b] = 1;
  c->prefilled = true;
  return read_frame(c, frame0, logits, B);
}

tf_status tf_prefill_seq(tf_ctx* c, int32_t slot, const int32_t* tokens, int32_t P) {
  if (!c) return TF_E_INVAL;
  if (c->poisoned) return fail(c, TF_E_STATE, "context poisoned by an earlier error");
  if (!tokens) return fail(c, TF_E_INVAL, "tokens are required");
  if (slot < 0 || slot >= c->Bmax) return fail(c, TF_E_INVAL, "slot must be in [0, max_batch)");
  if (P < 1 || P > c->T) return fail(c, TF_E_INVAL, "P must be in [1, max_seq_len]");
  std::string missing;
  if (!all_loaded(c, &missing)) return fail(c, TF_E_STATE, missing);
  for (int32_t i = 0; i < P; ++i)
    if (tokens[i] < 0 || tokens[i] >= c->Vt) return fail(c, TF_E_INVAL, "prompt id out of range");
  CK(cudaSetDevice(c->device));
  tf_status r;
  if ((r = release_slot(c, slot))) return r;
  if ((r = ensure_pages(c, slot, P - 1))) return r;
  if (P > 1) {  // every prompt id but the last through the prompt pass
    CK(cudaMemcpyAsync(c->tokens, tokens, sizeof(int32_t) * (P - 1), cudaMemcpyHostToDevice, c->stream));
    CK(cudaStreamSynchronize(c->stream));
    CK(prompt_pass(c, slot, 1, c->tokens, P - 1));
  }
  // the last prompt id is fed by the next decode step, which emits frame 0
  c->pos_host[slot] = P - 1;
  c->frame_host[slot] = 0;
  c->active_host[slot] = 1;
  c->pending_host[slot] = tokens[P - 1];
  if ((r = upload_slots(c))) return r;
  CK(cudaStreamSynchronize(c->stream));
  c->Bc = slots_in_use(c);
  c->uniform = false;
  c->prefilled = true;
  return TF_OK;
}

tf_status tf_release_seq(tf_ctx* c, int32_t slot) {
  if (!c) return TF_E_INVAL;
  if (c->poisoned) return fail(c, TF_E_STATE, "context poisoned by an earlier error");
  if (slot < 0 || slot >= c->Bmax) return fail(c, TF_E_INVAL, "slot must be in [0, max_batch)");
  CK(cudaSetDevice(c->device));
  tf_status r;
  if ((r = release_slot(c, slot))) return r;
  if ((r = upload_slots(c))) return r;
  CK(cudaStreamSynchronize(c->stream));
  c->Bc = std::max(1, slots_in_use(c));
  return TF_OK;
}

// Checks that every active slot can take n more frames and gives the paged
// caches the pages they will write.
static tf_status reserve_frames(tf_ctx* c, int n) {
  if (!slots_in_use(c)) return fail(c, TF_E_STATE, "no active sequence");
  for (int b = 0; b < c->Bc; ++b)
    if (c->active_host[b] && c->pos_host[b] + n > c->T)
      return fail(c, TF_E_CAPACITY, "KV cache full (slot " + std::to_string(b) + ")");
  for (int b = 0; b < c->Bc; ++b)
    if (c->active_host[b])
      if (tf_status r = ensure_pages(c, b, c->pos_host[b] + n - 1)) return r;
  return TF_OK;
}

// Host mirrors after n decode frames: every active slot advanced.
static void advance_slots(tf_ctx* c, int n) {
  for (int b = 0; b < c->Bc; ++b)
    if (c->active_host[b]) {
      c->pos_host[b] += n;
      c->frame_host[b] += n;
      c->pending_host[b] = -1;
    }
}

tf_status tf_decode_frame(tf_ctx* c, const tf_sampling* sampling, const int32_t* forced,
                          int32_t* frame, float* logits) {
  if (!c) return TF_E_INVAL;
  if (c->poisoned) return fail(c, TF_E_STATE, "context poisoned by an earlier error");
  if (!frame) return fail(c, TF_E_INVAL, "frame is required");
  if (!c->prefilled) return fail(c, TF_E_STATE, "tf_prefill must come first");
  tf_sampling s;
  tf_status r = check_sampling(c, sampling, &s);
  if (r) return r;
  CK(cudaSetDevice(c->device));
  if ((r = reserve_frames(c, 1))) return r;
  if ((r = set_forced(c, forced, c->Bc))) return r;
  if (c->inject_armed && c->Bc == 1) {
    // failure test: this frame runs outside the graph, its first GEMV
    // skipping one weight copy
    c->inject_armed = false;
    c->inject_skip = true;
    cudaError_t e = enqueue_decode_frame(c, &s);
    c->inject_skip = false;
    CK(e);
  } else {
    cudaGraphExec_t g;
    if ((r = get_graph(c, &s, &g))) return r;
    CK(cudaGraphLaunch(g, c->stream));
  }
  advance_slots(c, 1);
  return read_frame(c, frame, logits, c->Bc);
}

tf_status tf_test_inject(tf_ctx* c, int32_t what) {
  if (!c || what != TF_TEST_SKIP_ONE_COPY) return TF_E_INVAL;
  if (c->poisoned) return fail(c, TF_E_STATE, "context poisoned by an earlier error");
  if (c->Bmax != 1) return fail(c, TF_E_INVAL, "the copy-skip test needs a batch-1 context");
  c->inject_armed = true;
  return TF_OK;
}

void tf_test_fail_alloc(int32_t n) { g_fail_alloc.store(n > 0 ? n : 0); }

tf_status tf_decode_frames(tf_ctx* c, const tf_sampling* sampling, int32_t n, int32_t* frames) {
  if (!c) return TF_E_INVAL;
  if (c->poisoned) return fail(c, TF_E_STATE, "context poisoned by an earlier error");
  if (n < 0 || (n > 0 && !frames)) return fail(c, TF_E_INVAL, "bad n or frames");
  if (!c->prefilled) return fail(c, TF_E_STATE, "tf_prefill must come first");
  if (n == 0) return TF_OK;
  tf_sampling s;
  tf_status r = check_sampling(c, sampling, &s);
  if (r) return r;
  CK(cudaSetDevice(c->device));
  if ((r = reserve_frames(c, n))) return r;
  if ((r = set_forced(c, nullptr, c->Bc))) return r;
  const int32_t zero = 0;
  CK(cudaMemcpyAsync(&c->st->hist_idx, &zero, 4, cudaMemcpyHostToDevice, c->stream));
  cudaGraphExec_t g;
  if ((r = get_graph(c, &s, &g))) return r;
  for (int i = 0; i < n; ++i) CK(cudaGraphLaunch(g, c->stream));
  CK(cudaMemcpyAsync(frames, c->hist, sizeof(int32_t) * c->NCB * c->Bc * n, cudaMemcpyDeviceToHost,
                     c->stream));
  r = check_kernel_errors(c);  // synchronises the stream
  for (int i = 0; i < n; ++i)   // idle slots report -1
    for (int b = 0; b < c->Bc; ++b)
      if (!c->active_host[b])
        for (int j = 0; j < c->NCB; ++j) frames[((size_t)i * c->Bc + b) * c->NCB + j] = -1;
  advance_slots(c, n);
  return r;
}

tf_status tf_profile_kernel(tf_ctx* c, int32_t which, int32_t iters, float* ms_per_launch,
                            int64_t* bytes_per_launch) {
  if (!c || iters < 1 || which < 0 || which > 7) return TF_E_INVAL;
  if (c->poisoned) return fail(c, TF_E_STATE, "context poisoned by an earlier error");
  const bool batched = which >= 4;
  if (batched && c->Bmax < 2) return fail(c, TF_E_INVAL, "skinny-GEMM kernels need max_batch > 1");
  std::string missing;
  if (!all_loaded(c, &missing)) return fail(c, TF_E_STATE, missing);
  CK(cudaSetDevice(c->device));
  const int Ls = static_cast<int>(c->slow.size());
  const int Lf = static_cast<int>(c->fast.size());
  const int M = batched ? c->Bmax : 1;
  const int kind = which & 3;
  // Scratch input rows: finite values in every activation buffer the kernel reads.
  std::vector<float> ones(std::max({c->H, c->Q, c->F}), 0.01f);
  CK(cudaMemcpyAsync(c->pa, ones.data(), sizeof(float) * c->H, cudaMemcpyHostToDevice, c->stream));
  CK(cudaMemcpyAsync(c->po, ones.data(), sizeof(float) * c->Q, cudaMemcpyHostToDevice, c->stream));
  CK(cudaMemcpyAsync(c->pu, ones.data(), sizeof(float) * c->F, cudaMemcpyHostToDevice, c->stream));
  if (batched) {
    const size_t n = (size_t)2 * c->Bmax * std::max({c->H, c->Q, c->F});
    std::vector<uint16_t> hi(n, 0x3c24), lo(n, 0);  // bf16(0.01) and 0
    for (int i = 0; i < 2; ++i) {
      CK(cudaMemcpyAsync(c->bh[i], hi.data(), n * 2, cudaMemcpyHostToDevice, c->stream));
      CK(cudaMemcpyAsync(c->bl[i], lo.data(), n * 2, cudaMemcpyHostToDevice, c->stream));
    }
    std::vector<float> ss((size_t)hidden_tiles(c) * kSsqRows, 1.0f);
    CK(cudaMemcpyAsync(c->ssq, ss.data(), ss.size() * 4, cudaMemcpyHostToDevice, c->stream));
    CK(cudaMemsetAsync(c->xf, 0, sizeof(float) * 2 * c->Bmax * c->H, c->stream));
    CK(cudaStreamSynchronize(c->stream));
  }
  CK(cudaStreamSynchronize(c->stream));
  // The QKV epilogue appends K/V rows: it writes position 0 of the fast
  // decoder's caches, which every frame rewrites before it reads them.
  auto launch = [&](int i, bool pdl) -> cudaError_t {
    const Layer& L = c->slow[i % Ls];
    const Layer& F = c->fast[i % Lf];
    if (batched) {  // as in the frame: deferred RMSNorm in and out
      SkOpt o;
      switch (kind) {
        case 0:
          o.out_set = 1;
          o.ssq_n = hidden_tiles(c);
          return skinny(c, L.w13, 0, M, EPI_SWIGLU, nullptr, c->F, o);
        case 1:
          o.layer = &F;
          o.rps = 1;
          o.ssq_n = hidden_tiles(c);
          return skinny(c, L.qkv, 0, M, EPI_QKV, nullptr, 0, o);
        case 2:
          o.nw_next = L.ffn_norm;
          return skinny(c, L.o, 1, M, EPI_RESID, c->xf, c->H, o);
        default:
          o.nw_next = L.attn_norm;
          return skinny(c, L.w2, 1, M, EPI_RESID, c->xf, c->H, o);
      }
    }
    switch (kind) {
      case 0: return gemv(c, L.w13, PRO_NORM, c->pa, L.ffn_norm, EPI_SWIGLU, c->pq, c->F, 1, pdl);
      case 1: return gemv(c, L.qkv, PRO_NORM, c->pa, L.attn_norm, EPI_QKV, nullptr, 0, 1, pdl, &F,
                          nullptr, 0);
      case 2: return gemv(c, L.o, PRO_PLAIN, c->po, nullptr, EPI_RESID, c->px, c->H, 1, pdl);
      default: return gemv(c, L.w2, PRO_PLAIN, c->pu, nullptr, EPI_RESID, c->px, c->H, 1, pdl);
    }
  };
  // The launches are captured once as a graph (as the decode frame is), so
  // the time is the device's and not the host's launch rate; one warm-up
  // replay, then the timed one.
  cudaGraph_t g = nullptr;
  cudaGraphExec_t ge = nullptr;
  CK(cudaStreamBeginCapture(c->stream, cudaStreamCaptureModeThreadLocal));
  cudaError_t le = cudaSuccess;
  for (int i = 0; i < iters && le == cudaSuccess; ++i) le = launch(i, i > 0);
  cudaError_t ce = cudaStreamEndCapture(c->stream, &g);
  if (le != cudaSuccess || ce != cudaSuccess) {
    if (g) cudaGraphDestroy(g);
    return cuda_fail(c, le != cudaSuccess ? le : ce, "capture of the profiled launches");
  }
  cudaError_t ie = cudaGraphInstantiate(&ge, g, 0);
  cudaGraphDestroy(g);
  if (ie != cudaSuccess) return cuda_fail(c, ie, "cudaGraphInstantiate");
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  float ms = 0.f;
  cudaError_t te = cudaGraphLaunch(ge, c->stream);
  if (!te) te = cudaEventCreate(&e0);
  if (!te) te = cudaEventCreate(&e1);
  if (!te) te = cudaEventRecord(e0, c->stream);
  if (!te) te = cudaGraphLaunch(ge, c->stream);
  if (!te) te = cudaEventRecord(e1, c->stream);
  if (!te) te = cudaEventSynchronize(e1);
  if (!te) te = cudaEventElapsedTime(&ms, e0, e1);
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  cudaGraphExecDestroy(ge);
  if (te) return cuda_fail(c, te, "timing of the profiled launches");
  if (ms_per_launch) *ms_per_launch = ms / iters;
  const Layer& L0 = c->slow[0];
  const Lin& lin = kind == 0 ? L0.w13 : kind == 1 ? L0.qkv : kind == 2 ? L0.o : L0.w2;
  int64_t bytes = (int64_t)(lin.N * lin_row_bytes(c->wt, lin.K)) + (c->fp8 ? (int64_t)lin.N * 4 : 0);
  if (batched) {
    bytes += (int64_t)M * lin.K * 4;                   // activation rows in (bf16 hi + lo)
    bytes += (int64_t)M * (kind == 0 ? (int64_t)c->F * 4 : kind == 1 ? (int64_t)(c->Q * 4 + 2 * c->KV * 2)
                                                             : (int64_t)c->H * 8);
  } else {
    bytes += (int64_t)lin.K * 4;                        // activation row in
    if (kind == 0 || kind == 1) bytes += (int64_t)lin.K * 2;  // RMSNorm weight
    bytes += kind == 0 ? (int64_t)c->F * 4 : kind == 1 ? (int64_t)(c->Q * 4 + 2 * c->KV * 2)
                                                       : (int64_t)c->H * 8;  // out (+ residual read)
  }
  if (bytes_per_launch) *bytes_per_launch = bytes;
  return check_kernel_errors(c);
}

// ------------------------------------------------------------------ ops
tf_status tf_op_quantize_fp8(const uint16_t* w, int64_t rows, int64_t cols, uint8_t* codes,
                             float* scale, void* stream) {
  if (!w || !codes || !scale || rows < 1 || cols < 16 || cols % 16 || rows > (1 << 30))
    return TF_E_INVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  PackParams p = {};
  p.src = reinterpret_cast<const uint8_t*>(w);
  p.dst = codes;
  p.dst_scale = scale;
  p.rows = rows;
  p.cols = cols;
  p.map = MAP_IDENTITY;
  p.mode = 1;
  if (launch_pack(p, s) != cudaSuccess) return TF_E_CUDA;
  return cudaStreamSynchronize(s) == cudaSuccess ? TF_OK : TF_E_CUDA;
}

tf_status tf_op_quantize_nvfp4(const uint16_t* w, int64_t rows, int64_t cols, uint8_t* packed,
                               float* row_scale, void* stream) {
  if (!w || !packed || !row_scale || rows < 1 || cols < 256 || cols % 256 || rows > (1 << 30))
    return TF_E_INVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  PackParams p = {};
  p.src = reinterpret_cast<const uint8_t*>(w);
  p.dst = packed;
  p.dst_scale = row_scale;
  p.rows = rows;
  p.cols = cols;
  p.map = MAP_IDENTITY;
  p.mode = 4;
  if (launch_pack(p, s) != cudaSuccess) return TF_E_CUDA;
  return cudaStreamSynchronize(s) == cudaSuccess ? TF_OK : TF_E_CUDA;
}

tf_status tf_op_select(const float* logits, int32_t n, int32_t vocab, const tf_sampling* sampling,
                       int32_t frame, int32_t codebook0, int32_t sequence, const int32_t* recent,
                       int32_t n_recent, int32_t* ids, void* stream) {
  if (!logits || !ids || !sampling || n < 1 || vocab < 1 || vocab > 8192) return TF_E_INVAL;
  if (sampling->top_k < 0 || sampling->top_k > 256 || !(sampling->temperature > 0.f)) return TF_E_INVAL;
  if (!(sampling->top_p >= 0.f && sampling->top_p <= 1.0f) || !(sampling->rep_penalty >= 0.f) ||
      n_recent < 0 || n_recent > kRepRing || (n_recent > 0 && !recent))
    return TF_E_INVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t* err = nullptr;
  if (cudaMalloc(&err, sizeof(uint32_t)) != cudaSuccess) return TF_E_NOMEM;
  cudaMemsetAsync(err, 0, 4, s);
  SelectParams q = {};
  q.logits = logits;
  q.ld = vocab;
  q.vocab = vocab;
  q.n = n;
  q.top_k = sampling->top_k;
  q.temperature = sampling->temperature;
  q.top_p = sampling->top_p == 0.f ? 1.0f : sampling->top_p;
  q.rep_penalty = sampling->rep_penalty == 0.f ? 1.0f : sampling->rep_penalty;
  q.recent = n_recent > 0 ? recent : nullptr;
  q.n_recent = n_recent;
  q.key0 = static_cast<uint32_t>(sampling->seed & 0xFFFFFFFFull);
  q.key1 = static_cast<uint32_t>(sampling->seed >> 32);
  q.frame = frame;
  q.codebook0 = codebook0;
  q.sequence = sequence;
  q.sel = ids;
  q.err = err;
  tf_status r = TF_OK;
  if (launch_select(q, false, s) != cudaSuccess) r = TF_E_CUDA;
  uint32_t e = 0;
  if (r == TF_OK && (cudaMemcpyAsync(&e, err, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
                     cudaStreamSynchronize(s) != cudaSuccess))
    r = TF_E_CUDA;
  cudaFree(err);
  if (r == TF_OK && (e & ERR_NAN)) r = TF_E_NUMERIC;
  return r;
}

tf_status tf_op_attention(const float* q, const uint16_t* K, const uint16_t* V, int32_t T,
                          int32_t Hq, int32_t Hkv, int32_t D, int32_t rows, int32_t pos0,
                          int32_t splits, float* out, void* stream) {
  if (!q || !K || !V || !out || T < 1 || Hq < 1 || Hkv < 1 || rows < 1 || pos0 < 0 ||
      (int64_t)pos0 + rows > T || splits < 1 || splits > 64 || rows > 65535)
    return TF_E_INVAL;
  if ((D != 64 && D != 128) || Hq % Hkv) return TF_E_INVAL;
  const int g = Hq / Hkv;
  if (g != 1 && g != 2 && g != 4 && g != 8) return TF_E_INVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t part_bytes = (size_t)rows * Hq * splits * (D + 2) * sizeof(float);
  const size_t cnt_bytes = (size_t)rows * Hkv * sizeof(uint32_t);
  float* part = nullptr;
  uint32_t* cnt = nullptr;
  uint32_t* err = nullptr;
  if (cudaMalloc(&part, part_bytes) != cudaSuccess || cudaMalloc(&cnt, cnt_bytes) != cudaSuccess ||
      cudaMalloc(&err, sizeof(uint32_t)) != cudaSuccess) {
    (void)cudaGetLastError();
    cudaFree(part);
    cudaFree(cnt);
    cudaFree(err);
    return TF_E_NOMEM;
  }
  tf_status r = TF_OK;
  if (cudaMemsetAsync(cnt, 0, cnt_bytes, s) != cudaSuccess || cudaMemsetAsync(err, 0, 4, s) != cudaSuccess)
    r = TF_E_CUDA;
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
  if (r == TF_OK && launch_attention(a, rows, false, s) != cudaSuccess) r = TF_E_CUDA;
  uint32_t e = 0;
  if (r == TF_OK && (cudaMemcpyAsync(&e, err, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
                     cudaStreamSynchronize(s) != cudaSuccess))
    r = TF_E_CUDA;
  cudaFree(part);
  cudaFree(cnt);
  cudaFree(err);
  if (r == TF_OK && (e & ERR_TIMEOUT)) r = TF_E_TIMEOUT;
  else if (r == TF_OK && e) r = TF_E_INVAL;
  return r;
}

tf_status tf_op_attention_prompt(const float* q, const uint16_t* K, const uint16_t* V, int32_t T,
                                 int32_t Hq, int32_t Hkv, int32_t D, int32_t rows, int32_t pos0,
                                 float* out, void* stream) {
  if (!q || !K || !V || !out || T < 1 || Hq < 1 || Hkv < 1 || rows < 1 || pos0 < 0 ||
      (int64_t)pos0 + rows > T || !prompt_attention_tc_supported(D, Hq, Hkv) ||
      (int64_t)Hkv * T * D >= (1ll << 40))
    return TF_E_INVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t n = (size_t)rows * Hq * D;
  uint16_t *hi = nullptr, *lo = nullptr;
  uint32_t* err = nullptr;
  if (cudaMalloc(&hi, n * 2) != cudaSuccess || cudaMalloc(&lo, n * 2) != cudaSuccess ||
      cudaMalloc(&err, 4) != cudaSuccess) {
    (void)cudaGetLastError();
    cudaFree(hi);
    cudaFree(lo);
    cudaFree(err);
    return TF_E_NOMEM;
  }
  PromptAttnArgs a = {};
  a.P = rows;
  a.nseq = 1;
  a.pos0 = pos0;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.T = T;
  a.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt((double)D));
  a.out = out;
  a.err = err;
  tf_status r = TF_OK;
  if (cudaMemsetAsync(err, 0, 4, s) != cudaSuccess || launch_split_bf16(q, hi, lo, n, s) != cudaSuccess ||
      launch_prompt_attention_tc(hi, lo, K, V, (int64_t)Hkv * T, D, a, s) != cudaSuccess)
    r = TF_E_CUDA;
  uint32_t e = 0;
  if (r == TF_OK && (cudaMemcpyAsync(&e, err, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
                     cudaStreamSynchronize(s) != cudaSuccess))
    r = TF_E_CUDA;
  cudaFree(hi);
  cudaFree(lo);
  cudaFree(err);
  if (r == TF_OK && (e & ERR_TIMEOUT)) r = TF_E_TIMEOUT;
  else if (r == TF_OK && e) r = TF_E_INVAL;
  return r;
}

tf_status tf_op_gemm(const float* A, const uint16_t* W, int32_t M, int32_t N, int32_t K, float* C,
                     void* stream) {
  if (!A || !W || !C || M < 1 || N < 1 || K < 1 || !gemm_tc_supported(N, K)) return TF_E_INVAL;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return TF_E_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint16_t *hi = nullptr, *lo = nullptr;
  uint32_t *err = nullptr, *tickets = nullptr;
  float* part = nullptr;
  const size_t n = (size_t)M * K;
  const size_t pf = std::max<size_t>(gemm_tc_part_floats(M, N, K, sms), 4);
  const size_t nt = (size_t)((M + 127) / 128) * (N / 128);
  if (cudaMalloc(&hi, n * 2) != cudaSuccess || cudaMalloc(&lo, n * 2) != cudaSuccess ||
      cudaMalloc(&err, 4) != cudaSuccess || cudaMalloc(&tickets, nt * 4) != cudaSuccess ||
      cudaMalloc(&part, pf * 4) != cudaSuccess) {
    (void)cudaGetLastError();
    cudaFree(hi);
    cudaFree(lo);
    cudaFree(err);
    cudaFree(tickets);
    cudaFree(part);
    return TF_E_NOMEM;
  }
  tf_status r = TF_OK;
  GemvParams p = {};
  p.W = reinterpret_cast<const uint8_t*>(W);
  p.N = N;
  p.K = K;
  p.epi = EPI_STORE;
  p.out = C;
  p.ldo = N;
  p.err = err;
  if (cudaMemsetAsync(err, 0, 4, s) != cudaSuccess || cudaMemsetAsync(tickets, 0, nt * 4, s) != cudaSuccess ||
      launch_split_bf16(A, hi, lo, n, s) != cudaSuccess ||
      launch_gemm_tc(p, 0, hi, lo, M, part, tickets, sms, s) != cudaSuccess)
    r = TF_E_CUDA;
  uint32_t e = 0;
  if (r == TF_OK && (cudaMemcpyAsync(&e, err, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
                     cudaStreamSynchronize(s) != cudaSuccess))
    r = TF_E_CUDA;
  cudaFree(hi);
  cudaFree(lo);
  cudaFree(err);
  cudaFree(tickets);
  cudaFree(part);
  if (r == TF_OK && (e & ERR_TIMEOUT)) r = TF_E_TIMEOUT;
  return r;
}

namespace {
tf_status skinny_op(const float* A, const void* W, int wt, const float* row_scale, int32_t M, int32_t N,
                    int32_t K, float* C, void* stream) {
  if (!A || !W || !C || M < 1 || M > 64 || N < 2 || (N & 1) || K < 8 || (K % 8) ||
      (wt >= 1 && !row_scale) || (wt == 1 && K % 16) || (wt == 2 && K % 256))
    return TF_E_INVAL;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return TF_E_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint16_t *hi = nullptr, *lo = nullptr;
  uint32_t *err = nullptr, *tickets = nullptr;
  float* part = nullptr;
  const size_t n = (size_t)M * K;
  const size_t pf = std::max<size_t>(skinny_part_floats(N, K, M, sms), 4);
  const size_t nt = (size_t)(N + 127) / 128;
  if (cudaMalloc(&hi, n * 2) != cudaSuccess || cudaMalloc(&lo, n * 2) != cudaSuccess ||
      cudaMalloc(&err, 4) != cudaSuccess || cudaMalloc(&tickets, nt * 4) != cudaSuccess ||
      cudaMalloc(&part, pf * 4) != cudaSuccess) {
    (void)cudaGetLastError();
    cudaFree(hi);
    cudaFree(lo);
    cudaFree(err);
    cudaFree(tickets);
    cudaFree(part);
    return TF_E_NOMEM;
  }
  tf_status r = TF_OK;
  GemvParams p = {};
  p.W = reinterpret_cast<const uint8_t*>(W);
  p.scale = row_scale;
  p.N = N;
  p.K = K;
  p.epi = EPI_STORE;
  p.out = C;
  p.ldo = N;
  p.err = err;
  if (cudaMemsetAsync(err, 0, 4, s) != cudaSuccess || cudaMemsetAsync(tickets, 0, nt * 4, s) != cudaSuccess ||
      launch_split_bf16(A, hi, lo, n, s) != cudaSuccess ||
      launch_gemm_skinny(p, wt, hi, lo, M, part, tickets, sms, false, s) != cudaSuccess)
    r = TF_E_CUDA;
  uint32_t e = 0;
  if (r == TF_OK && (cudaMemcpyAsync(&e, err, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
                     cudaStreamSynchronize(s) != cudaSuccess))
    r = TF_E_CUDA;
  cudaFree(hi);
  cudaFree(lo);
  cudaFree(err);
  cudaFree(tickets);
  cudaFree(part);
  if (r == TF_OK && (e & ERR_TIMEOUT)) r = TF_E_TIMEOUT;
  return r;
}
}  // namespace

tf_status tf_op_gemm_skinny(const float* A, const uint16_t* W, int32_t M, int32_t N, int32_t K,
                            float* C, void* stream) {
  return skinny_op(A, W, 0, nullptr, M, N, K, C, stream);
}

tf_status tf_op_gemm_skinny_fp8(const float* A, const uint8_t* W, const float* row_scale, int32_t M,
                                int32_t N, int32_t K, float* C, void* stream) {
  return skinny_op(A, W, 1, row_scale, M, N, K, C, stream);
}

tf_status tf_op_gemm_skinny_nvfp4(const float* A, const uint8_t* W, const float* row_scale, int32_t M,
                                  int32_t N, int32_t K, float* C, void* stream) {
  return skinny_op(A, W, 2, row_scale, M, N, K, C, stream);
}

tf_status tf_op_gemv(const void* W, int32_t dtype, const float* row_scale, int64_t rows,
                     int64_t cols, const float* x, float* y, int32_t repeat, float* ms,
                     void* stream) {
  if (!W || !x || !y || rows < 1 || cols < 16 || rows > (1 << 30) || repeat < 1) return TF_E_INVAL;
  if (dtype != TF_DTYPE_BF16 && dtype != TF_DTYPE_FP8_E4M3 && dtype != TF_DTYPE_NVFP4) return TF_E_INVAL;
  if (dtype != TF_DTYPE_BF16 && !row_scale) return TF_E_INVAL;
  const int wt = dtype;  // TF_DTYPE_* matches the GEMV's format numbers
  const int eb = dtype == TF_DTYPE_BF16 ? 2 : 1;
  if ((cols * eb) % 16 || cols * eb / 16 > 5 * 256) return TF_E_INVAL;
  if (dtype == TF_DTYPE_NVFP4 && cols % 256) return TF_E_INVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (gemv_set_attributes() != cudaSuccess) return TF_E_CUDA;
  uint32_t* err = nullptr;
  if (cudaMalloc(&err, sizeof(uint32_t)) != cudaSuccess) return TF_E_NOMEM;
  cudaMemsetAsync(err, 0, 4, s);
  GemvParams p = {};
  p.N = static_cast<int32_t>(rows);
  p.K = static_cast<int32_t>(cols);
  p.pro = PRO_PLAIN;
  p.x = x;
  p.ldx = p.K;
  p.epi = EPI_STORE;
  p.out = y;
  p.ldo = 0;
  p.err = err;
  gemv_plan(p, wt, sms, 1);
  const int grid = gemv_grid(p, sms);
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  tf_status r = TF_OK;
  if (ms) {
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    cudaEventRecord(e0, s);
  }
  for (int i = 0; i < repeat && r == TF_OK; ++i) {
    p.W = static_cast<const uint8_t*>(W) + (size_t)i * rows * lin_row_bytes(wt, cols);
    p.scale = row_scale ? row_scale + (size_t)i * rows : nullptr;
    if (launch_gemv(p, wt, 1, grid, i > 0, s) != cudaSuccess) r = TF_E_CUDA;
  }
  if (ms) cudaEventRecord(e1, s);
  uint32_t e = 0;
  if (cudaMemcpyAsync(&e, err, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    r = TF_E_CUDA;
  if (ms && r == TF_OK) {
    float t = 0.f;
    cudaEventElapsedTime(&t, e0, e1);
    *ms = t / repeat;
  }
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  cudaFree(err);
  if (r == TF_OK && (e & ERR_TIMEOUT)) r = TF_E_TIMEOUT;
  return r;
}

}  // extern "C"
