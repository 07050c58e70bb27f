// Internal launch interface of the decode kernels (host side).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace tf {

// Error bits raised by kernels (the host maps them to tf_status).
enum : uint32_t {
  ERR_TIMEOUT = 1u << 0,   // a bounded wait expired
  ERR_NAN = 1u << 1,       // NaN logit met by a selection
  ERR_BAD_ID = 1u << 2,    // an id fed back was outside its table
  ERR_BAD_POS = 1u << 3,   // a position outside the KV cache
  ERR_BAD_CODE = 1u << 4,  // an e4m3 NaN code in a weight handed over as codes
};

// ----------------------------------------------------------------- GEMV
// Prologue: how the activation vector a[m][k] is formed.
enum Prologue : int32_t {
  PRO_PLAIN = 0,   // a = x
  PRO_NORM = 1,    // a = RMSNorm(x) * w   (w bf16 [K])
};
// Epilogue: what happens to y[m][r] = sum_k W[r][k] a[m][k].
enum Epilogue : int32_t {
  EPI_STORE = 0,   // out[m][r] = y
  EPI_RESID = 1,   // out[m][r] += y (in-place residual add)
  EPI_SWIGLU = 2,  // rows (2i, 2i+1) = (gate_i, up_i): out[m][i] = silu(g) * u
  EPI_QKV = 3,     // rows in RoPE-pair order: rotate q, k; q -> qout, k, v -> KV cache
  EPI_LOGITS = 4,  // out[r] = y (M = 1) and, if select, grid-wide argmax -> ids
};

struct GemvParams {
  const uint8_t* W;      // [N][K] row-major, bf16 or e4m3 bytes
  const float* scale;    // [N] per-row scale (fp8) or nullptr
  int32_t N, K;
  int32_t unit;          // rows per partition unit (2 for pair epilogues)
  int32_t units;         // N / unit
  int32_t rs;            // rows per pipeline stage
  int32_t nst;           // stages in the shared-memory ring
  int32_t stb;           // bytes per stage slot (multiple of 128)
  int32_t ctas_per_sm;   // 1 or 2 (set by gemv_plan)
  int32_t nt, J;         // consumer threads and 16-byte chunks per thread (gemv_plan)
  // prologue
  int32_t pro;
  const float* x;        // [M][ldx]
  int32_t ldx;
  const uint16_t* nw;    // RMSNorm weight (bf16 bits) [K]
  float eps;
  // epilogue
  int32_t epi;
  float* out;            // [M][ldo]
  int32_t ldo;
  uint16_t* out_hi;      // EPI_SWIGLU: if set, the result goes out as bf16
  uint16_t* out_lo;      // hi / lo parts [M][ldo] instead of fp32 to out
  // EPI_QKV
  int32_t q_dim, kv_dim, head_dim;
  float* qout;           // [M][q_dim]
  uint16_t* Kc;          // [Hkv][T][head_dim] bf16
  uint16_t* Vc;
  int32_t T;
  const int32_t* pos_ptr;  // row m sits at position pos_ptr[0] + m, or
  int32_t pos_fixed;       // pos_fixed + m when pos_ptr is null
  int32_t rps;           // rows per sequence: > 0 -> row m is row m % rps of
                         // sequence seq_base + m / rps (position pos_ptr[seq] +
                         // m % rps); 0 -> every row belongs to sequence seq_base
  int32_t seq_base;
  int64_t kv_seq;        // elements between two sequences' caches (dense caches)
  const int32_t* kv_tbl; // paged caches: page of (sequence, position / kKvPage) at
  int32_t kv_npp;        // kv_tbl[seq * kv_npp + position / kKvPage]; null: dense
  int32_t pos_uniform;   // every sequence sits at the same position (lockstep)
  const float2* rope;    // [T][head_dim/2] (cos, sin)
  // EPI_LOGITS
  int32_t select;        // 1: argmax -> sel[cb], fb[cb]
  unsigned long long* best;
  uint32_t* ticket;
  int32_t* sel;          // selected id slot
  int32_t* fb;           // fed-back id slot
  const int32_t* forced;     // forced id slot (if *forced_on)
  const int32_t* forced_on;
  uint32_t* err;
  // Deferred RMSNorm of the skinny tensor-core GEMM (batched decode).
  // RMSNorm(x) * w = rstd * (x * w) with rstd = 1 / sqrt(mean(x^2) + eps), a
  // per-row scalar, so W (RMSNorm(x) * w) = rstd * W (x * w): the GEMM that
  // produces x emits x * w as bf16 parts plus partial sums of x^2, and the
  // GEMM that consumes it scales its rows by rstd in the epilogue.
  const uint16_t* nw_next;   // producer (EPI_RESID): norm weight of the consumer
  uint16_t* nx_hi;           //   x * nw_next as bf16 hi / lo parts [M][ldo]
  uint16_t* nx_lo;
  float* ssq_out;            //   sum of x^2 over this tile's columns: [tile][kSsqRows]
  const float* ssq_in;       // consumer: partial sums [ssq_n][kSsqRows] of its rows
  int32_t ssq_n;
  int32_t in_rps;            // consumer row m is producer row m * in_rps + in_rps - 1
                             // (activation parts and sums); 0 or 1: the same row
  // Cross-kernel L2 prefetch (batch-1 GEMV): once CTA c has issued its last
  // weight copy, it asks L2 for the first pf_bytes of the row block that CTA
  // c of the next GEMV in the stream will stream (that GEMV's partition:
  // pf_units units of pf_unit rows of pf_rowbytes, over pf_grid CTAs), so
  // HBM keeps streaming across the kernel boundary.
  const uint8_t* pf_w;
  int32_t pf_units, pf_unit, pf_rowbytes, pf_grid, pf_bytes;
  // QKV GEMV of one sequence (dense caches): after its last weight copy each
  // CTA also asks L2 for its share of the layer's cached K and V rows
  // 0..pos-1, which the attention kernel that follows reads.
  int32_t kv_pf;
  // q/k RMSNorm option: the QKV epilogue stores the q and k pairs as they
  // are (RoPE-pair order, [M][q_dim + kv_dim]) for k_qknorm to finish
  float* qk_raw;
  const uint16_t* q_norm;  // k_qknorm: per-head RMSNorm weights [head_dim]
  const uint16_t* k_norm;
  // Failure test: CTA 0's producer arms its last stage's barrier without
  // issuing the copy, so that stage's bounded wait expires (ERR_TIMEOUT).
  int32_t test_skip_copy;
};
// Finishes q and k after a QKV GEMM that left them raw (GemvParams::qk_raw):
// each head of each row is RMSNorm-ed with q_norm / k_norm, rotated by RoPE
// at the row's position, q stored to qout and k appended to the KV cache.
cudaError_t launch_qknorm(const GemvParams& p, int M, bool pdl, cudaStream_t s);
constexpr int kSsqRows = 64;   // row stride of the partial sums of squares
// Paged KV caches: a page holds kKvPage positions of every KV head of one
// layer, laid out [page][Hkv][kKvPage][D]; page 0 is a scratch page.
constexpr int kKvPage = 32;

// Shared memory bytes a launch with these params needs.
size_t gemv_smem_bytes(const GemvParams& p, int M);
// Fills unit/units/rs/nst/stb/ctas_per_sm for a matrix of N x K elements
// stored as weight format wt (0 bf16, 1 e4m3 codes, 2 block-scaled 4-bit) and
// M activation rows.
void gemv_plan(GemvParams& p, int wt, int num_sms, int M);
// CTAs to launch for a planned GEMV.
int gemv_grid(const GemvParams& p, int num_sms);
// Launch (weight format wt: 0 bf16, 1 fp8, 2 block-scaled 4-bit) on `grid` CTAs; pdl = allow
// programmatic dependent launch on the previous kernel of the stream.
cudaError_t launch_gemv(const GemvParams& p, int wt, int M, int grid, bool pdl,
                        cudaStream_t s);
cudaError_t gemv_set_attributes();

// ----------------------------------------------------------------- attention
struct AttnParams {
  const float* q;        // [M][Hq*D] rotated queries
  const uint16_t* Kc;    // [Hkv][T][D] per sequence, or the page pool
  const uint16_t* Vc;
  int32_t T, Hq, Hkv, D;
  const int32_t* pos_ptr;  // per-sequence positions, or null: pos_fixed
  int32_t pos_fixed;
  int32_t rps;           // rows per sequence (as GemvParams::rps)
  int32_t seq_base;
  int64_t kv_seq;        // elements between two sequences' caches (dense)
  const int32_t* kv_tbl; // paged caches (as GemvParams::kv_tbl)
  int32_t kv_npp;
  int32_t S;             // splits over the key range (grid.x)
  float* part;           // [M][Hq][S][D + 2] partial (m, l, acc)
  uint32_t* counters;    // [M][Hkv], zero between launches
  float* out;            // [M][Hq*D]
  uint16_t* out_hi;      // if set: the output as bf16 hi / lo parts [M][Hq*D]
  uint16_t* out_lo;      // instead of fp32 to out
  uint32_t* err;
};
cudaError_t launch_attention(const AttnParams& p, int M, bool pdl, cudaStream_t s);
// The same attention for prompt rows (many rows, one long key slice each).
cudaError_t launch_attention_rows(const AttnParams& p, int M, bool pdl, cudaStream_t s);
// Causal attention of prompt rows on the tensor cores, nseq sequences of P
// rows: row m of a sequence sits at position pos0 + m and attends to keys
// 0..pos0 + m of that sequence.  The queries come as bf16 hi / lo parts
// [nseq * P][Hq*D]; Kc / Vc are dense caches [slots][Hkv][T][D] (kv_rows =
// slots*Hkv*T, sequence z in slot seq + z), or with kv_tbl the page pool
// [pages][Hkv][kKvPage][D] (kv_rows = pages*Hkv*kKvPage).  D = 64 or 128.
struct PromptAttnArgs {
  int32_t P, pos0, Hq, Hkv, T;
  int32_t nseq;            // sequences, P query rows each ([nseq][P] rows of q and out)
  int32_t seq;             // the first sequence's slot; sequence z is slot seq + z
  const int32_t* kv_tbl;   // paged: block table [slots][npp]; null: dense
  int32_t kv_npp;
  float scale_log2;        // log2(e) / sqrt(D)
  float* out;              // [P][Hq*D] fp32, or
  uint16_t* out_hi;        // bf16 hi / lo parts
  uint16_t* out_lo;
  uint32_t* err;
};
bool prompt_attention_tc_supported(int D, int Hq, int Hkv);
cudaError_t launch_prompt_attention_tc(const uint16_t* q_hi, const uint16_t* q_lo, const uint16_t* Kc,
                                       const uint16_t* Vc, int64_t kv_rows, int D,
                                       const PromptAttnArgs& a, cudaStream_t s);

// ----------------------------------------------------------------- misc
// Builds the input rows of a decoder pass.  Sequence b's ids sit at
// ids[b * id_stride] (the slot of the codebook the pass feeds from).
enum BuildMode : int32_t {
  BUILD_SLOW = 0,    // x[b] = text_embed[sem_base + fb_b[0]]
  BUILD_FAST1 = 1,   // x[2b] = RMSNorm(xs[b]) * w_final; x[2b+1] = cb_embed[0][fb_b[0]]
  BUILD_FASTJ = 2,   // x[b] = cb_embed[j-1][fb_b[j-1]]
  BUILD_TOKENS = 3,  // x[m] = text_embed[tokens[m]]  (prefill)
};
struct BuildParams {
  int32_t mode, j, H, M;
  // BUILD_SLOW: a sequence with pending[b] >= 0 still has that prompt id to
  // feed (it joined with its prompt pass done but for its last id): its row
  // is text_embed[pending[b]] (table + 0, text_rows ids) instead
  const int32_t* pending;
  int32_t text_rows;
  const uint16_t* table;   // embedding table base (text_embed or cb_embed[j-1])
  int32_t table_rows;      // rows the id may address
  int32_t row_base;        // added to the id (sem_base for BUILD_SLOW)
  const int32_t* ids;      // id source (fb slot, or tokens for BUILD_TOKENS)
  int32_t id_stride;       // ids between two sequences' slots
  const float* xs;         // slow residuals [B][H] (BUILD_FAST1)
  const uint16_t* nw;      // final slow norm (BUILD_FAST1)
  float eps;
  float* x;                // output rows [M][H]
  uint32_t* err;
  // BUILD_SLOW option: add the previous frame's codes 1..9 (id slots
  // ids[b * id_stride + j]) as rows of cb_sum [ncb - 1][cb_rows][H]
  const uint16_t* cb_sum;
  int32_t cb_rows;
  int32_t ncb;
  // optional, for the skinny GEMM that reads the rows next (see GemvParams):
  const uint16_t* nw_next; // x * nw_next as bf16 parts [M][H], sum of x^2 per row
  uint16_t* nx_hi;
  uint16_t* nx_lo;
  float* ssq_out;          // [kSsqRows]
};
cudaError_t launch_build(const BuildParams& p, bool pdl, cudaStream_t s);

// Per-frame bookkeeping after the last codebook: pos += advance,
// frame_index += 1, history[hist_idx++] = sel of every sequence.
struct FrameEndParams {
  int32_t* pos;          // per sequence
  int32_t advance;
  int32_t* frame_index;  // per sequence
  const int32_t* active; // null: every sequence; else only those with active[b]
  int32_t* pending;      // null, or cleared to -1 for the sequences that advance
  const int32_t* sel;    // sequence b's ids at sel[b * sel_stride]
  int32_t sel_stride;
  int32_t nseq;          // history row = [nseq][ncb]
  int32_t ncb;
  int32_t* hist;         // [hist_cap][ncb]
  int32_t* hist_idx;
  int32_t hist_cap;
  const int32_t* fb;     // ids fed back this frame, sequence b's at fb[b * sel_stride]
  int32_t* fb_ring;      // [nseq][kRepRing][kRepIds]: slot frame_index % kRepRing
};
// Frames of fed-back ids kept per sequence for the repetition window, and
// id slots per frame in that ring.
constexpr int kRepRing = 64;
constexpr int kRepIds = 16;
cudaError_t launch_frame_end(const FrameEndParams& p, bool pdl, cudaStream_t s);

// Top-k / argmax selection of one row of logits per CTA.
struct SelectParams {
  const float* logits;   // [n][ld]
  int32_t ld, vocab, n;
  int32_t top_k;
  float temperature;
  uint32_t key0, key1;   // Philox key (seed low / high)
  const int32_t* frame_ptr;  // per-sequence frame indices on the device (or null -> frame)
  int32_t frame;
  int32_t codebook0;     // row i uses codebook0 + i (seq_rows = 0)
  int32_t sequence;
  int32_t seq_rows;      // 1: row i is sequence `sequence + i` at codebook0,
                         // its slots sel/fb/forced[i * id_stride]
  int32_t id_stride;
  int32_t* sel;          // [n]
  int32_t* fb;           // [n] fed-back ids or null
  const int32_t* forced;
  const int32_t* forced_on;
  uint32_t* err;
  // nucleus and repetition window (see tf_sampling)
  float top_p;             // >= 1: no nucleus cut
  float rep_penalty;
  int32_t rep_window;      // frames of the ring the window covers (0: off)
  const int32_t* fb_ring;  // [sequences][kRepRing][kRepIds] fed-back ids
  const int32_t* recent;   // or explicit window ids [n][n_recent] (< 0: empty)
  int32_t n_recent;
};
cudaError_t launch_select(const SelectParams& p, bool pdl, cudaStream_t s);

// Weight re-layout and quantisation at load time.
enum RowMap : int32_t {
  MAP_IDENTITY = 0,
  MAP_QKV = 1,       // dst row order: RoPE pairs of q heads, k heads; v as is
  MAP_GATE = 2,      // src row i -> dst row 2i
  MAP_UP = 3,        // src row i -> dst row 2i + 1
};
struct PackParams {
  const uint8_t* src;    // [rows][cols] bf16 or e4m3
  const float* src_scale;  // e4m3 input: [rows]
  uint8_t* dst;          // packed destination (bf16 or e4m3)
  float* dst_scale;      // fp8 destination: [dst rows]
  int64_t rows, cols;
  int32_t map;
  int32_t q_dim, kv_dim, head_dim;
  int32_t mode;          // 0 copy bf16, 1 quantise bf16 -> fp8, 2 copy fp8 + scale,
                         // 4 quantise bf16 -> block-scaled 4-bit rows
  uint32_t* err;         // mode 2: ERR_BAD_CODE if a code is NaN (0x7F / 0xFF)
};
cudaError_t launch_pack(const PackParams& p, cudaStream_t s);

// ----------------------------------------------------------------- prefill
// Row-block GEMM on CUDA cores for prompts: out = epi(A[M][K] * W[N][K]^T)
// with the GEMV's prologue/epilogue semantics (positions: row m at pos m).
cudaError_t launch_gemm_rows(const GemvParams& p, int wt, int M, cudaStream_t s);
// Tensor-core (tcgen05) GEMM for prompts, bf16 weights:
// out = epi(A[M][K] * W[N][K]^T) with A given as bf16 hi/lo parts [M][K].
// K is split when the tiles alone would not fill the SMs (gemm_tc_splits);
// then part holds gemm_tc_part_floats() floats and tickets one zeroed word per
// output tile (returned to zero by the launch).
bool gemm_tc_supported(int N, int K);
size_t gemm_tc_smem_bytes();
// wt = 0: bf16 weights; 1: e4m3 codes (row scale in p.scale); 2: 4-bit rows
// as k_pack writes them (K a multiple of 256): quantised weights stream as
// they are and are converted to bf16 in shared memory (128-wide tiles).
int gemm_tc_splits(int M, int N, int K, int num_sms, int wt = 0);
size_t gemm_tc_part_floats(int M, int N, int K, int num_sms);
cudaError_t launch_gemm_tc(const GemvParams& p, int wt, const uint16_t* a_hi, const uint16_t* a_lo, int M,
                           float* part, uint32_t* tickets, int num_sms, cudaStream_t s);
// Skinny tensor-core GEMM for batched decode (M <= 64 activation rows):
// out = epi(A[M][K] * W[N][K]^T), the weight rows on the MMA's 128-row side,
// the activation rows (bf16 hi / lo parts, [M][K]) on its N side, split over K
// so that the grid covers the GPU; the last CTA of a weight tile sums the
// splits' partials in split order (part: skinny_part_floats(), tickets: one
// per weight tile, zero between launches).  wt = 0: bf16 weights; wt = 1:
// e4m3 codes (K a multiple of 16) converted to bf16 in shared memory, the
// fp32 row scale (p.scale) applied in the epilogue.
int skinny_splits(int N, int K, int num_sms);
size_t skinny_part_floats(int N, int K, int M, int num_sms);
cudaError_t launch_gemm_skinny(const GemvParams& p, int wt, const uint16_t* a_hi, const uint16_t* a_lo,
                               int M, float* part, uint32_t* tickets, int num_sms, bool pdl,
                               cudaStream_t s);
// Rows for a skinny GEMM with a deferred RMSNorm: a = x[m] * w as bf16 hi / lo
// parts [M][K] and ssq[m] = sum_k x[m][k]^2, for M rows x[m * ldx].
cudaError_t launch_rows_prep(const float* x, int ldx, int M, int K, const uint16_t* w,
                             uint16_t* hi, uint16_t* lo, float* ssq, bool pdl, cudaStream_t s);
// e4m3 codes -> bf16 bits of the same values (n even).
cudaError_t launch_e4m3_to_bf16(const uint8_t* q, uint16_t* out, size_t n, cudaStream_t s);
// Block-scaled 4-bit rows [N][K/2 + K/16] -> bf16 bits of e2m1 x block scale
// [N][K] (exact; the row scale is applied later, in the GEMM epilogue).
cudaError_t launch_nvfp4_to_bf16(const uint8_t* q, uint16_t* out, int N, int K, cudaStream_t s);
// hi = bf16(a), lo = bf16(a - hi) elementwise.
cudaError_t launch_split_bf16(const float* a, uint16_t* hi, uint16_t* lo, size_t n, cudaStream_t s);
// a[m] = RMSNorm(x[m]) * w for M rows (prefill prologue).
cudaError_t launch_rmsnorm_rows(const float* x, const uint16_t* w, float* a, int M, int H,
                                float eps, cudaStream_t s);
// The same rows as bf16 hi / lo parts (the tensor-core prompt GEMM's input).
cudaError_t launch_rmsnorm_split(const float* x, const uint16_t* w, uint16_t* hi, uint16_t* lo,
                                 int M, int H, float eps, cudaStream_t s);

}  // namespace tf
