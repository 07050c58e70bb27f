/*
 * tf.h - C ABI of the GB300 (sm_103a) Dual-AR decode library.
 *
 * The library runs the decode step of a Dual-AR (RQ-Transformer) text-to-
 * speech model shaped like Fish-Speech S2-Pro: per frame, one token through a
 * "slow" decoder along time (GQA attention with RoPE over a static KV cache,
 * SwiGLU MLP, RMSNorm) whose tied semantic head picks codebook 0, then a loop
 * of 9 steps through a "fast" decoder along depth that picks the residual
 * codebooks 1..9.  One decode call emits one frame of 10 codebook ids.
 *   - Dual-AR structure, 10 codebooks: fish-s2-pro-mlx-local-deploy README,
 *     architecture paragraph ("Slow AR ... time axis ... primary semantic
 *     codebook; Fast AR ... remaining 9 residual codebooks").
 *   - Shapes, static KV cache, bytes per decode step: tuna-fish README,
 *     "Inference estimation".
 *   - Per-row FP8 weights: drbaph s2-pro-fp8 model card, "Quantization Details".
 *
 * Conventions for every call:
 *   - The caller owns every pointer it passes; host buffers may be freed as
 *     soon as the call returns.  The library owns all device memory it
 *     allocates (tf_create) and frees it in tf_destroy.
 *   - Calls are synchronous with respect to the host: outputs are valid on
 *     return.  Work runs on the context's stream (tf_set_stream).
 *   - A context is used by one host thread at a time.
 *   - Errors: every call returns a tf_status; tf_last_error() gives a one-line
 *     message.  After TF_E_CUDA or TF_E_TIMEOUT the context is poisoned and
 *     every later call except tf_destroy returns TF_E_STATE.
 *   - Device kernels never trap: a kernel that detects a bad id, a NaN logit or
 *     an expired wait sets a flag that the call turns into TF_E_NUMERIC,
 *     TF_E_INVAL or TF_E_TIMEOUT.
 */
#ifndef TF_H
#define TF_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct tf_ctx tf_ctx;

typedef enum {
  TF_OK = 0,
  TF_E_INVAL = 1,     /* bad argument, shape, name or id; nothing changed       */
  TF_E_NOMEM = 2,     /* device allocation failed                               */
  TF_E_CUDA = 3,      /* CUDA runtime error; context poisoned                   */
  TF_E_STATE = 4,     /* call out of order (no weights, no prefill) or poisoned */
  TF_E_CAPACITY = 5,  /* KV cache full (position == max_seq_len); state kept    */
  TF_E_TIMEOUT = 6,   /* a bounded device wait expired; context poisoned        */
  TF_E_NUMERIC = 7    /* NaN logit met during selection                          */
} tf_status;

/* Weight formats of the linear layers (tf_config.weight_dtype).
 * TF_WEIGHT_NVFP4: block-scaled 4-bit weights (the tuna-fish README lists
 * nvfp4 among its formats): FP4 E2M1 codes, an e4m3 scale per 16 elements
 * of a row and a float32 scale per row; the library quantises bf16 linears
 * as tf_op_quantize_nvfp4 does.  Needs hidden, ffn and n_heads*head_dim
 * multiples of 256. */
enum { TF_WEIGHT_BF16 = 0, TF_WEIGHT_FP8 = 1, TF_WEIGHT_NVFP4 = 2 };
/* Element types of tensors handed to tf_load_weights (tf_tensor.dtype), and
 * of the weight given to tf_op_gemv (TF_DTYPE_NVFP4: rows as
 * tf_op_quantize_nvfp4 writes them). */
enum { TF_DTYPE_BF16 = 0, TF_DTYPE_FP8_E4M3 = 1, TF_DTYPE_NVFP4 = 2 };

/* Model shape.  All sizes are element counts.
 * head_dim must be 64 or 128; n_heads a multiple of n_kv_heads with
 * n_heads / n_kv_heads <= 8; hidden, ffn and n_heads*head_dim multiples of 16;
 * semantic_vocab <= text_vocab; n_codebooks = 10 (codebook 0 semantic). */
typedef struct {
  int32_t slow_layers, fast_layers;
  int32_t hidden, n_heads, n_kv_heads, head_dim, ffn;
  int32_t text_vocab;       /* rows of the tied text embedding                  */
  int32_t semantic_vocab;   /* slow head = text-embedding rows [text_vocab - semantic_vocab, text_vocab) */
  int32_t n_codebooks;      /* ids per frame (10)                               */
  int32_t codebook_size;    /* rows of the fast head and of each codebook table */
  int32_t max_seq_len;      /* static slow KV length T                          */
  int32_t max_batch;        /* sequences per context, 1..32 (lockstep batch)    */
  float rms_eps, rope_theta;
  int32_t weight_dtype;     /* TF_WEIGHT_BF16 or TF_WEIGHT_FP8                  */
  int32_t flags;            /* TF_FLAG_* model options, 0 = none                */
} tf_config;

/* Model options (tf_config.flags) for checkpoints that have them:
 * TF_FLAG_QK_NORM: every slow layer normalises each head of q and of k with
 *   an RMSNorm over head_dim ("slow.{i}.q_norm", "slow.{i}.k_norm",
 *   [head_dim] bf16) before RoPE.  The tuna-fish README's slowAR parameter
 *   count ("Inference estimation") holds these 2 x head_dim per layer.
 * TF_FLAG_QK_NORM_FAST: the same in the fast layers ("fast.{i}.q_norm", ...).
 * TF_FLAG_SLOW_CB_SUM: the slow input of a decoded frame adds the embeddings
 *   of the previous frame's codes 1..9 ("slow.cb_embed"
 *   [n_codebooks-1][codebook_size][hidden] bf16, table j-1 for code j) to the
 *   text-embedding row of its code 0. */
enum { TF_FLAG_QK_NORM = 1, TF_FLAG_QK_NORM_FAST = 2, TF_FLAG_SLOW_CB_SUM = 4, TF_FLAG_PAGED_KV = 8 };
/* TF_FLAG_PAGED_KV: the slow KV caches are pools of pages of 32 positions
 * shared by the sequence slots, found through a block table; a slot holds
 * pages only for the positions it has reached (the fish-s2-pro-mlx-local-
 * deploy README's architecture paragraph and the drbaph s2-pro-fp8 card's
 * "Architecture" name continuous batching with a paged KV cache for
 * serving).  Results equal the dense caches'. */

/* One named host (or device) tensor for tf_load_weights.
 * Names: "text_embed" [text_vocab][hidden];
 *        "slow.{i}.attn_norm" / "slow.{i}.ffn_norm" [hidden];
 *        "slow.{i}.wqkv" [n_heads*head_dim + 2*n_kv_heads*head_dim][hidden]
 *            (rows: q heads, then k heads, then v heads);
 *        "slow.{i}.wo" [hidden][n_heads*head_dim];
 *        "slow.{i}.w1" (gate), "slow.{i}.w3" (up) [ffn][hidden];
 *        "slow.{i}.w2" (down) [hidden][ffn];
 *        "slow.norm" [hidden];  the same for "fast.{i}.*" and "fast.norm";
 *        "fast.head" [codebook_size][hidden];
 *        "fast.cb_embed" [n_codebooks-1][max(semantic_vocab, codebook_size)][hidden]
 *            (table j-1 embeds the id fed at fast step j: code 0 at step 1,
 *            code j-1 after);
 *        with the TF_FLAG_* options also "slow.{i}.q_norm", "slow.{i}.k_norm",
 *        "fast.{i}.q_norm", "fast.{i}.k_norm" [head_dim] and "slow.cb_embed".
 * Linear weights are [out][in] row-major.  Embeddings and norms are bf16.
 * In an FP8 context a linear weight is given either as bf16 (the library
 * quantises it per row, exactly as tf_op_quantize_fp8) or as
 * TF_DTYPE_FP8_E4M3 codes with row_scale[out] (float32); codes must be
 * finite (NaN codes 0x7F / 0xFF are refused with TF_E_INVAL). */
typedef struct {
  const char* name;
  int32_t dtype;
  int32_t ndim;
  int64_t shape[3];
  const void* data;         /* host or device pointer                          */
  const float* row_scale;   /* FP8 codes only: [shape[0]] float32, else NULL   */
} tf_tensor;

/* Codebook-id selection ("Fish Speech" tour, "Why You Need This": the
 * generation loop samples with top-k and top-p and keeps repetition
 * windows).  top_k = 0 (or 1): greedy argmax (lowest index on ties).
 * top_k > 1: keep the top_k logits ordered by (logit desc, index asc),
 * weights exp((z - z_max) / temperature) summed in that order in float32,
 * u = (w0 >> 8) * 2^-24 from Philox4x32-10 with counter
 * (frame index, codebook, sequence, 0) and key (seed low, seed high 32 bits);
 * the pick is the first candidate whose running sum exceeds u * sum.
 * top_p in (0, 1) (top_k > 1 only): the draw is restricted to the shortest
 *   prefix of the ordered candidates whose running sum reaches
 *   top_p * sum (float32), with that prefix's sum in place of sum;
 *   top_p = 1 keeps every candidate.
 * rep_window W in [0, 64], rep_penalty r > 0: before selection, the logit of
 *   every id that codebook fed back in the previous W frames of the same
 *   sequence (each id once) becomes z / r if z > 0, else z * r (float32);
 *   W = 0 or r = 1 turns it off.  Returned logits are the model's, before
 *   the penalty. */
typedef struct {
  int32_t top_k;
  float temperature;
  uint64_t seed;
  float top_p;
  float rep_penalty;
  int32_t rep_window;
} tf_sampling;

/* Read-only facts about a context. */
typedef struct {
  int32_t position;         /* next slow position of sequence 0                */
  int32_t frame_index;      /* frames emitted since the last prefill           */
  int32_t num_sms;          /* SMs of the device                                */
  int32_t graph_nodes;      /* kernel launches in one captured decode frame     */
  int64_t weight_bytes;     /* device bytes of all weights as stored            */
  int64_t frame_weight_bytes; /* weight bytes one decode frame streams          */
  int64_t device_bytes;     /* all device memory the context owns               */
} tf_info;

/* Creates a context on CUDA device `device`: validates cfg, allocates weights,
 * KV caches and work buffers (all device memory is allocated here), creates
 * the context's stream.  On failure *out is NULL.  Errors: TF_E_INVAL (bad
 * shape), TF_E_NOMEM, TF_E_CUDA. */
tf_status tf_create(const tf_config* cfg, int device, tf_ctx** out);

/* Copies n named tensors into the context (host->device or device->device),
 * re-laying them out for the kernels and quantising bf16 linears in an FP8
 * context.  May be called several times; a decode needs every tensor loaded.
 * Errors: TF_E_INVAL (unknown name, wrong shape or dtype), TF_E_CUDA. */
tf_status tf_load_weights(tf_ctx* ctx, const tf_tensor* t, int32_t n);

/* Prompt in, frame 0 out.  tokens: host int32 [B][P], ids in [0, text_vocab),
 * 1 <= B <= max_batch: B independent sequences with prompts of one length P.
 * Resets every sequence to position 0, runs the slow decoder over each
 * prompt (positions 0..P-1, the sequence's own KV cache; max_seq_len / P
 * prompts share one pass of the tensor-core GEMMs), then selects frame 0 of
 * every sequence from its last row.  The B sequences then decode in
 * lockstep: each later decode call advances all B by one frame (B > 1 runs
 * every linear layer as one skinny tensor-core GEMM over the B rows, see
 * tf_op_gemm_skinny).  Sampling draws use the sequence index b as the
 * Philox counter's third word.
 * forced: NULL, or host int32 [B][n_codebooks] ids that replace the selected
 *   ids wherever they are fed back (teacher forcing); frame0 still reports the
 *   library's own selections.
 * frame0: host int32 [B][n_codebooks].  logits: NULL or host float
 *   [B][n_codebooks][max(semantic_vocab, codebook_size)] (row 0 semantic).
 * Errors: TF_E_INVAL (B, P or an id out of range), TF_E_STATE (weights
 * missing), TF_E_NUMERIC, TF_E_CUDA. */
tf_status tf_prefill(tf_ctx* ctx, const int32_t* tokens, int32_t B, int32_t P,
                     const tf_sampling* sampling, const int32_t* forced,
                     int32_t* frame0, float* logits);

/* Continuous batching: starts a sequence in slot `slot` (0 <= slot <
 * max_batch) while the other slots keep their state.  tokens: host int32
 * [P], ids in [0, text_vocab), 1 <= P <= max_seq_len.  Ids 0..P-2 run
 * through the prompt pass into the slot's KV caches; the last id is fed by
 * the next decode call, whose frame for this slot is the sequence's frame 0
 * (sampling counters restart: its frame index is 0).  A sequence already in
 * the slot is released first.  Prompt lengths may differ between slots: each
 * slot has its own position.  Errors: TF_E_INVAL, TF_E_STATE (weights
 * missing), TF_E_CAPACITY (no free KV page), TF_E_CUDA. */
tf_status tf_prefill_seq(tf_ctx* ctx, int32_t slot, const int32_t* tokens, int32_t P);

/* Ends the sequence in slot `slot`: the slot goes idle (its frames read -1)
 * and, with paged caches, its pages return to the pool.  Errors: TF_E_INVAL. */
tf_status tf_release_seq(tf_ctx* ctx, int32_t slot);

/* One decode frame: feeds each active sequence's last codebook-0 id (or the
 * last id of a prompt started with tf_prefill_seq) at its own next position
 * and emits the next frame of every slot up to the last active one (B =
 * that count; idle slots read -1).  forced, frame and logits as tf_prefill.
 * When an active slot is at position == max_seq_len returns TF_E_CAPACITY
 * and changes nothing; TF_E_STATE when no sequence is active. */
tf_status tf_decode_frame(tf_ctx* ctx, const tf_sampling* sampling,
                          const int32_t* forced, int32_t* frame, float* logits);

/* n decode frames back to back on the device (no host round trip between
 * frames); frames: host int32 [n][B][n_codebooks] (B and idle slots as
 * tf_decode_frame).  Fails with TF_E_CAPACITY before running anything if
 * the n frames do not fit. */
tf_status tf_decode_frames(tf_ctx* ctx, const tf_sampling* sampling, int32_t n,
                           int32_t* frames);

/* Sets the CUDA stream (cudaStream_t) all later work of ctx runs on; NULL
 * restores the context's own stream.  The caller keeps the stream alive. */
tf_status tf_set_stream(tf_ctx* ctx, void* stream);
/* The stream work is currently enqueued on. */
void* tf_get_stream(const tf_ctx* ctx);

tf_status tf_get_info(const tf_ctx* ctx, tf_info* info);

/* One-line description of the last error of ctx (or of the last failed
 * tf_create when ctx is NULL).  Never NULL; valid until the next call. */
const char* tf_last_error(const tf_ctx* ctx);

/* Frees everything the context owns.  NULL-safe. */
void tf_destroy(tf_ctx* ctx);

/* Times one kernel of the decode frame in its in-frame configuration
 * (same parameters, prologue, epilogue and launch chaining) on the context's
 * stream with CUDA events: `iters` back-to-back launches cycling through the
 * slow decoder's layers (so every launch streams a distinct weight from HBM),
 * captured as one CUDA graph like the decode frame and replayed once to
 * warm up, then once timed.
 * which: 0 = gate/up GEMV (RMSNorm prologue, SwiGLU epilogue),
 *        1 = QKV GEMV, 2 = O GEMV, 3 = down GEMV;
 *        4..7 = the same four layers as the batched step's skinny
 *        tensor-core GEMMs over max_batch activation rows (needs
 *        max_batch > 1; the RMSNorm runs in a separate row kernel there).
 * Outputs the mean device time per launch and the algorithmic bytes one
 * launch moves (weights + scales + activations in and out).  Touches only
 * scratch activations and position 0 of the fast decoder's KV caches (which
 * every frame rewrites before reading); the decode state is unchanged.
 * Needs loaded weights.  Errors: TF_E_INVAL, TF_E_STATE, TF_E_CUDA. */
tf_status tf_profile_kernel(tf_ctx* ctx, int32_t which, int32_t iters,
                            float* ms_per_launch, int64_t* bytes_per_launch);

/* ---------------------------------------------------------------------------
 * Failure tests.  They make a failure happen without faulting the GPU, so
 * that the error paths can be tested: a bounded device wait that runs out,
 * and a device allocation that is refused.
 * ------------------------------------------------------------------------- */
enum { TF_TEST_SKIP_ONE_COPY = 1 };
/* TF_TEST_SKIP_ONE_COPY: the next tf_decode_frame of this (batch-1) context
 * runs its kernels directly instead of from the captured graph, and in its
 * first weight-streaming GEMV one CTA arms the barrier of its last stage
 * without issuing the copy.  That stage's bounded wait (200 ms) runs out,
 * the call returns TF_E_TIMEOUT and the context is poisoned as for any
 * expired wait (every later call but tf_destroy returns TF_E_STATE).
 * Errors: TF_E_INVAL (unknown test, batched context), TF_E_STATE. */
tf_status tf_test_inject(tf_ctx* ctx, int32_t what);
/* The n-th device allocation the library makes from now on (any context,
 * any thread; tf_create allocates everything) is refused as if cudaMalloc
 * had failed: that call returns TF_E_NOMEM and frees what it had allocated.
 * n <= 0 turns it off.  Not thread-safe with respect to which call is hit. */
void tf_test_fail_alloc(int32_t n);

/* ---------------------------------------------------------------------------
 * Single-operation entry points, for parity tests and profiling.  Each runs
 * one kernel of the decode path on caller-provided DEVICE buffers on `stream`
 * (cudaStream_t, NULL = legacy default stream) and synchronises it.
 * ------------------------------------------------------------------------- */

/* Per-row symmetric FP8 quantisation (drbaph s2-pro-fp8 model card,
 * "Quantization Details"): w_bf16 [rows][cols] (bf16 bits) ->
 * codes [rows][cols] float8_e4m3fn, scale [rows] float32 with
 * scale = amax/448 (IEEE float32 division; 1 for an all-zero row) and
 * code = e4m3 round-to-nearest-even of clamp(w / scale, -448, 448).
 * cols must be a multiple of 16.  Errors: TF_E_INVAL, TF_E_CUDA. */
tf_status tf_op_quantize_fp8(const uint16_t* w_bf16, int64_t rows, int64_t cols,
                             uint8_t* codes, float* scale, void* stream);

/* Block-scaled 4-bit quantisation of a bf16 weight [rows][cols] (cols a
 * multiple of 256): per row s = amax / (6 * 448) (IEEE float32 division; 1
 * for an all-zero row); per 16-element block b = e4m3 round-to-nearest-even
 * of min(amax_block / (6 * s), 448); code = FP4 E2M1 round-to-nearest-even
 * (ties to the even code) of clamp(w / (value(b) * s), -6, 6), 0 where b is
 * 0 -- each step one float32 operation.  packed: [rows][cols/2 + cols/16]
 * bytes (the codes, two per byte with the even element in the low nibble,
 * then the block scales); row_scale: float32 [rows].  All device pointers.
 * The value of element k is e2m1(code) * e4m3(b) * s.
 * Errors: TF_E_INVAL, TF_E_CUDA. */
tf_status tf_op_quantize_nvfp4(const uint16_t* w_bf16, int64_t rows, int64_t cols,
                               uint8_t* packed, float* row_scale, void* stream);

/* Codebook-id selection over float32 logits [n][vocab] (device); row i uses
 * Philox counter (frame, codebook0 + i, sequence, 0).  Writes ids [n] (device,
 * int32).  sampling as tf_sampling (top_k 0 = argmax).  vocab <= 8192.
 * recent: NULL, or device int32 [n][n_recent] ids that row i's repetition
 * window holds (entries < 0 are empty; sampling->rep_window is ignored here,
 * rep_penalty applies to these ids).  n_recent <= 64.
 * Errors: TF_E_INVAL, TF_E_NUMERIC (NaN logit), TF_E_CUDA. */
tf_status tf_op_select(const float* logits, int32_t n, int32_t vocab,
                       const tf_sampling* sampling, int32_t frame,
                       int32_t codebook0, int32_t sequence, const int32_t* recent,
                       int32_t n_recent, int32_t* ids, void* stream);

/* Grouped-query decode attention ("Fish Speech" tour, "Why You Need This":
 * rotary embeddings and grouped-query attention; tuna-fish README,
 * "Inference estimation": static KV cache), the decode path's attention
 * kernel on its own: query row m (m < rows) sits at position pos0 + m and
 * attends to keys 0..pos0+m of its KV head (query head h reads KV head
 * h / (Hq/Hkv)), scores scaled by 1/sqrt(D), softmax over the keys.
 * q: float32 [rows][Hq*D] (already rotated); K, V: bf16 bits [Hkv][T][D];
 * out: float32 [rows][Hq*D]; all device pointers.  `splits` (1..64) is the
 * number of key slices per KV head (at least 32 keys each) whose partial
 * softmax results are merged afterwards.  Allocates its scratch (partials,
 * tickets, error word) with cudaMalloc and frees it before returning.
 * D must be 64 or 128, Hq / Hkv one of 1, 2, 4, 8, pos0 + rows <= T.
 * Errors: TF_E_INVAL (bad argument or position), TF_E_NOMEM, TF_E_CUDA,
 * TF_E_TIMEOUT (a bounded wait for a key/value copy expired). */
tf_status tf_op_attention(const float* q, const uint16_t* K, const uint16_t* V, int32_t T,
                          int32_t Hq, int32_t Hkv, int32_t D, int32_t rows, int32_t pos0,
                          int32_t splits, float* out, void* stream);

/* tf_op_attention without any device allocation.  The source pages have no
 * counterpart to this call; it exists for callers that must not allocate
 * device memory while they run (a real-time loop with no allocator calls, a
 * host that gives all device memory to its own pool, a plugin kept off the
 * global CUDA allocator).  Same arguments, results and errors as
 * tf_op_attention, but the scratch comes from one fixed array built into the
 * library (present on every GPU that loads it, until the process exits):
 * calls need rows*Hq*splits*(D+2) <= 524288 and rows*Hkv <= 1024, else
 * TF_E_INVAL.  The first call on a device (and the first after its context
 * was reset) looks up the array's device address: make it before any stream
 * capture.  All calls share the array:
 * calls that overlap on the GPU race on it. */
tf_status tf_op_attention_noalloc(const float* q, const uint16_t* K, const uint16_t* V, int32_t T,
                                  int32_t Hq, int32_t Hkv, int32_t D, int32_t rows, int32_t pos0,
                                  int32_t splits, float* out, void* stream);

/* Causal attention of prompt rows on the tensor cores (tcgen05), the
 * prefill's attention kernel ("Fish Speech" tour, "Why You Need This":
 * grouped-query attention).  Same arguments and results as tf_op_attention
 * without `splits`: row m (position pos0 + m) attends to keys 0..pos0 + m of
 * the dense cache K, V [Hkv][T][D] (bf16, device), scores scaled by
 * 1/sqrt(D), softmax with max subtraction.  The queries are split into bf16
 * hi and lo parts (about 16 significant bits); the probabilities enter the
 * second product as bf16; accumulation is fp32.  D must be 64 or 128 and Hq
 * a multiple of Hkv.  Allocates and frees its scratch.  Errors: TF_E_INVAL,
 * TF_E_NOMEM, TF_E_CUDA, TF_E_TIMEOUT. */
tf_status tf_op_attention_prompt(const float* q, const uint16_t* K, const uint16_t* V, int32_t T,
                                 int32_t Hq, int32_t Hkv, int32_t D, int32_t rows, int32_t pos0,
                                 float* out, void* stream);

/* Prompt GEMM on the tensor cores (tcgen05, fp32 accumulation in TMEM), the
 * prefill's matrix kernel: C[m][n] = sum_k A[m][k] W[n][k] for the prompt
 * rows m.  A: float32 [M][K] device; W: bf16 bits [N][K] device; C: float32
 * [M][N] device.  A is split into bf16 hi and lo parts that are both
 * multiplied with W, so the result carries about 16 significant bits of A.
 * N must be a multiple of 128 and K of 64.  Output tiles are 128 rows by 128
 * columns (by 256 when M > 512 and N is a multiple of 256).  When the tiles
 * would not fill the GPU, K is split and the splits' partials are added in
 * split order (results do not depend on timing).  One CTA per SM works
 * through the (tile, split) units.  Allocates and frees its scratch.
 * Errors: TF_E_INVAL, TF_E_NOMEM, TF_E_CUDA, TF_E_TIMEOUT. */
tf_status tf_op_gemm(const float* A, const uint16_t* W, int32_t M, int32_t N, int32_t K, float* C,
                     void* stream);

/* Skinny GEMM on the tensor cores, the batched decode step's matrix kernel
 * (each linear layer of B lockstep sequences is a GEMM with B activation
 * rows; tuna-fish README, "Inference estimation": decode streams every
 * weight once per step, so one weight pass serves all B rows):
 * C[m][n] = sum_k A[m][k] W[n][k] for M <= 64 rows.  Weight rows sit on the
 * 128-row side of tcgen05.mma and the activation rows on its N side; K is
 * split so that the grid covers the GPU and the splits are added in a fixed
 * order (deterministic).  A: float32 [M][K] device, split into bf16 hi and lo
 * parts as in tf_op_gemm; W: bf16 bits [N][K] device; C: float32 [M][N]
 * device.  N even, K a multiple of 8 (ragged tiles are zero-filled).
 * Allocates and frees its scratch.  Errors: TF_E_INVAL, TF_E_NOMEM,
 * TF_E_CUDA, TF_E_TIMEOUT. */
tf_status tf_op_gemm_skinny(const float* A, const uint16_t* W, int32_t M, int32_t N, int32_t K,
                            float* C, void* stream);

/* tf_op_gemm_skinny with e4m3 weights (the drbaph s2-pro-fp8 card,
 * "Quantization Details": e4m3 codes with a float32 scale per output row):
 * C[m][n] = row_scale[n] * sum_k A[m][k] e4m3(W[n][k]).  The codes stream
 * from memory as they are and are converted to bf16 (exactly) in shared
 * memory for the tensor cores.  W: uint8 codes [N][K] device; row_scale:
 * float32 [N] device.  K a multiple of 16; other arguments and errors as
 * tf_op_gemm_skinny.  Codes must be finite (tf_load_weights refuses NaN). */
tf_status tf_op_gemm_skinny_fp8(const float* A, const uint8_t* W, const float* row_scale, int32_t M,
                                int32_t N, int32_t K, float* C, void* stream);

/* tf_op_gemm_skinny with block-scaled 4-bit weights in the layout
 * tf_op_quantize_nvfp4 writes (per row: K/2 bytes of e2m1 codes, the even
 * element in the low nibble, then K/16 e4m3 block-scale bytes; row_scale
 * float32 [N]): C[m][n] = row_scale[n] * sum_k A[m][k] w[n][k] with w = e2m1
 * value x block scale.  The rows stream as they are and are decoded to bf16
 * (exactly) in shared memory.  K a multiple of 256; other arguments and
 * errors as tf_op_gemm_skinny. */
tf_status tf_op_gemm_skinny_nvfp4(const float* A, const uint8_t* W, const float* row_scale, int32_t M,
                                  int32_t N, int32_t K, float* C, void* stream);

/* Weight-streaming GEMV y[r] = sum_k W[r][k] x[k] (the decode path's matrix
 * kernel, no prologue or epilogue): W bf16 [rows][cols] (dtype
 * TF_DTYPE_BF16), e4m3 codes with row_scale[rows] (TF_DTYPE_FP8_E4M3), or
 * 4-bit rows as tf_op_quantize_nvfp4 writes them with row_scale[rows]
 * (TF_DTYPE_NVFP4, cols a multiple of 256);
 * x, y float32 device vectors.  `repeat` > 1 launches it that many times
 * back to back (each launch with weights W + i * rows * cols elements, so the
 * caller can rotate through distinct matrices) and returns the mean device
 * time per launch in *ms (CUDA events on `stream`), if ms is not NULL.
 * e4m3 codes must be finite: a NaN code (0x7F, 0xFF) gives an undefined
 * result here (tf_load_weights refuses them).
 * Errors: TF_E_INVAL, TF_E_CUDA. */
tf_status tf_op_gemv(const void* W, int32_t dtype, const float* row_scale,
                     int64_t rows, int64_t cols, const float* x, float* y,
                     int32_t repeat, float* ms, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* TF_H */
