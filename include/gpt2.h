/*
 * gpt2.h -- C ABI of the GB300 GPT-2 decode library (libgpt2gb.so).
 *
 * The library computes the GPT-2 124M forward pass described in the LeanExe
 * GPT-2 README (model description paragraph): token plus position embedding;
 * per block LayerNorm, query/key/value projection, causal attention, output
 * projection and residual, LayerNorm, GELU feed-forward network and residual;
 * final LayerNorm and the tied vocabulary projection.  It also provides the
 * int8 group-64 variant of "Quantized GPT-2 Inference with Exact WebAssembly
 * Proofs" (abstract).  All arithmetic runs in this library's CUDA kernels
 * (sm_103a); there is no CPU fallback.
 *
 * Conventions for every entry point:
 *  - Pointers named *_host are host memory owned by the caller; pointers
 *    named d_* are device memory owned by the caller; handles own their own
 *    device memory.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default).
 *  - On a validation failure an entry returns its status, writes 0 to every
 *    output length and launches no device work (LeanExe GPT-2 README: invalid
 *    inputs return empty byte arrays).
 *  - Device-side failures of asynchronous calls (an invalid device-resident
 *    token, non-finite logits, a wait that timed out) are recorded in the
 *    session and returned by the next gpt2_session_sync().
 */
#ifndef GPT2_GB300_H
#define GPT2_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Model dimensions.  max_pos is the number of accepted positions (positions
 * 0..max_pos-1): 128 for the README's entry points ("accepts positions zero
 * through 127"), up to n_pos (1024 stored position rows) for long contexts.
 * Supported shapes: (d_model, d_ff, d_model/n_head) = (768, 3072, 64),
 * (192, 384, 64) and (64, 256, 16). */
typedef struct gpt2_config {
    uint32_t n_layer, d_model, n_head, d_ff, vocab, n_pos, max_pos;
} gpt2_config;

typedef enum gpt2_status {
    GPT2_OK = 0,
    GPT2_ERR_WEIGHTS_LEN = 1, /* weights_len != 4 * checkpoint words */
    GPT2_ERR_TOKEN = 2,       /* a token id >= vocab */
    GPT2_ERR_POSITION = 3,    /* position >= max_pos (or a run would pass it) */
    GPT2_ERR_CACHE_LEN = 4,   /* cache_len != position * n_layer * 2 * d_model * 4 */
    GPT2_ERR_TOKENS_LEN = 5,  /* token array empty, not a multiple of 4 bytes, or > max_pos ids */
    GPT2_ERR_NONFINITE = 6,   /* a step produced a NaN or infinite logit */
    GPT2_ERR_CONFIG = 7,      /* unsupported shape, quantization or grid */
    GPT2_ERR_NOMEM = 8,       /* a device or host allocation failed */
    GPT2_ERR_TIMEOUT = 9,     /* a device-side wait exceeded its limit; the run was abandoned */
    GPT2_ERR_CUDA = 10,       /* a CUDA runtime call failed */
    GPT2_ERR_ARG = 11,        /* a NULL pointer or an out-of-range argument */
    GPT2_ERR_SCRATCH = 12     /* the call needs more scratch than gpt2_cached_step_noalloc's static area */
} gpt2_status;

typedef enum gpt2_quant {
    GPT2_F32 = 0,      /* binary32 weights and arithmetic */
    GPT2_INT8_G64 = 1, /* int8 weights and projection inputs, scales per 64 inputs, int32 sums */
    GPT2_F16 = 2,      /* the 48 block matrices and the tied embedding stored as binary16 (rounded to
                          nearest-even at load), widened to binary32 before every multiply-add;
                          everything else binary32 (the gpt2.s page's half-precision weight option) */
    GPT2_INT8_ROW = 3, /* as GPT2_INT8_G64, but one weight scale per output row (maxabs over the whole
                          row / 127); the rescale keeps the grouped order with the row's scale in every
                          group's place; projection inputs keep their group-64 scales */
    GPT2_INT8_ROW_ACT = 4 /* as GPT2_INT8_ROW, and every projection input quantized with one scale for
                             the whole vector (maxabs / 127) in every group's place: the per-activation-row
                             design the quantized GPT-2 abstract measured and rejected */
} gpt2_quant;

/* In a device token array: use the previous step's greedy choice. */
#define GPT2_TOKEN_GREEDY 0xFFFFFFFFu

typedef struct gpt2_model gpt2_model;
typedef struct gpt2_session gpt2_session;
typedef struct gpt2_batch gpt2_batch;

/* Most sessions one gpt2_batch steps together. */
#define GPT2_BATCH_MAX 256u

/* Packed checkpoint size in 32-bit words (LeanExe GPT-2 README, packed
 * checkpoint paragraph: wte, all stored position rows, the blocks, the final
 * normalization; 124,439,808 words for GPT-2 124M).  0 for a NULL config. */
size_t gpt2_weight_words(const gpt2_config* cfg);

/* Words of one cached position: n_layer * 2 * d_model (README, cachedStep
 * paragraph: 12 x 1536 for GPT-2 124M). */
size_t gpt2_cache_words_per_position(const gpt2_config* cfg);

/* ---------------------------------------------------------------------
 * Byte-level entries with the README's semantics (host buffers; each call
 * uploads the checkpoint, runs on the GPU and copies results back; slow by
 * design, use the session API for decoding).
 * ------------------------------------------------------------------- */

/* infer (README, infer paragraph): weights = packed little-endian binary32
 * checkpoint; tokens = 1..max_pos little-endian u32 ids.  Writes the final
 * row's vocab logits to logits_out_host (capacity vocab floats) and
 * *logits_out_len = vocab.  Checks, in order: weights_len, tokens_len, each
 * token.  Runs the tensor-core prefill (gpt2_session_prefill). */
gpt2_status gpt2_infer(const gpt2_config* cfg, const void* weights_host, size_t weights_len,
                       const void* tokens_host, size_t tokens_len, float* logits_out_host,
                       size_t* logits_out_len);

/* cachedStep (README, cachedStep paragraph): one token at `position`, given a
 * cache of position*n_layer*2*d_model little-endian binary32 words ordered by
 * prior position, then layer, then d_model keys and d_model values (word
 * (source*n_layer + layer)*2*d_model + offset).  Writes vocab logits and the
 * cache with this position's rows appended (cache_out_host capacity
 * cache_len + n_layer*2*d_model*4 bytes; it may be the same buffer as
 * cache_host).  Checks, in order: weights_len, token, position, cache_len. */
gpt2_status gpt2_cached_step(const gpt2_config* cfg, const void* weights_host, size_t weights_len,
                             const void* cache_host, size_t cache_len, uint32_t token, uint32_t position,
                             float* logits_out_host, size_t* logits_out_len, void* cache_out_host,
                             size_t* cache_out_len);

/* ---------------------------------------------------------------------
 * Device-resident model and session (the measured path).
 * ------------------------------------------------------------------- */

/* Uploads the packed checkpoint and builds the device weight streams
 * (K-major copies of the block matrices; for GPT2_INT8_G64 the int8 copies
 * of the 48 block matrices and the tied wte with their group scales, for
 * GPT2_INT8_ROW and GPT2_INT8_ROW_ACT with their row scales; for GPT2_F16
 * binary16 copies of both).
 * grid_ctas: CTAs of the persistent step kernel, 0 = one per SM.
 * Synchronous.  Checks weights_len, the shape and the quantization. */
gpt2_status gpt2_model_create(const gpt2_config* cfg, const void* weights_host, size_t weights_len, int quant,
                              int grid_ctas, gpt2_model** out);
void gpt2_model_destroy(gpt2_model* model);

/* Copies back one int8 matrix of the model as q[out][in] (int8) and
 * s[out][in/64] (float): index 4*layer + {0: qkv, 1: out-proj, 2: fc,
 * 3: mlp-proj}, or 4*n_layer for the tied wte.  GPT2_ERR_CONFIG for a
 * binary32 model. */
gpt2_status gpt2_model_read_q8(gpt2_model* model, int index, int8_t* q_host, float* s_host);

/* Which kernel runs this model's decode steps: 1 the cluster step kernel
 * (thread-block clusters that complete each projection's split-K partials
 * in distributed shared memory; binary32 and binary16 models created while
 * the environment variable GPT2_STEP_KERNEL was "cluster"), 0 the per-phase
 * step kernel (int8 models, and the others unless "cluster" was asked
 * for; "phase" asks for it explicitly).  For the cluster
 * kernel *clusters and *cluster_size receive its grid (clusters x CTAs per
 * cluster); for the other they receive 0 and its CTA count.  Either pointer
 * may be NULL.  Returns -1 for a NULL model. */
int gpt2_model_step_kernel(const gpt2_model* model, uint32_t* clusters, uint32_t* cluster_size);

/* A session owns a device KV cache of max_pos positions and the step
 * kernel's scratch; it starts empty at position 0.  Synchronous. */
gpt2_status gpt2_session_create(gpt2_model* model, gpt2_session** out);
void gpt2_session_destroy(gpt2_session* session);

/* Current position (= number of cached positions), as enqueued. */
uint32_t gpt2_session_position(const gpt2_session* session);

/* Replaces the cache with cache_len bytes in the boundary layout above and
 * sets the position to cache_len / (n_layer*2*d_model*4).  Synchronous.
 * GPT2_ERR_CACHE_LEN unless cache_len is a whole number of positions below
 * max_pos. */
gpt2_status gpt2_session_load_cache(gpt2_session* session, const void* cache_host, size_t cache_len);

/* Truncates the session to its first `position` cached positions (the
 * cache words beyond are overwritten by later steps) and clears the greedy
 * history, stream-ordered on the session's last stream.  GPT2_ERR_POSITION
 * if position exceeds the current position. */
gpt2_status gpt2_session_rewind(gpt2_session* session, uint32_t position);

/* Copies the cache (position positions, boundary layout) to cache_host
 * (capacity bytes).  Synchronous; waits for queued runs. */
gpt2_status gpt2_session_read_cache(gpt2_session* session, void* cache_host, size_t capacity, size_t* len);

/* Enqueues n_steps cached steps at positions position..position+n_steps-1 as
 * ONE persistent kernel launch on `stream`.  d_tokens_in: device array of
 * n_steps token ids; GPT2_TOKEN_GREEDY takes the previous step's greedy
 * choice (for step 0: the session's last choice).  d_logits (may be NULL):
 * device output, step s written at d_logits + s*logits_stride floats
 * (logits_stride 0 = every step overwrites one row).  d_tokens_out (may be
 * NULL): device array receiving each step's greedy choice (argmax, lowest
 * index on ties; 0xFFFFFFFF if a logit was not finite).  Host-side checks:
 * n_steps >= 1 and position + n_steps <= max_pos.  The position advances
 * when the call returns. */
gpt2_status gpt2_session_run(gpt2_session* session, const uint32_t* d_tokens_in, uint32_t n_steps,
                             float* d_logits, size_t logits_stride, uint32_t* d_tokens_out, void* stream);

/* Prefill (README, infer paragraph; the prompt half of a session): the
 * full-prefix forward pass of n prompt tokens (d_tokens: device u32 ids) on
 * the tensor cores.  Starts an empty session (position 0, else
 * GPT2_ERR_POSITION); writes the KV-cache rows of positions 0..n-1, the
 * vocab logits of the last prompt row to d_logits (device, vocab floats;
 * NULL: the session's own buffer), and the greedy choice of those logits
 * (largest, lowest index on ties) as the session's last choice and, if
 * d_next_token is not NULL, to *d_next_token; leaves the session at
 * position n, so that gpt2_session_run / gpt2_session_step continue the
 * prompt.  binary32 models only (GPT2_ERR_CONFIG otherwise); 1 <= n <=
 * max_pos (GPT2_ERR_TOKENS_LEN).  An out-of-range token or a non-finite
 * logit is reported by the next gpt2_session_sync.  The first call on a
 * model makes the TF32 remainders of its block matrices (a one-off copy of
 * their size) and allocates the session's prefill workspace; the first call
 * for a given length and buffers records the prefill's launches as a CUDA
 * graph, which later calls replay.  Asynchronous, ordered on `stream` (a
 * cudaStream_t; NULL is the default stream). */
gpt2_status gpt2_session_prefill(gpt2_session* session, const uint32_t* d_tokens, uint32_t n, float* d_logits,
                                 uint32_t* d_next_token, void* stream);

/* One step with a host token; outputs as in gpt2_session_run.  Asynchronous. */
gpt2_status gpt2_session_step(gpt2_session* session, uint32_t token, float* d_logits, uint32_t* d_next_token,
                              void* stream);

/* One step with host buffers end to end: the token goes in as a kernel
 * argument, the logits (vocab floats) and greedy choice are copied back to
 * host memory, and the call waits for them.  Returns any device status. */
gpt2_status gpt2_session_step_host(gpt2_session* session, uint32_t token, float* logits_host,
                                   uint32_t* next_token_host);

/* A run with host buffers end to end: n_steps token ids from host memory
 * (GPT2_TOKEN_GREEDY as in gpt2_session_run; every other id checked < vocab
 * on the host, else GPT2_ERR_TOKEN and nothing runs), one persistent launch,
 * then every step's logits (n_steps*vocab floats, row s at s*vocab) to
 * logits_host and the greedy choices (n_steps ids) to tokens_out_host; either
 * may be NULL.  Pinned host memory makes the copies asynchronous; the call
 * waits for them and returns any device status.  The device buffers are
 * session-owned and grow to the largest n_steps seen. */
gpt2_status gpt2_session_run_host(gpt2_session* session, const uint32_t* tokens_host, uint32_t n_steps,
                                  float* logits_host, uint32_t* tokens_out_host);

/* Waits for the session's queued work and returns (and clears) the first
 * device-side failure recorded since the last sync. */
gpt2_status gpt2_session_sync(gpt2_session* session);

/* ---------------------------------------------------------------------
 * Batched independent sessions: B decode sessions of one binary32 model
 * stepped together.  Every step is one cachedStep (README, cachedStep
 * paragraph) per session, each at its own position on its own KV cache;
 * the sessions share only the weights, whose bytes one step reads once for
 * all B rows (tensor-core projections).
 * ------------------------------------------------------------------- */

/* Creates a batch of n_sessions (1..GPT2_BATCH_MAX) empty sessions (position
 * 0, no previous choice) with device KV caches of max_pos positions each.
 * binary32 models of a shape the tensor-core path supports only
 * (GPT2_ERR_CONFIG otherwise; the same shapes as gpt2_session_prefill).  The
 * first batch of a model makes the TF32 remainders of its block matrices
 * and of the tied embedding (one-off copies of their size, owned by the
 * model).  The batch refers to the model, which must outlive it. */
gpt2_status gpt2_batch_create(gpt2_model* model, uint32_t n_sessions, gpt2_batch** out);
void gpt2_batch_destroy(gpt2_batch* batch);
uint32_t gpt2_batch_size(const gpt2_batch* batch);
/* Position of session `index` (0 for a bad batch or index). */
uint32_t gpt2_batch_position(const gpt2_batch* batch, uint32_t index);

/* Session `index`: copies a host cache of len bytes (a whole number of
 * positions, fewer than max_pos; boundary layout) into its cache, sets its
 * position to that number and forgets its previous choice.  Synchronous. */
gpt2_status gpt2_batch_load_cache(gpt2_batch* batch, uint32_t index, const void* cache_host, size_t len);

/* Session `index`: copies its cache (position positions) to cache_host
 * (capacity bytes).  Synchronous; waits for queued steps. */
gpt2_status gpt2_batch_read_cache(gpt2_batch* batch, uint32_t index, void* cache_host, size_t capacity,
                                  size_t* len);

/* Enqueues n_steps steps of every session on `stream` (a cudaStream_t; NULL
 * is the default stream).  d_tokens_in: device array [n_steps][B] of token
 * ids; GPT2_TOKEN_GREEDY takes that session's previous greedy choice.
 * d_logits (may be NULL): device output, session b of step s at d_logits +
 * s*logits_stride + b*vocab floats (logits_stride 0 = every step overwrites
 * one [B][vocab] block; else at least B*vocab).  d_tokens_out (may be NULL):
 * device array [n_steps][B] of greedy choices (largest, lowest index on
 * ties; 0xFFFFFFFF if a logit of that row was not finite).  Host-side
 * checks: n_steps >= 1, every position + n_steps <= max_pos.  The positions
 * advance when the call returns.  An out-of-range token, a greedy token
 * without a previous choice and non-finite logits are reported by the next
 * gpt2_batch_sync; after such a failure the caches and positions are
 * unspecified until reloaded.  The first call for a set of buffers records
 * one step's launches as a CUDA graph, replayed once per step. */
gpt2_status gpt2_batch_run(gpt2_batch* batch, const uint32_t* d_tokens_in, uint32_t n_steps, float* d_logits,
                           size_t logits_stride, uint32_t* d_tokens_out, void* stream);

/* Every session back to `position` (each must be at or past it, else
 * GPT2_ERR_POSITION and nothing changes), with no previous choice; its
 * cache rows below `position` are kept.  Asynchronous, ordered on `stream`. */
gpt2_status gpt2_batch_rewind(gpt2_batch* batch, uint32_t position, void* stream);

/* Waits for the batch's queued steps and returns (and clears) the first
 * device-side failure recorded since the last sync. */
gpt2_status gpt2_batch_sync(gpt2_batch* batch);

/* Debug: enqueue the next run with an activation trace.  d_trace receives,
 * for step 0 of that run only, per layer: x_in[d], LN1(x)[d], qkv[3d],
 * attention output[d], x_mid[d], LN2(x_mid)[d], gelu output[d_ff]; then
 * x_final[d], LN_f(x_final)[d].  Pass NULL to stop tracing. */
gpt2_status gpt2_session_set_trace(gpt2_session* session, float* d_trace);

/* Profiling: enqueue the next run with phase timestamps.  d_stamps
 * (device, (5*n_layer+1) * grid_ctas * 8 u64, phase-major) receives, for
 * step 0 of that run, per phase and CTA: [0..2] the device globaltimer (ns)
 * when the CTA started the phase, when its inputs were complete and when
 * its outputs were stored; [3..6] the SM's clock64 when its inputs were
 * complete, when its projection started (after LayerNorm / head merge /
 * quantization), when thread 0's projection work ended and when its outputs
 * were stored; [7] clock64 when the phase's first weight chunk was known to
 * have landed.  Attention phases fill [0..6] only.
 * Models on the cluster step kernel (gpt2_model_step_kernel == 1) use
 * another layout: d_stamps holds 8 + grid_ctas * (16*n_layer + 8) u64.
 * Words 0..5 receive, when a bounded wait of the run gives up, the wait's
 * kind (1 ring chunk, 2 distributed-shared-memory gather, 3 tagged words,
 * 4 greedy partials), the CTA, the step, the layer and two words about what
 * was awaited (for kind 4: (partial index << 32 | tag), and the word last
 * seen); all 0 when none gave up.  Then per CTA (CTA-major), for step 0,
 * per layer 16 words: the globaltimer (ns) when the block input was formed,
 * QKV partials done, q/k/v gathered, attention done, head outputs gathered,
 * out-projection partials stored, attention residual formed, FC partials
 * done, GELU outputs gathered, MLP partials stored (a CTA of a cluster
 * without a head leaves the second to sixth at 0); 6 words unused.  Then
 * final input formed, gathered, LN_f done, vocabulary rows done; then, if a wait of
 * this CTA gave up, (kind | 0x100 if it left because another CTA had
 * given up | thread index << 16), the step, the layer and what was
 * awaited.  Pass NULL to stop. */
gpt2_status gpt2_session_set_timing(gpt2_session* session, uint64_t* d_stamps);

/* Debug/test: make the next run's CTA 0 skip publishing one phase so that
 * the other CTAs' bounded waits expire and the run ends with
 * GPT2_ERR_TIMEOUT (no GPU fault, no hang).  wait_limit_ns bounds every
 * device-side wait of that run. */
gpt2_status gpt2_session_inject_stall(gpt2_session* session, uint32_t phase, uint64_t wait_limit_ns);

/* gpt2_cached_step_noalloc -- one cached step that allocates nothing.
 * The pages have no counterpart: this entry exists for callers that may not
 * allocate device memory while they run steps.  Examples are a plug-in or
 * embedded runtime whose host framework owns every device allocation within
 * a fixed budget, and a latency-critical loop that cannot afford cudaMalloc,
 * which may synchronise the device.  The caller still passes every input and
 * output:
 *   model         created once beforehand with gpt2_model_create;
 *   d_cache       caller-owned device KV cache in the cachedStep layout
 *                 above, holding positions 0..position-1, with room for
 *                 position+1 positions; this step's keys and values are
 *                 written at position `position`;
 *   token         this step's token id (< vocab; GPT2_TOKEN_GREEDY is
 *                 rejected);
 *   d_logits      device output of vocab floats, or NULL;
 *   d_next_token  device output of the greedy choice, or NULL; it reads
 *                 0xFFFFFFFF after the step if a logit was not finite or the
 *                 step gave up on a device-side wait.  It is the call's only
 *                 failure signal (the host reads no status back): pass it
 *                 whenever a failed step must be detected; with NULL a
 *                 failed step leaves d_logits partly written, unnoticed.
 * The step kernel's scratch is a file-scope static device array of 512 KiB
 * (GPT-2 124M uses about 360 KB on the cluster step kernel, 70 KB on the
 * per-phase kernel).  Every GPU that loads the library's device code holds
 * it until the process exits.  A model whose scratch would not fit is
 * rejected with GPT2_ERR_SCRATCH before any device work.  gpt2_model_create
 * loads the array's module and looks its device address up on the device
 * that is current (CUDA may load modules lazily, so this is where the array
 * comes into being); a call on a device where no model was created does that
 * set-up itself, so make such a first call before any stream capture.
 * No call allocates: no cudaMalloc, no cudaFree, no allocating library
 * routine.  All calls share the one array, and it keeps the previous call's
 * contents.  Each call clears, on `stream`, what must start at zero (phase
 * flags, status words).  Calls that overlap on the GPU race on the array:
 * order them on one stream, or otherwise serialize them.  Enqueued on
 * `stream`; host-side checks: model, d_cache, token, position < max_pos. */
gpt2_status gpt2_cached_step_noalloc(const gpt2_model* model, float* d_cache, uint32_t position, uint32_t token,
                                     float* d_logits, uint32_t* d_next_token, void* stream);

/* Test hook: applies projection `index` of the model (index convention of
 * gpt2_model_read_q8; the vocabulary projection has no bias) to the device
 * vector d_x (its input width in floats) and writes d_y (its output width),
 * using the step kernel's own device routines and the path it takes for that
 * matrix (rows spread over warps for block matrices, one warp per ring chunk
 * for the vocabulary): for int8 models the per-64 activation quantizer, the
 * dp4a group sums and the fixed-order rescale; for binary32 models the float4
 * dot products; for binary16 models the same on widened binary16 weights.
 * Enqueued on `stream`. */
gpt2_status gpt2_debug_project(gpt2_model* model, int index, const float* d_x, float* d_y, void* stream);

/* Test hook: the step kernel's greedy-choice routine over d_values[n]:
 * *d_index = index of the largest value (lowest index on ties), and
 * *d_nonfinite = 1 with *d_index = 0xFFFFFFFF if any value is NaN or
 * infinite.  Enqueued on `stream`. */
gpt2_status gpt2_debug_argmax(const float* d_values, uint32_t n, uint32_t* d_index, int* d_nonfinite,
                              void* stream);

/* The CUDA runtime error behind the most recent GPT2_ERR_CUDA / NOMEM of
 * this process (0 if none), and its name (e.g. "cudaErrorIllegalAddress"). */
int gpt2_last_cuda_error(const char** name);

/* Human-readable status name ("ok", "token", ...). */
const char* gpt2_status_name(gpt2_status status);

#ifdef __cplusplus
}
#endif
#endif /* GPT2_GB300_H */
