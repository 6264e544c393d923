/*
 * dec.h - C ABI of the GB300 (sm_103a) Qwen3-style speech-LLM decoder.
 *
 * The library runs the causal-LM decoder of the speech-LLM pipelines in
 * transcribe.cpp: audio-injected prompt rows go through a prefill, then a
 * greedy single-token step loop emits text token ids.  Each block is pre-LN
 * RMSNorm, GQA attention with per-head Q/K RMSNorm, NeoX RoPE and a KV-cache
 * write/read, then SwiGLU on a packed gate_up projection and the down
 * projection; a final RMSNorm and the tied lm_head with argmax close the
 * step.  (qwen3_asr/decoder.cpp, transcribe-cpp-sys 0.2.0: file header,
 * build_prefill_graph, build_step_graph; qwen3_asr/model.cpp, run.)
 *
 * Conventions shared by every entry point:
 *  - Every call returns a dec_status.  Invalid arguments are rejected before
 *    any work is queued (the pages' graph builders validate and return
 *    before building, decoder.cpp build_prefill_graph).
 *  - Memory: the caller owns the device workspace (size from
 *    dec_workspace_size) and every host buffer it passes.  The library never
 *    allocates device memory and never frees caller memory.  Weights are
 *    copied (and packed) into the workspace by dec_create; the caller may
 *    free its host copy afterwards.
 *  - Streams: all device work is queued on the stream given to dec_create.
 *    Calls that return host results (tokens, logits) synchronise that stream
 *    before returning.  A handle is not thread-safe.
 *  - Unless stated, pointers are host pointers.  Arguments named `on_device`
 *    select host (0) or device (1) memory for the data pointers of one call.
 *  - Matrices are row-major; weights use the [out, in] layout of the
 *    checkpoint format (a mul_mat of the weight against the activations).
 */
#ifndef SPEECH_DECODER_GB300_DEC_H
#define SPEECH_DECODER_GB300_DEC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes follow the pages' transcribe_status set (OK, invalid argument,
 * out of memory, input too long, output truncated, backend failure). */
typedef enum dec_status {
    DEC_OK = 0,
    DEC_ERR_INVALID_ARG = 1,       /* bad pointer, size or hyper-parameter            */
    DEC_ERR_OOM = 2,               /* workspace smaller than dec_workspace_size()      */
    DEC_ERR_INPUT_TOO_LONG = 3,    /* prompt + generation budget exceed the context    */
    DEC_ERR_OUTPUT_TRUNCATED = 4,  /* budget or context reached before EOS (ids valid) */
    DEC_ERR_CUDA = 5,              /* a CUDA runtime call failed                       */
    DEC_ERR_STATE = 6,             /* call out of order (e.g. step before prefill)     */
    DEC_ERR_DEVICE = 7             /* a kernel reported an error status                */
} dec_status;

/* DEC_E4M3 (weights only): the weights are passed as bf16; dec_create rounds
 * every row of the projection matrices and of the tied embedding to
 * 2^e * e4m3 as dec_quantize_e4m3_rows does, keeps the rounded values in bf16
 * for the prompt path (and the embedding lookup), and the single-sequence
 * step GEMVs stream the 1-byte codes with per-row scales.  Both paths compute
 * with the same (rounded) weights; norm weights are not rounded.  The
 * workspace (dec_workspace_size) holds both forms: one more byte per
 * projection and embedding weight and one float per row. */
typedef enum dec_dtype { DEC_BF16 = 0, DEC_F32 = 1, DEC_F16 = 2, DEC_E4M3 = 3 } dec_dtype;

/* Model shape and run limits (qwen3_asr/decoder.cpp, to_block_params:
 * n_heads, n_kv_heads, head_dim, max_position, rms_eps, rope_theta). */
typedef struct dec_hparams {
    int32_t n_layers;      /* decoder blocks                                    */
    int32_t hidden;        /* model width H; multiple of 256                   */
    int32_t n_heads;       /* query heads; multiple of n_kv_heads              */
    int32_t n_kv_heads;    /* key/value heads                                  */
    int32_t head_dim;      /* d: 64 or 128                                      */
    int32_t ffn;           /* SwiGLU width F; multiple of 128                  */
    int32_t vocab;         /* tied embedding / lm_head rows                    */
    float rms_eps;         /* RMSNorm epsilon (block, Q/K and final norms)      */
    float rope_theta;      /* NeoX RoPE base                                   */
    int32_t max_ctx;       /* KV slots one sequence may use (context ceiling)  */
    int32_t max_batch;     /* sequences per prefill/step call                  */
    int32_t max_tokens;    /* prompt rows per prefill call, summed over items  */
    int32_t max_new;       /* generation budget; the length gate rejects a
                              prompt with T + max_new > max_ctx                 */
    int32_t eos_id;        /* end-of-stream token, -1 for none                 */
    int32_t weight_dtype;  /* DEC_BF16 (production), DEC_E4M3 (bf16 in, e4m3
                              step weights) or DEC_F32 (debug build)           */
    int32_t kv_dtype;      /* DEC_F16 with BF16 or E4M3 weights; DEC_F32 with F32 */
} dec_hparams;

/* Host pointers to one block's weights, each in hparams.weight_dtype (bf16
 * as raw 16-bit patterns; bf16 for DEC_E4M3 too).  Shapes: attn_norm, ffn_norm [H]; q [n_heads*d, H];
 * k, v [n_kv_heads*d, H]; o [H, n_heads*d]; q_norm, k_norm [d] (one vector
 * shared by all heads); gate, up [F, H]; down [H, F]. */
typedef struct dec_layer_weights {
    const void *attn_norm, *q, *k, *v, *o, *q_norm, *k_norm, *ffn_norm, *gate, *up, *down;
} dec_layer_weights;

typedef struct dec_weights {
    const void *embed;                 /* [vocab, H]; also the tied lm_head */
    const void *final_norm;            /* [H]                               */
    const dec_layer_weights *layers;   /* n_layers entries                  */
} dec_weights;

typedef struct dec_handle dec_handle;

/* Bytes of device workspace dec_create needs for these hyper-parameters
 * (packed weights, KV pool of max_batch*max_ctx slots, activations, scratch).
 * Returns DEC_ERR_INVALID_ARG for unsupported shapes. */
dec_status dec_workspace_size(const dec_hparams *hp, size_t *bytes);

/* Validate hp, carve the caller's device workspace (256-byte aligned,
 * ws_bytes >= dec_workspace_size) and upload the weights: q|k|v packed into
 * one [(n_heads+2*n_kv_heads)*d, H] matrix and gate|up packed into one
 * [2F, H] matrix in blocks of 128 rows (gate rows of the block, then the up
 * rows of the same features; model.cpp, load: pack_gate_up).  `stream` is a
 * cudaStream_t; it must not be the legacy default stream, because the step
 * loop is captured into CUDA graphs.  NULL makes the handle create (and
 * later destroy) its own non-blocking stream.  Blocks until the upload is
 * done.  On success *out owns host-side objects only; free with dec_destroy. */
dec_status dec_create(const dec_hparams *hp, const dec_weights *w, void *workspace,
                      size_t ws_bytes, void *stream, dec_handle **out);

/* Release the handle's host objects and CUDA graphs (not the workspace). */
void dec_destroy(dec_handle *h);

/* Forget all sequences (n_past = 0).  KV memory is reused, not cleared:
 * every read is bounded by the sequence length (model.cpp, run: session
 * reuse clears the cache; bounding reads gives the same results). */
dec_status dec_reset(dec_handle *h);

/* Prefill one sequence from its input rows.  embeds: float32 [T, H], the
 * audio-injected prompt (prefix token embeddings | encoder rows | suffix
 * token embeddings), host or device memory per on_device.  Writes the KV
 * cache for positions 0..T-1 and returns the argmax of the last row's
 * logits in *first_token (decoder.cpp, build_prefill_graph; model.cpp, run).
 * Replaces any previous sequences.  DEC_ERR_INPUT_TOO_LONG when
 * T + max_new > max_ctx or T > max_tokens (model.cpp, run: input-length gate). */
dec_status dec_prefill(dec_handle *h, const float *embeds, int32_t T, int32_t on_device,
                       int32_t *first_token);

/* Chunked prefill of one sequence: embeds float32 [T, H] are the next T
 * prompt rows, at positions [p, p + T) where p counts the rows of earlier
 * chunks since the last reset or whole-prompt prefill; every block attends to
 * the cached keys of the earlier chunks (causal over the whole prompt).  The
 * sequence owns KV slots [0, max_ctx).  final_chunk != 0 also runs the head on
 * the last row: *first_token = the prompt's greedy token and the handle is
 * ready for dec_step / dec_generate, exactly as after dec_prefill of the whole
 * prompt; otherwise *first_token = -1, only the KV cache advances, and steps
 * return DEC_ERR_STATE until a final chunk.  DEC_ERR_INPUT_TOO_LONG if
 * p + T + max_new > max_ctx or T > max_tokens (no work done; the chunked
 * prompt is abandoned on any error).  The pages' long-prompt path feeds the
 * prompt in chunks against the growing KV cache (MOSS: chunked prefill with
 * chunked == single-shot logits). */
dec_status dec_prefill_chunk(dec_handle *h, const float *embeds, int32_t T, int32_t on_device,
                             int32_t final_chunk, int32_t *first_token);

/* Prefill one sequence from token ids and encoder rows, assembling the rows
 * on the device: rows = embed[ids[0:prefix_len]] | audio | embed[ids[prefix_len:]]
 * (decoder.cpp, build_prefill_graph: get_rows + 3-way concat).
 * ids: int32 [n_ids]; audio: float32 [n_audio, H]; T = n_ids + n_audio. */
dec_status dec_prefill_ids(dec_handle *h, const int32_t *ids, int32_t n_ids, const float *audio,
                           int32_t n_audio, int32_t prefix_len, int32_t on_device,
                           int32_t *first_token);

/* Ragged batched prefill of B sequences.  embeds: float32 [sum T_b, H] with
 * sequence b in rows cu_seqlens[b] .. cu_seqlens[b+1]-1; cu_seqlens: int32
 * [B+1] host memory, cu_seqlens[0] = 0.  Each sequence gets its own
 * positions 0..T_b-1 and an exact-fit KV range of T_b + max_new slots.
 * first_tokens: int32 [B].  (decoder.cpp, build_prefill_graph_batched;
 * rows are ragged, with no padding.) */
dec_status dec_prefill_batch(dec_handle *h, const float *embeds, const int32_t *cu_seqlens,
                             int32_t B, int32_t on_device, int32_t *first_tokens);

/* Ragged batched form of dec_prefill_ids: item b has token ids
 * ids[cu_ids[b] .. cu_ids[b+1]) and encoder rows audio[cu_audio[b] ..
 * cu_audio[b+1]) (float32 rows of width H), assembled on the device as
 * embed[ids[:prefix_lens[b]]] | audio rows | embed[ids[prefix_lens[b]:]].
 * cu_ids, cu_audio: int32 [B+1] and prefix_lens: int32 [B], host memory; ids
 * and audio in host or device memory per on_device.  first_tokens: int32 [B]. */
dec_status dec_prefill_ids_batch(dec_handle *h, const int32_t *ids, const int32_t *cu_ids,
                                 const float *audio, const int32_t *cu_audio,
                                 const int32_t *prefix_lens, int32_t B, int32_t on_device,
                                 int32_t *first_tokens);

/* One greedy step of sequence 0: `token` at position n_past, its K/V written
 * at slot n_past, returns the argmax of the logits (decoder.cpp,
 * build_step_graph).  DEC_ERR_STATE before a prefill; DEC_ERR_INPUT_TOO_LONG
 * when the sequence's KV range is full. */
dec_status dec_step(dec_handle *h, int32_t token, int32_t *next_token);

/* One step of every sequence of the last batched prefill.  tokens: int32
 * [B]; active: uint8 [B] (0 = skip the row: no KV write, no output) or NULL
 * for all; next_tokens: int32 [B] (-1 for skipped rows). */
dec_status dec_step_batch(dec_handle *h, const int32_t *tokens, const uint8_t *active,
                          int32_t *next_tokens);

/* Greedy loop of sequence 0 after dec_prefill (model.cpp, run): ids start
 * with the prefill's token; the loop stops at EOS, at max_new ids (the
 * prefill's token counts), or when the KV range is full.  A trailing EOS is
 * stripped.  out_ids: int32 [max_new]; *n_out ids written.  Returns
 * DEC_ERR_OUTPUT_TRUNCATED (ids still valid) when no EOS was produced.
 * max_new <= hparams.max_new.  The step loop runs on the device: tokens feed
 * the next step without a host round trip. */
dec_status dec_generate(dec_handle *h, int32_t max_new, int32_t *out_ids, int32_t *n_out);

/* Batched greedy loop with per-item EOS (model.cpp, run_batch:
 * run_batched_step_loop): finished rows stop writing KV and stay finished.
 * out_ids: int32 [B, max_new] row-major; n_out, truncated: int32 [B].
 * Returns DEC_OK even when some items were truncated (see truncated[]). */
dec_status dec_generate_batch(dec_handle *h, int32_t max_new, int32_t *out_ids, int32_t *n_out,
                              int32_t *truncated);

/* Generation budget of a run (moss/model.cpp of transcribe-cpp-sys 0.4.1,
 * run and run_batch: the budget handed to the greedy loop).  The page asks
 * for twice the audio rows plus 128 tokens (room above the plain audio-token
 * count for the transcript's markers), takes the fixed generation reserve as
 * the floor and the context left after the prompt as the cap; it shows the
 * call, not the helper's body.  Reading taken here:
 *     *budget = min(max(2 * n_audio + 128, floor_new), ceiling - T_prompt)
 * n_audio: encoder rows injected into the prompt (>= 0); T_prompt: prompt
 * rows (>= 1); floor_new: the generation reserve (the pages' 256; >= 1);
 * ceiling: the context ceiling in tokens (hparams.max_ctx for this library).
 * For a batch the page passes the longest audio and the longest prompt of
 * the batch.  DEC_ERR_INPUT_TOO_LONG when T_prompt + floor_new > ceiling
 * (the page's gate, checked before the budget); DEC_ERR_INVALID_ARG for a
 * null budget pointer or an argument out of range.  Host arithmetic only:
 * no device work.  Pass the result as max_new to dec_generate or
 * dec_generate_batch (a decoder whose hparams.max_new is at least the
 * budget); the loop then stops at EOS, at the budget, or when the KV range
 * is full. */
dec_status dec_decode_budget(int32_t n_audio, int32_t T_prompt, int32_t floor_new, int32_t ceiling,
                             int32_t *budget);

/* Copy the logits rows of the last prefill/step (one row per sequence,
 * float32 [rows, vocab]) into host memory.  rows <= sequences of that call. */
dec_status dec_debug_logits(dec_handle *h, float *out, int32_t rows);

/* Enable (1) or disable (0) capture of named intermediates during prefill
 * (the pages' dump points, decoder.cpp build_prefill_graph: dec.block.0.out,
 * dec.block.last.out, dec.out_before_head).  Off by default. */
dec_status dec_set_dumps(dec_handle *h, int32_t enable);

/* Copy a captured intermediate (float32) into host memory.  names:
 * "dec.audio_injected" [T, H], "dec.block.0.out" [T, H] (all rows),
 * "dec.block.last.out" [B, H] (last row of each sequence; the last block
 * runs its attention query, FFN and head on those rows only),
 * "dec.out_before_head" [B, H].  n_floats must equal the tensor size. */
dec_status dec_debug_dump(dec_handle *h, const char *name, float *out, size_t n_floats);

/* Kernel launches this handle has issued so far (a graph launch counts its
 * kernel nodes). */
dec_status dec_launch_count(const dec_handle *h, int64_t *count);

/* Device time (milliseconds, CUDA events on the handle's stream) of the last
 * prefill and of the last generate loop. */
dec_status dec_last_timings(const dec_handle *h, float *prefill_ms, float *generate_ms);

/* Time one family of decode kernels in isolation on the handle's stream
 * (CUDA events around `iters` rounds; each round launches the kernel once
 * per layer, so consecutive launches stream different weights and no
 * launch is served from L2).  op 0: the step's projection GEMVs of every
 * layer in step order (q|k|v, o, gate|up with SwiGLU, down), without the
 * attention between them; op 1: the lm_head + argmax GEMV; op 2: the
 * split-KV attention at the current lengths; op 3: one whole decode step
 * (the persistent step kernel when it is in use; *avg_ms is then per step
 * and *bytes_per_launch the step's algorithmic bytes).  Needs a prior prefill (it
 * reads and rewrites the step buffers; the KV cache and sequence state are
 * left as they were).  *avg_ms = mean duration of one launch;
 * *bytes_per_launch = algorithmic bytes one launch must move (weights,
 * activations, KV). */
dec_status dec_profile_kernel(dec_handle *h, int32_t op, int32_t iters, float *avg_ms,
                              double *bytes_per_launch);

/* ---------------------------------------------------------------------
 * Standalone kernel: the split-KV grouped-query attention of the step
 * (decoder.cpp, build_step_graph: attention of one new row per sequence
 * over its cached keys), for queries that are already Q-normed and rotated.
 * All data pointers are device memory; work is queued on `stream` and the
 * call returns without synchronising.
 *   q       float32 [B, n_heads, head_dim]
 *   K, V    pool [n_kv_heads, slots, head_dim] of kv_dtype (DEC_F16/DEC_F32)
 *   kv_off  int32 [B]: first pool slot of sequence b
 *   kv_len  int32 [B]: keys kv_off[b] .. kv_off[b]+kv_len[b]-1 are visible;
 *           rows with kv_len <= 0 or outside the pool are skipped and their
 *           output left unchanged
 *   out     float32 [B, n_heads, head_dim] = softmax(q k^T / sqrt(d)) v with
 *           query head h reading KV head h / (n_heads / n_kv_heads)
 *   scratch device memory of at least dec_attn_decode_scratch_size() bytes
 *           (per-split partials and arrival counters; zeroed by the call)
 * Shapes: head_dim 64 or 128, n_heads a multiple of n_kv_heads, at most 8
 * query heads per KV head.  Calls sharing one scratch buffer must not
 * overlap on the GPU. */
dec_status dec_attn_decode_scratch_size(int32_t B, int32_t n_heads, int32_t n_kv_heads,
                                        int32_t head_dim, size_t *bytes);
dec_status dec_attn_decode(const float *q, const void *K, const void *V, int32_t kv_dtype,
                           int32_t slots, const int32_t *kv_off, const int32_t *kv_len, int32_t B,
                           int32_t n_heads, int32_t n_kv_heads, int32_t head_dim, float *out,
                           void *scratch, size_t scratch_bytes, void *stream);

/* dec_attn_decode without the scratch argument, for callers that cannot
 * allocate device memory: code running inside a host engine or plugin
 * interface whose device memory belongs to someone else and offers no
 * allocator, or a latency-bound loop that must not call cudaMalloc (which can
 * synchronise the device).  The pages have no counterpart: their decoder
 * always owns a ggml scheduler that allocates its own buffers.
 *
 * Arguments and results are those of dec_attn_decode.  The partials and the
 * arrival counters live in one file-scope device array of 4 MiB, reserved on
 * every GPU that loads the library and held until the process exits; a shape
 * whose scratch (dec_attn_decode_scratch_size) exceeds 4 MiB returns
 * DEC_ERR_OOM without launching.  The call allocates nothing (no cudaMalloc,
 * cudaFree or allocating library routine); it zeroes the counters with
 * cudaMemsetAsync on `stream`.  The first call on a device looks up the
 * array's device address (cudaGetSymbolAddress) with that device current;
 * make that first call before any stream capture.  That address is kept for
 * the life of the process: after cudaDeviceReset, or once the device's
 * primary context was destroyed and created again, the kept address is stale,
 * so do not call this entry point on that device again.  Every call shares
 * the one array, so calls that overlap on the GPU (other streams, other
 * threads) race and corrupt each other's results: serialise them.  The
 * scratch a shape needs is dec_attn_decode_scratch_size(); for 8 KV heads of
 * 2 query heads each and head_dim 128 the array holds up to 502 sequences. */
dec_status dec_attn_decode_noalloc(const float *q, const void *K, const void *V, int32_t kv_dtype,
                                   int32_t slots, const int32_t *kv_off, const int32_t *kv_len,
                                   int32_t B, int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                                   float *out, void *stream);

/* Perception projection of encoder rows (canary_qwen/model.cpp, forward
 * shape: FastConformer encoder -> perception projection Linear(1024, 2048) +
 * bias -> rows scattered into the prompt): out[t][f] = sum_k W[f][k] enc[t][k]
 * + bias[f].  Device pointers: enc float32 [T, d_in]; W bf16 [d_out, d_in]
 * (HF [out, in]); bias float32 [d_out]; out float32 [T, d_out] (may be the
 * encoder rows that dec_prefill_ids then reads with on_device = 1).  The
 * activation enters the tensor-core GEMM as two bf16 planes (value and
 * rounding residual).  d_in a multiple of 64, d_out a multiple of 128;
 * scratch: caller-owned device memory of at least 2 * align256(T d_in 2) + 16 MiB
 * (DEC_ERR_OOM otherwise).  Runs on `stream` (NULL = legacy default stream);
 * returns after the launch. */
dec_status dec_perception_project(const float *enc, int32_t T, int32_t d_in, const void *W, const float *bias,
                                  int32_t d_out, float *out, void *scratch, size_t scratch_bytes, void *stream);

/* Per-row e4m3 rounding of bf16 weights, the DEC_E4M3 weight format (an
 * extension of the pages' weight-streaming decode; their decoder streams
 * bf16 or f32 weights).  Row r gets the scale 2^e_r, e_r the smallest integer
 * with max_k |w[r][k]| <= 448 * 2^e_r (scale 1 for an all-zero row); codes[r][k]
 * is the e4m3 value nearest w[r][k] / 2^e_r, ties to even (OCP 8-bit floating
 * point, E4M3: exponent bias 7, 3 mantissa bits, subnormals, largest finite
 * 448, byte = sign | exponent | mantissa); w_rounded[r][k] = value(codes[r][k])
 * * 2^e_r, exact in bf16.  Device pointers: w bf16 [rows, cols] (raw 16-bit
 * patterns); codes uint8 [rows, cols]; scales float32 [rows]; w_rounded bf16
 * [rows, cols], may equal w (rounded in place).  rows >= 1, cols >= 1.  Runs
 * on `stream` (NULL = legacy default stream); returns after the launch. */
dec_status dec_quantize_e4m3_rows(const void *w, int64_t rows, int32_t cols, uint8_t *codes, float *scales,
                                  void *w_rounded, void *stream);

/* Standalone kernel (test hook): one prompt-row projection of the prefill,
 * C = X W^T (epi 0: store, epi 1: add into C) or, with gate|up packed in
 * blocks of 128 rows (epi 2), Hout = silu(gate) * up in bf16.  X bf16 [T, K],
 * W bf16 [n_feat, K], C float32 [T, ldc], Hout bf16 [T, ldh]; all device
 * memory.  use_tc = 1 runs the tcgen05 GEMM, 0 the CUDA-core GEMM (epi 0/1
 * only).  splits > 0 forces the tcgen05 split-K count.  scratch: device
 * memory for split-K partial tiles, scratch_bytes >= 16 MB.  Queued on
 * `stream`. */
dec_status dec_debug_gemm(const void *X, int32_t T, const void *W, int32_t n_feat, int32_t K,
                          int32_t epi, float *C, int32_t ldc, void *Hout, int32_t ldh, int32_t use_tc,
                          int32_t splits, void *scratch, size_t scratch_bytes, void *stream);

/* Message of the last error on this handle ("" if none). */
const char *dec_last_error(const dec_handle *h);

/* Name of a status code. */
const char *dec_status_string(dec_status s);

#ifdef __cplusplus
}
#endif
#endif /* SPEECH_DECODER_GB300_DEC_H */
