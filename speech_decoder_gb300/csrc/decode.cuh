// Decode-path kernel interfaces (one token per sequence per step).
#pragma once
#include "common.cuh"

namespace dec {

enum GemvIn { IN_NORM = 0, IN_EMBED_NORM = 1, IN_PLAIN = 2, IN_SWIGLU = 3 };
// OUT_SWIGLU (producer-warp GEMV only): W is the packed gate|up matrix, N the
// ffn features, out[b][f] = silu(gate_f) * up_f
// OUT_QKV_ATTN (producer-warp GEMV, one sequence): W is the packed q|k|v
// matrix; OUT_STORE of the row, then the CTA that completes the last rows of
// a KV head's q, k and v runs that head's step attention (args a.at)
enum GemvOut { OUT_STORE = 0, OUT_RESID = 1, OUT_ARGMAX = 2, OUT_SWIGLU = 3, OUT_QKV_ATTN = 4 };

struct AttnDecArgs {
    const float *qkv;       // [B, (nq + 2 nkv) d] raw projections of the step's row
    const float *qn_w, *kn_w;
    float eps;
    const float2 *rope;     // [max_pos, d/2] (cos, sin)
    void *Kc, *Vc;          // this layer's pool [nkv][slots][d]
    int slots;
    float *o;               // [B, nq d]
    float *part;            // scratch [B][nkv][S][n_rep][d + 2]
    unsigned *counter;      // scratch [B][nkv], zero between launches
    SeqState *st;
    int nq, nkv, d;
    int B;                  // sequences (grid z)
    int append;             // 1: write the row's K/V at slot n_past first
    int min_chunk;          // step mode: keys per split at least (0: attn_step_min_chunk(B))
    // plain mode (no state, no norm/RoPE/append): q already normed and roped
    const float *q_plain;   // [B, nq, d]
    const int32_t *kv_off;  // [B] first slot of each sequence
    const int32_t *kv_len;  // [B] visible keys (rows with len <= 0 or out of range are skipped)
    __nv_bfloat16 *o_bf16;  // optional bf16 copy of o (input of the tensor-core O projection)
    __nv_bfloat16 *o_bf16_lo;  // with o_bf16: the bf16 rounding residual (may be null)

};

struct GemvArgs {
    const void *W;          // [N, K] weights (bf16 or f32; e4m3 codes when wscale is set)
    const float *wscale;    // [N] scale of each e4m3 row (null: W holds bf16 or f32 values)
    int N, K;
    const float *in;        // [B, K] activations (IN_NORM, IN_PLAIN); [B, 2*ffn] gate|up (IN_SWIGLU)
    const float *norm_w;    // [K] RMSNorm weight (IN_NORM, IN_EMBED_NORM)
    const void *embed;      // [V, K] embedding table (IN_EMBED_NORM)
    float *x_resid;         // [B, K] residual written from the embedding row (IN_EMBED_NORM)
    float *out;             // [B, N] (STORE / RESID: in-place add; ARGMAX: logits, may be null)
    float eps;
    int ffn;                // IN_SWIGLU
    SeqState *st;
    int B;
    // OUT_ARGMAX
    float *part_val;
    int *part_idx;
    unsigned *counter;
    int32_t *out_ids;       // [B, out_ids_cap]
    int out_ids_cap;
    // the weights of the kernel that runs next ([pf_N, pf_K] bf16, may be null):
    // each CTA pulls up to pf_bytes of its share of the rows into L2 once its
    // own rows are in flight, so HBM keeps streaming across the launch boundary
    const void *pf;
    int pf_N, pf_K, pf_bytes;
    int pf_wb;              // bytes per weight of the next kernel's rows (0: 2, bf16)
    int pre_bulk;           // ring chunks copied before the dependency wait (0: the whole first fill)
    // KV of this layer pulled into L2 for the attention that follows (may be null)
    const void *kvp_K, *kvp_V;
    int kvp_slots, kvp_nkv, kvp_row_bytes;
    // OUT_QKV_ATTN: the step attention of the row (at.qkv = out; at.counter
    // holds one completed-row count per KV head, zero between launches)
    AttnDecArgs at;
    float at_scale;
    // filled in by launch_gemv: shared-memory slots per warp, units per CTA
    int n_ring;
    int max_units;
};

struct GemvPlan {
    int n_ring, max_units;
    size_t smem;
    bool ok;
};
GemvPlan gemv_plan(int K, bool w_bf16, int nb, int N, int grid_x);
// tuning knobs (process-wide): GEMV implementation for bf16 weights (1
// registers, 4 producer-warp stream; SPEECH_DECODER_GEMV=ldg|stream) and the
// stream GEMV's ring size
void gemv_set_impl(int impl);
// re-read SPEECH_DECODER_GEMV and SPEECH_DECODER_GEMV_SLOTS (each decoder creation)
void gemv_reload_env();
int gemv_impl();


// Batched-step helpers (rows of several sequences through the tensor-core GEMM):
// x[b] = embed[cur_tok[b]] for live rows; row argmax of logits [B, V] that
// advances the greedy state exactly as the GEMV head does.
void launch_embed_rows(const void *embed, bool w_bf16, SeqState *st, float *x, int B, int H, cudaStream_t s);
void launch_argmax_rows(const float *logits, int B, int V, SeqState *st, int32_t *out_ids, int out_ids_cap,
                        cudaStream_t s);

void launch_gemv(int in_mode, int out_mode, bool w_bf16, const GemvArgs &a, int grid_x,
                 cudaStream_t s);
void launch_attn_decode(bool kv_f16, const AttnDecArgs &a, int splits, cudaStream_t s);
// plain-mode launch over caller buffers; a.part/a.counter are the scratch
void launch_attn_decode_plain(bool kv_f16, const AttnDecArgs &a, int splits, cudaStream_t s);
// split-KV partitions for B sequences and the scratch bytes they need
int attn_decode_splits(int B, int nkv, int num_sms);
size_t attn_decode_part_floats(int B, int nq, int nkv, int d, int splits);

// Standalone plain-mode attention over caller buffers (shared by the C entry
// points): checks shapes, zeroes the counters in `scratch` and launches.
// scratch = [partials (256-aligned)][B * nkv counters].
size_t attn_op_scratch_bytes(int B, int nq, int nkv, int d, int num_sms);
bool attn_op_shape_ok(int B, int nq, int nkv, int d, int slots, int kv_dtype_f16_or_f32);
cudaError_t attn_op_launch(const float *q, const void *K, const void *V, bool kv_f16, int slots,
                           const int32_t *kv_off, const int32_t *kv_len, int B, int nq, int nkv, int d,
                           float *out, void *scratch, int num_sms, cudaStream_t s);
int gemv_grid(int N, int num_sms, int ctas_per_sm);
void init_gemv_kernels();
// shared-memory opt-in of the step attention (called once per process, with init_gemv_kernels)
void init_attn_kernels();
// producer-warp GEMV (bf16 weights, one CTA per SM): plan, launch (false: shape
// not supported), ring size override (0 = automatic)
GemvPlan gemv_stream_plan(int in_mode, int K, int nb, int N, int grid_x);
bool launch_gemv_stream(int in_mode, int out_mode, const GemvArgs &a, int grid_x, cudaStream_t s);
void gemv_stream_set_slots(int slots);
// the fused gate|up + SwiGLU GEMV fits (hidden K, ffn features)
bool gemv_stream_swiglu_ok(int K, int nb, int ffn, int grid_x);
// the q|k|v GEMV of one sequence with the step attention fused (f16 KV,
// head_dim 128, two query heads per KV head) fits this shape
bool gemv_stream_qkv_attn_ok(int K, int grid_x, int nq, int nkv, int d, bool kv_f16);
// longest context for which one CTA per KV head runs the step attention
// (longer ones take the split-KV attention kernel)
constexpr int kFusedAttnMaxCtx = 1024;
void init_gemv_stream_kernels();
// Step attention of at most kGroupB sequences as one thread-block cluster per
// (sequence, KV head) whose CTAs split the keys and combine through
// distributed shared memory (f16 KV, head_dim 128, 1, 2 or 4 query heads per
// KV head).  attn_cluster_splits: the cluster size for contexts of up to
// `capacity` keys, 0 when this kernel does not apply.
void init_attn_cluster();
int attn_cluster_splits(int capacity, int nq, int nkv, int d, bool kv_f16, int B);
cudaError_t launch_attn_cluster(const AttnDecArgs &a, int S, cudaStream_t s);
// Per-row e4m3 rounding of bf16 weights [rows, cols]: codes, power-of-two row
// scales and the rounded values in bf16 (`out` may equal `w`)
void launch_quantize_e4m3_rows(const void *w, size_t rows, int cols, uint8_t *codes, float *scales, void *out,
                               cudaStream_t s);
// GEMV CTAs per SM that suit the selected implementation
int gemv_default_ctas_per_sm();

// activation rows x K floats of one GEMV CTA must fit: kGroupB * K * 4 <= kGemvMaxSmem
constexpr int kGemvMaxSmem = 216 * 1024;
// split-KV partitions per (sequence, kv head)
constexpr int kAttnMaxSplits = 32;
// keys per split at least (short sequences run few splits); the step attention
// of at most kGroupB sequences (one CTA per SM, two key tiles in flight) takes
// twice as many, so that contexts up to 512 keys need no split combine
constexpr int kAttnMinChunk = 256;
__host__ __device__ constexpr int attn_step_min_chunk(int B) {
    return B > kGroupB ? kAttnMinChunk : 2 * kAttnMinChunk;
}

// Keys [0, len) of one (sequence, kv head) are cut into splits of `chunk` keys
// (at least min_chunk); splits [0, n_used) hold keys.
__host__ __device__ __forceinline__ void attn_split(int len, int S, int &chunk, int &n_used,
                                                    int min_chunk = kAttnMinChunk) {
    chunk = (len + S - 1) / S;
    chunk = chunk < min_chunk ? min_chunk : chunk;
    n_used = (len + chunk - 1) / chunk;
}

}  // namespace dec
