// Prefill-path kernel interfaces (all prompt rows of one or more sequences).
#pragma once
#include "gemm_tc.cuh"

namespace dec {

// rows of x (float32 [T, H]) -> RMSNorm(x) * w in bf16 (act_bf16; out_lo, if not
// null, receives the bf16 rounding residual) or float32
// fp16 copy of bf16 values (the prompt GEMMs' fp16 weights)
void launch_bf16_to_f16(const void *src, void *dst, size_t n, cudaStream_t s);
// RMSNorm of rows into one fp16 plane (operands of the fp16 prompt GEMMs)
void launch_rmsnorm_rows_f16(const float *x, const float *w, float eps, void *out, int T, int H, cudaStream_t s);
void launch_rmsnorm_rows(const float *x, const float *w, float eps, void *out, void *out_lo, bool act_bf16, int T,
                         int H, cudaStream_t s);

// n float32 values -> bf16 hi = bf16(v) and lo = bf16(v - hi)
void launch_split_planes(const float *x, void *hi, void *lo, size_t n, cudaStream_t s);

// C[M, N] (float32, row stride ldc) = or += A[M, K] . W[N, K]^T on CUDA cores
void launch_gemm_simt(const void *A, bool a_bf16, const void *W, bool w_bf16, float *C, int ldc,
                      int M, int N, int K, int epi, cudaStream_t s);

// h[t, f] = silu(gate) * up from the packed gate|up rows (blocks of 128 + 128);
// h_lo as for launch_rmsnorm_rows
void launch_swiglu(const float *gu, void *h, void *h_lo, bool act_bf16, int T, int F, cudaStream_t s);

struct RopeKvArgs {
    const float *qkv;          // [T, (nq + 2 nkv) d]
    const float *qn_w, *kn_w;
    float eps;
    const float2 *rope;        // [max_pos, d/2]
    const int32_t *row_pos;    // [T] position of each row in its sequence
    const int32_t *row_slot;   // [T] KV slot of each row in the pool
    void *q_out;               // [T, nq, d] (f16 or f32, same type as the cache)
    void *Kc, *Vc;             // this layer's pool [nkv][slots][d]
    int slots, T, nq, nkv, d;
    // optional (fp16 KV): V transposed, vt[(g d + e) vt_ld + row_vtcol[t]], for
    // the tensor-core attention
    void *vt;
    const int32_t *row_vtcol;
    int vt_ld;
};
void launch_qk_rope_kv(bool kv_f16, const RopeKvArgs &a, cudaStream_t s);

// Tensor-core causal attention of the prompt rows (fp16 KV, head_dim 128).
// tiles[i] = (first global row, first position in its sequence, rows <= 128,
// item); keys of item b sit at pool slots kv_off[b] + position and at V^T
// columns vt_col[b] + position (vt_col a multiple of 128).
struct AttnPrefillTcArgs {
    const void *q;             // [q_rows][nq][d] fp16 (normed, roped)
    const void *Kc;            // pool [nkv][slots][d] fp16
    const void *vt;            // [nkv d][vt_ld] fp16
    const int4 *tiles;
    const int32_t *kv_off, *vt_col;
    __nv_bfloat16 *o, *o_lo;   // [rows][nq d] two bf16 planes (o_lo may be null)
    int o_f16;                 // 1: o holds one fp16 plane instead (o_lo unused)
    int *err;                  // device error code if a bounded wait expires
    int q_rows, nq, nkv, slots, vt_ld;
    float scale;
};
void init_attn_prefill_tc();
// fp16 V of keys [0, n_keys) of one sequence (pool slots kv_off + j, head_dim
// 128) into the transposed scratch at columns vt_col0 + j
void launch_vt_from_pool(const void *V, void *vt, int vt_ld, int slots, int nkv, int kv_off, int n_keys, int vt_col0,
                         cudaStream_t s);
bool attn_prefill_tc_ok(int d, bool kv_f16);
cudaError_t launch_attn_prefill_tc(const AttnPrefillTcArgs &a, int n_tiles, cudaStream_t s);

struct AttnPrefillArgs {
    const void *q;             // [T, nq, d] roped queries (cache type)
    const void *Kc, *Vc;       // pool [nkv][slots][d]
    const int32_t *row_pos, *row_slot;
    void *o;                   // [T, nq d] (bf16 or f32)
    void *o_lo;                // bf16 rounding residual of o (bf16 output; may be null)
    int slots, T, nq, nkv, d;
};
void launch_attn_prefill_simt(bool kv_f16, bool out_bf16, const AttnPrefillArgs &a, cudaStream_t s);

// out[b] = x[idx[b]] for b < B (float32 rows of width H)
void launch_gather_rows(const float *x, const int32_t *idx, float *out, int B, int H, cudaStream_t s);

// x[t] = audio[t - prefix] inside the audio span, else embed[ids[..]] (prompt assembly)
void launch_assemble(const void *embed, bool w_bf16, const int32_t *ids, const float *audio,
                     float *x, int T, int n_audio, int prefix_len, int H, cudaStream_t s);

}  // namespace dec
