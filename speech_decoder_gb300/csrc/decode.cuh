// Decode-path kernel interfaces (one token per sequence per step).
#pragma once
#include "common.cuh"

namespace dec {

enum GemvIn { IN_NORM = 0, IN_EMBED_NORM = 1, IN_PLAIN = 2, IN_SWIGLU = 3 };
enum GemvOut { OUT_STORE = 0, OUT_RESID = 1, OUT_ARGMAX = 2 };

struct GemvArgs {
    const void *W;          // [N, K] weights (bf16 or f32)
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
};

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
};

void launch_gemv(int in_mode, int out_mode, bool w_bf16, const GemvArgs &a, int grid_x,
                 cudaStream_t s);
void launch_attn_decode(bool kv_f16, const AttnDecArgs &a, int splits, cudaStream_t s);
int gemv_grid(int N, int num_sms);
void init_gemv_kernels();

// activation rows x K floats of one GEMV CTA must fit: kGroupB * K * 4 <= kGemvMaxSmem
constexpr int kGemvMaxSmem = 200 * 1024;

}  // namespace dec
