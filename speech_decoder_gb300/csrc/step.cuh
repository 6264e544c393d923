// Persistent decode step of one sequence (one cooperative launch per step).
#pragma once
#include <cuda.h>

#include "common.cuh"

namespace dec {

struct StepLayer {
    const __nv_bfloat16 *wqkv, *wo, *wgu, *wd;
    const float *attn_norm, *ffn_norm, *qn, *kn;
    __half *K, *V;
};

struct StepArgs {
    int L, H, F, nq, nkv, V, qkv_n, slots;
    int S;                            // attention splits per KV head (kAttnKeys keys each at most)
    int ring_stages;                  // filled in by launch_step
    float eps, scale;
    const StepLayer *layers;          // device array [L]
    const CUtensorMap *kv_maps;       // device array [L][2]: K and V pool of each layer (64-dim x 32-key boxes)
    const __nv_bfloat16 *embed;
    const float *final_norm;
    const float2 *rope;
    float *x;                         // [H] residual stream
    float *qkv;                       // [qkv_n]
    float *h;                         // [F] silu(gate) * up
    float *part;                      // [nkv][S][n_rep][D + 2] attention partials (sum, then max and sum of exp)
    float *logits;                    // [V]
    float *am_val;                    // [grid] per-CTA argmax candidates
    int *am_idx;
    unsigned *am_counter;             // zero between launches
    int32_t *out_ids;
    int out_ids_cap;
    SeqState *st;
    unsigned long long *bar;          // grid-barrier counter, zeroed before each launch
};

constexpr int kAttnKeys = 128;        // keys of one attention item of the step kernel

struct StepPlan {
    bool ok;
    int ring_stages;
    size_t smem;
};
StepPlan step_plan(int H, int F, int nqd);
// one sequence, bf16 weights, f16 KV, head_dim 128, 1, 2 or 4 query heads per
// KV head, n_kv_heads * ceil(max_ctx / kAttnKeys) attention items at most one
// per SM
bool step_supported(int head_dim, int n_rep, int nkv, int H, int F, int max_ctx, int num_sms);
int step_splits(int max_ctx);
// the K/V pool tensor maps of one layer ([nkv * slots][128] f16, 64 x 32 boxes)
bool step_kv_maps(CUtensorMap *k_map, CUtensorMap *v_map, const void *K, const void *V, int rows);
// zeroes the barrier counter and launches the cooperative step kernel (grid = num_sms)
cudaError_t launch_step(StepArgs a, int num_sms, cudaStream_t s);

}  // namespace dec
