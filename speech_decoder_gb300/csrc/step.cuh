// Persistent decode step (one cooperative launch per greedy step).
#pragma once
#include "common.cuh"

namespace dec {

struct StepLayer {
    const __nv_bfloat16 *wqkv, *wo, *wgu, *wd;
    const float *attn_norm, *ffn_norm, *qn, *kn;
    __half *K, *V;
};

struct StepArgs {
    int L, H, F, nq, nkv, V, qkv_n, B, slots, splits;
    int ring_stages, union_floats;    // shared-memory plan, filled in by launch_step
    float eps, scale;
    const StepLayer *layers;          // device array [L]
    const __nv_bfloat16 *embed;
    const float *final_norm;
    const float2 *rope;
    float *x, *qkv, *o, *gu, *logits;
    float *attn_part;
    unsigned *attn_counter;
    float *am_val;
    int *am_idx;
    unsigned *am_counter;
    int32_t *out_ids;
    int out_ids_cap;
    SeqState *st;
    unsigned long long *bar;          // grid-barrier counter, zeroed before each launch
};

struct StepPlan {
    bool ok;
    int ring_stages, union_floats;
    size_t smem;
};
StepPlan step_plan(int H, int F, int nqd, int B);
// head_dim 128, at most 4 query heads per KV head, 1..4 sequences, one CTA per SM
bool step_supported(int head_dim, int n_rep, int H, int F, int nqd, int max_b);
// zeroes the barrier counter and launches the cooperative step kernel (grid = num_sms)
cudaError_t launch_step(StepArgs a, int num_sms, cudaStream_t s);

}  // namespace dec
