// C ABI and runtime of the decoder: workspace layout, weight packing, the
// prefill sequence, the captured step graph, and the device-side greedy loop.
//
// Sources: qwen3_asr/decoder.cpp (transcribe-cpp-sys 0.2.0) build_prefill_graph,
// build_step_graph, build_*_batched; qwen3_asr/model.cpp run / run_batch
// (input-length gate, KV sizing, greedy loop, truncation, EOS strip).
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include "dec.h"
#include "decode.cuh"
#include "gemm_tc.cuh"
#include "prefill.cuh"
#include "step.cuh"

using namespace dec;

namespace {

struct DevLayer {
    void *wqkv = nullptr, *wo = nullptr, *wgu = nullptr, *wd = nullptr;
    // DEC_E4M3: the same matrices as e4m3 codes with per-row scales
    uint8_t *wqkv8 = nullptr, *wo8 = nullptr, *wgu8 = nullptr, *wd8 = nullptr;
    float *wqkv_s = nullptr, *wo_s = nullptr, *wgu_s = nullptr, *wd_s = nullptr;
    // fp16 copies of the (bf16) projection matrices for the prompt GEMMs' fp16 mode
    void *wqkv16 = nullptr, *wo16 = nullptr, *wgu16 = nullptr, *wd16 = nullptr;
    float *attn_norm = nullptr, *ffn_norm = nullptr, *qn = nullptr, *kn = nullptr;
    void *K = nullptr, *V = nullptr;
};

struct Bump {
    char *base;
    size_t off = 0;
    template <typename T> T *take(size_t count) {
        off = (off + 255) & ~size_t(255);
        T *p = base ? reinterpret_cast<T *>(base + off) : nullptr;
        off += count * sizeof(T);
        return p;
    }
};

constexpr int kGenChunk = 16;     // steps per captured generate graph
constexpr size_t kTcScratchFloats = size_t(12) << 20;   // 48 MB of split-K partial tiles

}  // namespace

struct dec_handle {
    dec_hparams hp{};
    cudaStream_t stream = nullptr;
    int num_sms = 0;
    bool w_bf16 = true, kv_f16 = true, use_tc = true;
    bool w_e4m3 = false;            // DEC_E4M3: bf16 weights rounded per row to e4m3; codes for the step GEMVs
    size_t slots = 0;
    // weights
    void *embed = nullptr;
    uint8_t *embed8 = nullptr;      // DEC_E4M3: the lm_head as e4m3 codes
    float *embed_s = nullptr;
    float *final_norm = nullptr;
    std::vector<DevLayer> L;
    float2 *rope = nullptr;
    // prefill activations
    float *x = nullptr, *qkv = nullptr, *gu = nullptr;
    void *xn = nullptr, *q16 = nullptr, *attn_o = nullptr, *hbuf = nullptr;
    // bf16 builds: second planes (rounding residuals) of the tensor-core GEMM inputs
    void *xn_lo = nullptr, *attn_o_lo = nullptr, *hbuf_lo = nullptr;
    int32_t *row_pos = nullptr, *row_slot = nullptr, *last_row = nullptr, *ids_dev = nullptr;
    // tensor-core prompt attention: V^T of the layer's prompt rows [nkv d][vt_ld]
    // (fp16, zeroed once), each row's V^T column, query tiles, per-item offsets
    void *vt = nullptr;
    int vt_ld = 0;
    int32_t *row_vtcol = nullptr, *item_kv_off = nullptr, *item_vt_col = nullptr;
    int4 *attn_tiles = nullptr;
    bool tc_attn = false;
    bool f16_copies = false;        // the workspace holds fp16 copies of the projection matrices
    bool pf16 = false;              // prompt GEMMs in fp16 (one activation plane), else bf16 (two planes)
    // decode activations and scratch
    float *xd = nullptr, *qkvd = nullptr, *od = nullptr, *gud = nullptr, *logits = nullptr;
    float *attn_part = nullptr;
    unsigned *attn_counter = nullptr;
    float *am_val = nullptr;
    int *am_idx = nullptr;
    unsigned *am_counter = nullptr;
    bool no_fold_rope = false;      // SPEECH_DECODER_FOLD_ROPE=0: the prompt's rope kernel runs separately
    bool no_fold_norm = false;      // SPEECH_DECODER_FOLD_NORM=0: RMSNorms of prompt / batch rows run separately
    bool norm_ready = false;        // batched step: xn already holds the next RMSNorm (written by the down GEMM)
    int lm_grid = 0;
    int32_t *out_ids = nullptr;
    SeqState *st = nullptr;
    // dumps
    float *dump_inj = nullptr, *dump_b0 = nullptr, *dump_blast = nullptr, *dump_final = nullptr;
    bool dumps = false;
    int dump_T = 0, dump_B = 0;
    bool dump_b0_valid = false;
    // host state
    SeqState hst{};
    int n_seq = 0;
    bool prefilled = false;
    int chunk_pos = 0;              // chunked prefill: rows of sequence 0 already in the KV cache
    int logits_rows = 0;
    std::vector<int32_t> h_row_pos, h_row_slot, h_last_row, h_row_vtcol, h_item_kv_off, h_item_vt_col;
    std::vector<int4> h_tiles;
    // graphs
    cudaGraphExec_t step_exec = nullptr;
    int step_B = -1;
    size_t step_nodes = 0;
    cudaGraphExec_t gen_exec = nullptr;
    int gen_B = -1;
    size_t gen_nodes = 0;
    int64_t launches = 0;
    int64_t enq = 0;                // kernels enqueued by the current enqueue pass
    std::string err;
    cudaEvent_t ev[4] = {};
    float prefill_ms = 0.f, gen_ms = 0.f;
    bool own_stream = false;
    int gemv_ctas = 1;              // GEMV CTAs per SM
    float *tc_scratch = nullptr;    // split-K partial tiles of the tensor-core GEMM
    int pf_bytes = 0;               // L2 look-ahead of the decode GEMVs, bytes per CTA
    int pre_bulk = 0;               // ring chunks a GEMV copies before its dependency wait (0: all)
    // persistent step kernel
    StepLayer *step_layers = nullptr;
    CUtensorMap *kv_maps = nullptr;  // [L][2] K and V pool maps of the step kernel's attention tiles
    unsigned long long *step_bar = nullptr;
    bool use_step = false;
    bool attn_fuse = false;         // single-sequence q|k|v GEMV runs the step attention (short contexts)
    bool attn_split_kernel = false; // step attention always on the split-KV kernel (no cluster kernel)
    int lo_planes = -1;             // prompt projections with two bf16 activation planes (-1: by prompt length)
    int lo_planes_now = 15;         // the set of the prompt being run
    int attn_chunk = 0;             // keys per step-attention split at least (0: attn_step_min_chunk)
};

// ------------------------------------------------------------------ helpers
static dec_status fail(dec_handle *h, dec_status s, const std::string &msg) {
    if (h) h->err = msg;
    return s;
}

#define CK(call)                                                                                \
    do {                                                                                        \
        cudaError_t e_ = (call);                                                                \
        if (e_ != cudaSuccess)                                                                  \
            return fail(h, DEC_ERR_CUDA, std::string(#call " failed: ") + cudaGetErrorString(e_)); \
    } while (0)

// bytes per weight as passed in and kept for the prompt path (DEC_E4M3: bf16)
static size_t wsize(const dec_hparams &hp) { return hp.weight_dtype == DEC_F32 ? 4 : 2; }
static size_t kvsize(const dec_hparams &hp) { return hp.kv_dtype == DEC_F16 ? 2 : 4; }
static int qkv_rows(const dec_hparams &hp) { return (hp.n_heads + 2 * hp.n_kv_heads) * hp.head_dim; }

static std::string validate(const dec_hparams *hp) {
    if (!hp) return "hparams is NULL";
    const dec_hparams &p = *hp;
    if (p.n_layers < 1) return "n_layers must be >= 1";
    if (p.hidden < 256 || p.hidden % 256) return "hidden must be a positive multiple of 256";
    if (p.head_dim != 64 && p.head_dim != 128) return "head_dim must be 64 or 128";
    if (p.n_kv_heads < 1 || p.n_heads < 1 || p.n_heads % p.n_kv_heads) return "n_heads must be a multiple of n_kv_heads";
    if (p.n_heads / p.n_kv_heads > 8) return "at most 8 query heads per KV head";
    if ((p.n_heads * p.head_dim) % 256) return "n_heads*head_dim must be a multiple of 256";
    if (p.ffn < 128 || p.ffn % 128) return "ffn must be a positive multiple of 128";
    if (p.vocab < 1) return "vocab must be >= 1";
    {
        // every projection of the step must fit the GEMV's shared-memory plan
        const int H = p.hidden, F = p.ffn, nqd = p.n_heads * p.head_dim;
        const int qkv = (p.n_heads + 2 * p.n_kv_heads) * p.head_dim;
        const int shapes[5][2] = {{qkv, H}, {H, nqd}, {2 * F, H}, {H, F}, {p.vocab, H}};
        for (auto &nk : shapes)
            if (!gemv_plan(nk[1], p.weight_dtype != DEC_F32, std::min(p.max_batch, kGroupB), nk[0], 152).ok)
                return "projection too large for the decode GEMV (hidden, ffn, n_heads*head_dim <= 6144)";
    }
    if (!(p.rms_eps >= 0.f) || !(p.rope_theta > 0.f)) return "rms_eps must be >= 0 and rope_theta > 0";
    if (p.max_batch < 1 || p.max_batch > kMaxBatch) return "max_batch must be in [1, 64]";
    if (p.max_new < 1) return "max_new must be >= 1";
    if (p.max_ctx < 2 || p.max_ctx <= p.max_new) return "max_ctx must exceed max_new";
    if (p.max_tokens < 1) return "max_tokens must be >= 1";
    if (p.eos_id < -1 || p.eos_id >= p.vocab) return "eos_id must be -1 or a vocabulary id";
    const bool ok = ((p.weight_dtype == DEC_BF16 || p.weight_dtype == DEC_E4M3) && p.kv_dtype == DEC_F16) ||
                    (p.weight_dtype == DEC_F32 && p.kv_dtype == DEC_F32);
    if (!ok) return "supported formats: bf16 or e4m3 weights with f16 KV, or f32 weights with f32 KV";
    return "";
}

// Keys per split of the step attention at least: attn_step_min_chunk(B), or
// SPEECH_DECODER_ATTN_CHUNK.
static int attn_min_chunk(const dec_handle *h, int B) {
    return h->attn_chunk > 0 ? h->attn_chunk : attn_step_min_chunk(B);
}

// Split-KV partitions of the step attention: a split holds at least
// attn_min_chunk keys, so more splits than the longest context can fill would
// only launch CTAs that exit at once (the step graph is captured once, so the
// bound is the context capacity, not the current length).
static int splits_for(const dec_handle *h, int B) {
    const int mc = attn_min_chunk(h, B);
    const int by_ctx = (h->hp.max_ctx + mc - 1) / mc;
    return std::max(1, std::min(attn_decode_splits(B, h->hp.n_kv_heads, h->num_sms), by_ctx));
}

static int gemv_ctas_per_sm() {
    const char *c = std::getenv("SPEECH_DECODER_GEMV_CTAS_PER_SM");
    return c ? std::max(1, std::min(4, std::atoi(c))) : gemv_default_ctas_per_sm();
}

// Assign every device buffer from the bump allocator (base == nullptr: size only).
static size_t plan(dec_handle *h, const dec_hparams &hp, char *base, int num_sms) {
    Bump b{base};
    gemv_reload_env();
    h->gemv_ctas = gemv_ctas_per_sm();
    {
        const char *c = std::getenv("SPEECH_DECODER_GEMV_PF_KB");
        h->pf_bytes = (c ? std::max(0, std::min(4096, std::atoi(c))) : 64) * 1024;
        const char *pf = std::getenv("SPEECH_DECODER_PROMPT_F16");
        h->f16_copies = !(pf && pf[0] == '0') && hp.weight_dtype != DEC_F32 && hp.hidden % 128 == 0 &&
                        hp.ffn % 128 == 0 && (hp.n_heads * hp.head_dim) % 128 == 0;
        const char *fn = std::getenv("SPEECH_DECODER_FOLD_NORM");
        h->no_fold_norm = fn && fn[0] == '0';
        const char *fr = std::getenv("SPEECH_DECODER_FOLD_ROPE");
        h->no_fold_rope = fr && fr[0] == '0';
        const char *pb = std::getenv("SPEECH_DECODER_GEMV_PRE");
        h->pre_bulk = pb ? std::max(0, std::min(64, std::atoi(pb))) : 8;
    }
    const size_t ws = wsize(hp), kvs = kvsize(hp), as = ws;   // activations use the weight format
    const size_t H = hp.hidden, d = hp.head_dim, nq = hp.n_heads, nkv = hp.n_kv_heads, F = hp.ffn;
    const size_t V = hp.vocab, Tm = hp.max_tokens, Bm = hp.max_batch;
    const size_t slots = (size_t)hp.max_batch * hp.max_ctx;
    h->slots = slots;
    const bool e4m3 = hp.weight_dtype == DEC_E4M3;
    h->embed = b.take<char>(V * H * ws);
    if (e4m3) {
        h->embed8 = b.take<uint8_t>(V * H);
        h->embed_s = b.take<float>(V);
    }
    h->final_norm = b.take<float>(H);
    h->L.assign(hp.n_layers, DevLayer{});
    for (auto &l : h->L) {
        l.wqkv = b.take<char>((size_t)qkv_rows(hp) * H * ws);
        l.wo = b.take<char>(H * nq * d * ws);
        l.wgu = b.take<char>(2 * F * H * ws);
        l.wd = b.take<char>(H * F * ws);
        if (h->f16_copies) {
            l.wqkv16 = b.take<char>((size_t)qkv_rows(hp) * H * 2);
            l.wo16 = b.take<char>(H * nq * d * 2);
            l.wgu16 = b.take<char>(2 * F * H * 2);
            l.wd16 = b.take<char>(H * F * 2);
        }
        if (e4m3) {
            l.wqkv8 = b.take<uint8_t>((size_t)qkv_rows(hp) * H);
            l.wo8 = b.take<uint8_t>(H * nq * d);
            l.wgu8 = b.take<uint8_t>(2 * F * H);
            l.wd8 = b.take<uint8_t>(H * F);
            l.wqkv_s = b.take<float>(qkv_rows(hp));
            l.wo_s = b.take<float>(H);
            l.wgu_s = b.take<float>(2 * F);
            l.wd_s = b.take<float>(H);
        }
        l.attn_norm = b.take<float>(H);
        l.ffn_norm = b.take<float>(H);
        l.qn = b.take<float>(d);
        l.kn = b.take<float>(d);
        l.K = b.take<char>(nkv * slots * d * kvs);
        l.V = b.take<char>(nkv * slots * d * kvs);
    }
    h->rope = b.take<float2>((size_t)hp.max_ctx * (d / 2));
    h->x = b.take<float>(Tm * H);
    const size_t Ta = std::max(Tm, Bm);                   // rows of the GEMM inputs (prompt rows or step rows)
    const size_t lo = as == 2 ? 1 : 0;
    h->xn = b.take<char>(Ta * std::max(H, F) * as);
    h->xn_lo = lo ? b.take<char>(Ta * std::max(H, F) * as) : nullptr;
    h->qkv = b.take<float>(Tm * qkv_rows(hp));
    h->q16 = b.take<char>(Tm * nq * d * kvs);
    h->attn_o = b.take<char>(Ta * nq * d * as);
    h->attn_o_lo = lo ? b.take<char>(Ta * nq * d * as) : nullptr;
    h->gu = b.take<float>(Tm * 2 * F);
    h->hbuf = b.take<char>(Ta * F * as);
    h->hbuf_lo = lo ? b.take<char>(Ta * F * as) : nullptr;
    h->row_pos = b.take<int32_t>(Tm);
    h->row_slot = b.take<int32_t>(Tm);
    h->last_row = b.take<int32_t>(Bm);
    // items start at multiples of 128 columns of V^T
    h->vt_ld = (int)(((std::max(Tm + 128 * Bm, (size_t)hp.max_ctx + 128)) + 127) / 128 * 128);
    h->vt = kvs == 2 && d == 128 ? b.take<char>(nkv * d * (size_t)h->vt_ld * 2) : nullptr;
    h->row_vtcol = b.take<int32_t>(Tm);
    h->item_kv_off = b.take<int32_t>(Bm);
    h->item_vt_col = b.take<int32_t>(Bm);
    h->attn_tiles = b.take<int4>(Tm / 128 + Bm + 1);
    h->ids_dev = b.take<int32_t>(Tm);
    h->xd = b.take<float>(Bm * H);
    h->qkvd = b.take<float>(Bm * qkv_rows(hp));
    h->od = b.take<float>(Bm * nq * d);
    h->gud = b.take<float>(Bm * 2 * F);
    h->logits = b.take<float>(Bm * V);
    h->attn_part = b.take<float>(Bm * nkv * kAttnMaxSplits * (nq / nkv) * (d + 2));
    h->attn_counter = b.take<unsigned>(Bm * nkv);
    h->lm_grid = gemv_grid((int)V, num_sms, h->gemv_ctas);
    h->am_val = b.take<float>(Bm * h->lm_grid);
    h->am_idx = b.take<int>(Bm * h->lm_grid);
    h->am_counter = b.take<unsigned>(64);
    h->out_ids = b.take<int32_t>(Bm * hp.max_new);
    h->st = b.take<SeqState>(1);
    h->tc_scratch = b.take<float>(kTcScratchFloats);
    h->step_layers = b.take<StepLayer>(hp.n_layers);
    h->kv_maps = b.take<CUtensorMap>(2 * (size_t)hp.n_layers);
    h->step_bar = b.take<unsigned long long>(1);
    h->dump_inj = b.take<float>(Tm * H);
    h->dump_b0 = b.take<float>(Tm * H);
    h->dump_blast = b.take<float>(Bm * H);
    h->dump_final = b.take<float>(Bm * H);
    return b.off + 256;
}

// ------------------------------------------------------------------ enqueue passes
static int *dev_error(dec_handle *h) { return &h->st->error; }

// Prompt-row projection C[M, N] (=|+=) A[M, K] W[N, K]^T: tcgen05 for bf16
// weights, CUDA cores for the fp32 debug build.
// A_lo: the second bf16 plane of A (bf16 builds), read by the tensor-core path.
// f16: W and A are fp16 (the prompt GEMMs' fp16 mode: A_lo unused; the
// shapes it is enabled for always plan on the tensor cores)
static void gemm(dec_handle *h, const void *A, const void *A_lo, const void *W, float *C, int ldc, int M, int N, int K,
                 int epi, bool f16 = false) {
    // long prompts: 256 weight rows per CTA share each activation tile
    const int groups = M > 256 && N % 256 == 0 ? 2 : 1;
    if (f16 || (h->use_tc && h->w_bf16 &&
                gemm_tc_plan(M, N, K, groups, h->num_sms, kTcScratchFloats, 0, A_lo ? 2 : 1).ok))
        launch_gemm_tc(A, A_lo, M, W, N, K, groups, epi, C, ldc, nullptr, nullptr, 0, h->tc_scratch, kTcScratchFloats,
                       dev_error(h), h->num_sms, h->stream, 0, nullptr, f16);   // a launch error surfaces at the end
    else
        launch_gemm_simt(A, h->w_bf16, W, h->w_bf16, C, ldc, M, N, K, epi, h->stream);
    h->enq++;
}

// A residual projection (o, down) of M rows whose split-K reduction also
// writes RMSNorm(C) * norm_w into the xn planes for the next projection.
// False (nothing launched) where that does not apply: then the caller runs
// gemm() and the RMSNorm kernel.
static bool gemm_resid_norm(dec_handle *h, const void *A, const void *A_lo, const void *W, float *C, int M, int N,
                            int K, const float *norm_w, bool f16 = false) {
    if (!h->use_tc || !h->w_bf16 || h->no_fold_norm || !norm_w) return false;
    const cudaError_t e = launch_gemm_tc_resid_norm(A, A_lo, M, W, N, K, C, N, norm_w, h->hp.rms_eps, h->xn, h->xn_lo,
                                                    h->tc_scratch, kTcScratchFloats, dev_error(h), h->num_sms,
                                                    h->stream, f16);
    if (e == cudaErrorNotSupported) return false;
    h->enq += 2;                                       // any launch error surfaces at the end of the pass
    return true;
}

// The second activation plane of a prompt projection, or null where the
// projection takes one bf16 plane (bit of h->lo_planes: 1 q|k|v, 2 o,
// 4 gate|up, 8 down).
static const void *lo_plane(const dec_handle *h, int bit, const void *lo) {
    return !h->pf16 && (h->lo_planes_now & bit) ? lo : nullptr;
}

// Projections that take the second plane in a prompt of `rows` rows: all of
// them for short prompts (bound by the weight bytes, where the second plane
// costs little), q|k|v, o and down for long ones (bound by the tensor pipe;
// the gate|up input, half of the block's FLOPs, in one plane).  The logits
// stay within about 1.4e-2 of the oracle's largest magnitude on the 1.7B
// shape at 8015 rows, and 2.4e-3 at 152 rows.
static int prompt_planes(const dec_handle *h, int rows) {
    if (h->lo_planes >= 0) return h->lo_planes;
    return rows >= 1024 ? (1 | 2 | 8) : 15;
}

// Gate|up projection and SwiGLU into h->hbuf (and its second plane).
static void gemm_swiglu(dec_handle *h, const void *A, const void *A_lo, const void *Wgu, int M, int F, int K,
                        bool f16 = false) {
    if (f16 || (h->use_tc && h->w_bf16 &&
                gemm_tc_plan(M, 2 * F, K, 2, h->num_sms, kTcScratchFloats, 0, A_lo ? 2 : 1).ok)) {
        launch_gemm_tc(A, A_lo, M, Wgu, 2 * F, K, 2, EPI_SWIGLU_BF16, nullptr, 0, h->hbuf, h->hbuf_lo, F,
                       h->tc_scratch, kTcScratchFloats, dev_error(h), h->num_sms, h->stream, 0, nullptr, f16);
        h->enq++;
    } else {
        launch_gemm_simt(A, h->w_bf16, Wgu, h->w_bf16, h->gu, 2 * F, M, 2 * F, K, EPI_STORE_F32, h->stream);
        launch_swiglu(h->gu, h->hbuf, h->hbuf_lo, h->w_bf16, M, F, h->stream);
        h->enq += 2;
    }
}

// Batched step rows go through the tensor-core GEMM once there are more
// sequences than one GEMV CTA keeps in shared memory.
static bool batched_path(const dec_handle *h, int B) {
    return B > kGroupB && h->use_tc && h->w_bf16 && gemm_tc_ready();
}

static void enqueue_decode_layer_tc(dec_handle *h, int l, int B, bool from_embed) {
    const dec_hparams &hp = h->hp;
    const DevLayer &L = h->L[l];
    const int H = hp.hidden, F = hp.ffn, nqd = hp.n_heads * hp.head_dim;
    cudaStream_t s = h->stream;
    if (from_embed && l == 0) {
        launch_embed_rows(h->embed, h->w_bf16, h->st, h->xd, B, H, s);
        h->enq++;
    }
    if (!(h->norm_ready && !(from_embed && l == 0))) {
        launch_rmsnorm_rows(h->xd, L.attn_norm, hp.rms_eps, h->xn, h->xn_lo, true, B, H, s);
        h->enq++;
    }
    h->norm_ready = false;
    gemm(h, h->xn, h->xn_lo, L.wqkv, h->qkvd, qkv_rows(hp), B, qkv_rows(hp), H, EPI_STORE_F32);

    AttnDecArgs a{};
    a.qkv = h->qkvd;
    a.qn_w = L.qn;
    a.kn_w = L.kn;
    a.eps = hp.rms_eps;
    a.rope = h->rope;
    a.Kc = L.K;
    a.Vc = L.V;
    a.slots = (int)h->slots;
    a.o = h->od;
    a.o_bf16 = static_cast<__nv_bfloat16 *>(h->attn_o);
    a.o_bf16_lo = static_cast<__nv_bfloat16 *>(h->attn_o_lo);
    a.part = h->attn_part;
    a.counter = h->attn_counter;
    a.st = h->st;
    a.nq = hp.n_heads;
    a.nkv = hp.n_kv_heads;
    a.d = hp.head_dim;
    a.B = B;
    a.append = 1;
    a.min_chunk = attn_min_chunk(h, B);
    launch_attn_decode(h->kv_f16, a, splits_for(h, B), s);
    h->enq++;
    if (!gemm_resid_norm(h, h->attn_o, h->attn_o_lo, L.wo, h->xd, B, H, nqd, L.ffn_norm)) {
        gemm(h, h->attn_o, h->attn_o_lo, L.wo, h->xd, H, B, H, nqd, EPI_RESID_F32);
        launch_rmsnorm_rows(h->xd, L.ffn_norm, hp.rms_eps, h->xn, h->xn_lo, true, B, H, s);
        h->enq++;
    }
    gemm_swiglu(h, h->xn, h->xn_lo, L.wgu, B, F, H);
    // the next layer's (or the head's) RMSNorm in the down projection's reduction
    const float *next_norm = l + 1 < hp.n_layers ? h->L[l + 1].attn_norm : h->final_norm;
    if (gemm_resid_norm(h, h->hbuf, h->hbuf_lo, L.wd, h->xd, B, H, F, next_norm)) h->norm_ready = true;
    else gemm(h, h->hbuf, h->hbuf_lo, L.wd, h->xd, H, B, H, F, EPI_RESID_F32);
}

// The matrix one step GEMV streams: e4m3 codes and row scales when the handle
// holds them and the step has one sequence (the GEMV's e4m3 form), else the
// bf16 (or f32) values.
struct WSrc {
    const void *W;
    const float *scale;
};
static bool e4m3_step(const dec_handle *h, int B) { return h->w_e4m3 && B == 1 && gemv_impl() == 4; }
static WSrc wsrc(const dec_handle *h, int B, const void *w, const uint8_t *codes, const float *scales) {
    return e4m3_step(h, B) ? WSrc{codes, scales} : WSrc{w, nullptr};
}
static double wbytes(const dec_handle *h, int B) { return e4m3_step(h, B) ? 1.0 : (double)wsize(h->hp); }

// The GEMV that runs next streams W [N, K]: let this one pull its first rows into L2.
static void set_prefetch(const dec_handle *h, GemvArgs &g, WSrc W, int N, int K) {
    g.pre_bulk = h->pre_bulk;
    if (!h->w_bf16 || h->pf_bytes <= 0) return;
    g.pf = W.W;
    g.pf_N = N;
    g.pf_K = K;
    g.pf_bytes = h->pf_bytes;
    g.pf_wb = W.scale ? 1 : 2;
}

// Step attention of layer l over the q|k|v rows in qkvd (K/V appended at n_past).
static AttnDecArgs step_attn_args(const dec_handle *h, int l, int B) {
    const dec_hparams &hp = h->hp;
    const DevLayer &L = h->L[l];
    AttnDecArgs a{};
    a.qkv = h->qkvd;
    a.qn_w = L.qn;
    a.kn_w = L.kn;
    a.eps = hp.rms_eps;
    a.rope = h->rope;
    a.Kc = L.K;
    a.Vc = L.V;
    a.slots = (int)h->slots;
    a.o = h->od;
    a.part = h->attn_part;
    a.counter = h->attn_counter;
    a.st = h->st;
    a.nq = hp.n_heads;
    a.nkv = hp.n_kv_heads;
    a.d = hp.head_dim;
    a.B = B;
    a.append = 1;
    a.min_chunk = attn_min_chunk(h, B);
    return a;
}

// Option (SPEECH_DECODER_STEP_ATTN=fused): a single sequence with a context
// capacity of at most kFusedAttnMaxCtx keys has the q|k|v GEMV finish each KV
// head's attention (one CTA per head, all keys) and no separate attention launch.
static bool qkv_attn_fused(const dec_handle *h, int B) {
    const dec_hparams &hp = h->hp;
    return B == 1 && h->attn_fuse && h->w_bf16 && !h->w_e4m3 && h->kv_f16 && gemv_impl() == 4 &&
           hp.max_ctx <= kFusedAttnMaxCtx &&
           gemv_stream_qkv_attn_ok(hp.hidden, gemv_grid(qkv_rows(hp), h->num_sms, h->gemv_ctas), hp.n_heads,
                                   hp.n_kv_heads, hp.head_dim, h->kv_f16);
}

// The decode step's launches of one block (one row per sequence).  Each
// projection helper returns the launch's algorithmic bytes (weights once, the
// activation rows in and out) for the profiler.
static double layer_qkv(dec_handle *h, int l, int B, bool from_embed, bool with_attn) {
    const dec_hparams &hp = h->hp;
    const DevLayer &L = h->L[l];
    const int H = hp.hidden, nqd = hp.n_heads * hp.head_dim;
    GemvArgs g{};
    g.st = h->st;
    g.B = B;
    g.eps = hp.rms_eps;
    const WSrc w = wsrc(h, B, L.wqkv, L.wqkv8, L.wqkv_s);
    g.W = w.W;
    g.wscale = w.scale;
    g.N = qkv_rows(hp);
    g.K = H;
    g.in = h->xd;
    g.norm_w = L.attn_norm;
    g.embed = h->embed;
    g.x_resid = h->xd;
    g.out = h->qkvd;
    set_prefetch(h, g, wsrc(h, B, L.wo, L.wo8, L.wo_s), H, nqd);
    if (h->w_bf16 && h->pf_bytes > 0) {
        g.kvp_K = L.K;
        g.kvp_V = L.V;
        g.kvp_slots = (int)h->slots;
        g.kvp_nkv = hp.n_kv_heads;
        g.kvp_row_bytes = (int)(hp.head_dim * kvsize(hp));
    }
    const bool emb = from_embed && l == 0;
    if (with_attn) {
        g.at = step_attn_args(h, l, B);
        g.at_scale = (float)(1.0 / std::sqrt((double)hp.head_dim));
    }
    launch_gemv(emb ? IN_EMBED_NORM : IN_NORM, with_attn ? OUT_QKV_ATTN : OUT_STORE, h->w_bf16, g,
                gemv_grid(g.N, h->num_sms, h->gemv_ctas), h->stream);
    h->enq++;
    return (double)g.N * H * wbytes(h, B) + (double)B * (H + g.N) * 4.0;
}

// Cluster size of the step attention for B sequences (0: the split-KV kernel).
static int cluster_splits(const dec_handle *h, int B) {
    if (h->attn_split_kernel) return 0;
    const dec_hparams &hp = h->hp;
    return attn_cluster_splits(hp.max_ctx, hp.n_heads, hp.n_kv_heads, hp.head_dim, h->kv_f16, B);
}

static void layer_attn(dec_handle *h, int l, int B) {
    AttnDecArgs a = step_attn_args(h, l, B);
    const int S = cluster_splits(h, B);
    if (S > 0 && launch_attn_cluster(a, S, h->stream) == cudaSuccess) {
        h->enq++;
        return;
    }
    launch_attn_decode(h->kv_f16, a, splits_for(h, B), h->stream);
    h->enq++;
}

static double layer_o(dec_handle *h, int l, int B) {
    const dec_hparams &hp = h->hp;
    const DevLayer &L = h->L[l];
    const int H = hp.hidden, F = hp.ffn, nqd = hp.n_heads * hp.head_dim;
    GemvArgs o{};
    o.st = h->st;
    o.B = B;
    o.eps = hp.rms_eps;
    const WSrc w = wsrc(h, B, L.wo, L.wo8, L.wo_s);
    o.W = w.W;
    o.wscale = w.scale;
    o.N = H;
    o.K = nqd;
    o.in = h->od;
    o.out = h->xd;
    set_prefetch(h, o, wsrc(h, B, L.wgu, L.wgu8, L.wgu_s), 2 * F, H);
    launch_gemv(IN_PLAIN, OUT_RESID, h->w_bf16, o, gemv_grid(H, h->num_sms, h->gemv_ctas), h->stream);
    h->enq++;
    return (double)H * nqd * wbytes(h, B) + (double)B * (nqd + 2 * H) * 4.0;
}

// gate|up: with the producer-warp GEMV each gate row meets its up row in one
// stage and the kernel writes silu(gate) * up; otherwise gate|up is stored and
// the down projection's prologue applies SwiGLU
static bool swiglu_fused(const dec_handle *h, int B) {
    const int H = h->hp.hidden, F = h->hp.ffn;
    return h->w_bf16 && gemv_impl() == 4 &&
           gemv_stream_swiglu_ok(H, std::min(B, kGroupB), F, gemv_grid(2 * F, h->num_sms, h->gemv_ctas));
}

static double layer_gu(dec_handle *h, int l, int B) {
    const dec_hparams &hp = h->hp;
    const DevLayer &L = h->L[l];
    const int H = hp.hidden, F = hp.ffn;
    const bool fused = swiglu_fused(h, B);
    GemvArgs f1{};
    f1.st = h->st;
    f1.B = B;
    f1.eps = hp.rms_eps;
    f1.K = H;
    f1.in = h->xd;
    const WSrc w = wsrc(h, B, L.wgu, L.wgu8, L.wgu_s);
    f1.W = w.W;
    f1.wscale = w.scale;
    f1.N = fused ? F : 2 * F;
    f1.norm_w = L.ffn_norm;
    f1.out = h->gud;
    set_prefetch(h, f1, wsrc(h, B, L.wd, L.wd8, L.wd_s), H, F);
    launch_gemv(IN_NORM, fused ? OUT_SWIGLU : OUT_STORE, h->w_bf16, f1, gemv_grid(2 * F, h->num_sms, h->gemv_ctas),
                h->stream);
    h->enq++;
    return (double)2 * F * H * wbytes(h, B) + (double)B * (H + f1.N) * 4.0;
}

static double layer_down(dec_handle *h, int l, int B) {
    const dec_hparams &hp = h->hp;
    const DevLayer &L = h->L[l];
    const int H = hp.hidden, F = hp.ffn;
    const bool fused = swiglu_fused(h, B);
    GemvArgs f2{};
    f2.st = h->st;
    f2.B = B;
    const WSrc w = wsrc(h, B, L.wd, L.wd8, L.wd_s);
    f2.W = w.W;
    f2.wscale = w.scale;
    f2.N = H;
    f2.K = F;
    f2.in = h->gud;
    f2.ffn = F;
    f2.out = h->xd;
    if (l + 1 < hp.n_layers) {
        const DevLayer &N = h->L[l + 1];
        set_prefetch(h, f2, wsrc(h, B, N.wqkv, N.wqkv8, N.wqkv_s), qkv_rows(hp), H);
    } else {
        set_prefetch(h, f2, wsrc(h, B, h->embed, h->embed8, h->embed_s), hp.vocab, H);
    }
    launch_gemv(fused ? IN_PLAIN : IN_SWIGLU, OUT_RESID, h->w_bf16, f2, gemv_grid(H, h->num_sms, h->gemv_ctas),
                h->stream);
    h->enq++;
    return (double)H * F * wbytes(h, B) + (double)B * ((fused ? 1 : 2) * F + 2 * H) * 4.0;
}

static void enqueue_decode_layer(dec_handle *h, int l, int B, bool from_embed) {
    if (batched_path(h, B)) {
        enqueue_decode_layer_tc(h, l, B, from_embed);
        return;
    }
    const bool fused = qkv_attn_fused(h, B);
    layer_qkv(h, l, B, from_embed, fused);
    if (!fused) layer_attn(h, l, B);
    layer_o(h, l, B);
    layer_gu(h, l, B);
    layer_down(h, l, B);
}

static void enqueue_head(dec_handle *h, int B) {
    if (batched_path(h, B)) {
        const dec_hparams &hp = h->hp;
        if (!h->norm_ready) {
            launch_rmsnorm_rows(h->xd, h->final_norm, hp.rms_eps, h->xn, h->xn_lo, true, B, hp.hidden, h->stream);
            h->enq++;
        }
        h->norm_ready = false;
        gemm(h, h->xn, h->xn_lo, h->embed, h->logits, hp.vocab, B, hp.vocab, hp.hidden, EPI_STORE_F32);
        launch_argmax_rows(h->logits, B, hp.vocab, h->st, h->out_ids, hp.max_new, h->stream);
        h->enq++;
        return;
    }
    GemvArgs g{};
    g.st = h->st;
    g.B = B;
    g.eps = h->hp.rms_eps;
    const WSrc w = wsrc(h, B, h->embed, h->embed8, h->embed_s);
    g.W = w.W;
    g.wscale = w.scale;
    g.N = h->hp.vocab;
    g.K = h->hp.hidden;
    g.in = h->xd;
    g.norm_w = h->final_norm;
    g.out = h->logits;
    g.part_val = h->am_val;
    g.part_idx = h->am_idx;
    g.counter = h->am_counter;
    g.out_ids = h->out_ids;
    g.out_ids_cap = h->hp.max_new;
    set_prefetch(h, g, wsrc(h, B, h->L[0].wqkv, h->L[0].wqkv8, h->L[0].wqkv_s), qkv_rows(h->hp), h->hp.hidden);
    launch_gemv(IN_NORM, OUT_ARGMAX, h->w_bf16, g, h->lm_grid, h->stream);
    h->enq++;
}

static StepArgs step_args(dec_handle *h) {
    const dec_hparams &hp = h->hp;
    StepArgs a{};
    a.L = hp.n_layers;
    a.H = hp.hidden;
    a.F = hp.ffn;
    a.nq = hp.n_heads;
    a.nkv = hp.n_kv_heads;
    a.V = hp.vocab;
    a.qkv_n = qkv_rows(hp);
    a.slots = (int)h->slots;
    a.S = step_splits(hp.max_ctx);
    a.eps = hp.rms_eps;
    a.scale = (float)(1.0 / std::sqrt((double)hp.head_dim));
    a.layers = h->step_layers;
    a.kv_maps = h->kv_maps;
    a.embed = static_cast<const __nv_bfloat16 *>(h->embed);
    a.final_norm = h->final_norm;
    a.rope = h->rope;
    a.x = h->xd;
    a.qkv = h->qkvd;
    a.h = h->gud;
    a.part = h->attn_part;
    a.logits = h->logits;
    a.am_val = h->am_val;
    a.am_idx = h->am_idx;
    a.am_counter = h->am_counter;
    a.out_ids = h->out_ids;
    a.out_ids_cap = hp.max_new;
    a.st = h->st;
    a.bar = h->step_bar;
    return a;
}

static bool step_path(const dec_handle *h, int B) { return h->use_step && B == 1; }

static void enqueue_step(dec_handle *h, int B) {
    h->norm_ready = false;
    if (step_path(h, B)) {
        launch_step(step_args(h), h->num_sms, h->stream);
        h->enq++;
        return;
    }
    for (int l = 0; l < h->hp.n_layers; ++l) enqueue_decode_layer(h, l, B, true);
    enqueue_head(h, B);
}

static dec_status capture(dec_handle *h, int steps, int B, cudaGraphExec_t *exec, size_t *nodes) {
    if (*exec) {
        cudaGraphExecDestroy(*exec);
        *exec = nullptr;
    }
    cudaGraph_t graph = nullptr;
    CK(cudaStreamBeginCapture(h->stream, cudaStreamCaptureModeThreadLocal));
    for (int i = 0; i < steps; ++i) enqueue_step(h, B);
    CK(cudaStreamEndCapture(h->stream, &graph));
    size_t n = 0;
    CK(cudaGraphGetNodes(graph, nullptr, &n));
    cudaError_t e = cudaGraphInstantiate(exec, graph, 0);
    cudaGraphDestroy(graph);
    if (e != cudaSuccess) return fail(h, DEC_ERR_CUDA, std::string("graph instantiate: ") + cudaGetErrorString(e));
    *nodes = n;
    return DEC_OK;
}

static dec_status sync_state(dec_handle *h) {
    CK(cudaMemcpyAsync(&h->hst, h->st, sizeof(SeqState), cudaMemcpyDeviceToHost, h->stream));
    CK(cudaStreamSynchronize(h->stream));
    if (h->hst.error) return fail(h, DEC_ERR_DEVICE, "device reported error " + std::to_string(h->hst.error));
    return DEC_OK;
}

// ------------------------------------------------------------------ prefill
// Rows are already in h->x (sum T_b rows); cu has B + 1 offsets.
// Chunked prefill of sequence 0: its rows start at position p0 of a context
// that owns KV slots [0, max_ctx); a non-final chunk writes the KV of every
// block and stops (no head).
struct Chunk {
    bool on = false;
    int p0 = 0;
    bool final = true;
};

static dec_status prefill_rows(dec_handle *h, const int32_t *cu, int B, int32_t *first_tokens, Chunk ck = Chunk()) {
    const dec_hparams &hp = h->hp;
    const int total = cu[B];
    const int H = hp.hidden, F = hp.ffn, nqd = hp.n_heads * hp.head_dim;
    cudaStream_t s = h->stream;
    h->enq = 0;

    h->h_row_pos.resize(total);
    h->h_row_slot.resize(total);
    h->h_last_row.resize(B);
    h->h_row_vtcol.resize(total);
    h->h_item_kv_off.resize(B);
    h->h_item_vt_col.resize(B);
    h->h_tiles.clear();
    int vt_col = 0;
    SeqState &st = h->hst;
    std::memset(&st, 0, sizeof(st));
    int off = 0;
    const int p0 = ck.on ? ck.p0 : 0;        // position of the first row (B == 1 when chunked)
    for (int b = 0; b < B; ++b) {
        const int T = cu[b + 1] - cu[b];
        const int cap = ck.on ? hp.max_ctx : T + hp.max_new;
        for (int t = 0; t < T; ++t) {
            h->h_row_pos[cu[b] + t] = p0 + t;
            h->h_row_slot[cu[b] + t] = off + p0 + t;
            h->h_row_vtcol[cu[b] + t] = vt_col + p0 + t;
        }
        h->h_item_kv_off[b] = off;
        h->h_item_vt_col[b] = vt_col;
        for (int q0 = 0; q0 < T; q0 += 128)
            h->h_tiles.push_back(make_int4(cu[b] + q0, p0 + q0, std::min(128, T - q0), b));
        vt_col += (p0 + T + 127) / 128 * 128;
        h->h_last_row[b] = cu[b + 1] - 1;
        st.n_past[b] = p0 + T - 1;       // the head pass processes the last row
        st.kv_off[b] = off;
        st.kv_cap[b] = cap;
        st.active[b] = 1;
        off += cap;
    }
    st.max_new = hp.max_new;
    st.eos_id = hp.eos_id;
    st.n_seq = B;
    CK(cudaMemcpyAsync(h->row_pos, h->h_row_pos.data(), total * 4, cudaMemcpyHostToDevice, s));
    CK(cudaMemcpyAsync(h->row_slot, h->h_row_slot.data(), total * 4, cudaMemcpyHostToDevice, s));
    CK(cudaMemcpyAsync(h->last_row, h->h_last_row.data(), B * 4, cudaMemcpyHostToDevice, s));
    if (h->tc_attn) {
        // longest causal ranges first: the tail of the grid is short tiles
        std::stable_sort(h->h_tiles.begin(), h->h_tiles.end(),
                         [](const int4 &u, const int4 &v) { return u.y + u.z > v.y + v.z; });
        CK(cudaMemcpyAsync(h->row_vtcol, h->h_row_vtcol.data(), total * 4, cudaMemcpyHostToDevice, s));
        CK(cudaMemcpyAsync(h->item_kv_off, h->h_item_kv_off.data(), B * 4, cudaMemcpyHostToDevice, s));
        CK(cudaMemcpyAsync(h->item_vt_col, h->h_item_vt_col.data(), B * 4, cudaMemcpyHostToDevice, s));
        CK(cudaMemcpyAsync(h->attn_tiles, h->h_tiles.data(), h->h_tiles.size() * sizeof(int4),
                           cudaMemcpyHostToDevice, s));
    }
    CK(cudaMemcpyAsync(h->st, &st, sizeof(SeqState), cudaMemcpyHostToDevice, s));

    if (h->dumps) {
        CK(cudaMemcpyAsync(h->dump_inj, h->x, (size_t)total * H * 4, cudaMemcpyDeviceToDevice, s));
        h->dump_T = total;
        h->dump_B = B;
        h->dump_b0_valid = false;
    }
    h->lo_planes_now = prompt_planes(h, total);
    bool norm_ready = false;                       // xn holds this block's input norm (the down GEMM wrote it)
    const bool f16 = h->pf16;                      // prompt GEMMs in fp16 (one plane), else bf16 planes
    for (int l = 0; l < hp.n_layers; ++l) {
        const DevLayer &L = h->L[l];
        if (!norm_ready) {
            if (f16) launch_rmsnorm_rows_f16(h->x, L.attn_norm, hp.rms_eps, h->xn, total, H, s);
            else launch_rmsnorm_rows(h->x, L.attn_norm, hp.rms_eps, h->xn, h->xn_lo, h->w_bf16, total, H, s);
        }
        norm_ready = false;
        RopeKvArgs r{};
        r.qkv = h->qkv;
        r.qn_w = L.qn;
        r.kn_w = L.kn;
        r.eps = hp.rms_eps;
        r.rope = h->rope;
        r.row_pos = h->row_pos;
        r.row_slot = h->row_slot;
        r.q_out = h->q16;
        r.Kc = L.K;
        r.Vc = L.V;
        r.slots = (int)h->slots;
        r.T = total;
        r.nq = hp.n_heads;
        r.nkv = hp.n_kv_heads;
        r.d = hp.head_dim;
        if (h->tc_attn && l + 1 < hp.n_layers) {
            r.vt = h->vt;
            r.row_vtcol = h->row_vtcol;
            r.vt_ld = h->vt_ld;
            // a later chunk also attends to the keys of the earlier ones: their
            // V rows come back from the pool into the transposed scratch
            if (p0 > 0) {
                launch_vt_from_pool(L.V, h->vt, h->vt_ld, (int)h->slots, hp.n_kv_heads, 0, p0, 0, s);
                h->enq++;
            }
        }
        // q|k|v projection; where it runs split-K, the per-head Q/K norm, RoPE
        // and KV write happen in its reduction (no q|k|v round trip)
        if (!(h->use_tc && h->w_bf16 && h->kv_f16 && hp.head_dim == 128 && !h->no_fold_rope &&
              launch_gemm_tc_qkv_rope(h->xn, lo_plane(h, 1, h->xn_lo), total, f16 ? L.wqkv16 : L.wqkv, qkv_rows(hp),
                                      H, r, h->tc_scratch, kTcScratchFloats, dev_error(h), h->num_sms, s,
                                      f16) == cudaSuccess)) {
            gemm(h, h->xn, lo_plane(h, 1, h->xn_lo), f16 ? L.wqkv16 : L.wqkv, h->qkv, qkv_rows(hp), total,
                 qkv_rows(hp), H, EPI_STORE_F32, f16);
            launch_qk_rope_kv(h->kv_f16, r, s);
            h->enq++;
        } else {
            h->enq++;                                   // the GEMM and its reduction (gemm() counts one)
        }
        h->enq++;
        if (l + 1 == hp.n_layers && ck.on && !ck.final) break;   // KV of every block written; no head
        if (l + 1 < hp.n_layers) {
            AttnPrefillArgs a{};
            a.q = h->q16;
            a.Kc = L.K;
            a.Vc = L.V;
            a.row_pos = h->row_pos;
            a.row_slot = h->row_slot;
            a.o = h->attn_o;
            a.o_lo = h->attn_o_lo;
            a.slots = (int)h->slots;
            a.T = total;
            a.nq = hp.n_heads;
            a.nkv = hp.n_kv_heads;
            a.d = hp.head_dim;
            if (h->tc_attn) {
                AttnPrefillTcArgs t{};
                t.q = h->q16;
                t.Kc = L.K;
                t.vt = h->vt;
                t.tiles = h->attn_tiles;
                t.kv_off = h->item_kv_off;
                t.vt_col = h->item_vt_col;
                t.o = static_cast<__nv_bfloat16 *>(h->attn_o);
                t.o_lo = static_cast<__nv_bfloat16 *>(h->attn_o_lo);
                t.o_f16 = f16 ? 1 : 0;
                t.err = dev_error(h);
                t.q_rows = total;
                t.nq = hp.n_heads;
                t.nkv = hp.n_kv_heads;
                t.slots = (int)h->slots;
                t.vt_ld = h->vt_ld;
                t.scale = (float)(1.0 / std::sqrt((double)hp.head_dim));
                launch_attn_prefill_tc(t, (int)h->h_tiles.size(), s);
            } else {
                launch_attn_prefill_simt(h->kv_f16, h->w_bf16, a, s);
            }
            // residual projections whose split-K reduction also writes the next RMSNorm
            const void *wo = f16 ? L.wo16 : L.wo, *wgu = f16 ? L.wgu16 : L.wgu, *wd = f16 ? L.wd16 : L.wd;
            if (!gemm_resid_norm(h, h->attn_o, lo_plane(h, 2, h->attn_o_lo), wo, h->x, total, H, nqd, L.ffn_norm,
                                 f16)) {
                gemm(h, h->attn_o, lo_plane(h, 2, h->attn_o_lo), wo, h->x, H, total, H, nqd, EPI_RESID_F32, f16);
                if (f16) launch_rmsnorm_rows_f16(h->x, L.ffn_norm, hp.rms_eps, h->xn, total, H, s);
                else launch_rmsnorm_rows(h->x, L.ffn_norm, hp.rms_eps, h->xn, h->xn_lo, h->w_bf16, total, H, s);
                h->enq++;
            }
            gemm_swiglu(h, h->xn, lo_plane(h, 4, h->xn_lo), wgu, total, F, H, f16);
            if (gemm_resid_norm(h, h->hbuf, lo_plane(h, 8, h->hbuf_lo), wd, h->x, total, H, F, h->L[l + 1].attn_norm,
                                f16))
                norm_ready = true;
            else
                gemm(h, h->hbuf, lo_plane(h, 8, h->hbuf_lo), wd, h->x, H, total, H, F, EPI_RESID_F32, f16);
            h->enq++;
            if (h->dumps && l == 0) {
                CK(cudaMemcpyAsync(h->dump_b0, h->x, (size_t)total * H * 4, cudaMemcpyDeviceToDevice, s));
                h->dump_b0_valid = true;
            }
        } else {
            // slice_last: the last block's query side, FFN and head run on the
            // last row of each sequence only (decoder.cpp, build_prefill_graph)
            launch_gather_rows(h->x, h->last_row, h->xd, B, H, s);
            h->enq++;
            enqueue_decode_layer(h, l, B, false);
        }
    }
    if (ck.on && !ck.final) {
        CK(cudaGetLastError());
        h->launches += h->enq;
        dec_status rc = sync_state(h);
        if (rc != DEC_OK) return rc;
        h->prefilled = false;
        for (int b = 0; b < B; ++b) first_tokens[b] = -1;
        return DEC_OK;
    }
    if (h->dumps) {
        CK(cudaMemcpyAsync(h->dump_blast, h->xd, (size_t)B * H * 4, cudaMemcpyDeviceToDevice, s));
        launch_rmsnorm_rows(h->xd, h->final_norm, hp.rms_eps, h->dump_final, nullptr, false, B, H, s);
    }
    enqueue_head(h, B);
    CK(cudaGetLastError());
    h->launches += h->enq;
    dec_status rc = sync_state(h);
    if (rc != DEC_OK) return rc;
    h->n_seq = B;
    h->prefilled = true;
    h->logits_rows = B;
    for (int b = 0; b < B; ++b) first_tokens[b] = h->hst.cur_tok[b];
    return DEC_OK;
}

static dec_status check_lengths(dec_handle *h, const int32_t *cu, int B) {
    const dec_hparams &hp = h->hp;
    if (B < 1 || B > hp.max_batch) return fail(h, DEC_ERR_INVALID_ARG, "batch size out of range");
    if (cu[0] != 0) return fail(h, DEC_ERR_INVALID_ARG, "cu_seqlens[0] must be 0");
    for (int b = 0; b < B; ++b) {
        const int T = cu[b + 1] - cu[b];
        if (T < 1) return fail(h, DEC_ERR_INVALID_ARG, "every sequence needs at least one row");
        if (T + hp.max_new > hp.max_ctx)
            return fail(h, DEC_ERR_INPUT_TOO_LONG,
                        "prompt of " + std::to_string(T) + " rows + generation budget " +
                            std::to_string(hp.max_new) + " exceeds the context of " + std::to_string(hp.max_ctx));
    }
    if (cu[B] > hp.max_tokens)
        return fail(h, DEC_ERR_INPUT_TOO_LONG, "prompt rows exceed max_tokens");
    return DEC_OK;
}

static dec_status timed_prefill(dec_handle *h, const int32_t *cu, int B, int32_t *first, Chunk ck = Chunk()) {
    if (!ck.on) h->chunk_pos = 0;            // a whole-prompt prefill ends any chunked one
    cudaEventRecord(h->ev[0], h->stream);
    dec_status rc = prefill_rows(h, cu, B, first, ck);
    cudaEventRecord(h->ev[1], h->stream);
    cudaEventSynchronize(h->ev[1]);
    cudaEventElapsedTime(&h->prefill_ms, h->ev[0], h->ev[1]);
    return rc;
}

// ------------------------------------------------------------------ generate
static dec_status run_step_graph(dec_handle *h, int B) {
    if (h->step_B != B) {
        h->enq = 0;
        dec_status rc = capture(h, 1, B, &h->step_exec, &h->step_nodes);
        if (rc != DEC_OK) return rc;
        h->step_B = B;
    }
    CK(cudaGraphLaunch(h->step_exec, h->stream));
    h->launches += (int64_t)h->step_nodes;
    return DEC_OK;
}

static dec_status generate_core(dec_handle *h, int max_new) {
    const int B = h->n_seq;
    SeqState &st = h->hst;
    st.max_new = max_new;
    for (int b = 0; b < B; ++b) {
        if (!st.active[b]) continue;
        st.done[b] = (st.cur_tok[b] == st.eos_id) || st.gen[b] >= max_new || st.n_past[b] + 1 > st.kv_cap[b];
    }
    CK(cudaMemcpyAsync(h->st, &st, sizeof(SeqState), cudaMemcpyHostToDevice, h->stream));
    if (h->gen_B != B) {
        h->enq = 0;
        dec_status rc = capture(h, kGenChunk, B, &h->gen_exec, &h->gen_nodes);
        if (rc != DEC_OK) return rc;
        h->gen_B = B;
    }
    CK(cudaEventRecord(h->ev[2], h->stream));
    for (;;) {
        bool live = false;
        for (int b = 0; b < B; ++b) live |= st.active[b] && !st.done[b];
        if (!live) break;
        CK(cudaGraphLaunch(h->gen_exec, h->stream));
        h->launches += (int64_t)h->gen_nodes;
        dec_status rc = sync_state(h);
        if (rc != DEC_OK) return rc;
    }
    CK(cudaEventRecord(h->ev[3], h->stream));
    CK(cudaEventSynchronize(h->ev[3]));
    cudaEventElapsedTime(&h->gen_ms, h->ev[2], h->ev[3]);
    h->logits_rows = B;
    return DEC_OK;
}

// ================================================================== C ABI
extern "C" {

const char *dec_status_string(dec_status s) {
    switch (s) {
    case DEC_OK: return "DEC_OK";
    case DEC_ERR_INVALID_ARG: return "DEC_ERR_INVALID_ARG";
    case DEC_ERR_OOM: return "DEC_ERR_OOM";
    case DEC_ERR_INPUT_TOO_LONG: return "DEC_ERR_INPUT_TOO_LONG";
    case DEC_ERR_OUTPUT_TRUNCATED: return "DEC_ERR_OUTPUT_TRUNCATED";
    case DEC_ERR_CUDA: return "DEC_ERR_CUDA";
    case DEC_ERR_STATE: return "DEC_ERR_STATE";
    case DEC_ERR_DEVICE: return "DEC_ERR_DEVICE";
    }
    return "unknown";
}

const char *dec_last_error(const dec_handle *h) { return h ? h->err.c_str() : "null handle"; }

dec_status dec_workspace_size(const dec_hparams *hp, size_t *bytes) {
    if (!bytes) return DEC_ERR_INVALID_ARG;
    if (!validate(hp).empty()) return DEC_ERR_INVALID_ARG;
    dec_handle tmp;
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaGetLastError();
    *bytes = plan(&tmp, *hp, nullptr, sms);
    return DEC_OK;
}

static void to_f32_host(const void *src, bool bf16, size_t n, float *dst) {
    if (!bf16) {
        std::memcpy(dst, src, n * 4);
        return;
    }
    const uint16_t *s = static_cast<const uint16_t *>(src);
    for (size_t i = 0; i < n; ++i) {
        const uint32_t u = (uint32_t)s[i] << 16;
        std::memcpy(dst + i, &u, 4);
    }
}

dec_status dec_create(const dec_hparams *hp, const dec_weights *w, void *workspace, size_t ws_bytes,
                      void *stream, dec_handle **out) {
    if (!out) return DEC_ERR_INVALID_ARG;
    *out = nullptr;
    const std::string why = validate(hp);
    if (!why.empty()) return DEC_ERR_INVALID_ARG;
    if (!w || !w->embed || !w->final_norm || !w->layers || !workspace) return DEC_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) % 256) return DEC_ERR_INVALID_ARG;
    for (int l = 0; l < hp->n_layers; ++l) {
        const dec_layer_weights &L = w->layers[l];
        if (!L.attn_norm || !L.q || !L.k || !L.v || !L.o || !L.q_norm || !L.k_norm || !L.ffn_norm || !L.gate ||
            !L.up || !L.down)
            return DEC_ERR_INVALID_ARG;
    }
    dec_handle *h = new dec_handle();
    h->hp = *hp;
    h->stream = static_cast<cudaStream_t>(stream);
    if (!h->stream) {
        // the step loop is captured into CUDA graphs, which the legacy default stream cannot do
        if (cudaStreamCreateWithFlags(&h->stream, cudaStreamNonBlocking) != cudaSuccess) {
            delete h;
            return DEC_ERR_CUDA;
        }
        h->own_stream = true;
    }
    h->w_bf16 = hp->weight_dtype != DEC_F32;
    h->w_e4m3 = hp->weight_dtype == DEC_E4M3;
    h->kv_f16 = hp->kv_dtype == DEC_F16;
    const char *g = std::getenv("SPEECH_DECODER_GEMM");
    h->use_tc = !(g && std::strcmp(g, "simt") == 0);

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        delete h;
        return DEC_ERR_CUDA;
    }
    const size_t need = plan(h, *hp, nullptr, h->num_sms);
    if (ws_bytes < need) {
        delete h;
        return DEC_ERR_OOM;
    }
    plan(h, *hp, static_cast<char *>(workspace), h->num_sms);
    for (auto &e : h->ev) cudaEventCreate(&e);

    auto fail_create = [&](dec_status s) {
        dec_destroy(h);
        return s;
    };
#define CKC(call)                                   \
    do {                                            \
        if ((call) != cudaSuccess) return fail_create(DEC_ERR_CUDA); \
    } while (0)

    init_gemv_kernels();
    init_gemm_tc();
    init_attn_prefill_tc();
    cudaStream_t s = h->stream;
    const size_t ws = wsize(*hp), H = hp->hidden, F = hp->ffn, d = hp->head_dim;
    const size_t nq = hp->n_heads, nkv = hp->n_kv_heads;
    CKC(cudaMemcpyAsync(h->embed, w->embed, (size_t)hp->vocab * H * ws, cudaMemcpyHostToDevice, s));
    if (h->w_e4m3) {
        launch_quantize_e4m3_rows(h->embed, (size_t)hp->vocab, (int)H, h->embed8, h->embed_s, h->embed, s);
        CKC(cudaGetLastError());
    }
    std::vector<float> nbuf(std::max(H, d));
    std::vector<char> gu_host(2 * F * H * ws);
    auto put_norm = [&](float *dst, const void *src, size_t n) -> cudaError_t {
        to_f32_host(src, h->w_bf16, n, nbuf.data());
        cudaError_t e = cudaMemcpyAsync(dst, nbuf.data(), n * 4, cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        return e;
    };
    CKC(put_norm(h->final_norm, w->final_norm, H));
    for (int l = 0; l < hp->n_layers; ++l) {
        const dec_layer_weights &W = w->layers[l];
        DevLayer &D = h->L[l];
        char *q = static_cast<char *>(D.wqkv);
        CKC(cudaMemcpyAsync(q, W.q, nq * d * H * ws, cudaMemcpyHostToDevice, s));
        CKC(cudaMemcpyAsync(q + nq * d * H * ws, W.k, nkv * d * H * ws, cudaMemcpyHostToDevice, s));
        CKC(cudaMemcpyAsync(q + (nq + nkv) * d * H * ws, W.v, nkv * d * H * ws, cudaMemcpyHostToDevice, s));
        CKC(cudaMemcpyAsync(D.wo, W.o, H * nq * d * ws, cudaMemcpyHostToDevice, s));
        CKC(cudaMemcpyAsync(D.wd, W.down, H * F * ws, cudaMemcpyHostToDevice, s));
        // gate|up packed per 128 features: [gate rows of the block | up rows of the block]
        const size_t blk = 128 * H * ws;
        CKC(cudaStreamSynchronize(s));
        for (size_t j = 0; j < F / 128; ++j) {
            std::memcpy(gu_host.data() + (2 * j) * blk, static_cast<const char *>(W.gate) + j * blk, blk);
            std::memcpy(gu_host.data() + (2 * j + 1) * blk, static_cast<const char *>(W.up) + j * blk, blk);
        }
        CKC(cudaMemcpyAsync(D.wgu, gu_host.data(), 2 * F * H * ws, cudaMemcpyHostToDevice, s));
        if (h->w_e4m3) {
            // rounded in place: the prompt path then computes with the same weights as the codes
            launch_quantize_e4m3_rows(D.wqkv, qkv_rows(*hp), (int)H, D.wqkv8, D.wqkv_s, D.wqkv, s);
            launch_quantize_e4m3_rows(D.wo, H, (int)(nq * d), D.wo8, D.wo_s, D.wo, s);
            launch_quantize_e4m3_rows(D.wgu, 2 * F, (int)H, D.wgu8, D.wgu_s, D.wgu, s);
            launch_quantize_e4m3_rows(D.wd, H, (int)F, D.wd8, D.wd_s, D.wd, s);
            CKC(cudaGetLastError());
        }
        if (h->f16_copies) {
            // the same (rounded) values in fp16: exact for bf16 values in fp16's normal range
            launch_bf16_to_f16(D.wqkv, D.wqkv16, (size_t)qkv_rows(*hp) * H, s);
            launch_bf16_to_f16(D.wo, D.wo16, H * nq * d, s);
            launch_bf16_to_f16(D.wgu, D.wgu16, 2 * F * H, s);
            launch_bf16_to_f16(D.wd, D.wd16, H * F, s);
            CKC(cudaGetLastError());
        }
        CKC(cudaStreamSynchronize(s));
        CKC(put_norm(D.attn_norm, W.attn_norm, H));
        CKC(put_norm(D.ffn_norm, W.ffn_norm, H));
        CKC(put_norm(D.qn, W.q_norm, d));
        CKC(put_norm(D.kn, W.k_norm, d));
    }
    // RoPE table: angle p * theta^(-2i/d) in double, stored as float (cos, sin)
    {
        const size_t P = hp->max_ctx, half = d / 2;
        std::vector<float2> tab(P * half);
        for (size_t i = 0; i < half; ++i) {
            const double inv = std::pow((double)hp->rope_theta, -2.0 * (double)i / (double)d);
            for (size_t p = 0; p < P; ++p) {
                const double a = (double)p * inv;
                tab[p * half + i] = make_float2((float)std::cos(a), (float)std::sin(a));
            }
        }
        CKC(cudaMemcpyAsync(h->rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice, s));
        CKC(cudaStreamSynchronize(s));
    }
    {
        std::vector<StepLayer> sl(hp->n_layers);
        for (int l = 0; l < hp->n_layers; ++l) {
            const DevLayer &D = h->L[l];
            sl[l] = StepLayer{static_cast<const __nv_bfloat16 *>(D.wqkv), static_cast<const __nv_bfloat16 *>(D.wo),
                              static_cast<const __nv_bfloat16 *>(D.wgu), static_cast<const __nv_bfloat16 *>(D.wd),
                              D.attn_norm, D.ffn_norm, D.qn, D.kn, static_cast<__half *>(D.K),
                              static_cast<__half *>(D.V)};
        }
        CKC(cudaMemcpyAsync(h->step_layers, sl.data(), sl.size() * sizeof(StepLayer), cudaMemcpyHostToDevice, s));
        // the per-op kernel sequence is the default; SPEECH_DECODER_STEP=persistent
        // selects the single cooperative launch per step of one sequence where
        // it is supported
        const char *env = std::getenv("SPEECH_DECODER_STEP");
        bool maps_ok = true;
        std::vector<CUtensorMap> maps(2 * (size_t)hp->n_layers);
        if (h->w_bf16 && !h->w_e4m3 && h->kv_f16 && d == 128)
            for (int l = 0; l < hp->n_layers && maps_ok; ++l)
                maps_ok = step_kv_maps(&maps[2 * l], &maps[2 * l + 1], h->L[l].K, h->L[l].V, (int)(nkv * h->slots));
        else
            maps_ok = false;
        if (maps_ok)
            CKC(cudaMemcpyAsync(h->kv_maps, maps.data(), maps.size() * sizeof(CUtensorMap), cudaMemcpyHostToDevice,
                                s));
        CKC(cudaStreamSynchronize(s));
        h->use_step = maps_ok && env && !std::strcmp(env, "persistent") &&
                      step_supported((int)d, (int)(nq / nkv), (int)nkv, (int)H, (int)F, hp->max_ctx, h->num_sms) &&
                      step_splits(hp->max_ctx) <= kAttnMaxSplits;
        cudaGetLastError();
    }
    CKC(cudaMemsetAsync(h->attn_counter, 0, (size_t)hp->max_batch * nkv * sizeof(unsigned), s));
    {
        // SPEECH_DECODER_STEP_ATTN=fused lets the q|k|v GEMV of a single sequence
        // run the step attention (measured slower than the split-KV kernel on
        // the 0.6B and 1.7B shapes: one 9-warp CTA per KV head over every key)
        const char *sa = std::getenv("SPEECH_DECODER_STEP_ATTN");
        h->attn_fuse = sa && !std::strcmp(sa, "fused");
        h->attn_split_kernel = sa && !std::strcmp(sa, "split");
        const char *pl = std::getenv("SPEECH_DECODER_PLANES");
        h->lo_planes = pl ? std::max(0, std::min(15, std::atoi(pl))) : -1;
        const char *ac = std::getenv("SPEECH_DECODER_ATTN_CHUNK");
        h->attn_chunk = ac ? std::max(0, std::min(1 << 20, std::atoi(ac))) : 0;
    }
    {
        // tensor-core prompt attention: V^T columns past a sequence's keys meet
        // zero probabilities and must hold finite values, so the scratch starts at 0
        const char *pa = std::getenv("SPEECH_DECODER_PREFILL_ATTN");
        h->tc_attn = h->use_tc && h->vt && attn_prefill_tc_ok((int)d, h->kv_f16) && !(pa && !std::strcmp(pa, "simt"));
        // prompt GEMMs in fp16: fp16 weights and one fp16 activation plane
        // (an fp16 rounding, 8 times finer than bf16's, of each projection input)
        h->pf16 = h->f16_copies && h->w_bf16 && h->tc_attn && h->kv_f16 && d == 128;
        if (h->vt) CKC(cudaMemsetAsync(h->vt, 0, (size_t)nkv * d * h->vt_ld * 2, s));
    }
    CKC(cudaMemsetAsync(h->am_counter, 0, 64 * sizeof(unsigned), s));
    std::memset(&h->hst, 0, sizeof(SeqState));
    h->hst.eos_id = hp->eos_id;
    CKC(cudaMemcpyAsync(h->st, &h->hst, sizeof(SeqState), cudaMemcpyHostToDevice, s));
    CKC(cudaStreamSynchronize(s));
#undef CKC
    *out = h;
    return DEC_OK;
}

void dec_destroy(dec_handle *h) {
    if (!h) return;
    if (h->step_exec) cudaGraphExecDestroy(h->step_exec);
    if (h->gen_exec) cudaGraphExecDestroy(h->gen_exec);
    for (auto &e : h->ev)
        if (e) cudaEventDestroy(e);
    if (h->own_stream) cudaStreamDestroy(h->stream);
    delete h;
}

dec_status dec_reset(dec_handle *h) {
    if (!h) return DEC_ERR_INVALID_ARG;
    h->prefilled = false;
    h->chunk_pos = 0;
    h->n_seq = 0;
    h->logits_rows = 0;
    std::memset(&h->hst, 0, sizeof(SeqState));
    h->hst.eos_id = h->hp.eos_id;
    CK(cudaMemcpyAsync(h->st, &h->hst, sizeof(SeqState), cudaMemcpyHostToDevice, h->stream));
    CK(cudaStreamSynchronize(h->stream));
    h->err.clear();
    return DEC_OK;
}

static dec_status copy_in(dec_handle *h, void *dst, const void *src, size_t bytes, int on_device) {
    CK(cudaMemcpyAsync(dst, src, bytes, on_device ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice,
                       h->stream));
    return DEC_OK;
}

dec_status dec_prefill(dec_handle *h, const float *embeds, int32_t T, int32_t on_device, int32_t *first_token) {
    if (!h || !embeds || !first_token || T < 1) return fail(h, DEC_ERR_INVALID_ARG, "bad prefill arguments");
    const int32_t cu[2] = {0, T};
    dec_status rc = check_lengths(h, cu, 1);
    if (rc != DEC_OK) return rc;
    rc = copy_in(h, h->x, embeds, (size_t)T * h->hp.hidden * 4, on_device);
    if (rc != DEC_OK) return rc;
    return timed_prefill(h, cu, 1, first_token);
}

dec_status dec_prefill_chunk(dec_handle *h, const float *embeds, int32_t T, int32_t on_device, int32_t final_chunk,
                             int32_t *first_token) {
    if (!h || !embeds || !first_token || T < 1) return fail(h, DEC_ERR_INVALID_ARG, "bad prefill_chunk arguments");
    const dec_hparams &hp = h->hp;
    const int p0 = h->chunk_pos;
    h->chunk_pos = 0;                        // any error abandons the chunked prompt
    if (T > hp.max_tokens) return fail(h, DEC_ERR_INPUT_TOO_LONG, "chunk rows exceed max_tokens");
    if ((long long)p0 + T + hp.max_new > hp.max_ctx)
        return fail(h, DEC_ERR_INPUT_TOO_LONG,
                    "context of " + std::to_string(p0 + T) + " rows + generation budget " + std::to_string(hp.max_new) +
                        " exceeds the context of " + std::to_string(hp.max_ctx));
    dec_status rc = copy_in(h, h->x, embeds, (size_t)T * hp.hidden * 4, on_device);
    if (rc != DEC_OK) return rc;
    const int32_t cu[2] = {0, T};
    Chunk ck;
    ck.on = true;
    ck.p0 = p0;
    ck.final = final_chunk != 0;
    rc = timed_prefill(h, cu, 1, first_token, ck);
    if (rc != DEC_OK) return rc;
    h->chunk_pos = ck.final ? 0 : p0 + T;
    return DEC_OK;
}

dec_status dec_prefill_ids(dec_handle *h, const int32_t *ids, int32_t n_ids, const float *audio, int32_t n_audio,
                           int32_t prefix_len, int32_t on_device, int32_t *first_token) {
    if (!h || !first_token || n_ids < 0 || n_audio < 0 || prefix_len < 0 || prefix_len > n_ids ||
        (n_ids > 0 && !ids) || (n_audio > 0 && !audio) || n_ids + n_audio < 1)
        return fail(h, DEC_ERR_INVALID_ARG, "bad prefill_ids arguments");
    const int T = n_ids + n_audio;
    const int32_t cu[2] = {0, T};
    dec_status rc = check_lengths(h, cu, 1);
    if (rc != DEC_OK) return rc;
    if (n_ids > 0) {
        std::vector<int32_t> hid(n_ids);
        if (on_device) CK(cudaMemcpy(hid.data(), ids, n_ids * 4, cudaMemcpyDeviceToHost));
        else std::memcpy(hid.data(), ids, n_ids * 4);
        for (int i = 0; i < n_ids; ++i)
            if (hid[i] < 0 || hid[i] >= h->hp.vocab) return fail(h, DEC_ERR_INVALID_ARG, "token id out of range");
        CK(cudaMemcpyAsync(h->ids_dev, hid.data(), n_ids * 4, cudaMemcpyHostToDevice, h->stream));
        CK(cudaStreamSynchronize(h->stream));
    }
    const size_t H = h->hp.hidden;
    float *span = h->x + (size_t)prefix_len * H;
    if (n_audio > 0) {
        rc = copy_in(h, span, audio, (size_t)n_audio * H * 4, on_device);
        if (rc != DEC_OK) return rc;
    }
    launch_assemble(h->embed, h->w_bf16, h->ids_dev, span, h->x, T, n_audio, prefix_len, (int)H, h->stream);
    h->launches++;
    return timed_prefill(h, cu, 1, first_token);
}

dec_status dec_prefill_ids_batch(dec_handle *h, const int32_t *ids, const int32_t *cu_ids, const float *audio,
                                 const int32_t *cu_audio, const int32_t *prefix_lens, int32_t B, int32_t on_device,
                                 int32_t *first_tokens) {
    if (!h || !cu_ids || !cu_audio || !prefix_lens || !first_tokens || B < 1 || B > h->hp.max_batch)
        return fail(h, DEC_ERR_INVALID_ARG, "bad prefill_ids_batch arguments");
    if (cu_ids[0] != 0 || cu_audio[0] != 0) return fail(h, DEC_ERR_INVALID_ARG, "offsets must start at 0");
    std::vector<int32_t> cu(B + 1, 0);
    for (int b = 0; b < B; ++b) {
        const int ni = cu_ids[b + 1] - cu_ids[b], na = cu_audio[b + 1] - cu_audio[b];
        if (ni < 0 || na < 0 || prefix_lens[b] < 0 || prefix_lens[b] > ni || ni + na < 1)
            return fail(h, DEC_ERR_INVALID_ARG, "bad item lengths");
        cu[b + 1] = cu[b] + ni + na;
    }
    if ((cu_ids[B] > 0 && !ids) || (cu_audio[B] > 0 && !audio)) return fail(h, DEC_ERR_INVALID_ARG, "null data");
    dec_status rc = check_lengths(h, cu.data(), B);
    if (rc != DEC_OK) return rc;
    const int n_ids = cu_ids[B];
    if (n_ids > 0) {
        std::vector<int32_t> hid(n_ids);
        if (on_device) CK(cudaMemcpy(hid.data(), ids, (size_t)n_ids * 4, cudaMemcpyDeviceToHost));
        else std::memcpy(hid.data(), ids, (size_t)n_ids * 4);
        for (int i = 0; i < n_ids; ++i)
            if (hid[i] < 0 || hid[i] >= h->hp.vocab) return fail(h, DEC_ERR_INVALID_ARG, "token id out of range");
        CK(cudaMemcpyAsync(h->ids_dev, hid.data(), (size_t)n_ids * 4, cudaMemcpyHostToDevice, h->stream));
        CK(cudaStreamSynchronize(h->stream));
    }
    const size_t H = h->hp.hidden;
    for (int b = 0; b < B; ++b) {
        const int na = cu_audio[b + 1] - cu_audio[b], T = cu[b + 1] - cu[b];
        float *span = h->x + ((size_t)cu[b] + prefix_lens[b]) * H;
        if (na > 0) {
            rc = copy_in(h, span, audio + (size_t)cu_audio[b] * H, (size_t)na * H * 4, on_device);
            if (rc != DEC_OK) return rc;
        }
        launch_assemble(h->embed, h->w_bf16, h->ids_dev + cu_ids[b], span, h->x + (size_t)cu[b] * H, T, na,
                        prefix_lens[b], (int)H, h->stream);
        h->launches++;
    }
    return timed_prefill(h, cu.data(), B, first_tokens);
}

dec_status dec_prefill_batch(dec_handle *h, const float *embeds, const int32_t *cu_seqlens, int32_t B,
                             int32_t on_device, int32_t *first_tokens) {
    if (!h || !embeds || !cu_seqlens || !first_tokens) return fail(h, DEC_ERR_INVALID_ARG, "null argument");
    dec_status rc = check_lengths(h, cu_seqlens, B);
    if (rc != DEC_OK) return rc;
    rc = copy_in(h, h->x, embeds, (size_t)cu_seqlens[B] * h->hp.hidden * 4, on_device);
    if (rc != DEC_OK) return rc;
    return timed_prefill(h, cu_seqlens, B, first_tokens);
}

static dec_status step_rows(dec_handle *h, const int32_t *tokens, const uint8_t *active, int32_t *next) {
    SeqState &st = h->hst;
    const int B = h->n_seq;
    for (int b = 0; b < B; ++b) {
        const bool on = active ? active[b] != 0 : true;
        if (on && (tokens[b] < 0 || tokens[b] >= h->hp.vocab))
            return fail(h, DEC_ERR_INVALID_ARG, "token id out of range");
        if (on && st.n_past[b] + 1 > st.kv_cap[b])
            return fail(h, DEC_ERR_INPUT_TOO_LONG, "KV range of the sequence is full");
    }
    for (int b = 0; b < B; ++b) {
        const bool on = active ? active[b] != 0 : true;
        st.active[b] = on;
        st.done[b] = 0;
        if (on) st.cur_tok[b] = tokens[b];
    }
    st.max_new = 0x7fffffff;
    CK(cudaMemcpyAsync(h->st, &st, sizeof(SeqState), cudaMemcpyHostToDevice, h->stream));
    dec_status rc = run_step_graph(h, B);
    if (rc != DEC_OK) return rc;
    rc = sync_state(h);
    if (rc != DEC_OK) return rc;
    for (int b = 0; b < B; ++b) next[b] = st.active[b] ? st.cur_tok[b] : -1;
    for (int b = 0; b < B; ++b) st.active[b] = 1;
    h->logits_rows = B;
    return DEC_OK;
}

dec_status dec_step(dec_handle *h, int32_t token, int32_t *next_token) {
    if (!h || !next_token) return fail(h, DEC_ERR_INVALID_ARG, "null argument");
    if (!h->prefilled) return fail(h, DEC_ERR_STATE, "dec_step before dec_prefill");
    if (h->n_seq != 1) return fail(h, DEC_ERR_STATE, "dec_step needs a single-sequence prefill");
    return step_rows(h, &token, nullptr, next_token);
}

dec_status dec_step_batch(dec_handle *h, const int32_t *tokens, const uint8_t *active, int32_t *next_tokens) {
    if (!h || !tokens || !next_tokens) return fail(h, DEC_ERR_INVALID_ARG, "null argument");
    if (!h->prefilled) return fail(h, DEC_ERR_STATE, "dec_step_batch before a prefill");
    return step_rows(h, tokens, active, next_tokens);
}

static void finish_ids(dec_handle *h, int b, int max_new, int32_t *out, int32_t *n_out, int32_t *trunc,
                       const std::vector<int32_t> &all) {
    int n = std::min(h->hst.gen[b], max_new);
    const int32_t *src = all.data() + (size_t)b * h->hp.max_new;
    std::copy(src, src + n, out);
    const bool eos = n > 0 && src[n - 1] == h->hp.eos_id;
    if (eos) --n;
    *n_out = n;
    *trunc = eos ? 0 : 1;
}

dec_status dec_generate(dec_handle *h, int32_t max_new, int32_t *out_ids, int32_t *n_out) {
    if (!h || !out_ids || !n_out) return fail(h, DEC_ERR_INVALID_ARG, "null argument");
    if (!h->prefilled || h->n_seq != 1) return fail(h, DEC_ERR_STATE, "dec_generate needs a single-sequence prefill");
    if (max_new < 1 || max_new > h->hp.max_new) return fail(h, DEC_ERR_INVALID_ARG, "max_new out of range");
    dec_status rc = generate_core(h, max_new);
    if (rc != DEC_OK) return rc;
    std::vector<int32_t> all((size_t)h->hp.max_new * h->n_seq);
    CK(cudaMemcpy(all.data(), h->out_ids, all.size() * 4, cudaMemcpyDeviceToHost));
    int32_t trunc = 0;
    finish_ids(h, 0, max_new, out_ids, n_out, &trunc, all);
    return trunc ? fail(h, DEC_ERR_OUTPUT_TRUNCATED, "generation budget or context reached before EOS") : DEC_OK;
}

dec_status dec_generate_batch(dec_handle *h, int32_t max_new, int32_t *out_ids, int32_t *n_out, int32_t *truncated) {
    if (!h || !out_ids || !n_out || !truncated) return fail(h, DEC_ERR_INVALID_ARG, "null argument");
    if (!h->prefilled) return fail(h, DEC_ERR_STATE, "dec_generate_batch before a prefill");
    if (max_new < 1 || max_new > h->hp.max_new) return fail(h, DEC_ERR_INVALID_ARG, "max_new out of range");
    dec_status rc = generate_core(h, max_new);
    if (rc != DEC_OK) return rc;
    std::vector<int32_t> all((size_t)h->hp.max_new * h->n_seq);
    CK(cudaMemcpy(all.data(), h->out_ids, all.size() * 4, cudaMemcpyDeviceToHost));
    for (int b = 0; b < h->n_seq; ++b)
        finish_ids(h, b, max_new, out_ids + (size_t)b * max_new, n_out + b, truncated + b, all);
    return DEC_OK;
}

dec_status dec_decode_budget(int32_t n_audio, int32_t T_prompt, int32_t floor_new, int32_t ceiling,
                             int32_t *budget) {
    if (!budget || n_audio < 0 || T_prompt < 1 || floor_new < 1 || ceiling < 1) return DEC_ERR_INVALID_ARG;
    if ((int64_t)T_prompt + floor_new > (int64_t)ceiling) return DEC_ERR_INPUT_TOO_LONG;
    const int64_t asked = 2 * (int64_t)n_audio + 128;
    const int64_t room = (int64_t)ceiling - T_prompt;
    *budget = (int32_t)std::min(std::max(asked, (int64_t)floor_new), room);
    return DEC_OK;
}

dec_status dec_debug_logits(dec_handle *h, float *out, int32_t rows) {
    if (!h || !out || rows < 1) return fail(h, DEC_ERR_INVALID_ARG, "bad arguments");
    if (rows > h->logits_rows) return fail(h, DEC_ERR_STATE, "fewer logits rows available");
    CK(cudaMemcpyAsync(out, h->logits, (size_t)rows * h->hp.vocab * 4, cudaMemcpyDeviceToHost, h->stream));
    CK(cudaStreamSynchronize(h->stream));
    return DEC_OK;
}

dec_status dec_set_dumps(dec_handle *h, int32_t enable) {
    if (!h) return DEC_ERR_INVALID_ARG;
    h->dumps = enable != 0;
    return DEC_OK;
}

dec_status dec_debug_dump(dec_handle *h, const char *name, float *out, size_t n_floats) {
    if (!h || !name || !out) return fail(h, DEC_ERR_INVALID_ARG, "null argument");
    const size_t H = h->hp.hidden;
    const float *src = nullptr;
    size_t n = 0;
    if (!std::strcmp(name, "dec.audio_injected")) { src = h->dump_inj; n = (size_t)h->dump_T * H; }
    else if (!std::strcmp(name, "dec.block.0.out") && h->dump_b0_valid) { src = h->dump_b0; n = (size_t)h->dump_T * H; }
    else if (!std::strcmp(name, "dec.block.last.out")) { src = h->dump_blast; n = (size_t)h->dump_B * H; }
    else if (!std::strcmp(name, "dec.out_before_head")) { src = h->dump_final; n = (size_t)h->dump_B * H; }
    if (!src || n == 0) return fail(h, DEC_ERR_STATE, std::string("no capture named ") + name);
    if (n != n_floats) return fail(h, DEC_ERR_INVALID_ARG, "size mismatch for " + std::string(name));
    CK(cudaMemcpyAsync(out, src, n * 4, cudaMemcpyDeviceToHost, h->stream));
    CK(cudaStreamSynchronize(h->stream));
    return DEC_OK;
}

dec_status dec_launch_count(const dec_handle *h, int64_t *count) {
    if (!h || !count) return DEC_ERR_INVALID_ARG;
    *count = h->launches;
    return DEC_OK;
}

dec_status dec_profile_kernel(dec_handle *h, int32_t op, int32_t iters, float *avg_ms, double *bytes_per_launch) {
    if (!h || !avg_ms || !bytes_per_launch || iters < 1 || op < 0 || op > 3)
        return fail(h, DEC_ERR_INVALID_ARG, "bad profile arguments");
    if (!h->prefilled) return fail(h, DEC_ERR_STATE, "profile needs a prefill first");
    dec_status rc = sync_state(h);
    if (rc != DEC_OK) return rc;
    const SeqState saved = h->hst;
    SeqState live = saved;                      // profile every row, whatever the loop state
    for (int b = 0; b < h->n_seq; ++b) {
        live.active[b] = 1;
        live.done[b] = 0;
    }
    CK(cudaMemcpyAsync(h->st, &live, sizeof(SeqState), cudaMemcpyHostToDevice, h->stream));
    const dec_hparams &hp = h->hp;
    const int B = h->n_seq, H = hp.hidden, F = hp.ffn, d = hp.head_dim, nkv = hp.n_kv_heads;
    const double ws = (double)wsize(hp), kvs = (double)kvsize(hp);
    cudaStream_t s = h->stream;
    int64_t launches = 0;
    double bytes = 0.0;
    CK(cudaEventRecord(h->ev[2], s));
    for (int it = 0; it < iters; ++it) {
        if (op == 3) {
            // the whole step as one persistent launch (or the kernel sequence when it is unavailable)
            CK(cudaMemcpyAsync(h->st, &live, sizeof(SeqState), cudaMemcpyHostToDevice, s));
            h->enq = 0;
            enqueue_step(h, B);
            launches += h->enq;
            double kv = 0.0;
            for (int b = 0; b < B; ++b) kv += 2.0 * nkv * (double)(saved.n_past[b] + 1) * d * kvs * hp.n_layers;
            const double per_layer = ((double)qkv_rows(hp) * H + (double)H * hp.n_heads * d + 2.0 * F * H +
                                      (double)H * F) * ws;
            bytes += per_layer * hp.n_layers + (double)hp.vocab * H * ws + kv;
            continue;
        }
        if (op == 1) {
            // keep every row live so each launch does the full work
            CK(cudaMemcpyAsync(h->st, &live, sizeof(SeqState), cudaMemcpyHostToDevice, s));
            enqueue_head(h, B);
            ++launches;
            bytes += (double)hp.vocab * H * ws + (double)B * (H + hp.vocab) * 4.0;
            continue;
        }
        for (int l = 0; l < hp.n_layers; ++l) {
            const DevLayer &L = h->L[l];
            if (op == 0 && batched_path(h, B)) {
                // tensor-core projections of the batched step (GEMM + split-K reduction each)
                gemm(h, h->xn, h->xn_lo, L.wqkv, h->qkvd, qkv_rows(hp), B, qkv_rows(hp), H, EPI_STORE_F32);
                bytes += (double)qkv_rows(hp) * H * ws + (double)B * H * 4.0 + (double)B * qkv_rows(hp) * 4.0;
                gemm_swiglu(h, h->xn, h->xn_lo, L.wgu, B, F, H);
                bytes += (double)2 * F * H * ws + (double)B * H * 4.0 + (double)B * F * 4.0;
                launches += 2;
            } else if (op == 0) {
                // the step's four projection GEMVs of the layer, as the step launches them
                bytes += layer_qkv(h, l, B, false, false);
                bytes += layer_o(h, l, B);
                bytes += layer_gu(h, l, B);
                bytes += layer_down(h, l, B);
                launches += 4;
            } else {
                AttnDecArgs a{};
                a.qkv = h->qkvd;
                a.qn_w = L.qn;
                a.kn_w = L.kn;
                a.eps = hp.rms_eps;
                a.rope = h->rope;
                a.Kc = L.K;
                a.Vc = L.V;
                a.slots = (int)h->slots;
                a.o = h->od;
                a.part = h->attn_part;
                a.counter = h->attn_counter;
                a.st = h->st;
                a.nq = hp.n_heads;
                a.nkv = nkv;
                a.d = d;
                a.B = B;
                a.append = 0;
                a.min_chunk = attn_min_chunk(h, B);
                launch_attn_decode(h->kv_f16, a, splits_for(h, B), s);
                for (int b = 0; b < B; ++b)
                    bytes += 2.0 * nkv * (double)(saved.n_past[b] + 1) * d * kvs;
                bytes += (double)B * (qkv_rows(hp) + hp.n_heads * d) * 4.0;
                ++launches;
            }
        }
    }
    CK(cudaEventRecord(h->ev[3], s));
    CK(cudaEventSynchronize(h->ev[3]));
    CK(cudaGetLastError());
    float ms = 0.f;
    cudaEventElapsedTime(&ms, h->ev[2], h->ev[3]);
    h->launches += launches;
    h->hst = saved;
    CK(cudaMemcpyAsync(h->st, &h->hst, sizeof(SeqState), cudaMemcpyHostToDevice, s));
    CK(cudaStreamSynchronize(s));
    *avg_ms = ms / (float)launches;
    *bytes_per_launch = bytes / (double)launches;
    return DEC_OK;
}

static int current_sms() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return sms;
}

dec_status dec_attn_decode_scratch_size(int32_t B, int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                                        size_t *bytes) {
    if (!bytes || !attn_op_shape_ok(B, n_heads, n_kv_heads, head_dim, 1, 1)) return DEC_ERR_INVALID_ARG;
    const int sms = current_sms();
    if (sms <= 0) return DEC_ERR_CUDA;
    *bytes = attn_op_scratch_bytes(B, n_heads, n_kv_heads, head_dim, sms);
    return DEC_OK;
}

dec_status dec_attn_decode(const float *q, const void *K, const void *V, int32_t kv_dtype, int32_t slots,
                           const int32_t *kv_off, const int32_t *kv_len, int32_t B, int32_t n_heads,
                           int32_t n_kv_heads, int32_t head_dim, float *out, void *scratch, size_t scratch_bytes,
                           void *stream) {
    if (!q || !K || !V || !kv_off || !kv_len || !out || !scratch ||
        !attn_op_shape_ok(B, n_heads, n_kv_heads, head_dim, slots, kv_dtype == DEC_F16 || kv_dtype == DEC_F32))
        return DEC_ERR_INVALID_ARG;
    const int sms = current_sms();
    if (sms <= 0) return DEC_ERR_CUDA;
    if (scratch_bytes < attn_op_scratch_bytes(B, n_heads, n_kv_heads, head_dim, sms)) return DEC_ERR_OOM;
    cudaError_t e = attn_op_launch(q, K, V, kv_dtype == DEC_F16, slots, kv_off, kv_len, B, n_heads, n_kv_heads,
                                   head_dim, out, scratch, sms, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DEC_OK : DEC_ERR_CUDA;
}

dec_status dec_perception_project(const float *enc, int32_t T, int32_t d_in, const void *W, const float *bias,
                                  int32_t d_out, float *out, void *scratch, size_t scratch_bytes, void *stream) {
    if (!enc || !W || !bias || !out || !scratch || T < 1 || d_in < 64 || d_in % 64 || d_out < 128 || d_out % 128)
        return DEC_ERR_INVALID_ARG;
    const size_t plane = ((size_t)T * d_in * 2 + 255) / 256 * 256;
    if (scratch_bytes < 2 * plane + (size_t(16) << 20)) return DEC_ERR_OOM;
    const int sms = current_sms();
    if (sms <= 0) return DEC_ERR_CUDA;
    init_gemm_tc();
    if (!gemm_tc_ready()) return DEC_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char *base = static_cast<char *>(scratch);
    void *hi = base, *lo = base + plane;
    float *part = reinterpret_cast<float *>(base + 2 * plane);
    const size_t floats = (scratch_bytes - 2 * plane) / 4;
    launch_split_planes(enc, hi, lo, (size_t)T * d_in, s);
    cudaError_t e = launch_gemm_tc(hi, lo, T, W, d_out, d_in, 1, EPI_BIAS_F32, out, d_out, nullptr, nullptr, 0, part,
                                   floats, nullptr, sms, s, 0, bias);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return DEC_ERR_CUDA;
    }
    return cudaGetLastError() == cudaSuccess ? DEC_OK : DEC_ERR_CUDA;
}

dec_status dec_quantize_e4m3_rows(const void *w, int64_t rows, int32_t cols, uint8_t *codes, float *scales,
                                  void *w_rounded, void *stream) {
    if (!w || !codes || !scales || !w_rounded || rows < 1 || rows > INT32_MAX || cols < 1) return DEC_ERR_INVALID_ARG;
    launch_quantize_e4m3_rows(w, (size_t)rows, cols, codes, scales, w_rounded, static_cast<cudaStream_t>(stream));
    return cudaGetLastError() == cudaSuccess ? DEC_OK : DEC_ERR_CUDA;
}

dec_status dec_debug_gemm(const void *X, int32_t T, const void *W, int32_t n_feat, int32_t K, int32_t epi, float *C,
                          int32_t ldc, void *Hout, int32_t ldh, int32_t use_tc, int32_t splits, void *scratch,
                          size_t scratch_bytes, void *stream) {
    if (!X || !W || T < 1 || n_feat < 1 || K < 1 || epi < 0 || epi > 2 || !scratch ||
        scratch_bytes < (size_t(16) << 20) || (epi == 2 ? !Hout : !C))
        return DEC_ERR_INVALID_ARG;
    const int sms = current_sms();
    if (sms <= 0) return DEC_ERR_CUDA;
    init_gemm_tc();
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t floats = scratch_bytes / 4;
    if (use_tc) {
        // the tile shape the prefill takes for this projection (256 weight rows
        // per CTA for long prompts; gate|up always)
        const int groups = epi == 2 || (T > 256 && n_feat % 256 == 0) ? 2 : 1;
        if (!gemm_tc_plan(T, n_feat, K, groups, sms, floats, splits).ok) return DEC_ERR_INVALID_ARG;
        cudaError_t e = launch_gemm_tc(X, nullptr, T, W, n_feat, K, groups, epi, C, ldc, Hout, nullptr, ldh,
                                       static_cast<float *>(scratch), floats, nullptr, sms, s, splits);
        if (e != cudaSuccess) cudaGetLastError();
        return e == cudaSuccess ? DEC_OK : DEC_ERR_CUDA;
    }
    if (epi == 2) return DEC_ERR_INVALID_ARG;
    launch_gemm_simt(X, true, W, true, C, ldc, T, n_feat, K, epi, s);
    return cudaGetLastError() == cudaSuccess ? DEC_OK : DEC_ERR_CUDA;
}

dec_status dec_last_timings(const dec_handle *h, float *prefill_ms, float *generate_ms) {
    if (!h) return DEC_ERR_INVALID_ARG;
    if (prefill_ms) *prefill_ms = h->prefill_ms;
    if (generate_ms) *generate_ms = h->gen_ms;
    return DEC_OK;
}

}  // extern "C"
