// C ABI of the EAGLE-3 MLA draft head: handle, argument checks, workspace, launch sequence.
//
// Two execution paths share one handle and one workspace:
//  * rows <= 8 (batch-1 / small-batch decode): every linear layer is a weight-streaming GEMV on fp32
//    activations (bound by reading the weights once);
//  * rows > 8 with bf16 weights: every linear layer runs on the tcgen05 tensor-core GEMM with bf16
//    activations produced by the preceding kernel, and the per-head absorb / value up-projection are
//    batched tensor-core GEMMs.
// Attention is the same absorbed split-K kernel on both paths.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <map>
#include <mutex>
#include <new>
#include <utility>
#include <vector>

#include "../../include/eagle3.h"
#include "kernels.h"

using namespace e3;
typedef __nv_bfloat16 bf16_t;

cudaError_t e3::smem_optin(const void* kernel, int bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static std::mutex mu;
    static std::map<std::pair<const void*, int>, int> done;   // (kernel, device) -> bytes opted in
    std::lock_guard<std::mutex> lock(mu);
    const auto key = std::make_pair(kernel, dev);
    const auto it = done.find(key);
    if (it != done.end() && it->second >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done[key] = bytes;
    return e;
}

static thread_local int g_last_cuda_error = 0;

namespace {
enum Kind {
    K_FC = 0, K_EMBED, K_QKV_A, K_LATENT, K_Q_B, K_ABSORB, K_ATTN, K_COMBINE, K_O_PROJ, K_POST_NORM,
    K_GATE_UP, K_DOWN, K_FINAL, K_LM_HEAD, K_ARGMAX, K_EMIT, K_ROPE_Q, K_UNABSORB, K_KV_GATHER, K_KV_EXPAND,
    K_PREFILL_TILES, K_SAMPLE, K_DEQUANT, K_COUNT
};
static_assert(K_COUNT <= EAGLE3_PROF_KINDS, "profile kinds");
const char* kKindNames[EAGLE3_PROF_KINDS] = {
    "fc", "embed_norms", "q_a_kv_a", "latent_rope_append", "q_b", "absorb", "attention", "merge_splits",
    "o_proj", "post_attn_norm", "gate_up_silu", "down", "final_norm", "lm_head_argmax", "argmax_remap",
    "emit_first", "rope_q", "unabsorb", "kv_gather", "kv_expand", "prefill_tiles", "sample", "dequant_fp8", ""};
constexpr int kProfPairs = 32768;
constexpr int kGemvMaxRows = 8;          // rows above this take the tensor-core path (bf16 heads)
constexpr int kAttnWaves = 8;            // waves of attention CTAs planned for fixed-chunk splits
constexpr int kAttnChunkRows = 16;       // rows from which attention splits use fixed chunks
constexpr size_t kSplitKBytes = 64u << 20;
constexpr int kPrefillMinRows = 1024;    // extends of at least this many rows may take the unabsorbed path
}  // namespace

struct eagle3_draft {
    eagle3_config_t cfg;
    eagle3_weights_t w;
    int device = 0;
    int num_sms = 0;
    void* ws = nullptr;
    size_t ws_bytes = 0;
    int m_cap = 0;          // rows per call
    int splits_cap = 0;     // attention splits bound
    int npart = 0;          // lm_head argmax partials per row of the latest scoring
    bool tc_ok = false;     // the tensor-core path is available for this head
    // workspace views (fp32 unless named _bf)
    float *f = nullptr, *carry = nullptr, *x = nullptr, *cqkv = nullptr, *cq_hat = nullptr, *q = nullptr,
          *qa = nullptr, *part_o = nullptr, *part_ml = nullptr, *o = nullptr, *h1 = nullptr, *y = nullptr,
          *mlp = nullptr, *h2 = nullptr, *z = nullptr, *pval = nullptr, *rope_cos = nullptr,
          *rope_sin = nullptr, *tc_part = nullptr, *olat = nullptr, *logits = nullptr;
    bf16_t *qa_bf = nullptr, *x_bf = nullptr, *cqh_bf = nullptr, *q_bf = nullptr, *olat_bf = nullptr,
           *o_bf = nullptr, *y_bf = nullptr, *m_bf = nullptr, *z_bf = nullptr, *wukt = nullptr;
    // unabsorbed extend attention (allocated when the configuration allows long extends)
    bf16_t *xc = nullptr, *xpe = nullptr, *kvx = nullptr;
    int4* tiles = nullptr;
    int tiles_cap = 0;
    // FP8 heads on the tensor-core path: the bf16 expansion of the matrix being multiplied
    bf16_t* wdq = nullptr;
    int *pidx = nullptr, *row_seq = nullptr, *row_pos = nullptr, *d0 = nullptr, *tok_in = nullptr,
        *err = nullptr;
    size_t part_rows = 0;   // capacity of the attention partials in (row, split) pairs
    int batch = 0;
    bool have_extend = false;
    // native tracing: event pairs around launches, accumulated per kernel kind
    uint32_t prof_mask = 0;   // kinds whose launches are timed
    std::vector<cudaEvent_t> prof_ev;
    std::vector<int> prof_kind;
    int prof_used = 0;
    double prof_ms[EAGLE3_PROF_KINDS] = {};
    int64_t prof_n[EAGLE3_PROF_KINDS] = {};
    int64_t launches[EAGLE3_PROF_KINDS] = {};
};

namespace {

// Runs `launch` (returning cudaError_t) bracketed by profiling events when enabled.
template <typename F>
cudaError_t traced(eagle3_draft& d, int kind, cudaStream_t st, F&& launch) {
    d.launches[kind] += 1;
    const bool rec = ((d.prof_mask >> kind) & 1u) && d.prof_used < kProfPairs;
    // Inside stream capture an event record must be "external" to become a timestamp node of the graph.
    unsigned int flags = cudaEventRecordDefault;
    if (rec) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        cudaError_t e = cudaStreamIsCapturing(st, &cs);
        if (e != cudaSuccess) return e;
        if (cs == cudaStreamCaptureStatusActive) flags = cudaEventRecordExternal;
        e = cudaEventRecordWithFlags(d.prof_ev[2 * d.prof_used], st, flags);
        if (e != cudaSuccess) return e;
    }
    cudaError_t e = launch();
    if (e != cudaSuccess) return e;
    if (rec) {
        e = cudaEventRecordWithFlags(d.prof_ev[2 * d.prof_used + 1], st, flags);
        if (e != cudaSuccess) return e;
        d.prof_kind[d.prof_used] = kind;
        d.prof_used += 1;
    }
    return cudaSuccess;
}

cudaError_t prof_flush(eagle3_draft& d) {
    if (d.prof_used == 0) return cudaSuccess;
    cudaError_t e = cudaEventSynchronize(d.prof_ev[2 * d.prof_used - 1]);
    if (e != cudaSuccess) return e;
    for (int i = 0; i < d.prof_used; ++i) {
        float ms = 0.f;
        e = cudaEventElapsedTime(&ms, d.prof_ev[2 * i], d.prof_ev[2 * i + 1]);
        if (e != cudaSuccess) return e;
        d.prof_ms[d.prof_kind[i]] += ms;
        d.prof_n[d.prof_kind[i]] += 1;
    }
    d.prof_used = 0;
    return cudaSuccess;
}

eagle3_status_t cuda_fail(cudaError_t e) {
    g_last_cuda_error = (int)e;
    return EAGLE3_ERR_CUDA;
}

#define E3_CUDA(call)                                  \
    do {                                               \
        cudaError_t _e = (call);                       \
        if (_e != cudaSuccess) return cuda_fail(_e);   \
    } while (0)
#define E3_TRY(call)                                   \
    do {                                               \
        cudaError_t _e = (call);                       \
        if (_e != cudaSuccess) return _e;              \
    } while (0)

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Attention split plan for M rows.  With few rows the context of each row is divided evenly over
// enough splits for two CTAs per SM.  From kAttnChunkRows rows on, contexts are cut into fixed chunks
// instead (about kAttnWaves waves of CTAs over the longest possible context), so rows of very different
// lengths give CTAs of similar work; splits past a row's context exit at once.
void attn_plan(const eagle3_draft& d, int M, int* splits, int* chunk) {
    const int hpc = attention_heads_per_cta(d.cfg.dtype == EAGLE3_BF16 ? BF16 : F32, d.cfg.kv_lora_rank,
                                            d.cfg.qk_rope_dim);
    const long hg = (d.cfg.n_heads + hpc - 1) / hpc;
    const long rows = (long)M * hg, ctx = d.cfg.max_ctx;
    *chunk = 0;
    if (M < kAttnChunkRows) {
        // Each row's context is divided evenly over the splits.  The 64-head mma.sync kernel holds one
        // CTA per SM: its (split, head block, row) CTAs fill one wave, so the longest context takes the
        // fewest 32-slot tiles per CTA (4097 slots: 2 tiles over 76 splits instead of 3 over 64 in a
        // second wave's worth of CTAs); the merge fused with the value projection takes up to 128 splits
        // (at most 8 rows), the plain merge 64.  Other kernels plan two CTAs per SM.
        const bool dt_bf = d.cfg.dtype == EAGLE3_BF16;
        const bool one = attention_one_cta_per_sm(dt_bf ? BF16 : F32, d.cfg.kv_lora_rank, d.cfg.qk_rope_dim);
        long s = one ? d.num_sms / rows : (2L * d.num_sms + rows - 1) / rows;
        long cap = d.splits_cap;
        if (one && dt_bf && M <= 8 && d.cfg.kv_lora_rank == 512 && d.cfg.v_head_dim == 128) {
            cap = (d.cfg.max_ctx + 31) / 32;
            if (cap > kMergeUnabsorbMaxSplits) cap = kMergeUnabsorbMaxSplits;
        }
        if (s > cap) s = cap;
        if (s < 1) s = 1;
        while (s > 1 && (size_t)M * s > d.part_rows) --s;
        *splits = (int)s;
        return;
    }
    long ch = (ctx * rows + (long)kAttnWaves * d.num_sms - 1) / ((long)kAttnWaves * d.num_sms);
    if (ch < 256) ch = 256;
    ch = (ch + 31) / 32 * 32;
    long s = (ctx + ch - 1) / ch;
    // at most splits_cap splits, and the (row, split) partials must fit the workspace
    while (s > 1 && (s > d.splits_cap || (size_t)M * s > d.part_rows)) {
        ch *= 2;
        s = (ctx + ch - 1) / ch;
    }
    *splits = (int)s;
    *chunk = s > 1 ? (int)ch : 0;
}

// The tcgen05 latent attention serves the DeepseekV3 geometry in bf16 (128 heads, latent 512, rope 64)
// with cache pages of a multiple of 64 slots, from kAttnChunkRows rows per call.  Below that (batch-1
// decode) the mma.sync kernel's lighter launch (no cluster, no TMEM) is the faster one.
bool attention_tc_ok(const eagle3_draft& d, int M) {
    const eagle3_config_t& c = d.cfg;
    return M >= kAttnChunkRows && c.dtype == EAGLE3_BF16 && c.attention != EAGLE3_ATTN_MHA && c.n_heads == 128 &&
           c.kv_lora_rank == 512 && c.qk_rope_dim == 64 && c.page_size % 64 == 0;
}

// Split plan of the tcgen05 attention: fixed chunks of whole 64-slot tiles (splits past a row's context
// exit at once and the merge skips them), sized so the CTA pairs of the longest possible contexts fill
// about one wave (few rows), four waves, or eight from 128 rows (ragged contexts then leave a shorter
// tail of long chunks: batch 256, 1.31 -> 1.24 ms per call), with at most splits_cap splits and the
// partials within the workspace.
void attn_plan_tc(const eagle3_draft& d, int M, int* splits, int* chunk) {
    const long pairs = d.num_sms / 2 > 0 ? d.num_sms / 2 : 1, ctx = d.cfg.max_ctx;
    const long waves = M < kAttnChunkRows ? 1 : (M >= 128 ? 8 : 4);
    long ch = (ctx * M + waves * pairs - 1) / (waves * pairs);
    const long ch_min = (ctx + d.splits_cap - 1) / d.splits_cap;
    if (ch < ch_min) ch = ch_min;
    if (ch < 128) ch = 128;
    ch = (ch + 63) / 64 * 64;
    long s = (ctx + ch - 1) / ch;
    while (s > 1 && (s > d.splits_cap || (size_t)M * s > d.part_rows)) {
        ch *= 2;
        s = (ctx + ch - 1) / ch;
    }
    *splits = (int)s;
    *chunk = (int)((s > 1 ? ch : (ctx + 63) / 64 * 64));
}

bool mha_head(const eagle3_config_t& c) { return c.attention == EAGLE3_ATTN_MHA; }
int fc_inputs(const eagle3_config_t& c) { return c.fc_inputs == 0 ? 3 : c.fc_inputs; }
// width rotated by RoPE: d_r (MLA) or the whole head_dim (MHA)
int rope_dim(const eagle3_config_t& c) { return mha_head(c) ? c.head_dim : c.qk_rope_dim; }

// The Llama-style MHA head's configuration (its MLA sizes are not read).
eagle3_status_t check_config_mha(const eagle3_config_t* c) {
    const int dims[] = {c->hidden, c->n_heads, c->n_kv_heads, c->head_dim, c->intermediate, c->target_vocab,
                        c->draft_vocab, c->max_batch, c->max_tokens_per_extend, c->max_ctx, c->page_size,
                        c->max_pages_per_seq};
    for (int v : dims)
        if (v <= 0) return EAGLE3_ERR_INVALID_ARG;
    if (c->n_heads % c->n_kv_heads) return EAGLE3_ERR_INVALID_ARG;
    if (!mha_supported(c->n_heads, c->n_kv_heads, c->head_dim)) return EAGLE3_ERR_UNSUPPORTED;
    if (c->dtype != EAGLE3_F32 && c->dtype != EAGLE3_BF16) return EAGLE3_ERR_INVALID_ARG;
    if (c->weight_format != EAGLE3_WEIGHTS_DTYPE) return EAGLE3_ERR_UNSUPPORTED;
    if (c->hidden % 8 || c->intermediate % 8) return EAGLE3_ERR_UNSUPPORTED;
    if (c->draft_vocab > c->target_vocab) return EAGLE3_ERR_INVALID_ARG;
    if (c->hidden > 16384) return EAGLE3_ERR_UNSUPPORTED;
    if (!(c->rms_eps > 0.f) || !(c->rope_theta > 1.f) || !(c->yarn_factor >= 1.f) ||
        c->yarn_original_max_pos <= 0)
        return EAGLE3_ERR_INVALID_ARG;
    if ((long)c->max_ctx > (long)c->max_pages_per_seq * c->page_size) return EAGLE3_ERR_INVALID_ARG;
    return EAGLE3_OK;
}

eagle3_status_t check_config(const eagle3_config_t* c) {
    if (!c) return EAGLE3_ERR_INVALID_ARG;
    if (c->attention != EAGLE3_ATTN_MLA && c->attention != EAGLE3_ATTN_MHA) return EAGLE3_ERR_INVALID_ARG;
    if (fc_inputs(*c) != 3 && !(mha_head(*c) && fc_inputs(*c) == 2)) return EAGLE3_ERR_INVALID_ARG;
    if (mha_head(*c)) return check_config_mha(c);
    const int dims[] = {c->hidden, c->n_heads, c->q_lora_rank, c->kv_lora_rank, c->qk_nope_dim, c->qk_rope_dim,
                        c->v_head_dim, c->intermediate, c->target_vocab, c->draft_vocab, c->max_batch,
                        c->max_tokens_per_extend, c->max_ctx, c->page_size, c->max_pages_per_seq};
    for (int v : dims)
        if (v <= 0) return EAGLE3_ERR_INVALID_ARG;
    if (c->qk_rope_dim % 2) return EAGLE3_ERR_INVALID_ARG;
    if (c->rope_interleave != 1) return EAGLE3_ERR_UNSUPPORTED;
    if (c->dtype != EAGLE3_F32 && c->dtype != EAGLE3_BF16) return EAGLE3_ERR_INVALID_ARG;
    if (c->weight_format != EAGLE3_WEIGHTS_DTYPE && c->weight_format != EAGLE3_WEIGHTS_FP8 &&
        c->weight_format != EAGLE3_WEIGHTS_NVFP4)
        return EAGLE3_ERR_INVALID_ARG;
    if (c->weight_format != EAGLE3_WEIGHTS_DTYPE) {
        // the FP8 kernels load 16 codes per lane, the NVFP4 kernels 32: every quantized matrix's K is a
        // multiple of that
        const int u = c->weight_format == EAGLE3_WEIGHTS_FP8 ? 16 : 32;
        if (c->dtype != EAGLE3_BF16) return EAGLE3_ERR_UNSUPPORTED;
        if (c->hidden % u || c->q_lora_rank % u || (c->n_heads * c->v_head_dim) % u || c->intermediate % u)
            return EAGLE3_ERR_UNSUPPORTED;
    }
    // inner (K) dimensions of every linear layer stream in 8-element chunks
    const long inner[] = {c->hidden, c->q_lora_rank, c->kv_lora_rank, (long)c->n_heads * c->v_head_dim,
                          c->intermediate, c->kv_lora_rank + c->qk_rope_dim};
    for (long v : inner)
        if (v % 8) return EAGLE3_ERR_UNSUPPORTED;
    if (!attention_supported(c->kv_lora_rank, c->qk_rope_dim, c->qk_nope_dim, c->v_head_dim))
        return EAGLE3_ERR_UNSUPPORTED;
    if (c->draft_vocab > c->target_vocab) return EAGLE3_ERR_INVALID_ARG;
    // row kernels hold a row in registers: H <= 16384, q_lora_rank and kv_lora_rank <= 2048
    if (c->hidden > 16384 || c->q_lora_rank > 2048 || c->kv_lora_rank > 2048) return EAGLE3_ERR_UNSUPPORTED;
    if (!(c->rms_eps > 0.f) || !(c->rope_theta > 1.f) || !(c->yarn_factor >= 1.f) ||
        c->yarn_original_max_pos <= 0)
        return EAGLE3_ERR_INVALID_ARG;
    if ((long)c->max_ctx > (long)c->max_pages_per_seq * c->page_size) return EAGLE3_ERR_INVALID_ARG;
    return EAGLE3_OK;
}

eagle3_status_t check_weights(const eagle3_config_t& c, const eagle3_weights_t* w) {
    if (!w) return EAGLE3_ERR_INVALID_ARG;
    if (mha_head(c)) {
        const void* p[] = {w->embed, w->fc, w->input_norm, w->hidden_norm, w->q_proj, w->k_proj, w->v_proj, w->o,
                           w->post_attn_norm, w->gate, w->up, w->down, w->final_norm, w->lm_head};
        for (const void* v : p)
            if (!v || !aligned16(v)) return EAGLE3_ERR_INVALID_ARG;
        return EAGLE3_OK;
    }
    const void* p[] = {w->embed, w->fc, w->input_norm, w->hidden_norm, w->q_a, w->q_a_norm, w->q_b,
                       w->kv_a, w->kv_a_norm, w->kv_b, w->o, w->post_attn_norm, w->gate, w->up, w->down,
                       w->final_norm, w->lm_head};
    for (const void* v : p)
        if (!v || !aligned16(v)) return EAGLE3_ERR_INVALID_ARG;
    if (c.weight_format != EAGLE3_WEIGHTS_DTYPE) {
        // FP8 row scales are fp32; NVFP4 block scales are read two bytes at a time
        const uintptr_t align = c.weight_format == EAGLE3_WEIGHTS_FP8 ? 3u : 1u;
        const void* s[] = {w->fc_scale, w->q_a_scale, w->kv_a_scale, w->q_b_scale, w->o_scale, w->gate_scale,
                           w->up_scale, w->down_scale, w->lm_head_scale};
        for (const void* v : s)
            if (!v || ((uintptr_t)v & align)) return EAGLE3_ERR_INVALID_ARG;
        if (c.weight_format == EAGLE3_WEIGHTS_NVFP4 && (!w->matrix_scales || ((uintptr_t)w->matrix_scales & 3u)))
            return EAGLE3_ERR_INVALID_ARG;
    }
    return EAGLE3_OK;
}

// The head stores its projection matrices quantized (FP8 or NVFP4).
bool quant_head(const eagle3_config_t& c) { return c.weight_format != EAGLE3_WEIGHTS_DTYPE; }
// Index of each quantized matrix in eagle3_weights_t::matrix_scales.
enum QMat { QM_FC = 0, QM_QA, QM_KVA, QM_QB, QM_O, QM_GATE, QM_UP, QM_DOWN, QM_LM };

// Elements of the largest quantized matrix pair one tensor-core GEMM reads (q_a | kv_a and gate | up are
// expanded together).
size_t quant_max_matrix(const eagle3_config_t& c) {
    const size_t H = c.hidden, nh = c.n_heads, D = c.kv_lora_rank + c.qk_rope_dim;
    const size_t m[] = {H * 3 * H, (c.q_lora_rank + D) * 2 * H, nh * (c.qk_nope_dim + c.qk_rope_dim) * c.q_lora_rank,
                        H * nh * c.v_head_dim, 2 * (size_t)c.intermediate * H, H * c.intermediate,
                        (size_t)c.draft_vocab * H};
    size_t best = 0;
    for (size_t v : m) best = v > best ? v : best;
    return best;
}

// The tensor-core path needs bf16 weights, every GEMM K a multiple of 64 and the q_a | kv_a split on a
// 128-row tile boundary; otherwise large calls stay on the GEMV path.
bool tc_supported(const eagle3_config_t& c) {
    if (c.dtype != EAGLE3_BF16) return false;
    if (mha_head(c)) {
        // K of every GEMM a multiple of 64, the k | v split on a 128-row tile boundary
        const long ks[] = {c.hidden, (long)c.n_heads * c.head_dim, c.intermediate};
        for (long k : ks)
            if (k % 64) return false;
        return ((long)c.n_kv_heads * c.head_dim) % 128 == 0;
    }
    const long ks[] = {c.hidden, c.q_lora_rank, c.kv_lora_rank, c.qk_nope_dim, (long)c.n_heads * c.v_head_dim,
                       c.intermediate, c.qk_nope_dim + c.qk_rope_dim};
    for (long k : ks)
        if (k % 64) return false;
    return c.q_lora_rank % 128 == 0 && c.kv_lora_rank == 512 && c.qk_rope_dim == 64;
}

// Workspace layout: one allocation carved into 256-byte aligned views.
struct Layout {
    size_t off = 0;
    size_t take(size_t bytes) {
        size_t o = off;
        off += (bytes + 255) & ~(size_t)255;
        return o;
    }
};

struct Offsets {
    size_t f, carry, x, cqkv, cq_hat, q, qa, qa_bf, part_o, part_ml, o, h1, y, mlp, h2, z, pval, pidx, rope_cos,
        rope_sin, row_seq, row_pos, d0, tok_in, err, olat, x_bf, cqh_bf, q_bf, olat_bf, o_bf, y_bf, m_bf, z_bf, wukt,
        tc_part, xc, xpe, kvx, tiles, logits, wdq, total;
    int tiles_cap;
    int m_cap, splits_cap, npart;
    size_t part_rows;
};

// The unabsorbed extend path exists for bf16 heads with the DeepseekV3 head geometry whose
// configuration allows extends of at least kPrefillMinRows rows.
bool prefill_allowed(const eagle3_config_t& c) {
    return !mha_head(c) && tc_supported(c) && c.max_tokens_per_extend >= kPrefillMinRows &&
           prefill_supported(c.dtype == EAGLE3_BF16 ? BF16 : F32, c.qk_nope_dim, c.qk_rope_dim, c.v_head_dim);
}

Offsets plan(const eagle3_config_t& c, int num_sms) {
    Offsets o;
    const long M = c.max_tokens_per_extend > c.max_batch ? c.max_tokens_per_extend : c.max_batch;
    const long H = c.hidden, nh = c.n_heads, dqk = c.qk_nope_dim + c.qk_rope_dim;
    const long D = c.kv_lora_rank + c.qk_rope_dim, B = c.max_batch;
    const bool tc = tc_supported(c);
    const bool mha = mha_head(c);
    const long hd = c.head_dim, nkv = c.n_kv_heads;
    // per-row widths: projections into cqkv ([q_a | kv_a] or [k | v]), queries, attention output; the
    // attention partials' width per head; MLA-only buffers are empty for an MHA head
    const long w_cqkv = mha ? 2 * nkv * hd : c.q_lora_rank + D;
    const long w_q = mha ? nh * hd : nh * dqk, w_o = mha ? nh * hd : nh * c.v_head_dim;
    const long w_part = mha ? hd : c.kv_lora_rank;
    const long mla = mha ? 0 : 1;
    const long Mt = tc ? M : 0;       // rows of the bf16 activation copies
    o.m_cap = (int)M;
    o.splits_cap = (c.max_ctx + 31) / 32;
    if (o.splits_cap > 64) o.splits_cap = 64;
    // argmax partials per scored row: the GEMV writes one per CTA, the tensor-core GEMM one per 128 rows
    o.npart = gemv_argmax_parts(c.draft_vocab, num_sms);
    if (tc && (c.draft_vocab + 127) / 128 > o.npart) o.npart = (c.draft_vocab + 127) / 128;
    // (row, split) partials: few rows use at most M + 2 * num_sms pairs (splits = ceil(2 SMs / row groups),
    // or SMs / row groups for the one-CTA-per-SM kernel);
    // fixed chunks are planned for about kAttnWaves * num_sms pairs and shrunk to fit this capacity
    o.part_rows = (size_t)M + (size_t)kAttnWaves * num_sms + 1;
    Layout L;
    const size_t f4 = 4, b2 = 2;
    o.f = L.take(M * H * f4);
    o.carry = L.take(B * H * f4);
    o.x = L.take(M * 2 * H * f4);
    o.cqkv = L.take(M * w_cqkv * f4);
    o.cq_hat = L.take(mla * M * c.q_lora_rank * f4);
    o.q = L.take(M * w_q * f4);
    o.qa = L.take(mla * M * nh * D * f4);
    o.qa_bf = L.take(mla * M * nh * D * b2);
    o.part_o = L.take(o.part_rows * nh * w_part * f4);
    o.part_ml = L.take(o.part_rows * nh * 2 * f4);
    o.o = L.take(M * w_o * f4);
    o.h1 = L.take(M * H * f4);
    o.y = L.take(M * H * f4);
    o.mlp = L.take(M * (size_t)c.intermediate * f4);
    o.h2 = L.take(M * H * f4);
    o.z = L.take(B * H * f4);
    o.pval = L.take(B * o.npart * f4);
    o.pidx = L.take(B * o.npart * 4);
    o.rope_cos = L.take((size_t)c.max_ctx * (rope_dim(c) / 2) * f4);
    o.rope_sin = L.take((size_t)c.max_ctx * (rope_dim(c) / 2) * f4);
    o.row_seq = L.take(M * 4);
    o.row_pos = L.take(M * 4);
    o.d0 = L.take(B * 4);
    o.tok_in = L.take(B * 4);
    o.err = L.take(4);
    o.olat = L.take(mla * (tc && M > 8 ? 8 : M) * nh * c.kv_lora_rank * f4);
    o.x_bf = L.take(Mt * 2 * H * b2);
    o.cqh_bf = L.take(mla * Mt * c.q_lora_rank * b2);
    o.q_bf = L.take(mla * Mt * nh * dqk * b2);
    o.olat_bf = L.take(mla * Mt * nh * c.kv_lora_rank * b2);
    o.o_bf = L.take(Mt * w_o * b2);
    o.y_bf = L.take(Mt * H * b2);
    o.m_bf = L.take(Mt * (size_t)c.intermediate * b2);
    o.z_bf = L.take((tc ? B : 0) * H * b2);
    o.wukt = L.take(tc && !mha ? (size_t)nh * c.kv_lora_rank * c.qk_nope_dim * b2 : 0);
    o.tc_part = L.take(tc ? kSplitKBytes : 0);
    o.logits = L.take(B * (size_t)c.draft_vocab * f4);   // lm_head outputs of a sampled decode step
    // unabsorbed extend attention: gathered latent rows, expanded keys/values, query tile map
    const bool pre = prefill_allowed(c);
    const size_t slots = pre ? (size_t)B * c.max_ctx : 0;
    o.tiles_cap = pre ? prefill_tiles_cap((int)M, (int)B, 64) : 0;   // the finer of the two tile heights
    o.xc = L.take(slots * c.kv_lora_rank * b2);
    o.xpe = L.take(slots * c.qk_rope_dim * b2);
    o.kvx = L.take(slots * nh * (c.qk_nope_dim + c.v_head_dim) * b2);
    o.tiles = L.take((size_t)o.tiles_cap * sizeof(int4));
    o.wdq = L.take(tc && quant_head(c) && M > kGemvMaxRows ? quant_max_matrix(c) * b2 : 0);
    o.total = L.off;
    return o;
}

// YaRN rotary frequencies (the published YaRN construction; the pages name DeepseekYarnRotaryEmbedding
// and its rope_scaling betas, "Eagle3 DeepseekV3 in MAX" §4-§5): pair i keeps theta^(-2i/d) where its
// wavelength fits >= beta_fast times in the original window, is divided by the factor where it fits
// < beta_slow times, and is blended linearly in between.
void yarn_table(const eagle3_config_t& c, std::vector<float>& cs, std::vector<float>& sn) {
    const int d = rope_dim(c), half = d / 2;
    const double theta = c.rope_theta, f = c.yarn_factor, L0 = c.yarn_original_max_pos;
    auto band = [&](double beta) { return d * log(L0 / (2.0 * M_PI * beta)) / (2.0 * log(theta)); };
    double lo = floor(band(c.yarn_beta_fast));
    if (lo < 0) lo = 0;
    double hi = ceil(band(c.yarn_beta_slow));
    if (hi > d - 1) hi = d - 1;
    if (lo == hi) hi += 0.001;
    std::vector<double> inv(half);
    for (int i = 0; i < half; ++i) {
        const double plain = pow(theta, -2.0 * i / d);
        double t = (i - lo) / (hi - lo);
        t = t < 0 ? 0 : (t > 1 ? 1 : t);
        inv[i] = (plain / f) * t + plain * (1.0 - t);
    }
    auto mag = [&](double mu) { return f <= 1.0 ? 1.0 : 0.1 * mu * log(f) + 1.0; };
    const double scale = mag(c.yarn_mscale) / mag(c.yarn_mscale_all_dim);
    cs.resize((size_t)c.max_ctx * half);
    sn.resize((size_t)c.max_ctx * half);
    for (long p = 0; p < c.max_ctx; ++p)
        for (int i = 0; i < half; ++i) {
            const double ang = (double)p * inv[i];
            cs[p * half + i] = (float)(cos(ang) * scale);
            sn[p * half + i] = (float)(sin(ang) * scale);
        }
}

float attention_scale(const eagle3_config_t& c) {
    const double f = c.yarn_factor;
    const double m = f <= 1.0 ? 1.0 : 0.1 * c.yarn_mscale_all_dim * log(f) + 1.0;
    const int dqk = mha_head(c) ? c.head_dim : c.qk_nope_dim + c.qk_rope_dim;
    return (float)(m * m / sqrt((double)dqk));
}

RowArgs row_args(const eagle3_draft& d, const eagle3_kv_t* kv) {
    RowArgs a;
    const eagle3_config_t& c = d.cfg;
    a.H = c.hidden; a.dq = c.q_lora_rank; a.dc = c.kv_lora_rank; a.dr = c.qk_rope_dim;
    a.nh = c.n_heads; a.dn = c.qk_nope_dim; a.dv = c.v_head_dim;
    a.Vt = c.target_vocab; a.max_ctx = c.max_ctx; a.page_size = c.page_size; a.max_pages = c.max_pages_per_seq;
    a.num_pages = kv ? kv->num_pages : 0;
    a.eps = c.rms_eps;
    a.dt = c.dtype == EAGLE3_BF16 ? BF16 : F32;
    a.err = d.err;
    return a;
}

// ---------------------------------------------------------------------------------------------- linear
// One bias-free linear layer y = X W^T + epilogue, on whichever path the row count selects.
struct Lin {
    int M = 0, N = 0, K = 0, epi = EPI_STORE;
    // activations: up to 3 K-segments; fp32 for the GEMV path, bf16 for the tensor-core path
    int na = 1;
    const void* a32[3] = {nullptr, nullptr, nullptr};
    bool a32_is_bf16 = false;       // the GEMV path may read bf16 activations (the aux states)
    const bf16_t* a16[3] = {nullptr, nullptr, nullptr};
    long lda[3] = {0, 0, 0};
    int ka[3] = {0, 0, 0};
    // weights: segment 0 rows [0, n0rows), segment 1 the rest (GLU: gate and up, N rows each)
    const void* w0 = nullptr;
    const void* w1 = nullptr;
    int n0rows = 0, n1rows = 0;
    // quantized weights (set by quant()): the format, the scales of w0 / w1 (FP8 fp32 row scales or
    // NVFP4 E4M3 block scales) and, for NVFP4, the two matrices' fp32 scales
    int wq = EAGLE3_WEIGHTS_DTYPE;
    const void* s0 = nullptr;
    const void* s1 = nullptr;
    const float* g0 = nullptr;
    const float* g1 = nullptr;
    float* y = nullptr; long ldy = 0;          // fp32 output (GEMV path always; tensor path when set)
    bf16_t* ybf = nullptr; long ldybf = 0;     // bf16 output for the next tensor-core GEMM
    const float* resid = nullptr; long ldr = 0;
    float* logits = nullptr; long ldl = 0;     // ARGMAX debug output
    // grouped rows (GEMV path only): see GemvArgs
    int w_grp = 0; long w_grp_stride = 0; int w_row0 = 0;
    bool force_tc = false;   // run on the tensor-core GEMM whatever the row count
    int a_grp = 0; long a_grp_stride = 0;
};

bool use_tc(const eagle3_draft& d, int M) { return d.tc_ok && M > kGemvMaxRows; }

// The lm_head scores 5 to 8 rows on the tensor cores too: the GEMV would multiply every weight by each
// row's activations from L1, and at that many rows the L1 reads, not HBM, set its pace.  (Quantized heads
// keep the GEMV: their expansion buffer exists only for heads that take more than 8 rows.)
bool head_tc(const eagle3_draft& d, int rows) {
    return use_tc(d, rows) || (d.tc_ok && rows >= 5 && !quant_head(d.cfg) && d.z_bf != nullptr);
}

// Split-K count for a tensor-core GEMM: the count that minimises a wave model of the launch.  One CTA
// per SM at a time; a CTA streams its share of the weight tile at the SM's share of the HBM bandwidth (or
// runs its MMAs, when they take longer), plus a fixed start and drain cost; CTAs run in waves of num_sms,
// so a grid just past a multiple of the SM count pays a whole extra wave.  Every split adds a write and a
// read of the fp32 partial planes, and the reduction kernel's launch.  Fewer splits win ties.
int tc_splits(const eagle3_draft& d, int M, int N, int K, int bn, bool glu) {
    const long tiles = (long)((N + 127) / 128) * ((M + bn - 1) / bn);
    const int nkb = K / 64;
    const int smax = nkb / 4 < 64 ? nkb / 4 : 64;   // at least 4 K-blocks per split
    if (smax < 2) return 1;
    const double hbm = 6.0e12, sm_bw = hbm / d.num_sms;   // achievable bytes/s, whole GPU and per SM
    const double mac_rate = 7.0e12;                       // dense bf16 MACs/s of one SM's tensor core
    const double c0 = 2.0e-6, c_sum = 4.0e-6;             // per-CTA start/drain; the reduction launch
    const double np = glu ? 2.0 : 1.0;
    const double plane = np * M * N * 4.0;
    int best = 1;
    double t_best = 1e30;
    for (int s = 1; s <= smax; ++s) {
        const int per = (nkb + s - 1) / s, eff = (nkb + per - 1) / per;   // the launcher's split count
        if (eff != s) continue;
        if (s > 1 && s * plane > (double)kSplitKBytes) break;
        const long waves = (tiles * s + d.num_sms - 1) / d.num_sms;
        const double t_mem = np * 128.0 * per * 64 * 2 / sm_bw;
        const double t_mma = np * 128.0 * bn * per * 64 / mac_rate;
        double t = waves * ((t_mem > t_mma ? t_mem : t_mma) + c0);
        if (s > 1) t += 2.0 * s * plane / hbm + c_sum;
        if (t < 0.97 * t_best) {
            t_best = t;
            best = s;
        }
    }
    return best;
}

cudaError_t run_linear(eagle3_draft& d, const Lin& L, int kind, cudaStream_t st) {
    if (!L.force_tc && !use_tc(d, L.M)) {
        GemvArgs g;
        memset(&g, 0, sizeof(g));
        for (int i = 0; i < L.na; ++i) { g.a[i] = L.a32[i]; g.lda[i] = L.lda[i]; g.ka[i] = L.ka[i]; }
        g.na = L.na;
        g.w[0] = L.w0; g.w[1] = L.w1;
        g.nw[0] = L.n0rows; g.nw[1] = L.n1rows;
        g.nseg_w = (L.epi != EPI_GLU && L.w1) ? 2 : 1;
        g.M = L.M; g.N = L.N; g.K = L.K;
        g.a_type = L.a32_is_bf16 ? BF16 : F32;
        g.w_type = d.cfg.dtype == EAGLE3_BF16 ? BF16 : F32;
        if (L.wq == EAGLE3_WEIGHTS_FP8) {
            g.w_type = FP8;
            g.wscale[0] = static_cast<const float*>(L.s0); g.wscale[1] = static_cast<const float*>(L.s1);
        } else if (L.wq == EAGLE3_WEIGHTS_NVFP4) {
            g.w_type = FP4;
            g.wscale[0] = L.g0; g.wscale[1] = L.g1;
            g.wbs[0] = static_cast<const uint8_t*>(L.s0); g.wbs[1] = static_cast<const uint8_t*>(L.s1);
        }
        g.y = L.y; g.ldy = L.ldy;
        g.resid = L.resid; g.ldr = L.ldr;
        g.pval = d.pval; g.pidx = d.pidx; g.logits = L.logits; g.ldl = L.ldl;
        g.w_grp = L.w_grp; g.w_grp_stride = L.w_grp_stride; g.w_row0 = L.w_row0;
        g.a_grp = L.a_grp; g.a_grp_stride = L.a_grp_stride;
        g.err = d.err;
        const cudaError_t e = traced(d, kind, st, [&] { return launch_gemv(g, L.epi, d.num_sms, st); });
        if (L.epi == EPI_ARGMAX) d.npart = g.npart;   // partials per row that this launch wrote
        return e;
    }
    TcParams p;
    memset(&p, 0, sizeof(p));
    int bn = tc_pick_bn(L.M);
    const bool glu = L.epi == EPI_GLU;
    const void* w0 = L.w0;
    const void* w1 = L.w1;
    const long r0 = glu ? L.N : L.n0rows, r1 = glu ? L.N : L.n1rows;
    if (L.wq != EAGLE3_WEIGHTS_DTYPE) {
        // quantized weights: expand the codes to bf16 (decoded value times its scales, rounded) in the
        // workspace; the GEMM then runs as for a bf16 head
        if (!d.wdq || (size_t)(r0 + (L.w1 ? r1 : 0)) * L.K > quant_max_matrix(d.cfg) || (L.w1 && !L.s1))
            return cudaErrorInvalidValue;
        auto expand = [&](const void* codes, const void* sc, const float* gs, long rows, bf16_t* out) {
            return traced(d, K_DEQUANT, st, [&] {
                if (L.wq == EAGLE3_WEIGHTS_FP8)
                    return launch_dequant_e4m3(static_cast<const uint8_t*>(codes), static_cast<const float*>(sc),
                                               rows, L.K, out, d.num_sms, st);
                return launch_dequant_nvfp4(static_cast<const uint8_t*>(codes), static_cast<const uint8_t*>(sc), gs,
                                            rows, L.K, out, d.num_sms, st);
            });
        };
        E3_TRY(expand(L.w0, L.s0, L.g0, r0, d.wdq));
        w0 = d.wdq;
        if (L.w1) {
            E3_TRY(expand(L.w1, L.s1, L.g1, r1, d.wdq + r0 * L.K));
            w1 = d.wdq + r0 * L.K;
        }
    }
    if (!make_tma_2d(&p.mw[0], w0, r0, L.K, L.K, 128)) return cudaErrorInvalidValue;
    if (w1 && !make_tma_2d(&p.mw[1], w1, r1, L.K, L.K, 128)) return cudaErrorInvalidValue;
    p.np0 = L.w1 && !glu ? L.n0rows : 1 << 30;
    p.N = L.N; p.M = L.M; p.K = L.K;
    p.kseg[0] = L.na > 1 ? L.ka[0] / 64 : 1 << 30;
    p.kseg[1] = L.na > 2 ? (L.ka[0] + L.ka[1]) / 64 : 1 << 30;
    p.epi = L.epi;
    p.y = L.y; p.ldy = L.ldy; p.ybf = L.ybf; p.ldybf = L.ldybf;
    p.resid = L.resid; p.ldr = L.ldr;
    p.part = d.tc_part;
    p.pval = d.pval; p.pidx = d.pidx; p.logits = L.logits; p.ldl = L.ldl;
    p.err = d.err;
    p.nbatch = 1;
    int splits = L.epi == EPI_ARGMAX ? 1 : tc_splits(d, L.M, L.N, L.K, bn, glu);
    // Large problems take 256 weight rows per CTA: the staged activation tile then feeds two MMAs,
    // halving the shared-memory traffic per FLOP, which bounds 128-row tiles on long-K layers.
    // Persistent CTAs (one per SM, the next tile's loads and MMAs overlapping this tile's epilogue) for
    // unsplit one-matrix GEMMs with more tiles than SMs whose epilogue is a large share of a tile: the
    // lm_head's argmax, short K, or a single token tile (decode batches).
    long tiles = (long)((L.N + 127) / 128) * ((L.M + bn - 1) / bn);
    const bool persist = !glu && splits == 1 && tiles > d.num_sms && (L.epi == EPI_ARGMAX || L.K <= 2048 || L.M <= bn);
    const long pair_tiles = (long)((L.N + 255) / 256) * ((L.M + bn - 1) / bn);
    if (persist) {
        // one token tile of up to 256 rows leaves each CTA one or two weight tiles, so half of them idle
        // through the last; narrower token tiles (down to 64 rows) give every CTA four or more (batch 256:
        // q_b 44 -> 38 us).  Not for the argmax epilogue, whose per-tile reduction then runs four times
        // over (batch-256 lm_head 168 -> 181 us).
        while (L.epi != EPI_ARGMAX && bn > 64 && L.M <= bn && tiles < 4L * d.num_sms) {
            bn /= 2;
            tiles = (long)((L.N + 127) / 128) * ((L.M + bn - 1) / bn);
        }
        p.persist = d.num_sms;
    } else if (!glu && L.epi != EPI_ARGMAX && bn == 256 && pair_tiles >= 2L * d.num_sms) {
        p.pair = 1;
        splits = 1;
    }
    for (int i = 0; i < L.na; ++i)
        if (!make_tma_2d(&p.mx[i], L.a16[i], L.M, L.ka[i], L.lda[i], bn)) return cudaErrorInvalidValue;
    cudaError_t e = traced(d, kind, st, [&] { return launch_tc_gemm(p, bn, splits, st); });
    if (L.epi == EPI_ARGMAX) d.npart = p.npart;
    return e;
}

// Marks L's weights as the head's quantized matrices m0 (and m1, the second segment or the up matrix) with
// scales s0 / s1; nothing for a head with dtype weights.
void quant(const eagle3_draft& d, Lin& L, int m0, const void* s0, int m1 = -1, const void* s1 = nullptr) {
    if (!quant_head(d.cfg)) return;
    L.wq = d.cfg.weight_format;
    L.s0 = s0; L.s1 = s1;
    if (L.wq == EAGLE3_WEIGHTS_NVFP4) {
        L.g0 = d.w.matrix_scales + m0;
        L.g1 = m1 >= 0 ? d.w.matrix_scales + m1 : nullptr;
    }
}

Lin lin1(const eagle3_draft& d, int M, const float* a32, const bf16_t* a16, int K, const void* w, int N) {
    Lin L;
    L.M = M; L.N = N; L.K = K;
    L.a32[0] = a32; L.a16[0] = a16; L.lda[0] = K; L.ka[0] = K;
    L.w0 = w; L.n0rows = N;
    (void)d;
    return L;
}

// Per-head batched tensor-core GEMM: for head h, out[:, h*ycol + n] = X[:, h*kx : h*kx + K] W_h^T with
// W_h the rows [h*wrows_stride + wrow0, + N) of `w` (row length K).
cudaError_t run_batched(eagle3_draft& d, int kind, int M, const bf16_t* x, long ldx, int kx_per_head, const void* w,
                        long wrows_total, int wrow0, int wrows_stride, int N, int K, float* y, bf16_t* ybf, long ldy,
                        long ycol, cudaStream_t st) {
    TcParams p;
    memset(&p, 0, sizeof(p));
    const int bn = tc_pick_bn(M);
    // the map starts at row wrow0 so that batch h's tile row is h * wrows_stride
    const bf16_t* wb = reinterpret_cast<const bf16_t*>(w) + (long)wrow0 * K;
    if (!make_tma_2d(&p.mw[0], wb, wrows_total - wrow0, K, K, 128)) return cudaErrorInvalidValue;
    if (!make_tma_2d(&p.mx[0], x, M, ldx, ldx, bn)) return cudaErrorInvalidValue;
    p.np0 = 1 << 30;
    p.N = N; p.M = M; p.K = K;
    p.kseg[0] = p.kseg[1] = 1 << 30;
    p.epi = EPI_STORE;
    p.y = y; p.ldy = ldy; p.ybf = ybf; p.ldybf = ldy;
    p.err = d.err;
    p.nbatch = d.cfg.n_heads;
    p.bw_rows = wrows_stride;
    p.bq_kb = kx_per_head / 64;
    p.by_col = ycol;
    return traced(d, kind, st, [&] { return launch_tc_gemm(p, bn, 1, st); });
}

// The decoder chain from the concatenated input x to h2.
// fused: the residual stream of the rows (fc output in extend, the carried hidden in decode).
// Unabsorbed causal attention of a long extend: rotate q_pe in the bf16 query rows, gather and expand
// every live slot's keys and values once, then flash-attention tiles write o_h per head (bf16).
cudaError_t run_prefill_attention(eagle3_draft& d, eagle3_kv_t* kv, int M, int batch, const int32_t* row_offsets,
                                  cudaStream_t st) {
    const eagle3_config_t& c = d.cfg;
    const int nh = c.n_heads, dkv = c.qk_nope_dim + c.v_head_dim;
    PrefillArgs pa;
    memset(&pa, 0, sizeof(pa));
    pa.M = M; pa.B = batch; pa.nh = nh; pa.max_ctx = c.max_ctx;
    pa.page_size = c.page_size; pa.max_pages = c.max_pages_per_seq; pa.num_pages = kv->num_pages;
    pa.sigma = attention_scale(c);
    pa.row_offsets = row_offsets; pa.row_pos = d.row_pos; pa.block_table = kv->block_table; pa.cache = kv->data;
    pa.xc = d.xc; pa.xpe = d.xpe; pa.kv = d.kvx; pa.q = d.q_bf; pa.qf = nullptr;
    pa.rope_cos = d.rope_cos; pa.rope_sin = d.rope_sin;
    pa.tiles = d.tiles; pa.o_bf = d.o_bf; pa.err = d.err;
    // 128-row query tiles on tcgen05; the mma.sync kernel (64-row tiles) where TMA cannot address the rows
    pa.bq = 128;
    const bool tc_pf = prefill_tc_supported(pa);
    if (!tc_pf) pa.bq = 64;
    pa.ntiles_cap = prefill_tiles_cap(M, batch, pa.bq);
    if (pa.ntiles_cap > d.tiles_cap) return cudaErrorInvalidValue;
    E3_TRY(traced(d, K_ROPE_Q, st, [&] { return launch_rope_q_rows(pa, st); }));
    E3_TRY(traced(d, K_KV_GATHER, st, [&] { return launch_kv_gather(pa, st); }));
    {
        Lin L = lin1(d, batch * c.max_ctx, nullptr, d.xc, c.kv_lora_rank, d.w.kv_b, nh * dkv);
        L.ybf = d.kvx; L.ldybf = (long)nh * dkv;
        E3_TRY(run_linear(d, L, K_KV_EXPAND, st));
    }
    E3_TRY(traced(d, K_PREFILL_TILES, st, [&] { return launch_prefill_tiles(pa, st); }));
    return traced(d, K_ATTN, st, [&] { return tc_pf ? launch_prefill_tc(pa, st) : launch_prefill_attention(pa, st); });
}

// The MLA attention block of a layer: q_a | kv_a, latent norms and cache append, q_b, then absorbed
// attention (or, for a long extend, the unabsorbed path); leaves o (GEMV path) or o_bf (tensor-core path).
cudaError_t run_attention_mla(eagle3_draft& d, eagle3_kv_t* kv, int M, cudaStream_t st, int batch,
                              const int32_t* row_offsets) {
    const eagle3_config_t& c = d.cfg;
    const eagle3_weights_t& w = d.w;
    const int H = c.hidden, dq = c.q_lora_rank, dc = c.kv_lora_rank, dr = c.qk_rope_dim, dn = c.qk_nope_dim;
    const int nh = c.n_heads, dqk = dn + dr, D = dc + dr, dv = c.v_head_dim;
    const bool tc = use_tc(d, M);
    RowArgs ra = row_args(d, kv);
    // q_a | kv_a over the 2H input
    {
        Lin L = lin1(d, M, d.x, d.x_bf, 2 * H, w.q_a, dq + D);
        L.w1 = w.kv_a; L.n0rows = dq; L.n1rows = D;
        quant(d, L, QM_QA, w.q_a_scale, QM_KVA, w.kv_a_scale);
        L.y = d.cqkv; L.ldy = dq + D;
        E3_TRY(run_linear(d, L, K_QKV_A, st));
    }
    E3_TRY(traced(d, K_LATENT, st, [&] {
        return launch_latent(ra, M, d.cqkv, w.q_a_norm, w.kv_a_norm, d.rope_cos, d.rope_sin, d.row_seq, d.row_pos,
                             kv->block_table, kv->data, d.cq_hat, tc ? d.cqh_bf : nullptr, st);
    }));
    {
        Lin L = lin1(d, M, d.cq_hat, d.cqh_bf, dq, w.q_b, nh * dqk);
        quant(d, L, QM_QB, w.q_b_scale);
        // the tensor-core path keeps only the bf16 rows: every consumer (absorb GEMM, rope, attention)
        // reads bf16
        if (tc) { L.ybf = d.q_bf; L.ldybf = (long)nh * dqk; } else { L.y = d.q; L.ldy = (long)nh * dqk; }
        E3_TRY(run_linear(d, L, K_Q_B, st));
    }
    const bool prefill = d.tiles && row_offsets && M >= kPrefillMinRows && 2L * M >= (long)batch * c.max_ctx;
    if (prefill) {
        E3_TRY(run_prefill_attention(d, kv, M, batch, row_offsets, st));
    } else {
        AttnArgs aa;
        memset(&aa, 0, sizeof(aa));
        aa.M = M; aa.nh = nh; aa.dn = dn; aa.dr = dr; aa.dc = dc; aa.dv = dv;
        aa.sigma = attention_scale(c);
        aa.page_size = c.page_size; aa.max_pages = c.max_pages_per_seq; aa.num_pages = kv->num_pages; aa.err = d.err;
        const bool tc_attn = attention_tc_ok(d, M);
        if (tc_attn) attn_plan_tc(d, M, &aa.splits, &aa.chunk);
        else attn_plan(d, M, &aa.splits, &aa.chunk);
        aa.dt = ra.dt;
        aa.row_seq = d.row_seq; aa.row_pos = d.row_pos; aa.block_table = kv->block_table;
        aa.cache = kv->data; aa.kv_b = w.kv_b; aa.q = d.q; aa.rope_cos = d.rope_cos; aa.rope_sin = d.rope_sin;
        aa.qa = tc ? nullptr : d.qa; aa.qa_bf = ra.dt == BF16 ? d.qa_bf : nullptr;
        aa.q_bf = tc ? d.q_bf : nullptr;
        aa.part_o = d.part_o; aa.part_ml = d.part_ml; aa.o = d.o;
        if (tc) {
            // rope part, then q_lat,h = q_nope,h W_UK,h as a per-head GEMM against the transposed key weights
            E3_TRY(traced(d, K_ROPE_Q, st, [&] { return launch_rope_q(aa, st); }));
            E3_TRY(run_batched(d, K_ABSORB, M, d.q_bf, (long)nh * dqk, dqk, d.wukt, (long)nh * dc, 0, dc, dc, dn,
                               nullptr, d.qa_bf, (long)nh * D, D, st));
        } else {
            E3_TRY(traced(d, K_ABSORB, st, [&] { return launch_absorb(aa, st); }));
        }
        // o_lat: written by the attention kernel itself for a single split, else by the split merge; then
        // o_h = W_UV,h o_lat,h over the value rows of kv_b
        if (tc) aa.olat_bf = d.olat_bf; else aa.olat = d.olat;
        // few rows with split partials: the merge and the value up-projection in one kernel (more than 64
        // splits only there)
        bool fused = !tc && aa.splits > 1 && merge_unabsorb_supported(aa);
        if (!fused && aa.splits > 64) {
            aa.splits = 64;
            fused = !tc && merge_unabsorb_supported(aa);
        }
        E3_TRY(traced(d, K_ATTN, st, [&] { return tc_attn ? launch_attention_tc(aa, st) : launch_attention(aa, st); }));
        if (fused) {
            E3_TRY(traced(d, K_UNABSORB, st, [&] { return launch_merge_unabsorb(aa, st); }));
            return cudaSuccess;
        }
        if (aa.splits > 1) E3_TRY(traced(d, K_COMBINE, st, [&] { return launch_merge(aa, st); }));
        if (tc) {
            E3_TRY(run_batched(d, K_UNABSORB, M, d.olat_bf, (long)nh * dc, dc, w.kv_b, (long)nh * (dn + dv), dn, dn + dv,
                               dv, dc, nullptr, d.o_bf, (long)nh * dv, dv, st));
        } else {
            Lin L = lin1(d, M, d.olat, nullptr, dc, w.kv_b, nh * dv);
            L.lda[0] = (long)nh * dc;
            L.w_grp = dv; L.w_grp_stride = dn + dv; L.w_row0 = dn;
            L.a_grp = dv; L.a_grp_stride = dc;
            L.y = d.o; L.ldy = (long)nh * dv;
            E3_TRY(run_linear(d, L, K_UNABSORB, st));
        }
    }
    return cudaSuccess;
}

// Split plan of the MHA attention: 128-slot chunks (one 32-slot tile per warp), doubled while the
// (row, key/value head, split) CTAs exceed about 8 per SM, the rows' splits exceed the partials, or a
// row has more splits than the merge stages (1024).
void mha_plan(const eagle3_draft& d, int M, int* splits, int* chunk) {
    const int ctx = d.cfg.max_ctx;
    auto ns = [&](int ch) { return (ctx + ch - 1) / ch; };
    int ch = 128;
    while (ns(ch) > 1 && ((long)M * d.cfg.n_kv_heads * ns(ch) > 8L * d.num_sms || (size_t)M * ns(ch) > d.part_rows ||
                          ns(ch) > 1024))
        ch *= 2;
    *chunk = ch;
    *splits = ns(ch);
}

// The MHA attention block ("Eagle3 DeepseekV3 in MAX" §11): q and k | v projections at 2H input, rotate-
// half RoPE with the cache append, grouped-query attention over the head's own cache and the split
// merge; leaves o (GEMV path) or o_bf (tensor-core path).
cudaError_t run_attention_mha(eagle3_draft& d, eagle3_kv_t* kv, int M, cudaStream_t st) {
    const eagle3_config_t& c = d.cfg;
    const eagle3_weights_t& w = d.w;
    const int H = c.hidden, nh = c.n_heads, nkv = c.n_kv_heads, hd = c.head_dim;
    const bool tc = use_tc(d, M);
    {
        Lin L = lin1(d, M, d.x, d.x_bf, 2 * H, w.q_proj, nh * hd);
        L.y = d.q; L.ldy = (long)nh * hd;
        E3_TRY(run_linear(d, L, K_Q_B, st));
    }
    {
        Lin L = lin1(d, M, d.x, d.x_bf, 2 * H, w.k_proj, 2 * nkv * hd);
        L.w1 = w.v_proj; L.n0rows = nkv * hd; L.n1rows = nkv * hd;
        L.y = d.cqkv; L.ldy = 2L * nkv * hd;
        E3_TRY(run_linear(d, L, K_QKV_A, st));
    }
    MhaArgs ma;
    memset(&ma, 0, sizeof(ma));
    ma.M = M; ma.nh = nh; ma.nkv = nkv; ma.d = hd;
    ma.sigma = attention_scale(c);
    ma.page_size = c.page_size; ma.max_pages = c.max_pages_per_seq; ma.num_pages = kv->num_pages;
    ma.dt = c.dtype == EAGLE3_BF16 ? BF16 : F32;
    ma.row_seq = d.row_seq; ma.row_pos = d.row_pos; ma.block_table = kv->block_table; ma.cache = kv->data;
    ma.q = d.q; ma.kv = d.cqkv; ma.rope_cos = d.rope_cos; ma.rope_sin = d.rope_sin;
    ma.part_o = d.part_o; ma.part_ml = d.part_ml;
    if (tc) ma.o_bf = d.o_bf; else ma.o = d.o;
    ma.err = d.err;
    mha_plan(d, M, &ma.splits, &ma.chunk);
    E3_TRY(traced(d, K_LATENT, st, [&] { return launch_mha_rope_append(ma, st); }));
    E3_TRY(traced(d, K_ATTN, st, [&] { return launch_mha_attention(ma, st); }));
    if (ma.splits > 1) E3_TRY(traced(d, K_COMBINE, st, [&] { return launch_mha_merge(ma, st); }));
    return cudaSuccess;
}

// One decoder layer over M rows: the attention block of the head's kind, then o_proj with the residual,
// the post-attention norm and the dense SiLU MLP.  row_offsets (extend only) lets a long extend of an
// MLA head take the unabsorbed attention path.
cudaError_t run_layer(eagle3_draft& d, eagle3_kv_t* kv, int M, const float* fused, cudaStream_t st, int batch = 0,
                      const int32_t* row_offsets = nullptr) {
    const eagle3_config_t& c = d.cfg;
    const eagle3_weights_t& w = d.w;
    const int H = c.hidden, I = c.intermediate;
    const int w_o = mha_head(c) ? c.n_heads * c.head_dim : c.n_heads * c.v_head_dim;
    const bool tc = use_tc(d, M);
    RowArgs ra = row_args(d, kv);
    if (mha_head(c)) E3_TRY(run_attention_mha(d, kv, M, st));
    else E3_TRY(run_attention_mla(d, kv, M, st, batch, row_offsets));
    // o_proj + residual
    {
        Lin L = lin1(d, M, d.o, d.o_bf, w_o, w.o, H);
        quant(d, L, QM_O, w.o_scale);
        L.epi = EPI_RESID; L.resid = fused; L.ldr = H;
        L.y = d.h1; L.ldy = H;
        E3_TRY(run_linear(d, L, K_O_PROJ, st));
    }
    E3_TRY(traced(d, K_POST_NORM, st, [&] {
        // the tensor-core GEMM reads only the bf16 copy
        return launch_rmsnorm(M, H, c.rms_eps, ra.dt, d.h1, w.post_attn_norm, tc ? nullptr : d.y, tc ? d.y_bf : nullptr,
                              st);
    }));
    {
        Lin L = lin1(d, M, d.y, d.y_bf, H, w.gate, I);
        L.epi = EPI_GLU; L.w1 = w.up; L.n1rows = I;
        quant(d, L, QM_GATE, w.gate_scale, QM_UP, w.up_scale);
        if (tc) { L.ybf = d.m_bf; L.ldybf = I; } else { L.y = d.mlp; L.ldy = I; }
        E3_TRY(run_linear(d, L, K_GATE_UP, st));
    }
    {
        Lin L = lin1(d, M, d.mlp, d.m_bf, I, w.down, H);
        quant(d, L, QM_DOWN, w.down_scale);
        L.epi = EPI_RESID; L.resid = d.h1; L.ldr = H;
        L.y = d.h2; L.ldy = H;
        E3_TRY(run_linear(d, L, K_DOWN, st));
    }
    return cudaSuccess;
}

cudaError_t run_head(eagle3_draft& d, int batch, float* logits_out, cudaStream_t st) {
    Lin L = lin1(d, batch, d.z, d.z_bf, d.cfg.hidden, d.w.lm_head, d.cfg.draft_vocab);
    quant(d, L, QM_LM, d.w.lm_head_scale);
    L.epi = EPI_ARGMAX; L.logits = logits_out; L.ldl = d.cfg.draft_vocab;
    L.force_tc = head_tc(d, batch);
    return run_linear(d, L, K_LM_HEAD, st);
}

bool kv_ok(const eagle3_kv_t* kv) {
    return kv && kv->data && kv->block_table && kv->lengths && kv->num_pages > 0;
}

}  // namespace

extern "C" {

const char* eagle3_status_string(eagle3_status_t s) {
    switch (s) {
        case EAGLE3_OK: return "ok";
        case EAGLE3_ERR_INVALID_ARG: return "invalid argument";
        case EAGLE3_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case EAGLE3_ERR_STATE: return "invalid state (decode before extend?)";
        case EAGLE3_ERR_OOM: return "out of device memory";
        case EAGLE3_ERR_CUDA: return "CUDA error";
        case EAGLE3_ERR_DEVICE_RANGE: return "device-side range error";
        case EAGLE3_ERR_SCRATCH_LIMIT: return "M * N exceeds the fixed scratch of eagle3_linear_noalloc";
    }
    return "unknown status";
}

int32_t eagle3_last_cuda_error(void) { return g_last_cuda_error; }

eagle3_status_t eagle3_draft_workspace_bytes(const eagle3_config_t* config, size_t* bytes) {
    eagle3_status_t s = check_config(config);
    if (s != EAGLE3_OK) return s;
    if (!bytes) return EAGLE3_ERR_INVALID_ARG;
    *bytes = plan(*config, 152).total;
    return EAGLE3_OK;
}

eagle3_status_t eagle3_draft_create(const eagle3_config_t* config, const eagle3_weights_t* weights,
                                    eagle3_draft_t** out) {
    if (!out) return EAGLE3_ERR_INVALID_ARG;
    *out = nullptr;
    eagle3_status_t s = check_config(config);
    if (s != EAGLE3_OK) return s;
    if ((s = check_weights(*config, weights)) != EAGLE3_OK) return s;
    eagle3_draft* d = new (std::nothrow) eagle3_draft();
    if (!d) return EAGLE3_ERR_OOM;
    d->cfg = *config;
    d->w = *weights;
    cudaError_t e = cudaGetDevice(&d->device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d->num_sms, cudaDevAttrMultiProcessorCount, d->device);
    if (e != cudaSuccess) { delete d; return cuda_fail(e); }
    Offsets o = plan(d->cfg, d->num_sms);
    e = cudaMalloc(&d->ws, o.total);
    if (e != cudaSuccess) {
        g_last_cuda_error = (int)e;
        cudaGetLastError();
        delete d;
        return EAGLE3_ERR_OOM;
    }
    d->ws_bytes = o.total;
    d->m_cap = o.m_cap;
    d->splits_cap = o.splits_cap;
    d->npart = o.npart;
    d->part_rows = o.part_rows;
    d->tc_ok = tc_supported(d->cfg);
    char* base = (char*)d->ws;
    auto F = [&](size_t off) { return (float*)(base + off); };
    auto Bf = [&](size_t off) { return (bf16_t*)(base + off); };
    auto I = [&](size_t off) { return (int*)(base + off); };
    d->f = F(o.f); d->carry = F(o.carry); d->x = F(o.x); d->cqkv = F(o.cqkv); d->cq_hat = F(o.cq_hat);
    d->q = F(o.q); d->qa = F(o.qa); d->qa_bf = Bf(o.qa_bf); d->part_o = F(o.part_o); d->part_ml = F(o.part_ml);
    d->o = F(o.o); d->h1 = F(o.h1); d->y = F(o.y); d->mlp = F(o.mlp); d->h2 = F(o.h2); d->z = F(o.z);
    d->pval = F(o.pval); d->pidx = I(o.pidx); d->rope_cos = F(o.rope_cos); d->rope_sin = F(o.rope_sin);
    d->row_seq = I(o.row_seq); d->row_pos = I(o.row_pos); d->d0 = I(o.d0); d->tok_in = I(o.tok_in);
    d->err = I(o.err); d->olat = F(o.olat);
    d->x_bf = Bf(o.x_bf); d->cqh_bf = Bf(o.cqh_bf); d->q_bf = Bf(o.q_bf); d->olat_bf = Bf(o.olat_bf);
    d->o_bf = Bf(o.o_bf); d->y_bf = Bf(o.y_bf); d->m_bf = Bf(o.m_bf); d->z_bf = Bf(o.z_bf); d->wukt = Bf(o.wukt);
    d->tc_part = F(o.tc_part);
    d->xc = Bf(o.xc); d->xpe = Bf(o.xpe); d->kvx = Bf(o.kvx);
    d->logits = F(o.logits);
    d->tiles = o.tiles_cap ? reinterpret_cast<int4*>(base + o.tiles) : nullptr;
    d->tiles_cap = o.tiles_cap;
    d->wdq = quant_head(d->cfg) && d->tc_ok && o.m_cap > kGemvMaxRows ? Bf(o.wdq) : nullptr;
    std::vector<float> cs, sn;
    yarn_table(d->cfg, cs, sn);
    e = cudaMemcpy(d->rope_cos, cs.data(), cs.size() * sizeof(float), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(d->rope_sin, sn.data(), sn.size() * sizeof(float), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemset(d->err, 0, sizeof(int));
    if (e == cudaSuccess) e = cudaMemset(d->carry, 0, (size_t)d->cfg.max_batch * d->cfg.hidden * sizeof(float));
    if (e == cudaSuccess && d->tc_ok && !mha_head(d->cfg))
        e = launch_transpose_wuk(d->w.kv_b, d->cfg.n_heads, d->cfg.qk_nope_dim, d->cfg.v_head_dim,
                                 d->cfg.kv_lora_rank, d->wukt, 0);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        cudaFree(d->ws);
        delete d;
        return cuda_fail(e);
    }
    *out = d;
    return EAGLE3_OK;
}

eagle3_status_t eagle3_draft_extend(eagle3_draft_t* d, const void* const aux_hidden[3], const int32_t* tokens,
                                    const int32_t* positions, const int32_t* row_offsets, int32_t batch,
                                    int32_t num_tokens, eagle3_kv_t* cache, float* hidden_out, float* logits_out,
                                    void* stream) {
    if (!d || !aux_hidden || !tokens || !positions || !row_offsets || !kv_ok(cache)) return EAGLE3_ERR_INVALID_ARG;
    const eagle3_config_t& c = d->cfg;
    const int nfc = fc_inputs(c);
    for (int i = 0; i < nfc; ++i)
        if (!aux_hidden[i] || !aligned16(aux_hidden[i])) return EAGLE3_ERR_INVALID_ARG;
    if (batch < 1 || batch > c.max_batch || num_tokens < batch || num_tokens > c.max_tokens_per_extend)
        return EAGLE3_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    const int H = c.hidden, M = num_tokens;
    const bool tc = use_tc(*d, M);
    RowArgs ra = row_args(*d, cache);
    // fc: f = [a_early | a_mid | a_late] W_fc^T  (3H -> H, no bias; an MHA head may fuse two states)
    {
        Lin L;
        L.M = M; L.N = H; L.K = nfc * H; L.na = nfc;
        for (int i = 0; i < nfc; ++i) {
            L.a32[i] = aux_hidden[i];
            L.a16[i] = (const bf16_t*)aux_hidden[i];
            L.lda[i] = H; L.ka[i] = H;
        }
        L.a32_is_bf16 = ra.dt == BF16;
        L.w0 = d->w.fc; L.n0rows = H;
        quant(*d, L, QM_FC, d->w.fc_scale);
        L.y = d->f; L.ldy = H;
        E3_CUDA(run_linear(*d, L, K_FC, st));
    }
    E3_CUDA(traced(*d, K_EMBED, st, [&] {
        return launch_embed_norms(ra, false, M, tokens, positions, row_offsets, batch, nullptr, nullptr, d->f,
                                  d->w.embed, d->w.input_norm, d->w.hidden_norm, tc ? nullptr : d->x, tc ? d->x_bf : nullptr,
                                  d->row_seq, d->row_pos, st);
    }));
    E3_CUDA(run_layer(*d, cache, M, d->f, st, batch, row_offsets));
    const bool tch = head_tc(*d, batch);
    E3_CUDA(traced(*d, K_FINAL, st, [&] {
        return launch_final(ra, true, batch, M, row_offsets, d->h2, d->w.final_norm, d->row_pos, d->carry, d->z,
                            tch ? d->z_bf : nullptr, hidden_out, cache->lengths, st);
    }));
    E3_CUDA(run_head(*d, batch, logits_out, st));
    E3_CUDA(traced(*d, K_ARGMAX, st, [&] {
        return launch_argmax_final(batch, d->npart, d->pval, d->pidx, 0, nullptr, c.target_vocab, d->d0, nullptr, 0,
                                   0, nullptr, d->err, st);
    }));
    d->batch = batch;
    d->have_extend = true;
    return EAGLE3_OK;
}

eagle3_status_t eagle3_draft_decode(eagle3_draft_t* d, int32_t gamma, const int32_t* d2t, eagle3_kv_t* cache,
                                    int32_t* draft_tokens, float* hidden_out, float* logits_out, void* stream) {
    if (!d || !draft_tokens || !kv_ok(cache)) return EAGLE3_ERR_INVALID_ARG;
    if (gamma < 1 || gamma > 64) return EAGLE3_ERR_INVALID_ARG;
    if (!d->have_extend) return EAGLE3_ERR_STATE;
    const eagle3_config_t& c = d->cfg;
    cudaStream_t st = (cudaStream_t)stream;
    const int B = d->batch, H = c.hidden;
    const bool tc = use_tc(*d, B);
    RowArgs ra = row_args(*d, cache);
    E3_CUDA(traced(*d, K_EMIT, st, [&] {
        return launch_emit_first(B, d->d0, d2t, c.target_vocab, draft_tokens, gamma, d->tok_in, d->err, st);
    }));
    for (int s = 1; s < gamma; ++s) {
        E3_CUDA(traced(*d, K_EMBED, st, [&] {
            return launch_embed_norms(ra, true, B, nullptr, nullptr, nullptr, B, d->tok_in, cache->lengths, d->carry,
                                      d->w.embed, d->w.input_norm, d->w.hidden_norm, tc ? nullptr : d->x, tc ? d->x_bf : nullptr,
                                      d->row_seq, d->row_pos, st);
        }));
        E3_CUDA(run_layer(*d, cache, B, d->carry, st));
        float* ho = hidden_out ? hidden_out + (size_t)(s - 1) * B * H : nullptr;
        float* lo = logits_out ? logits_out + (size_t)(s - 1) * B * c.draft_vocab : nullptr;
        E3_CUDA(traced(*d, K_FINAL, st, [&] {
            return launch_final(ra, false, B, B, nullptr, d->h2, d->w.final_norm, d->row_pos, d->carry, d->z,
                                head_tc(*d, B) ? d->z_bf : nullptr, ho, cache->lengths, st);
        }));
        E3_CUDA(run_head(*d, B, lo, st));
        E3_CUDA(traced(*d, K_ARGMAX, st, [&] {
            return launch_argmax_final(B, d->npart, d->pval, d->pidx, 1, d2t, c.target_vocab, nullptr, draft_tokens,
                                       gamma, s, d->tok_in, d->err, st);
        }));
    }
    return EAGLE3_OK;
}

namespace {
bool sampling_ok(const eagle3_sampling_t* p) {
    return p && p->temperature >= 0.f && p->top_k >= 0 && p->top_k <= 1024 && p->top_p > 0.f && p->top_p <= 1.f &&
           !(p->temperature > 0.f && p->top_k == 0 && p->top_p < 1.f);
}
}  // namespace

eagle3_status_t eagle3_draft_decode_sampled(eagle3_draft_t* d, int32_t gamma, const int32_t* d2t,
                                            eagle3_kv_t* cache, const eagle3_sampling_t* params,
                                            const float* first_logits, const float* uniforms, int32_t* draft_tokens,
                                            float* draft_probs, int32_t probs_len, int32_t probs_in_target,
                                            float* hidden_out, float* logits_out, void* stream) {
    if (!d || !draft_tokens || !first_logits || !uniforms || !kv_ok(cache) || !sampling_ok(params))
        return EAGLE3_ERR_INVALID_ARG;
    if (gamma < 1 || gamma > 64) return EAGLE3_ERR_INVALID_ARG;
    if (!d->have_extend) return EAGLE3_ERR_STATE;
    const eagle3_config_t& c = d->cfg;
    const int B = d->batch, H = c.hidden, Vd = c.draft_vocab;
    if (draft_probs && probs_len < (probs_in_target && d2t ? c.target_vocab : Vd)) return EAGLE3_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    const bool tc = use_tc(*d, B);
    RowArgs ra = row_args(*d, cache);
    // step s draws with uniforms[s] from the step's logits: the extend's for s = 0, else the decode step's
    auto sample = [&](int s, const float* logits) {
        SampleArgs sa;
        memset(&sa, 0, sizeof(sa));
        sa.logits = logits; sa.ldl = Vd; sa.rows = B; sa.V = Vd;
        sa.temperature = params->temperature; sa.top_k = params->top_k; sa.top_p = params->top_p;
        sa.uniforms = uniforms + (size_t)s * B; sa.d2t = d2t; sa.target_vocab = c.target_vocab;
        sa.tokens = d->tok_in; sa.tokens2 = draft_tokens + s; sa.tok2_stride = gamma;
        // [batch, gamma, probs_len]: the layout eagle3_accept_residual reads
        sa.probs = draft_probs ? draft_probs + (size_t)s * probs_len : nullptr; sa.ldp = (long)gamma * probs_len;
        sa.probs_len = probs_len; sa.probs_target = probs_in_target ? 1 : 0;
        sa.err = d->err;
        return traced(*d, K_SAMPLE, st, [&] { return launch_sample(sa, st); });
    };
    E3_CUDA(sample(0, first_logits));
    for (int s = 1; s < gamma; ++s) {
        E3_CUDA(traced(*d, K_EMBED, st, [&] {
            return launch_embed_norms(ra, true, B, nullptr, nullptr, nullptr, B, d->tok_in, cache->lengths, d->carry,
                                      d->w.embed, d->w.input_norm, d->w.hidden_norm, tc ? nullptr : d->x, tc ? d->x_bf : nullptr,
                                      d->row_seq, d->row_pos, st);
        }));
        E3_CUDA(run_layer(*d, cache, B, d->carry, st));
        float* ho = hidden_out ? hidden_out + (size_t)(s - 1) * B * H : nullptr;
        float* lo = logits_out ? logits_out + (size_t)(s - 1) * B * Vd : d->logits;
        E3_CUDA(traced(*d, K_FINAL, st, [&] {
            return launch_final(ra, false, B, B, nullptr, d->h2, d->w.final_norm, d->row_pos, d->carry, d->z,
                                head_tc(*d, B) ? d->z_bf : nullptr, ho, cache->lengths, st);
        }));
        {
            Lin L = lin1(*d, B, d->z, d->z_bf, H, d->w.lm_head, Vd);
            quant(*d, L, QM_LM, d->w.lm_head_scale);
            L.y = lo; L.ldy = Vd;
            E3_CUDA(run_linear(*d, L, K_LM_HEAD, st));
        }
        E3_CUDA(sample(s, lo));
    }
    return EAGLE3_OK;
}

eagle3_status_t eagle3_linear(eagle3_draft_t* d, const void* x, const void* w, float* y, int32_t M, int32_t N,
                              int32_t K, void* stream) {
    if (!d || !x || !w || !y || M < 1 || N < 1 || K < 8 || K % 8) return EAGLE3_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w) || !aligned16(y)) return EAGLE3_ERR_INVALID_ARG;
    if (d->cfg.dtype != EAGLE3_BF16) return EAGLE3_ERR_UNSUPPORTED;
    if (use_tc(*d, M) && K % 64) return EAGLE3_ERR_UNSUPPORTED;
    Lin L;
    L.M = M; L.N = N; L.K = K; L.na = 1;
    L.a32[0] = x; L.a32_is_bf16 = true; L.a16[0] = (const bf16_t*)x; L.lda[0] = K; L.ka[0] = K;
    L.w0 = w; L.n0rows = N;
    L.y = y; L.ldy = N;
    E3_CUDA(run_linear(*d, L, K_FC, (cudaStream_t)stream));
    return EAGLE3_OK;
}

eagle3_status_t eagle3_accept(const int32_t* draft, const int32_t* target, int32_t batch, int32_t gamma,
                              int32_t* accepted_len, int32_t* hist, void* stream) {
    if (!draft || !target || !accepted_len) return EAGLE3_ERR_INVALID_ARG;
    if (batch < 1 || gamma < 1 || gamma > 4096) return EAGLE3_ERR_INVALID_ARG;
    E3_CUDA(launch_accept(draft, target, batch, gamma, accepted_len, hist, (cudaStream_t)stream));
    return EAGLE3_OK;
}

eagle3_status_t eagle3_accept_relaxed(const int32_t* draft, const int32_t* topk_ids, const float* topk_logprobs,
                                      const uint8_t* in_thinking, int32_t batch, int32_t gamma, int32_t k, float delta,
                                      int32_t* accepted_len, int32_t* hist, void* stream) {
    if (!draft || !topk_ids || !topk_logprobs || !accepted_len) return EAGLE3_ERR_INVALID_ARG;
    if (batch < 1 || gamma < 1 || gamma > 4096 || k < 1 || k > 1024 || !(delta >= 0.f)) return EAGLE3_ERR_INVALID_ARG;
    E3_CUDA(launch_accept_relaxed(draft, topk_ids, topk_logprobs, in_thinking, batch, gamma, k, delta, accepted_len,
                                  hist, (cudaStream_t)stream));
    return EAGLE3_OK;
}


eagle3_status_t eagle3_sample(const float* logits, int32_t rows, int32_t V, int64_t ld,
                              const eagle3_sampling_t* params, const float* uniforms, const int32_t* d2t,
                              int32_t target_vocab, int32_t* tokens, float* token_prob, float* probs,
                              int32_t probs_len, int32_t probs_in_target, void* stream) {
    if (!logits || !uniforms || !tokens || rows < 1 || rows > 65535 || V < 1 || V > 131072 || ld < V ||
        !sampling_ok(params))
        return EAGLE3_ERR_INVALID_ARG;
    if (d2t && target_vocab < 1) return EAGLE3_ERR_INVALID_ARG;
    if (probs && probs_len < (probs_in_target && d2t ? target_vocab : V)) return EAGLE3_ERR_INVALID_ARG;
    SampleArgs sa;
    memset(&sa, 0, sizeof(sa));
    sa.logits = logits; sa.ldl = ld; sa.rows = rows; sa.V = V;
    sa.temperature = params->temperature; sa.top_k = params->top_k; sa.top_p = params->top_p;
    sa.uniforms = uniforms; sa.d2t = d2t; sa.target_vocab = d2t ? target_vocab : V;
    sa.tokens = tokens; sa.token_prob = token_prob;
    sa.probs = probs; sa.ldp = probs_len; sa.probs_len = probs_len; sa.probs_target = probs_in_target ? 1 : 0;
    sa.err = nullptr;
    E3_CUDA(launch_sample(sa, (cudaStream_t)stream));
    return EAGLE3_OK;
}

eagle3_status_t eagle3_accept_typical(const int32_t* draft, const float* target_probs, int32_t batch, int32_t gamma,
                                      int32_t V, float epsilon, float delta, int32_t* accepted_len, int32_t* hist,
                                      void* stream) {
    if (!draft || !target_probs || !accepted_len) return EAGLE3_ERR_INVALID_ARG;
    if (batch < 1 || gamma < 1 || gamma > 4096 || V < 1 || !(epsilon >= 0.f) || !(delta >= 0.f))
        return EAGLE3_ERR_INVALID_ARG;
    E3_CUDA(launch_accept_typical(draft, target_probs, batch, gamma, V, epsilon, delta, accepted_len, hist,
                                  (cudaStream_t)stream));
    return EAGLE3_OK;
}

eagle3_status_t eagle3_philox_uniforms(uint64_t seed, uint64_t offset, int64_t n, float* out, void* stream) {
    if (n < 0 || (n > 0 && !out)) return EAGLE3_ERR_INVALID_ARG;
    E3_CUDA(launch_philox_uniforms(seed, offset, (long)n, out, (cudaStream_t)stream));
    return EAGLE3_OK;
}

eagle3_status_t eagle3_accept_residual(const int32_t* draft, const float* draft_probs, const float* target_probs,
                                       const float* u_accept, const float* u_resample, int32_t batch, int32_t gamma,
                                       int32_t V, int32_t* accepted_len, int32_t* next_token, int32_t* hist,
                                       void* stream) {
    if (!draft || !draft_probs || !target_probs || !u_accept || !u_resample || !accepted_len || !next_token)
        return EAGLE3_ERR_INVALID_ARG;
    if (batch < 1 || gamma < 1 || gamma > 4096 || V < 1) return EAGLE3_ERR_INVALID_ARG;
    ResidualArgs ra;
    memset(&ra, 0, sizeof(ra));
    ra.draft = draft; ra.draft_probs = draft_probs; ra.target_probs = target_probs;
    ra.u_accept = u_accept; ra.u_resample = u_resample; ra.batch = batch; ra.gamma = gamma; ra.V = V;
    ra.accepted_len = accepted_len; ra.next_token = next_token; ra.hist = hist;
    E3_CUDA(launch_accept_residual(ra, (cudaStream_t)stream));
    return EAGLE3_OK;
}

eagle3_status_t eagle3_draft_get_error(eagle3_draft_t* d, int32_t* device_error) {
    if (!d || !device_error) return EAGLE3_ERR_INVALID_ARG;
    E3_CUDA(cudaDeviceSynchronize());
    E3_CUDA(cudaMemcpy(device_error, d->err, sizeof(int32_t), cudaMemcpyDeviceToHost));
    return *device_error ? EAGLE3_ERR_DEVICE_RANGE : EAGLE3_OK;
}

eagle3_status_t eagle3_draft_clear_error(eagle3_draft_t* d, void* stream) {
    if (!d) return EAGLE3_ERR_INVALID_ARG;
    E3_CUDA(cudaMemsetAsync(d->err, 0, sizeof(int32_t), (cudaStream_t)stream));
    return EAGLE3_OK;
}

eagle3_status_t eagle3_draft_profile_enable(eagle3_draft_t* d, int32_t kind_mask) {
    if (!d) return EAGLE3_ERR_INVALID_ARG;
    if (kind_mask && d->prof_ev.empty()) {
        d->prof_ev.resize(2 * kProfPairs);
        d->prof_kind.resize(kProfPairs);
        for (auto& ev : d->prof_ev) E3_CUDA(cudaEventCreate(&ev));
    }
    if (!kind_mask) E3_CUDA(prof_flush(*d));
    d->prof_mask = (uint32_t)kind_mask;
    return EAGLE3_OK;
}

eagle3_status_t eagle3_draft_profile_read(eagle3_draft_t* d, int32_t kind, double* total_ms, int64_t* timed,
                                          int64_t* launches, const char** name) {
    if (!d || kind < 0 || kind >= EAGLE3_PROF_KINDS) return EAGLE3_ERR_INVALID_ARG;
    E3_CUDA(prof_flush(*d));
    if (total_ms) *total_ms = d->prof_ms[kind];
    if (timed) *timed = d->prof_n[kind];
    if (launches) *launches = d->launches[kind];
    if (name) *name = kKindNames[kind];
    return EAGLE3_OK;
}

eagle3_status_t eagle3_draft_profile_reset(eagle3_draft_t* d) {
    if (!d) return EAGLE3_ERR_INVALID_ARG;
    E3_CUDA(prof_flush(*d));
    for (int k = 0; k < EAGLE3_PROF_KINDS; ++k) { d->prof_ms[k] = 0.0; d->prof_n[k] = 0; d->launches[k] = 0; }
    return EAGLE3_OK;
}

eagle3_status_t eagle3_draft_destroy(eagle3_draft_t* d) {
    if (!d) return EAGLE3_OK;
    cudaDeviceSynchronize();
    for (auto& ev : d->prof_ev) cudaEventDestroy(ev);
    cudaError_t e = cudaFree(d->ws);
    delete d;
    if (e != cudaSuccess) return cuda_fail(e);
    return EAGLE3_OK;
}

}  // extern "C"
