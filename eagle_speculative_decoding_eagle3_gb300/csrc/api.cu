// C ABI of the EAGLE-3 MLA draft head: handle, argument checks, workspace, launch sequence.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <new>
#include <vector>

#include "../../include/eagle3.h"
#include "kernels.h"

using namespace e3;

static thread_local int g_last_cuda_error = 0;

struct eagle3_draft {
    eagle3_config_t cfg;
    eagle3_weights_t w;
    int device = 0;
    int num_sms = 0;
    void* ws = nullptr;
    size_t ws_bytes = 0;
    int m_cap = 0;          // rows per call
    int splits_cap = 0;     // attention splits bound
    int npart_lm = 0;       // lm_head argmax partials per row
    // workspace views
    float *f = nullptr, *carry = nullptr, *x = nullptr, *cqkv = nullptr, *cq_hat = nullptr, *q = nullptr,
          *qa = nullptr, *part_o = nullptr, *part_ml = nullptr, *o = nullptr, *h1 = nullptr, *y = nullptr,
          *mlp = nullptr, *h2 = nullptr, *z = nullptr, *pval = nullptr, *rope_cos = nullptr,
          *rope_sin = nullptr;
    int *pidx = nullptr, *row_seq = nullptr, *row_pos = nullptr, *d0 = nullptr, *tok_in = nullptr,
        *err = nullptr;
    size_t part_rows = 0;   // capacity of the attention partials in (row, split) pairs
    int batch = 0;
    bool have_extend = false;
};

namespace {

eagle3_status_t cuda_fail(cudaError_t e) {
    g_last_cuda_error = (int)e;
    return EAGLE3_ERR_CUDA;
}

#define E3_CUDA(call)                                  \
    do {                                               \
        cudaError_t _e = (call);                       \
        if (_e != cudaSuccess) return cuda_fail(_e);   \
    } while (0)

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }


constexpr int kHeadsPerCta = 16;

int attn_splits(const eagle3_draft& d, int M) {
    const int hg = (d.cfg.n_heads + kHeadsPerCta - 1) / kHeadsPerCta;
    const long want = 2L * d.num_sms;
    long s = (want + (long)M * hg - 1) / ((long)M * hg);
    if (s < 1) s = 1;
    if (s > d.splits_cap) s = d.splits_cap;
    return (int)s;
}

eagle3_status_t check_config(const eagle3_config_t* c) {
    if (!c) return EAGLE3_ERR_INVALID_ARG;
    const int dims[] = {c->hidden, c->n_heads, c->q_lora_rank, c->kv_lora_rank, c->qk_nope_dim, c->qk_rope_dim,
                        c->v_head_dim, c->intermediate, c->target_vocab, c->draft_vocab, c->max_batch,
                        c->max_tokens_per_extend, c->max_ctx, c->page_size, c->max_pages_per_seq};
    for (int v : dims)
        if (v <= 0) return EAGLE3_ERR_INVALID_ARG;
    if (c->qk_rope_dim % 2) return EAGLE3_ERR_INVALID_ARG;
    if (c->rope_interleave != 1) return EAGLE3_ERR_UNSUPPORTED;
    if (c->dtype != EAGLE3_F32 && c->dtype != EAGLE3_BF16) return EAGLE3_ERR_INVALID_ARG;
    // inner (K) dimensions of every linear layer stream in 8-element chunks
    const long inner[] = {c->hidden, c->q_lora_rank, c->kv_lora_rank, (long)c->n_heads * c->v_head_dim,
                          c->intermediate, c->kv_lora_rank + c->qk_rope_dim};
    for (long v : inner)
        if (v % 8) return EAGLE3_ERR_UNSUPPORTED;
    if (!attention_supported(c->kv_lora_rank, c->qk_rope_dim, c->qk_nope_dim, c->v_head_dim))
        return EAGLE3_ERR_UNSUPPORTED;
    if (c->draft_vocab > c->target_vocab) return EAGLE3_ERR_INVALID_ARG;
    if (!(c->rms_eps > 0.f) || !(c->rope_theta > 1.f) || !(c->yarn_factor >= 1.f) ||
        c->yarn_original_max_pos <= 0)
        return EAGLE3_ERR_INVALID_ARG;
    if ((long)c->max_ctx > (long)c->max_pages_per_seq * c->page_size) return EAGLE3_ERR_INVALID_ARG;
    return EAGLE3_OK;
}

eagle3_status_t check_weights(const eagle3_weights_t* w) {
    if (!w) return EAGLE3_ERR_INVALID_ARG;
    const void* p[] = {w->embed, w->fc, w->input_norm, w->hidden_norm, w->q_a, w->q_a_norm, w->q_b,
                       w->kv_a, w->kv_a_norm, w->kv_b, w->o, w->post_attn_norm, w->gate, w->up, w->down,
                       w->final_norm, w->lm_head};
    for (const void* v : p)
        if (!v || !aligned16(v)) return EAGLE3_ERR_INVALID_ARG;
    return EAGLE3_OK;
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
    size_t f, carry, x, cqkv, cq_hat, q, qa, part_o, part_ml, o, h1, y, mlp, h2, z, pval, pidx, rope_cos,
        rope_sin, row_seq, row_pos, d0, tok_in, err, total;
    int m_cap, splits_cap, npart;
    size_t part_rows;
};

Offsets plan(const eagle3_config_t& c, int num_sms) {
    Offsets o;
    const long M = c.max_tokens_per_extend > c.max_batch ? c.max_tokens_per_extend : c.max_batch;
    const long H = c.hidden, nh = c.n_heads, dqk = c.qk_nope_dim + c.qk_rope_dim;
    const long D = c.kv_lora_rank + c.qk_rope_dim;
    o.m_cap = (int)M;
    o.splits_cap = (c.max_ctx + 31) / 32;
    if (o.splits_cap > 64) o.splits_cap = 64;
    o.npart = gemv_argmax_parts(c.draft_vocab, num_sms);
    // rows x splits never exceeds M + 2 * num_sms (splits = ceil(2 * SMs / (M * groups)) for small M)
    o.part_rows = (size_t)M + 2 * (size_t)num_sms + 1;
    Layout L;
    const size_t f4 = 4;
    o.f = L.take(M * H * f4);
    o.carry = L.take((size_t)c.max_batch * H * f4);
    o.x = L.take(M * 2 * H * f4);
    o.cqkv = L.take(M * (c.q_lora_rank + D) * f4);
    o.cq_hat = L.take(M * c.q_lora_rank * f4);
    o.q = L.take(M * nh * dqk * f4);
    o.qa = L.take(M * nh * D * f4);
    o.part_o = L.take(o.part_rows * nh * c.kv_lora_rank * f4);
    o.part_ml = L.take(o.part_rows * nh * 2 * f4);
    o.o = L.take(M * nh * c.v_head_dim * f4);
    o.h1 = L.take(M * H * f4);
    o.y = L.take(M * H * f4);
    o.mlp = L.take(M * (size_t)c.intermediate * f4);
    o.h2 = L.take(M * H * f4);
    o.z = L.take((size_t)c.max_batch * H * f4);
    o.pval = L.take((size_t)c.max_batch * o.npart * f4);
    o.pidx = L.take((size_t)c.max_batch * o.npart * 4);
    o.rope_cos = L.take((size_t)c.max_ctx * (c.qk_rope_dim / 2) * f4);
    o.rope_sin = L.take((size_t)c.max_ctx * (c.qk_rope_dim / 2) * f4);
    o.row_seq = L.take(M * 4);
    o.row_pos = L.take(M * 4);
    o.d0 = L.take((size_t)c.max_batch * 4);
    o.tok_in = L.take((size_t)c.max_batch * 4);
    o.err = L.take(4);
    o.total = L.off;
    return o;
}

// YaRN rotary frequencies (the published YaRN construction; the pages name DeepseekYarnRotaryEmbedding
// and its rope_scaling betas, "Eagle3 DeepseekV3 in MAX" §4-§5): pair i keeps theta^(-2i/d) where its
// wavelength fits >= beta_fast times in the original window, is divided by the factor where it fits
// < beta_slow times, and is blended linearly in between.
void yarn_table(const eagle3_config_t& c, std::vector<float>& cs, std::vector<float>& sn) {
    const int d = c.qk_rope_dim, half = d / 2;
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
    return (float)(m * m / sqrt((double)(c.qk_nope_dim + c.qk_rope_dim)));
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

GemvArgs gemv1(const eagle3_draft& d, const float* a, long lda, int K, const void* w, int N, float* y, long ldy) {
    GemvArgs g;
    memset(&g, 0, sizeof(g));
    g.a[0] = a; g.lda[0] = lda; g.ka[0] = K; g.na = 1;
    g.w[0] = w; g.nw[0] = N; g.nseg_w = 1;
    g.N = N; g.K = K;
    g.a_type = F32;
    g.w_type = d.cfg.dtype == EAGLE3_BF16 ? BF16 : F32;
    g.y = y; g.ldy = ldy;
    return g;
}

// The decoder chain from the concatenated input x to the scored hidden / argmax partials.
// fused: the residual stream of the rows (fc output in extend, the carried hidden in decode).
cudaError_t run_layer(eagle3_draft& d, eagle3_kv_t* kv, int M, const float* fused, cudaStream_t st) {
    const eagle3_config_t& c = d.cfg;
    const eagle3_weights_t& w = d.w;
    const int H = c.hidden, dq = c.q_lora_rank, dc = c.kv_lora_rank, dr = c.qk_rope_dim;
    const int nh = c.n_heads, dqk = c.qk_nope_dim + dr, D = dc + dr;
    RowArgs ra = row_args(d, kv);
    cudaError_t e;
    // q_a | kv_a over the 2H input
    {
        GemvArgs g = gemv1(d, d.x, 2L * H, 2 * H, w.q_a, dq + D, d.cqkv, dq + D);
        g.w[1] = w.kv_a; g.nw[0] = dq; g.nw[1] = D; g.nseg_w = 2; g.M = M;
        if ((e = launch_gemv(g, EPI_STORE, d.num_sms, st)) != cudaSuccess) return e;
    }
    if ((e = launch_latent(ra, M, d.cqkv, w.q_a_norm, w.kv_a_norm, d.rope_cos, d.rope_sin, d.row_seq, d.row_pos,
                           kv->block_table, kv->data, d.cq_hat, st)) != cudaSuccess)
        return e;
    {
        GemvArgs g = gemv1(d, d.cq_hat, dq, dq, w.q_b, nh * dqk, d.q, (long)nh * dqk);
        g.M = M;
        if ((e = launch_gemv(g, EPI_STORE, d.num_sms, st)) != cudaSuccess) return e;
    }
    AttnArgs aa;
    aa.M = M; aa.nh = nh; aa.dn = c.qk_nope_dim; aa.dr = dr; aa.dc = dc; aa.dv = c.v_head_dim;
    aa.sigma = attention_scale(c);
    aa.page_size = c.page_size; aa.max_pages = c.max_pages_per_seq;
    aa.splits = attn_splits(d, M);
    aa.dt = ra.dt;
    aa.row_seq = d.row_seq; aa.row_pos = d.row_pos; aa.block_table = kv->block_table;
    aa.cache = kv->data; aa.kv_b = w.kv_b; aa.q = d.q; aa.rope_cos = d.rope_cos; aa.rope_sin = d.rope_sin;
    aa.qa = d.qa; aa.part_o = d.part_o; aa.part_ml = d.part_ml; aa.o = d.o;
    if ((e = launch_absorb(aa, st)) != cudaSuccess) return e;
    if ((e = launch_attention(aa, st)) != cudaSuccess) return e;
    if ((e = launch_combine(aa, st)) != cudaSuccess) return e;
    // o_proj + residual
    {
        GemvArgs g = gemv1(d, d.o, (long)nh * c.v_head_dim, nh * c.v_head_dim, w.o, H, d.h1, H);
        g.M = M; g.resid = fused; g.ldr = H;
        if ((e = launch_gemv(g, EPI_RESID, d.num_sms, st)) != cudaSuccess) return e;
    }
    if ((e = launch_rmsnorm(M, H, c.rms_eps, ra.dt, d.h1, w.post_attn_norm, d.y, st)) != cudaSuccess) return e;
    {
        GemvArgs g = gemv1(d, d.y, H, H, w.gate, c.intermediate, d.mlp, c.intermediate);
        g.w[1] = w.up; g.nw[1] = c.intermediate; g.M = M;
        if ((e = launch_gemv(g, EPI_GLU, d.num_sms, st)) != cudaSuccess) return e;
    }
    {
        GemvArgs g = gemv1(d, d.mlp, c.intermediate, c.intermediate, w.down, H, d.h2, H);
        g.M = M; g.resid = d.h1; g.ldr = H;
        if ((e = launch_gemv(g, EPI_RESID, d.num_sms, st)) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t run_head(eagle3_draft& d, int batch, float* logits_out, cudaStream_t st) {
    GemvArgs g = gemv1(d, d.z, d.cfg.hidden, d.cfg.hidden, d.w.lm_head, d.cfg.draft_vocab, nullptr, 0);
    g.M = batch; g.pval = d.pval; g.pidx = d.pidx; g.logits = logits_out; g.ldl = d.cfg.draft_vocab;
    return launch_gemv(g, EPI_ARGMAX, d.num_sms, st);
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
    if ((s = check_weights(weights)) != EAGLE3_OK) return s;
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
    d->npart_lm = o.npart;
    d->part_rows = o.part_rows;
    char* base = (char*)d->ws;
    d->f = (float*)(base + o.f); d->carry = (float*)(base + o.carry); d->x = (float*)(base + o.x);
    d->cqkv = (float*)(base + o.cqkv); d->cq_hat = (float*)(base + o.cq_hat); d->q = (float*)(base + o.q);
    d->qa = (float*)(base + o.qa); d->part_o = (float*)(base + o.part_o); d->part_ml = (float*)(base + o.part_ml);
    d->o = (float*)(base + o.o); d->h1 = (float*)(base + o.h1); d->y = (float*)(base + o.y);
    d->mlp = (float*)(base + o.mlp); d->h2 = (float*)(base + o.h2); d->z = (float*)(base + o.z);
    d->pval = (float*)(base + o.pval); d->pidx = (int*)(base + o.pidx);
    d->rope_cos = (float*)(base + o.rope_cos); d->rope_sin = (float*)(base + o.rope_sin);
    d->row_seq = (int*)(base + o.row_seq); d->row_pos = (int*)(base + o.row_pos);
    d->d0 = (int*)(base + o.d0); d->tok_in = (int*)(base + o.tok_in); d->err = (int*)(base + o.err);
    std::vector<float> cs, sn;
    yarn_table(d->cfg, cs, sn);
    e = cudaMemcpy(d->rope_cos, cs.data(), cs.size() * sizeof(float), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(d->rope_sin, sn.data(), sn.size() * sizeof(float), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemset(d->err, 0, sizeof(int));
    if (e == cudaSuccess) e = cudaMemset(d->carry, 0, (size_t)d->cfg.max_batch * d->cfg.hidden * sizeof(float));
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
    for (int i = 0; i < 3; ++i)
        if (!aux_hidden[i] || !aligned16(aux_hidden[i])) return EAGLE3_ERR_INVALID_ARG;
    const eagle3_config_t& c = d->cfg;
    if (batch < 1 || batch > c.max_batch || num_tokens < batch || num_tokens > c.max_tokens_per_extend)
        return EAGLE3_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    const int H = c.hidden, M = num_tokens;
    RowArgs ra = row_args(*d, cache);
    // fc: f = [a_early | a_mid | a_late] W_fc^T  (3H -> H, no bias)
    {
        GemvArgs g;
        memset(&g, 0, sizeof(g));
        for (int i = 0; i < 3; ++i) { g.a[i] = aux_hidden[i]; g.lda[i] = H; g.ka[i] = H; }
        g.na = 3;
        g.w[0] = d->w.fc; g.nw[0] = H; g.nseg_w = 1;
        g.M = M; g.N = H; g.K = 3 * H;
        g.a_type = ra.dt; g.w_type = ra.dt;
        g.y = d->f; g.ldy = H;
        E3_CUDA(launch_gemv(g, EPI_STORE, d->num_sms, st));
    }
    E3_CUDA(launch_embed_norms(ra, false, M, tokens, positions, row_offsets, batch, nullptr, nullptr, d->f,
                               d->w.embed, d->w.input_norm, d->w.hidden_norm, d->x, d->row_seq, d->row_pos, st));
    E3_CUDA(run_layer(*d, cache, M, d->f, st));
    E3_CUDA(launch_final(ra, true, batch, row_offsets, d->h2, d->w.final_norm, d->row_pos, d->carry, d->z,
                         hidden_out, cache->lengths, st));
    E3_CUDA(run_head(*d, batch, logits_out, st));
    E3_CUDA(launch_argmax_final(batch, d->npart_lm, d->pval, d->pidx, 0, nullptr, c.target_vocab, d->d0, nullptr,
                                0, 0, nullptr, d->err, st));
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
    RowArgs ra = row_args(*d, cache);
    E3_CUDA(launch_emit_first(B, d->d0, d2t, c.target_vocab, draft_tokens, gamma, d->tok_in, d->err, st));
    for (int s = 1; s < gamma; ++s) {
        E3_CUDA(launch_embed_norms(ra, true, B, nullptr, nullptr, nullptr, B, d->tok_in, cache->lengths, d->carry,
                                   d->w.embed, d->w.input_norm, d->w.hidden_norm, d->x, d->row_seq, d->row_pos,
                                   st));
        E3_CUDA(run_layer(*d, cache, B, d->carry, st));
        float* ho = hidden_out ? hidden_out + (size_t)(s - 1) * B * H : nullptr;
        float* lo = logits_out ? logits_out + (size_t)(s - 1) * B * c.draft_vocab : nullptr;
        E3_CUDA(launch_final(ra, false, B, nullptr, d->h2, d->w.final_norm, d->row_pos, d->carry, d->z, ho,
                             cache->lengths, st));
        E3_CUDA(run_head(*d, B, lo, st));
        E3_CUDA(launch_argmax_final(B, d->npart_lm, d->pval, d->pidx, 1, d2t, c.target_vocab, nullptr, draft_tokens,
                                    gamma, s, d->tok_in, d->err, st));
    }
    return EAGLE3_OK;
}

eagle3_status_t eagle3_accept(const int32_t* draft, const int32_t* target, int32_t batch, int32_t gamma,
                              int32_t* accepted_len, int32_t* hist, void* stream) {
    if (!draft || !target || !accepted_len) return EAGLE3_ERR_INVALID_ARG;
    if (batch < 1 || gamma < 1 || gamma > 4096) return EAGLE3_ERR_INVALID_ARG;
    E3_CUDA(launch_accept(draft, target, batch, gamma, accepted_len, hist, (cudaStream_t)stream));
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

eagle3_status_t eagle3_draft_destroy(eagle3_draft_t* d) {
    if (!d) return EAGLE3_OK;
    cudaDeviceSynchronize();
    cudaError_t e = cudaFree(d->ws);
    delete d;
    if (e != cudaSuccess) return cuda_fail(e);
    return EAGLE3_OK;
}

}  // extern "C"
