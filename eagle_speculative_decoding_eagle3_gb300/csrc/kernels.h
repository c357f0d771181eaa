// Internal launch interface of the draft-head kernels.  Host code (api.cu) fills these structs;
// every launch_* enqueues its kernel(s) on `st` and returns the launch error.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace e3 {

enum DType { F32 = 0, BF16 = 1 };

// ---------------------------------------------------------------- weight-streaming GEMM
// y[m, n] = sum_k A[m, k] * W[n, k] for m < M, n < N, with
//   A given as up to 3 consecutive K-segments (a[s], row stride lda[s], width ka[s]),
//   W given as up to 2 consecutive N-segments (w[s], rows nw[s]); every W row has K = sum ka.
enum Epi { EPI_STORE = 0, EPI_RESID = 1, EPI_GLU = 2, EPI_ARGMAX = 3 };

struct GemvArgs {
    const void* a[3];
    long lda[3];
    int ka[3];
    int na;
    const void* w[2];   // EPI_GLU: w[0] = gate rows, w[1] = up rows, both N rows
    int nw[2];
    int nseg_w;
    int M, N, K;
    DType a_type, w_type;
    float* y;  long ldy;              // STORE / RESID / GLU output
    const float* resid; long ldr;     // RESID
    float* pval; int* pidx;           // ARGMAX partials [M, npart]
    int npart;                        // ARGMAX: grid.x used (set by the launcher)
    float* logits; long ldl;          // ARGMAX: optional full logits
};
cudaError_t launch_gemv(GemvArgs& g, int epi, int num_sms, cudaStream_t st);
int gemv_argmax_parts(int N, int num_sms);   // partial count of an ARGMAX launch over N columns

// ---------------------------------------------------------------- row kernels
struct RowArgs {
    int H, dq, dc, dr, nh, dn, dv;
    int Vt, max_ctx, page_size, max_pages, num_pages;
    float eps;
    DType dt;             // storage type of weights / embed / cache
    int* err;
};

// extend: rows r < M; token = tokens[r], pos = positions[r], fused = f[r]
// decode: rows r < M (= batch); token = tok_in[r], pos = lengths[r], fused = carry[r]
cudaError_t launch_embed_norms(const RowArgs& a, bool decode, int M, const int* tokens, const int* positions,
                               const int* row_offsets, int batch, const int* tok_in, const int* lengths,
                               const float* fused, const void* embed, const void* w_in, const void* w_hid,
                               float* x, int* row_seq, int* row_pos, cudaStream_t st);

// latent norms, k_rope rotation and cache append
cudaError_t launch_latent(const RowArgs& a, int M, const float* cqkv, const void* w_qa, const void* w_kva,
                          const float* rope_cos, const float* rope_sin, const int* row_seq, const int* row_pos,
                          const int* block_table, void* cache, float* cq_hat, cudaStream_t st);

cudaError_t launch_rmsnorm(int M, int H, float eps, DType wt, const float* x, const void* w, float* y,
                           cudaStream_t st);

// scored rows: b < batch; src row = extend ? row_offsets[b+1]-1 : b
cudaError_t launch_final(const RowArgs& a, bool extend, int batch, const int* row_offsets, const float* h2,
                         const void* w_final, const int* row_pos, float* carry, float* z, float* hidden_out,
                         int* lengths, cudaStream_t st);

// argmax over partials; mode 0 (extend): d0[b] = d; mode 1 (decode step s): t = remap(d),
// out_tokens[b*gamma + s] = t, tok_in[b] = t
cudaError_t launch_argmax_final(int batch, int npart, const float* pval, const int* pidx, int mode,
                                const int* d2t, int Vt, int* d0, int* out_tokens, int gamma, int s,
                                int* tok_in, int* err, cudaStream_t st);

// decode start: t = remap(d0[b]); out_tokens[b*gamma] = t; tok_in[b] = t
cudaError_t launch_emit_first(int batch, const int* d0, const int* d2t, int Vt, int* out_tokens, int gamma,
                              int* tok_in, int* err, cudaStream_t st);

cudaError_t launch_accept(const int* draft, const int* target, int batch, int gamma, int* acc, int* hist,
                          cudaStream_t st);

// ---------------------------------------------------------------- MLA attention (absorbed)
struct AttnArgs {
    int M, nh, dn, dr, dc, dv;
    float sigma;
    int page_size, max_pages, splits;
    DType dt;
    const int* row_seq; const int* row_pos; const int* block_table;
    const void* cache;
    const void* kv_b;
    const float* q;      // [M, nh*(dn+dr)]
    const float* rope_cos; const float* rope_sin;
    float* qa;           // [M, nh, dc+dr]   absorbed latent query | rotated rope query
    float* part_o;       // [M, nh, splits, dc]
    float* part_ml;      // [M, nh, splits, 2]
    float* o;            // [M, nh*dv]
};
cudaError_t launch_absorb(const AttnArgs& a, cudaStream_t st);
cudaError_t launch_attention(const AttnArgs& a, cudaStream_t st);
cudaError_t launch_combine(const AttnArgs& a, cudaStream_t st);
bool attention_supported(int dc, int dr, int dn, int dv);

}  // namespace e3
