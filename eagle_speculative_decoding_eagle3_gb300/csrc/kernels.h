// Internal launch interface of the draft-head kernels.  Host code (api.cu) fills these structs;
// every launch_* enqueues its kernel(s) on `st` and returns the launch error.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace e3 {

// FP8: E4M3 codes with per-row fp32 scales; FP4: NVFP4 (E2M1 codes, E4M3 scales per 16, fp32 per matrix)
enum DType { F32 = 0, BF16 = 1, FP8 = 2, FP4 = 3 };

// Opts `kernel` in to `bytes` of dynamic shared memory on the current device.  The opt-in is a property
// of the device's context, so it is made once per (kernel, device) and remembered under a lock.
cudaError_t smem_optin(const void* kernel, int bytes);

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
    // grouped rows (per-head GEMVs over one weight tensor), off when 0:
    //   output row n reads weight row (n / w_grp) * w_grp_stride + w_row0 + n % w_grp of w[0]
    //   and the activation slice starting at element (n / a_grp) * a_grp_stride of a[0]
    int w_grp; long w_grp_stride; int w_row0;
    int a_grp; long a_grp_stride;
    int* err;                         // device error word (bounded waits that ran out)
    // w_type FP8: per-output-row scales of w[0] / w[1] (y[m, n] = scale[n] * sum_k A[m, k] code[n, k]);
    // w_type FP4: each matrix's one fp32 scale, with its E4M3 block scales [rows, K / 16] in wbs
    const float* wscale[2];
    const uint8_t* wbs[2];
};
cudaError_t launch_gemv(GemvArgs& g, int epi, int num_sms, cudaStream_t st);
cudaError_t launch_gemv_fp8(GemvArgs& g, int epi, int num_sms, cudaStream_t st);   // w_type FP8
cudaError_t launch_gemv_fp4(GemvArgs& g, int epi, int num_sms, cudaStream_t st);   // w_type FP4
// bf16 expansion of an NVFP4 matrix (K a multiple of 32)
cudaError_t launch_dequant_nvfp4(const uint8_t* codes, const uint8_t* block_scales, const float* global, long rows,
                                 int K, __nv_bfloat16* out, int num_sms, cudaStream_t st);
// bf16 expansion of an FP8 E4M3 matrix with per-row scales (K a multiple of 8)
cudaError_t launch_dequant_e4m3(const uint8_t* codes, const float* scales, long rows, int K, __nv_bfloat16* out,
                                int num_sms, cudaStream_t st);
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
                               float* x, __nv_bfloat16* x_bf, int* row_seq, int* row_pos, cudaStream_t st);

// latent norms, k_rope rotation and cache append
cudaError_t launch_latent(const RowArgs& a, int M, const float* cqkv, const void* w_qa, const void* w_kva,
                          const float* rope_cos, const float* rope_sin, const int* row_seq, const int* row_pos,
                          const int* block_table, void* cache, float* cq_hat, __nv_bfloat16* cqh_bf,
                          cudaStream_t st);

cudaError_t launch_rmsnorm(int M, int H, float eps, DType wt, const float* x, const void* w, float* y,
                           __nv_bfloat16* y_bf, cudaStream_t st);

// scored rows: b < batch; src row = extend ? row_offsets[b+1]-1 : b
cudaError_t launch_final(const RowArgs& a, bool extend, int batch, int M, const int* row_offsets, const float* h2,
                         const void* w_final, const int* row_pos, float* carry, float* z, __nv_bfloat16* z_bf,
                         float* hidden_out, int* lengths, cudaStream_t st);

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
cudaError_t launch_accept_relaxed(const int* draft, const int* ids, const float* lp, const unsigned char* think,
                                  int batch, int gamma, int k, float delta, int* acc, int* hist, cudaStream_t st);

// ---------------------------------------------------------------- sampled drafts, residual acceptance
struct SampleArgs {
    const float* logits; long ldl;     // [rows, V] draft-vocabulary logits
    int rows, V;
    float temperature;                 // 0: greedy argmax
    int top_k;                         // 0: whole vocabulary (top_p must then be 1); else 1..1024
    float top_p;                       // (0, 1]
    const float* uniforms;             // [rows] in [0, 1)
    const int* d2t;                    // [V] additive draft-to-target map or null
    int target_vocab;
    int* tokens;                       // [rows] out: target-vocabulary ids
    int* tokens2; long tok2_stride;    // optional second copy of the ids, row r at r * tok2_stride
    int* draft_ids;                    // [rows] out (optional): draft-vocabulary ids
    float* token_prob;                 // [rows] out (optional): the sampled token's final probability
    float* probs; long ldp;            // [rows, probs_len] out (optional): final distribution
    int probs_len;
    int probs_target;                  // probs indexed by target ids (through d2t) instead of draft ids
    int* err;
};
struct ResidualArgs {
    const int* draft;                  // [B, gamma] target-vocabulary ids
    const float* draft_probs;          // [B, gamma, V] draft distributions over the target vocabulary
    const float* target_probs;         // [B, gamma + 1, V]
    const float* u_accept;             // [B, gamma]
    const float* u_resample;           // [B, gamma]
    int batch, gamma, V;
    int* accepted_len;                 // [B]
    int* next_token;                   // [B] the token emitted after the accepted prefix
    int* hist;                         // [gamma + 1] or null
};
cudaError_t launch_sample(const SampleArgs& s, cudaStream_t st);
cudaError_t launch_accept_residual(const ResidualArgs& a, cudaStream_t st);
// typical acceptance: accept x while p(x) > min(epsilon, delta exp(-H(p))); target_probs [B, gamma, V]
cudaError_t launch_accept_typical(const int* draft, const float* target_probs, int batch, int gamma, int V,
                                  float epsilon, float delta, int* accepted_len, int* hist, cudaStream_t st);
// out[i] = uniform i of the Philox4x64-10 stream (seed, offset), i < n
cudaError_t launch_philox_uniforms(uint64_t seed, uint64_t offset, long n, float* out, cudaStream_t st);

// ---------------------------------------------------------------- causal attention of a long extend
// (unabsorbed; DeepseekV3 geometry d_n 128, d_r 64, d_v 128)
struct PrefillArgs {
    int M, B, nh, max_ctx, page_size, max_pages, num_pages;
    int ntiles_cap;                    // entries of `tiles` (prefill_tiles_cap)
    int bq;                            // query rows per tile: 64 (mma.sync kernel) or 128 (tcgen05 kernel)
    float sigma;
    const int* row_offsets;            // [B + 1] rows of each sequence in this extend
    const int* row_pos;                // [M] positions
    const int* block_table;            // [B, max_pages]
    const void* cache;                 // bf16 [pages, page_size, 576]
    __nv_bfloat16* xc;                 // [B * max_ctx, 512] gathered latent rows
    __nv_bfloat16* xpe;                // [B * max_ctx, 64] gathered rotated k_pe
    const __nv_bfloat16* kv;           // [B * max_ctx, nh * 256] expanded [k_nope | v] per head
    __nv_bfloat16* q;                  // [M, nh * 192] bf16 query rows (rope part rotated in place)
    const float* qf;                   // [M, nh * 192] fp32 query rows (source of the rope part), or
                                       // null to rotate the bf16 rows of q in place
    const float* rope_cos;             // [max_ctx, 32]
    const float* rope_sin;
    int4* tiles;                       // [ntiles_cap] (sequence, first row, rows) or sequence -1
    __nv_bfloat16* o_bf;               // [M, nh * 128] attention output per head
    int* err;
};
bool prefill_supported(int dt, int dn, int dr, int dv);
int prefill_tiles_cap(int M, int B, int bq);
cudaError_t launch_kv_gather(const PrefillArgs& a, cudaStream_t st);
cudaError_t launch_prefill_tiles(const PrefillArgs& a, cudaStream_t st);
cudaError_t launch_rope_q_rows(const PrefillArgs& a, cudaStream_t st);
cudaError_t launch_prefill_attention(const PrefillArgs& a, cudaStream_t st);
// tcgen05 flash attention of the same extend (bq 128): the same o_bf output
bool prefill_tc_supported(const PrefillArgs& a);
cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t st);

// ---------------------------------------------------------------- MHA attention (Llama-style head)
struct MhaArgs {
    int M, nh, nkv, d;
    float sigma;
    int page_size, max_pages, num_pages;
    int splits, chunk;        // split s of a row covers slots [s chunk, (s + 1) chunk) of its context
    DType dt;                 // cache storage
    const int* row_seq;
    const int* row_pos;
    const int* block_table;
    void* cache;              // [num_pages, page_size, 2 nkv d]
    float* q;                 // [M, nh d], rotated in place by the append kernel
    const float* kv;          // [M, 2 nkv d] k then v projections
    const float* rope_cos;    // [max_ctx, d / 2]
    const float* rope_sin;
    float* part_o;            // [M splits, nh, d] (splits > 1)
    float* part_ml;           // [M splits, nh, 2]
    float* o;                 // [M, nh d] fp32 output (or null)
    __nv_bfloat16* o_bf;      // [M, nh d] bf16 output (or null)
    int* err;
};
bool mha_supported(int nh, int nkv, int d);
cudaError_t launch_mha_rope_append(const MhaArgs& a, cudaStream_t st);
cudaError_t launch_mha_attention(const MhaArgs& a, cudaStream_t st);
cudaError_t launch_mha_merge(const MhaArgs& a, cudaStream_t st);

// ---------------------------------------------------------------- MLA attention (absorbed)
struct AttnArgs {
    int M, nh, dn, dr, dc, dv;
    float sigma;
    int page_size, max_pages, num_pages, splits;
    int chunk;                // > 0: split s covers slots [s chunk, (s + 1) chunk) of every row (splits past a
                              // row's context are empty); 0: a row's context is divided evenly over splits
    int* err;
    DType dt;
    const int* row_seq; const int* row_pos; const int* block_table;
    const void* cache;
    const void* kv_b;
    const float* q;      // [M, nh*(dn+dr)]
    const __nv_bfloat16* q_bf;   // bf16 copy of q; when set, rope_q reads the rope part from it
    const float* rope_cos; const float* rope_sin;
    float* qa;           // [M, nh, dc+dr]   absorbed latent query | rotated rope query
    __nv_bfloat16* qa_bf;  // bf16 copy of qa for the tensor-core kernel (nullptr: not written)
    float* part_o;       // [M, nh, splits, dc]
    float* part_ml;      // [M, nh, splits, 2]
    float* o;            // [M, nh*dv]
    __nv_bfloat16* olat_bf;  // merged latent output o_lat [M, nh, dc] in bf16 (optional)
    float* olat;             // merged latent output o_lat [M, nh, dc] in fp32 (optional)
};
cudaError_t launch_absorb(const AttnArgs& a, cudaStream_t st);
cudaError_t launch_attention(const AttnArgs& a, cudaStream_t st);
// split-K merge into o_lat (olat and/or olat_bf); the value up-projection then runs as a GEMM
cudaError_t launch_merge(const AttnArgs& a, cudaStream_t st);
// split merge fused with o = W_UV o_lat into a.o (fp32), for at most 8 rows of a bf16 head with d_c 512,
// d_v 128 and 2 .. kMergeUnabsorbMaxSplits splits (the plain merge takes at most 64)
constexpr int kMergeUnabsorbMaxSplits = 128;
bool merge_unabsorb_supported(const AttnArgs& a);
cudaError_t launch_merge_unabsorb(const AttnArgs& a, cudaStream_t st);
// rotated rope query into qa / qa_bf[:, :, dc:] (the tensor-core path forms q_lat separately)
cudaError_t launch_rope_q(const AttnArgs& a, cudaStream_t st);
// W_UK,h^T for every head: out[h, c, i] = kv_b[h*(dn+dv) + i, c]  (bf16)
cudaError_t launch_transpose_wuk(const void* kv_b, int nh, int dn, int dv, int dc, __nv_bfloat16* out,
                                 cudaStream_t st);
bool attention_supported(int dc, int dr, int dn, int dv);
int attention_heads_per_cta(int dt, int dc, int dr);
// true where the latent attention kernel holds one CTA per SM (the 64-head mma.sync kernel)
bool attention_one_cta_per_sm(int dt, int dc, int dr);
// tcgen05 latent attention (bf16 cache, 128 heads, latent 512 + rope 64, fixed-chunk splits of 64k
// slots, pages of 64k slots): one CTA pair per (split, row); same partial / o_lat outputs as above
bool attention_tc_supported(const AttnArgs& a);
cudaError_t launch_attention_tc(const AttnArgs& a, cudaStream_t st);

// ---------------------------------------------------------------- tcgen05 GEMM (bf16, many rows)
// out[m, n] = sum_k W[n, k] X[m, k]; W from mw[0] (rows < np0) and mw[1] (rows >= np0, or the up
// projection for GLU), X from mx[s] for K-blocks in segment s (boundaries kseg, in 64-wide blocks).
struct TcParams {
    CUtensorMap mw[2];
    CUtensorMap mx[3];
    int np0;
    int N, M, K;
    int kseg[2];
    int nkb, kb_per_split, splits;   // set by the launcher
    int nbatch;                   // batched GEMMs: batch z reads W rows + z*bw_rows, X K-blocks + z*bq_kb,
    int bw_rows, bq_kb;           // and writes output columns + z*by_col (one X segment, no split)
    long by_col;
    int epi;                      // EPI_STORE / EPI_RESID / EPI_GLU / EPI_ARGMAX
    int pair;                     // STORE / RESID at 256 tokens per tile: each CTA takes two 128-row
                                  // weight tiles that share the activation tile (0 = one tile)
    int persist;                  // > 0: one-matrix, unsplit GEMMs with more tiles than this run on this
                                  // many persistent CTAs (double-buffered TMEM accumulators); 0 = a CTA per tile
    float* y; long ldy;           // fp32 output (optional)
    __nv_bfloat16* ybf; long ldybf;  // bf16 output (optional)
    const float* resid; long ldr;
    float* part;                  // split-K partials [splits][GLU ? 2 : 1][M][N]
    float* pval; int* pidx; int npart;   // ARGMAX partials [M, npart] (npart set by the launcher)
    float* logits; long ldl;
    int* err;
};
bool make_tma_2d(CUtensorMap* map, const void* ptr, long rows, long cols, long ld, int box_rows);
bool make_tma_chunks(CUtensorMap* map, const void* ptr, long rows, long cols, int box_rows, int box_chunks);
int tc_pick_bn(int M);
cudaError_t launch_tc_gemm(TcParams& p, int bn, int splits, cudaStream_t st);

}  // namespace e3
