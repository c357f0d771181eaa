/*
 * eagle3.h — C ABI of the GB300 (sm_103a) EAGLE-3 draft head for an MLA (DeepseekV3-shaped) target.
 *
 * The head, per token: fc fuses three target hidden states (early, middle, late; 3H -> H, no
 * bias); the token embedding (the target's table) and the fused state are RMS-normalised
 * separately and concatenated to 2H; one MLA decoder layer runs at 2H input (q_a -> q_lora,
 * kv_a -> kv_lora + rope, interleaved YaRN RoPE, attention over a one-layer latent KV cache,
 * o_proj heads*v_head_dim -> H, residual), then a dense SiLU-gated MLP with residual; the
 * final RMSNorm and the head's own lm_head give logits whose argmax, mapped through the
 * optional d2t table, is the draft token.  Drafting runs autoregressively for gamma tokens;
 * greedy acceptance compares drafts with target tokens.
 *
 * Sources (page title, section):
 *   "Eagle3 DeepseekV3 speculative decoding architecture: a full walkthrough of MAX's
 *    eagle3_deepseekV3 module" (xxmr.cn) — §4 Eagle3MLADraft forward, §5 weight sharing and
 *    rope_scaling override, §7 one-layer draft KV, §9 prefill = step 0 / decode = steps 1..K,
 *    §10 greedy acceptance without mid-graph allocation;
 *   "max.pipelines.architectures.eagle3_deepseekV3" API reference (max.modular.com) —
 *    Eagle3DeepseekV3DraftConfig defaults, construct_kv_params (one-layer view of the cache);
 *   "EAGLE head deep dive: inside Model Optimizer's speculative-decoding draft model"
 *    (discosf.com) — part 2 fc fusion, part 3 doubled first-layer input, part 4 draft
 *    vocabulary lm_head and the additive d2t table.
 *
 * Conventions for every call:
 *   - Pointers are DEVICE pointers unless the comment says "host".
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).  All
 *     compute calls are asynchronous on it and allocate nothing, so they can be recorded in a
 *     CUDA graph.
 *   - Weight and cache memory is BORROWED: the caller owns it and keeps it alive and
 *     unchanged (weights) while the handle uses it.  The handle owns only its workspace.
 *   - Arguments the host can check are checked before anything is launched; a failed check
 *     returns a status and launches nothing.  Range errors that only the device can see
 *     (a token >= target_vocab, a d2t result outside [0, target_vocab), a position >= max_ctx,
 *     a page index outside the cache) are clamped into range, set a bit in the handle's
 *     sticky device error word, and are reported by eagle3_draft_get_error.
 *   - Weights are row-major [out, in] like nn.Linear.  Pointers must be 16-byte aligned and
 *     every inner dimension a multiple of 8.
 */
#ifndef EAGLE3_H
#define EAGLE3_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define EAGLE3_API __attribute__((visibility("default")))
#else
#define EAGLE3_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    EAGLE3_OK = 0,
    EAGLE3_ERR_INVALID_ARG = 1,   /* null pointer, size out of the configured bounds, misalignment */
    EAGLE3_ERR_UNSUPPORTED = 2,   /* a shape or dtype the library does not implement */
    EAGLE3_ERR_STATE = 3,         /* decode before any extend, or batch mismatch */
    EAGLE3_ERR_OOM = 4,           /* workspace allocation failed at create */
    EAGLE3_ERR_CUDA = 5,          /* a CUDA runtime call failed (see eagle3_last_cuda_error) */
    EAGLE3_ERR_DEVICE_RANGE = 6,  /* returned by eagle3_draft_get_error when the error word is set */
    EAGLE3_ERR_SCRATCH_LIMIT = 7  /* eagle3_linear_noalloc: M * N exceeds what its fixed scratch holds */
} eagle3_status_t;

typedef enum { EAGLE3_F32 = 0, EAGLE3_BF16 = 1 } eagle3_dtype_t;

/* Storage of the nine projection matrices (fc, q_a, kv_a, q_b, o, gate, up, down, lm_head).
 *   EAGLE3_WEIGHTS_DTYPE  the configured dtype, like every other weight;
 *   EAGLE3_WEIGHTS_FP8    FP8 E4M3 codes (OCP 8-bit floating point: sign, 4 exponent bits with bias 7,
 *                         3 mantissa bits, largest finite 448) [rows, cols] row-major, one byte each, with
 *                         one fp32 scale per output row: weight[n, k] = decode(code[n, k]) * scale[n].
 *                         The post-training FP8 quantization of the drafter ("EAGLE head deep dive",
 *                         deployment); eagle3_quantize_e4m3 produces this form from bf16 / fp32 weights.
 *                         Requires dtype == EAGLE3_BF16.  kv_b, the embedding and the norm weights keep
 *                         the configured dtype.
 *   EAGLE3_WEIGHTS_NVFP4  NVFP4: E2M1 codes (OCP FP4: sign, 2 exponent bits with bias 1, 1 mantissa bit,
 *                         largest 6), two per byte with the even element in the low nibble, [rows, cols/2];
 *                         one E4M3 scale per 16 consecutive weights of a row, [rows, cols/16] bytes; one
 *                         fp32 scale per matrix: weight = decode(code) * decode(block scale) * matrix
 *                         scale (the drafter's NVFP4 post-training quantization, same page and section;
 *                         eagle3_quantize_nvfp4 produces this form).  Requires dtype == EAGLE3_BF16, an MLA
 *                         head, and every quantized matrix's cols a multiple of 32. */
typedef enum { EAGLE3_WEIGHTS_DTYPE = 0, EAGLE3_WEIGHTS_FP8 = 1, EAGLE3_WEIGHTS_NVFP4 = 2 } eagle3_weight_format_t;

/* Attention of the head's decoder layer.
 *   EAGLE3_ATTN_MLA  the DeepseekV3 draft (Eagle3DeepseekV2ForCausalLM): latent q/kv projections, one
 *                    latent cache row [c_kv_hat | k_rope] per token ("Eagle3 DeepseekV3 in MAX" §4, §7);
 *   EAGLE3_ATTN_MHA  the Llama-style draft (LlamaForCausalLMEagle3, "Eagle3 DeepseekV3 in MAX" §11):
 *                    q/k/v projections at 2H input, rotate-half RoPE on q and k (dimension i pairs with
 *                    i + head_dim/2), grouped-query attention (query head h reads key/value head
 *                    h / (n_heads / n_kv_heads)) over the head's own cache, whose row per token is
 *                    [k_rot (n_kv_heads x head_dim) | v (n_kv_heads x head_dim)]; softmax scale
 *                    head_dim^-1/2 times the squared YaRN attention factor.  The MLA sizes of the config
 *                    (q_lora_rank, kv_lora_rank, qk_nope_dim, qk_rope_dim, v_head_dim, rope_interleave) are
 *                    not used. */
typedef enum { EAGLE3_ATTN_MLA = 0, EAGLE3_ATTN_MHA = 1 } eagle3_attention_t;

/* Device error word bits (eagle3_draft_get_error). */
#define EAGLE3_DEVERR_TOKEN    1   /* an input token id was outside [0, target_vocab) */
#define EAGLE3_DEVERR_POSITION 2   /* a position was >= max_ctx */
#define EAGLE3_DEVERR_D2T      4   /* d + d2t[d] was outside [0, target_vocab) */
#define EAGLE3_DEVERR_PAGE     8   /* a position's page was outside the block table or the cache */
#define EAGLE3_DEVERR_ROWS     16  /* row_offsets were not non-decreasing within [0, num_tokens] */
#define EAGLE3_DEVERR_TIMEOUT  32  /* a bounded wait inside a tensor-core kernel ran out (work skipped) */

/* Head configuration (host struct, copied by create).  Field names follow the DeepseekV3 config
 * (MAX API reference, Eagle3DeepseekV3DraftConfig). */
typedef struct {
    int32_t hidden;               /* H */
    int32_t n_heads;              /* n_h */
    int32_t q_lora_rank;          /* d_q */
    int32_t kv_lora_rank;         /* d_c, the latent width cached per token */
    int32_t qk_nope_dim;          /* d_n */
    int32_t qk_rope_dim;          /* d_r, even */
    int32_t v_head_dim;           /* d_v */
    int32_t intermediate;         /* I of the dense MLP */
    int32_t target_vocab;         /* V_t: rows of the (borrowed, target's) embedding */
    int32_t draft_vocab;          /* V_d: rows of lm_head (== V_t when no d2t is used) */
    int32_t max_batch;            /* sequences per call */
    int32_t max_tokens_per_extend;/* rows per extend call */
    int32_t max_ctx;              /* positions must be < max_ctx */
    int32_t page_size;            /* cache slots per page */
    int32_t max_pages_per_seq;    /* columns of the block table */
    float rms_eps;                /* 1e-6 */
    float rope_theta;             /* 1e4 */
    float yarn_factor;            /* 1 disables YaRN */
    float yarn_beta_fast;         /* 32 */
    float yarn_beta_slow;         /* 1 */
    float yarn_mscale;            /* 1 */
    float yarn_mscale_all_dim;    /* 1 */
    int32_t yarn_original_max_pos;/* 4096 */
    int32_t rope_interleave;      /* must be 1: pairs (2i, 2i+1) rotate together */
    eagle3_dtype_t dtype;         /* storage type of weights, aux states and cache */
    eagle3_weight_format_t weight_format; /* storage of the projection matrices (0 = dtype) */
    eagle3_attention_t attention; /* 0 = MLA (the fields above), 1 = MHA (the fields below) */
    int32_t n_kv_heads;           /* MHA: key/value heads; n_heads a multiple of it (n_heads / n_kv_heads
                                   * in {1, 2, 4, 7, 8}) */
    int32_t head_dim;             /* MHA: d in {32, 64, 128} */
    int32_t fc_inputs;            /* aux states fc fuses: 3 (0 means 3), or 2 for an MHA head whose fc is
                                   * [H, 2H] (§11: the width is read from fc.weight) */
} eagle3_config_t;

/* Device pointers to the head's weights (BORROWED).  Shapes [rows, cols], row-major. */
typedef struct {
    const void *embed;          /* [V_t, H]   the target's embedding table */
    const void *fc;             /* [H, 3H]    columns: early | middle | late */
    const void *input_norm;     /* [H]        RMSNorm weight of the embedding stream */
    const void *hidden_norm;    /* [H]        RMSNorm weight of the fused stream */
    const void *q_a;            /* [d_q, 2H] */
    const void *q_a_norm;       /* [d_q] */
    const void *q_b;            /* [n_h*(d_n+d_r), d_q]  per head: nope rows then rope rows */
    const void *kv_a;           /* [d_c+d_r, 2H]         latent rows then rope rows */
    const void *kv_a_norm;      /* [d_c] */
    const void *kv_b;           /* [n_h*(d_n+d_v), d_c]  per head: key rows then value rows */
    const void *o;              /* [H, n_h*d_v] */
    const void *post_attn_norm; /* [H] */
    const void *gate;           /* [I, H] */
    const void *up;             /* [I, H] */
    const void *down;           /* [H, I] */
    const void *final_norm;     /* [H] */
    const void *lm_head;        /* [V_d, H] */
    /* Scales of the quantized matrices above (ignored for EAGLE3_WEIGHTS_DTYPE), for the matrix of the
     * same name: EAGLE3_WEIGHTS_FP8, the fp32 per-output-row scales [rows]; EAGLE3_WEIGHTS_NVFP4, the
     * E4M3 block scales [rows, cols/16] (bytes). */
    const void *fc_scale, *q_a_scale, *kv_a_scale, *q_b_scale, *o_scale, *gate_scale, *up_scale,
        *down_scale, *lm_head_scale;
    /* EAGLE3_ATTN_MHA only (its q_a, q_a_norm, q_b, kv_a, kv_a_norm and kv_b are unused and may be NULL;
     * its fc is [H, fc_inputs H] and its o [H, n_heads head_dim]): */
    const void *q_proj;         /* [n_heads head_dim, 2H] */
    const void *k_proj;         /* [n_kv_heads head_dim, 2H] */
    const void *v_proj;         /* [n_kv_heads head_dim, 2H] */
    /* EAGLE3_WEIGHTS_NVFP4 only: the nine matrix scales, fp32 [9], in the order fc, q_a, kv_a, q_b, o,
     * gate, up, down, lm_head. */
    const float *matrix_scales;
} eagle3_weights_t;

/* The one-layer latent cache (BORROWED).  Slot p of sequence b is row (p % page_size) of page
 * block_table[b * max_pages_per_seq + p / page_size].  A row is [c_kv_hat (d_c) | k_rope (d_r)],
 * the normalised latent and the ROTATED rope key, in the configured dtype. */
typedef struct {
    void *data;                 /* [num_pages, page_size, d_c + d_r] */
    const int32_t *block_table; /* [batch, max_pages_per_seq] */
    int32_t *lengths;           /* [batch] cached tokens per sequence; extend/decode advance it */
    int32_t num_pages;          /* host: pages in `data` */
} eagle3_kv_t;

typedef struct eagle3_draft eagle3_draft_t;

/* Create a head.  Validates the config (sizes > 0, d_r even, inner dims multiples of 8,
 * rope_interleave == 1), copies it, records the weight pointers, builds the YaRN cos/sin table
 * (fp64 on the host, stored fp32) and allocates the workspace on the current device.
 * Returns EAGLE3_ERR_INVALID_ARG / _UNSUPPORTED / _OOM / _CUDA; *out is NULL on failure. */
EAGLE3_API eagle3_status_t eagle3_draft_create(const eagle3_config_t *config, const eagle3_weights_t *weights,
                                    eagle3_draft_t **out);

/* Bytes of device workspace create allocates for `config` (host-only; no CUDA call). */
EAGLE3_API eagle3_status_t eagle3_draft_workspace_bytes(const eagle3_config_t *config, size_t *bytes);

/* Extend (draft step 0, "Eagle3 DeepseekV3 in MAX" §4 and §9): runs the whole head over
 * `num_tokens` new rows of `batch` sequences.
 *   aux_hidden  host array of 3 device pointers, each [num_tokens, H] (early, middle, late); with
 *               fc_inputs 2 only the first two are read (early, late) and the third may be NULL
 *   tokens      [num_tokens] target-vocab ids paired with the aux rows
 *   positions   [num_tokens] slot of each row; within a sequence strictly increasing, and every
 *               slot below a row's position must already hold that sequence's cache entry
 *   row_offsets [batch + 1] rows of sequence b are [row_offsets[b], row_offsets[b+1]), each >= 1
 * Appends each row's latent entry at its position, sets lengths[b] = last position + 1, keeps
 * the last row's hidden (before the final norm) and its draft-vocab argmax in the handle.
 * Optional debug outputs (NULL to skip): hidden_out [batch, H] fp32, logits_out [batch, V_d] fp32
 * of the last rows.  1 <= batch <= max_batch, batch <= num_tokens <= max_tokens_per_extend. */
EAGLE3_API eagle3_status_t eagle3_draft_extend(eagle3_draft_t *d, const void *const aux_hidden[3],
                                    const int32_t *tokens, const int32_t *positions,
                                    const int32_t *row_offsets, int32_t batch, int32_t num_tokens,
                                    eagle3_kv_t *cache, float *hidden_out, float *logits_out,
                                    void *stream);

/* Decode (draft steps 1..gamma-1, "Eagle3 DeepseekV3 in MAX" §9): writes
 * draft_tokens[b, 0] = remap(d0) for the argmax d0 kept by extend, then runs gamma - 1
 * autoregressive steps: step s embeds draft_tokens[:, s-1] at position lengths[b] with the
 * previous step's hidden as the fused state (fc skipped), appends its latent entry, advances
 * lengths, and writes draft_tokens[b, s].  remap(d) = d + d2t[d] when d2t is given ("EAGLE head
 * deep dive" part 4), else d.
 *   d2t           [V_d] int32 or NULL
 *   draft_tokens  [batch, gamma] int32 out, target-vocab ids
 *   hidden_out    [gamma - 1, batch, H] fp32 or NULL (hidden of each decode step)
 *   logits_out    [gamma - 1, batch, V_d] fp32 or NULL
 * `batch` is the last extend's.  Returns EAGLE3_ERR_STATE before any extend.  A second decode
 * without a new extend continues from the same kept state and appends after the current lengths. */
EAGLE3_API eagle3_status_t eagle3_draft_decode(eagle3_draft_t *d, int32_t gamma, const int32_t *d2t,
                                    eagle3_kv_t *cache, int32_t *draft_tokens, float *hidden_out,
                                    float *logits_out, void *stream);

/* One bias-free linear layer of the head's engine, exposed for callers and tests:
 * y[m, n] = sum_k x[m, k] w[n, k] with x [M, K] and w [N, K] bf16 (row-major), y [M, N] fp32.
 * It runs on the engine the head itself uses for M rows: the weight-streaming GEMV for M <= 8, the
 * tcgen05 tensor-core GEMM above (K must then be a multiple of 64).  Uses the handle's workspace
 * (so calls on one handle must not overlap) and reports timeouts in its error word.
 * Returns EAGLE3_ERR_UNSUPPORTED for an fp32 head. */
EAGLE3_API eagle3_status_t eagle3_linear(eagle3_draft_t *d, const void *x, const void *w, float *y, int32_t M,
                                         int32_t N, int32_t K, void *stream);

/* ---- Allocation-free linear layer.  The pages have no counterpart: this is an engineering addition
 * for callers that cannot allocate device memory on their call path.
 *
 * Computes the same product as eagle3_linear, y[m, n] = sum_k x[m, k] w[n, k] (x [M, K] and w [N, K]
 * bf16 row-major, y [M, N] fp32 row-major; device pointers, 16-byte aligned, owned by the caller), always
 * on the tcgen05 split-K tensor-core GEMM.  It takes no handle.  Its split-K partial sums live in one
 * fixed scratch array per device (EAGLE3_NOALLOC_SCRATCH_BYTES plus a 256-byte header) that the library
 * defines statically in device memory: every GPU that loads the library holds it until the process exits.
 * Neither the call nor its set-up calls cudaMalloc, cudaFree or any allocating library routine.
 *
 * Who needs it: a serving runtime that hands nearly all HBM to its own pool up front (weights, KV pages),
 * so a handle's workspace, sized for the largest batch, does not fit or would fragment that pool; and
 * latency-critical loops that must not reach cudaMalloc or cudaFree, which can synchronise the device.
 * Callers that can allocate should use eagle3_linear.
 *
 * Limits: M, N >= 1; K a multiple of 64; M * N <= EAGLE3_NOALLOC_SCRATCH_BYTES / 8 (= 2^21: two fp32
 * partial planes must fit).  A larger M * N returns EAGLE3_ERR_SCRATCH_LIMIT before any work is queued.
 * Set-up: the first call on each device (made with that device current) looks the scratch array's
 * address up with cudaGetSymbolAddress; make that first call before any stream capture begins.
 * Sharing: all calls on one device share the one scratch array, which keeps the last call's contents.
 * Calls ordered on one stream are safe; calls that can overlap on the GPU (different streams, or host
 * threads whose streams are not ordered) race on the scratch and corrupt each other's results.
 * Each call clears the scratch's device error word on `stream` before the GEMM.  A bounded wait that runs
 * out inside the GEMM (a failing device) leaves zeros in the affected outputs; this call does not report
 * it.  Returns EAGLE3_ERR_INVALID_ARG for a null or misaligned pointer or M, N, K < 1,
 * EAGLE3_ERR_UNSUPPORTED when K is not a multiple of 64, EAGLE3_ERR_CUDA when a CUDA call fails. */
#define EAGLE3_NOALLOC_SCRATCH_BYTES (16u << 20)
EAGLE3_API eagle3_status_t eagle3_linear_noalloc(const void *x, const void *w, float *y, int32_t M, int32_t N,
                                                 int32_t K, void *stream);

/* Greedy acceptance ("Eagle3 DeepseekV3 in MAX" §10): accepted_len[b] = number of leading
 * positions i with draft[b, i] == target[b, i] (0..gamma).  hist (optional, [gamma + 1]) is
 * overwritten with hist[k] = number of sequences with accepted_len == k.  No handle needed. */
EAGLE3_API eagle3_status_t eagle3_accept(const int32_t *draft, const int32_t *target, int32_t batch,
                              int32_t gamma, int32_t *accepted_len, int32_t *hist, void *stream);

/* Relaxed acceptance inside thinking blocks ("Eagle3 DeepseekV3 in MAX" §10: use_relaxed_acceptance_for_
 * thinking with relaxed_topk (default 10) and relaxed_delta (default 0.6); §8: the per-row
 * in_thinking_phase flag).  For each position i of sequence b the target supplies its k candidate
 * tokens and their log-probabilities.  A row whose in_thinking flag is set accepts the drafted token when
 * it is one of the candidates with log-probability >= the best candidate's log-probability - delta
 * (the threshold formed in fp64 from the single-precision inputs: the exact comparison); every other row accepts only the best candidate (the first listed among equal best).
 * accepted_len[b] = number of leading accepted positions (0..gamma).
 *   draft           [batch, gamma] int32
 *   topk_ids        [batch, gamma, k] int32
 *   topk_logprobs   [batch, gamma, k] fp32
 *   in_thinking     [batch] uint8 (non-zero = thinking) or NULL (no row is thinking: the greedy rule)
 *   accepted_len    [batch] int32 out; hist [gamma + 1] int32 out or NULL, as in eagle3_accept
 * All device pointers; no handle needed.  Returns EAGLE3_ERR_INVALID_ARG for null required pointers,
 * batch or gamma < 1, k < 1 or k > 1024, or a negative delta. */
EAGLE3_API eagle3_status_t eagle3_accept_relaxed(const int32_t *draft, const int32_t *topk_ids,
                                                 const float *topk_logprobs, const uint8_t *in_thinking,
                                                 int32_t batch, int32_t gamma, int32_t k, float delta,
                                                 int32_t *accepted_len, int32_t *hist, void *stream);

/* ---- Sampled drafts and residual acceptance ("Eagle3 DeepseekV3 in MAX" §3.1, §10: the sampling
 * parameters of the drafts and the rejection-sampling strategies; §8: a seed counter feeds the sampler).
 * The uniform random numbers are inputs (device arrays in [0, 1)), so every consumer of a draw sees the
 * same number. */
typedef struct {
    float temperature;   /* 0: greedy argmax (lowest index among equal maxima) */
    int32_t top_k;       /* 0: the whole vocabulary (top_p must then be 1); else 1..1024 */
    float top_p;         /* (0, 1]: keep the shortest prefix of the top_k tokens, by probability, whose mass
                            reaches top_p of their total */
} eagle3_sampling_t;

/* Draw one token per row from filtered logits: x = logits / temperature; keep the top_k largest x (lower
 * indices first among equal values; x is ordered as the logits are, so this set is exact), then the top_p
 * prefix in the order (x descending, index ascending) by the softmax mass of x (fp32 weights
 * exp((l - l_max) / temperature)); renormalise the kept weights and pick by inverse CDF over the kept
 * tokens in ascending index order with uniforms[r].
 *   logits       [rows, ld] fp32, the first V entries of each row are the draft-vocabulary logits
 *   uniforms     [rows] fp32
 *   d2t          [V] int32 additive draft-to-target map or NULL (tokens are then draft ids)
 *   tokens       [rows] int32 out, target-vocabulary ids
 *   token_prob   [rows] fp32 out or NULL: the drawn token's final probability
 *   probs        [rows, probs_len] fp32 out or NULL: the final distribution, indexed by target ids when
 *                probs_in_target is non-zero (zeros elsewhere), else by draft ids
 * One thread-block cluster of 8 CTAs per row, each CTA owning an eighth of the row's logits.  Returns
 * EAGLE3_ERR_INVALID_ARG for null required pointers, rows outside 1..65535, V < 1, V > 131072, ld < V, top_k
 * outside 0..1024, top_p outside (0, 1], top_p < 1 without top_k, or a negative temperature. */
EAGLE3_API eagle3_status_t eagle3_sample(const float *logits, int32_t rows, int32_t V, int64_t ld,
                                         const eagle3_sampling_t *params, const float *uniforms, const int32_t *d2t,
                                         int32_t target_vocab, int32_t *tokens, float *token_prob, float *probs,
                                         int32_t probs_len, int32_t probs_in_target, void *stream);

/* The decode of a sampled round: like eagle3_draft_decode, but every draft token is drawn with
 * eagle3_sample's rule instead of the argmax.  Token 0 is drawn from first_logits (the extend's logits of
 * the scored rows, [batch, V_d], from eagle3_draft_extend's logits_out) with uniforms[0, :]; decode step
 * s (1 <= s < gamma) draws from its own logits with uniforms[s, :] and feeds the drawn token (target id,
 * through d2t) to the next step.
 *   uniforms     [gamma, batch] fp32 in [0, 1)
 *   draft_tokens [batch, gamma] int32 out, target-vocabulary ids
 *   draft_probs  [batch, gamma, probs_len] fp32 out or NULL: each step's final distribution, indexed by
 *                target ids when probs_in_target is non-zero (the layout eagle3_accept_residual reads)
 *   hidden_out, logits_out: as in eagle3_draft_decode (logits of decode steps 1..gamma-1)
 * Returns EAGLE3_ERR_STATE before any extend, EAGLE3_ERR_INVALID_ARG as eagle3_sample and
 * eagle3_draft_decode do. */
EAGLE3_API eagle3_status_t eagle3_draft_decode_sampled(eagle3_draft_t *d, int32_t gamma, const int32_t *d2t,
                                                       eagle3_kv_t *cache, const eagle3_sampling_t *params,
                                                       const float *first_logits, const float *uniforms,
                                                       int32_t *draft_tokens, float *draft_probs, int32_t probs_len,
                                                       int32_t probs_in_target, float *hidden_out, float *logits_out,
                                                       void *stream);

/* Residual (rejection-sampling) acceptance: position i of sequence b accepts its drafted token x when
 * u_accept[b, i] * q(x) < p(x) (probability min(1, p(x) / q(x))); the first rejected position emits a
 * token drawn from max(0, p - q) renormalised, by inverse CDF in ascending token order with
 * u_resample[b, i]; if all gamma positions are accepted the emitted token is drawn from p_gamma with
 * u_resample[b, gamma - 1].
 *   draft         [batch, gamma] int32 target-vocabulary ids
 *   draft_probs   [batch, gamma, V] fp32: the draft's final distributions over the target vocabulary
 *   target_probs  [batch, gamma + 1, V] fp32
 *   u_accept, u_resample  [batch, gamma] fp32
 *   accepted_len  [batch] int32 out; next_token [batch] int32 out; hist [gamma + 1] int32 out or NULL
 * One CTA per sequence.  Returns EAGLE3_ERR_INVALID_ARG for null required pointers or sizes < 1. */
EAGLE3_API eagle3_status_t eagle3_accept_residual(const int32_t *draft, const float *draft_probs,
                                                  const float *target_probs, const float *u_accept,
                                                  const float *u_resample, int32_t batch, int32_t gamma, int32_t V,
                                                  int32_t *accepted_len, int32_t *next_token, int32_t *hist,
                                                  void *stream);

/* Typical acceptance ("Eagle3 DeepseekV3 in MAX" §10 names the typical-acceptance strategy of
 * --rejection-sampling-strategy without stating it; the rule here is the published one of Medusa, Cai
 * et al. 2024): position i of sequence b accepts its drafted token x while
 *   p_i(x) > min(epsilon, delta * exp(-H(p_i))),   H(p_i) = -sum_v p_i(v) ln p_i(v)  (nats),
 * p_i the target's distribution at that position; accepted_len[b] = number of leading accepted positions
 * (0..gamma); an id outside [0, V) is never accepted.  No bonus token is drawn: the caller takes the
 * target's own next token, as for greedy acceptance.  Medusa's defaults are epsilon 0.09, delta 0.3.
 *   draft         [batch, gamma] int32 target-vocabulary ids
 *   target_probs  [batch, gamma, V] fp32
 *   accepted_len  [batch] int32 out; hist [gamma + 1] int32 out or NULL, as in eagle3_accept
 * One CTA per sequence; the entropy is summed in fp32.  Returns EAGLE3_ERR_INVALID_ARG for null required
 * pointers, batch, gamma or V < 1, gamma > 4096, or a negative (or NaN) epsilon or delta. */
EAGLE3_API eagle3_status_t eagle3_accept_typical(const int32_t *draft, const float *target_probs, int32_t batch,
                                                 int32_t gamma, int32_t V, float epsilon, float delta,
                                                 int32_t *accepted_len, int32_t *hist, void *stream);

/* Device uniforms from a seed and a counter ("Eagle3 DeepseekV3 in MAX" §8: a seed counter feeds the
 * sampler), so a sampled round draws its random numbers without a host copy.  The generator is
 * Philox4x64-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011):
 * out[i] is word i mod 4 of the block whose 256-bit counter is offset + floor(i / 4) (little-endian
 * 64-bit words) under the key (seed, 0), its top 24 bits times 2^-24 (a value in [0, 1) exact in fp32).
 * Successive calls take fresh numbers by advancing offset by ceil(n / 4).
 *   out  [n] fp32 out (device memory)
 * Returns EAGLE3_ERR_INVALID_ARG for n < 0 or a null out with n > 0; n == 0 launches nothing. */
EAGLE3_API eagle3_status_t eagle3_philox_uniforms(uint64_t seed, uint64_t offset, int64_t n, float *out,
                                                  void *stream);

/* Per-row FP8 E4M3 quantization of one weight matrix (the drafter's post-training FP8 quantization,
 * "EAGLE head deep dive", deployment; the form EAGLE3_WEIGHTS_FP8 reads).  For every row n of w:
 *   scale[n] = max_k |w[n, k]| / 448 in fp32 (1 for an all-zero row),
 *   code[n, k] = E4M3(w[n, k] / scale[n]): the fp32 quotient rounded to the nearest E4M3 value, ties to
 *   the even code, magnitudes above 448 saturating to 448.
 *   w       [N, K] of `dtype` (bf16 or fp32), row-major
 *   codes   [N, K] uint8 out; scales [N] fp32 out (both caller-owned device memory)
 * One CTA per row.  Returns EAGLE3_ERR_INVALID_ARG for null pointers or sizes < 1, _UNSUPPORTED for
 * another dtype. */
EAGLE3_API eagle3_status_t eagle3_quantize_e4m3(const void *w, eagle3_dtype_t dtype, int32_t N, int32_t K,
                                                uint8_t *codes, float *scales, void *stream);

/* NVFP4 quantization of one weight matrix (the drafter's post-training NVFP4 quantization, "EAGLE head
 * deep dive", deployment; the form EAGLE3_WEIGHTS_NVFP4 reads), all in fp32:
 *   g = max |w| / 2688 (= 448 * 6; 1 for an all-zero matrix),
 *   s_b = E4M3(max_{k in block b} |w[n, k]| / (6 g)) for each 16 consecutive weights of a row (6 g rounded
 *   first; nearest, ties to even, saturating),
 *   e_b = decode(s_b) * g, code = E2M1(w / e_b) (nearest, ties to the even code, saturating at 6; 0 where
 *   e_b is 0).
 *   w             [N, K] of `dtype` (bf16 or fp32), K a multiple of 32
 *   codes         [N, K/2] uint8 out, two codes per byte, the even element in the low nibble
 *   block_scales  [N, K/16] uint8 out (E4M3); global_scale [1] fp32 out (g)
 * Four launches (matrix maximum, codes, scale).  Returns EAGLE3_ERR_INVALID_ARG for null pointers or
 * sizes < 1, _UNSUPPORTED for K not a multiple of 32 or another dtype. */
EAGLE3_API eagle3_status_t eagle3_quantize_nvfp4(const void *w, eagle3_dtype_t dtype, int32_t N, int32_t K,
                                                 uint8_t *codes, uint8_t *block_scales, float *global_scale,
                                                 void *stream);

/* Read the sticky device error word (synchronises the device).  *device_error (host) receives
 * the EAGLE3_DEVERR_* bits; returns EAGLE3_ERR_DEVICE_RANGE when any bit is set. */
EAGLE3_API eagle3_status_t eagle3_draft_get_error(eagle3_draft_t *d, int32_t *device_error);

/* Clear the sticky device error word (asynchronous on `stream`). */
EAGLE3_API eagle3_status_t eagle3_draft_clear_error(eagle3_draft_t *d, void *stream);

/* Free the workspace and the handle (synchronises the device).  NULL is accepted. */
EAGLE3_API eagle3_status_t eagle3_draft_destroy(eagle3_draft_t *d);

/* ---- Per-kernel timing (native tracing).  Every launch of a kernel kind whose bit is set in
 * `kind_mask` (bit k = kind k; -1 = all kinds, 0 = off) is bracketed by CUDA events recorded on the
 * launch stream (as graph timestamp nodes when the stream is being captured); read() synchronises and
 * accumulates the event intervals per kind.  Launches are counted whether or not they are timed.
 * Turning timing off flushes the pending intervals. */
#define EAGLE3_PROF_KINDS 24
EAGLE3_API eagle3_status_t eagle3_draft_profile_enable(eagle3_draft_t *d, int32_t kind_mask);
/* For kernel kind `kind` (0 <= kind < EAGLE3_PROF_KINDS) since the last reset: total milliseconds over
 * the timed launches, the number of timed launches, and the number of launches (timed or not; the
 * event pool times at most 32768 launches between reads).  Synchronises the device.  Launches recorded
 * inside a CUDA graph report the intervals of the graph's latest replay.  *name (host, optional)
 * receives a static kernel name. */
EAGLE3_API eagle3_status_t eagle3_draft_profile_read(eagle3_draft_t *d, int32_t kind, double *total_ms,
                                                     int64_t *timed, int64_t *launches, const char **name);
EAGLE3_API eagle3_status_t eagle3_draft_profile_reset(eagle3_draft_t *d);

/* Static string for a status code. */
EAGLE3_API const char *eagle3_status_string(eagle3_status_t s);

/* The last CUDA error code seen by this library on this thread (0 if none). */
EAGLE3_API int32_t eagle3_last_cuda_error(void);

#ifdef __cplusplus
}
#endif
#endif /* EAGLE3_H */
