// Per-row kernels of the draft head: the embedding gather with the two input RMSNorms and the
// 2H concat, the latent norms with rope-key rotation and the cache append, RMSNorm, the
// scored-row epilogue, the argmax reduction with the d2t remap, and greedy acceptance.
#include <float.h>
#include <limits.h>

#include "common.cuh"
#include "kernels.h"
#include "../../include/eagle3.h"

namespace e3 {

constexpr int kRowThreads = 256;
constexpr int kVecThreads = 1024;   // row kernels over H: one 8-element chunk per thread (two above 8192)
constexpr int kVecChunks = 2;

// Block-wide sums of two values; `scratch` holds >= 64 floats.
__device__ __forceinline__ float2 block_sum2(float a, float b, float* scratch) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    a = warp_sum(a);
    b = warp_sum(b);
    __syncthreads();
    if (lane == 0) { scratch[w] = a; scratch[32 + w] = b; }
    __syncthreads();
    float ta = (lane < nw) ? scratch[lane] : 0.f, tb = (lane < nw) ? scratch[32 + lane] : 0.f;
    return make_float2(warp_sum(ta), warp_sum(tb));
}

template <typename T> __device__ __forceinline__ void load_row8(const T* p, float* v) { widen(ld8<false>(p), v); }
__device__ __forceinline__ void store_bf8(bf16* p, const float* v) {
    uint4 u;
    u.x = pack2_bf16(v[0], v[1]); u.y = pack2_bf16(v[2], v[3]);
    u.z = pack2_bf16(v[4], v[5]); u.w = pack2_bf16(v[6], v[7]);
    *reinterpret_cast<uint4*>(p) = u;
}
__device__ __forceinline__ void store_row8(float* p, const float* v) {
    reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}

// x[r] = [ RMS(E[token]) * w_in | RMS(fused[r]) * w_hid ]  (2H wide), in fp32 (x, for the GEMV) and/or bf16
// (x_bf, for the tensor-core GEMM); either may be null.
// The token embedding is the target's table ("Eagle3 DeepseekV3 in MAX" §5); the two streams are
// normalised separately and concatenated ("EAGLE head deep dive" part 3; MAX §4).
template <typename T>
__global__ void __launch_bounds__(kVecThreads)
embed_norms_kernel(RowArgs a, int decode, const int* tokens, const int* positions, const int* row_offsets,
                   int batch, int M, const int* tok_in, const int* lengths, const float* fused,
                   const T* embed, const T* w_in, const T* w_hid, float* x, bf16* x_bf, int* row_seq,
                   int* row_pos) {
    pdl_trigger();
    pdl_wait();
    __shared__ float red[64];
    const int r = blockIdx.x;
    int b, tok, pos;
    if (decode) {
        b = r;
        tok = tok_in[r];
        pos = lengths[r];
    } else {
        tok = tokens[r];
        pos = positions[r];
        int lo = 0, hi = batch - 1;   // largest b with row_offsets[b] <= r
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (row_offsets[mid] <= r) lo = mid; else hi = mid - 1;
        }
        b = lo;
        if (r == 0) {
            for (int t = threadIdx.x; t < batch; t += blockDim.x) {
                const bool bad = row_offsets[t] >= row_offsets[t + 1] || (t == 0 && row_offsets[0] != 0) ||
                                 (t == batch - 1 && row_offsets[batch] != M);
                if (bad) set_err(a.err, EAGLE3_DEVERR_ROWS);
            }
        }
    }
    if (tok < 0 || tok >= a.Vt) {
        if (threadIdx.x == 0) set_err(a.err, EAGLE3_DEVERR_TOKEN);
        tok = tok < 0 ? 0 : a.Vt - 1;
    }
    if (pos < 0 || pos >= a.max_ctx) {
        if (threadIdx.x == 0) set_err(a.err, EAGLE3_DEVERR_POSITION);
        pos = pos < 0 ? 0 : a.max_ctx - 1;
    }
    if (threadIdx.x == 0) { row_seq[r] = b; row_pos[r] = pos; }
    const int H = a.H, nch = H / 8;
    const T* e = embed + (long)tok * H;
    const float* f = fused + (long)r * H;
    float ev[kVecChunks][8], fv[kVecChunks][8];
    float se = 0.f, sf = 0.f;
#pragma unroll
    for (int i = 0; i < kVecChunks; ++i) {
        const int c = threadIdx.x + i * blockDim.x;
        if (c < nch) {
            load_row8(e + 8 * c, ev[i]);
            load_row8(f + 8 * c, fv[i]);
#pragma unroll
            for (int k = 0; k < 8; ++k) { se += ev[i][k] * ev[i][k]; sf += fv[i][k] * fv[i][k]; }
        }
    }
    const float2 ss = block_sum2(se, sf, red);
    const float ie = rsqrtf(ss.x / H + a.eps), iff = rsqrtf(ss.y / H + a.eps);
    float* xr = x + (long)r * 2 * H;
#pragma unroll
    for (int i = 0; i < kVecChunks; ++i) {
        const int c = threadIdx.x + i * blockDim.x;
        if (c < nch) {
            float wi[8], wh[8], o1[8], o2[8];
            load_row8(w_in + 8 * c, wi);
            load_row8(w_hid + 8 * c, wh);
#pragma unroll
            for (int k = 0; k < 8; ++k) { o1[k] = ev[i][k] * ie * wi[k]; o2[k] = fv[i][k] * iff * wh[k]; }
            if (x) {
                store_row8(xr + 8 * c, o1);
                store_row8(xr + H + 8 * c, o2);
            }
            if (x_bf) {
                store_bf8(x_bf + (long)r * 2 * H + 8 * c, o1);
                store_bf8(x_bf + (long)r * 2 * H + H + 8 * c, o2);
            }
        }
    }
}

// c_q_hat = RMS(c_q) * w_qa;  c_kv_hat = RMS(c_kv) * w_kva;  k_rope rotated at the row's position;
// [c_kv_hat | k_rope_rot] appended to the one-layer cache at slot = position.
template <typename T>
__global__ void __launch_bounds__(kRowThreads)
latent_kernel(RowArgs a, const float* cqkv, const T* w_qa, const T* w_kva, const float* rope_cos,
              const float* rope_sin, const int* row_seq, const int* row_pos, const int* block_table, T* cache,
              float* cq_hat, bf16* cqh_bf) {
    pdl_trigger();
    pdl_wait();
    __shared__ float red[64];
    const int r = blockIdx.x;
    const int dq = a.dq, dc = a.dc, dr = a.dr;
    const float* cq = cqkv + (long)r * (dq + dc + dr);
    const float* ckv = cq + dq;
    const float* kr = ckv + dc;
    const int t = threadIdx.x;
    float qv[8], cv[8];
    float s1 = 0.f, s2 = 0.f;
    if (t < dq / 8) {
        load_row8(cq + 8 * t, qv);
#pragma unroll
        for (int k = 0; k < 8; ++k) s1 += qv[k] * qv[k];
    }
    if (t < dc / 8) {
        load_row8(ckv + 8 * t, cv);
#pragma unroll
        for (int k = 0; k < 8; ++k) s2 += cv[k] * cv[k];
    }
    const float2 ss = block_sum2(s1, s2, red);
    const float i1 = rsqrtf(ss.x / dq + a.eps), i2 = rsqrtf(ss.y / dc + a.eps);
    if (t < dq / 8) {
        float w[8];
        load_row8(w_qa + 8 * t, w);
#pragma unroll
        for (int k = 0; k < 8; ++k) qv[k] *= i1 * w[k];
        store_row8(cq_hat + (long)r * dq + 8 * t, qv);
        if (cqh_bf) store_bf8(cqh_bf + (long)r * dq + 8 * t, qv);
    }
    const int b = row_seq[r], pos = row_pos[r];
    const int pi = pos / a.page_size;
    int page = -1;
    if (pi < a.max_pages) page = block_table[(long)b * a.max_pages + pi];
    if (page < 0 || page >= a.num_pages) {
        if (t == 0) set_err(a.err, EAGLE3_DEVERR_PAGE);
        return;
    }
    T* dst = cache + ((long)page * a.page_size + pos % a.page_size) * (dc + dr);
    if (t < dc / 8) {
        float w[8];
        load_row8(w_kva + 8 * t, w);
#pragma unroll
        for (int k = 0; k < 8; ++k) dst[8 * t + k] = from_f<T>(cv[k] * i2 * w[k]);
    }
    const int half = dr / 2;
    for (int i = t; i < half; i += blockDim.x) {
        const float c = rope_cos[(long)pos * half + i], s = rope_sin[(long)pos * half + i];
        const float x0 = kr[2 * i], x1 = kr[2 * i + 1];
        dst[dc + 2 * i] = from_f<T>(x0 * c - x1 * s);
        dst[dc + 2 * i + 1] = from_f<T>(x0 * s + x1 * c);
    }
}

template <typename T>
__global__ void __launch_bounds__(kVecThreads)
rmsnorm_kernel(int H, float eps, const float* x, const T* w, float* y, bf16* y_bf) {
    pdl_trigger();
    pdl_wait();
    __shared__ float red[64];
    const long r = blockIdx.x;
    const int nch = H / 8;
    const float* xr = x + r * H;
    float v[kVecChunks][8];
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kVecChunks; ++i) {
        const int c = threadIdx.x + i * blockDim.x;
        if (c < nch) {
            load_row8(xr + 8 * c, v[i]);
#pragma unroll
            for (int k = 0; k < 8; ++k) s += v[i][k] * v[i][k];
        }
    }
    const float inv = rsqrtf(block_sum2(s, 0.f, red).x / H + eps);
#pragma unroll
    for (int i = 0; i < kVecChunks; ++i) {
        const int c = threadIdx.x + i * blockDim.x;
        if (c < nch) {
            float wv[8];
            load_row8(w + 8 * c, wv);
#pragma unroll
            for (int k = 0; k < 8; ++k) v[i][k] *= inv * wv[k];
            if (y) store_row8(y + r * H + 8 * c, v[i]);
            if (y_bf) store_bf8(y_bf + r * H + 8 * c, v[i]);
        }
    }
}

// Scored row of each sequence (the last new row in extend, MAX §4 "gather last token"):
// carry its hidden to the next step, normalise it for the lm_head, advance the cache length.
template <typename T>
__global__ void __launch_bounds__(kVecThreads)
final_kernel(RowArgs a, int extend, int M, const int* row_offsets, const float* h2, const T* w_final,
             const int* row_pos, float* carry, float* z, bf16* z_bf, float* hidden_out, int* lengths) {
    pdl_trigger();
    pdl_wait();
    __shared__ float red[64];
    const int b = blockIdx.x;
    int src = extend ? row_offsets[b + 1] - 1 : b;
    if (src < 0 || src >= M) {   // malformed row_offsets (also flagged by the embedding kernel)
        if (threadIdx.x == 0) set_err(a.err, EAGLE3_DEVERR_ROWS);
        src = src < 0 ? 0 : M - 1;
    }
    const int H = a.H, nch = H / 8;
    const float* h = h2 + (long)src * H;
    float v[kVecChunks][8];
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kVecChunks; ++i) {
        const int c = threadIdx.x + i * blockDim.x;
        if (c < nch) {
            load_row8(h + 8 * c, v[i]);
#pragma unroll
            for (int k = 0; k < 8; ++k) s += v[i][k] * v[i][k];
            store_row8(carry + (long)b * H + 8 * c, v[i]);
            if (hidden_out) store_row8(hidden_out + (long)b * H + 8 * c, v[i]);
        }
    }
    const float inv = rsqrtf(block_sum2(s, 0.f, red).x / H + a.eps);
#pragma unroll
    for (int i = 0; i < kVecChunks; ++i) {
        const int c = threadIdx.x + i * blockDim.x;
        if (c < nch) {
            float wv[8];
            load_row8(w_final + 8 * c, wv);
#pragma unroll
            for (int k = 0; k < 8; ++k) v[i][k] *= inv * wv[k];
            store_row8(z + (long)b * H + 8 * c, v[i]);
            if (z_bf) store_bf8(z_bf + (long)b * H + 8 * c, v[i]);
        }
    }
    if (threadIdx.x == 0) lengths[b] = row_pos[src] + 1;
}

__device__ __forceinline__ int remap_token(int d, const int* d2t, int Vt, int* err) {
    long t = d;
    if (d2t != nullptr) t += d2t[d];
    if (t < 0 || t >= Vt) {
        set_err(err, EAGLE3_DEVERR_D2T);
        t = t < 0 ? 0 : Vt - 1;
    }
    return (int)t;
}

__global__ void __launch_bounds__(kRowThreads)
argmax_final_kernel(int npart, const float* pval, const int* pidx, int mode, const int* d2t, int Vt, int* d0,
                    int* out_tokens, int gamma, int s, int* tok_in, int* err) {
    pdl_trigger();
    pdl_wait();
    __shared__ float sv[kRowThreads / 32];
    __shared__ int si[kRowThreads / 32];
    const int b = blockIdx.x;
    float bv = -FLT_MAX;
    int bi = INT_MAX;
    for (int p = threadIdx.x; p < npart; p += blockDim.x) {
        const float v = pval[(long)b * npart + p];
        const int i = pidx[(long)b * npart + p];
        if (better(v, i, bv, bi)) { bv = v; bi = i; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float v = __shfl_xor_sync(0xffffffffu, bv, o);
        const int i = __shfl_xor_sync(0xffffffffu, bi, o);
        if (better(v, i, bv, bi)) { bv = v; bi = i; }
    }
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    if (lane == 0) { sv[w] = bv; si[w] = bi; }
    __syncthreads();
    if (threadIdx.x == 0) {
        bv = sv[0]; bi = si[0];
        for (int k = 1; k < (int)(blockDim.x >> 5); ++k)
            if (better(sv[k], si[k], bv, bi)) { bv = sv[k]; bi = si[k]; }
        if (bi == INT_MAX) bi = 0;   // every logit NaN: keep a valid id
        if (mode == 0) {
            d0[b] = bi;
        } else {
            const int t = remap_token(bi, d2t, Vt, err);
            out_tokens[(long)b * gamma + s] = t;
            tok_in[b] = t;
        }
    }
}

__global__ void emit_first_kernel(int batch, const int* d0, const int* d2t, int Vt, int* out_tokens, int gamma,
                                  int* tok_in, int* err) {
    pdl_trigger();
    pdl_wait();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= batch) return;
    const int t = remap_token(d0[b], d2t, Vt, err);
    out_tokens[(long)b * gamma] = t;
    tok_in[b] = t;
}

// accepted_len[b] = leading positions where draft == target ("Eagle3 DeepseekV3 in MAX" §10).
__global__ void __launch_bounds__(kRowThreads)
accept_kernel(const int* draft, const int* target, int batch, int gamma, int* acc, int* hist) {
    pdl_trigger();
    pdl_wait();
    extern __shared__ int sh[];
    for (int k = threadIdx.x; k <= gamma; k += blockDim.x) sh[k] = 0;
    __syncthreads();
    for (int b = threadIdx.x; b < batch; b += blockDim.x) {
        int k = 0;
        while (k < gamma && draft[(long)b * gamma + k] == target[(long)b * gamma + k]) ++k;
        acc[b] = k;
        if (hist) atomicAdd(&sh[k], 1);
    }
    __syncthreads();
    if (hist)
        for (int k = threadIdx.x; k <= gamma; k += blockDim.x) hist[k] = sh[k];
}

// Relaxed acceptance ("Eagle3 DeepseekV3 in MAX" §10: use_relaxed_acceptance_for_thinking, relaxed_topk,
// relaxed_delta; §8: the per-row in_thinking_phase flag).  Position i of a thinking row accepts a draft
// token listed among the target's k candidates with log-probability >= the best candidate's - delta;
// other rows accept only the best candidate (the first listed among equal best).  One thread per row.
// The threshold is formed in fp64 from the single-precision inputs, so the comparison is the exact
// real-number one and not subject to a single-precision rounding of best - delta.
__global__ void __launch_bounds__(kRowThreads)
accept_relaxed_kernel(const int* draft, const int* ids, const float* lp, const unsigned char* think, int batch,
                      int gamma, int k, float delta, int* acc, int* hist) {
    pdl_trigger();
    pdl_wait();
    extern __shared__ int sh[];
    for (int j = threadIdx.x; j <= gamma; j += blockDim.x) sh[j] = 0;
    __syncthreads();
    for (int b = threadIdx.x; b < batch; b += blockDim.x) {
        const bool relaxed = think != nullptr && think[b] != 0;
        int n = 0;
        for (; n < gamma; ++n) {
            const long pos = (long)b * gamma + n;
            const int* ci = ids + pos * k;
            const float* cl = lp + pos * k;
            const int tok = draft[pos];
            float best = cl[0];
            int first = 0;
            for (int j = 1; j < k; ++j)
                if (cl[j] > best) { best = cl[j]; first = j; }
            bool ok;
            if (!relaxed) {
                ok = tok == ci[first];
            } else {
                const double thr = (double)best - (double)delta;
                ok = false;
                for (int j = 0; j < k; ++j) ok = ok || (ci[j] == tok && (double)cl[j] >= thr);
            }
            if (!ok) break;
        }
        acc[b] = n;
        if (hist) atomicAdd(&sh[n], 1);
    }
    __syncthreads();
    if (hist)
        for (int j = threadIdx.x; j <= gamma; j += blockDim.x) hist[j] = sh[j];
}

// ------------------------------------------------------------------------------------------ launchers
cudaError_t launch_embed_norms(const RowArgs& a, bool decode, int M, const int* tokens, const int* positions,
                               const int* row_offsets, int batch, const int* tok_in, const int* lengths,
                               const float* fused, const void* embed, const void* w_in, const void* w_hid,
                               float* x, __nv_bfloat16* x_bf, int* row_seq, int* row_pos, cudaStream_t st) {
    if (a.dt == BF16)
        launch_pdl(embed_norms_kernel<bf16>, dim3(M), dim3(kVecThreads), 0, st, a, decode, tokens, positions, row_offsets, batch, M,
            tok_in, lengths, fused, (const bf16*)embed, (const bf16*)w_in, (const bf16*)w_hid, x, x_bf, row_seq, row_pos);
    else
        launch_pdl(embed_norms_kernel<float>, dim3(M), dim3(kVecThreads), 0, st, a, decode, tokens, positions, row_offsets, batch, M,
            tok_in, lengths, fused, (const float*)embed, (const float*)w_in, (const float*)w_hid, x, x_bf, row_seq, row_pos);
    return cudaGetLastError();
}

cudaError_t launch_latent(const RowArgs& a, int M, const float* cqkv, const void* w_qa, const void* w_kva,
                          const float* rope_cos, const float* rope_sin, const int* row_seq, const int* row_pos,
                          const int* block_table, void* cache, float* cq_hat, __nv_bfloat16* cqh_bf, cudaStream_t st) {
    if (a.dt == BF16)
        launch_pdl(latent_kernel<bf16>, dim3(M), dim3(kRowThreads), 0, st, a, cqkv, (const bf16*)w_qa, (const bf16*)w_kva, rope_cos,
            rope_sin, row_seq, row_pos, block_table, (bf16*)cache, cq_hat, cqh_bf);
    else
        launch_pdl(latent_kernel<float>, dim3(M), dim3(kRowThreads), 0, st, a, cqkv, (const float*)w_qa, (const float*)w_kva, rope_cos,
            rope_sin, row_seq, row_pos, block_table, (float*)cache, cq_hat, cqh_bf);
    return cudaGetLastError();
}

cudaError_t launch_rmsnorm(int M, int H, float eps, DType wt, const float* x, const void* w, float* y,
                           __nv_bfloat16* y_bf, cudaStream_t st) {
    if (wt == BF16) launch_pdl(rmsnorm_kernel<bf16>, dim3(M), dim3(kVecThreads), 0, st, H, eps, x, (const bf16*)w, y, y_bf);
    else launch_pdl(rmsnorm_kernel<float>, dim3(M), dim3(kVecThreads), 0, st, H, eps, x, (const float*)w, y, y_bf);
    return cudaGetLastError();
}

cudaError_t launch_final(const RowArgs& a, bool extend, int batch, int M, const int* row_offsets, const float* h2,
                         const void* w_final, const int* row_pos, float* carry, float* z, __nv_bfloat16* z_bf,
                         float* hidden_out, int* lengths, cudaStream_t st) {
    if (a.dt == BF16)
        launch_pdl(final_kernel<bf16>, dim3(batch), dim3(kVecThreads), 0, st, a, extend, M, row_offsets, h2, (const bf16*)w_final,
                                                          row_pos, carry, z, z_bf, hidden_out, lengths);
    else
        launch_pdl(final_kernel<float>, dim3(batch), dim3(kVecThreads), 0, st, a, extend, M, row_offsets, h2, (const float*)w_final,
                                                           row_pos, carry, z, z_bf, hidden_out, lengths);
    return cudaGetLastError();
}

cudaError_t launch_argmax_final(int batch, int npart, const float* pval, const int* pidx, int mode,
                                const int* d2t, int Vt, int* d0, int* out_tokens, int gamma, int s,
                                int* tok_in, int* err, cudaStream_t st) {
    launch_pdl(argmax_final_kernel, dim3(batch), dim3(kRowThreads), 0, st, npart, pval, pidx, mode, d2t, Vt, d0, out_tokens, gamma, s,
                                                       tok_in, err);
    return cudaGetLastError();
}

cudaError_t launch_emit_first(int batch, const int* d0, const int* d2t, int Vt, int* out_tokens, int gamma,
                              int* tok_in, int* err, cudaStream_t st) {
    launch_pdl(emit_first_kernel, dim3((batch + 127) / 128), dim3(128), 0, st, batch, d0, d2t, Vt, out_tokens, gamma, tok_in, err);
    return cudaGetLastError();
}

cudaError_t launch_accept(const int* draft, const int* target, int batch, int gamma, int* acc, int* hist,
                          cudaStream_t st) {
    launch_pdl(accept_kernel, dim3(1), dim3(kRowThreads), (gamma + 1) * sizeof(int), st, draft, target, batch, gamma, acc, hist);
    return cudaGetLastError();
}

cudaError_t launch_accept_relaxed(const int* draft, const int* ids, const float* lp, const unsigned char* think,
                                  int batch, int gamma, int k, float delta, int* acc, int* hist, cudaStream_t st) {
    launch_pdl(accept_relaxed_kernel, dim3(1), dim3(kRowThreads), (gamma + 1) * sizeof(int), st, draft, ids, lp, think,
               batch, gamma, k, delta, acc, hist);
    return cudaGetLastError();
}

}  // namespace e3
