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

// x[r] = [ RMS(E[token]) * w_in | RMS(fused[r]) * w_hid ]  (2H wide).
// The token embedding is the target's table ("Eagle3 DeepseekV3 in MAX" §5); the two streams are
// normalised separately and concatenated ("EAGLE head deep dive" part 3; MAX §4).
template <typename T>
__global__ void __launch_bounds__(kRowThreads)
embed_norms_kernel(RowArgs a, int decode, const int* tokens, const int* positions, const int* row_offsets,
                   int batch, int M, const int* tok_in, const int* lengths, const float* fused,
                   const T* embed, const T* w_in, const T* w_hid, float* x, int* row_seq, int* row_pos) {
    __shared__ float red[32];
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
    const int H = a.H;
    const T* e = embed + (long)tok * H;
    const float* f = fused + (long)r * H;
    float se = 0.f, sf = 0.f;
    for (int k = threadIdx.x; k < H; k += blockDim.x) {
        const float ev = to_f(e[k]);
        const float fv = f[k];
        se += ev * ev;
        sf += fv * fv;
    }
    se = block_sum(se, red);
    sf = block_sum(sf, red);
    const float ie = rsqrtf(se / H + a.eps), iff = rsqrtf(sf / H + a.eps);
    float* xr = x + (long)r * 2 * H;
    for (int k = threadIdx.x; k < H; k += blockDim.x) {
        xr[k] = to_f(e[k]) * ie * to_f(w_in[k]);
        xr[H + k] = f[k] * iff * to_f(w_hid[k]);
    }
}

// c_q_hat = RMS(c_q) * w_qa;  c_kv_hat = RMS(c_kv) * w_kva;  k_rope rotated at the row's position;
// [c_kv_hat | k_rope_rot] appended to the one-layer cache at slot = position.
template <typename T>
__global__ void __launch_bounds__(kRowThreads)
latent_kernel(RowArgs a, const float* cqkv, const T* w_qa, const T* w_kva, const float* rope_cos,
              const float* rope_sin, const int* row_seq, const int* row_pos, const int* block_table, T* cache,
              float* cq_hat) {
    __shared__ float red[32];
    const int r = blockIdx.x;
    const int dq = a.dq, dc = a.dc, dr = a.dr;
    const float* cq = cqkv + (long)r * (dq + dc + dr);
    const float* ckv = cq + dq;
    const float* kr = ckv + dc;
    float s1 = 0.f, s2 = 0.f;
    for (int k = threadIdx.x; k < dq; k += blockDim.x) s1 += cq[k] * cq[k];
    for (int k = threadIdx.x; k < dc; k += blockDim.x) s2 += ckv[k] * ckv[k];
    s1 = block_sum(s1, red);
    s2 = block_sum(s2, red);
    const float i1 = rsqrtf(s1 / dq + a.eps), i2 = rsqrtf(s2 / dc + a.eps);
    for (int k = threadIdx.x; k < dq; k += blockDim.x) cq_hat[(long)r * dq + k] = cq[k] * i1 * to_f(w_qa[k]);

    const int b = row_seq[r], pos = row_pos[r];
    const int pi = pos / a.page_size;
    int page = -1;
    if (pi < a.max_pages) page = block_table[(long)b * a.max_pages + pi];
    if (page < 0 || page >= a.num_pages) {
        if (threadIdx.x == 0) set_err(a.err, EAGLE3_DEVERR_PAGE);
        return;
    }
    T* dst = cache + ((long)page * a.page_size + pos % a.page_size) * (dc + dr);
    for (int k = threadIdx.x; k < dc; k += blockDim.x) dst[k] = from_f<T>(ckv[k] * i2 * to_f(w_kva[k]));
    const int half = dr / 2;
    for (int i = threadIdx.x; i < half; i += blockDim.x) {
        const float c = rope_cos[(long)pos * half + i], s = rope_sin[(long)pos * half + i];
        const float x0 = kr[2 * i], x1 = kr[2 * i + 1];
        dst[dc + 2 * i] = from_f<T>(x0 * c - x1 * s);
        dst[dc + 2 * i + 1] = from_f<T>(x0 * s + x1 * c);
    }
}

template <typename T>
__global__ void __launch_bounds__(kRowThreads)
rmsnorm_kernel(int H, float eps, const float* x, const T* w, float* y) {
    __shared__ float red[32];
    const long r = blockIdx.x;
    const float* xr = x + r * H;
    float s = 0.f;
    for (int k = threadIdx.x; k < H; k += blockDim.x) s += xr[k] * xr[k];
    s = block_sum(s, red);
    const float inv = rsqrtf(s / H + eps);
    for (int k = threadIdx.x; k < H; k += blockDim.x) y[r * H + k] = xr[k] * inv * to_f(w[k]);
}

// Scored row of each sequence (the last new row in extend, MAX §4 "gather last token"):
// carry its hidden to the next step, normalise it for the lm_head, advance the cache length.
template <typename T>
__global__ void __launch_bounds__(kRowThreads)
final_kernel(RowArgs a, int extend, const int* row_offsets, const float* h2, const T* w_final, const int* row_pos,
             float* carry, float* z, float* hidden_out, int* lengths) {
    __shared__ float red[32];
    const int b = blockIdx.x;
    const int src = extend ? row_offsets[b + 1] - 1 : b;
    const int H = a.H;
    const float* h = h2 + (long)(src < 0 ? 0 : src) * H;
    float s = 0.f;
    for (int k = threadIdx.x; k < H; k += blockDim.x) {
        const float v = h[k];
        s += v * v;
        carry[(long)b * H + k] = v;
        if (hidden_out) hidden_out[(long)b * H + k] = v;
    }
    s = block_sum(s, red);
    const float inv = rsqrtf(s / H + a.eps);
    for (int k = threadIdx.x; k < H; k += blockDim.x) z[(long)b * H + k] = h[k] * inv * to_f(w_final[k]);
    if (threadIdx.x == 0) lengths[b] = row_pos[src < 0 ? 0 : src] + 1;
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
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= batch) return;
    const int t = remap_token(d0[b], d2t, Vt, err);
    out_tokens[(long)b * gamma] = t;
    tok_in[b] = t;
}

// accepted_len[b] = leading positions where draft == target ("Eagle3 DeepseekV3 in MAX" §10).
__global__ void __launch_bounds__(kRowThreads)
accept_kernel(const int* draft, const int* target, int batch, int gamma, int* acc, int* hist) {
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

// ------------------------------------------------------------------------------------------ launchers
cudaError_t launch_embed_norms(const RowArgs& a, bool decode, int M, const int* tokens, const int* positions,
                               const int* row_offsets, int batch, const int* tok_in, const int* lengths,
                               const float* fused, const void* embed, const void* w_in, const void* w_hid,
                               float* x, int* row_seq, int* row_pos, cudaStream_t st) {
    if (a.dt == BF16)
        embed_norms_kernel<bf16><<<M, kRowThreads, 0, st>>>(a, decode, tokens, positions, row_offsets, batch, M,
            tok_in, lengths, fused, (const bf16*)embed, (const bf16*)w_in, (const bf16*)w_hid, x, row_seq, row_pos);
    else
        embed_norms_kernel<float><<<M, kRowThreads, 0, st>>>(a, decode, tokens, positions, row_offsets, batch, M,
            tok_in, lengths, fused, (const float*)embed, (const float*)w_in, (const float*)w_hid, x, row_seq, row_pos);
    return cudaGetLastError();
}

cudaError_t launch_latent(const RowArgs& a, int M, const float* cqkv, const void* w_qa, const void* w_kva,
                          const float* rope_cos, const float* rope_sin, const int* row_seq, const int* row_pos,
                          const int* block_table, void* cache, float* cq_hat, cudaStream_t st) {
    if (a.dt == BF16)
        latent_kernel<bf16><<<M, kRowThreads, 0, st>>>(a, cqkv, (const bf16*)w_qa, (const bf16*)w_kva, rope_cos,
            rope_sin, row_seq, row_pos, block_table, (bf16*)cache, cq_hat);
    else
        latent_kernel<float><<<M, kRowThreads, 0, st>>>(a, cqkv, (const float*)w_qa, (const float*)w_kva, rope_cos,
            rope_sin, row_seq, row_pos, block_table, (float*)cache, cq_hat);
    return cudaGetLastError();
}

cudaError_t launch_rmsnorm(int M, int H, float eps, DType wt, const float* x, const void* w, float* y,
                           cudaStream_t st) {
    if (wt == BF16) rmsnorm_kernel<bf16><<<M, kRowThreads, 0, st>>>(H, eps, x, (const bf16*)w, y);
    else rmsnorm_kernel<float><<<M, kRowThreads, 0, st>>>(H, eps, x, (const float*)w, y);
    return cudaGetLastError();
}

cudaError_t launch_final(const RowArgs& a, bool extend, int batch, const int* row_offsets, const float* h2,
                         const void* w_final, const int* row_pos, float* carry, float* z, float* hidden_out,
                         int* lengths, cudaStream_t st) {
    if (a.dt == BF16)
        final_kernel<bf16><<<batch, kRowThreads, 0, st>>>(a, extend, row_offsets, h2, (const bf16*)w_final, row_pos,
                                                          carry, z, hidden_out, lengths);
    else
        final_kernel<float><<<batch, kRowThreads, 0, st>>>(a, extend, row_offsets, h2, (const float*)w_final,
                                                           row_pos, carry, z, hidden_out, lengths);
    return cudaGetLastError();
}

cudaError_t launch_argmax_final(int batch, int npart, const float* pval, const int* pidx, int mode,
                                const int* d2t, int Vt, int* d0, int* out_tokens, int gamma, int s,
                                int* tok_in, int* err, cudaStream_t st) {
    argmax_final_kernel<<<batch, kRowThreads, 0, st>>>(npart, pval, pidx, mode, d2t, Vt, d0, out_tokens, gamma, s,
                                                       tok_in, err);
    return cudaGetLastError();
}

cudaError_t launch_emit_first(int batch, const int* d0, const int* d2t, int Vt, int* out_tokens, int gamma,
                              int* tok_in, int* err, cudaStream_t st) {
    emit_first_kernel<<<(batch + 127) / 128, 128, 0, st>>>(batch, d0, d2t, Vt, out_tokens, gamma, tok_in, err);
    return cudaGetLastError();
}

cudaError_t launch_accept(const int* draft, const int* target, int batch, int gamma, int* acc, int* hist,
                          cudaStream_t st) {
    accept_kernel<<<1, kRowThreads, (gamma + 1) * sizeof(int), st>>>(draft, target, batch, gamma, acc, hist);
    return cudaGetLastError();
}

}  // namespace e3
