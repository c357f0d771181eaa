// Attention of the Llama-style MHA draft head ("Eagle3 DeepseekV3 in MAX" §11: LlamaForCausalLMEagle3 on a
// DeepseekV3 target; "max.pipelines.architectures.eagle3_deepseekV3", Eagle3MHADeepseekV3DraftArchConfig:
// the head keeps its own one-layer key/value cache).
//
//   mha_rope_append_kernel   rotate q (in place) and k by the rotate-half RoPE (dimension i pairs with
//                            i + d/2), write the row's [k | v] entry into the paged cache at its position
//   mha_attention_kernel     grouped-query attention, split over the context: a CTA takes one row, one
//                            key/value head (the G query heads that share it) and one chunk of slots
//   mha_merge_kernel         combines the splits' (max, sum, unnormalised output) of every row and head
//
// Cache row of slot p: [k_rot (n_kv x d) | v (n_kv x d)] in the configured dtype.  A row at position p
// attends to slots 0..p of its sequence (causal; a decode row sees itself, after its own append).
#include <float.h>
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "mma_sync.cuh"
#include "../../include/eagle3.h"

namespace e3 {

constexpr int kMhaThreads = 128;          // 4 warps; each takes 32-slot tiles of the chunk in turn
constexpr int kMhaWarps = kMhaThreads / 32;
constexpr int kMhaAppendThreads = 256;
constexpr int kMhaMaxSplits = 1024;       // split statistics a merge CTA stages in shared memory

// Grid (rows, chunks of 256 work items): item i < (n_h + n_kv) d/2 rotates one (i, i + d/2) pair of q (in
// place) or of k (into the cache); item i < n_kv d also copies one v element.  One item per thread, so no
// thread waits on a chain of loads.
template <typename T>
__global__ void __launch_bounds__(kMhaAppendThreads) mha_rope_append_kernel(const MhaArgs a) {
    pdl_trigger();
    pdl_wait();
    const int r = blockIdx.x;
    const int nh = a.nh, nkv = a.nkv, d = a.d, half = d / 2;
    const int i = blockIdx.y * kMhaAppendThreads + threadIdx.x;
    const int b = a.row_seq[r], pos = a.row_pos[r];
    const float* cs = a.rope_cos + (long)pos * half;
    const float* sn = a.rope_sin + (long)pos * half;
    if (i < nh * half) {
        float* q = a.q + (long)r * nh * d;
        const int h = i / half, j = i % half;
        const float x0 = q[h * d + j], x1 = q[h * d + j + half];
        q[h * d + j] = x0 * cs[j] - x1 * sn[j];
        q[h * d + j + half] = x0 * sn[j] + x1 * cs[j];
    }
    const bool krot = i >= nh * half && i < (nh + nkv) * half;
    const bool vcopy = i < nkv * d;
    if (!krot && !vcopy) return;
    const int pi = pos / a.page_size;
    int page = -1;
    if (pi < a.max_pages) page = a.block_table[(long)b * a.max_pages + pi];
    if (page < 0 || page >= a.num_pages) {
        if (threadIdx.x == 0 && blockIdx.y == 0) set_err(a.err, EAGLE3_DEVERR_PAGE);
        return;
    }
    const float* kv = a.kv + (long)r * 2 * nkv * d;
    T* dst = static_cast<T*>(a.cache) + ((long)page * a.page_size + pos % a.page_size) * (2L * nkv * d);
    if (krot) {
        const int ik = i - nh * half, h = ik / half, j = ik % half;
        const float x0 = kv[h * d + j], x1 = kv[h * d + j + half];
        dst[h * d + j] = from_f<T>(x0 * cs[j] - x1 * sn[j]);
        dst[h * d + j + half] = from_f<T>(x0 * sn[j] + x1 * cs[j]);
    }
    if (vcopy) dst[nkv * d + i] = from_f<T>(kv[nkv * d + i]);
}

// One CTA: row r, key/value head g, slots [s chunk, min((s + 1) chunk, pos + 1)).  Each warp takes
// 32-slot tiles in turn.  The tile's value rows go to the warp's shared-memory buffer by cp.async first;
// meanwhile each lane loads its slot's whole key row (every load of the row in flight at once) and forms
// the G dot products (the G query rows sit in shared memory and are read as broadcasts).  Values: each
// lane owns d/32 output dimensions of every head and walks the staged rows, with each slot's
// probabilities shuffled from its lane.
template <typename T, int D>
constexpr int mha_vstage_bytes() { return kMhaWarps * 32 * D * (int)sizeof(T); }

template <typename T, int D, int G>
__global__ void __launch_bounds__(kMhaThreads) mha_attention_kernel(const MhaArgs a) {
    constexpr int DL = D / 32;                       // output dimensions per lane
    constexpr int CPR = D * (int)sizeof(T) / 16;     // 16-byte chunks of a value row
    extern __shared__ __align__(16) unsigned char mha_dyn[];
    __shared__ float qs[G][D];
    __shared__ float wm[kMhaWarps][G], wl[kMhaWarps][G];
    __shared__ float so[G][D];
    pdl_trigger();
    pdl_wait();
    const int r = blockIdx.x, g = blockIdx.y, s = blockIdx.z;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int b = a.row_seq[r], pos = a.row_pos[r];
    const int start = s * a.chunk, end = min(pos + 1, start + a.chunk);
    if (start >= end) return;                       // past this row's context: the merge skips it
    const long rowlen = 2L * a.nkv * D;
    for (int i = threadIdx.x; i < G * D; i += kMhaThreads) {
        qs[i / D][i % D] = a.q[(long)r * a.nh * D + (long)g * G * D + i] * a.sigma;
        so[i / D][i % D] = 0.f;
    }
    __syncthreads();
    const T* cache = static_cast<const T*>(a.cache);
    const int* bt = a.block_table + (long)b * a.max_pages;

    float m[G], l[G], o[G][DL];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.f;
#pragma unroll
        for (int e = 0; e < DL; ++e) o[h][e] = 0.f;
    }
    T* vs = reinterpret_cast<T*>(mha_dyn) + (long)warp * 32 * D;   // this warp's staged value rows
    for (int tb = start + 32 * warp; tb < end; tb += 32 * kMhaWarps) {
        const int j = tb + lane;
        bool valid = j < end;
        long off = 0;                                // this lane's slot row, in elements
        if (valid) {
            const int pi = j / a.page_size;
            const int page = pi < a.max_pages ? bt[pi] : -1;
            if (page < 0 || page >= a.num_pages) {
                set_err(a.err, EAGLE3_DEVERR_PAGE);
                valid = false;
            } else {
                off = ((long)page * a.page_size + j % a.page_size) * rowlen;
            }
        }
        // the tile's value rows into shared memory (chunk c: row c / CPR, 16 bytes c % CPR)
        __syncwarp();                                // the previous tile's rows have been read
#pragma unroll 4
        for (int c = lane; c < 32 * CPR; c += 32) {
            const int row = c / CPR, q = c % CPR;
            const long ro = __shfl_sync(0xffffffffu, off, row);
            const bool rv = __shfl_sync(0xffffffffu, valid ? 1 : 0, row) != 0;
            if (rv)
                cp_async16(smem_u32(vs + (long)row * D) + 16 * q,
                           reinterpret_cast<const unsigned char*>(cache + ro + (long)a.nkv * D + (long)g * D) + 16 * q);
        }
        cp_async_commit();
        float sc[G];
#pragma unroll
        for (int h = 0; h < G; ++h) sc[h] = 0.f;
        if (valid) {
            const T* kr = cache + off + (long)g * D;
            Raw8<T> kraw[D / 8];
#pragma unroll
            for (int c = 0; c < D / 8; ++c) kraw[c] = ld8<false>(kr + 8 * c);
#pragma unroll
            for (int c = 0; c < D / 8; ++c) {
                float kv8[8];
                widen(kraw[c], kv8);
#pragma unroll
                for (int h = 0; h < G; ++h)
#pragma unroll
                    for (int e = 0; e < 8; ++e) sc[h] = fmaf(qs[h][8 * c + e], kv8[e], sc[h]);
            }
        }
        float p[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float x = valid ? sc[h] : -INFINITY;
            const float mt = warp_max(x);
            const float mn = fmaxf(m[h], mt);        // finite: lane 0's slot is always valid or flagged
            const float mref = mn == -INFINITY ? 0.f : mn;
            p[h] = valid ? __expf(x - mref) : 0.f;
            const float corr = __expf(m[h] - mref);  // 0 while m is still -inf
            l[h] = l[h] * corr + warp_sum(p[h]);
#pragma unroll
            for (int e = 0; e < DL; ++e) o[h][e] *= corr;
            m[h] = mn;
        }
        const int nt = min(32, end - tb);
        const unsigned vmask = __ballot_sync(0xffffffffu, valid);
        cp_async_wait<0>();
        __syncwarp();
#pragma unroll 4
        for (int jj = 0; jj < nt; ++jj) {
            if (!((vmask >> jj) & 1u)) continue;     // a slot without a row (flagged) adds nothing
            const T* vr = vs + (long)jj * D + lane * DL;
            float v[DL];
#pragma unroll
            for (int e = 0; e < DL; ++e) v[e] = to_f(vr[e]);
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float ph = __shfl_sync(0xffffffffu, p[h], jj);
#pragma unroll
                for (int e = 0; e < DL; ++e) o[h][e] = fmaf(ph, v[e], o[h][e]);
            }
        }
    }
    // combine the warps: common maximum per head, rescaled sums
    if (lane == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) { wm[warp][h] = m[h]; wl[warp][h] = l[h]; }
    }
    __syncthreads();
    float M[G], L[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        M[h] = wm[0][h];
        for (int w = 1; w < kMhaWarps; ++w) M[h] = fmaxf(M[h], wm[w][h]);
        L[h] = 0.f;
        for (int w = 0; w < kMhaWarps; ++w)
            if (wm[w][h] != -INFINITY) L[h] += wl[w][h] * __expf(wm[w][h] - M[h]);
    }
    for (int w = 0; w < kMhaWarps; ++w) {
        if (warp == w && m[0] != -INFINITY) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float f = __expf(m[h] - M[h]);
#pragma unroll
                for (int e = 0; e < DL; ++e) so[h][lane * DL + e] += o[h][e] * f;
            }
        }
        __syncthreads();
    }
    const int head0 = g * G;
    if (a.splits == 1) {
        for (int i = threadIdx.x; i < G * D; i += kMhaThreads) {
            const int h = i / D, e = i % D;
            const float v = so[h][e] / L[h];
            const long idx = (long)r * a.nh * D + (long)(head0 + h) * D + e;
            if (a.o) a.o[idx] = v;
            if (a.o_bf) a.o_bf[idx] = __float2bfloat16_rn(v);
        }
    } else {
        const long pr = (long)r * a.splits + s;
        for (int i = threadIdx.x; i < G * D; i += kMhaThreads) {
            const int h = i / D, e = i % D;
            a.part_o[(pr * a.nh + head0 + h) * D + e] = so[h][e];
        }
        if (threadIdx.x < G) {
            const int h = threadIdx.x;
            a.part_ml[(pr * a.nh + head0 + h) * 2] = M[h];
            a.part_ml[(pr * a.nh + head0 + h) * 2 + 1] = L[h];
        }
    }
}

// One CTA per (row, head), one thread per output dimension: o = sum_s e^(m_s - M) o_s / sum_s e^(m_s - M) l_s
// over the splits that hold any of the row's slots.  The splits' (m, l) are staged in shared memory first,
// so the loop over o_s issues independent loads.
__global__ void __launch_bounds__(256) mha_merge_kernel(const MhaArgs a) {
    __shared__ float sm[kMhaMaxSplits], sl[kMhaMaxSplits];
    __shared__ float red[8];
    pdl_trigger();
    pdl_wait();
    const int r = blockIdx.x, h = blockIdx.y, e = threadIdx.x;
    const int pos = a.row_pos[r];
    const int nvalid = min(min(a.splits, kMhaMaxSplits), (pos + a.chunk) / a.chunk);
    const long pr0 = (long)r * a.splits;
    float mx = -INFINITY;
    for (int s = e; s < nvalid; s += blockDim.x) {
        sm[s] = a.part_ml[((pr0 + s) * a.nh + h) * 2];
        sl[s] = a.part_ml[((pr0 + s) * a.nh + h) * 2 + 1];
        mx = fmaxf(mx, sm[s]);
    }
    mx = warp_max(mx);
    if ((e & 31) == 0) red[e >> 5] = mx;
    __syncthreads();
    float M = red[0];
    for (int w = 1; w < (int)(blockDim.x + 31) / 32; ++w) M = fmaxf(M, red[w]);
    // eight splits' partial outputs in flight at a time (independent loads, then the weighted sum in
    // split order)
    float L = 0.f, acc = 0.f;
    for (int s0 = 0; s0 < nvalid; s0 += 8) {
        float po[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
            po[u] = (s0 + u < nvalid && e < a.d) ? a.part_o[((pr0 + s0 + u) * a.nh + h) * a.d + e] : 0.f;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            if (s0 + u >= nvalid) break;
            const float f = sm[s0 + u] == -INFINITY ? 0.f : __expf(sm[s0 + u] - M);
            L += f * sl[s0 + u];
            acc += f * po[u];
        }
    }
    if (e < a.d) {
        const float v = acc / L;
        const long idx = (long)r * a.nh * a.d + (long)h * a.d + e;
        if (a.o) a.o[idx] = v;
        if (a.o_bf) a.o_bf[idx] = __float2bfloat16_rn(v);
    }
}

bool mha_supported(int nh, int nkv, int d) {
    if (nkv < 1 || nh % nkv) return false;
    const int G = nh / nkv;
    return (d == 32 || d == 64 || d == 128) && (G == 1 || G == 2 || G == 4 || G == 7 || G == 8);
}

cudaError_t launch_mha_rope_append(const MhaArgs& a, cudaStream_t st) {
    const int items = (a.nh + a.nkv) * (a.d / 2) > a.nkv * a.d ? (a.nh + a.nkv) * (a.d / 2) : a.nkv * a.d;
    const dim3 grid(a.M, (items + kMhaAppendThreads - 1) / kMhaAppendThreads);
    if (a.dt == BF16) return launch_pdl(mha_rope_append_kernel<bf16>, grid, dim3(kMhaAppendThreads), 0, st, a);
    return launch_pdl(mha_rope_append_kernel<float>, grid, dim3(kMhaAppendThreads), 0, st, a);
}

template <typename T, int D, int G>
static cudaError_t launch_attn_dg(const MhaArgs& a, dim3 grid, cudaStream_t st) {
    constexpr int smem = mha_vstage_bytes<T, D>();
    cudaError_t e = smem_optin((const void*)mha_attention_kernel<T, D, G>, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(mha_attention_kernel<T, D, G>, grid, dim3(kMhaThreads), (size_t)smem, st, a);
}

template <typename T, int D>
static cudaError_t launch_attn_g(const MhaArgs& a, dim3 grid, cudaStream_t st) {
    switch (a.nh / a.nkv) {
        case 1: return launch_attn_dg<T, D, 1>(a, grid, st);
        case 2: return launch_attn_dg<T, D, 2>(a, grid, st);
        case 4: return launch_attn_dg<T, D, 4>(a, grid, st);
        case 7: return launch_attn_dg<T, D, 7>(a, grid, st);
        case 8: return launch_attn_dg<T, D, 8>(a, grid, st);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T>
static cudaError_t launch_attn_t(const MhaArgs& a, dim3 grid, cudaStream_t st) {
    switch (a.d) {
        case 32: return launch_attn_g<T, 32>(a, grid, st);
        case 64: return launch_attn_g<T, 64>(a, grid, st);
        case 128: return launch_attn_g<T, 128>(a, grid, st);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_mha_attention(const MhaArgs& a, cudaStream_t st) {
    if (!mha_supported(a.nh, a.nkv, a.d) || a.chunk < 1 || a.splits < 1) return cudaErrorInvalidValue;
    const dim3 grid(a.M, a.nkv, a.splits);
    return a.dt == BF16 ? launch_attn_t<bf16>(a, grid, st) : launch_attn_t<float>(a, grid, st);
}

cudaError_t launch_mha_merge(const MhaArgs& a, cudaStream_t st) {
    if (a.splits > kMhaMaxSplits) return cudaErrorInvalidValue;
    const int threads = (a.d + 31) / 32 * 32;
    return launch_pdl(mha_merge_kernel, dim3(a.M, a.nh), dim3(threads), 0, st, a);
}

}  // namespace e3
