// MLA attention over the one-layer latent cache, in absorbed form.
//
// The draft head's single MLA layer ("Eagle3 DeepseekV3 in MAX" §4) attends over a one-layer view
// of the cache ("max.pipelines.architectures.eagle3_deepseekV3", construct_kv_params) whose rows
// are [c_kv_hat | k_rope].  With W_UK,h / W_UV,h the key / value rows of kv_b for head h:
//   score_t = sigma (q_nope,h . W_UK,h c_t + q_pe,h . k_t) = sigma (q_lat,h . c_t + q_pe,h . k_t),
//   o_h = sum_t p_t W_UV,h c_t = W_UV,h (sum_t p_t c_t),      q_lat,h = W_UK,h^T q_nope,h.
// So the kernels never expand per-head keys or values: absorb forms q_lat; attention runs split-K
// over the ragged context with a warp-level online softmax and writes per-split partials;
// combine merges the splits and applies W_UV,h.
#include <float.h>

#include "common.cuh"
#include "kernels.h"

namespace e3 {

constexpr int kAbsRows = 4;
constexpr int kTile = 32;
constexpr int kAttnWarps = 8;
constexpr int kHeadsPerWarp = 2;
constexpr int kHeadsPerCta = kAttnWarps * kHeadsPerWarp;
constexpr int kCombRows = 4;

// qa[r, h] = [ W_UK,h^T q_nope[r, h] | RoPE(q_pe[r, h], pos_r) ]
template <typename T>
__global__ void __launch_bounds__(256) absorb_kernel(const AttnArgs a) {
    extern __shared__ float qn[];   // [kAbsRows][dn]
    const int h = blockIdx.x, r0 = blockIdx.y * kAbsRows;
    const int nr = min(kAbsRows, a.M - r0);
    const int dqk = a.dn + a.dr, D = a.dc + a.dr;
    for (int t = threadIdx.x; t < nr * a.dn; t += blockDim.x) {
        const int i = t / a.dn, k = t % a.dn;
        qn[i * a.dn + k] = a.q[((long)(r0 + i) * a.nh + h) * dqk + k];
    }
    const int half = a.dr / 2;
    for (int t = threadIdx.x; t < nr * half; t += blockDim.x) {
        const int i = t / half, p = t % half;
        const int pos = a.row_pos[r0 + i];
        const float c = a.rope_cos[(long)pos * half + p], s = a.rope_sin[(long)pos * half + p];
        const float* qp = a.q + ((long)(r0 + i) * a.nh + h) * dqk + a.dn;
        const float x0 = qp[2 * p], x1 = qp[2 * p + 1];
        float* dst = a.qa + ((long)(r0 + i) * a.nh + h) * D + a.dc;
        dst[2 * p] = x0 * c - x1 * s;
        dst[2 * p + 1] = x0 * s + x1 * c;
    }
    __syncthreads();
    const T* W = reinterpret_cast<const T*>(a.kv_b) + (long)h * (a.dn + a.dv) * a.dc;
    for (int c = threadIdx.x; c < a.dc; c += blockDim.x) {
        float acc[kAbsRows];
#pragma unroll
        for (int i = 0; i < kAbsRows; ++i) acc[i] = 0.f;
        for (int k = 0; k < a.dn; ++k) {
            const float w = to_f(W[(long)k * a.dc + c]);
#pragma unroll
            for (int i = 0; i < kAbsRows; ++i) acc[i] = fmaf(qn[i * a.dn + k], w, acc[i]);
        }
        for (int i = 0; i < nr; ++i) a.qa[((long)(r0 + i) * a.nh + h) * D + c] = acc[i];
    }
}

// One (split, head group, row) per CTA.  Row r at position p attends to slots [0, p]; split s covers
// a contiguous tile-aligned chunk of those slots.  Each warp owns two heads; lane j scores token j of
// the staged tile, then the warp updates its running max / sum / output (lane holds DC/32 outputs).
template <typename T, int DC, int DR>
__global__ void __launch_bounds__(kAttnWarps * 32) attention_kernel(const AttnArgs a) {
    constexpr int D = DC + DR;
    constexpr int EPW = 4 / sizeof(T);          // elements per 32-bit word
    constexpr int WORDS = D / EPW;
    constexpr int ROWW = WORDS | 1;             // odd word stride: lane-per-row reads hit distinct banks
    constexpr int NO = DC / 32;
    extern __shared__ float smem[];
    float* qs = smem;                                           // [kHeadsPerCta][D]
    uint32_t* kvs = reinterpret_cast<uint32_t*>(qs + kHeadsPerCta * D);   // [kTile][ROWW]

    const int s = blockIdx.x, hg = blockIdx.y, r = blockIdx.z;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int b = a.row_seq[r], pos = a.row_pos[r], n = pos + 1;
    int chunk = (n + a.splits - 1) / a.splits;
    chunk = (chunk + kTile - 1) / kTile * kTile;
    const int t0 = s * chunk, t1 = min(n, t0 + chunk);
    const int h0 = hg * kHeadsPerCta;

    for (int t = threadIdx.x; t < kHeadsPerCta * D; t += blockDim.x) {
        const int hh = t / D, d = t % D, h = h0 + hh;
        qs[t] = (h < a.nh) ? a.qa[((long)r * a.nh + h) * D + d] : 0.f;
    }
    const float* qA = qs + (warp * kHeadsPerWarp) * D;
    const float* qB = qA + D;
    float m[2] = {-FLT_MAX, -FLT_MAX}, l[2] = {0.f, 0.f};
    float o[2][NO];
#pragma unroll
    for (int i = 0; i < NO; ++i) { o[0][i] = 0.f; o[1][i] = 0.f; }
    bool any = false;

    const T* cache = reinterpret_cast<const T*>(a.cache);
    const int* bt = a.block_table + (long)b * a.max_pages;
    for (int tt = t0; tt < t1; tt += kTile) {
        const int cnt = min(kTile, t1 - tt);
        __syncthreads();
        for (int t = threadIdx.x; t < cnt * WORDS; t += blockDim.x) {
            const int j = t / WORDS, w = t % WORDS;
            const int slot = tt + j;
            const int page = bt[slot / a.page_size];
            const uint32_t* src = reinterpret_cast<const uint32_t*>(
                cache + ((long)page * a.page_size + slot % a.page_size) * D);
            kvs[j * ROWW + w] = src[w];
        }
        __syncthreads();
        float sa = 0.f, sb = 0.f;
        if (lane < cnt) {
            const uint32_t* kr = kvs + lane * ROWW;
            if constexpr (EPW == 2) {
#pragma unroll 8
                for (int w = 0; w < WORDS; ++w) {
                    const uint32_t u = kr[w];
                    const float k0 = bf_lo(u), k1 = bf_hi(u);
                    const float2 a2 = *reinterpret_cast<const float2*>(qA + 2 * w);
                    const float2 b2 = *reinterpret_cast<const float2*>(qB + 2 * w);
                    sa = fmaf(a2.x, k0, fmaf(a2.y, k1, sa));
                    sb = fmaf(b2.x, k0, fmaf(b2.y, k1, sb));
                }
            } else {
#pragma unroll 8
                for (int w = 0; w < WORDS; ++w) {
                    const float k0 = __uint_as_float(kr[w]);
                    sa = fmaf(qA[w], k0, sa);
                    sb = fmaf(qB[w], k0, sb);
                }
            }
        }
        const bool valid = lane < cnt;
        float p[2];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const float sc = valid ? (hh ? sb : sa) * a.sigma : -FLT_MAX;
            const float mt = warp_max(sc);
            const float mn = fmaxf(m[hh], mt);
            const float alpha = any ? __expf(m[hh] - mn) : 0.f;
            p[hh] = valid ? __expf(sc - mn) : 0.f;
            l[hh] = l[hh] * alpha + warp_sum(p[hh]);
#pragma unroll
            for (int i = 0; i < NO; ++i) o[hh][i] *= alpha;
            m[hh] = mn;
        }
        any = true;
        for (int j = 0; j < cnt; ++j) {
            const float p0 = __shfl_sync(0xffffffffu, p[0], j);
            const float p1 = __shfl_sync(0xffffffffu, p[1], j);
            const T* row = reinterpret_cast<const T*>(kvs + j * ROWW);
#pragma unroll
            for (int i = 0; i < NO; ++i) {
                const float v = to_f(row[lane + 32 * i]);
                o[0][i] = fmaf(p0, v, o[0][i]);
                o[1][i] = fmaf(p1, v, o[1][i]);
            }
        }
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int h = h0 + warp * kHeadsPerWarp + hh;
        if (h >= a.nh) continue;
        const long base = ((long)r * a.nh + h) * a.splits + s;
        if (lane == 0) {
            a.part_ml[base * 2] = any ? m[hh] : -FLT_MAX;
            a.part_ml[base * 2 + 1] = l[hh];
        }
#pragma unroll
        for (int i = 0; i < NO; ++i) a.part_o[base * DC + lane + 32 * i] = o[hh][i];
    }
}

// o[r, h*dv + j] = W_UV,h[j] . (sum_s e^{m_s - M} o_s / sum_s e^{m_s - M} l_s)
template <typename T, int DC>
__global__ void __launch_bounds__(256) combine_kernel(const AttnArgs a) {
    __shared__ float ol[kCombRows][DC];
    const int h = blockIdx.x, r0 = blockIdx.y * kCombRows;
    const int nr = min(kCombRows, a.M - r0);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int i = 0; i < nr; ++i) {
        const long base = ((long)(r0 + i) * a.nh + h) * a.splits;
        float mx = -FLT_MAX;
        for (int s = 0; s < a.splits; ++s) mx = fmaxf(mx, a.part_ml[(base + s) * 2]);
        float den = 0.f;
        for (int s = 0; s < a.splits; ++s) {
            const float l = a.part_ml[(base + s) * 2 + 1];
            if (l > 0.f) den += __expf(a.part_ml[(base + s) * 2] - mx) * l;
        }
        const float inv = den > 0.f ? 1.f / den : 0.f;
        for (int c = threadIdx.x; c < DC; c += blockDim.x) {
            float num = 0.f;
            for (int s = 0; s < a.splits; ++s) {
                const float l = a.part_ml[(base + s) * 2 + 1];
                if (l > 0.f) num += __expf(a.part_ml[(base + s) * 2] - mx) * a.part_o[(base + s) * DC + c];
            }
            ol[i][c] = num * inv;
        }
    }
    __syncthreads();
    const T* W = reinterpret_cast<const T*>(a.kv_b) + ((long)h * (a.dn + a.dv) + a.dn) * DC;
    for (int j = warp; j < a.dv; j += blockDim.x >> 5) {
        const T* wr = W + (long)j * DC;
        float acc[kCombRows];
#pragma unroll
        for (int i = 0; i < kCombRows; ++i) acc[i] = 0.f;
        for (int c = lane; c < DC; c += 32) {
            const float w = to_f(wr[c]);
#pragma unroll
            for (int i = 0; i < kCombRows; ++i) acc[i] = fmaf(w, ol[i][c], acc[i]);
        }
        for (int i = 0; i < nr; ++i) {
            const float v = warp_sum(acc[i]);
            if (lane == 0) a.o[(long)(r0 + i) * a.nh * a.dv + h * a.dv + j] = v;
        }
    }
}

bool attention_supported(int dc, int dr, int dn, int dv) {
    (void)dn; (void)dv;
    return (dc == 512 && dr == 64) || (dc == 32 && dr == 16);
}

cudaError_t launch_absorb(const AttnArgs& a, cudaStream_t st) {
    dim3 grid(a.nh, (a.M + kAbsRows - 1) / kAbsRows);
    const size_t sm = (size_t)kAbsRows * a.dn * sizeof(float);
    if (a.dt == BF16) absorb_kernel<bf16><<<grid, 256, sm, st>>>(a);
    else absorb_kernel<float><<<grid, 256, sm, st>>>(a);
    return cudaGetLastError();
}

template <typename T, int DC, int DR>
static cudaError_t attn_launch(const AttnArgs& a, cudaStream_t st) {
    constexpr int D = DC + DR;
    constexpr int WORDS = D / (4 / sizeof(T));
    const size_t sm = (size_t)kHeadsPerCta * D * sizeof(float) + (size_t)kTile * (WORDS | 1) * sizeof(uint32_t);
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(attention_kernel<T, DC, DR>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    dim3 grid(a.splits, (a.nh + kHeadsPerCta - 1) / kHeadsPerCta, a.M);
    attention_kernel<T, DC, DR><<<grid, kAttnWarps * 32, sm, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_attention(const AttnArgs& a, cudaStream_t st) {
    if (a.dc == 512 && a.dr == 64)
        return a.dt == BF16 ? attn_launch<bf16, 512, 64>(a, st) : attn_launch<float, 512, 64>(a, st);
    if (a.dc == 32 && a.dr == 16)
        return a.dt == BF16 ? attn_launch<bf16, 32, 16>(a, st) : attn_launch<float, 32, 16>(a, st);
    return cudaErrorInvalidValue;
}

cudaError_t launch_combine(const AttnArgs& a, cudaStream_t st) {
    dim3 grid(a.nh, (a.M + kCombRows - 1) / kCombRows);
    if (a.dc == 512) {
        if (a.dt == BF16) combine_kernel<bf16, 512><<<grid, 256, 0, st>>>(a);
        else combine_kernel<float, 512><<<grid, 256, 0, st>>>(a);
    } else if (a.dc == 32) {
        if (a.dt == BF16) combine_kernel<bf16, 32><<<grid, 256, 0, st>>>(a);
        else combine_kernel<float, 32><<<grid, 256, 0, st>>>(a);
    } else {
        return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace e3
