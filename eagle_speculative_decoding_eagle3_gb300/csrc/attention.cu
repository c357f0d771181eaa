// MLA attention over the one-layer latent cache, in absorbed form.
//
// The draft head's single MLA layer ("Eagle3 DeepseekV3 in MAX" §4) attends over a one-layer view
// of the cache ("max.pipelines.architectures.eagle3_deepseekV3", construct_kv_params) whose rows
// are [c_kv_hat | k_rope].  With W_UK,h / W_UV,h the key / value rows of kv_b for head h:
//   score_t = sigma (q_nope,h . W_UK,h c_t + q_pe,h . k_t) = sigma (q_lat,h . c_t + q_pe,h . k_t),
//   o_h = sum_t p_t W_UV,h c_t = W_UV,h (sum_t p_t c_t),      q_lat,h = W_UK,h^T q_nope,h.
// So no kernel expands per-head keys or values: absorb forms q_lat; attention runs split-K over the
// ragged context with an online softmax and writes per-split partials; merge combines the splits into
// o_lat and a grouped GEMM applies W_UV,h.
//
// Two attention kernels share the partial format:
//  * attention_mma_kernel (bf16 cache, d_c 512 / d_r 64): 64 heads x 32-token tiles on the tensor
//    cores with mma.sync m16n8k16 (heads are the MMA rows, so the 64 heads of a CTA share one staged
//    KV tile); the KV tiles are double-buffered with cp.async through the block table.
//  * attention_kernel (any dtype, small latent): CUDA-core fallback used by the fp32 head.
#include <float.h>
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "mma_sync.cuh"
#include "../../include/eagle3.h"

namespace e3 {

constexpr int kAbsRows = 4;
constexpr int kTile = 32;
constexpr int kAttnWarps = 8;
constexpr int kHeadsPerWarp = 2;
constexpr int kHeadsPerCta = kAttnWarps * kHeadsPerWarp;

// Slots of row r (context n = pos + 1) per split: the fixed chunk, else ceil(n / splits); either way
// rounded up to whole 32-slot tiles, so the leading splits cover the context and the rest are empty.
__device__ __forceinline__ int split_chunk(const AttnArgs& a, int n) {
    const int chunk = a.chunk > 0 ? a.chunk : (n + a.splits - 1) / a.splits;
    return (chunk + kTile - 1) / kTile * kTile;
}
// Splits of row r that hold partials (an empty split writes none and the merges read none)
__device__ __forceinline__ int live_splits(const AttnArgs& a, int r) {
    const int n = a.row_pos[r] + 1;
    const int chunk = split_chunk(a, n);
    return min(a.splits, (n + chunk - 1) / chunk);
}

// qa[r, h] = [ W_UK,h^T q_nope[r, h] | RoPE(q_pe[r, h], pos_r) ]  (fp32, plus a bf16 copy when asked)
// Grid (head, column block of kAbsCols latent columns, block of ROWS rows).  Thread (cc, rg) owns 8
// columns and the W_UK rows rg, rg + RG, ...: all of its (dn / RG) 16-byte weight loads are issued
// together, then the RG row groups are reduced through shared memory.  The rope part is written by
// column block 0.  A single bf16 row (batch-1 decode) takes ROWS = 1: its accumulators fit four CTAs per
// SM, so the 128 heads x 4 column blocks run as one wave instead of two.
constexpr int kAbsCols = 128;
template <typename T, int ROWS>
__global__ void __launch_bounds__(256, ROWS == 1 ? 4 : 0) absorb_kernel(const AttnArgs a) {
    extern __shared__ float sm[];           // [ROWS][dn] q_nope, then [RG][ROWS][cols] partials
    constexpr int kMaxLoads = 8;
    const int h = blockIdx.x, cb = blockIdx.y, r0 = blockIdx.z * ROWS;
    const int nr = min(ROWS, a.M - r0);
    const int dqk = a.dn + a.dr, D = a.dc + a.dr;
    const int cols = min(kAbsCols, a.dc), c0 = cb * cols;
    const int nchunk = cols / 8;
    const int RG = blockDim.x / nchunk;
    const int cc = threadIdx.x % nchunk, rg = threadIdx.x / nchunk;
    const T* W = reinterpret_cast<const T*>(a.kv_b) + (long)h * (a.dn + a.dv) * a.dc + c0 + 8 * cc;
    // the first batch of weight loads (all of them for d_n <= RG * kMaxLoads) precedes the wait on the
    // kernel that produced q
    pdl_trigger();
    Raw8<T> wr[kMaxLoads];
#pragma unroll
    for (int j = 0; j < kMaxLoads; ++j) {
        const int k = rg + j * RG;
        wr[j] = (rg < RG && k < a.dn) ? ld8<true>(W + (long)k * a.dc) : zero8((T*)nullptr);
    }
    pdl_wait();
    float* qn = sm;
    float* part = sm + ROWS * a.dn;
    for (int t = threadIdx.x; t < ROWS * a.dn; t += blockDim.x) {
        const int i = t / a.dn, k = t % a.dn;
        qn[t] = (i < nr) ? a.q[((long)(r0 + i) * a.nh + h) * dqk + k] : 0.f;
    }
    const int half = a.dr / 2;
    if (cb == 0) {
        for (int t = threadIdx.x; t < nr * half; t += blockDim.x) {
            const int i = t / half, p = t % half;
            const int pos = a.row_pos[r0 + i];
            const float c = a.rope_cos[(long)pos * half + p], s = a.rope_sin[(long)pos * half + p];
            const float* qp = a.q + ((long)(r0 + i) * a.nh + h) * dqk + a.dn;
            const float x0 = qp[2 * p], x1 = qp[2 * p + 1];
            const float y0 = x0 * c - x1 * s, y1 = x0 * s + x1 * c;
            const long o = ((long)(r0 + i) * a.nh + h) * D + a.dc + 2 * p;
            a.qa[o] = y0;
            a.qa[o + 1] = y1;
            if (a.qa_bf) { a.qa_bf[o] = __float2bfloat16_rn(y0); a.qa_bf[o + 1] = __float2bfloat16_rn(y1); }
        }
    }
    __syncthreads();
    float acc[ROWS][8];
#pragma unroll
    for (int i = 0; i < ROWS; ++i)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[i][e] = 0.f;
    for (int k0 = rg; rg < RG && k0 < a.dn; k0 += RG * kMaxLoads) {
        if (k0 != rg) {
#pragma unroll
            for (int j = 0; j < kMaxLoads; ++j) {
                const int k = k0 + j * RG;
                wr[j] = k < a.dn ? ld8<true>(W + (long)k * a.dc) : zero8((T*)nullptr);
            }
        }
#pragma unroll
        for (int j = 0; j < kMaxLoads; ++j) {
            const int k = k0 + j * RG;
            if (k < a.dn) {
                float w[8];
                widen(wr[j], w);
#pragma unroll
                for (int i = 0; i < ROWS; ++i) {
                    const float q = qn[i * a.dn + k];
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[i][e] = fmaf(q, w[e], acc[i][e]);
                }
            }
        }
    }
    if (rg < RG) {
#pragma unroll
        for (int i = 0; i < ROWS; ++i) {
            float4* dst = reinterpret_cast<float4*>(part + ((long)rg * ROWS + i) * cols + 8 * cc);
            dst[0] = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
            dst[1] = make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
        }
    }
    __syncthreads();
    for (int t = threadIdx.x; t < nr * cols; t += blockDim.x) {
        const int i = t / cols, c = t % cols;
        float v = 0.f;
        for (int g = 0; g < RG; ++g) v += part[((long)g * ROWS + i) * cols + c];
        const long o = ((long)(r0 + i) * a.nh + h) * D + c0 + c;
        a.qa[o] = v;
        if (a.qa_bf) a.qa_bf[o] = __float2bfloat16_rn(v);
    }
}

// ------------------------------------------------------------------------------------------------
// CUDA-core split-K attention (fp32 cache or small latent widths).
// One (split, head group, row) per CTA.  Row r at position p attends to slots [0, p]; split s covers
// a contiguous tile-aligned chunk of those slots.  Each warp owns two heads; lane j scores token j of
// the staged tile, then the warp updates its running max / sum / output (lane holds DC/32 outputs).
template <typename T, int DC, int DR>
__global__ void __launch_bounds__(kAttnWarps * 32) attention_kernel(const AttnArgs a) {
    pdl_trigger();
    pdl_wait();
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
    const int chunk = split_chunk(a, n);
    const int t0 = s * chunk, t1 = min(n, t0 + chunk);
    const int h0 = hg * kHeadsPerCta;
    if (t0 >= t1) return;   // past this row's context: an empty split that the merge skips

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
            if (page < 0 || page >= a.num_pages) {   // a bad block table reads zeros and is flagged
                kvs[j * ROWW + w] = 0u;
                if (w == 0) set_err(a.err, 8);
                continue;
            }
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
        if (a.splits == 1) {   // a single split is already the whole softmax: o_lat = o / l
            const float inv = l[hh] > 0.f ? 1.f / l[hh] : 0.f;
            const long ob = ((long)r * a.nh + h) * DC;
#pragma unroll
            for (int i = 0; i < NO; ++i) {
                const float v = o[hh][i] * inv;
                if (a.olat) a.olat[ob + lane + 32 * i] = v;
                if (a.olat_bf) a.olat_bf[ob + lane + 32 * i] = __float2bfloat16_rn(v);
            }
            continue;
        }
        const long base = ((long)r * a.nh + h) * a.splits + s;
        if (lane == 0) {
            a.part_ml[base * 2] = any ? m[hh] : -FLT_MAX;
            a.part_ml[base * 2 + 1] = l[hh];
        }
#pragma unroll
        for (int i = 0; i < NO; ++i) a.part_o[base * DC + lane + 32 * i] = o[hh][i];
    }
}

// ------------------------------------------------------------------------------------------------
// Tensor-core split-K attention for the DeepseekV3 latent geometry (bf16, d_c 512, d_r 64).
namespace mla_mma {
constexpr int T = 32;             // tokens per tile
constexpr int HEADS = 64;         // heads per CTA: four MMA row groups of 16 share each staged KV tile
constexpr int D = 576, DC = 512;
constexpr int ROW = D + 8;        // bf16 row stride: 1168 B, 16-byte aligned, an odd number of 16 B units
constexpr int SROW = T + 4;       // fp32 score row stride
constexpr int WARPS = 8;          // warp w: head group g = w & 3, latent half c = w >> 2
constexpr size_t SMEM = (size_t)HEADS * ROW * 2 + 2 * (size_t)T * ROW * 2 + (size_t)HEADS * SROW * 4;
}  // namespace mla_mma


// One (split, 64-head block, row) per CTA; 8 warps.  Warp (g, c) scores tokens [16c, 16c + 16) of every
// tile for heads 16g..16g+15 (two 8-token MMA column tiles, four independent accumulators), the scores go
// through shared memory, both warps of a head group run the same online softmax over the 32-token tile,
// and warp (g, c) accumulates O[16 heads, 256c .. 256c + 256) = P V.  Q (64 heads x 576) and the
// double-buffered KV tiles are staged with cp.async; the KV rows come through the block table.
__global__ void __launch_bounds__(mla_mma::WARPS * 32, 1) attention_mma_kernel(const AttnArgs a) {
    using namespace mla_mma;
    pdl_trigger();
    pdl_wait();
    extern __shared__ __align__(16) unsigned char smraw[];
    bf16* qs = reinterpret_cast<bf16*>(smraw);                  // [HEADS][ROW]
    bf16* kvb = qs + HEADS * ROW;                              // [2][T][ROW]
    float* ss = reinterpret_cast<float*>(kvb + 2 * T * ROW);   // [HEADS][SROW]
    const int s = blockIdx.x, hb = blockIdx.y, r = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gq = lane >> 2, tig = lane & 3;
    const int hgrp = warp & 3, half = warp >> 2;
    const int b = a.row_seq[r], pos = a.row_pos[r], n = pos + 1;
    static_assert(T == kTile, "split chunks are whole 32-slot tiles");
    const int chunk = split_chunk(a, n);
    const int t0 = s * chunk, t1 = min(n, t0 + chunk);
    const int h0 = hb * HEADS;
    if (t0 >= t1) return;   // past this row's context: an empty split that the merge skips

    // Q: heads h0 .. h0 + 63 of row r (zero rows past n_heads)
    for (int c = tid; c < HEADS * (D / 8); c += WARPS * 32) {
        const int hh = c / (D / 8), q = c % (D / 8), h = h0 + hh;
        bf16* d = qs + hh * ROW + 8 * q;
        if (h < a.nh) cp_async16(smem_u32(d), a.qa_bf + ((long)r * a.nh + h) * D + 8 * q);
        else *reinterpret_cast<uint4*>(d) = make_uint4(0, 0, 0, 0);
    }
    const bf16* cache = reinterpret_cast<const bf16*>(a.cache);
    const int* bt = a.block_table + (long)b * a.max_pages;
    // tile loader: thread t copies row t % T, chunks t / T + k * (threads / T): one block-table lookup per tile
    constexpr int kChunkStep = WARPS * 32 / T;
    auto load_tile = [&](int buf, int tt) {
        const int j = tid % T, slot = tt + j;
        bf16* d = kvb + buf * T * ROW + j * ROW;
        const int page = (slot < t1) ? bt[slot / a.page_size] : -1;
        if (page >= 0 && page < a.num_pages) {
            const bf16* src = cache + ((long)page * a.page_size + slot % a.page_size) * D;
            for (int q = tid / T; q < D / 8; q += kChunkStep) cp_async16(smem_u32(d + 8 * q), src + 8 * q);
        } else {
            for (int q = tid / T; q < D / 8; q += kChunkStep) *reinterpret_cast<uint4*>(d + 8 * q) = make_uint4(0, 0, 0, 0);
            if (slot < t1 && tid < T) set_err(a.err, 8);
        }
        cp_async_commit();
    };

    float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};
    float o[32][4];
#pragma unroll
    for (int i = 0; i < 32; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

    if (t0 < t1) load_tile(0, t0);
    else cp_async_commit();
    int it = 0;
    // A-fragment rows of this warp's head group; B rows: tokens 16c + (lane & 7) + 8 (lane >> 4)
    const uint32_t qrow = smem_u32(qs + (16 * hgrp + (lane & 7) + ((lane >> 3) & 1) * 8) * ROW + (lane >> 4) * 8);
    for (int tt = t0; tt < t1; tt += T, ++it) {
        const int cnt = min(T, t1 - tt);
        if (tt + T < t1) {
            load_tile((it + 1) & 1, tt + T);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const bf16* K = kvb + (it & 1) * T * ROW;
        // ---- scores: heads 16g.., tokens 16c + [0, 16)
        float sacc[2][2][4];
#pragma unroll
        for (int x = 0; x < 2; ++x)
#pragma unroll
            for (int y = 0; y < 2; ++y) sacc[x][y][0] = sacc[x][y][1] = sacc[x][y][2] = sacc[x][y][3] = 0.f;
        const uint32_t krow = smem_u32(K + (16 * half + (lane & 7) + (lane >> 4) * 8) * ROW + ((lane >> 3) & 1) * 8);
#pragma unroll 4
        for (int ks = 0; ks < D / 16; ++ks) {
            uint32_t qa[4], kb[4];
            ldsm_x4(qrow + ks * 32, qa);
            ldsm_x4(krow + ks * 32, kb);
            mma_bf16_16816(sacc[ks & 1][0], qa, kb[0], kb[1]);
            mma_bf16_16816(sacc[ks & 1][1], qa, kb[2], kb[3]);
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int col = 16 * half + 8 * nt + 2 * tig;
            float v[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) v[i] = (sacc[0][nt][i] + sacc[1][nt][i]) * a.sigma;
            if (col >= cnt) v[0] = v[2] = -INFINITY;
            if (col + 1 >= cnt) v[1] = v[3] = -INFINITY;
            float* row0 = ss + (16 * hgrp + gq) * SROW + col;
            float* row1 = row0 + 8 * SROW;
            row0[0] = v[0]; row0[1] = v[1];
            row1[0] = v[2]; row1[1] = v[3];
        }
        __syncthreads();
        // ---- online softmax over the tile for rows gq and gq + 8 of the head group
        float p[2][2][4];   // [k-step][row][cols 2tig, 2tig+1, 2tig+8, 2tig+9]
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const float* row = ss + (16 * hgrp + gq + 8 * rr) * SROW + kk * 16 + 2 * tig;
                p[kk][rr][0] = row[0];
                p[kk][rr][1] = row[1];
                p[kk][rr][2] = row[8];
                p[kk][rr][3] = row[9];
#pragma unroll
                for (int e = 0; e < 4; ++e) mx[rr] = fmaxf(mx[rr], p[kk][rr][e]);
            }
        float alpha[2];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 1));
            mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 2));
            const float mn = fmaxf(m_r[rr], mx[rr]);
            alpha[rr] = (m_r[rr] == -INFINITY) ? 0.f : __expf(m_r[rr] - mn);
            float ls = 0.f;
#pragma unroll
            for (int kk = 0; kk < 2; ++kk)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    p[kk][rr][e] = __expf(p[kk][rr][e] - mn);
                    ls += p[kk][rr][e];
                }
            ls += __shfl_xor_sync(0xffffffffu, ls, 1);
            ls += __shfl_xor_sync(0xffffffffu, ls, 2);
            l_r[rr] = l_r[rr] * alpha[rr] + ls;
            m_r[rr] = mn;
        }
#pragma unroll
        for (int nt = 0; nt < 32; ++nt) {
            o[nt][0] *= alpha[0]; o[nt][1] *= alpha[0];
            o[nt][2] *= alpha[1]; o[nt][3] *= alpha[1];
        }
        // ---- O[:, 256c : 256c + 256) += P V
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            uint32_t pa[4];
            pa[0] = pack_bf16(p[kk][0][0], p[kk][0][1]);
            pa[1] = pack_bf16(p[kk][1][0], p[kk][1][1]);
            pa[2] = pack_bf16(p[kk][0][2], p[kk][0][3]);
            pa[3] = pack_bf16(p[kk][1][2], p[kk][1][3]);
            const uint32_t vrow = smem_u32(K + (kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * ROW + 256 * half +
                                           (lane >> 4) * 8);
#pragma unroll
            for (int nt = 0; nt < 32; nt += 2) {
                uint32_t vb[4];
                ldsm_x4_t(vrow + nt * 16, vb);
                mma_bf16_16816(o[nt], pa, vb[0], vb[1]);
                mma_bf16_16816(o[nt + 1], pa, vb[2], vb[3]);
            }
        }
        __syncthreads();
    }
    cp_async_wait<0>();
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        const int h = h0 + 16 * hgrp + gq + 8 * rr;
        if (h >= a.nh) continue;
        if (a.splits == 1) {   // a single split is already the whole softmax: o_lat = o / l
            const float inv = l_r[rr] > 0.f ? 1.f / l_r[rr] : 0.f;
            const long ob = ((long)r * a.nh + h) * DC;
#pragma unroll
            for (int nt = 0; nt < 32; ++nt) {
                const int col = 256 * half + nt * 8 + 2 * tig;
                const float v0 = o[nt][2 * rr] * inv, v1 = o[nt][2 * rr + 1] * inv;
                if (a.olat) *reinterpret_cast<float2*>(a.olat + ob + col) = make_float2(v0, v1);
                if (a.olat_bf) *reinterpret_cast<uint32_t*>(a.olat_bf + ob + col) = pack2_bf16(v0, v1);
            }
            continue;
        }
        const long base = ((long)r * a.nh + h) * a.splits + s;
        if (half == 0 && tig == 0) {
            a.part_ml[base * 2] = m_r[rr];
            a.part_ml[base * 2 + 1] = l_r[rr];
        }
#pragma unroll
        for (int nt = 0; nt < 32; ++nt) {
            const int col = 256 * half + nt * 8 + 2 * tig;
            *reinterpret_cast<float2*>(a.part_o + base * DC + col) = make_float2(o[nt][2 * rr], o[nt][2 * rr + 1]);
        }
    }
}

// Split-K merge: o_lat[r, h] = sum_s e^{m_s - M} o_s / sum_s e^{m_s - M} l_s (fp32 and/or bf16).
// One CTA per (head, row); thread t owns the four latent columns 4 (t % C4) .. + 4 (C4 = d_c / 4) of the
// splits s = t / C4 + j G (j < J).  It issues all of its partial loads first, so they are in flight
// while warp 0 turns the (m_s, l_s) pairs into split weights.  Up to 16 splits one group of C4 threads
// holds them all; beyond that G groups (about four splits per thread, up to kMergeThreads threads) meet
// in shared memory.  With fixed-chunk splits only the splits that reach into the row's context are read.
constexpr int kMergeThreads = 512;
constexpr int kMergeJ = 16;          // splits per thread: G >= 4 covers the 64-split maximum
template <int J, bool MULTI>         // J splits per thread at most; MULTI: several split groups
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const AttnArgs a) {
    pdl_trigger();
    pdl_wait();
    __shared__ float wsp[64];
    __shared__ float4 red[MULTI ? kMergeThreads : 1];
    const int h = blockIdx.x, r = blockIdx.y;
    const int S = a.splits;
    const long base = ((long)r * a.nh + h) * S;
    const int C4 = a.dc / 4, G = MULTI ? blockDim.x / C4 : 1;
    // only the splits that cover part of this row's context hold partials
    const int Sv = live_splits(a, r);
    const int t = threadIdx.x, col4 = t % C4, grp = t / C4;
    const bool active = grp < G;
    float4 o[J];
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int sp = grp + j * G;
        o[j] = (active && sp < Sv) ? *reinterpret_cast<const float4*>(a.part_o + (base + sp) * a.dc + 4 * col4)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (t < 32) {
        float m0 = -FLT_MAX, m1 = -FLT_MAX, l0 = 0.f, l1 = 0.f;
        if (t < Sv) { m0 = a.part_ml[(base + t) * 2]; l0 = a.part_ml[(base + t) * 2 + 1]; }
        if (t + 32 < Sv) { m1 = a.part_ml[(base + t + 32) * 2]; l1 = a.part_ml[(base + t + 32) * 2 + 1]; }
        const float mx = warp_max(fmaxf(m0, m1));
        const float e0 = l0 > 0.f ? __expf(m0 - mx) : 0.f;
        const float e1 = l1 > 0.f ? __expf(m1 - mx) : 0.f;
        const float den = warp_sum(e0 * l0 + e1 * l1);
        const float inv = den > 0.f ? 1.f / den : 0.f;
        wsp[t] = e0 * inv;
        wsp[t + 32] = e1 * inv;
    }
    __syncthreads();
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int sp = grp + j * G;
        const float w = (active && sp < Sv) ? wsp[sp] : 0.f;
        v.x = fmaf(w, o[j].x, v.x); v.y = fmaf(w, o[j].y, v.y);
        v.z = fmaf(w, o[j].z, v.z); v.w = fmaf(w, o[j].w, v.w);
    }
    if (MULTI) {
        red[t] = v;
        __syncthreads();
        if (grp != 0) return;
        for (int g = 1; g < G; ++g) {
            const float4 u = red[g * C4 + col4];
            v.x += u.x; v.y += u.y; v.z += u.z; v.w += u.w;
        }
    } else if (!active) {
        return;
    }
    const long off = ((long)r * a.nh + h) * a.dc + 4 * col4;
    if (a.olat) *reinterpret_cast<float4*>(a.olat + off) = v;
    if (a.olat_bf) {
        uint2 u;
        u.x = pack2_bf16(v.x, v.y);
        u.y = pack2_bf16(v.z, v.w);
        *reinterpret_cast<uint2*>(a.olat_bf + off) = u;
    }
}

// Split merge fused with the value up-projection, for few rows (the weight-streaming path): CTA h
// stages W_UV,h (the d_v value rows of kv_b for head h, d_v x d_c bf16, contiguous) into shared memory
// with one bulk copy issued before the wait on the attention kernel, merges the head's split partials
// of every row into o_lat (shared memory), then forms o[r, h] = W_UV,h o_lat[r, h] (warp w: rows
// v = 16w .. 16w + 15, lanes over d_c, a warp reduction per output).  d_c 512, d_v 128, M <= 8 rows.
namespace mu {
constexpr int DC = 512, DV = 128, THREADS = 256, MAXR = 8;
constexpr int W_BYTES = DV * DC * 2;
constexpr size_t SMEM = (size_t)W_BYTES + (size_t)MAXR * DC * 4 + 64;
}  // namespace mu

__global__ void __launch_bounds__(mu::THREADS, 1) merge_unabsorb_kernel(const AttnArgs a) {
    using namespace mu;
    pdl_trigger();
    extern __shared__ __align__(128) unsigned char msm[];
    bf16* w = reinterpret_cast<bf16*>(msm);                              // [DV][DC]
    float* ol = reinterpret_cast<float*>(msm + W_BYTES);                 // [M][DC]
    uint64_t* bar = reinterpret_cast<uint64_t*>(msm + W_BYTES + MAXR * DC * 4);
    __shared__ float wsp[kMergeUnabsorbMaxSplits];
    const int h = blockIdx.x, t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const uint32_t sbar = smem_u32(bar);
    if (t == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(sbar));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(sbar), "r"(W_BYTES) : "memory");
        const bf16* src = reinterpret_cast<const bf16*>(a.kv_b) + ((long)h * (a.dn + a.dv) + a.dn) * DC;
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                     ::"r"(smem_u32(w)), "l"(src), "r"(W_BYTES), "r"(sbar) : "memory");
    }
    pdl_wait();
    const int S = a.splits;
    for (int r = 0; r < a.M; ++r) {
        const long base = ((long)r * a.nh + h) * S;
        const int Sv = live_splits(a, r);
        __syncthreads();   // wsp of the previous row is consumed
        if (t < 32) {      // lane t weighs splits t, t + 32, t + 64, t + 96
            constexpr int J = kMergeUnabsorbMaxSplits / 32;
            float m[J], l[J];
            float mx = -FLT_MAX;
#pragma unroll
            for (int j = 0; j < J; ++j) {
                const int sp = t + 32 * j;
                m[j] = sp < Sv ? a.part_ml[(base + sp) * 2] : -FLT_MAX;
                l[j] = sp < Sv ? a.part_ml[(base + sp) * 2 + 1] : 0.f;
                mx = fmaxf(mx, m[j]);
            }
            mx = warp_max(mx);
            float den = 0.f;
#pragma unroll
            for (int j = 0; j < J; ++j) {
                m[j] = l[j] > 0.f ? __expf(m[j] - mx) : 0.f;
                den = fmaf(m[j], l[j], den);
            }
            den = warp_sum(den);
            const float inv = den > 0.f ? 1.f / den : 0.f;
#pragma unroll
            for (int j = 0; j < J; ++j) wsp[t + 32 * j] = m[j] * inv;
        }
        __syncthreads();
        // thread t: columns 4 (t % 128) .. + 3 of the splits sp = t / 128, + 2, ...: 16-byte loads, eight in
        // flight per thread; the two halves meet in shared memory
        const int cq = t & 127, g = t >> 7;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int sp0 = g; sp0 < Sv; sp0 += 16) {
            float4 pv[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int sp = sp0 + 2 * j;
                pv[j] = sp < Sv ? *reinterpret_cast<const float4*>(a.part_o + (base + sp) * DC + 4 * cq)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int sp = sp0 + 2 * j;
                const float ws = sp < Sv ? wsp[sp] : 0.f;
                v.x = fmaf(ws, pv[j].x, v.x); v.y = fmaf(ws, pv[j].y, v.y);
                v.z = fmaf(ws, pv[j].z, v.z); v.w = fmaf(ws, pv[j].w, v.w);
            }
        }
        float4* row = reinterpret_cast<float4*>(ol + r * DC);
        if (g == 1) row[cq] = v;
        __syncthreads();
        if (g == 0) {
            const float4 u = row[cq];
            row[cq] = make_float4(v.x + u.x, v.y + u.y, v.z + u.z, v.w + u.w);
        }
    }
    // the staged weights (bounded wait; a wait that runs out flags the call and leaves the outputs alone)
    bool ok = false;
    for (uint32_t i = 0; i < (1u << 22) && !ok; ++i) {
        uint32_t done;
        asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n selp.u32 %0, 1, 0, p;\n}\n"
                     : "=r"(done) : "r"(sbar) : "memory");
        ok = done != 0;
    }
    __syncthreads();
    if (!ok) {
        if (t == 0) set_err(a.err, EAGLE3_DEVERR_TIMEOUT);
        return;
    }
    for (int r = 0; r < a.M; ++r) {
        float x[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) x[j] = ol[r * DC + lane * 16 + j];
        for (int v = warp * 16; v < warp * 16 + 16; ++v) {
            const uint4* wr = reinterpret_cast<const uint4*>(w + (long)v * DC + lane * 16);
            float f[16];
            unpack_bf16x8(wr[0], f);
            unpack_bf16x8(wr[1], f + 8);
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < 16; ++j) acc = fmaf(f[j], x[j], acc);
            acc = warp_sum(acc);
            if (lane == 0) a.o[((long)r * a.nh + h) * DV + v] = acc;
        }
    }
}

bool merge_unabsorb_supported(const AttnArgs& a) {
    return a.dt == BF16 && a.dc == mu::DC && a.dv == mu::DV && a.M <= mu::MAXR && a.splits >= 1 && a.splits <= kMergeUnabsorbMaxSplits &&
           a.o != nullptr && ((uintptr_t)a.kv_b & 15u) == 0;
}

cudaError_t launch_merge_unabsorb(const AttnArgs& a, cudaStream_t st) {
    if (!merge_unabsorb_supported(a)) return cudaErrorInvalidValue;
    cudaError_t e = smem_optin((const void*)merge_unabsorb_kernel, (int)mu::SMEM);
    if (e != cudaSuccess) return e;
    return launch_pdl(merge_unabsorb_kernel, dim3(a.nh), dim3(mu::THREADS), mu::SMEM, st, a);
}

cudaError_t launch_merge(const AttnArgs& a, cudaStream_t st) {
    if (a.splits < 1 || a.splits > 64 || a.dc % 4 || a.dc > 4 * kMergeThreads) return cudaErrorInvalidValue;
    const int C4 = a.dc / 4;
    // up to 16 splits: one group whose threads hold all of them, no cross-group reduction
    const dim3 one((C4 + 31) / 32 * 32);
    if (a.splits <= 4) return launch_pdl(merge_kernel<4, false>, dim3(a.nh, a.M), one, 0, st, a);
    if (a.splits <= 8) return launch_pdl(merge_kernel<8, false>, dim3(a.nh, a.M), one, 0, st, a);
    if (a.splits <= 16) return launch_pdl(merge_kernel<16, false>, dim3(a.nh, a.M), one, 0, st, a);
    int G = (a.splits + 3) / 4;
    if (G > kMergeThreads / C4) G = kMergeThreads / C4;
    if ((long)G * kMergeJ < a.splits) return cudaErrorInvalidValue;   // G split groups of kMergeJ splits
    const int threads = (C4 * G + 31) / 32 * 32;
    return launch_pdl(merge_kernel<kMergeJ, true>, dim3(a.nh, a.M), dim3(threads), 0, st, a);
}

// Rotated rope part of the query: qa[r, h, dc:] = RoPE(q_pe[r, h], pos_r) (fp32 and bf16).
__global__ void rope_q_kernel(const AttnArgs a) {
    pdl_trigger();
    pdl_wait();
    const int r = blockIdx.x;
    const int half = a.dr / 2, dqk = a.dn + a.dr, D = a.dc + a.dr;
    const int pos = a.row_pos[r];
    for (int t = threadIdx.x; t < a.nh * half; t += blockDim.x) {
        const int h = t / half, p = t % half;
        const float c = a.rope_cos[(long)pos * half + p], s = a.rope_sin[(long)pos * half + p];
        const long qi = ((long)r * a.nh + h) * dqk + a.dn + 2 * p;
        float x0, x1;
        if (a.q_bf) {
            x0 = __bfloat162float(a.q_bf[qi]);
            x1 = __bfloat162float(a.q_bf[qi + 1]);
        } else {
            x0 = a.q[qi];
            x1 = a.q[qi + 1];
        }
        const float y0 = x0 * c - x1 * s, y1 = x0 * s + x1 * c;
        const long o = ((long)r * a.nh + h) * D + a.dc + 2 * p;
        if (a.qa) {
            a.qa[o] = y0;
            a.qa[o + 1] = y1;
        }
        if (a.qa_bf) *reinterpret_cast<uint32_t*>(a.qa_bf + o) = pack2_bf16(y0, y1);
    }
}

// out[h, c, i] = kv_b[h (dn + dv) + i, c]: the key up-projection of each head, transposed so that the
// absorbed query q_lat,h = W_UK,h^T q_nope,h is a K-major GEMM over i.
__global__ void transpose_wuk_kernel(const bf16* kv_b, int nh, int dn, int dv, int dc, bf16* out) {
    __shared__ bf16 tile[32][33];
    const int h = blockIdx.z, c0 = blockIdx.x * 32, i0 = blockIdx.y * 32;
    const bf16* W = kv_b + (long)h * (dn + dv) * dc;
    for (int k = threadIdx.y; k < 32; k += blockDim.y) {
        const int i = i0 + k, c = c0 + threadIdx.x;
        tile[k][threadIdx.x] = (i < dn && c < dc) ? W[(long)i * dc + c] : __float2bfloat16_rn(0.f);
    }
    __syncthreads();
    for (int k = threadIdx.y; k < 32; k += blockDim.y) {
        const int c = c0 + k, i = i0 + threadIdx.x;
        if (c < dc && i < dn) out[((long)h * dc + c) * dn + i] = tile[threadIdx.x][k];
    }
}

cudaError_t launch_rope_q(const AttnArgs& a, cudaStream_t st) {
    launch_pdl(rope_q_kernel, dim3(a.M), dim3(256), 0, st, a);
    return cudaGetLastError();
}

cudaError_t launch_transpose_wuk(const void* kv_b, int nh, int dn, int dv, int dc, bf16* out, cudaStream_t st) {
    dim3 grid((dc + 31) / 32, (dn + 31) / 32, nh);
    transpose_wuk_kernel<<<grid, dim3(32, 8), 0, st>>>(reinterpret_cast<const bf16*>(kv_b), nh, dn, dv, dc, out);
    return cudaGetLastError();
}

bool attention_supported(int dc, int dr, int dn, int dv) {
    (void)dn; (void)dv;
    return (dc == 512 && dr == 64) || (dc == 32 && dr == 16);
}

int attention_heads_per_cta(int dt, int dc, int dr) {
    return (dt == BF16 && dc == 512 && dr == 64) ? mla_mma::HEADS : kHeadsPerCta;
}

bool attention_one_cta_per_sm(int dt, int dc, int dr) {
    return dt == BF16 && dc == 512 && dr == 64;   // mla_mma::SMEM (158 KB) leaves room for one CTA
}

cudaError_t launch_absorb(const AttnArgs& a, cudaStream_t st) {
    const int cols = a.dc < kAbsCols ? a.dc : kAbsCols;
    if (a.dc % cols) return cudaErrorInvalidValue;
    const bool one = a.dt == BF16 && a.M == 1;
    const int rows = one ? 1 : kAbsRows;
    dim3 grid(a.nh, a.dc / cols, (a.M + rows - 1) / rows);
    const int RG = 256 / (cols / 8);
    const size_t sm = ((size_t)rows * a.dn + (size_t)RG * rows * cols) * sizeof(float);
    const void* k = one ? (const void*)absorb_kernel<bf16, 1>
                        : a.dt == BF16 ? (const void*)absorb_kernel<bf16, kAbsRows> : (const void*)absorb_kernel<float, kAbsRows>;
    {
        cudaError_t e = smem_optin(k, 96 * 1024);
        if (e != cudaSuccess) return e;
    }
    if (sm > 96 * 1024) return cudaErrorInvalidValue;
    if (one) launch_pdl(absorb_kernel<bf16, 1>, dim3(grid), dim3(256), sm, st, a);
    else if (a.dt == BF16) launch_pdl(absorb_kernel<bf16, kAbsRows>, dim3(grid), dim3(256), sm, st, a);
    else launch_pdl(absorb_kernel<float, kAbsRows>, dim3(grid), dim3(256), sm, st, a);
    return cudaGetLastError();
}

template <typename T, int DC, int DR>
static cudaError_t attn_launch(const AttnArgs& a, cudaStream_t st) {
    constexpr int D = DC + DR;
    constexpr int WORDS = D / (4 / sizeof(T));
    const size_t sm = (size_t)kHeadsPerCta * D * sizeof(float) + (size_t)kTile * (WORDS | 1) * sizeof(uint32_t);
    {
        cudaError_t e = smem_optin((const void*)attention_kernel<T, DC, DR>, (int)sm);
        if (e != cudaSuccess) return e;
    }
    dim3 grid(a.splits, (a.nh + kHeadsPerCta - 1) / kHeadsPerCta, a.M);
    launch_pdl(attention_kernel<T, DC, DR>, dim3(grid), dim3(kAttnWarps * 32), sm, st, a);
    return cudaGetLastError();
}

cudaError_t launch_attention(const AttnArgs& a, cudaStream_t st) {
    if (a.dc == 512 && a.dr == 64) {
        if (a.dt == BF16) {
            {
                cudaError_t e = smem_optin((const void*)attention_mma_kernel, (int)mla_mma::SMEM);
                if (e != cudaSuccess) return e;
            }
            if (!a.qa_bf) return cudaErrorInvalidValue;
            dim3 grid(a.splits, (a.nh + mla_mma::HEADS - 1) / mla_mma::HEADS, a.M);
            launch_pdl(attention_mma_kernel, dim3(grid), dim3(mla_mma::WARPS * 32), mla_mma::SMEM, st, a);
            return cudaGetLastError();
        }
        return attn_launch<float, 512, 64>(a, st);
    }
    if (a.dc == 32 && a.dr == 16)
        return a.dt == BF16 ? attn_launch<bf16, 32, 16>(a, st) : attn_launch<float, 32, 16>(a, st);
    return cudaErrorInvalidValue;
}


}  // namespace e3
