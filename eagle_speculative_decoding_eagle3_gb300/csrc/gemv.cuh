// Weight-streaming GEMM for few activation rows (decode and small extends).
//
// y[m, n] = sum_k A[m, k] W[n, k] — the bias-free linear layers of the draft head (fc, q_a | kv_a,
// q_b, o_proj, gate | up, down, lm_head, the per-head value up-projection; "Eagle3 DeepseekV3 in MAX"
// §4).  At a handful of rows a layer is bound by streaming W from HBM once, so the kernel is laid out
// for HBM:
//  * one balanced wave: the grid holds gemv_cps CTAs per SM (two; three for FP8 weights outside the GLU,
//    where the arithmetic per byte leaves a warp computing for longer between its load batches and a
//    third CTA with half the loads per batch keeps more of them in flight) and every warp owns an equal
//    range of weight rows (rows_per_warp), so no SM idles in a half-empty last wave;
//  * a warp streams R of its rows at once (R = 1 or 4), each with U 16-byte non-allocating loads per
//    lane (lane l reads elements [8l + 256c, +8) of a row; FP8: [16l + 512c, +16)), so gemv_loads (16 at
//    two CTAs per SM, 8 at three) loads of 16 B are in flight per lane whatever the row length;
//  * the activation rows (up to MR) stay L1/L2 resident and are loaded once per chunk for all R rows;
//  * at the end of each pass the warp reduces its partial dot products and applies the fused epilogue:
//    store, residual add, SiLU(gate) * up (two weight rows per output), or a running row argmax with
//    the lowest index winning ties (the logits never round-trip through HBM unless a debug buffer asks
//    for them).
// Two kernels share this layout: gemv_kernel gives each warp whole rows; gemv_ks_kernel splits every row
// across the warps of a row group, for layers whose rows are long and few per warp.
// Weights are fp32, bf16, FP8 E4M3 codes with one fp32 scale per output row, or NVFP4 (E2M1 codes, an
// E4M3 scale per 16 weights, an fp32 scale per matrix): the drafter's FP8 / NVFP4 post-training
// quantization, "EAGLE head deep dive", deployment.  The FP8 kernels widen the codes exactly to fp32,
// accumulate code * activation and multiply each output column's sum by its row scale; the NVFP4 path
// (whole-row kernel only) sums each block of 16 products, multiplies it by the block's scale, and the
// output by the matrix scale.  The templates live in this header; gemv.cu instantiates the fp32 / bf16
// weights, gemv_fp8.cu the FP8 and gemv_fp4.cu the NVFP4 ones.
#pragma once
#include <float.h>
#include <limits.h>

#include "common.cuh"
#include "kernels.h"

namespace e3 {

constexpr int kGemvWarps = 8;
constexpr int kGemvMaxCtasPerSm = 3;   // the largest gemv_cps: sizes the argmax partials

template <typename T> constexpr bool kIsFp8 = false;
template <> constexpr bool kIsFp8<fp8e4> = true;
// CTAs per SM of a GEMV launch and the 16-byte weight loads per lane and iteration that fit its registers
template <typename TW, int EPI> constexpr int gemv_cps() { return kIsFp8<TW> && EPI != EPI_GLU ? 3 : 2; }
template <typename TW, int EPI> constexpr int gemv_loads() { return gemv_cps<TW, EPI>() >= 3 ? 8 : 16; }
template <typename T> constexpr bool kIsFp4 = false;
template <> constexpr bool kIsFp4<fp4x2> = true;

// The unit a lane loads from a weight row: 8 elements (fp32: two 16-byte loads, bf16: one), 16 E4M3
// codes or 32 E2M1 codes (one 16-byte load).  A warp covers kChunk<TW> = 32 units' elements per row and
// step.  PK elements share one TW (two E2M1 codes per byte).
template <typename TW> struct WUnit {
    static constexpr int EL = 8, BYTES = 8 * (int)sizeof(TW), PK = 1;
    using Raw = Raw8<TW>;
};
template <> struct WUnit<fp8e4> { static constexpr int EL = 16, BYTES = 16, PK = 1; using Raw = Raw16e4; };
template <> struct WUnit<fp4x2> { static constexpr int EL = 32, BYTES = 16, PK = 2; using Raw = Raw16e4; };
template <typename TW> constexpr int kChunk = 32 * WUnit<TW>::EL;
template <typename TW> __device__ __forceinline__ typename WUnit<TW>::Raw ldw(const TW* p) {
    if constexpr (kIsFp8<TW> || kIsFp4<TW>) return Raw16e4{ld_stream16(p)}; else return ld8<true>(p);
}
template <typename TW> __device__ __forceinline__ typename WUnit<TW>::Raw zerow() {
    if constexpr (kIsFp8<TW> || kIsFp4<TW>) return Raw16e4{make_uint4(0, 0, 0, 0)}; else return zero8((TW*)nullptr);
}
// The two E4M3 block scales of an NVFP4 unit (32 codes = 2 blocks of 16), as a 16-bit load.
__device__ __forceinline__ uint32_t ld_scale_pair(const uint8_t* p) {
    unsigned short v;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}
// EL activations of row `p` (fp32 or bf16) widened to fp32
template <int EL, typename TA> __device__ __forceinline__ void ld_act(const TA* p, float* v) {
#pragma unroll
    for (int h = 0; h < EL / 8; ++h) widen(ld8<false>(p + 8 * h), v + 8 * h);
}

// Scale of output column n of an FP8 GEMV (GLU: q selects the gate or up matrix; else the segment).
__device__ __forceinline__ float row_scale(const GemvArgs& g, bool glu, int n, int q) {
    if (glu) return __ldg(g.wscale[q] + n);
    const int seg = (g.nseg_w > 1 && n >= g.nw[0]) ? 1 : 0;
    return __ldg(g.wscale[seg] + (seg ? n - g.nw[0] : n));
}
// The NVFP4 matrix scale of output column n's matrix.
__device__ __forceinline__ float matrix_scale(const GemvArgs& g, bool glu, int n, int q) {
    const int seg = glu ? q : ((g.nseg_w > 1 && n >= g.nw[0]) ? 1 : 0);
    return __ldg(g.wscale[seg]);
}

template <typename TA, typename TW, int MR, int EPI, int R>
__global__ void __launch_bounds__(kGemvWarps * 32, gemv_cps<TW, EPI>()) gemv_kernel(const GemvArgs g, int rows_per_warp) {
    constexpr int NW = (EPI == EPI_GLU) ? 2 : 1;   // weight rows read per output column
    constexpr int EL = WUnit<TW>::EL, CW = kChunk<TW>, PK = WUnit<TW>::PK;
    constexpr bool F4 = kIsFp4<TW>;
    constexpr int U0 = gemv_loads<TW, EPI>() / (R * NW) * 16 / WUnit<TW>::BYTES;
    constexpr int U = U0 < 1 ? 1 : U0;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int m0 = blockIdx.x * MR;
    const int mcount = min(MR, g.M - m0);
    const int K = g.K;
    const int r_begin = (blockIdx.y * kGemvWarps + warp) * rows_per_warp;
    const int r_end = min(g.N, r_begin + rows_per_warp);
    const int ka0 = g.ka[0], ka01 = g.ka[0] + g.ka[1];

    const long KW = K / PK;                          // TW per weight row
    auto wrow = [&](int n, int q) -> const TW* {
        if (EPI == EPI_GLU) return reinterpret_cast<const TW*>(g.w[q]) + (long)n * KW;
        if (g.w_grp)
            return reinterpret_cast<const TW*>(g.w[0]) +
                   ((long)(n / g.w_grp) * g.w_grp_stride + g.w_row0 + n % g.w_grp) * KW;
        const int seg = (g.nseg_w > 1 && n >= g.nw[0]) ? 1 : 0;
        return reinterpret_cast<const TW*>(g.w[seg]) + (long)(seg ? n - g.nw[0] : n) * KW;
    };
    // NVFP4 block scales of row n: K / 16 bytes
    auto bsrow = [&](int n, int q) -> const uint8_t* {
        const int seg = EPI == EPI_GLU ? q : ((g.nseg_w > 1 && n >= g.nw[0]) ? 1 : 0);
        return g.wbs[seg] + (long)(seg && EPI != EPI_GLU ? n - g.nw[0] : n) * (K / 16);
    };

    float best_v[MR];
    int best_i[MR];
#pragma unroll
    for (int i = 0; i < MR; ++i) { best_v[i] = -FLT_MAX; best_i[i] = INT_MAX; }

    // The first batch of weight loads does not depend on the previous kernel: issue it, then wait.
    pdl_trigger();
    bool waited = false;
    for (int p0 = r_begin; p0 < r_end; p0 += R) {
        const int nr = min(R, r_end - p0);
        const TW* wp[R][NW];
        const uint8_t* bp[R][NW];
#pragma unroll
        for (int j = 0; j < R; ++j)
#pragma unroll
            for (int q = 0; q < NW; ++q) {
                wp[j][q] = wrow(p0 + (j < nr ? j : 0), q);
                if constexpr (F4) bp[j][q] = bsrow(p0 + (j < nr ? j : 0), q);
            }
        // the per-head GEMVs use one activation slice per row group; all rows of a pass share it
        const long aoff = g.a_grp ? (long)(p0 / g.a_grp) * g.a_grp_stride : 0;
        float sc[R][NW];                      // FP8 row / NVFP4 matrix scales, loaded with the first weights
#pragma unroll
        for (int j = 0; j < R; ++j)
#pragma unroll
            for (int q = 0; q < NW; ++q)
                sc[j][q] = kIsFp8<TW> ? row_scale(g, EPI == EPI_GLU, p0 + (j < nr ? j : 0), q)
                                      : (F4 ? matrix_scale(g, EPI == EPI_GLU, p0 + (j < nr ? j : 0), q) : 1.f);
        float acc[MR][R][NW];
#pragma unroll
        for (int i = 0; i < MR; ++i)
#pragma unroll
            for (int j = 0; j < R; ++j)
#pragma unroll
                for (int q = 0; q < NW; ++q) acc[i][j][q] = 0.f;

        for (int k0 = lane * EL; k0 < K; k0 += CW * U) {
            typename WUnit<TW>::Raw wr[U][R][NW];
            uint32_t bs[U][R][NW];                   // NVFP4: the unit's two block scales
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int k = k0 + u * CW;
#pragma unroll
                for (int j = 0; j < R; ++j)
#pragma unroll
                    for (int q = 0; q < NW; ++q) {
                        wr[u][j][q] = (k < K && j < nr) ? ldw(wp[j][q] + k / PK) : zerow<TW>();
                        if constexpr (F4) bs[u][j][q] = (k < K && j < nr) ? ld_scale_pair(bp[j][q] + k / 16) : 0u;
                    }
            }
            if (!waited) { pdl_wait(); waited = true; }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int k = k0 + u * CW;
                if (k < K) {
                    const int s = (k >= ka0) + (k >= ka01);
                    const int kl = k - (s == 0 ? 0 : (s == 1 ? ka0 : ka01));
                    const TA* ap = reinterpret_cast<const TA*>(g.a[s]) + (long)m0 * g.lda[s] + aoff + kl;
#pragma unroll
                    for (int i = 0; i < MR; ++i) {
                        if (i < mcount) {
                            if constexpr (F4) {
                                // two blocks of 16: sum code x activation, then times the block's scale
#pragma unroll
                                for (int h = 0; h < 2; ++h) {
                                    float av[16];
                                    ld_act<16>(ap + i * g.lda[s] + 16 * h, av);
#pragma unroll
                                    for (int j = 0; j < R; ++j)
#pragma unroll
                                        for (int q = 0; q < NW; ++q) {
                                            float wv[16];
                                            const uint4 w4 = wr[u][j][q].a;
                                            e2m1x16_to_f32(h ? w4.z : w4.x, h ? w4.w : w4.y, wv);
                                            float p = 0.f;
#pragma unroll
                                            for (int e = 0; e < 16; ++e) p = fmaf(wv[e], av[e], p);
                                            acc[i][j][q] = fmaf(p, e4m3_to_f32(bs[u][j][q] >> (8 * h)), acc[i][j][q]);
                                        }
                                }
                            } else {
                                float av[EL];
                                ld_act<EL>(ap + i * g.lda[s], av);
#pragma unroll
                                for (int j = 0; j < R; ++j)
#pragma unroll
                                    for (int q = 0; q < NW; ++q) {
                                        float wv[EL];
                                        widen(wr[u][j][q], wv);
#pragma unroll
                                        for (int e = 0; e < EL; ++e) acc[i][j][q] = fmaf(wv[e], av[e], acc[i][j][q]);
                                    }
                            }
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int i = 0; i < MR; ++i)
#pragma unroll
            for (int j = 0; j < R; ++j)
#pragma unroll
                for (int q = 0; q < NW; ++q) acc[i][j][q] = warp_sum(acc[i][j][q]) * sc[j][q];
#pragma unroll
        for (int i = 0; i < MR; ++i) {
            if (i >= mcount) continue;
            const long m = m0 + i;
#pragma unroll
            for (int j = 0; j < R; ++j) {
                if (j >= nr) continue;
                const int n = p0 + j;
                if (EPI == EPI_ARGMAX) {
                    if (better(acc[i][j][0], n, best_v[i], best_i[i])) { best_v[i] = acc[i][j][0]; best_i[i] = n; }
                    if (g.logits != nullptr && lane == (i * R + j) % 32) g.logits[m * g.ldl + n] = acc[i][j][0];
                } else if (lane == (i * R + j) % 32) {
                    float v;
                    if (EPI == EPI_GLU) v = silu(acc[i][j][0]) * acc[i][j][NW - 1];
                    else if (EPI == EPI_RESID) v = acc[i][j][0] + g.resid[m * g.ldr + n];
                    else v = acc[i][j][0];
                    g.y[m * g.ldy + n] = v;
                }
            }
        }
    }

    if (!waited) pdl_wait();
    if (EPI == EPI_ARGMAX) {
        __shared__ float sv[kGemvWarps][MR];
        __shared__ int si[kGemvWarps][MR];
        if (lane == 0) {
#pragma unroll
            for (int i = 0; i < MR; ++i) { sv[warp][i] = best_v[i]; si[warp][i] = best_i[i]; }
        }
        __syncthreads();
        if (threadIdx.x < MR && (int)threadIdx.x < mcount) {
            const int i = threadIdx.x;
            float bv = sv[0][i];
            int bi = si[0][i];
            for (int w = 1; w < kGemvWarps; ++w)
                if (better(sv[w][i], si[w][i], bv, bi)) { bv = sv[w][i]; bi = si[w][i]; }
            g.pval[(long)(m0 + i) * g.npart + blockIdx.y] = bv;
            g.pidx[(long)(m0 + i) * g.npart + blockIdx.y] = bi;
        }
    }
}

// K-split variant for long rows (bf16 or FP8 weights, no row grouping).  A CTA owns `rpc` consecutive output
// columns; its 8 warps form RG = 8 / KS row groups of KS warps, and the KS warps of a group split K
// (warp k of a group reads the warp chunks [k nch / KS, (k + 1) nch / KS) of every row).  A group
// streams R rows at once (U chunks each, gemv_loads loads of 16 B in flight per lane), so one activation load
// feeds R rows instead of the whole-row kernel's few, and a layer with few rows per warp (q_a | kv_a:
// 2112 rows for 2432 warps) still keeps every warp busy.  Each round the RG groups take one pass of R
// rows each; the KS partial sums of every output meet in shared memory, where the epilogue is applied.
template <typename TA, typename TW, int MR, int EPI, int R>
__global__ void __launch_bounds__(kGemvWarps * 32, gemv_cps<TW, EPI>()) gemv_ks_kernel(const GemvArgs g, int rpc, int KS) {
    constexpr int NW = (EPI == EPI_GLU) ? 2 : 1;
    constexpr int EL = WUnit<TW>::EL, CW = kChunk<TW>;
    static_assert(!kIsFp4<TW>, "NVFP4 weights stream through the whole-row kernel");
    constexpr int U0 = gemv_loads<TW, EPI>() / (R * NW) * 16 / WUnit<TW>::BYTES;
    static_assert(R * MR <= 32, "one epilogue thread per (row group, row, activation row)");
    constexpr int U = U0 < 1 ? 1 : U0;
    constexpr int OUT = MR * R * NW;                 // partial sums per warp and pass
    __shared__ float red[kGemvWarps][OUT];
    __shared__ float fin[kGemvWarps * R * MR];       // ARGMAX: the round's reduced scores
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int RG = kGemvWarps / KS, ks = warp % KS, rg = warp / KS;
    const int m0 = blockIdx.x * MR, mcount = min(MR, g.M - m0);
    const int K = g.K, nch = (K + CW - 1) / CW;
    const int c0 = ks * nch / KS, c1 = (ks + 1) * nch / KS;
    const int row0 = blockIdx.y * rpc, row1 = min(g.N, row0 + rpc);
    const int npass = (row1 - row0 + R - 1) / R, nround = (npass + RG - 1) / RG;
    const int ka0 = g.ka[0], ka01 = g.ka[0] + g.ka[1];

    auto wrow = [&](int n, int q) -> const TW* {
        if (EPI == EPI_GLU) return reinterpret_cast<const TW*>(g.w[q]) + (long)n * K;
        const int seg = (g.nseg_w > 1 && n >= g.nw[0]) ? 1 : 0;
        return reinterpret_cast<const TW*>(g.w[seg]) + (long)(seg ? n - g.nw[0] : n) * K;
    };

    float best_v[MR];
    int best_i[MR];
#pragma unroll
    for (int i = 0; i < MR; ++i) { best_v[i] = -FLT_MAX; best_i[i] = INT_MAX; }

    pdl_trigger();
    bool waited = false;
    for (int q = 0; q < nround; ++q) {
        const int p0 = row0 + (q * RG + rg) * R;
        const int nr = max(0, min(R, row1 - p0));
        // this thread's output of the round's epilogue (at most one: RG * R * MR <= 8 * 32) and, for FP8,
        // its row scales, loaded with the round's first weights
        const int et = threadIdx.x, egrp = et / (R * MR), ej = (et % (R * MR)) / MR, ei = et % MR;
        const int en = row0 + (q * RG + egrp) * R + ej;
        const bool eown = et < RG * R * MR;
        float esc0 = 1.f, esc1 = 1.f;
        if (kIsFp8<TW> && eown && en < row1) {
            esc0 = row_scale(g, EPI == EPI_GLU, en, 0);
            if (NW == 2) esc1 = row_scale(g, true, en, 1);
        }
        float acc[MR][R][NW];
#pragma unroll
        for (int i = 0; i < MR; ++i)
#pragma unroll
            for (int j = 0; j < R; ++j)
#pragma unroll
                for (int w = 0; w < NW; ++w) acc[i][j][w] = 0.f;
        if (nr > 0) {
            const TW* wp[R][NW];
#pragma unroll
            for (int j = 0; j < R; ++j)
#pragma unroll
                for (int w = 0; w < NW; ++w) wp[j][w] = wrow(p0 + (j < nr ? j : 0), w);
            for (int c = c0; c < c1; c += U) {
                typename WUnit<TW>::Raw wr[U][R][NW];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int k = (c + u) * CW + lane * EL;
                    const bool ok = c + u < c1 && k < K;
#pragma unroll
                    for (int j = 0; j < R; ++j)
#pragma unroll
                        for (int w = 0; w < NW; ++w)
                            wr[u][j][w] = (ok && j < nr) ? ldw(wp[j][w] + k) : zerow<TW>();
                }
                if (!waited) { pdl_wait(); waited = true; }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int k = (c + u) * CW + lane * EL;
                    if (c + u < c1 && k < K) {
                        const int s = (k >= ka0) + (k >= ka01);
                        const int kl = k - (s == 0 ? 0 : (s == 1 ? ka0 : ka01));
                        const TA* ap = reinterpret_cast<const TA*>(g.a[s]) + (long)m0 * g.lda[s] + kl;
#pragma unroll
                        for (int i = 0; i < MR; ++i) {
                            if (i < mcount) {
                                float av[EL];
                                ld_act<EL>(ap + i * g.lda[s], av);
#pragma unroll
                                for (int j = 0; j < R; ++j)
#pragma unroll
                                    for (int w = 0; w < NW; ++w) {
                                        float wv[EL];
                                        widen(wr[u][j][w], wv);
#pragma unroll
                                        for (int e = 0; e < EL; ++e) acc[i][j][w] = fmaf(wv[e], av[e], acc[i][j][w]);
                                    }
                            }
                        }
                    }
                }
            }
        }
        if (!waited) { pdl_wait(); waited = true; }
#pragma unroll
        for (int i = 0; i < MR; ++i)
#pragma unroll
            for (int j = 0; j < R; ++j)
#pragma unroll
                for (int w = 0; w < NW; ++w) {
                    const float v = warp_sum(acc[i][j][w]);
                    if (lane == 0) red[warp][(i * R + j) * NW + w] = v;
                }
        __syncthreads();
        // one thread per (row group, row of the pass, activation row)
        if (eown) {
            const int t = et, grp = egrp, j = ej, i = ei, n = en;
            float v0 = 0.f, v1 = 0.f;
            for (int k = 0; k < KS; ++k) {
                v0 += red[grp * KS + k][(i * R + j) * NW];
                if (NW == 2) v1 += red[grp * KS + k][(i * R + j) * NW + NW - 1];
            }
            v0 *= esc0;
            v1 *= esc1;
            const bool valid = i < mcount && n < row1;
            const long m = m0 + i;
            if (EPI == EPI_ARGMAX) {
                fin[t] = valid ? v0 : -FLT_MAX;
                if (valid && g.logits != nullptr) g.logits[m * g.ldl + n] = v0;
            } else if (valid) {
                float v;
                if (EPI == EPI_GLU) v = silu(v0) * v1;
                else if (EPI == EPI_RESID) v = v0 + g.resid[m * g.ldr + n];
                else v = v0;
                g.y[m * g.ldy + n] = v;
            }
        }
        if (EPI == EPI_ARGMAX) {
            __syncthreads();
            const int t = threadIdx.x;
            if (t < MR) {
                // ascending column order; better() keeps the lowest index on ties
                for (int grp = 0; grp < RG; ++grp)
                    for (int j = 0; j < R; ++j) {
                        const int n = row0 + (q * RG + grp) * R + j;
                        const float v = fin[(grp * R + j) * MR + t];
                        if (n < row1 && better(v, n, best_v[t], best_i[t])) { best_v[t] = v; best_i[t] = n; }
                    }
            }
        }
        __syncthreads();
    }
    if (!waited) pdl_wait();
    if (EPI == EPI_ARGMAX && (int)threadIdx.x < mcount) {
        const int i = threadIdx.x;
        g.pval[(long)(m0 + i) * g.npart + blockIdx.y] = best_v[i];
        g.pidx[(long)(m0 + i) * g.npart + blockIdx.y] = best_i[i];
    }
}

// K slices per row group, from the row's nch warp chunks (kChunk elements each): 8 when they split evenly
// into at least two per warp or are many enough (>= 64) that an uneven split costs under an eighth; else
// the largest of {4, 2} that splits them evenly into at least two per warp; else 1 (whole rows, as in
// gemv_kernel).
static int gemv_ks_slices(int nch) {
    if ((nch % 8 == 0 && nch >= 16) || nch >= 64) return 8;
    for (int ks = 4; ks >= 2; ks >>= 1)
        if (nch % ks == 0 && nch / ks >= 2) return ks;
    return 1;
}

// Rows per pass of the K-split kernel: the accumulators within the register budget of two CTAs per SM
// (the FP8 kernels at three CTAs per SM take the same rows with half the loads per pass).
template <int MR, int EPI>
constexpr int gemv_ks_rows() {
    return (EPI == EPI_GLU ? 4 : 8) / (MR >= 8 ? 4 : (MR >= 4 ? 2 : 1));
}

// Columns per CTA of the K-split kernel: one balanced wave of cps CTAs per SM, whole passes.
static void gemv_ks_split(int N, int num_sms, int cps, int R, int* rpc, int* ctas) {
    const long slots = (long)num_sms * cps;
    int r = (int)((N + slots - 1) / slots);
    r = (r + R - 1) / R * R;
    *rpc = r;
    *ctas = (N + r - 1) / r;
}

// Rows per warp and CTAs along N for one balanced wave of cps CTAs per SM.  A grouped GEMV keeps every pass
// of R rows inside one activation group.
static void gemv_split(int N, int num_sms, int cps, int group, int* rows_per_warp, int* ctas, int* R) {
    const long warps = (long)num_sms * cps * kGemvWarps;
    int rpw = (int)((N + warps - 1) / warps);
    if (rpw < 1) rpw = 1;
    *R = rpw < 4 ? rpw : 4;                              // the loads of a batch spread over R rows
    if (group && *R > 1) {                               // passes must not straddle a group
        *R = 4;
        int r = (rpw + 3) / 4 * 4;
        while (r <= group && group % r) r += 4;
        if (r <= group && group % r == 0) rpw = r;
        else *R = 1;                                     // one-row passes never straddle
    }
    *rows_per_warp = rpw;
    *ctas = (N + kGemvWarps * rpw - 1) / (kGemvWarps * rpw);
}

template <typename TA, typename TW, int MR, int EPI>
static cudaError_t launch_r(const GemvArgs& g, int R, int rpw, int ctas, cudaStream_t st) {
    dim3 grid((g.M + MR - 1) / MR, ctas);
    dim3 block(kGemvWarps * 32);
    switch (R) {
        case 1: return launch_pdl(gemv_kernel<TA, TW, MR, EPI, 1>, grid, block, 0, st, g, rpw);
        case 2: return launch_pdl(gemv_kernel<TA, TW, MR, EPI, 2>, grid, block, 0, st, g, rpw);
        case 3: return launch_pdl(gemv_kernel<TA, TW, MR, EPI, 3>, grid, block, 0, st, g, rpw);
        default: return launch_pdl(gemv_kernel<TA, TW, MR, EPI, 4>, grid, block, 0, st, g, rpw);
    }
}

template <typename TA, typename TW, int MR, int EPI>
static cudaError_t launch_ks(GemvArgs& g, int KS, int num_sms, cudaStream_t st) {
    constexpr int R = gemv_ks_rows<MR, EPI>();
    int rpc, ctas;
    gemv_ks_split(g.N, num_sms, gemv_cps<TW, EPI>(), R, &rpc, &ctas);
    if (EPI == EPI_ARGMAX) g.npart = ctas;
    dim3 grid((g.M + MR - 1) / MR, ctas);
    return launch_pdl(gemv_ks_kernel<TA, TW, MR, EPI, R>, grid, dim3(kGemvWarps * 32), 0, st, g, rpc, KS);
}

template <typename TA, typename TW, int EPI>
static cudaError_t launch_mr(GemvArgs& g, int num_sms, cudaStream_t st) {
    const int MR = g.M >= 5 ? 8 : (g.M >= 3 ? 4 : (g.M == 2 ? 2 : 1));
    // The K-split kernel wins where the whole-row kernel has few rows per warp (long rows: fc, q_a | kv_a,
    // o_proj, down); with four or more rows per pass the whole-row kernel already reuses each activation
    // load and streams slightly faster (gate | up, lm_head, q_b on a GB300).
    const int KS = gemv_ks_slices((g.K + kChunk<TW> - 1) / kChunk<TW>);
    int rpw, ctas, R;
    gemv_split(g.N, num_sms, gemv_cps<TW, EPI>(), g.a_grp, &rpw, &ctas, &R);
    if constexpr (!kIsFp4<TW>) {
        if (sizeof(TW) <= 2 && KS > 1 && rpw <= 4 && !g.w_grp && !g.a_grp) {
            switch (MR) {
                case 1: return launch_ks<TA, TW, 1, EPI>(g, KS, num_sms, st);
                case 2: return launch_ks<TA, TW, 2, EPI>(g, KS, num_sms, st);
                case 4: return launch_ks<TA, TW, 4, EPI>(g, KS, num_sms, st);
                default: return launch_ks<TA, TW, 8, EPI>(g, KS, num_sms, st);
            }
        }
    }
    if (EPI == EPI_ARGMAX) g.npart = ctas;
    switch (MR) {
        case 1: return launch_r<TA, TW, 1, EPI>(g, R, rpw, ctas, st);
        case 2: return launch_r<TA, TW, 2, EPI>(g, R, rpw, ctas, st);
        case 4: return launch_r<TA, TW, 4, EPI>(g, R, rpw, ctas, st);
        default: return launch_r<TA, TW, 8, EPI>(g, R, rpw, ctas, st);
    }
}

template <typename TA, typename TW>
static cudaError_t launch_epi(GemvArgs& g, int epi, int num_sms, cudaStream_t st) {
    switch (epi) {
        case EPI_STORE: return launch_mr<TA, TW, EPI_STORE>(g, num_sms, st);
        case EPI_RESID: return launch_mr<TA, TW, EPI_RESID>(g, num_sms, st);
        case EPI_GLU: return launch_mr<TA, TW, EPI_GLU>(g, num_sms, st);
        default: return launch_mr<TA, TW, EPI_ARGMAX>(g, num_sms, st);
    }
}

}  // namespace e3
