// Weight-streaming GEMM for few activation rows (decode and small extends).
//
// y[m, n] = sum_k A[m, k] W[n, k] — the bias-free linear layers of the draft head (fc, q_a | kv_a,
// q_b, o_proj, gate | up, down, lm_head, the per-head value up-projection; "Eagle3 DeepseekV3 in MAX"
// §4).  At a handful of rows a layer is bound by streaming W from HBM once, so the kernel is laid out
// for HBM:
//  * one balanced wave: the grid holds kGemvCtasPerSm CTAs per SM and every warp owns an equal range of
//    weight rows (rows_per_warp), so no SM idles in a half-empty last wave;
//  * a warp streams R of its rows at once (R = 1 or 4), each with U 16-byte non-allocating loads per
//    lane (lane l reads elements [8l + 256c, +8) of a row), so about 16 loads of 16 B are in flight per
//    lane and ~128 KB per SM whatever the row length;
//  * the activation rows (up to MR) stay L1/L2 resident and are loaded once per chunk for all R rows;
//  * at the end of each pass the warp reduces its partial dot products and applies the fused epilogue:
//    store, residual add, SiLU(gate) * up (two weight rows per output), or a running row argmax with
//    the lowest index winning ties (the logits never round-trip through HBM unless a debug buffer asks
//    for them).
#include <float.h>
#include <limits.h>

#include "common.cuh"
#include "kernels.h"

namespace e3 {

constexpr int kGemvWarps = 8;
constexpr int kGemvCtasPerSm = 2;
constexpr int kLoadsInFlight = 16;     // 16-byte weight loads per lane per iteration

template <typename TA, typename TW, int MR, int EPI, int R>
__global__ void __launch_bounds__(kGemvWarps * 32, kGemvCtasPerSm) gemv_kernel(const GemvArgs g, int rows_per_warp) {
    constexpr int NW = (EPI == EPI_GLU) ? 2 : 1;   // weight rows read per output column
    constexpr int U0 = kLoadsInFlight / (R * NW) * 2 / (int)sizeof(TW);
    constexpr int U = U0 < 1 ? 1 : U0;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int m0 = blockIdx.x * MR;
    const int mcount = min(MR, g.M - m0);
    const int K = g.K;
    const int r_begin = (blockIdx.y * kGemvWarps + warp) * rows_per_warp;
    const int r_end = min(g.N, r_begin + rows_per_warp);
    const int ka0 = g.ka[0], ka01 = g.ka[0] + g.ka[1];

    auto wrow = [&](int n, int q) -> const TW* {
        if (EPI == EPI_GLU) return reinterpret_cast<const TW*>(g.w[q]) + (long)n * K;
        if (g.w_grp)
            return reinterpret_cast<const TW*>(g.w[0]) +
                   ((long)(n / g.w_grp) * g.w_grp_stride + g.w_row0 + n % g.w_grp) * K;
        const int seg = (g.nseg_w > 1 && n >= g.nw[0]) ? 1 : 0;
        return reinterpret_cast<const TW*>(g.w[seg]) + (long)(seg ? n - g.nw[0] : n) * K;
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
#pragma unroll
        for (int j = 0; j < R; ++j)
#pragma unroll
            for (int q = 0; q < NW; ++q) wp[j][q] = wrow(p0 + (j < nr ? j : 0), q);
        // the per-head GEMVs use one activation slice per row group; all rows of a pass share it
        const long aoff = g.a_grp ? (long)(p0 / g.a_grp) * g.a_grp_stride : 0;
        float acc[MR][R][NW];
#pragma unroll
        for (int i = 0; i < MR; ++i)
#pragma unroll
            for (int j = 0; j < R; ++j)
#pragma unroll
                for (int q = 0; q < NW; ++q) acc[i][j][q] = 0.f;

        for (int k0 = lane * 8; k0 < K; k0 += 256 * U) {
            Raw8<TW> wr[U][R][NW];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int k = k0 + u * 256;
#pragma unroll
                for (int j = 0; j < R; ++j)
#pragma unroll
                    for (int q = 0; q < NW; ++q)
                        wr[u][j][q] = (k < K && j < nr) ? ld8<true>(wp[j][q] + k) : zero8((TW*)nullptr);
            }
            if (!waited) { pdl_wait(); waited = true; }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int k = k0 + u * 256;
                if (k < K) {
                    const int s = (k >= ka0) + (k >= ka01);
                    const int kl = k - (s == 0 ? 0 : (s == 1 ? ka0 : ka01));
                    const TA* ap = reinterpret_cast<const TA*>(g.a[s]) + (long)m0 * g.lda[s] + aoff + kl;
#pragma unroll
                    for (int i = 0; i < MR; ++i) {
                        if (i < mcount) {
                            float av[8];
                            widen(ld8<false>(ap + i * g.lda[s]), av);
#pragma unroll
                            for (int j = 0; j < R; ++j)
#pragma unroll
                                for (int q = 0; q < NW; ++q) {
                                    float wv[8];
                                    widen(wr[u][j][q], wv);
#pragma unroll
                                    for (int e = 0; e < 8; ++e) acc[i][j][q] = fmaf(wv[e], av[e], acc[i][j][q]);
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
                for (int q = 0; q < NW; ++q) acc[i][j][q] = warp_sum(acc[i][j][q]);
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

// Rows per warp and CTAs along N for one balanced wave of kGemvCtasPerSm CTAs per SM.  A grouped GEMV
// keeps every pass of R rows inside one activation group.
static void gemv_split(int N, int num_sms, int group, int* rows_per_warp, int* ctas, int* R) {
    const long warps = (long)num_sms * kGemvCtasPerSm * kGemvWarps;
    int rpw = (int)((N + warps - 1) / warps);
    if (rpw < 1) rpw = 1;
    *R = rpw < 4 ? rpw : 4;                              // 16 / R loads per row keep 16 in flight
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

int gemv_argmax_parts(int N, int num_sms) {
    int rpw, ctas, R;
    gemv_split(N, num_sms, 0, &rpw, &ctas, &R);
    return ctas;
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

template <typename TA, typename TW, int EPI>
static cudaError_t launch_mr(GemvArgs& g, int num_sms, cudaStream_t st) {
    const int MR = g.M >= 5 ? 8 : (g.M >= 3 ? 4 : (g.M == 2 ? 2 : 1));
    int rpw, ctas, R;
    gemv_split(g.N, num_sms, g.a_grp, &rpw, &ctas, &R);
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

cudaError_t launch_gemv(GemvArgs& g, int epi, int num_sms, cudaStream_t st) {
    if (g.M <= 0 || g.N <= 0) return cudaSuccess;
    for (int s = g.na; s < 3; ++s) g.ka[s] = 1 << 30;   // unused K segments never match
    if (g.w_type == F32) {
        if (g.a_type != F32) return cudaErrorInvalidValue;
        return launch_epi<float, float>(g, epi, num_sms, st);
    }
    if (g.a_type == F32) return launch_epi<float, bf16>(g, epi, num_sms, st);
    if (epi != EPI_STORE) return cudaErrorInvalidValue;
    return launch_mr<bf16, bf16, EPI_STORE>(g, num_sms, st);
}

}  // namespace e3
