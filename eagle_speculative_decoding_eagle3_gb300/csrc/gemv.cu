// Weight-streaming GEMM for few activation rows (decode and small extends).
//
// y[m, n] = sum_k A[m, k] W[n, k] — the bias-free linear layers of the draft head (fc, q_a | kv_a,
// q_b, o_proj, gate | up, down, lm_head; "Eagle3 DeepseekV3 in MAX" §4).  At a handful of rows a
// layer is bound by streaming W from HBM once, so each warp owns NR weight rows (two rows per
// output column for the gated MLP), streams them with 16-byte non-allocating loads (U loads per row
// in flight per lane), and multiplies them against up to MR activation rows that stay L1/L2
// resident.  Fused epilogues: residual add, SiLU(gate) * up, and a row argmax with the lowest index
// winning ties (the logits never round-trip through HBM unless a debug buffer asks for them).
#include <float.h>
#include <limits.h>

#include "common.cuh"
#include "kernels.h"

namespace e3 {

constexpr int kGemvWarps = 8;

template <typename TW, int MR> struct GemvUnroll { static constexpr int v = MR <= 2 ? 8 : 4; };
template <int MR> struct GemvUnroll<float, MR> { static constexpr int v = MR <= 2 ? 4 : 2; };

template <int EPI> struct RowsPerWarp { static constexpr int v = 2; };
template <> struct RowsPerWarp<EPI_GLU> { static constexpr int v = 1; };

template <typename TA, typename TW, int MR, int EPI>
__global__ void __launch_bounds__(kGemvWarps * 32) gemv_kernel(const GemvArgs g) {
    constexpr int NW = (EPI == EPI_GLU) ? 2 : 1;   // weight rows read per output column
    constexpr int NR = RowsPerWarp<EPI>::v;       // output columns per warp
    constexpr int U = GemvUnroll<TW, MR>::v;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int m0 = blockIdx.x * MR;
    const int mcount = min(MR, g.M - m0);
    const int K = g.K;
    const int n0 = (blockIdx.y * kGemvWarps + warp) * NR;

    const TW* wrow[NR][NW];
#pragma unroll
    for (int j = 0; j < NR; ++j) {
        const int n = min(n0 + j, g.N - 1);
        if (EPI == EPI_GLU) {
            wrow[j][0] = reinterpret_cast<const TW*>(g.w[0]) + (long)n * K;
            wrow[j][NW - 1] = reinterpret_cast<const TW*>(g.w[1]) + (long)n * K;
        } else {
            const int seg = (g.nseg_w > 1 && n >= g.nw[0]) ? 1 : 0;
            const int nn = seg ? n - g.nw[0] : n;
            wrow[j][0] = reinterpret_cast<const TW*>(g.w[seg]) + (long)nn * K;
        }
    }
    float acc[MR][NR][NW];
#pragma unroll
    for (int i = 0; i < MR; ++i)
#pragma unroll
        for (int j = 0; j < NR; ++j)
#pragma unroll
            for (int q = 0; q < NW; ++q) acc[i][j][q] = 0.f;

    if (n0 < g.N) {
        int kbase = 0;
        for (int s = 0; s < g.na; ++s) {
            const TA* ap = reinterpret_cast<const TA*>(g.a[s]) + (long)m0 * g.lda[s];
            const long lda = g.lda[s];
            const int ks = g.ka[s];
            for (int k0 = lane * 8; k0 < ks; k0 += 32 * 8 * U) {
                Raw8<TW> wr[U][NR][NW];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int k = k0 + u * 256;
#pragma unroll
                    for (int j = 0; j < NR; ++j)
#pragma unroll
                        for (int q = 0; q < NW; ++q)
                            wr[u][j][q] = (k < ks) ? ld8<true>(wrow[j][q] + kbase + k) : zero8((TW*)nullptr);
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int k = k0 + u * 256;
                    if (k < ks) {
                        float wv[NR][NW][8];
#pragma unroll
                        for (int j = 0; j < NR; ++j)
#pragma unroll
                            for (int q = 0; q < NW; ++q) widen(wr[u][j][q], wv[j][q]);
#pragma unroll
                        for (int i = 0; i < MR; ++i) {
                            if (i < mcount) {
                                float av[8];
                                widen(ld8<false>(ap + i * lda + k), av);
#pragma unroll
                                for (int j = 0; j < NR; ++j)
#pragma unroll
                                    for (int q = 0; q < NW; ++q)
#pragma unroll
                                        for (int e = 0; e < 8; ++e)
                                            acc[i][j][q] = fmaf(wv[j][q][e], av[e], acc[i][j][q]);
                            }
                        }
                    }
                }
            }
            kbase += ks;
        }
    }
#pragma unroll
    for (int i = 0; i < MR; ++i)
#pragma unroll
        for (int j = 0; j < NR; ++j)
#pragma unroll
            for (int q = 0; q < NW; ++q) acc[i][j][q] = warp_sum(acc[i][j][q]);

    if (EPI == EPI_ARGMAX) {
        __shared__ float sv[kGemvWarps][MR];
        __shared__ int si[kGemvWarps][MR];
#pragma unroll
        for (int i = 0; i < MR; ++i) {
            float bv = -FLT_MAX;
            int bi = INT_MAX;
#pragma unroll
            for (int j = 0; j < NR; ++j) {
                const int n = n0 + j;
                if (n < g.N && i < mcount) {
                    if (better(acc[i][j][0], n, bv, bi)) { bv = acc[i][j][0]; bi = n; }
                    if (g.logits != nullptr && lane == (i * NR + j) % 32)
                        g.logits[(long)(m0 + i) * g.ldl + n] = acc[i][j][0];
                }
            }
            if (lane == 0) { sv[warp][i] = bv; si[warp][i] = bi; }
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
        return;
    }
#pragma unroll
    for (int i = 0; i < MR; ++i) {
#pragma unroll
        for (int j = 0; j < NR; ++j) {
            const int n = n0 + j;
            if (i >= mcount || n >= g.N || lane != (i * NR + j) % 32) continue;
            const long m = m0 + i;
            float v;
            if (EPI == EPI_GLU) v = silu(acc[i][j][0]) * acc[i][j][NW - 1];
            else if (EPI == EPI_RESID) v = acc[i][j][0] + g.resid[m * g.ldr + n];
            else v = acc[i][j][0];
            g.y[m * g.ldy + n] = v;
        }
    }
}

int gemv_argmax_parts(int N, int num_sms) {
    (void)num_sms;
    const int per_cta = kGemvWarps * RowsPerWarp<EPI_ARGMAX>::v;
    return (N + per_cta - 1) / per_cta;
}

template <typename TA, typename TW, int EPI>
static cudaError_t launch_mr(GemvArgs& g, int num_sms, cudaStream_t st) {
    const int MR = g.M >= 5 ? 8 : (g.M >= 3 ? 4 : (g.M == 2 ? 2 : 1));
    const int per_cta = kGemvWarps * RowsPerWarp<EPI>::v;
    const int ncol = (g.N + per_cta - 1) / per_cta;
    if (EPI == EPI_ARGMAX) g.npart = gemv_argmax_parts(g.N, num_sms);
    dim3 grid((g.M + MR - 1) / MR, ncol);
    dim3 block(kGemvWarps * 32);
    switch (MR) {
        case 1: gemv_kernel<TA, TW, 1, EPI><<<grid, block, 0, st>>>(g); break;
        case 2: gemv_kernel<TA, TW, 2, EPI><<<grid, block, 0, st>>>(g); break;
        case 4: gemv_kernel<TA, TW, 4, EPI><<<grid, block, 0, st>>>(g); break;
        default: gemv_kernel<TA, TW, 8, EPI><<<grid, block, 0, st>>>(g); break;
    }
    return cudaGetLastError();
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
    if (g.w_type == F32) {
        if (g.a_type != F32) return cudaErrorInvalidValue;
        return launch_epi<float, float>(g, epi, num_sms, st);
    }
    if (g.a_type == F32) return launch_epi<float, bf16>(g, epi, num_sms, st);
    if (epi != EPI_STORE) return cudaErrorInvalidValue;
    return launch_mr<bf16, bf16, EPI_STORE>(g, num_sms, st);
}

}  // namespace e3
