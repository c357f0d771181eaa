// Weight-streaming GEMM for few activation rows (decode and small extends).
//
// y[m, n] = sum_k A[m, k] W[n, k] — the bias-free linear layers of the draft head (fc, q_a | kv_a,
// q_b, o_proj, gate | up, down, lm_head; "Eagle3 DeepseekV3 in MAX" §4).  At a handful of
// rows the layer is bound by streaming W from HBM once, so each warp owns one W row, streams
// it with 16-byte non-allocating loads (kUnroll loads in flight per lane), and multiplies it
// against up to MR activation rows that stay L1/L2 resident.  Fused epilogues: residual add,
// SiLU(gate) * up, and a row argmax with the lowest index winning ties (no logits round trip).
#include <float.h>
#include <limits.h>

#include "common.cuh"
#include "kernels.h"

namespace e3 {

constexpr int kGemvWarps = 8;

template <typename TW> struct GemvUnroll { static constexpr int v = 8; };
template <> struct GemvUnroll<float> { static constexpr int v = 4; };

template <typename TA, typename TW, int MR, int EPI>
__global__ void __launch_bounds__(kGemvWarps * 32) gemv_kernel(const GemvArgs g) {
    constexpr int NW = (EPI == EPI_GLU) ? 2 : 1;   // weight rows read per output column
    constexpr int U = GemvUnroll<TW>::v;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int m0 = blockIdx.x * MR;
    const int mcount = min(MR, g.M - m0);
    const int K = g.K;

    float best_v[MR];
    int best_i[MR];
#pragma unroll
    for (int i = 0; i < MR; ++i) { best_v[i] = -FLT_MAX; best_i[i] = INT_MAX; }

    for (int n = blockIdx.y * kGemvWarps + warp; n < g.N; n += gridDim.y * kGemvWarps) {
        const TW* wrow[NW];
        if (EPI == EPI_GLU) {
            wrow[0] = reinterpret_cast<const TW*>(g.w[0]) + (long)n * K;
            if (NW > 1) wrow[NW - 1] = reinterpret_cast<const TW*>(g.w[1]) + (long)n * K;
        } else {
            const int seg = (g.nseg_w > 1 && n >= g.nw[0]) ? 1 : 0;
            const int nn = seg ? n - g.nw[0] : n;
            wrow[0] = reinterpret_cast<const TW*>(g.w[seg]) + (long)nn * K;
        }
        float acc[MR][NW];
#pragma unroll
        for (int i = 0; i < MR; ++i)
#pragma unroll
            for (int q = 0; q < NW; ++q) acc[i][q] = 0.f;

        int kbase = 0;
        for (int s = 0; s < g.na; ++s) {
            const TA* ap = reinterpret_cast<const TA*>(g.a[s]) + (long)m0 * g.lda[s];
            const long lda = g.lda[s];
            const int ks = g.ka[s];
            for (int k0 = lane * 8; k0 < ks; k0 += 32 * 8 * U) {
                Raw8<TW> wr[U][NW];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int k = k0 + u * 256;
#pragma unroll
                    for (int q = 0; q < NW; ++q)
                        wr[u][q] = (k < ks) ? ld8<true>(wrow[q] + kbase + k) : zero8((TW*)nullptr);
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int k = k0 + u * 256;
                    if (k < ks) {
                        float wv[NW][8];
#pragma unroll
                        for (int q = 0; q < NW; ++q) widen(wr[u][q], wv[q]);
#pragma unroll
                        for (int i = 0; i < MR; ++i) {
                            if (i < mcount) {
                                float av[8];
                                widen(ld8<false>(ap + i * lda + k), av);
#pragma unroll
                                for (int q = 0; q < NW; ++q)
#pragma unroll
                                    for (int e = 0; e < 8; ++e) acc[i][q] = fmaf(wv[q][e], av[e], acc[i][q]);
                            }
                        }
                    }
                }
            }
            kbase += ks;
        }
#pragma unroll
        for (int i = 0; i < MR; ++i)
#pragma unroll
            for (int q = 0; q < NW; ++q) acc[i][q] = warp_sum(acc[i][q]);

#pragma unroll
        for (int i = 0; i < MR; ++i) {
            if (i >= mcount) continue;
            const long m = m0 + i;
            if (EPI == EPI_ARGMAX) {
                const float v = acc[i][0];
                if (better(v, n, best_v[i], best_i[i])) { best_v[i] = v; best_i[i] = n; }
                if (g.logits != nullptr && lane == i % 32) g.logits[m * g.ldl + n] = v;
            } else if (lane == i % 32) {
                float v;
                if (EPI == EPI_GLU) v = silu(acc[i][0]) * acc[i][NW - 1];
                else if (EPI == EPI_RESID) v = acc[i][0] + g.resid[m * g.ldr + n];
                else v = acc[i][0];
                g.y[m * g.ldy + n] = v;
            }
        }
    }

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

int gemv_argmax_parts(int N, int num_sms) {
    const int groups = (N + kGemvWarps - 1) / kGemvWarps;
    return groups < 2 * num_sms ? groups : 2 * num_sms;
}

template <typename TA, typename TW, int EPI>
static cudaError_t launch_mr(GemvArgs& g, int num_sms, cudaStream_t st) {
    int MR = g.M >= 5 ? 8 : (g.M >= 3 ? 4 : (g.M == 2 ? 2 : 1));
    dim3 block(kGemvWarps * 32);
    int ncol = (g.N + kGemvWarps - 1) / kGemvWarps;
    if (EPI == EPI_ARGMAX) {
        ncol = gemv_argmax_parts(g.N, num_sms);
        g.npart = ncol;
    }
    dim3 grid((g.M + MR - 1) / MR, ncol);
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
