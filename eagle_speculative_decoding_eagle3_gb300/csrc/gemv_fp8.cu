// Weight-streaming GEMM for few activation rows: the FP8 E4M3 weight instantiations (per-row scales;
// the kernels and their launch logic are in gemv.cuh).
#include "gemv.cuh"

namespace e3 {

cudaError_t launch_gemv_fp8(GemvArgs& g, int epi, int num_sms, cudaStream_t st) {
    if (g.M <= 0 || g.N <= 0) return cudaSuccess;
    if (g.w_type != FP8 || !g.wscale[0] || (g.nseg_w > 1 && !g.wscale[1]) || (epi == EPI_GLU && !g.wscale[1]) ||
        g.w_grp || g.a_grp)
        return cudaErrorInvalidValue;
    // lanes load 16 codes at a time: K and the activation segments are whole 16-element units
    if (g.K % 16) return cudaErrorInvalidValue;
    for (int s = 0; s < g.na; ++s)
        if (g.ka[s] % 16) return cudaErrorInvalidValue;
    for (int s = g.na; s < 3; ++s) g.ka[s] = 1 << 30;   // unused K segments never match
    if (g.a_type == F32) return launch_epi<float, fp8e4>(g, epi, num_sms, st);
    if (epi != EPI_STORE) return cudaErrorInvalidValue;
    return launch_mr<bf16, fp8e4, EPI_STORE>(g, num_sms, st);
}

}  // namespace e3
