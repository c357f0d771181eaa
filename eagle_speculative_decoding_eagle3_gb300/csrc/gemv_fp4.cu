// Weight-streaming GEMM for few activation rows: the NVFP4 weight instantiations (E2M1 codes, E4M3 scales
// per 16 weights, one fp32 scale per matrix; the kernels and their launch logic are in gemv.cuh).
#include "gemv.cuh"

namespace e3 {

cudaError_t launch_gemv_fp4(GemvArgs& g, int epi, int num_sms, cudaStream_t st) {
    if (g.M <= 0 || g.N <= 0) return cudaSuccess;
    if (g.w_type != FP4 || !g.wscale[0] || !g.wbs[0] || ((g.nseg_w > 1 || epi == EPI_GLU) && (!g.wscale[1] || !g.wbs[1])) ||
        g.w_grp || g.a_grp)
        return cudaErrorInvalidValue;
    // lanes load 32 codes at a time: K and the activation segments are whole 32-element units
    if (g.K % 32) return cudaErrorInvalidValue;
    for (int s = 0; s < g.na; ++s)
        if (g.ka[s] % 32) return cudaErrorInvalidValue;
    for (int s = g.na; s < 3; ++s) g.ka[s] = 1 << 30;   // unused K segments never match
    if (g.a_type == F32) return launch_epi<float, fp4x2>(g, epi, num_sms, st);
    if (epi != EPI_STORE) return cudaErrorInvalidValue;
    return launch_mr<bf16, fp4x2, EPI_STORE>(g, num_sms, st);
}

}  // namespace e3
