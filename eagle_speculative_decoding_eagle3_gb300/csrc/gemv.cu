// Weight-streaming GEMM for few activation rows: the fp32 and bf16 weight instantiations (the
// kernels and their launch logic are in gemv.cuh).
#include "gemv.cuh"

namespace e3 {

// Upper bound of the ARGMAX partials per row (one per CTA): both kernels run one wave of at most
// kGemvMaxCtasPerSm CTAs per SM.  The launch reports the count it used in GemvArgs::npart.
int gemv_argmax_parts(int N, int num_sms) {
    const long slots = (long)num_sms * kGemvMaxCtasPerSm;
    return (int)(N < slots ? N : slots);
}

cudaError_t launch_gemv(GemvArgs& g, int epi, int num_sms, cudaStream_t st) {
    if (g.w_type == FP8) return launch_gemv_fp8(g, epi, num_sms, st);
    if (g.w_type == FP4) return launch_gemv_fp4(g, epi, num_sms, st);
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
