// FP8 E4M3 draft weights: the per-row quantizer (eagle3_quantize_e4m3) and the expansion of an FP8
// matrix to bf16 that the tensor-core GEMM reads when a call has more rows than the GEMV path serves.
//
// The drafter's post-training quantization to FP8 ("EAGLE head deep dive", deployment) stores each
// projection matrix as E4M3 codes with one fp32 scale per output row:
//   scale[n] = max_k |W[n, k]| / 448 (1 for an all-zero row), code[n, k] = E4M3(W[n, k] / scale[n]),
// with the quotient rounded to nearest (ties to the even code) and saturated at +-448 by the hardware
// conversion cvt.rn.satfinite.e4m3x2.f32, and the head then uses decode(code) * scale.
#include "common.cuh"
#include "eagle3.h"
#include "kernels.h"

namespace e3 {

constexpr int kQuantThreads = 256;

// One CTA per row: the row's absolute maximum, then the codes, two per conversion.
template <typename T>
__global__ void __launch_bounds__(kQuantThreads) quantize_e4m3_kernel(const T* __restrict__ w, int K,
                                                                       uint8_t* __restrict__ codes,
                                                                       float* __restrict__ scales) {
    __shared__ float red[kQuantThreads / kWarp];
    const long n = blockIdx.x;
    const T* row = w + n * K;
    float amax = 0.f;
    for (int k = threadIdx.x; k < K; k += kQuantThreads) amax = fmaxf(amax, fabsf(to_f(row[k])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int i = 1; i < kQuantThreads / kWarp; ++i) amax = fmaxf(amax, red[i]);
    const float scale = amax > 0.f ? amax / 448.f : 1.f;     // IEEE fp32 division
    if (threadIdx.x == 0) scales[n] = scale;
    uint8_t* out = codes + n * K;
    for (int k = 2 * threadIdx.x; k < K; k += 2 * kQuantThreads) {
        const float a = to_f(row[k]) / scale;
        const float b = k + 1 < K ? to_f(row[k + 1]) / scale : 0.f;
        uint16_t pair;
        // the first source operand lands in the upper byte: b, then a, puts element k in the low byte
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pair) : "f"(b), "f"(a));
        out[k] = (uint8_t)(pair & 0xFF);
        if (k + 1 < K) out[k + 1] = (uint8_t)(pair >> 8);
    }
}

// out[n, k] = bf16(decode(code[n, k]) * scale[n]) for rows [0, rows), K a multiple of 8: one thread per
// 8 codes (an 8-byte load, a 16-byte store), a grid-stride loop over one wave.
__global__ void __launch_bounds__(256) dequant_e4m3_kernel(const uint8_t* __restrict__ codes,
                                                           const float* __restrict__ scales, long rows, int K,
                                                           bf16* __restrict__ out) {
    const long chunks_per_row = K / 8, total = rows * chunks_per_row;
    for (long c = (long)blockIdx.x * blockDim.x + threadIdx.x; c < total; c += (long)gridDim.x * blockDim.x) {
        const long n = c / chunks_per_row;
        const Raw8<fp8e4> r = ld8<true>(reinterpret_cast<const fp8e4*>(codes) + c * 8);
        float v[8];
        widen(r, v);
        const float s = __ldg(scales + n);
        uint32_t p[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i] * s, v[2 * i + 1] * s);
            p[i] = *reinterpret_cast<const uint32_t*>(&h);
        }
        *reinterpret_cast<uint4*>(out + c * 8) = make_uint4(p[0], p[1], p[2], p[3]);
    }
}

cudaError_t launch_dequant_e4m3(const uint8_t* codes, const float* scales, long rows, int K, bf16* out,
                                int num_sms, cudaStream_t st) {
    if (rows <= 0) return cudaSuccess;
    if (K % 8) return cudaErrorInvalidValue;
    const long chunks = rows * (K / 8);
    long ctas = (chunks + 255) / 256;
    if (ctas > 8L * num_sms) ctas = 8L * num_sms;
    dequant_e4m3_kernel<<<(int)ctas, 256, 0, st>>>(codes, scales, rows, K, out);
    return cudaGetLastError();
}

// ----------------------------------------------------------------------------------------------- NVFP4
// NVFP4 ("EAGLE head deep dive", deployment: the drafter quantized to NVFP4): E2M1 codes, one E4M3 scale per
// 16 consecutive weights of a row, one fp32 scale per matrix, in the order the quantizer forms them:
//   g = max|W| / 2688 (448 * 6; 1 for a zero matrix), s_b = E4M3(max_b |W| / (6 g)),
//   e_b = decode(s_b) g, code = E2M1(W / e_b) (0 where e_b == 0).

// The matrix's absolute maximum as fp32 bits (non-negative floats order as their bit patterns), by an
// atomic maximum into *amax_bits (zeroed by the caller).
template <typename T>
__global__ void __launch_bounds__(256) absmax_kernel(const T* __restrict__ w, long n, unsigned* amax_bits) {
    float m = 0.f;
    for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x)
        m = fmaxf(m, fabsf(to_f(w[i])));
    m = warp_max(m);
    if ((threadIdx.x & 31) == 0) atomicMax(amax_bits, __float_as_uint(m));
}

__device__ __forceinline__ float nvfp4_global(unsigned amax_bits) {
    const float amax = __uint_as_float(amax_bits);
    return amax > 0.f ? amax / 2688.f : 1.f;
}

// One CTA per row, one thread per 16-weight block (looping): the block scale, then 16 codes as 8 bytes.
template <typename T>
__global__ void __launch_bounds__(kQuantThreads) quantize_nvfp4_kernel(const T* __restrict__ w, int K,
                                                                        const unsigned* amax_bits,
                                                                        uint8_t* __restrict__ codes,
                                                                        uint8_t* __restrict__ bscales) {
    const long n = blockIdx.x;
    const float g = nvfp4_global(*amax_bits);
    const float six_g = 6.f * g;
    const T* row = w + n * K;
    for (int b = threadIdx.x; b < K / 16; b += kQuantThreads) {
        float x[16], bmax = 0.f;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            x[e] = to_f(row[16 * b + e]);
            bmax = fmaxf(bmax, fabsf(x[e]));
        }
        const float q = bmax / six_g;
        uint16_t sp;
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(sp) : "f"(0.f), "f"(q));
        const uint8_t sb = (uint8_t)(sp & 0xFF);
        bscales[n * (K / 16) + b] = sb;
        const float eff = e4m3_to_f32(sb) * g;
        uint32_t packed[2] = {0u, 0u};
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
            const float a = eff > 0.f ? x[e] / eff : 0.f;
            const float c = eff > 0.f ? x[e + 1] / eff : 0.f;
            uint32_t byte;
            // the first source lands in the upper nibble: element e + 1 high, element e low
            asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
                : "=r"(byte) : "f"(c), "f"(a));
            packed[e / 8] |= (byte & 0xFFu) << (8 * ((e % 8) / 2));
        }
        *reinterpret_cast<uint2*>(codes + n * (K / 2) + 8 * b) = make_uint2(packed[0], packed[1]);
    }
}

__global__ void nvfp4_finish_kernel(unsigned* slot) {
    *slot = __float_as_uint(nvfp4_global(*slot));   // the matrix maximum becomes the matrix scale
}

// out[n, k] = bf16(decode(code) * decode(s_b) * g) for rows [0, rows), K a multiple of 32: one thread per
// 16 codes (an 8-byte load, two 16-byte stores), a grid-stride loop over one wave.
__global__ void __launch_bounds__(256) dequant_nvfp4_kernel(const uint8_t* __restrict__ codes,
                                                            const uint8_t* __restrict__ bscales,
                                                            const float* __restrict__ global, long rows, int K,
                                                            bf16* __restrict__ out) {
    const float g = __ldg(global);
    const long blocks = rows * (K / 16);
    for (long b = (long)blockIdx.x * blockDim.x + threadIdx.x; b < blocks; b += (long)gridDim.x * blockDim.x) {
        const uint2 c = __ldg(reinterpret_cast<const uint2*>(codes + 8 * b));
        const float s = e4m3_to_f32(__ldg(bscales + b)) * g;
        float v[16];
        e2m1x16_to_f32(c.x, c.y, v);
        uint32_t p[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i] * s, v[2 * i + 1] * s);
            p[i] = *reinterpret_cast<const uint32_t*>(&h);
        }
        uint4* o = reinterpret_cast<uint4*>(out + 16 * b);
        o[0] = make_uint4(p[0], p[1], p[2], p[3]);
        o[1] = make_uint4(p[4], p[5], p[6], p[7]);
    }
}

cudaError_t launch_dequant_nvfp4(const uint8_t* codes, const uint8_t* block_scales, const float* global, long rows,
                                 int K, bf16* out, int num_sms, cudaStream_t st) {
    if (rows <= 0) return cudaSuccess;
    if (K % 32) return cudaErrorInvalidValue;
    const long blocks = rows * (K / 16);
    long ctas = (blocks + 255) / 256;
    if (ctas > 8L * num_sms) ctas = 8L * num_sms;
    dequant_nvfp4_kernel<<<(int)ctas, 256, 0, st>>>(codes, block_scales, global, rows, K, out);
    return cudaGetLastError();
}

}  // namespace e3

extern "C" eagle3_status_t eagle3_quantize_nvfp4(const void* w, eagle3_dtype_t dtype, int32_t N, int32_t K,
                                                 uint8_t* codes, uint8_t* block_scales, float* global_scale,
                                                 void* stream) {
    using namespace e3;
    if (!w || !codes || !block_scales || !global_scale || N < 1 || K < 1) return EAGLE3_ERR_INVALID_ARG;
    if (K % 32) return EAGLE3_ERR_UNSUPPORTED;
    if (dtype != EAGLE3_BF16 && dtype != EAGLE3_F32) return EAGLE3_ERR_UNSUPPORTED;
    const cudaStream_t st = (cudaStream_t)stream;
    unsigned* slot = reinterpret_cast<unsigned*>(global_scale);
    if (cudaMemsetAsync(slot, 0, sizeof(unsigned), st) != cudaSuccess) return EAGLE3_ERR_CUDA;
    const long n = (long)N * K;
    const int ctas = (int)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
    if (dtype == EAGLE3_BF16) {
        absmax_kernel<bf16><<<ctas, 256, 0, st>>>(static_cast<const bf16*>(w), n, slot);
        quantize_nvfp4_kernel<bf16><<<N, kQuantThreads, 0, st>>>(static_cast<const bf16*>(w), K, slot, codes,
                                                                 block_scales);
    } else {
        absmax_kernel<float><<<ctas, 256, 0, st>>>(static_cast<const float*>(w), n, slot);
        quantize_nvfp4_kernel<float><<<N, kQuantThreads, 0, st>>>(static_cast<const float*>(w), K, slot, codes,
                                                                  block_scales);
    }
    nvfp4_finish_kernel<<<1, 1, 0, st>>>(slot);
    return cudaGetLastError() == cudaSuccess ? EAGLE3_OK : EAGLE3_ERR_CUDA;
}

extern "C" eagle3_status_t eagle3_quantize_e4m3(const void* w, eagle3_dtype_t dtype, int32_t N, int32_t K,
                                                uint8_t* codes, float* scales, void* stream) {
    using namespace e3;
    if (!w || !codes || !scales || N < 1 || K < 1) return EAGLE3_ERR_INVALID_ARG;
    const cudaStream_t st = (cudaStream_t)stream;
    if (dtype == EAGLE3_BF16)
        quantize_e4m3_kernel<bf16><<<N, kQuantThreads, 0, st>>>(static_cast<const bf16*>(w), K, codes, scales);
    else if (dtype == EAGLE3_F32)
        quantize_e4m3_kernel<float><<<N, kQuantThreads, 0, st>>>(static_cast<const float*>(w), K, codes, scales);
    else
        return EAGLE3_ERR_UNSUPPORTED;
    return cudaGetLastError() == cudaSuccess ? EAGLE3_OK : EAGLE3_ERR_CUDA;
}
