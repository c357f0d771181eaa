// Shared device helpers of the EAGLE-3 draft-head kernels (sm_103a).
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <utility>

namespace e3 {

typedef __nv_bfloat16 bf16;

constexpr int kWarp = 32;

// --------------------------------------------------------------------------------------------
// scalar conversions
__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(bf16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float x) { return __float2bfloat16_rn(x); }

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// --------------------------------------------------------------------------------------------
// 16-byte loads.  `stream` loads bypass L1 allocation: weights are touched once per call.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}
__device__ __forceinline__ uint4 ld_cached16(const void* p) {
    return __ldg(reinterpret_cast<const uint4*>(p));
}

// Eight consecutive elements widened to fp32.
struct F8 { float v[8]; };

__device__ __forceinline__ void unpack_bf16x8(const uint4& u, float* v) {
    v[0] = bf_lo(u.x); v[1] = bf_hi(u.x); v[2] = bf_lo(u.y); v[3] = bf_hi(u.y);
    v[4] = bf_lo(u.z); v[5] = bf_hi(u.z); v[6] = bf_lo(u.w); v[7] = bf_hi(u.w);
}
__device__ __forceinline__ void unpack_f32x4(const uint4& u, float* v) {
    v[0] = __uint_as_float(u.x); v[1] = __uint_as_float(u.y);
    v[2] = __uint_as_float(u.z); v[3] = __uint_as_float(u.w);
}

template <typename T> struct Raw8;                     // raw storage of 8 elements
template <> struct Raw8<bf16> { uint4 a; };
template <> struct Raw8<float> { uint4 a, b; };

template <bool kStream, typename T> __device__ __forceinline__ Raw8<T> ld8(const T* p);
template <> __device__ __forceinline__ Raw8<bf16> ld8<true, bf16>(const bf16* p) { return {ld_stream16(p)}; }
template <> __device__ __forceinline__ Raw8<bf16> ld8<false, bf16>(const bf16* p) { return {ld_cached16(p)}; }
template <> __device__ __forceinline__ Raw8<float> ld8<true, float>(const float* p) {
    return {ld_stream16(p), ld_stream16(p + 4)};
}
template <> __device__ __forceinline__ Raw8<float> ld8<false, float>(const float* p) {
    return {ld_cached16(p), ld_cached16(p + 4)};
}
__device__ __forceinline__ void widen(const Raw8<bf16>& r, float* v) { unpack_bf16x8(r.a, v); }
__device__ __forceinline__ void widen(const Raw8<float>& r, float* v) {
    unpack_f32x4(r.a, v); unpack_f32x4(r.b, v + 4);
}
__device__ __forceinline__ Raw8<bf16> zero8(bf16*) { return {make_uint4(0, 0, 0, 0)}; }
__device__ __forceinline__ Raw8<float> zero8(float*) { return {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)}; }

// One FP8 E4M3 code (OCP 8-bit floating point: sign, 4 exponent bits with bias 7, 3 mantissa bits).
struct fp8e4 { uint8_t v; };
template <> struct Raw8<fp8e4> { uint2 a; };
template <> __device__ __forceinline__ Raw8<fp8e4> ld8<true, fp8e4>(const fp8e4* p) {
    uint2 r;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
    return {r};
}
template <> __device__ __forceinline__ Raw8<fp8e4> ld8<false, fp8e4>(const fp8e4* p) {
    return {__ldg(reinterpret_cast<const uint2*>(p))};
}
// Four E4M3 codes (byte i = element i) to fp32.  Every E4M3 value is exact in fp16 (and so in fp32):
// the hardware conversion e4m3x2 -> f16x2 puts the low byte in the low half.
__device__ __forceinline__ void e4m3x4_to_f32(uint32_t w, float* v) {
    uint32_t h01, h23;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, lo;\n\tcvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
        : "=r"(h01), "=r"(h23) : "r"(w));
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&h01));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&h23));
    v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
}
__device__ __forceinline__ void widen(const Raw8<fp8e4>& r, float* v) {
    e4m3x4_to_f32(r.a.x, v); e4m3x4_to_f32(r.a.y, v + 4);
}
__device__ __forceinline__ Raw8<fp8e4> zero8(fp8e4*) { return {make_uint2(0, 0)}; }
// One byte holding two E2M1 codes (OCP FP4: sign, 2 exponent bits with bias 1, 1 mantissa bit): the
// element at the even index in the low nibble.
struct fp4x2 { uint8_t v; };
// Sixteen E4M3 codes, or 32 E2M1 codes: one 16-byte load, the streaming unit of the FP8 / NVFP4 kernels.
struct Raw16e4 { uint4 a; };
// Sixteen E2M1 codes (8 bytes) to fp32; every E2M1 value is exact in fp16.
__device__ __forceinline__ void e2m1x16_to_f32(uint32_t w0, uint32_t w1, float* v) {
    const uint32_t w[2] = {w0, w1};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        uint32_t h[4];
        asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
            "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
            "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
            : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3]) : "r"(w[i]));
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[k]));
            v[8 * i + 2 * k] = f.x;
            v[8 * i + 2 * k + 1] = f.y;
        }
    }
}
// The E4M3 code in the low byte of b, as fp32.
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
    uint32_t h;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}" : "=r"(h) : "r"(b & 0xFFu));
    return __half2float(__ushort_as_half((unsigned short)(h & 0xFFFFu)));
}
__device__ __forceinline__ void widen(const Raw16e4& r, float* v) {
    e4m3x4_to_f32(r.a.x, v); e4m3x4_to_f32(r.a.y, v + 4); e4m3x4_to_f32(r.a.z, v + 8); e4m3x4_to_f32(r.a.w, v + 12);
}

// --------------------------------------------------------------------------------------------
// reductions
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
// Block-wide sum; `scratch` holds >= 32 floats.  All threads receive the result.
__device__ __forceinline__ float block_sum(float v, float* scratch) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    v = warp_sum(v);
    __syncthreads();
    if (lane == 0) scratch[w] = v;
    __syncthreads();
    float t = (lane < nw) ? scratch[lane] : 0.f;
    return warp_sum(t);
}

// (value, index) maximum with the lowest index winning ties; NaN never wins.
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
    return v > bv || (v == bv && i < bi);
}

__device__ __forceinline__ void set_err(int* err, int bit) { atomicOr(err, bit); }

__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ float silu(float x) { return x / (1.f + __expf(-x)); }

// Programmatic dependent launch.  Every kernel is launched so that the next one on the stream may be
// scheduled once all of this kernel's CTAs have started (pdl_trigger at their start); each kernel
// calls pdl_wait before it touches anything the previous kernels wrote, and may only read constant
// inputs (weights, tables) before that.  Both are no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

}  // namespace e3

// Host-side launch with programmatic stream serialization (see pdl_wait / pdl_trigger).
template <typename... KArgs, typename... Args>
static inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                     Args&&... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}
