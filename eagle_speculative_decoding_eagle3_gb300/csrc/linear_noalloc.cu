// Allocation-free entry point of the linear-layer engine: eagle3_linear_noalloc.
//
// The same product as eagle3_linear, y = x W^T, always on the tcgen05 split-K GEMM.  Where
// eagle3_linear keeps the split-K partial sums in a handle's workspace, this entry point keeps them in
// a fixed array defined below at file scope in device memory, so it needs no handle and allocates
// nothing: the array is reserved when the library's CUDA module is loaded on a device and stays there
// until the process exits; each call only looks its address up (once per device) and launches kernels.
// It exists for callers that cannot allocate device memory on their call path (the declaration in
// eagle3.h says who they are and why).
#include <string.h>

#include <mutex>

#include "eagle3.h"
#include "kernels.h"

// Scratch layout: [0, 256) the device error word that the GEMM's bounded waits write (it must start at
// zero: every call clears it); [256, 256 + EAGLE3_NOALLOC_SCRATCH_BYTES) the fp32 split-K partials
// [splits][M][N] (every split writes every element of its plane, so they need no clearing).
// Host code must not pass `g_noalloc_scratch` itself to a kernel: on the host that name is only a
// stand-in for the device array; its device address comes from cudaGetSymbolAddress below.
static constexpr size_t kNoallocHeadBytes = 256;
static constexpr size_t kNoallocPartBytes = EAGLE3_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocHeadBytes + kNoallocPartBytes];

namespace {

constexpr int kMaxDevices = 64;
constexpr long kMaxElems = (long)(kNoallocPartBytes / (2 * sizeof(float)));   // two partial planes fit

struct DeviceSlot {
    unsigned char* scratch = nullptr;   // device address of g_noalloc_scratch on this device
    int num_sms = 0;
};
std::mutex g_slot_mutex;
DeviceSlot g_slots[kMaxDevices];

// Set-up, once per device, with that device current: the scratch array's device address and the SM
// count.  Later calls on the device reuse them.
cudaError_t device_slot(DeviceSlot* out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_slot_mutex);
    DeviceSlot& s = g_slots[dev];
    if (!s.scratch) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        if (!p || ((uintptr_t)p & 255u) || sms < 1) return cudaErrorInvalidDevicePointer;
        s.num_sms = sms;
        s.scratch = static_cast<unsigned char*>(p);
    }
    *out = s;
    return cudaSuccess;
}

// Split count: one when the (N-tile, M-tile) CTAs already cover every SM (the GEMM then writes y itself
// and the scratch is not touched); else enough split CTAs for two per SM, at least four K-blocks per
// split, and no more splits than the scratch holds (two always fit under the M * N limit).
int noalloc_splits(int num_sms, int M, int N, int K, int bn) {
    const long tiles = (long)((N + 127) / 128) * ((M + bn - 1) / bn);
    if (tiles >= num_sms) return 1;
    long s = (2L * num_sms + tiles - 1) / tiles;
    const long kmax = K / 64 / 4;
    if (s > kmax) s = kmax;
    while (s > 2 && s * (long)M * N * (long)sizeof(float) > (long)kNoallocPartBytes) --s;
    return s < 1 ? 1 : (int)s;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace

extern "C" eagle3_status_t eagle3_linear_noalloc(const void* x, const void* w, float* y, int32_t M, int32_t N,
                                                 int32_t K, void* stream) {
    using namespace e3;
    if (!x || !w || !y || M < 1 || N < 1 || K < 1) return EAGLE3_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w) || !aligned16(y)) return EAGLE3_ERR_INVALID_ARG;
    if (K % 64) return EAGLE3_ERR_UNSUPPORTED;
    if ((long)M * N > kMaxElems) return EAGLE3_ERR_SCRATCH_LIMIT;
    DeviceSlot slot;
    if (device_slot(&slot) != cudaSuccess) return EAGLE3_ERR_CUDA;
    const cudaStream_t st = (cudaStream_t)stream;
    int* err = reinterpret_cast<int*>(slot.scratch);
    float* part = reinterpret_cast<float*>(slot.scratch + kNoallocHeadBytes);
    if (cudaMemsetAsync(err, 0, sizeof(int), st) != cudaSuccess) return EAGLE3_ERR_CUDA;

    TcParams p;
    memset(&p, 0, sizeof(p));
    const int bn = tc_pick_bn(M);
    if (!make_tma_2d(&p.mw[0], w, N, K, K, 128)) return EAGLE3_ERR_INVALID_ARG;
    if (!make_tma_2d(&p.mx[0], x, M, K, K, bn)) return EAGLE3_ERR_INVALID_ARG;
    p.np0 = 1 << 30;
    p.N = N; p.M = M; p.K = K;
    p.kseg[0] = 1 << 30;
    p.kseg[1] = 1 << 30;
    p.epi = EPI_STORE;
    p.y = y; p.ldy = N;
    p.part = part;
    p.err = err;
    p.nbatch = 1;
    const int splits = noalloc_splits(slot.num_sms, M, N, K, bn);
    if (launch_tc_gemm(p, bn, splits, st) != cudaSuccess) return EAGLE3_ERR_CUDA;
    return EAGLE3_OK;
}
