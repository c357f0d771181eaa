// Sampled drafts and residual (rejection-sampling) acceptance.
//
// "Eagle3 DeepseekV3 in MAX" §3.1 and §10 name the sampling parameters of the drafts (temperature,
// top-k, top-p) and the rejection-sampling strategies (greedy, residual, ...), and §8 a seed counter
// that feeds the sampler.  The uniform random numbers are inputs (drawn by the caller, or on the device by
// philox_uniforms_kernel below), so every consumer of a draw sees the same number.
//
// sample_kernel: one thread-block cluster of kCluster CTAs per row; CTA g owns the logits of slice g of
// the row and keeps their order-preserving integer keys in shared memory.  x = logits / temperature; since
// the temperature is positive, x is ordered exactly as the logits are, so
//  * top_k keeps the top_k largest logits, lower indices first among equal values.  Each CTA finds the
//    top_k of its slice by a radix select on the 64-bit value (key, ~index), which is distinct for every
//    token and orders the tokens exactly as the rule does; CTA 0 gathers the cluster's candidates through
//    distributed shared memory and selects the top_k among them the same way.  The kept tokens are sorted
//    (logit descending, index ascending) by a bitonic sort; their softmax weights are
//    exp((l - l_max) / temperature) in fp32; top_p keeps the shortest prefix whose mass reaches top_p of
//    the kept mass; the kept weights are renormalised and u picks the token by inverse CDF in ascending
//    index order.
//  * without top_k the whole vocabulary is kept (top_p must be 1): each CTA sums exp((l - m_g) / T) over
//    its slice, the cluster combines the slice masses in units of the row maximum, and the CTA whose
//    slice holds the draw u * total finds the token by a block scan of its slice in index order.
//  * temperature 0 is the greedy argmax (largest (key, ~index)).
// A probability row that maps through d2t is zeroed by all CTAs of the cluster before the cluster barrier
// that precedes the writes of the kept probabilities.
//
// accept_residual_kernel: one CTA per sequence; the speculative-sampling rule (accept x with
// probability min(1, p(x) / q(x)); at the first rejection draw from max(0, p - q) renormalised; after
// gamma acceptances draw the bonus token from the target's next distribution).
#include <float.h>
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace e3 {

namespace smp {
constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kCluster = 8;                       // CTAs per row
constexpr int kMaxTopK = 1024;
constexpr int kMaxV = 131072;                     // logits per row
constexpr int kMaxSlice = kMaxV / kCluster;       // keys per CTA
constexpr int kSmemMax = kMaxSlice * 4 + kCluster * kMaxTopK * 8;
}  // namespace smp

// order-preserving image of a float: larger floats give larger unsigned keys
__device__ __forceinline__ uint32_t fkey(float x) {
    const uint32_t b = __float_as_uint(x);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
// the float of a key (exact inverse of fkey)
__device__ __forceinline__ float unkey(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}
// The selection value of token i with key k: larger logits first, lower indices first among equal ones.
__device__ __forceinline__ unsigned long long cval(uint32_t k, int i) {
    return ((unsigned long long)k << 32) | (uint32_t)~(uint32_t)i;
}
__device__ __forceinline__ int cidx(unsigned long long c) { return (int)~(uint32_t)c; }

// inclusive block scan of one float per thread (kThreads threads); returns the thread's inclusive sum
__device__ float block_inclusive_scan(float v, float* warp_tot) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    __syncthreads();
    if (lane == 31) warp_tot[warp] = v;
    __syncthreads();
    if (warp == 0) {
        float t = lane < (int)(blockDim.x >> 5) ? warp_tot[lane] : 0.f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float n = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += n;
        }
        warp_tot[lane] = t;   // inclusive totals per warp
    }
    __syncthreads();
    return v + (warp > 0 ? warp_tot[warp - 1] : 0.f);
}

// bitonic sort of the first n (a power of two <= kThreads) packed (key, index) pairs in shared memory,
// ascending.  Thread t holds element t in a register; a compare-exchange with a partner in the same warp
// (distance j < 32) goes through a shuffle, only the longer distances through shared memory and barriers.
__device__ void bitonic_sort(unsigned long long* a, int n) {
    const int t = threadIdx.x;
    unsigned long long v = t < n ? a[t] : ~0ull;
    for (int k = 2; k <= n; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            unsigned long long w;
            if (j >= 32) {
                __syncthreads();   // the previous exchange's reads are done
                if (t < n) a[t] = v;
                __syncthreads();
                w = t < n ? a[t ^ j] : v;
            } else {
                w = __shfl_xor_sync(0xffffffffu, v, j);
            }
            // of the pair (t, t ^ j) the lower index keeps the minimum in an ascending block (t & k) == 0
            const bool up = (t & k) == 0, lower = (t & j) == 0;
            const unsigned long long lo = v < w ? v : w, hi = v < w ? w : v;
            v = up == lower ? lo : hi;
        }
    }
    __syncthreads();
    if (t < n) a[t] = v;
    __syncthreads();
}

struct SelectShared {
    int whist[smp::kWarps][256];   // per-warp radix histograms (keeps the atomics of different warps apart)
    int hist[256];
    int sh[4];
};

// The K largest of n distinct 64-bit values get(0..n-1), 1 <= K <= n: on return exactly the values with
// (v & mask) >= prefix are the K largest.  Radix select from the top byte; the search ends early once every
// value left in the chosen bin is kept.
template <typename Get>
__device__ void select_largest(int n, int K, Get get, SelectShared& S, unsigned long long& prefix_out,
                               unsigned long long& mask_out) {
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    unsigned long long prefix = 0, mask = 0;
    int need = K;
    for (int shift = 56; shift >= 0; shift -= 8) {
        for (int i = t; i < smp::kWarps * 256; i += blockDim.x) (&S.whist[0][0])[i] = 0;
        __syncthreads();
        for (int i0 = 0; i0 < n; i0 += blockDim.x) {
            const int i = i0 + t;
            int bin = 256;
            if (i < n) {
                const unsigned long long v = get(i);
                if ((v & mask) == prefix) bin = (int)((v >> shift) & 255u);
            }
            // lanes sharing lane 0's bin add once through lane 0; the others add one by one
            const int b0 = __shfl_sync(0xffffffffu, bin, 0);
            const unsigned same = __ballot_sync(0xffffffffu, bin == b0);
            if (bin < 256) {
                if (bin != b0) atomicAdd(&S.whist[warp][bin], 1);
                else if (lane == 0) atomicAdd(&S.whist[warp][b0], __popc(same));
            }
        }
        __syncthreads();
        for (int b = t; b < 256; b += blockDim.x) {
            int c = 0;
#pragma unroll 8
            for (int w = 0; w < smp::kWarps; ++w) c += S.whist[w][b];
            S.hist[b] = c;
        }
        __syncthreads();
        if (warp == 0) {
            // lane L holds bins 255 - 8L down to 248 - 8L; the bin where the count from the top reaches
            // `need` is found by a warp scan, then inside the lane's eight bins
            int c8 = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) c8 += S.hist[255 - 8 * lane - q];
            int incl = c8;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int x = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += x;
            }
            const unsigned hit = __ballot_sync(0xffffffffu, incl >= need);
            if (lane == __ffs(hit) - 1) {
                int acc = incl - c8, d = 255 - 8 * lane;
                for (int q = 0; q < 7; ++q, --d) {
                    if (acc + S.hist[d] >= need) break;
                    acc += S.hist[d];
                }
                S.sh[0] = d;
                S.sh[1] = acc;
                S.sh[2] = S.hist[d];
            }
        }
        __syncthreads();
        const int d = S.sh[0], above = S.sh[1], inbin = S.sh[2];
        prefix |= (unsigned long long)d << shift;
        mask |= 255ull << shift;
        need -= above;
        if (inbin == need) break;   // block-uniform: the whole bin is kept
    }
    prefix_out = prefix;
    mask_out = mask;
}

// Largest 64-bit value over the block (every thread gets it).
__device__ unsigned long long block_max_u64(unsigned long long v, unsigned long long* scratch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
    __syncthreads();
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    v = lane < (int)(blockDim.x >> 5) ? scratch[lane] : 0ull;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ float block_max_f32(float v, float* scratch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_max(v);
    __syncthreads();
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    v = lane < (int)(blockDim.x >> 5) ? scratch[lane] : -INFINITY;
    return warp_max(v);
}

__global__ void __launch_bounds__(smp::kThreads, 1) sample_kernel(SampleArgs s) {
    using namespace smp;
    using namespace tc;
    pdl_trigger();
    pdl_wait();
    __shared__ SelectShared S;
    __shared__ unsigned long long sorted[kThreads];   // (~key, index) packed
    __shared__ unsigned long long red64[kWarps];
    __shared__ float ftot[kWarps];
    __shared__ int sh_int[4];
    __shared__ float sh_f[2];
    __shared__ unsigned long long xchg;                // read by the peers: greedy best / candidate count
    __shared__ float xm, xs;                           // read by the peers: slice maximum and mass
    __shared__ int cnts[kCluster];
    __shared__ float pm[kCluster], psum[kCluster];
    extern __shared__ __align__(16) unsigned char dyn[];
    const int r = blockIdx.y, t = threadIdx.x, V = s.V;
    const int g = (int)cluster_rank();
    const int SL = (V + kCluster - 1) / kCluster;
    const int base = min(V, g * SL), n = min(V, base + SL) - base;   // this CTA's slice [base, base + n)
    uint32_t* keys = reinterpret_cast<uint32_t*>(dyn);
    unsigned long long* cand = reinterpret_cast<unsigned long long*>(dyn + (((size_t)SL * 4 + 15) & ~(size_t)15));
    const float* l = s.logits + (long)r * s.ldl;
    float* probs = s.probs ? s.probs + (long)r * s.ldp : nullptr;
    const bool mapped = s.probs_target && s.d2t;
    const bool greedy = s.temperature <= 0.f, full = !greedy && s.top_k <= 0;
    const float T = s.temperature;
    const float u = s.uniforms[r];

    // the slice's keys: eight loads in flight per thread
    for (int i0 = 0; i0 < n; i0 += 8 * kThreads) {
        float v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int i = i0 + q * kThreads + t;
            v[q] = i < n ? __ldg(l + base + i) : 0.f;
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int i = i0 + q * kThreads + t;
            if (i < n) keys[i] = fkey(v[q]);
        }
    }
    // zero the probability row where only some entries get written, a share per CTA
    if (probs && (!full || mapped)) {
        const int PL = s.probs_len, ch = (PL + kCluster - 1) / kCluster;
        const int z0 = min(PL, g * ch), z1 = min(PL, z0 + ch);
        for (int i = z0 + t; i < z1; i += kThreads) probs[i] = 0.f;
    }
    __syncthreads();

    int token = -1;       // >= 0 in the CTA that writes the row's outputs
    float qtok = 1.f;
    if (greedy) {
        unsigned long long best = 0;
        for (int i = t; i < n; i += kThreads) best = max(best, cval(keys[i], base + i));
        best = block_max_u64(best, red64);
        if (t == 0) xchg = best;
        cluster_sync();
        if (g == 0 && t < 32) {
            unsigned long long b = 0;
            if (t < kCluster && t * SL < V) b = ld_cluster_u64(mapa(su32(&xchg), t));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) b = max(b, __shfl_xor_sync(0xffffffffu, b, o));
            if (t == 0) sh_int[0] = cidx(b);
        }
        cluster_sync();   // the peers' words have been read
        if (g != 0) return;
        __syncthreads();
        token = sh_int[0];
        if (probs && t == 0) {
            const int o = mapped ? token + s.d2t[token] : token;
            if (o >= 0 && o < s.probs_len) probs[o] = 1.f;
        }
    } else if (!full) {
        const int K = min(s.top_k, V);
        // this slice's top K (all of it when it holds no more than K tokens)
        if (n <= K) {
            for (int i = t; i < n; i += kThreads) cand[i] = cval(keys[i], base + i);
            if (t == 0) xchg = (unsigned long long)n;
        } else {
            unsigned long long pre, msk;
            select_largest(n, K, [&](int i) { return cval(keys[i], base + i); }, S, pre, msk);
            if (t == 0) sh_int[2] = 0;
            __syncthreads();
            for (int i = t; i < n; i += kThreads) {
                const unsigned long long c = cval(keys[i], base + i);
                if ((c & msk) >= pre) cand[atomicAdd(&sh_int[2], 1)] = c;
            }
            if (t == 0) xchg = (unsigned long long)K;
        }
        cluster_sync();   // every CTA's candidates and count are visible to CTA 0
        if (g == 0) {
            if (t < kCluster) cnts[t] = t * SL < V ? (int)ld_cluster_u64(mapa(su32(&xchg), t)) : 0;
            __syncthreads();
            // the peers' candidates after this CTA's own (at most K <= kThreads per CTA: one per thread)
            unsigned long long v[kCluster];
            int off = cnts[0];
#pragma unroll
            for (int h = 1; h < kCluster; ++h)
                v[h] = t < cnts[h] ? ld_cluster_u64(mapa(su32(cand + t), h)) : 0ull;
#pragma unroll
            for (int h = 1; h < kCluster; ++h) {
                if (t < cnts[h]) cand[off + t] = v[h];
                off += cnts[h];
            }
            if (t == 0) sh_int[3] = off;
        }
        cluster_sync();   // CTA 0 holds every candidate; the peers are done
        if (g != 0) return;
        const int total = sh_int[3];
        unsigned long long pre = 0, msk = 0;   // keeps every candidate when there are no more than K
        if (total > K) select_largest(total, K, [&](int i) { return cand[i]; }, S, pre, msk);
        if (t == 0) sh_int[2] = 0;
        sorted[t] = ~0ull;
        __syncthreads();
        for (int i = t; i < total; i += kThreads) {
            const unsigned long long c = cand[i];
            if ((c & msk) >= pre) sorted[atomicAdd(&sh_int[2], 1)] = ~c;   // (~key, index)
        }
        __syncthreads();
        const int nk = min(K, total);
        // (logit descending, index ascending) == (~key ascending, index ascending)
        int np2 = 2;
        while (np2 < nk) np2 <<= 1;
        bitonic_sort(sorted, np2);
        const bool live = t < nk;
        const int idx = live ? (int)(sorted[t] & 0xffffffffu) : 0;
        const float lt = live ? unkey(~(uint32_t)(sorted[t] >> 32)) : 0.f;
        const float l0 = unkey(~(uint32_t)(sorted[0] >> 32));
        const float w = live ? __expf((lt - l0) / T) : 0.f;
        const float cum = block_inclusive_scan(w, ftot);
        const float totw = ftot[kWarps - 1];
        // top-p: the shortest prefix whose mass reaches top_p of the total
        int keep = nk;
        if (s.top_p < 1.f) {
            if (t == 0) sh_int[3] = nk;
            __syncthreads();
            const float lim = s.top_p * totw;
            const float prev = cum - w;
            if (live && cum >= lim && prev < lim) sh_int[3] = t + 1;
            __syncthreads();
            keep = sh_int[3];
        }
        // inverse CDF over the kept tokens in index order
        const bool kept = t < keep;
        __syncthreads();
        sorted[t] = kept ? (((unsigned long long)(uint32_t)idx << 32) | __float_as_uint(w)) : ~0ull;
        __syncthreads();
        bitonic_sort(sorted, np2);
        const bool k2 = t < keep;
        const float w2 = k2 ? __uint_as_float((uint32_t)(sorted[t] & 0xffffffffu)) : 0.f;
        const int i2 = k2 ? (int)(sorted[t] >> 32) : 0;
        const float c2 = block_inclusive_scan(w2, ftot);
        const float kept_total = ftot[kWarps - 1];
        const float target = u * kept_total;
        if (t == 0) {   // u rounding past the kept total: the last kept token
            sh_int[0] = (int)(sorted[keep - 1] >> 32);
            sh_f[1] = __uint_as_float((uint32_t)(sorted[keep - 1] & 0xffffffffu));
        }
        __syncthreads();
        if (k2 && c2 - w2 <= target && target < c2) { sh_int[0] = i2; sh_f[1] = w2; }
        __syncthreads();
        token = sh_int[0];
        qtok = sh_f[1] / kept_total;
        if (probs && k2) {
            const int o = mapped ? i2 + s.d2t[i2] : i2;
            if (o >= 0 && o < s.probs_len) probs[o] = w2 / kept_total;
        }
    } else {
        // whole vocabulary: this slice's maximum and mass, in index order (a contiguous run per thread)
        float mloc = -INFINITY;
        for (int i = t; i < n; i += kThreads) mloc = fmaxf(mloc, unkey(keys[i]));
        mloc = block_max_f32(mloc, ftot);
        const int seg = (n + kThreads - 1) / kThreads, i0 = min(n, t * seg), i1 = min(n, i0 + seg);
        float part = 0.f;
        for (int i = i0; i < i1; ++i) part += __expf((unkey(keys[i]) - mloc) / T);
        const float incl = block_inclusive_scan(part, ftot);
        if (t == 0) { xm = mloc; xs = ftot[kWarps - 1]; }
        cluster_sync();
        if (t < kCluster) {
            const bool any = t * SL < V;
            pm[t] = any ? ld_cluster_f32(mapa(su32(&xm), t)) : -INFINITY;
            psum[t] = any ? ld_cluster_f32(mapa(su32(&xs), t)) : 0.f;
        }
        cluster_sync();   // the peers' words have been read
        // the row maximum, every slice's mass in its units and this slice's offset (the same arithmetic in
        // every CTA, so the slices' ranges tile [0, total))
        float m = -INFINITY;
#pragma unroll
        for (int h = 0; h < kCluster; ++h) m = fmaxf(m, pm[h]);
        float total = 0.f, cg = 0.f, wg = 0.f, sg = 1.f;
#pragma unroll
        for (int h = 0; h < kCluster; ++h) {
            const float sc = psum[h] > 0.f ? __expf((pm[h] - m) / T) : 0.f;
            const float wh = psum[h] * sc;
            if (h == g) { cg = total; wg = wh; sg = sc; }
            total += wh;
        }
        const float target = u * total;
        const int last = (V - 1) / SL;   // the last CTA with tokens takes a draw that rounds past the total
        const bool mine = n > 0 && target >= cg && (target < cg + wg || g == last);
        if (mine) {
            const float tl = (target - cg) / sg;   // the draw in this slice's units
            if (t == 0) sh_int[0] = base + n - 1;
            __syncthreads();
            int found = -1;
            if (incl - part <= tl && tl < incl) {
                float c = incl - part;
                for (int i = i0; i < i1; ++i) {
                    c += __expf((unkey(keys[i]) - mloc) / T);
                    if (tl < c) { found = i; break; }
                }
                if (found < 0) found = i1 - 1;
            }
            __syncthreads();
            if (found >= 0) sh_int[0] = base + found;
            __syncthreads();
            token = sh_int[0];
            qtok = __expf((unkey(keys[token - base]) - m) / T) / total;
        }
        if (probs) {
            for (int i = t; i < n; i += kThreads) {
                const int v = base + i;
                const int o = mapped ? v + s.d2t[v] : v;
                if (o >= 0 && o < s.probs_len) probs[o] = __expf((unkey(keys[i]) - m) / T) / total;
            }
        }
    }
    if (token >= 0 && t == 0) {
        int out = token;
        if (s.d2t) {
            out = token + s.d2t[token];
            if (out < 0 || out >= s.target_vocab) {
                if (s.err) set_err(s.err, 4);
                out = out < 0 ? 0 : s.target_vocab - 1;
            }
        }
        s.tokens[r] = out;
        if (s.tokens2) s.tokens2[(long)r * s.tok2_stride] = out;
        if (s.draft_ids) s.draft_ids[r] = token;
        if (s.token_prob) s.token_prob[r] = qtok;
    }
}

// Residual acceptance; one CTA per sequence.  Thread 0 walks the gamma positions (accept x while
// u_accept * q(x) < p(x)); then the block draws the emitted token by inverse CDF in index order over the
// residual max(0, p - q) of the first rejected position, or over p_gamma after gamma acceptances.  p and
// q are over the target vocabulary: p [B, gamma + 1, V], q [B, gamma, V].
__global__ void __launch_bounds__(smp::kThreads) accept_residual_kernel(ResidualArgs a) {
    using namespace smp;
    pdl_trigger();
    pdl_wait();
    __shared__ float ftot[32];
    __shared__ int sh[2];
    const int b = blockIdx.x, t = threadIdx.x, V = a.V, G = a.gamma;
    if (t == 0) {
        int k = 0;
        for (; k < G; ++k) {
            const long pos = (long)b * G + k;
            const int x = a.draft[pos];
            if (x < 0 || x >= V) break;   // an id outside the vocabulary is never accepted
            const float qx = a.draft_probs[pos * V + x];
            const float px = a.target_probs[((long)b * (G + 1) + k) * V + x];
            if (!(a.u_accept[pos] * qx < px)) break;
        }
        sh[0] = k;
        sh[1] = -1;
    }
    __syncthreads();
    const int k = sh[0];
    const float* p = a.target_probs + ((long)b * (G + 1) + k) * V;
    const float* q = k < G ? a.draft_probs + ((long)b * G + k) * V : nullptr;
    const float u = a.u_resample[(long)b * G + (k < G ? k : G - 1)];
    const int seg = (V + kThreads - 1) / kThreads, i0 = t * seg, i1 = min(V, i0 + seg);
    float part = 0.f;
    int last = -1;
    for (int i = i0; i < i1; ++i) {
        const float w = q ? fmaxf(p[i] - q[i], 0.f) : p[i];
        part += w;
        if (w > 0.f) last = i;
    }
    const float incl = block_inclusive_scan(part, ftot);
    const float total = ftot[kThreads / 32 - 1];
    const float target = u * total;
    // the last positive weight is the fallback when u * total rounds past the sum
    if (last >= 0) atomicMax(&sh[1], last);
    __syncthreads();
    const int fallback = sh[1] >= 0 ? sh[1] : V - 1;
    __syncthreads();
    if (t == 0) sh[1] = fallback;
    int found = -1;
    float cum = incl - part;
    if (cum <= target && target < incl) {
        for (int i = i0; i < i1; ++i) {
            const float w = q ? fmaxf(p[i] - q[i], 0.f) : p[i];
            cum += w;
            if (w > 0.f && target < cum) { found = i; break; }
        }
    }
    __syncthreads();
    if (found >= 0) sh[1] = found;
    __syncthreads();
    if (t == 0) {
        a.accepted_len[b] = k;
        a.next_token[b] = sh[1];
    }
}

// Typical acceptance: the published rule of Medusa (Cai et al. 2024), read for the "typical-acceptance"
// strategy that "Eagle3 DeepseekV3 in MAX" §10 names: position i accepts its drafted token x while
// p_i(x) > min(epsilon, delta exp(-H(p_i))), H the entropy (nats) of the target's distribution there.
// One CTA per sequence; the entropy of each position is a block reduction (fp32, log of each positive
// probability), and the walk stops at the first rejection.
__global__ void __launch_bounds__(smp::kThreads)
accept_typical_kernel(const int* draft, const float* target_probs, int gamma, int V, float epsilon, float delta,
                      int* accepted_len) {
    pdl_trigger();
    pdl_wait();
    __shared__ float red[32];
    __shared__ int decision;
    const int b = blockIdx.x, t = threadIdx.x;
    int k = 0;
    for (; k < gamma; ++k) {
        const long pos = (long)b * gamma + k;
        const int x = draft[pos];
        if (x < 0 || x >= V) break;          // an id outside the vocabulary is never accepted
        const float* p = target_probs + pos * V;
        float h = 0.f;
        for (int v = t; v < V; v += blockDim.x) {
            const float q = p[v];
            if (q > 0.f) h -= q * logf(q);
        }
        h = block_sum(h, red);
        if (t == 0) decision = p[x] > fminf(epsilon, delta * expf(-h)) ? 1 : 0;
        __syncthreads();
        const int ok = decision;
        __syncthreads();
        if (!ok) break;
    }
    if (t == 0) accepted_len[b] = k;
}

// Philox4x64-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011): ten
// rounds of two 64 x 64 -> 128-bit products over a 4-word counter; the 2-word key is bumped by the Weyl
// constants after each round.
__device__ __forceinline__ void philox4x64_10(uint64_t* c, uint64_t k0, uint64_t k1) {
    constexpr uint64_t M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
    constexpr uint64_t W0 = 0x9E3779B97F4A7C15ull, W1 = 0xBB67AE8584CAA73Bull;
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint64_t hi0 = __umul64hi(M0, c[0]), lo0 = M0 * c[0];
        const uint64_t hi1 = __umul64hi(M1, c[2]), lo1 = M1 * c[2];
        const uint64_t x0 = hi1 ^ c[1] ^ k0, x2 = hi0 ^ c[3] ^ k1;
        c[0] = x0; c[1] = lo1; c[2] = x2; c[3] = lo0;
        k0 += W0;
        k1 += W1;
    }
}

// out[i] = word i % 4 of the block whose counter is the 256-bit integer offset + i / 4, key (seed, 0): its
// top 24 bits times 2^-24, a uniform in [0, 1) that fp32 holds exactly.  One block per thread.
__global__ void philox_uniforms_kernel(uint64_t seed, uint64_t offset, long n, float* out) {
    pdl_trigger();
    pdl_wait();
    const long nb = (n + 3) / 4;
    for (long j = (long)blockIdx.x * blockDim.x + threadIdx.x; j < nb; j += (long)gridDim.x * blockDim.x) {
        uint64_t c[4];
        c[0] = offset + (uint64_t)j;
        c[1] = c[0] < offset ? 1ull : 0ull;   // carry into the next counter word
        c[2] = 0;
        c[3] = 0;
        philox4x64_10(c, seed, 0);
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const long i = 4 * j + w;
            if (i < n) out[i] = (float)(uint32_t)(c[w] >> 40) * 0x1p-24f;
        }
    }
}

__global__ void acceptance_hist_kernel(const int* acc, int batch, int gamma, int* hist) {
    pdl_trigger();
    pdl_wait();
    extern __shared__ int hsh[];
    for (int k = threadIdx.x; k <= gamma; k += blockDim.x) hsh[k] = 0;
    __syncthreads();
    for (int b = threadIdx.x; b < batch; b += blockDim.x) atomicAdd(&hsh[min(max(acc[b], 0), gamma)], 1);
    __syncthreads();
    for (int k = threadIdx.x; k <= gamma; k += blockDim.x) hist[k] = hsh[k];
}

cudaError_t launch_sample(const SampleArgs& s, cudaStream_t st) {
    using namespace smp;
    if (s.V < 1 || s.V > kMaxV || s.rows < 1 || s.rows > 65535 || s.top_k > kMaxTopK ||
        (s.temperature > 0.f && s.top_k <= 0 && s.top_p < 1.f))
        return cudaErrorInvalidValue;
    cudaError_t e = smem_optin((const void*)sample_kernel, kSmemMax + 16);
    if (e != cudaSuccess) return e;
    const int SL = (s.V + kCluster - 1) / kCluster;
    const bool topk = s.temperature > 0.f && s.top_k > 0;
    const size_t smem = (((size_t)SL * 4 + 15) & ~(size_t)15) +
                        (topk ? (size_t)kCluster * (s.top_k < s.V ? s.top_k : s.V) * 8 : 0);
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kCluster, s.rows);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, sample_kernel, s);
}

cudaError_t launch_accept_typical(const int* draft, const float* target_probs, int batch, int gamma, int V,
                                  float epsilon, float delta, int* accepted_len, int* hist, cudaStream_t st) {
    if (batch < 1 || gamma < 1 || V < 1) return cudaErrorInvalidValue;
    cudaError_t e = launch_pdl(accept_typical_kernel, dim3(batch), dim3(smp::kThreads), 0, st, draft, target_probs, gamma, V,
                               epsilon, delta, accepted_len);
    if (e != cudaSuccess || !hist) return e;
    return launch_pdl(acceptance_hist_kernel, dim3(1), dim3(256), (gamma + 1) * sizeof(int), st, (const int*)accepted_len,
                      batch, gamma, hist);
}

cudaError_t launch_philox_uniforms(uint64_t seed, uint64_t offset, long n, float* out, cudaStream_t st) {
    if (n < 0) return cudaErrorInvalidValue;
    if (n == 0) return cudaSuccess;
    const long nb = (n + 3) / 4;
    const long blocks = (nb + 255) / 256;
    return launch_pdl(philox_uniforms_kernel, dim3((unsigned)(blocks < 1184 ? blocks : 1184)), dim3(256), 0, st, seed,
                      offset, n, out);
}

cudaError_t launch_accept_residual(const ResidualArgs& a, cudaStream_t st) {
    if (a.batch < 1 || a.gamma < 1 || a.V < 1) return cudaErrorInvalidValue;
    cudaError_t e = launch_pdl(accept_residual_kernel, dim3(a.batch), dim3(smp::kThreads), 0, st, a);
    if (e != cudaSuccess || !a.hist) return e;
    return launch_pdl(acceptance_hist_kernel, dim3(1), dim3(256), (a.gamma + 1) * sizeof(int), st, a.accepted_len,
                      a.batch, a.gamma, a.hist);
}

}  // namespace e3
