// Sampled drafts and residual (rejection-sampling) acceptance.
//
// "Eagle3 DeepseekV3 in MAX" §3.1 and §10 name the sampling parameters of the drafts (temperature,
// top-k, top-p) and the rejection-sampling strategies (greedy, residual, ...), and §8 a seed counter
// that feeds the sampler.  Here the uniform random numbers are inputs, so a caller (or a test) draws
// them once and every consumer uses the same ones.
//
// sample_kernel: one CTA of kThreads per row.  x = logits / temperature; since the temperature is
// positive, x is ordered exactly as the logits are, so top_k keeps the top_k largest logits (lower
// indices first among equal values), found by a radix select on the order-preserving integer image of
// the logits; the kept tokens are sorted (logit descending, index ascending) by a bitonic sort in shared
// memory; their softmax weights are exp((l - l_max) / temperature) in fp32; top_p keeps the shortest
// prefix whose mass reaches top_p of the kept mass; the kept weights are renormalised and u picks the
// token by inverse CDF in ascending index order.
// temperature 0 is the greedy argmax.  Without top_k the whole vocabulary is kept (top_p must be 1) and
// the inverse CDF runs over it with a block-wide scan.
//
// accept_residual_kernel: one CTA per sequence; the speculative-sampling rule (accept x with
// probability min(1, p(x) / q(x)); at the first rejection draw from max(0, p - q) renormalised; after
// gamma acceptances draw the bonus token from the target's next distribution).
#include <float.h>
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace e3 {

namespace smp {
constexpr int kThreads = 1024;
constexpr int kMaxTopK = 1024;
constexpr int kKeyCache = 40960;   // rows up to this many logits keep their sort keys in shared memory
constexpr int kMaxChunks = 4096;   // rows of at most 131072 logits
}  // namespace smp

// order-preserving image of a float: larger floats give larger unsigned keys
__device__ __forceinline__ uint32_t fkey(float x) {
    const uint32_t b = __float_as_uint(x);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

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

__device__ int block_inclusive_scan_int(int v, int* warp_tot) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    __syncthreads();
    if (lane == 31) warp_tot[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int t = lane < (int)(blockDim.x >> 5) ? warp_tot[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += n;
        }
        warp_tot[lane] = t;
    }
    __syncthreads();
    return v + (warp > 0 ? warp_tot[warp - 1] : 0);
}

// bitonic sort of the first n (a power of two <= kThreads) packed (key, index) pairs in shared memory,
// ascending
__device__ void bitonic_sort(unsigned long long* a, int n) {
    const int t = threadIdx.x;
    for (int k = 2; k <= n; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            const int p = t ^ j;
            if (t < n && p > t) {
                const bool up = (t & k) == 0;
                const unsigned long long x = a[t], y = a[p];
                if ((x > y) == up) { a[t] = y; a[p] = x; }
            }
            __syncthreads();
        }
    }
}

__global__ void __launch_bounds__(smp::kThreads) sample_kernel(SampleArgs s) {
    using namespace smp;
    pdl_trigger();
    pdl_wait();
    __shared__ unsigned long long sorted[kThreads];   // (key, index) packed; reused
    __shared__ float wv[kThreads];
    __shared__ int hist[256];
    __shared__ int whist[kThreads / 32][256];         // per-warp radix histograms
    __shared__ int ccount[kMaxChunks];                // equal-key counts, then prefixes, per 32 indices
    __shared__ float ftot[32];
    __shared__ int itot[32];
    __shared__ int sh_int[4];
    __shared__ float sh_f[2];
    extern __shared__ uint32_t keycache[];             // [V] keys of the logits when V fits
    const int r = blockIdx.x, t = threadIdx.x, V = s.V;
    const float* l = s.logits + (long)r * s.ldl;
    float* probs = s.probs ? s.probs + (long)r * s.ldp : nullptr;
    const float u = s.uniforms[r];
    int token = 0;
    float qtok = 1.f;

    if (s.temperature <= 0.f) {
        // greedy: max with the lowest index
        float bv = -INFINITY;
        int bi = INT_MAX;
        for (int i = t; i < V; i += kThreads)
            if (l[i] > bv) { bv = l[i]; bi = i; }
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        if ((t & 31) == 0) { wv[t >> 5] = bv; sorted[t >> 5] = (unsigned long long)bi; }
        __syncthreads();
        if (t == 0) {
            float b = wv[0];
            int bidx = (int)sorted[0];
            for (int w = 1; w < kThreads / 32; ++w)
                if (wv[w] > b || (wv[w] == b && (int)sorted[w] < bidx)) { b = wv[w]; bidx = (int)sorted[w]; }
            sh_int[0] = bidx;
        }
        __syncthreads();
        token = sh_int[0];
        if (probs) {
            const int o = s.probs_target && s.d2t ? token + s.d2t[token] : token;
            for (int i = t; i < s.probs_len; i += kThreads) probs[i] = i == o ? 1.f : 0.f;
        }
    } else if (s.top_k <= 0) {
        // whole vocabulary: softmax of x = l / T and inverse CDF in index order
        const float T = s.temperature;
        float m = -INFINITY;
        for (int i = t; i < V; i += kThreads) m = fmaxf(m, l[i]);
        m = warp_max(m);
        if ((t & 31) == 0) wv[t >> 5] = m;
        __syncthreads();
        if (t < 32) {
            float mm = wv[t];
            mm = warp_max(mm);
            if (t == 0) sh_f[0] = mm;
        }
        __syncthreads();
        m = sh_f[0];
        // contiguous segment per thread, so the block scan follows the index order
        const int seg = (V + kThreads - 1) / kThreads, i0 = t * seg, i1 = min(V, i0 + seg);
        float part = 0.f;
        for (int i = i0; i < i1; ++i) part += __expf((l[i] - m) / T);
        const float incl = block_inclusive_scan(part, ftot);
        const float total = ftot[kThreads / 32 - 1];
        const float target = u * total;
        float cum = incl - part;
        int found = -1;
        if (cum <= target && target < incl) {
            for (int i = i0; i < i1; ++i) {
                cum += __expf((l[i] - m) / T);
                if (target < cum) { found = i; break; }
            }
            if (found < 0) found = i1 - 1;
        }
        if (t == 0) sh_int[0] = V - 1;   // u rounding past the total: the last token
        __syncthreads();
        if (found >= 0) sh_int[0] = found;
        __syncthreads();
        token = sh_int[0];
        qtok = __expf((l[token] - m) / T) / total;
        if (probs) {
            if (s.probs_target && s.d2t) {
                for (int i = t; i < s.probs_len; i += kThreads) probs[i] = 0.f;
                __syncthreads();
            }
            for (int i = t; i < V; i += kThreads) {
                const int o = s.probs_target && s.d2t ? i + s.d2t[i] : i;
                if (o >= 0 && o < s.probs_len) probs[o] = __expf((l[i] - m) / T) / total;
            }
        }
    } else {
        const float T = s.temperature;
        const int K = min(s.top_k, min(kMaxTopK, V));
        const bool cached = V <= kKeyCache;
        if (cached) {
            for (int i = t; i < V; i += kThreads) keycache[i] = fkey(l[i]);
            __syncthreads();
        }
        auto key_of = [&](int i) { return cached ? keycache[i] : fkey(l[i]); };
        // radix select of the K-th largest key, 8 bits at a time from the top
        uint32_t prefix = 0, pmask = 0;
        int need = K;
        const int warp = t >> 5;
        for (int shift = 24; shift >= 0; shift -= 8) {
            for (int i = t; i < (kThreads / 32) * 256; i += kThreads) (&whist[0][0])[i] = 0;
            __syncthreads();
            // logits cluster in a few exponents, so most keys share a bin: every warp counts into its own
            // histogram, which keeps the atomics of different warps apart
            for (int i0 = 0; i0 < V; i0 += kThreads) {
                const int i = i0 + t;
                int bin = 256;
                if (i < V) {
                    const uint32_t k = key_of(i);
                    if ((k & pmask) == prefix) bin = (int)((k >> shift) & 255u);
                }
                // lanes sharing lane 0's bin add once through lane 0; the others add one by one
                const int b0 = __shfl_sync(0xffffffffu, bin, 0);
                const unsigned same = __ballot_sync(0xffffffffu, bin == b0);
                if (bin < 256) {
                    if (bin != b0) atomicAdd(&whist[warp][bin], 1);
                    else if ((t & 31) == 0) atomicAdd(&whist[warp][b0], __popc(same));
                }
            }
            __syncthreads();
            for (int b = t; b < 256; b += kThreads) {
                int c = 0;
                for (int w = 0; w < kThreads / 32; ++w) c += whist[w][b];
                hist[b] = c;
            }
            __syncthreads();
            if (t == 0) {
                int acc = 0, d = 255;
                for (; d > 0; --d) {
                    if (acc + hist[d] >= need) break;
                    acc += hist[d];
                }
                sh_int[0] = d;
                sh_int[1] = acc;
                sh_int[3] = hist[d];   // after the last pass: the number of keys equal to the threshold
            }
            __syncthreads();
            prefix |= (uint32_t)sh_int[0] << shift;
            pmask |= 255u << shift;
            need -= sh_int[1];
            __syncthreads();
        }
        const uint32_t kth = prefix;   // keys > kth are all kept; `need` of the keys == kth, lowest index first
        // gather: keys above the threshold, then the first `need` equal keys in index order
        if (t == 0) sh_int[2] = 0;
        sorted[t] = ~0ull;
        __syncthreads();
        // when every key equal to the threshold is kept (the usual case) one pass gathers them all
        const bool all_eq = sh_int[3] == need;
        for (int i = t; i < V; i += kThreads) {
            const uint32_t k = key_of(i);
            if (k > kth || (all_eq && k == kth)) {
                const int slot = atomicAdd(&sh_int[2], 1);
                sorted[slot] = ((unsigned long long)(~k) << 32) | (uint32_t)i;
            }
        }
        __syncthreads();
        if (!all_eq)
        {
            // equal keys in index order: per 32-index chunk counts by ballot, one scan over the chunk counts,
            // then ranks inside the chunks that hold any of the `need` first equal keys
            const int base = sh_int[2];
            const int nchunk = (V + 31) / 32;
            for (int c = warp; c < nchunk; c += kThreads / 32) {
                const int i = c * 32 + (t & 31);
                const unsigned bal = __ballot_sync(0xffffffffu, i < V && key_of(i) == kth);
                if ((t & 31) == 0) ccount[c] = __popc(bal);
            }
            __syncthreads();
            const int per = (nchunk + kThreads - 1) / kThreads, c0 = t * per, c1 = min(nchunk, c0 + per);
            int mine = 0;
            for (int c = c0; c < c1; ++c) mine += ccount[c];
            int run = block_inclusive_scan_int(mine, itot) - mine;
            for (int c = c0; c < c1; ++c) {
                const int cn = ccount[c];
                ccount[c] = run;
                run += cn;
            }
            __syncthreads();
            for (int c = warp; c < nchunk; c += kThreads / 32) {
                const int start = ccount[c];
                if (start >= need) continue;   // warp-uniform
                const int i = c * 32 + (t & 31);
                const bool eq = i < V && key_of(i) == kth;
                const unsigned bal = __ballot_sync(0xffffffffu, eq);
                const int rank = start + __popc(bal & ((1u << (t & 31)) - 1u));
                if (eq && rank < need) sorted[base + rank] = ((unsigned long long)(~kth) << 32) | (uint32_t)i;
            }
            __syncthreads();
        }
        const int n = K;
        // (logit descending, index ascending) == (~key ascending, index ascending)
        int np2 = 2;
        while (np2 < n) np2 <<= 1;
        bitonic_sort(sorted, np2);
        const bool live = t < n;
        const int idx = live ? (int)(sorted[t] & 0xffffffffu) : 0;
        const float l0 = l[(int)(sorted[0] & 0xffffffffu)];
        const float w = live ? __expf((l[idx] - l0) / T) : 0.f;
        const float cum = block_inclusive_scan(w, ftot);
        const float total = ftot[kThreads / 32 - 1];
        // top-p: the shortest prefix whose mass reaches top_p of the total
        int keep = n;
        if (s.top_p < 1.f) {
            if (t == 0) sh_int[3] = n;
            __syncthreads();
            const float lim = s.top_p * total;
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
        const float kept_total = ftot[kThreads / 32 - 1];
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
        if (probs) {
            for (int i = t; i < s.probs_len; i += kThreads) probs[i] = 0.f;
            __syncthreads();
            if (k2) {
                const int o = s.probs_target && s.d2t ? i2 + s.d2t[i2] : i2;
                if (o >= 0 && o < s.probs_len) probs[o] = w2 / kept_total;
            }
        }
    }
    if (t == 0) {
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
    if (s.V < 1 || s.V > 32 * smp::kMaxChunks || s.rows < 1 || (s.top_k > smp::kMaxTopK) ||
        (s.temperature > 0.f && s.top_k <= 0 && s.top_p < 1.f))
        return cudaErrorInvalidValue;
    {
        cudaError_t e = smem_optin((const void*)sample_kernel, (int)(smp::kKeyCache * sizeof(uint32_t)));
        if (e != cudaSuccess) return e;
    }
    const bool cached = s.temperature > 0.f && s.top_k > 0 && s.V <= smp::kKeyCache;
    const size_t smem = cached ? (size_t)s.V * sizeof(uint32_t) : 0;
    return launch_pdl(sample_kernel, dim3(s.rows), dim3(smp::kThreads), smem, st, s);
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
