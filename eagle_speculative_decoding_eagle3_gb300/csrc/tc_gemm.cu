// tcgen05 (5th-generation tensor core) GEMM for the linear layers at many activation rows.
//
// out[m, n] = sum_k W[n, k] X[m, k] for the bias-free projections of the draft head (fc, q_a | kv_a,
// q_b, o_proj, gate | up, down, lm_head; "Eagle3 DeepseekV3 in MAX" §4) once the rows no longer fit
// the weight-streaming GEMV (extend, or decode at large batch).
//
// Orientation: the WEIGHT tile is the MMA "A" operand (128 rows of W, the MMA M) and the ACTIVATION
// tile is the MMA "B" operand (BN rows of X, the MMA N), so one tile is D^T[n, m] in TMEM with
// lane = output feature n and column = token m.  A small batch then still fills the 128-row MMA, and
// the epilogue's warp writes 32 consecutive features of one token: coalesced stores.
//
// Per CTA (192 threads): warp 0 issues TMA loads (128-byte swizzle, K-major) into a STAGES-deep
// ring; warp 1 owns the TMEM accumulator and one elected lane issues tcgen05.mma (kind::f16, bf16
// in, fp32 accumulate) and tcgen05.commit to release stages; warps 2-5 wait for the accumulator,
// read it with tcgen05.ld and apply the epilogue (store, residual add, SiLU(gate) * up, row argmax,
// or split-K partials).  Every mbarrier wait is bounded: a wait that runs out sets an error bit,
// the CTA skips the rest of its work, drains its own copies (bounded), frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <float.h>
#include <limits.h>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"
#include "../../include/eagle3.h"

namespace e3 {
namespace tc {

constexpr int BM = 128;                 // weight rows per tile (MMA M)
constexpr int BK = 64;                  // K per stage: one 128-byte swizzle atom of bf16
constexpr int kThreads = 192;
constexpr int kSmemBudget = 200 * 1024;

// MODE: kSingle (one 128-row weight tile), kGlu (gate and up tiles of the same rows, SiLU(gate) * up)
// or kPair (two consecutive 128-row tiles of one weight matrix sharing the activation tile: the CTA
// covers 256 output features, so each staged activation tile feeds twice the MMA work).
constexpr int kSingle = 0, kGlu = 1, kPair = 2;
template <int BN, int MODE> struct Cfg {
    static constexpr int NP = MODE == kSingle ? 1 : 2;
    static constexpr int P_BYTES = BM * BK * 2;
    static constexpr int Q_BYTES = BN * BK * 2;
    static constexpr int STAGE = NP * P_BYTES + Q_BYTES;
    static constexpr int STAGES = (kSmemBudget / STAGE) > 6 ? 6 : (kSmemBudget / STAGE);
    static constexpr int COLS_USED = NP * BN;
    static constexpr int TMEM_COLS = COLS_USED <= 32 ? 32 : COLS_USED <= 64 ? 64 : COLS_USED <= 128 ? 128
                                   : COLS_USED <= 256 ? 256 : 512;
    static constexpr int SMEM = STAGES * STAGE + 1024 + 256;
};

template <int BN, int MODE>
__global__ void __launch_bounds__(kThreads, 1) tc_gemm_kernel(const __grid_constant__ TcParams p) {
    pdl_trigger();
    using C = Cfg<BN, MODE>;
    constexpr bool GLU = MODE == kGlu, PAIR = MODE == kPair;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* base = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + C::STAGES * C::STAGE);
    // bars[0..S) full, bars[S..2S) empty, bars[2S] accumulator ready
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * C::STAGES + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // tile order: groups of up to 8 token tiles run back to back on each weight tile, so the CTAs in
    // flight share weight panels in L2 instead of streaming every weight panel once per token tile
    int ntile = blockIdx.x, mtile = blockIdx.y;
    if (gridDim.y > 1) {
        constexpr int G = 8;
        const int lin = blockIdx.x + gridDim.x * blockIdx.y;
        const int g = lin / (G * gridDim.x), in = lin % (G * gridDim.x);
        const int gsize = min(G, (int)gridDim.y - g * G);
        mtile = g * G + in % gsize;
        ntile = in / gsize;
    }
    const int n0 = ntile * (PAIR ? 2 * BM : BM), m0 = mtile * BN;
    const int split = blockIdx.z % p.splits, batch = blockIdx.z / p.splits;
    const int kb0 = split * p.kb_per_split;
    const int kb1 = min(p.nkb, kb0 + p.kb_per_split);
    const int nkb = kb1 - kb0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(su32(&bars[s]), 1);
            mbar_init(su32(&bars[C::STAGES + s]), 1);
        }
        mbar_init(su32(&bars[2 * C::STAGES]), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                     "r"(C::TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    int issued = 0;
    pdl_wait();

    if (warp == 0 && lane == 0 && nkb > 0) {
        // ---------------- TMA producer
        const bool second = !GLU && n0 >= p.np0;
        const CUtensorMap* mw = second ? &p.mw[1] : &p.mw[0];
        const int wrow = (second ? n0 - p.np0 : n0) + batch * p.bw_rows;
        for (int i = 0; i < nkb; ++i) {
            const int s = i % C::STAGES;
            const uint32_t ph = (uint32_t)(i / C::STAGES) & 1u;
            if (!mbar_wait(su32(&bars[C::STAGES + s]), ph ^ 1u)) { *abort_flag = 1; break; }
            if (*abort_flag) break;
            unsigned char* st = base + s * C::STAGE;
            const uint32_t full = su32(&bars[s]);
            mbar_expect_tx(full, C::STAGE);
            const int kb = kb0 + i;
            tma_load_2d(su32(st), mw, full, kb * BK, wrow);
            if (GLU) tma_load_2d(su32(st + C::P_BYTES), &p.mw[1], full, kb * BK, n0 + batch * p.bw_rows);
            if (PAIR) {   // rows n0 + 128 .. of the same weights (segment chosen per tile)
                const int n1 = n0 + BM;
                const bool sec1 = n1 >= p.np0;
                tma_load_2d(su32(st + C::P_BYTES), sec1 ? &p.mw[1] : &p.mw[0], full, kb * BK, sec1 ? n1 - p.np0 : n1);
            }
            const int qs = kb >= p.kseg[1] ? 2 : (kb >= p.kseg[0] ? 1 : 0);
            const int kl = kb - (qs == 0 ? 0 : p.kseg[qs - 1]) + batch * p.bq_kb;
            tma_load_2d(su32(st + C::NP * C::P_BYTES), &p.mx[qs], full, kl * BK, m0);
            ++issued;
        }
    } else if (warp == 1 && lane == 0 && nkb > 0) {
        // ---------------- MMA issuer
        constexpr uint32_t idesc = instr_desc(BN);
        for (int i = 0; i < nkb; ++i) {
            const int s = i % C::STAGES;
            const uint32_t ph = (uint32_t)(i / C::STAGES) & 1u;
            if (!mbar_wait(su32(&bars[s]), ph)) { *abort_flag = 1; break; }
            tc_fence_after();
            const uint32_t st = su32(base + s * C::STAGE);
            const uint64_t da = smem_desc(st);
            const uint64_t da2 = smem_desc(st + C::P_BYTES);
            const uint64_t db = smem_desc(st + C::NP * C::P_BYTES);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
                const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
                mma_bf16(tmem, da + 2 * kk, db + 2 * kk, idesc, acc);
                if (GLU || PAIR) mma_bf16(tmem + BN, da2 + 2 * kk, db + 2 * kk, idesc, acc);
            }
            mma_commit(su32(&bars[C::STAGES + s]));
        }
        mma_commit(su32(&bars[2 * C::STAGES]));
    } else if (warp >= 2) {
        // ---------------- epilogue: TMEM lanes [32q, 32q+32) are readable by warp q = warp % 4
        const int q = warp & 3;
        const int n_base = n0 + 32 * q + lane;
        bool ok = nkb > 0 && mbar_wait(su32(&bars[2 * C::STAGES]), 0);
        ok = __all_sync(0xffffffffu, ok);   // tcgen05.ld is warp-collective
        if (!ok && nkb > 0) *abort_flag = 1;
        tc_fence_after();
        const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16);
        const bool splitk = p.splits > 1;   // write fp32 partials for the reduction kernel
        // bf16-only outputs are staged through the (now idle) stage ring as [token][feature] rows and
        // leave in 16-byte row chunks: output rows are far apart (tens of KB), and one 64-byte piece
        // per row per store instruction left the writes at a fraction of the bandwidth
        constexpr int TW = PAIR ? 2 * BM : BM;      // output features of this CTA
        constexpr int OPITCH = TW + 8;              // staged row pitch (bf16), 16-byte multiple
        static_assert((size_t)BN * OPITCH * 2 <= (size_t)C::STAGES * C::STAGE, "staged tile fits the ring");
        const bool staged = !splitk && p.epi != EPI_ARGMAX && p.epi != EPI_RESID && p.y == nullptr && p.ybf != nullptr;
        __nv_bfloat16* obuf = reinterpret_cast<__nv_bfloat16*>(base);
        // kPair: columns [0, BN) of the accumulator hold features n, columns [BN, 2 BN) features n + 128
        constexpr int CW = BN >= 32 ? 32 : 16;   // accumulator columns per TMEM load
        for (int cc = 0; cc < (PAIR ? 2 * BN : BN); cc += CW) {
            const int c = PAIR ? cc % BN : cc;
            const int n = n_base + (PAIR && cc >= BN ? BM : 0);
            const long ncol = n + (long)batch * p.by_col;
            const bool nvalid = n < p.N;
            float v[CW], u[CW];
            if (ok) {
                if (CW == 32) {
                    tmem_ld32(trow + cc, v);
                    if (GLU) tmem_ld32(trow + BN + c, u);
                } else {
                    tmem_ld16(trow + cc, v);
                    if (GLU) tmem_ld16(trow + BN + c, u);
                }
            } else {
#pragma unroll
                for (int j = 0; j < CW; ++j) { v[j] = 0.f; u[j] = 0.f; }
            }
            if (p.epi == EPI_ARGMAX) {
                // per token: (max, argmax) over this warp's 32 features, lowest index on ties
#pragma unroll
                for (int j = 0; j < CW; ++j) {
                    float bvv = nvalid ? v[j] : -FLT_MAX;
                    int bi = nvalid ? n : INT_MAX;
                    const int m = m0 + c + j;
                    if (p.logits && nvalid && m < p.M) p.logits[(long)m * p.ldl + ncol] = v[j];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        const float ov = __shfl_xor_sync(0xffffffffu, bvv, o);
                        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                        if (better(ov, oi, bvv, bi)) { bvv = ov; bi = oi; }
                    }
                    if (lane == 0) {
                        float* rv = reinterpret_cast<float*>(base);          // stage memory is idle now
                        int* ri = reinterpret_cast<int*>(base + 4 * BN * sizeof(float));
                        rv[q * BN + c + j] = bvv;
                        ri[q * BN + c + j] = bi;
                    }
                }
                continue;
            }
            // residual operands first: all CW loads are in flight before the first store (the output
            // may alias nothing, but the compiler cannot know that)
            float rv16[CW];
            if (p.epi == EPI_RESID && !splitk) {
#pragma unroll
                for (int j = 0; j < CW; ++j) {
                    const int m = m0 + c + j;
                    rv16[j] = (nvalid && m < p.M) ? p.resid[(long)m * p.ldr + ncol] : 0.f;
                }
            }
#pragma unroll
            for (int j = 0; j < CW; ++j) {
                const int m = m0 + c + j;
                if (!nvalid || m >= p.M) continue;
                if (splitk) {
                    const long plane = (long)p.M * p.N;
                    float* part = p.part + (long)split * (GLU ? 2 : 1) * plane;
                    part[(long)m * p.N + n] = v[j];
                    if (GLU) part[plane + (long)m * p.N + n] = u[j];
                    continue;
                }
                float out;
                if (GLU) out = silu(v[j]) * u[j];
                else if (p.epi == EPI_RESID) out = v[j] + rv16[j];
                else out = v[j];
                if (staged) {
                    obuf[(c + j) * OPITCH + (n - n0)] = __float2bfloat16_rn(out);
                    continue;
                }
                if (p.y) p.y[(long)m * p.ldy + ncol] = out;
                if (p.ybf) p.ybf[(long)m * p.ldybf + ncol] = __float2bfloat16_rn(out);
            }
        }
        if (staged) {
            asm volatile("bar.sync 1, 128;" ::: "memory");   // the four epilogue warps
            constexpr int CPR = TW / 8;                       // 16-byte chunks per staged row
            const long col0 = (long)batch * p.by_col;
            for (int i = threadIdx.x - 64; i < BN * CPR; i += 128) {
                const int row = i / CPR, ch = i % CPR;
                const int m = m0 + row, nf = n0 + ch * 8;
                if (m >= p.M || nf >= p.N) continue;
                *reinterpret_cast<uint4*>(p.ybf + (long)m * p.ldybf + col0 + nf) =
                    *reinterpret_cast<const uint4*>(obuf + row * OPITCH + ch * 8);
            }
        }
        if (p.epi == EPI_ARGMAX) {
            asm volatile("bar.sync 1, 128;" ::: "memory");   // the four epilogue warps
            const float* rv = reinterpret_cast<const float*>(base);
            const int* ri = reinterpret_cast<const int*>(base + 4 * BN * sizeof(float));
            for (int j = threadIdx.x - 64; j < BN; j += 128) {
                const int m = m0 + j;
                if (m >= p.M) continue;
                float b = rv[j];
                int bi = ri[j];
                for (int w = 1; w < 4; ++w)
                    if (better(rv[w * BN + j], ri[w * BN + j], b, bi)) { b = rv[w * BN + j]; bi = ri[w * BN + j]; }
                p.pval[(long)m * p.npart + ntile] = b;
                p.pidx[(long)m * p.npart + ntile] = bi;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {
        if (threadIdx.x == 0) atomicOr(p.err, EAGLE3_DEVERR_TIMEOUT);
        // drain this CTA's own copies still in flight (bounded) before its shared memory goes away
        if (warp == 0 && lane == 0) {
            for (int i = max(0, issued - C::STAGES); i < issued; ++i)
                mbar_wait(su32(&bars[i % C::STAGES]), (uint32_t)(i / C::STAGES) & 1u);
        }
        __syncthreads();
    }
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS));
    }
}

// Persistent variant for one-matrix GEMMs with more output tiles than SMs and no split (the lm_head with its
// argmax, q_b, and short-K GEMMs of an extend).  One CTA per SM walks the tiles lin = blockIdx.x,
// + gridDim.x, ... in the grouped order above.  The TMA ring runs across tile boundaries and two TMEM
// accumulators alternate (MMA into one while the epilogue warps drain the other), so a tile's epilogue
// and the next tile's pipeline fill overlap its neighbours' loads and MMAs.  The epilogue scratch (the
// argmax partials of the four warps, or the staged bf16 output tile) has its own shared memory, since
// the ring keeps streaming.
template <int BN> struct PCfg {
    static constexpr int P_BYTES = BM * BK * 2;
    static constexpr int Q_BYTES = BN * BK * 2;
    static constexpr int STAGE = P_BYTES + Q_BYTES;
    static constexpr int OPITCH = BM + 8;                  // staged row pitch (bf16), 16-byte multiple
    static constexpr int OBUF = BN * OPITCH * 2;
    static constexpr int ABUF = 4 * BN * 8;
    static constexpr int SCRATCH = ((OBUF > ABUF ? OBUF : ABUF) + 1023) / 1024 * 1024;
    static constexpr int STAGES0 = (222 * 1024 - SCRATCH - 2048) / STAGE;
    static constexpr int STAGES = STAGES0 > 6 ? 6 : STAGES0;
    static constexpr int TMEM_COLS = 2 * BN <= 32 ? 32 : 2 * BN <= 64 ? 64 : 2 * BN <= 128 ? 128 : 2 * BN <= 256 ? 256 : 512;
    static constexpr int SMEM = STAGES * STAGE + SCRATCH + 1024 + 256;
    static_assert(STAGES >= 2, "at least a double-buffered ring");
    static_assert(SMEM <= 227 * 1024, "shared memory");
};

template <int BN>
__global__ void __launch_bounds__(kThreads, 1) tc_gemm_persist_kernel(const __grid_constant__ TcParams p) {
    pdl_trigger();
    using C = PCfg<BN>;
    constexpr int S = C::STAGES;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* base = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    unsigned char* scratch = base + S * C::STAGE;
    uint64_t* bars = reinterpret_cast<uint64_t*>(scratch + C::SCRATCH);
    // bars[0..S) full, bars[S..2S) empty, bars[2S + b] accumulator b ready, bars[2S + 2 + b] accumulator b free
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 4);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    auto bar = [&](int i) { return su32(&bars[i]); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nx = (p.N + BM - 1) / BM, ny = (p.M + BN - 1) / BN, ntiles = nx * ny;
    const int my_tiles = blockIdx.x < ntiles ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    auto tile_of = [&](int lin, int& ntile, int& mtile) {
        if (ny > 1) {
            constexpr int G = 8;
            const int g = lin / (G * nx), in = lin % (G * nx);
            const int gsize = min(G, ny - g * G);
            mtile = g * G + in % gsize;
            ntile = in / gsize;
        } else {
            ntile = lin;
            mtile = 0;
        }
    };
    const int nkb = p.nkb;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar(s), 1);
            mbar_init(bar(S + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(2 * S + b), 1);
            mbar_init(bar(2 * S + 2 + b), 4);   // one arrival per epilogue warp
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                     "r"(C::TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    int issued = 0;
    pdl_wait();

    if (warp == 0 && lane == 0 && nkb > 0) {
        // ---------------- TMA producer: every k-block of every tile of this CTA, one ring
        int i = 0;
        for (int t = 0; t < my_tiles; ++t) {
            int ntile, mtile;
            tile_of(blockIdx.x + t * gridDim.x, ntile, mtile);
            const int n0 = ntile * BM, m0 = mtile * BN;
            const bool second = n0 >= p.np0;
            const CUtensorMap* mw = second ? &p.mw[1] : &p.mw[0];
            const int wrow = second ? n0 - p.np0 : n0;
            for (int kb = 0; kb < nkb; ++kb, ++i) {
                const int s = i % S;
                if (!mbar_wait(bar(S + s), ((uint32_t)(i / S) & 1u) ^ 1u)) { *abort_flag = 1; break; }
                if (*abort_flag) break;
                unsigned char* st = base + s * C::STAGE;
                const uint32_t full = bar(s);
                mbar_expect_tx(full, C::STAGE);
                tma_load_2d(su32(st), mw, full, kb * BK, wrow);
                const int qs = kb >= p.kseg[1] ? 2 : (kb >= p.kseg[0] ? 1 : 0);
                const int kl = kb - (qs == 0 ? 0 : p.kseg[qs - 1]);
                tma_load_2d(su32(st + C::P_BYTES), &p.mx[qs], full, kl * BK, m0);
                ++issued;
            }
            if (*abort_flag) break;
        }
    } else if (warp == 1 && lane == 0 && nkb > 0) {
        // ---------------- MMA issuer: tile t accumulates into TMEM columns [BN (t & 1), + BN)
        constexpr uint32_t idesc = instr_desc(BN);
        int i = 0;
        bool ok = true;
        for (int t = 0; t < my_tiles && ok; ++t) {
            const int b = t & 1;
            ok = mbar_wait(bar(2 * S + 2 + b), ((uint32_t)(t >> 1) & 1u) ^ 1u) && !*abort_flag;
            if (!ok) break;
            tc_fence_after();
            for (int kb = 0; kb < nkb; ++kb, ++i) {
                const int s = i % S;
                if (!mbar_wait(bar(s), (uint32_t)(i / S) & 1u)) { ok = false; break; }
                tc_fence_after();
                const uint32_t st = su32(base + s * C::STAGE);
                const uint64_t da = smem_desc(st), db = smem_desc(st + C::P_BYTES);
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)
                    mma_bf16(tmem + BN * b, da + 2 * kk, db + 2 * kk, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
                mma_commit(bar(S + s));
            }
            if (ok) mma_commit(bar(2 * S + b));
        }
        if (!ok) *abort_flag = 1;
    } else if (warp >= 2) {
        // ---------------- epilogue: TMEM lanes [32q, 32q + 32) are readable by warp q = warp % 4
        const int q = warp & 3;
        const int et = threadIdx.x - 64;   // 0..127 over the four epilogue warps
        const bool staged = p.epi != EPI_ARGMAX && p.epi != EPI_RESID && p.y == nullptr && p.ybf != nullptr;
        __nv_bfloat16* obuf = reinterpret_cast<__nv_bfloat16*>(scratch);
        float* rv = reinterpret_cast<float*>(scratch);
        int* ri = reinterpret_cast<int*>(scratch + 4 * BN * sizeof(float));
        constexpr int CW = BN >= 32 ? 32 : 16;
        for (int t = 0; t < my_tiles; ++t) {
            const int b = t & 1;
            int ntile, mtile;
            tile_of(blockIdx.x + t * gridDim.x, ntile, mtile);
            const int n0 = ntile * BM, m0 = mtile * BN;
            const int n = n0 + 32 * q + lane;
            const bool nvalid = n < p.N;
            // every epilogue warp runs every tile (the named barriers below count on it); after a wait ran
            // out the tiles are written as zeros
            bool ok = nkb > 0 && !*abort_flag && mbar_wait(bar(2 * S + b), (uint32_t)(t >> 1) & 1u);
            ok = __all_sync(0xffffffffu, ok);   // tcgen05.ld is warp-collective
            if (!ok && nkb > 0) *abort_flag = 1;
            tc_fence_after();
            const uint32_t trow = tmem + BN * b + ((uint32_t)(32 * q) << 16);
            for (int c = 0; c < BN; c += CW) {
                float v[CW];
                if (ok) {
                    if (CW == 32) tmem_ld32(trow + c, v);
                    else tmem_ld16(trow + c, v);
                } else {
#pragma unroll
                    for (int j = 0; j < CW; ++j) v[j] = 0.f;
                }
                if (p.epi == EPI_ARGMAX) {
                    // per token: (max, argmax) over this warp's 32 features, lowest index on ties
#pragma unroll
                    for (int j = 0; j < CW; ++j) {
                        float bvv = nvalid ? v[j] : -FLT_MAX;
                        int bi = nvalid ? n : INT_MAX;
                        const int m = m0 + c + j;
                        if (p.logits && nvalid && m < p.M) p.logits[(long)m * p.ldl + n] = v[j];
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) {
                            const float ov = __shfl_xor_sync(0xffffffffu, bvv, o);
                            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                            if (better(ov, oi, bvv, bi)) { bvv = ov; bi = oi; }
                        }
                        if (lane == 0) {
                            rv[q * BN + c + j] = bvv;
                            ri[q * BN + c + j] = bi;
                        }
                    }
                    continue;
                }
                float rr[CW];
                if (p.epi == EPI_RESID) {
#pragma unroll
                    for (int j = 0; j < CW; ++j) {
                        const int m = m0 + c + j;
                        rr[j] = (nvalid && m < p.M) ? p.resid[(long)m * p.ldr + n] : 0.f;
                    }
                }
#pragma unroll
                for (int j = 0; j < CW; ++j) {
                    const int m = m0 + c + j;
                    if (!nvalid || m >= p.M) continue;
                    const float out = p.epi == EPI_RESID ? v[j] + rr[j] : v[j];
                    if (staged) {
                        obuf[(c + j) * C::OPITCH + (n - n0)] = __float2bfloat16_rn(out);
                        continue;
                    }
                    if (p.y) p.y[(long)m * p.ldy + n] = out;
                    if (p.ybf) p.ybf[(long)m * p.ldybf + n] = __float2bfloat16_rn(out);
                }
            }
            // the accumulator is read out: the MMA warp may start the tile after next in it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(2 * S + 2 + b));
            if (staged || p.epi == EPI_ARGMAX) {
                asm volatile("bar.sync 1, 128;" ::: "memory");   // the four epilogue warps
                if (staged) {
                    constexpr int CPR = BM / 8;                   // 16-byte chunks per staged row
                    for (int i = et; i < BN * CPR; i += 128) {
                        const int row = i / CPR, ch = i % CPR;
                        const int m = m0 + row, nf = n0 + ch * 8;
                        if (m >= p.M || nf >= p.N) continue;
                        *reinterpret_cast<uint4*>(p.ybf + (long)m * p.ldybf + nf) =
                            *reinterpret_cast<const uint4*>(obuf + row * C::OPITCH + ch * 8);
                    }
                } else {
                    for (int j = et; j < BN; j += 128) {
                        const int m = m0 + j;
                        if (m >= p.M) continue;
                        float bb = rv[j];
                        int bi = ri[j];
                        for (int w = 1; w < 4; ++w)
                            if (better(rv[w * BN + j], ri[w * BN + j], bb, bi)) { bb = rv[w * BN + j]; bi = ri[w * BN + j]; }
                        p.pval[(long)m * p.npart + ntile] = bb;
                        p.pidx[(long)m * p.npart + ntile] = bi;
                    }
                }
                asm volatile("bar.sync 1, 128;" ::: "memory");   // scratch is free for the next tile
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {
        if (threadIdx.x == 0) atomicOr(p.err, EAGLE3_DEVERR_TIMEOUT);
        // drain this CTA's own copies still in flight (bounded) before its shared memory goes away
        if (warp == 0 && lane == 0) {
            for (int i = max(0, issued - S); i < issued; ++i)
                mbar_wait(bar(i % S), (uint32_t)(i / S) & 1u);
        }
        __syncthreads();
    }
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS));
    }
}

// Split-K reduction: out = epi(sum_z part[z]) for STORE / RESID / GLU, the planes summed in split order.
// With N a multiple of 4 a thread takes four consecutive outputs and keeps four planes' loads in flight.
__global__ void tc_splitk_reduce(const TcParams p, int splits, int glu) {
    pdl_trigger();
    pdl_wait();
    const long total = (long)p.M * p.N;
    const long plane = total;
    const int np = glu ? 2 : 1;
    if ((p.N & 3) == 0) {
        for (long i4 = blockIdx.x * (long)blockDim.x + threadIdx.x; i4 < total / 4; i4 += (long)gridDim.x * blockDim.x) {
            const long i = 4 * i4;
            float v[4] = {0.f, 0.f, 0.f, 0.f}, u[4] = {0.f, 0.f, 0.f, 0.f};
            int z = 0;
            for (; z + 4 <= splits; z += 4) {
                float4 a[4], b[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    a[q] = __ldcg(reinterpret_cast<const float4*>(p.part + (long)(z + q) * np * plane + i));
                    if (glu) b[q] = __ldcg(reinterpret_cast<const float4*>(p.part + (long)(z + q) * np * plane + plane + i));
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    v[0] += a[q].x; v[1] += a[q].y; v[2] += a[q].z; v[3] += a[q].w;
                    if (glu) { u[0] += b[q].x; u[1] += b[q].y; u[2] += b[q].z; u[3] += b[q].w; }
                }
            }
            for (; z < splits; ++z) {
                const float4 a = __ldcg(reinterpret_cast<const float4*>(p.part + (long)z * np * plane + i));
                v[0] += a.x; v[1] += a.y; v[2] += a.z; v[3] += a.w;
                if (glu) {
                    const float4 b = __ldcg(reinterpret_cast<const float4*>(p.part + (long)z * np * plane + plane + i));
                    u[0] += b.x; u[1] += b.y; u[2] += b.z; u[3] += b.w;
                }
            }
            const long m = i / p.N, n = i % p.N;
            float r[4] = {0.f, 0.f, 0.f, 0.f};
            if (!glu && p.epi == EPI_RESID) {
#pragma unroll
                for (int e = 0; e < 4; ++e) r[e] = p.resid[m * p.ldr + n + e];
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float out = glu ? silu(v[e]) * u[e] : v[e] + r[e];
                if (p.y) p.y[m * p.ldy + n + e] = out;
                if (p.ybf) p.ybf[m * p.ldybf + n + e] = __float2bfloat16_rn(out);
            }
        }
        return;
    }
    for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total; i += (long)gridDim.x * blockDim.x) {
        float v = 0.f, u = 0.f;
        for (int z = 0; z < splits; ++z) {
            v += p.part[(long)z * np * plane + i];
            if (glu) u += p.part[(long)z * np * plane + plane + i];
        }
        const long m = i / p.N, n = i % p.N;
        float out;
        if (glu) out = silu(v) * u;
        else if (p.epi == EPI_RESID) out = v + p.resid[m * p.ldr + n];
        else out = v;
        if (p.y) p.y[m * p.ldy + n] = out;
        if (p.ybf) p.ybf[m * p.ldybf + n] = __float2bfloat16_rn(out);
    }
}

}  // namespace tc

// ------------------------------------------------------------------------------------------ host
static PFN_cuTensorMapEncodeTiled_v12000 tma_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void* f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
    return fn;
}

// 2-D bf16 tensor map over a row-major [rows, cols] matrix with row stride `ld` elements; box = 64 x box_rows.
bool make_tma_2d(CUtensorMap* map, const void* ptr, long rows, long cols, long ld, int box_rows) {
    auto enc = tma_encoder();
    if (!enc || !ptr || ((uintptr_t)ptr & 15) || (ld * 2) % 16 || cols % 8) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    cuuint32_t box[2] = {(cuuint32_t)tc::BK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A row-major bf16 matrix [rows, cols] viewed as 64-column chunks: dimension 0 the 64 columns of a chunk,
// dimension 1 the rows, dimension 2 the chunk index (stride 128 B), so one box of box_rows rows and
// box_chunks chunks lands in shared memory chunk-major: [chunk][row][64 columns], 128-byte swizzled.
bool make_tma_chunks(CUtensorMap* map, const void* ptr, long rows, long cols, int box_rows, int box_chunks) {
    auto enc = tma_encoder();
    if (!enc || !ptr || ((uintptr_t)ptr & 15) || cols % 64) return false;
    cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(cols / 64)};
    cuuint64_t strides[2] = {(cuuint64_t)cols * 2, 128};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, (cuuint32_t)box_chunks};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN>
static cudaError_t tc_launch_persist(const TcParams& p, int ctas, cudaStream_t st) {
    using C = tc::PCfg<BN>;
    cudaError_t e = smem_optin((const void*)tc::tc_gemm_persist_kernel<BN>, (int)C::SMEM);
    if (e != cudaSuccess) return e;
    return launch_pdl(tc::tc_gemm_persist_kernel<BN>, dim3(ctas), dim3(tc::kThreads), (size_t)C::SMEM, st, p);
}

template <int BN, int MODE>
static cudaError_t tc_launch_bn(const TcParams& p, dim3 grid, cudaStream_t st) {
    using C = tc::Cfg<BN, MODE>;
    {
        cudaError_t e = smem_optin((const void*)tc::tc_gemm_kernel<BN, MODE>, (int)C::SMEM);
        if (e != cudaSuccess) return e;
    }
    cudaError_t le = launch_pdl(tc::tc_gemm_kernel<BN, MODE>, grid, dim3(tc::kThreads), (size_t)C::SMEM, st, p);
    if (le != cudaSuccess) return le;
    return cudaGetLastError();
}

int tc_pick_bn(int M) {
    if (M <= 16) return 16;
    if (M <= 32) return 32;
    if (M <= 64) return 64;
    if (M <= 128) return 128;
    return 256;
}

cudaError_t launch_tc_gemm(TcParams& p, int bn, int splits, cudaStream_t st) {
    p.nkb = p.K / tc::BK;
    if (splits < 1 || p.nbatch > 1) splits = 1;
    if (p.nbatch < 1) p.nbatch = 1;
    p.kb_per_split = (p.nkb + splits - 1) / splits;
    splits = (p.nkb + p.kb_per_split - 1) / p.kb_per_split;
    p.splits = splits;
    const bool glu = p.epi == EPI_GLU;
    const bool pair = p.pair && bn == 256 && !glu && p.epi != EPI_ARGMAX && p.nbatch == 1;
    const int rows_per_cta = pair ? 2 * tc::BM : tc::BM;
    dim3 grid((p.N + rows_per_cta - 1) / rows_per_cta, (p.M + bn - 1) / bn, splits * p.nbatch);
    if (p.epi == EPI_ARGMAX) p.npart = grid.x;
    cudaError_t e;
    const long tiles = (long)grid.x * grid.y;
    if (p.persist > 0 && !pair && !glu && splits == 1 && p.nbatch == 1 && tiles > p.persist) {
        const int ctas = p.persist;
        switch (bn) {
            case 16: return tc_launch_persist<16>(p, ctas, st);
            case 32: return tc_launch_persist<32>(p, ctas, st);
            case 64: return tc_launch_persist<64>(p, ctas, st);
            case 128: return tc_launch_persist<128>(p, ctas, st);
            case 256: return tc_launch_persist<256>(p, ctas, st);
            default: return cudaErrorInvalidValue;
        }
    }
#define TC_CASE(B)                                                                                       \
    case B:                                                                                              \
        e = glu ? tc_launch_bn<B, tc::kGlu>(p, grid, st) : tc_launch_bn<B, tc::kSingle>(p, grid, st);   \
        break;
    if (pair) {
        e = tc_launch_bn<256, tc::kPair>(p, grid, st);
    } else switch (bn) {
        TC_CASE(16)
        TC_CASE(32)
        TC_CASE(64)
        TC_CASE(128)
        TC_CASE(256)
        default: return cudaErrorInvalidValue;
    }
#undef TC_CASE
    if (e != cudaSuccess || splits == 1) return e;
    const long total = (long)p.M * p.N;
    const long items = (p.N & 3) == 0 ? total / 4 : total;
    int blocks = (int)((items + 255) / 256);
    if (blocks > 4096) blocks = 4096;
    return launch_pdl(tc::tc_splitk_reduce, dim3(blocks), dim3(256), 0, st, p, splits, glu ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace e3
