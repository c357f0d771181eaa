// Causal attention of a long extend on the 5th-generation tensor cores (unabsorbed keys and values of
// the DeepseekV3 geometry: q/k 192 = nope 128 + rope 64, v 128).
//
// The draft layer is one DeepseekV3 decoder layer ("Eagle3 DeepseekV3 in MAX" §4); over an extend, each
// new row at position p attends to its sequence's slots 0..p (MLAPrefillMetadata: causal prefill).  The
// keys and values of every slot are expanded once (kv_gather + the kv_b GEMM, prefill_attention.cu) and
// this kernel runs flash attention over them:
//   * one CTA per (128-row query tile of one sequence, head); the query tile is the MMA M dimension;
//   * 128-slot key/value tiles staged by TMA into a 2-deep ring: K = [k_nope | k_pe] (three 64-column
//     chunks, k_pe shared by all heads), V (two chunks);
//   * S = Q K^T (tcgen05.mma M 128, N 128, K 16: 12 steps, A = Q from shared memory) into one of two TMEM
//     score buffers;
//   * one softmax thread per query row (TMEM lane = row): causal mask t <= p, online softmax in base 2
//     with a lazily updated maximum, P rounded to bf16 and written back into TMEM;
//   * O += P V (M 128, N 128, K 16: 8 steps, A = P from TMEM, B = V MN-major from the staged chunks),
//     O in TMEM; each accumulation chain reads its A operand from one place only.
// Key tiles above the diagonal are never loaded (a query tile stops at its last row's position).  Rows of
// a partial query tile past the sequence see no slot and write nothing.  Every mbarrier wait is bounded;
// a wait that runs out sets EAGLE3_DEVERR_TIMEOUT and the CTA winds down without writing its rows.
#include <float.h>
#include <math.h>
#include <string.h>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"
#include "../../include/eagle3.h"

namespace e3 {
namespace pft {

constexpr int BQ = 128;                 // query rows per tile (MMA M)
constexpr int BKV = 128;                // slots per key/value tile (MMA N of the scores)
constexpr int DN = 128, DR = 64, DQK = 192, DV = 128;
constexpr int CHUNK = 128 * 128;        // one 64-column, 128-row bf16 chunk, 128-byte swizzled: 16 KB
constexpr int Q_BYTES = 3 * CHUNK;      // [q_nope | q_pe]
constexpr int K_BYTES = 3 * CHUNK;      // [k_nope | k_pe]
constexpr int V_BYTES = 2 * CHUNK;
constexpr int STAGE = K_BYTES + V_BYTES;
constexpr int STAGES = 2;
constexpr int OFF_Q = 0;
constexpr int OFF_KV = OFF_Q + Q_BYTES;
constexpr int OFF_BAR = OFF_KV + STAGES * STAGE;
// barriers: q_full, kv_full[2], kv_empty[2], s_full[2], s_empty[2], p_full[2], p_empty[2], o_done, o_full
constexpr int B_Q = 0, B_KV_FULL = 1, B_KV_EMPTY = 3, B_S_FULL = 5, B_S_EMPTY = 7, B_P_FULL = 9, B_P_EMPTY = 11,
              B_O_DONE = 13, B_O_FULL = 14, NBARS = 15;
constexpr int OFF_MISC = OFF_BAR + NBARS * 8;
constexpr int SMEM = OFF_MISC + 16 + 1024;
constexpr int TMEM_COLS = 512;
constexpr int TM_S = 0, TM_O = 256, TM_P = 384;   // two score buffers | O | two P buffers (bf16 pairs)
constexpr int THREADS = 192;                      // warp 0 TMA, warp 1 MMA, warps 2-5 softmax
constexpr float TAU = 8.f;                        // lazy rescale threshold (base-2 exponent units)
constexpr uint32_t WAIT = 1u << 22;
static_assert(SMEM <= 227 * 1024, "shared memory");
static_assert(OFF_KV % 1024 == 0 && STAGE % 1024 == 0, "swizzle atoms 1024-aligned");

struct Params {
    PrefillArgs a;
    CUtensorMap mq;    // q rows [M, nh * 192], box 64 x 128
    CUtensorMap mkv;   // expanded [k_nope | v] rows [B * max_ctx, nh * 256], box 64 x 128
    CUtensorMap mpe;   // rotated k_pe rows [B * max_ctx, 64], box 64 x 128
};

}  // namespace pft

using namespace tc;

__global__ void __launch_bounds__(pft::THREADS, 1) prefill_tc_kernel(const __grid_constant__ pft::Params p) {
    using namespace pft;
    pdl_trigger();
    const PrefillArgs& a = p.a;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* base = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + OFF_BAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base + OFF_MISC + 4);
    auto bar = [&](int i) { return su32(&bars[i]); };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.y;

    if (threadIdx.x == 0) {
        mbar_init(bar(B_Q), 1);
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(bar(B_KV_FULL + i), 1);
            mbar_init(bar(B_KV_EMPTY + i), 1);
            mbar_init(bar(B_S_FULL + i), 1);
            mbar_init(bar(B_S_EMPTY + i), 4);
            mbar_init(bar(B_P_FULL + i), 4);
            mbar_init(bar(B_P_EMPTY + i), 1);
        }
        mbar_init(bar(B_O_DONE), 1);
        mbar_init(bar(B_O_FULL), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                     "r"(TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();

    const int4 tile = a.tiles[blockIdx.x];
    const int b = tile.x, r0 = tile.y, nrow = tile.z;
    // positions ascend within a sequence: the tile's last row sees the most slots
    const int pmax = b >= 0 ? min(a.row_pos[r0 + nrow - 1], a.max_ctx - 1) : -1;
    const int nkv = b >= 0 ? pmax / BKV + 1 : 0;
    const int kvrow0 = b >= 0 ? b * a.max_ctx : 0;
    unsigned char* qs = base + OFF_Q;
    unsigned char* kvs = base + OFF_KV;
    int issued = 0;

    if (nkv > 0) {
        if (warp == 0) {
            // ------------------------------------------------------------ TMA producer
            if (lane == 0) {
                mbar_expect_tx(bar(B_Q), Q_BYTES);
                for (int c = 0; c < 3; ++c) tma_load_2d(su32(qs + c * CHUNK), &p.mq, bar(B_Q), h * DQK + 64 * c, r0);
                for (int j = 0; j < nkv; ++j) {
                    const int st = j % STAGES;
                    if (!mbar_wait(bar(B_KV_EMPTY + st), ((j / STAGES) & 1) ^ 1, WAIT)) { *abort_flag = 1; break; }
                    if (*abort_flag) break;
                    unsigned char* sp = kvs + st * STAGE;
                    const uint32_t fb = bar(B_KV_FULL + st);
                    const int row = kvrow0 + j * BKV;
                    mbar_expect_tx(fb, STAGE);
                    tma_load_2d(su32(sp), &p.mkv, fb, h * (DN + DV), row);                       // k_nope 0..63
                    tma_load_2d(su32(sp + CHUNK), &p.mkv, fb, h * (DN + DV) + 64, row);          // k_nope 64..127
                    tma_load_2d(su32(sp + 2 * CHUNK), &p.mpe, fb, 0, row);                       // k_pe
                    tma_load_2d(su32(sp + 3 * CHUNK), &p.mkv, fb, h * (DN + DV) + DN, row);      // v 0..63
                    tma_load_2d(su32(sp + 4 * CHUNK), &p.mkv, fb, h * (DN + DV) + DN + 64, row); // v 64..127
                    ++issued;
                }
            }
        } else if (warp == 1) {
            // ------------------------------------------------------------ MMA issuer (event loop)
            if (lane == 0) {
                constexpr uint32_t idesc_s = instr_desc_mn(128, BKV, false);
                constexpr uint32_t idesc_pv = instr_desc_mn(128, DV, true);
                bool ok = mbar_wait(bar(B_Q), 0, WAIT);
                int js = 0, jp = 0;
                uint32_t idle = 0;
                while (ok && jp < nkv) {
                    bool progressed = false;
                    if (js < nkv) {
                        const int st = js % STAGES, sb = js % 2;
                        if (mbar_try(bar(B_KV_FULL + st), (js / STAGES) & 1) &&
                            mbar_try(bar(B_S_EMPTY + sb), ((js / 2) & 1) ^ 1)) {
                            tc_fence_after();
                            const uint32_t sp = su32(kvs + st * STAGE);
#pragma unroll
                            for (int ks = 0; ks < DQK / 16; ++ks) {
                                const int c = ks / 4, kk = ks % 4;
                                mma_bf16(tmem + TM_S + BKV * sb, smem_desc(su32(qs + c * CHUNK)) + 2 * kk,
                                         smem_desc(sp + c * CHUNK) + 2 * kk, idesc_s, ks > 0 ? 1u : 0u);
                            }
                            mma_commit(bar(B_S_FULL + sb));
                            ++js;
                            progressed = true;
                        }
                    }
                    if (jp < js) {
                        const int st = jp % STAGES, pb = jp % 2;
                        if (mbar_try(bar(B_P_FULL + pb), (jp / 2) & 1)) {
                            tc_fence_after();
                            const uint32_t vp = su32(kvs + st * STAGE + K_BYTES);
#pragma unroll
                            for (int kk = 0; kk < BKV / 16; ++kk)
                                mma_bf16_ta(tmem + TM_O, tmem + TM_P + 64 * pb + 8 * kk,
                                            smem_desc_mn(vp + kk * 16 * 128, CHUNK), idesc_pv, (jp > 0 || kk > 0) ? 1u : 0u);
                            mma_commit(bar(B_KV_EMPTY + st));
                            mma_commit(bar(B_P_EMPTY + pb));
                            mma_commit(bar(B_O_DONE));
                            ++jp;
                            progressed = true;
                        }
                    }
                    if (progressed) idle = 0;
                    else if (++idle > WAIT || *abort_flag) ok = false;
                }
                if (!ok) *abort_flag = 1;
                else mma_commit(bar(B_O_FULL));
            }
        } else {
            // ------------------------------------------------------------ softmax: one thread per query row
            const int q = warp & 3, row = 32 * q + lane;
            const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16);
            const int pos = row < nrow ? min(a.row_pos[r0 + row], a.max_ctx - 1) : -1;   // -1: sees no slot
            const float scale2 = a.sigma * 1.4426950408889634f;
            float m_ref = -INFINITY, l = 0.f;
            bool ok = true;
            for (int j = 0; j < nkv; ++j) {
                const int sb = j % 2;
                ok = __all_sync(0xffffffffu, ok && !*abort_flag && mbar_wait(bar(B_S_FULL + sb), (j / 2) & 1, WAIT));
                if (!ok) break;
                tc_fence_after();
                float s[BKV];
#pragma unroll
                for (int c = 0; c < BKV; c += 32) tmem_ld32(trow + TM_S + BKV * sb + c, s + c);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_S_EMPTY + sb));
                // causal mask (slot t visible when t <= pos), scale, tile maximum (eight partial maxima)
                const int t0 = j * BKV;
                float mx[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) mx[k] = -INFINITY;
#pragma unroll
                for (int k = 0; k < BKV; ++k) {
                    s[k] = t0 + k <= pos ? s[k] * scale2 : -INFINITY;
                    mx[k & 7] = fmaxf(mx[k & 7], s[k]);
                }
                const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                       fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
                float alpha = 1.f;
                if (m_ref == -INFINITY) {
                    m_ref = mt;
                } else if (mt > m_ref + TAU) {
                    alpha = exp2f(m_ref - mt);
                    l *= alpha;
                    m_ref = mt;
                }
                const bool live = m_ref != -INFINITY;   // false only for rows past the sequence
                float ps[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) ps[k] = 0.f;
#pragma unroll
                for (int k = 0; k < BKV; ++k) {
                    s[k] = live ? ex2_approx(s[k] - m_ref) : 0.f;   // P is rounded to bf16; ~2 ulp exp2 is plenty
                    ps[k & 7] += s[k];
                }
                l += ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
                // the P buffer's previous tile (j - 2) has been consumed by its P V
                ok = __all_sync(0xffffffffu, j < 2 || mbar_wait(bar(B_P_EMPTY + sb), ((j / 2) & 1) ^ 1, WAIT));
                if (!ok) break;
                if (__any_sync(0xffffffffu, alpha != 1.f)) {
                    // O += P V of tile j - 1 has landed before its rows are scaled
                    ok = __all_sync(0xffffffffu, mbar_wait(bar(B_O_DONE), (j - 1) & 1, WAIT));
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < DV; c += 32) {
                        float v[32];
                        tmem_ld32(trow + TM_O + c, v);
#pragma unroll
                        for (int k = 0; k < 32; ++k) v[k] *= alpha;
                        tmem_st32(trow + TM_O + c, v);
                    }
                }
                // P (bf16 pairs, the even slot in the low half) into this row's TMEM lane: the A operand of P V
#pragma unroll
                for (int c = 0; c < BKV; c += 32) {
                    uint32_t pk[16];
#pragma unroll
                    for (int k = 0; k < 16; ++k) pk[k] = pack2_bf16(s[c + 2 * k], s[c + 2 * k + 1]);
                    tmem_st16u(trow + TM_P + 64 * sb + c / 2, pk);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_P_FULL + sb));
            }
            ok = __all_sync(0xffffffffu, ok && mbar_wait(bar(B_O_FULL), 0, WAIT));
            if (!ok) {
                *abort_flag = 1;
            } else {
                tc_fence_after();
                const float inv = l > 0.f ? 1.f / l : 0.f;
                bf16* dst = a.o_bf + (long)(r0 + row) * a.nh * DV + (long)h * DV;
#pragma unroll 1
                for (int c = 0; c < DV; c += 32) {
                    float v[32];
                    tmem_ld32(trow + TM_O + c, v);   // warp-collective: every lane takes part
                    if (row < nrow) {
                        uint4* d4 = reinterpret_cast<uint4*>(dst + c);
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            d4[k] = make_uint4(pack2_bf16(v[8 * k] * inv, v[8 * k + 1] * inv),
                                               pack2_bf16(v[8 * k + 2] * inv, v[8 * k + 3] * inv),
                                               pack2_bf16(v[8 * k + 4] * inv, v[8 * k + 5] * inv),
                                               pack2_bf16(v[8 * k + 6] * inv, v[8 * k + 7] * inv));
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {
        if (threadIdx.x == 0) atomicOr(a.err, EAGLE3_DEVERR_TIMEOUT);
        // this CTA's own copies still in flight land before its shared memory goes away (bounded)
        if (warp == 0 && lane == 0) {
            mbar_wait(bar(B_Q), 0, WAIT);
            for (int j = max(0, issued - STAGES); j < issued; ++j)
                mbar_wait(bar(B_KV_FULL + j % STAGES), (uint32_t)(j / STAGES) & 1u, WAIT);
        }
        __syncthreads();
    }
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS));
    }
}

// ------------------------------------------------------------------------------------------ host
bool prefill_tc_supported(const PrefillArgs& a) {
    return a.nh >= 1 && a.bq == pft::BQ && ((uintptr_t)a.q & 15u) == 0 && ((uintptr_t)a.kv & 15u) == 0 &&
           ((uintptr_t)a.xpe & 15u) == 0 && ((uintptr_t)a.o_bf & 15u) == 0;
}

cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t st) {
    using namespace pft;
    if (!prefill_tc_supported(a)) return cudaErrorInvalidValue;
    Params p;
    memset(&p, 0, sizeof(p));
    p.a = a;
    const long kvrows = (long)a.B * a.max_ctx;
    if (!make_tma_2d(&p.mq, a.q, a.M, (long)a.nh * DQK, (long)a.nh * DQK, BQ)) return cudaErrorInvalidValue;
    if (!make_tma_2d(&p.mkv, a.kv, kvrows, (long)a.nh * (DN + DV), (long)a.nh * (DN + DV), BKV))
        return cudaErrorInvalidValue;
    if (!make_tma_2d(&p.mpe, a.xpe, kvrows, DR, DR, BKV)) return cudaErrorInvalidValue;
    cudaError_t e = smem_optin((const void*)prefill_tc_kernel, SMEM);
    if (e != cudaSuccess) return e;
    return launch_pdl(prefill_tc_kernel, dim3(a.ntiles_cap, a.nh), dim3(THREADS), (size_t)SMEM, st, p);
}

}  // namespace e3
