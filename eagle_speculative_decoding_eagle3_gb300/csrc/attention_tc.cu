// Latent (absorbed MLA) decode attention on the 5th-generation tensor cores, for the DeepseekV3 geometry
// (128 heads, latent 512 + rope 64, bf16 cache).
//
// The head's one MLA layer ("Eagle3 DeepseekV3 in MAX" §4) attends over the one-layer latent cache
// ("max.pipelines.architectures.eagle3_deepseekV3", construct_kv_params).  For one row r and its slots
// t < n:  S[h, t] = sigma (q_lat[h] . c_t + q_pe[h] . k_t)  (the 576-wide dot product of the absorbed
// query with the cached row), P = softmax_t(S), O[h] = sum_t P[h, t] c_t (512 wide).  Split s of the row
// covers a fixed chunk of slots and writes O unnormalised with its (max, sum) for the split merge, or
// o_lat = O / sum itself when the row has one split.
//
// Design.  All 128 heads of a row are the MMA M dimension, so every staged cache tile feeds all heads
// once.  O for 128 heads x 512 columns in fp32 fills a whole TMEM (512 columns), leaving no room for
// the scores, so a pair of CTAs (a thread-block cluster of 2) shares each (row, split):
//   * CTA c holds O[:, 256c : 256c + 256) in TMEM columns [0, 256) and stages cache columns
//     [256c, 256c + 320) of each 64-slot tile (five 64-column chunks; the middle one by both);
//   * the scores are split over K: CTA 0 forms the partial dot products over columns [0, 288) and
//     CTA 1 over [288, 576) (tcgen05.mma, M 128, N 64 slots, K 16: 18 steps) into one TMEM score
//     buffer.  A CTA's 288 query columns are the MMA's A operand in TMEM (144 columns), so the shared
//     memory holds only cache tiles, P and the exchange buffers.  (An accumulation chain that took some
//     A steps from shared memory and others from TMEM gave wrong sums past its first tile; every step
//     here reads TMEM.)  The tensor core takes at least ~45 cycles per MMA whatever N is, so N = 64
//     slots per tile keeps the score steps at ~70% of its rate (N = 32 was 36%);
//   * CTA c owns the softmax of heads [64c, 64c + 64): the other CTA sends its partial scores for
//     those heads through distributed shared memory, the owner adds them, runs the online softmax
//     (thread = head, fp32, base 2) and writes the head's row of P (bf16) into both CTAs.  Each
//     transfer into the peer is one bulk shared-to-shared copy per tile (the 64 rows are staged
//     locally first) whose bytes complete a transaction count on the peer's mbarrier, so no thread
//     waits for cluster-wide visibility of its stores (a cluster-scope release costs about a
//     microsecond) and no warp issues a remote store per row (about 40 ns each);
//   * each CTA then accumulates its half of O += P V (M 128, N 256, K 64 slots; V is the MN-major B
//     operand read straight from the staged cache chunks).
// The running maximum is updated lazily (only when a tile's maximum exceeds it by more than 2^8), so
// O is rescaled in TMEM only on those rare tiles.
//
// Warps: 0 TMA producer (the cache tiles through the block table, one 3D box of five 64-column chunks
// per tile, a 4-deep ring; the shared memory goes to cache stages rather than to second P and exchange
// buffers, since a stage stays occupied until its tile's P V completes);
// 1 TMEM owner and MMA issuer; 2-5 query loaders, then score readers (TMEM lanes = heads; a warp either
// sends its heads' partial scores to the peer or owns their softmax); 6-9 rescale O rows when asked,
// zero the cache rows past the context in the last tile (their P is 0, but 0 x NaN would poison O), and
// write the output.  Every mbarrier wait is bounded; a wait that runs out sets EAGLE3_DEVERR_TIMEOUT and
// the CTA pair winds down without touching its outputs.
#include <float.h>
#include <math.h>
#include <string.h>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"
#include "../../include/eagle3.h"

namespace e3 {
namespace mla_tc {

constexpr int HEADS = 128;
constexpr int D = 576, DC = 512;
constexpr int T = 64;                  // slots per tile
constexpr int NCH = 5;                 // 64-column chunks staged per CTA
constexpr int KSPLIT = 288;            // score columns of CTA 0 (CTA 1 takes the rest)
constexpr int KSTEPS = KSPLIT / 16;
constexpr int STAGES = 4;
constexpr int NS = 1, NB = 1, NX = 1;  // score buffers (TMEM), P / alpha buffers, exchange buffers
constexpr float TAU = 8.f;             // lazy rescale threshold, in base-2 exponent units
constexpr int KV_CHUNK = T * 128;      // 8 KB: 64 rows x 64 bf16
constexpr int KV_STAGE = NCH * KV_CHUNK;
constexpr int P_BYTES = HEADS * 128;   // one 128 x 64 K-major bf16 tile per P buffer
constexpr int XROW = T + 4;            // floats per exchange row: 272 B, 16-byte aligned, bank-spread
constexpr int X_BYTES = 64 * XROW * 4;
constexpr int OFF_KV = 0;
constexpr int OFF_P = OFF_KV + STAGES * KV_STAGE;
constexpr int OFF_X = OFF_P + NB * P_BYTES;        // partial scores received from the peer
constexpr int OFF_XO = OFF_X + NX * X_BYTES;       // partial scores staged for the peer
constexpr int OFF_ALPHA = OFF_XO + NX * X_BYTES;
constexpr int OFF_LM = OFF_ALPHA + NB * HEADS * 4;
constexpr int OFF_BAR = OFF_LM + HEADS * 2 * 4;
// barriers
constexpr int B_KV_FULL = 0, B_KV_EMPTY = B_KV_FULL + STAGES, B_Q_FULL = B_KV_EMPTY + STAGES,
              B_S_FULL = B_Q_FULL + 1, B_S_EMPTY = B_S_FULL + NS, B_X_FULL = B_S_EMPTY + NS,
              B_X_EMPTY = B_X_FULL + NX, B_A_FULL = B_X_EMPTY + NX, B_R_DONE = B_A_FULL + NB,
              B_P_FREE = B_R_DONE + NB, B_O_READY = B_P_FREE + NB, B_LM_FULL = B_O_READY + 1,
              B_SEND_SYNC = B_LM_FULL + 1, B_OWN_SYNC = B_SEND_SYNC + 1, NBARS = B_OWN_SYNC + 1;
constexpr int OFF_MISC = OFF_BAR + NBARS * 8;          // tmem slot, abort flag
constexpr int SMEM = OFF_MISC + 16 + 1024;             // + alignment slack of the dynamic window
constexpr int TMEM_COLS = 512;
constexpr int QCOLS = KSPLIT / 2;                      // TMEM columns of a CTA's query part (bf16 pairs)
constexpr int TM_O = 0, TM_Q = 256, TM_S = 448;        // O half | query part | scores
constexpr int THREADS = 320;
// bytes a CTA receives through st.async: per tile the peer's partial scores of its 64 heads (x_full)
// and the peer's P rows and rescale factors of its 64 heads (a_full); at the end its final sums
constexpr uint32_t X_TX = X_BYTES, A_TX = 64 * (T * 2 + 4), LM_TX = 64 * 8;

// polls before a wait gives up: every wait here is on work of the same CTA pair that takes microseconds
constexpr uint32_t WAIT = 1u << 20;
static_assert(TM_Q + QCOLS <= TM_S && TM_S + NS * T <= TMEM_COLS, "TMEM columns");
static_assert(OFF_P % 1024 == 0 && KV_STAGE % 1024 == 0, "swizzle atoms 1024-aligned");
static_assert(SMEM <= 227 * 1024, "shared memory");

struct Params {
    AttnArgs a;
    CUtensorMap mkv;   // cache rows as 64-column chunks [chunk][row][64], box 5 chunks x 64 rows
};

}  // namespace mla_tc

using namespace tc;

__global__ void __launch_bounds__(mla_tc::THREADS, 1) attention_tc_kernel(const __grid_constant__ mla_tc::Params p) {
    using namespace mla_tc;
    pdl_trigger();
    const AttnArgs& a = p.a;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* base = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + OFF_BAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base + OFF_MISC + 4);
    auto bar = [&](int i) { return su32(&bars[i]); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t c = cluster_rank(), peer = c ^ 1u;
    const int s = blockIdx.x >> 1, r = blockIdx.y;

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) { mbar_init(bar(B_KV_FULL + i), 1); mbar_init(bar(B_KV_EMPTY + i), 1); }
        mbar_init(bar(B_Q_FULL), 4);   // the four query-loading warps
        for (int i = 0; i < NS; ++i) { mbar_init(bar(B_S_FULL + i), 1); mbar_init(bar(B_S_EMPTY + i), 4); }
        // x_full: armed with the expected bytes, completed by the peer's bulk copy; x_empty: one arrival
        // from the peer's owners once they have read it
        for (int i = 0; i < NX; ++i) { mbar_init(bar(B_X_FULL + i), 1); mbar_init(bar(B_X_EMPTY + i), 1); }
        // a_full: 64 owners here + the arming (the peer's bulk copy completes it); r_done: the four rescale
        // warps; p_free: the P V commits of both CTAs
        for (int i = 0; i < NB; ++i) {
            mbar_init(bar(B_A_FULL + i), 65);
            mbar_init(bar(B_R_DONE + i), 4);
            mbar_init(bar(B_P_FREE + i), 2);
        }
        mbar_init(bar(B_O_READY), 1);
        mbar_init(bar(B_LM_FULL), 2);   // the owners' final sums here (one arrival) + the arming
        // the two sending warps and the two owning warps meet on these (a bounded barrier: a warp that
        // gave up on a wait does not leave the other blocked)
        mbar_init(bar(B_SEND_SYNC), 64);
        mbar_init(bar(B_OWN_SYNC), 64);
        // the first uses of the receive barriers are armed here; later uses by an owner thread once the
        // previous use has been consumed
        for (int i = 0; i < NX; ++i) mbar_expect_tx(bar(B_X_FULL + i), X_TX);
        for (int i = 0; i < NB; ++i) mbar_expect_tx(bar(B_A_FULL + i), A_TX);
        mbar_expect_tx(bar(B_LM_FULL), LM_TX);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                     "r"(TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    cluster_sync();   // both CTAs' barriers exist before any remote arrival
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();

    const int b = a.row_seq[r], pos = a.row_pos[r], n = pos + 1;
    const int t0 = s * a.chunk, t1 = min(n, t0 + a.chunk);
    const int ntiles = t0 < t1 ? (t1 - t0 + T - 1) / T : 0;
    const float scale2 = a.sigma * 1.4426950408889634f;   // scores in base-2 exponent units
    unsigned char* kvs = base + OFF_KV;
    unsigned char* ps = base + OFF_P;
    float* xs = reinterpret_cast<float*>(base + OFF_X);
    float* xo = reinterpret_cast<float*>(base + OFF_XO);
    float* alpha_s = reinterpret_cast<float*>(base + OFF_ALPHA);
    float* lm = reinterpret_cast<float*>(base + OFF_LM);
    int issued = 0;

    if (ntiles > 0) {
        if (warp == 0) {
            // ------------------------------------------------------------ TMA producer
            if (lane == 0) {
                const int* bt = a.block_table + (long)b * a.max_pages;
                for (int i = 0; i < ntiles; ++i) {
                    const int st = i % STAGES;
                    if (!mbar_wait(bar(B_KV_EMPTY + st), ((i / STAGES) & 1) ^ 1, WAIT)) { *abort_flag = 1; break; }
                    if (*abort_flag) break;
                    const int tt = t0 + i * T;
                    const int pi = tt / a.page_size;
                    const int page = pi < a.max_pages ? bt[pi] : -1;
                    unsigned char* stage = kvs + st * KV_STAGE;
                    if (page >= 0 && page < a.num_pages) {
                        mbar_expect_tx(bar(B_KV_FULL + st), KV_STAGE);
                        const int row = page * a.page_size + tt % a.page_size;
                        tma_load_3d(su32(stage), &p.mkv, bar(B_KV_FULL + st), 0, row, 4 * (int)c);   // 5 chunks
                        ++issued;
                    } else {   // a page outside the cache reads as zeros and is flagged
                        for (int q = 0; q < KV_STAGE / 16; ++q)
                            reinterpret_cast<uint4*>(stage)[q] = make_uint4(0, 0, 0, 0);
                        set_err(a.err, EAGLE3_DEVERR_PAGE);
                        fence_proxy_async_cta();
                        mbar_arrive(bar(B_KV_FULL + st));
                    }
                }
            }
        } else if (warp == 1) {
            // ------------------------------------------------------------ MMA issuer
            if (lane == 0) {
                constexpr uint32_t idesc_s = instr_desc_mn(128, T, false);
                constexpr uint32_t idesc_pv = instr_desc_mn(128, 256, true);
                bool ok = mbar_wait(bar(B_Q_FULL), 0, WAIT);
                tc_fence_after();
                // Event loop: the scores of tile j go out as soon as their cache tile has landed and the
                // score buffer has been read, and P V of tile i as soon as its P rows are in place, so
                // neither waits behind the other (the tensor core runs them in issue order).
                int js = 0, ipv = 0;
                uint32_t idle = 0;
                while (ok && ipv < ntiles) {
                    bool progressed = false;
                    if (js < ntiles) {
                        const int st = js % STAGES, sb = js % NS;
                        if (mbar_try(bar(B_KV_FULL + st), (js / STAGES) & 1) &&
                            mbar_try(bar(B_S_EMPTY + sb), ((js / NS) & 1) ^ 1)) {
                            tc_fence_after();
                            const uint32_t stage = su32(kvs + st * KV_STAGE);
                            const uint32_t d = tmem + TM_S + T * sb;
                            // K step ks covers cache columns KSPLIT c + 16 ks: local chunk (col / 64 - 4c), step
                            // (col % 64) / 16 of its 128-byte rows; its query part is TMEM columns 8 ks ..
#pragma unroll
                            for (int ks = 0; ks < KSTEPS; ++ks) {
                                const int col = KSPLIT * (int)c + 16 * ks;
                                const int lc = col / 64 - 4 * (int)c, kk = (col % 64) / 16;
                                mma_bf16_ta(d, tmem + TM_Q + 8 * ks, smem_desc(stage + lc * KV_CHUNK) + 2 * kk, idesc_s,
                                            ks > 0 ? 1u : 0u);
                            }
                            mma_commit(bar(B_S_FULL + sb));
                            ++js;
                            progressed = true;
                        }
                    }
                    if (ipv < js) {
                        const int pb = ipv % NB, st = ipv % STAGES;
                        if (mbar_try(bar(B_R_DONE + pb), (ipv / NB) & 1)) {
                            tc_fence_after();
                            const uint32_t stage = su32(kvs + st * KV_STAGE);
#pragma unroll
                            for (int kk = 0; kk < T / 16; ++kk)
                                mma_bf16(tmem + TM_O, smem_desc(su32(ps + pb * P_BYTES)) + 2 * kk,
                                         smem_desc_mn(stage + kk * 16 * 128, KV_CHUNK), idesc_pv,
                                         (ipv > 0 || kk > 0) ? 1u : 0u);
                            mma_commit(bar(B_KV_EMPTY + st));
                            mma_commit_multicast(bar(B_P_FREE + pb), 0x3);
                            ++ipv;
                            progressed = true;
                        }
                    }
                    if (progressed) idle = 0;
                    else if (++idle > WAIT || *abort_flag) ok = false;
                }
                if (!ok) *abort_flag = 1;
                else mma_commit(bar(B_O_READY));
            }
        } else if (warp < 6) {
            // ------------------------------------------------------------ score readers / softmax owners
            const int q = warp & 3, h = 32 * q + lane;
            const bool own = (h >> 6) == (int)c;
            const bool arming = own && (h & 63) == 0;   // one owner thread re-arms the receive barriers
            const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16);
            {
                // this head's query part (the absorbed query, bf16, columns [KSPLIT c, KSPLIT c + KSPLIT))
                // into TMEM lane h as the A operand of the score MMAs: 144 columns of packed bf16 pairs
                const uint4* src = reinterpret_cast<const uint4*>(a.qa_bf + ((long)r * a.nh + h) * D + KSPLIT * c);
                for (int cc = 0; cc < QCOLS; cc += 16) {
                    uint32_t v[16];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint4 u = src[cc / 4 + j];
                        v[4 * j] = u.x; v[4 * j + 1] = u.y; v[4 * j + 2] = u.z; v[4 * j + 3] = u.w;
                    }
                    tmem_st16u(trow + TM_Q + cc, v);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_Q_FULL));
            }
            float m_ref = -INFINITY, l = 0.f;
            bool ok = true;
            uint32_t gsync = 0;   // uses of this warp pair's group barrier
            auto group_sync = [&](int which) -> bool {
                mbar_arrive(bar(which));
                const bool done = mbar_wait(bar(which), gsync & 1u, WAIT);
                ++gsync;
                return done;
            };
            for (int i = 0; i < ntiles; ++i) {
                const int sb = i % NS, xb = i % NX, pb = i % NB;
                ok = __all_sync(0xffffffffu, ok && !*abort_flag && mbar_wait(bar(B_S_FULL + sb), (i / NS) & 1, WAIT));
                if (!ok) break;
                tc_fence_after();
                float sv[T];
                tmem_ld32(trow + TM_S + T * sb, sv);
                tmem_ld32(trow + TM_S + T * sb + 32, sv + 32);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_S_EMPTY + sb));
                if (!own) {
                    // this lane's head belongs to the peer: stage the partial scores, then one thread copies
                    // the 64 rows into the peer's exchange buffer (the peer having read its previous
                    // contents also means the copy out of this staging buffer two tiles ago is done)
                    if (i >= NX && !mbar_wait_cluster(bar(B_X_EMPTY + xb), ((i / NX) & 1) ^ 1, WAIT)) { ok = false; }
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    float4* dst = reinterpret_cast<float4*>(xo + xb * (X_BYTES / 4) + (h - 64 * (int)peer) * XROW);
#pragma unroll
                    for (int j = 0; j < T / 4; ++j) dst[j] = make_float4(sv[4 * j], sv[4 * j + 1], sv[4 * j + 2], sv[4 * j + 3]);
                    fence_proxy_async_cta();
                    ok = __all_sync(0xffffffffu, group_sync(B_SEND_SYNC));
                    if (!ok) break;
                    if ((h & 63) == 0) {
                        bulk_copy_to_peer(mapa(su32(xs + xb * (X_BYTES / 4)), peer), su32(xo + xb * (X_BYTES / 4)), X_BYTES,
                                          mapa(bar(B_X_FULL + xb), peer));
                        bulk_commit();
                    }
                    continue;
                }
                // owned head: add the peer's partial, online softmax, P row into both CTAs
                ok = __all_sync(0xffffffffu, mbar_wait_cluster(bar(B_X_FULL + xb), (i / NX) & 1, WAIT));
                if (!ok) break;
                const float4* xr = reinterpret_cast<const float4*>(xs + xb * (X_BYTES / 4) + (h - 64 * (int)c) * XROW);
                const int cnt = min(T, t1 - (t0 + i * T));
#pragma unroll
                for (int j = 0; j < T / 4; ++j) {
                    const float4 v = xr[j];
                    sv[4 * j] = (sv[4 * j] + v.x) * scale2;
                    sv[4 * j + 1] = (sv[4 * j + 1] + v.y) * scale2;
                    sv[4 * j + 2] = (sv[4 * j + 2] + v.z) * scale2;
                    sv[4 * j + 3] = (sv[4 * j + 3] + v.w) * scale2;
                }
                if (cnt < T) {
#pragma unroll
                    for (int j = 0; j < T; ++j)
                        if (j >= cnt) sv[j] = -INFINITY;
                }
                float mx[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) mx[k] = sv[k];
#pragma unroll
                for (int j = 8; j < T; ++j) mx[j & 7] = fmaxf(mx[j & 7], sv[j]);
                const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
                float alpha = 1.f;
                if (m_ref == -INFINITY) {
                    m_ref = mt;
                } else if (mt > m_ref + TAU) {
                    alpha = exp2f(m_ref - mt);
                    l *= alpha;
                    m_ref = mt;
                }
                float ps8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int j = 0; j < T; ++j) {
                    sv[j] = ex2_approx(sv[j] - m_ref);   // P is rounded to bf16; exp2 to ~2 ulp is plenty
                    ps8[j & 7] += sv[j];
                }
                l += ((ps8[0] + ps8[1]) + (ps8[2] + ps8[3])) + ((ps8[4] + ps8[5]) + (ps8[6] + ps8[7]));
                // the previous use of this P buffer (tile i - NB) must be consumed in both CTAs
                ok = __all_sync(0xffffffffu, i < NB || mbar_wait_cluster(bar(B_P_FREE + pb), ((i / NB) & 1) ^ 1, WAIT));
                if (!ok) break;
                // tile i - NB's use of a_full[pb] is complete (its P V ran, which also means the copy of
                // this P buffer into the peer two tiles ago has landed): arm it for tile i
                if (arming && i >= NB) mbar_expect_tx(bar(B_A_FULL + pb), A_TX);
                unsigned char* prow = ps + pb * P_BYTES + h * 128;
#pragma unroll
                for (int j = 0; j < T / 8; ++j) {
                    const uint4 chunk = make_uint4(pack2_bf16(sv[8 * j], sv[8 * j + 1]), pack2_bf16(sv[8 * j + 2], sv[8 * j + 3]),
                                                   pack2_bf16(sv[8 * j + 4], sv[8 * j + 5]), pack2_bf16(sv[8 * j + 6], sv[8 * j + 7]));
                    *reinterpret_cast<uint4*>(prow + ((j ^ (h & 7)) << 4)) = chunk;
                }
                alpha_s[pb * HEADS + h] = alpha;
                fence_proxy_async_cta();
                ok = __all_sync(0xffffffffu, group_sync(B_OWN_SYNC));
                if (!ok) break;
                if (arming) {
                    // this CTA's 64 P rows (contiguous: 128 B each) and rescale factors into the peer
                    const uint32_t abar = mapa(bar(B_A_FULL + pb), peer);
                    const uint32_t prows = su32(ps + pb * P_BYTES + 64 * (int)c * 128);
                    const uint32_t arows = su32(alpha_s + pb * HEADS + 64 * (int)c);
                    bulk_copy_to_peer(mapa(prows, peer), prows, 64 * T * 2, abar);
                    bulk_copy_to_peer(mapa(arows, peer), arows, 64 * 4, abar);
                    bulk_commit();
                    // X[xb] is consumed (its values went into P): re-arm it for tile i + NX, then let the
                    // peer overwrite it
                    if (i + NX < ntiles) mbar_expect_tx(bar(B_X_FULL + xb), X_TX);
                    mbar_arrive_remote_cta(mapa(bar(B_X_EMPTY + xb), peer));
                }
                mbar_arrive(bar(B_A_FULL + pb));
            }
            if (!ok) *abort_flag = 1;
            if (own && ok) {
                lm[2 * h] = l;
                lm[2 * h + 1] = m_ref;
                fence_proxy_async_cta();
                if (!__all_sync(0xffffffffu, group_sync(B_OWN_SYNC))) *abort_flag = 1;
                if (a.splits > 1) {
                    const long pr = ((long)r * a.nh + h) * a.splits + s;
                    a.part_ml[2 * pr] = m_ref * 0.6931471805599453f;   // natural-log units
                    a.part_ml[2 * pr + 1] = l;
                }
                if (arming) {
                    const uint32_t rows = su32(lm + 128 * (int)c);   // this CTA's 64 heads: 512 B
                    bulk_copy_to_peer(mapa(rows, peer), rows, LM_TX, mapa(bar(B_LM_FULL), peer));
                    bulk_commit();
                    mbar_arrive(bar(B_LM_FULL));
                }
            }
            // the bulk copies this thread issued have read their sources before the shared memory goes
            bulk_wait_read_all();
        } else {
            // ------------------------------------------------------------ rescale / tail fix-up / output
            const int q = warp & 3, h = 32 * q + lane;
            const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16);
            const int tid = threadIdx.x - 192;   // 0..127
            bool ok = true;
            for (int i = 0; i < ntiles; ++i) {
                const int pb = i % NB, st = i % STAGES;
                ok = __all_sync(0xffffffffu, ok && !*abort_flag && mbar_wait_cluster(bar(B_A_FULL + pb), (i / NB) & 1, WAIT));
                if (!ok) break;
                const float alpha = alpha_s[pb * HEADS + h];
                if (__any_sync(0xffffffffu, alpha != 1.f)) {
                    // O += P V of tile i - 1 must have landed before its rows are scaled
                    ok = __all_sync(0xffffffffu, mbar_wait_cluster(bar(B_P_FREE + (i - 1) % NB), ((i - 1) / NB) & 1, WAIT));
                    if (!ok) break;
                    tc_fence_after();
                    for (int cc = 0; cc < 256; cc += 32) {
                        float v[32];
                        tmem_ld32(trow + TM_O + cc, v);
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] *= alpha;
                        tmem_st32(trow + TM_O + cc, v);
                    }
                    tmem_wait_st();
                }
                const int cnt = min(T, t1 - (t0 + i * T));
                if (cnt < T) {   // cache rows past the context: zero the value chunks of this CTA
                    unsigned char* stage = kvs + st * KV_STAGE;
                    const int per_chunk = (T - cnt) * 8;          // 16-byte pieces per chunk
                    for (int w = tid; w < 4 * per_chunk; w += 128) {
                        const int lc = w / per_chunk, rem = w % per_chunk;
                        const int row = cnt + rem / 8, piece = rem % 8;
                        *reinterpret_cast<uint4*>(stage + lc * KV_CHUNK + row * 128 + piece * 16) = make_uint4(0, 0, 0, 0);
                    }
                }
                // the P rows (written here and, through st.async, by the peer) and the zeroed rows are read
                // by the tensor core next
                fence_proxy_async_cta();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_R_DONE + pb));
            }
            ok = __all_sync(0xffffffffu, ok && mbar_wait(bar(B_O_READY), 0, WAIT) && mbar_wait_cluster(bar(B_LM_FULL), 0, WAIT));
            if (!ok) {
                *abort_flag = 1;
            } else {
                tc_fence_after();
                const float l = lm[2 * h];
                const float inv = l > 0.f ? 1.f / l : 0.f;
                const long rowbase = ((long)r * a.nh + h) * DC + 256 * c;
                for (int cc = 0; cc < 256; cc += 32) {
                    float v[32];
                    tmem_ld32(trow + TM_O + cc, v);
                    if (a.splits == 1) {
                        if (a.olat) {
                            float4* d4 = reinterpret_cast<float4*>(a.olat + rowbase + cc);
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                d4[j] = make_float4(v[4 * j] * inv, v[4 * j + 1] * inv, v[4 * j + 2] * inv, v[4 * j + 3] * inv);
                        }
                        if (a.olat_bf) {
                            uint4* d4 = reinterpret_cast<uint4*>(a.olat_bf + rowbase + cc);
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                d4[j] = make_uint4(pack2_bf16(v[8 * j] * inv, v[8 * j + 1] * inv),
                                                   pack2_bf16(v[8 * j + 2] * inv, v[8 * j + 3] * inv),
                                                   pack2_bf16(v[8 * j + 4] * inv, v[8 * j + 5] * inv),
                                                   pack2_bf16(v[8 * j + 6] * inv, v[8 * j + 7] * inv));
                        }
                    } else {
                        const long pr = ((long)r * a.nh + h) * a.splits + s;
                        float4* d4 = reinterpret_cast<float4*>(a.part_o + pr * DC + 256 * c + cc);
#pragma unroll
                        for (int j = 0; j < 8; ++j) d4[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
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
            for (int i = max(0, issued - STAGES); i < issued; ++i)
                mbar_wait(bar(B_KV_FULL + i % STAGES), (uint32_t)(i / STAGES) & 1u, WAIT);
        }
        __syncthreads();
    }
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS));
    }
    cluster_sync();   // neither CTA leaves while the other may still write into its shared memory
}

// ------------------------------------------------------------------------------------------ host
bool attention_tc_supported(const AttnArgs& a) {
    return a.dt == BF16 && a.nh == mla_tc::HEADS && a.dc == mla_tc::DC && a.dr == mla_tc::D - mla_tc::DC &&
           a.page_size % mla_tc::T == 0 && a.qa_bf != nullptr && a.chunk > 0 && a.chunk % mla_tc::T == 0 &&
           ((uintptr_t)a.cache & 15u) == 0 && ((uintptr_t)a.qa_bf & 15u) == 0;
}

cudaError_t launch_attention_tc(const AttnArgs& a, cudaStream_t st) {
    using namespace mla_tc;
    if (!attention_tc_supported(a)) return cudaErrorInvalidValue;
    Params p;
    memset(&p, 0, sizeof(p));
    p.a = a;
    if (!make_tma_chunks(&p.mkv, a.cache, (long)a.num_pages * a.page_size, D, T, NCH)) return cudaErrorInvalidValue;
    cudaError_t e = smem_optin((const void*)attention_tc_kernel, SMEM);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * a.splits, a.M);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = SMEM;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, attention_tc_kernel, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace e3
