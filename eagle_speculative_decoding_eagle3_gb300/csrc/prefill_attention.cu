// Causal MLA attention of a long extend, in unabsorbed form.
//
// The draft layer is one DeepseekV3 decoder layer ("Eagle3 DeepseekV3 in MAX" §4); over an extend,
// each new row at position p attends to its sequence's slots 0..p: the cached prefix and the new rows
// up to itself.  Per (row, head, slot) the absorbed form used for decode costs 2 x (576 + 512) FLOPs
// against the latent row; materialising keys and values costs 2 x (192 + 128), plus one expansion of
// every slot.  When an extend brings many rows per sequence the expansion is shared by all of them, so
// this path expands once and runs flash-attention tiles:
//   1. kv_gather_kernel packs every slot t < L_b of every sequence into X_c [B * max_ctx, d_c] and
//      X_pe [B * max_ctx, d_r] (bf16, zeros for t >= L_b);
//   2. the tensor-core GEMM KV = X_c kv_b^T gives, per slot and head, [k_nope (d_n) | v (d_v)] in bf16
//      (kv_b rows per head: W_UK then W_UV);
//   3. rope_q_rows_kernel rotates q_pe inside the bf16 query rows, so row r, head h holds
//      [q_nope | RoPE(q_pe, pos_r)];
//   4. prefill_attention_kernel: one CTA per (tile of 64 query rows of one sequence, head).  S = Q K^T
//      with K = [k_nope | k_pe] on mma.sync m16n8k16, causal mask t <= pos, online softmax in
//      registers, O += P V with P re-used from the score registers as the A operand, then
//      o_h = O / l in bf16 for o_proj.  No split merge and no value up-projection follow.
// Geometry: d_n 128, d_r 64, d_v 128 (DeepseekV3); other geometries keep the absorbed path.
#include <float.h>
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "mma_sync.cuh"

namespace e3 {

namespace pf {
constexpr int BQ = 64;           // query rows per CTA: 4 warps x 16
constexpr int BKV = 64;          // slots per key/value tile
constexpr int DN = 128, DR = 64, DQK = 192, DV = 128;
constexpr int QROW = DQK + 8;    // bf16 stride of Q and K rows (400 B: ldmatrix rows hit distinct banks)
constexpr int VROW = DV + 8;     // bf16 stride of V rows (272 B)
constexpr int WARPS = 4;
constexpr int THREADS = WARPS * 32;
constexpr size_t SMEM = ((size_t)BQ * QROW + 2 * (size_t)BKV * QROW + 2 * (size_t)BKV * VROW) * 2;
constexpr int kGatherSlots = 8;  // slots per CTA of the gather
}  // namespace pf

bool prefill_supported(int dt, int dn, int dr, int dv) {
    return dt == BF16 && dn == pf::DN && dr == pf::DR && dv == pf::DV;
}

// Length after this extend of sequence b: its last new row's position + 1 (0 without new rows).
__device__ __forceinline__ int extend_length(const PrefillArgs& a, int b) {
    const int r0 = max(0, min(a.M, a.row_offsets[b])), r1 = max(r0, min(a.M, a.row_offsets[b + 1]));
    return r1 > r0 ? min(a.max_ctx, a.row_pos[r1 - 1] + 1) : 0;
}

// X_c / X_pe rows of slots [blockIdx.x * kGatherSlots, + kGatherSlots) of sequence blockIdx.y.
__global__ void __launch_bounds__(256) kv_gather_kernel(const PrefillArgs a) {
    pdl_trigger();
    pdl_wait();
    constexpr int CH = (512 + 64) / 8;   // 16-byte chunks per latent row
    const int b = blockIdx.y, t0 = blockIdx.x * pf::kGatherSlots;
    const int len = extend_length(a, b);
    const bf16* cache = reinterpret_cast<const bf16*>(a.cache);
    for (int c = threadIdx.x; c < pf::kGatherSlots * CH; c += blockDim.x) {
        const int j = c / CH, q = c % CH, t = t0 + j;
        if (t >= a.max_ctx) continue;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (t < len) {
            const int pg = t / a.page_size;
            const int page = pg < a.max_pages ? a.block_table[(long)b * a.max_pages + pg] : -1;
            if (page >= 0 && page < a.num_pages)
                v = *reinterpret_cast<const uint4*>(cache + ((long)page * a.page_size + t % a.page_size) * 576 + 8 * q);
            else if (q == 0)
                set_err(a.err, 8);
        }
        const long row = (long)b * a.max_ctx + t;
        if (q < 64) *reinterpret_cast<uint4*>(a.xc + row * 512 + 8 * q) = v;
        else *reinterpret_cast<uint4*>(a.xpe + row * 64 + 8 * (q - 64)) = v;
    }
}

// Tile map: for each sequence its ceil(T_b / bq) query tiles, last (heaviest) first; unused entries
// get sequence -1.  One CTA; thread 0 scans the tile counts.
__global__ void __launch_bounds__(256) prefill_tiles_kernel(const PrefillArgs a) {
    pdl_trigger();
    pdl_wait();
    extern __shared__ int start[];   // [B + 1] first tile index of each sequence
    if (threadIdx.x == 0) {
        int acc = 0;
        for (int b = 0; b < a.B; ++b) {
            start[b] = acc;
            const int r0 = max(0, min(a.M, a.row_offsets[b])), r1 = max(r0, min(a.M, a.row_offsets[b + 1]));
            acc += (r1 - r0 + a.bq - 1) / a.bq;
        }
        start[a.B] = min(acc, a.ntiles_cap);
    }
    __syncthreads();
    for (int b = threadIdx.x; b < a.B; b += blockDim.x) {
        const int r0 = max(0, min(a.M, a.row_offsets[b])), r1 = max(r0, min(a.M, a.row_offsets[b + 1]));
        const int nt = (r1 - r0 + a.bq - 1) / a.bq;
        for (int i = 0; i < nt; ++i) {
            const int idx = start[b] + (nt - 1 - i);
            if (idx >= a.ntiles_cap) continue;
            const int row = r0 + i * a.bq;
            a.tiles[idx] = make_int4(b, row, min(a.bq, r1 - row), 0);
        }
    }
    for (int i = start[a.B] + threadIdx.x; i < a.ntiles_cap; i += blockDim.x) a.tiles[i] = make_int4(-1, 0, 0, 0);
}

// q_bf[r, h, d_n:] = RoPE(q[r, h, d_n:], pos_r) in bf16 (interleaved pairs).
__global__ void __launch_bounds__(256) rope_q_rows_kernel(const PrefillArgs a) {
    pdl_trigger();
    pdl_wait();
    const int r = blockIdx.x;
    const int half = pf::DR / 2;
    const int pos = min(max(a.row_pos[r], 0), a.max_ctx - 1);
    for (int t = threadIdx.x; t < a.nh * half; t += blockDim.x) {
        const int h = t / half, p = t % half;
        const float c = a.rope_cos[(long)pos * half + p], s = a.rope_sin[(long)pos * half + p];
        const long o = ((long)r * a.nh + h) * pf::DQK + pf::DN + 2 * p;
        const float x0 = a.qf ? a.qf[o] : __bfloat162float(a.q[o]);
        const float x1 = a.qf ? a.qf[o + 1] : __bfloat162float(a.q[o + 1]);
        *reinterpret_cast<uint32_t*>(a.q + o) = pack_bf16(x0 * c - x1 * s, x0 * s + x1 * c);
    }
}

__global__ void __launch_bounds__(pf::THREADS, 2) prefill_attention_kernel(const PrefillArgs a) {
    using namespace pf;
    pdl_trigger();
    pdl_wait();
    extern __shared__ __align__(16) unsigned char smraw[];
    bf16* qs = reinterpret_cast<bf16*>(smraw);   // [BQ][QROW]
    bf16* ksm = qs + BQ * QROW;                  // [2][BKV][QROW]
    bf16* vsm = ksm + 2 * BKV * QROW;            // [2][BKV][VROW]
    const int4 tile = a.tiles[blockIdx.x];
    if (tile.x < 0) return;
    const int b = tile.x, r0 = tile.y, nrow = tile.z, h = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gq = lane >> 2, tig = lane & 3;
    const int pmax = min(a.row_pos[r0 + nrow - 1], a.max_ctx - 1);   // positions ascend within a sequence
    const int nkv = (pmax + BKV) / BKV;                               // tiles covering slots 0..pmax
    const long kvrow0 = (long)b * a.max_ctx;
    const long ldkv = (long)a.nh * (DN + DV);
    const long ldq = (long)a.nh * DQK;

    for (int c = tid; c < BQ * (DQK / 8); c += THREADS) {
        const int i = c / (DQK / 8), q = c % (DQK / 8);
        bf16* d = qs + i * QROW + 8 * q;
        if (i < nrow) cp_async16(smem_u32(d), a.q + (long)(r0 + i) * ldq + (long)h * DQK + 8 * q);
        else *reinterpret_cast<uint4*>(d) = make_uint4(0, 0, 0, 0);
    }
    // K rows: [k_nope (16 chunks) | k_pe (8 chunks)], V rows: 16 chunks; slots past max_ctx re-read the
    // last slot (masked)
    auto load_kv = [&](int buf, int t0) {
        bf16* kd = ksm + buf * BKV * QROW;
        bf16* vd = vsm + buf * BKV * VROW;
        for (int c = tid; c < BKV * 40; c += THREADS) {
            const int j = c / 40, q = c % 40;
            const long row = kvrow0 + min(t0 + j, a.max_ctx - 1);
            if (q < 16) cp_async16(smem_u32(kd + j * QROW + 8 * q), a.kv + row * ldkv + (long)h * (DN + DV) + 8 * q);
            else if (q < 24) cp_async16(smem_u32(kd + j * QROW + DN + 8 * (q - 16)), a.xpe + row * DR + 8 * (q - 16));
            else cp_async16(smem_u32(vd + j * VROW + 8 * (q - 24)), a.kv + row * ldkv + (long)h * (DN + DV) + DN + 8 * (q - 24));
        }
        cp_async_commit();
    };

    const int ra = 16 * warp + gq, rb = ra + 8;
    const int pos_a = ra < nrow ? a.row_pos[r0 + ra] : -1;   // -1: padding row, sees no slot
    const int pos_b = rb < nrow ? a.row_pos[r0 + rb] : -1;
    const float sl2 = a.sigma * 1.4426950408889634f;         // scores in log2 units
    float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};
    float o[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    uint32_t qf[DQK / 16][4];

    load_kv(0, 0);
    for (int it = 0; it < nkv; ++it) {
        if (it + 1 < nkv) {
            load_kv((it + 1) & 1, (it + 1) * BKV);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        if (it == 0) {
            const uint32_t qaddr = smem_u32(qs + (16 * warp + (lane & 7) + ((lane >> 3) & 1) * 8) * QROW + (lane >> 4) * 8);
#pragma unroll
            for (int ks = 0; ks < DQK / 16; ++ks) ldsm_x4(qaddr + ks * 32, qf[ks]);
        }
        const bf16* K = ksm + (it & 1) * BKV * QROW;
        const bf16* V = vsm + (it & 1) * BKV * VROW;
        float s[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
        const uint32_t kaddr = smem_u32(K + ((lane & 7) + (lane >> 4) * 8) * QROW + ((lane >> 3) & 1) * 8);
#pragma unroll
        for (int ks = 0; ks < DQK / 16; ++ks) {
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t kb[4];
                ldsm_x4(kaddr + np * 16 * QROW * 2 + ks * 32, kb);
                mma_bf16_16816(s[2 * np], qf[ks], kb[0], kb[1]);
                mma_bf16_16816(s[2 * np + 1], qf[ks], kb[2], kb[3]);
            }
        }
        // causal mask and scale, then the online softmax of rows ra (e = 0, 1) and rb (e = 2, 3)
        const int t0 = it * BKV;
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int t = t0 + nt * 8 + 2 * tig + (e & 1);
                const int p = e < 2 ? pos_a : pos_b;
                const float v = t <= p ? s[nt][e] * sl2 : -INFINITY;
                s[nt][e] = v;
                mx[e >> 1] = fmaxf(mx[e >> 1], v);
            }
        float alpha[2];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 1));
            mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 2));
            const float mn = fmaxf(m_r[rr], mx[rr]);
            alpha[rr] = m_r[rr] == -INFINITY ? 0.f : exp2f(m_r[rr] - mn);
            m_r[rr] = mn;
        }
        float ls[2] = {0.f, 0.f};
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int rr = e >> 1;
                const float p = s[nt][e] == -INFINITY ? 0.f : exp2f(s[nt][e] - m_r[rr]);
                s[nt][e] = p;
                ls[rr] += p;
            }
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            ls[rr] += __shfl_xor_sync(0xffffffffu, ls[rr], 1);
            ls[rr] += __shfl_xor_sync(0xffffffffu, ls[rr], 2);
            l_r[rr] = l_r[rr] * alpha[rr] + ls[rr];
        }
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            o[nt][0] *= alpha[0]; o[nt][1] *= alpha[0];
            o[nt][2] *= alpha[1]; o[nt][3] *= alpha[1];
        }
        // O += P V: the score accumulators of slots 16kk .. 16kk + 15 are the A fragment
#pragma unroll
        for (int kk = 0; kk < BKV / 16; ++kk) {
            uint32_t pa[4];
            pa[0] = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
            pa[1] = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
            pa[2] = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
            pa[3] = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
            const uint32_t vaddr = smem_u32(V + (kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * VROW + (lane >> 4) * 8);
#pragma unroll
            for (int np = 0; np < 8; ++np) {
                uint32_t vb[4];
                ldsm_x4_t(vaddr + np * 32, vb);
                mma_bf16_16816(o[2 * np], pa, vb[0], vb[1]);
                mma_bf16_16816(o[2 * np + 1], pa, vb[2], vb[3]);
            }
        }
        __syncthreads();
    }
    cp_async_wait<0>();
    const long ldo = (long)a.nh * DV;
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        const int row = rr ? rb : ra;
        if (row >= nrow) continue;
        const float inv = l_r[rr] > 0.f ? 1.f / l_r[rr] : 0.f;
        bf16* dst = a.o_bf + (long)(r0 + row) * ldo + (long)h * DV + 2 * tig;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt)
            *reinterpret_cast<uint32_t*>(dst + nt * 8) = pack_bf16(o[nt][2 * rr] * inv, o[nt][2 * rr + 1] * inv);
    }
}

cudaError_t launch_kv_gather(const PrefillArgs& a, cudaStream_t st) {
    dim3 grid((a.max_ctx + pf::kGatherSlots - 1) / pf::kGatherSlots, a.B);
    return launch_pdl(kv_gather_kernel, grid, dim3(256), 0, st, a);
}

cudaError_t launch_prefill_tiles(const PrefillArgs& a, cudaStream_t st) {
    return launch_pdl(prefill_tiles_kernel, dim3(1), dim3(256), (size_t)(a.B + 1) * sizeof(int), st, a);
}

cudaError_t launch_rope_q_rows(const PrefillArgs& a, cudaStream_t st) {
    return launch_pdl(rope_q_rows_kernel, dim3(a.M), dim3(256), 0, st, a);
}

cudaError_t launch_prefill_attention(const PrefillArgs& a, cudaStream_t st) {
    if (a.bq != pf::BQ) return cudaErrorInvalidValue;
    {
        cudaError_t e = smem_optin((const void*)prefill_attention_kernel, (int)pf::SMEM);
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(prefill_attention_kernel, dim3(a.ntiles_cap, a.nh), dim3(pf::THREADS), pf::SMEM, st, a);
}

int prefill_tiles_cap(int M, int B, int bq) { return (M + bq - 1) / bq + B; }

}  // namespace e3
