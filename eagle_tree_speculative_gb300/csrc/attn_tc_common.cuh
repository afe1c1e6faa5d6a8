// Pieces shared by the two tcgen05 attention kernels (tree attention and the
// training-time-test attention): the TMEM layout, the MMA issue loop and the online
// softmax of one 128-key tile for one query row.
//
// TMEM (512 columns): S[buf] at buf * 128 (P[buf], bf16 pairs, is written over the
// first 64 columns of S[buf]), O at 256, Q (bf16 pairs) at 384.  Both kernels keep
// their K and V tiles in two rings of NS stages of 32 KB (two 64-dim boxes of 128
// rows, 128-byte swizzle) and use the barrier protocol described in their headers.
#pragma once

#include "common.cuh"
#include "tc_common.cuh"

namespace eagle {
namespace attn_common {

constexpr int TBN = 128;                          // keys per tile
constexpr int NSBUF = 2;                          // S and P buffers in TMEM
constexpr int KV_BOX_BYTES = TBN * 64 * 2;        // 16 KB: 128 keys x 64 dims
constexpr int K_BYTES = 2 * KV_BOX_BYTES;         // 32 KB (one K or V tile)
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t S_COL0 = 0, O_COL0 = 256, Q_COL0 = 384;
constexpr float kRescaleThreshold = 8.f;          // log2 units

constexpr uint32_t kIdescQK = idesc_bf16(128, TBN, 0, 0);
constexpr uint32_t kIdescPV = idesc_bf16(128, kHeadDim, 0, 1);

// The MMA issuer (one thread) for tiles 0 .. T-1 held in ring stage j % NS:
// S[j % 2] = Q K_j^T (Q from TMEM, K a K-major shared-memory operand) and O += P_j V_j
// (P from TMEM over S[j % 2], V an MN-major operand).  After the first two QK^T it
// issues whichever is ready first, the QK^T of tile js (its S buffer free once the PV of
// tile js-2 has read its P; its K tile landed) or the PV of tile jp (its P written, its
// V tile landed), so a late K tile never holds back a PV and the reverse.  Each
// completion tested is the next one of its barrier, so one parity bit names it.  Every
// wait is bounded; the thread finally waits for its own MMAs to drain.
// Descriptors are built once; every operand differs from its base only in the 14-bit
// start-address field (all addresses < 256 KB), so an MMA costs two adds.
template <int NS, class Bars>
__device__ __forceinline__ void mma_issue_loop(Bars* bars, uint32_t tmem, uint8_t* sK, uint8_t* sV,
                                               int T, volatile int* abort_flag) {
    const uint64_t dK0 = sw128_desc(s32(sK));
    const uint64_t dV0 = sw128_desc_mn(s32(sV), KV_BOX_BYTES, 1024);
    const uint32_t ocol = tmem + O_COL0;
    auto issue_qk = [&](int j) {     // S[j % 2] = Q K_j^T; frees K stage j
        const uint64_t dk = dK0 + (uint64_t)(((j % NS) * K_BYTES) >> 4);
        const uint32_t scol = tmem + S_COL0 + (uint32_t)((j % NSBUF) * TBN);
#pragma unroll
        for (int k = 0; k < kHeadDim / 16; ++k)   // 16 dims = 8 packed TMEM columns
            umma_f16_ts(scol, tmem + Q_COL0 + k * 8,
                        dk + (uint64_t)((((k >> 2) * KV_BOX_BYTES) + (k & 3) * 32) >> 4), kIdescQK,
                        k > 0 ? 1u : 0u);
        umma_commit(s32(&bars->s_full[j % NSBUF]));
        umma_commit(s32(&bars->k_empty[j % NS]));
    };
    auto issue_pv = [&](int j) {     // O += P[j % 2] V_j; frees V stage j
        const uint64_t dv = dV0 + (uint64_t)(((j % NS) * K_BYTES) >> 4);
        const uint32_t pcol = tmem + S_COL0 + (uint32_t)((j % NSBUF) * TBN);
        const uint32_t acc0 = j > 0 ? 1u : 0u;
#pragma unroll
        for (int k = 0; k < TBN / 16; ++k)   // 16 keys = 8 packed TMEM columns
            umma_f16_ts(ocol, pcol + k * 8, dv + (uint64_t)((k * 16 * 128) >> 4), kIdescPV,
                        k > 0 ? 1u : acc0);
        umma_commit(s32(&bars->pv_done[j % NSBUF]));
        umma_commit(s32(&bars->v_empty[j % NS]));
    };
    auto wait_on = [&](uint64_t* bar, uint32_t parity) {
        if (!mbar_wait(s32(bar), parity, abort_flag)) return false;
        tc_fence_after();
        return true;
    };
    bool ok = wait_on(&bars->q_full, 0u);
    for (int j = 0; ok && j < min(T, NSBUF); ++j) {
        ok = wait_on(&bars->k_full[j % NS], ((uint32_t)j / NS) & 1u);
        if (ok) issue_qk(j);
    }
    int js = min(T, NSBUF), jp = 0;
    long long t_last = clock64();
    uint32_t idle = 0;
    while (ok && jp < T) {
        bool progressed = false;
        if (js < T &&
            mbar_try_wait(s32(&bars->pv_done[js % NSBUF]), ((uint32_t)(js - NSBUF) / NSBUF) & 1u) &&
            mbar_try_wait(s32(&bars->k_full[js % NS]), ((uint32_t)js / NS) & 1u)) {
            tc_fence_after();
            issue_qk(js++);
            progressed = true;
        }
        if (jp < js && mbar_try_wait(s32(&bars->p_full[jp % NSBUF]), ((uint32_t)jp / NSBUF) & 1u) &&
            mbar_try_wait(s32(&bars->v_full[jp % NS]), ((uint32_t)jp / NS) & 1u)) {
            tc_fence_after();
            issue_pv(jp++);
            progressed = true;
        }
        if (progressed) {
            t_last = clock64();
        } else if ((++idle & 63u) == 0u) {
            if (*abort_flag) ok = false;
            else if (clock64() - t_last > kTimeoutCycles) { *abort_flag = 1; ok = false; }
        }
    }
    umma_commit(s32(&bars->drain));
    mbar_wait(s32(&bars->drain), 0u, abort_flag, /*honour_abort=*/false);
}

// The online softmax of tile j for this thread's row, its 128 scores already masked in
// x (-inf for keys it may not see).  The running (reference max, sum) are in the exp2
// domain (sc = scale * log2 e); the reference is raised only when the tile's maximum
// exceeds it by more than kRescaleThreshold, and then O is rescaled in TMEM after the
// PV of tile j-1 (the one before, once a PV ran).  P = 2^(s sc - ref) goes as bf16 pairs
// over S[j % 2], where the PV MMA reads it, and the warp arrives on p_full.  Returns
// false (uniformly in the warp) if a wait ran out.
template <class Bars>
__device__ __forceinline__ bool softmax_tile(Bars* bars, float (&x)[TBN], float sc, float& mref,
                                             float& l, uint32_t s_addr, uint32_t o_addr, int j,
                                             int lane, volatile int* abort_flag) {
    // row max over the tile: eight independent chains, then a tree
    float m8[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) m8[e] = x[e];
#pragma unroll
    for (int c = 8; c < TBN; c += 8)
#pragma unroll
        for (int e = 0; e < 8; ++e) m8[e] = fmaxf(m8[e], x[c + e]);
    float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                     fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
    mx *= sc;                              // scale > 0 commutes with max
    float alpha = 1.f;
    if (mx > mref + kRescaleThreshold || (mref == -INFINITY && mx > -INFINITY)) {
        alpha = mref == -INFINITY ? 0.f : exp2f(mref - mx);
        mref = mx;
        l *= alpha;
    }
    // P of tile j goes over S of tile j, whose MMA was issued after the PV of tile j-2
    // had finished with that buffer.  PV of tile j-1 is awaited only before the output
    // accumulator is rescaled.
    if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        const bool got = mbar_wait(s32(&bars->pv_done[(j - 1) % NSBUF]),
                                   ((uint32_t)(j - 1) / NSBUF) & 1u, abort_flag);
        if (!__all_sync(0xffffffffu, got)) return false;
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < kHeadDim / 32; ++cc) {
            uint32_t o[32];
            tmem_ld32(o_addr + cc * 32, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(o_addr + cc * 32, o);
        }
    }
    const float base = mref == -INFINITY ? 0.f : mref;
    float ps[4] = {0.f, 0.f, 0.f, 0.f};      // four partial sums, no long FADD chain
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t pk[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            const float p0 = ex2_approx(fmaf(x[64 * h + 2 * e], sc, -base));
            const float p1 = ex2_approx(fmaf(x[64 * h + 2 * e + 1], sc, -base));
            ps[e & 3] += p0 + p1;
            pk[e] = pack2(p0, p1);
        }
        tmem_st32(s_addr + (uint32_t)(32 * h), pk);   // P, bf16 pairs, over S
    }
    l += (ps[0] + ps[1]) + (ps[2] + ps[3]);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(s32(&bars->p_full[j % NSBUF]));
    return true;
}

// The 128 scores of this thread's row of S[buf] (TMEM), four loads then one wait.
__device__ __forceinline__ void load_scores(uint32_t s_addr, float (&x)[TBN]) {
    uint32_t u0[32], u1[32], u2[32], u3[32];
    tmem_ld32_nowait(s_addr, u0);
    tmem_ld32_nowait(s_addr + 32, u1);
    tmem_ld32_nowait(s_addr + 64, u2);
    tmem_ld32_nowait(s_addr + 96, u3);
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
    for (int c = 0; c < 32; ++c) {
        x[c] = __uint_as_float(u0[c]);
        x[32 + c] = __uint_as_float(u1[c]);
        x[64 + c] = __uint_as_float(u2[c]);
        x[96 + c] = __uint_as_float(u3[c]);
    }
}

}  // namespace attn_common
}  // namespace eagle
