// Training-time-test attention on the 5th-generation tensor cores.
//
// Method (TTT page, section "训练时的 attention mask 为什么要特殊处理"): round 0 runs
// on the original tokens with the causal mask; in round r >= 1 every position i
// holds the token the previous round predicted there, and that token may see only
// its ancestors: the original tokens 0..i and the round-1..r tokens at position i.
// The original-token part is a dense causal attention; the part between simulated
// rounds is one key per earlier round on the diagonal, which the page says to
// compute as per-position dot products rather than as a mostly-masked matrix
// product.  This kernel does exactly that split.
//
// One CTA owns 128 query rows (row = position * G + head-in-group, G = Hq / Hkv)
// of one (sequence, kv head); its positions are imin .. imin + PB - 1 at most.
//   - The causal part runs like the tree-attention kernel: 128-key K and V tiles of
//     round 0 stream by TMA through two 3-stage rings; S = Q K^T and O += P V are
//     tcgen05 MMAs with Q, S, P and O in TMEM; one thread per row runs the online
//     softmax with the causal mask on the tiles that cross the diagonal.
//   - Diagonal tiles follow the causal tiles through the same rings and the same
//     MMAs, so they load while the last causal tiles are computed.  The rows of rounds
//     1..r at the tile's positions are contiguous per round, so one 4-D TMA box (64
//     dims x PB positions x RB rounds, PB * RB = 128) fills a K stage and the same box
//     of V the V stage.  A row sees, of such a tile, only the keys of its own position
//     in rounds up to r (at most RB of the 128): the softmax masks the rest, so the
//     diagonal part costs ND = ceil(r / RB) more tiles of the same pipeline instead of
//     per-position dot products on the CUDA cores after it.
// The row tiles nearest the end of the sequence have the most keys, so the grid
// runs them first.  Every wait is bounded.
//
// Barriers (each completes once per use; a waiter is never more than one
// completion behind):
//   k_full/v_full[s]     stage s landed (TMA)                   producer -> MMA
//   k_empty/v_empty[s]   tile in stage s consumed (MMA)         MMA -> producer
//   q_full, s_full/p_full/pv_done[tile % 2]  as in the tree-attention kernel.
#pragma once

#include "common.cuh"
#include "tc_common.cuh"
#include "attn_tc_common.cuh"

namespace eagle {
namespace ttt_tc {

using attn_common::TBN;
using attn_common::NSBUF;
using attn_common::KV_BOX_BYTES;
using attn_common::K_BYTES;
using attn_common::TMEM_COLS;
using attn_common::S_COL0;
using attn_common::O_COL0;
using attn_common::Q_COL0;
using attn_common::kRescaleThreshold;

constexpr int NSTAGES = 3;                        // K ring and V ring
constexpr int kPrefetch = 3;
constexpr int ROWS_PER_CTA = 128;
constexpr int SMEM_BYTES = 2 * NSTAGES * K_BYTES + 2048;
constexpr int kThreads = 256;                     // warps 0-3 roles, 4-7 softmax
constexpr int kMaxRounds = 16;                    // rounds stored (original + simulated)

struct Args {
    const uint16_t* q;        // [B, S, Hq, 128], the queries of round r
    uint16_t* out;            // [B, S, Hq, 128]
    int B, S, Hq, Hkv, G, R1, r;
    int PB;                   // positions per diagonal box (>= positions of any row tile)
    int RB;                   // rounds per diagonal box (PB * RB = 128)
    int ND;                   // diagonal tiles: ceil(r / RB)
    int tiles;                // row tiles per (sequence, kv head)
    float scale_log2;
    int32_t* dev_status;
};

struct Bars {
    uint64_t k_full[NSTAGES];
    uint64_t k_empty[NSTAGES];
    uint64_t v_full[NSTAGES];
    uint64_t v_empty[NSTAGES];
    uint64_t s_full[NSBUF];
    uint64_t q_full;
    uint64_t p_full[NSBUF];
    uint64_t pv_done[NSBUF];
    uint64_t drain;
    uint32_t tmem_slot;
    int abort_flag;
};

__global__ void __launch_bounds__(kThreads, 1)
ttt_attn_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,    // round 0, 3-D
                   const __grid_constant__ CUtensorMap tmap_v,
                   const __grid_constant__ CUtensorMap tmap_kd,   // all rounds, 4-D
                   const __grid_constant__ CUtensorMap tmap_vd, Args a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* sK = smem;                                   // [NSTAGES][32 KB]
    uint8_t* sV = sK + NSTAGES * K_BYTES;                 // [NSTAGES][32 KB]
    Bars* bars = reinterpret_cast<Bars*>(sV + NSTAGES * K_BYTES);
    volatile int* abort_flag = &bars->abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int kvz = (int)(blockIdx.x / (unsigned)a.tiles);   // (sequence, kv head) slab
    const int b = kvz / a.Hkv, kvh = kvz % a.Hkv;
    // within a slab, the row tiles with the most keys first
    const int rg = a.tiles - 1 - (int)(blockIdx.x % (unsigned)a.tiles);
    const int G = a.G, S = a.S, rows = S * G;
    const int row0 = rg * ROWS_PER_CTA;
    const int row_end = min(row0 + ROWS_PER_CTA, rows);
    const int imin = row0 / G;                            // first position of the tile
    const int ke = (row_end - 1) / G + 1;                 // round-0 keys 0 .. ke-1 reach the tile
    const int T = (ke + TBN - 1) / TBN;                   // causal tiles
    const int ND = a.ND;                                  // diagonal tiles, loaded last

    uint4 qrow[kHeadDim / 8];
    if (warp >= 4) {
        const int r = row0 + (warp & 3) * 32 + lane;
#pragma unroll
        for (int u = 0; u < kHeadDim / 8; ++u) qrow[u] = make_uint4(0u, 0u, 0u, 0u);
        if (r < rows) {
            const uint4* src = reinterpret_cast<const uint4*>(
                a.q + (((int64_t)b * S + r / G) * a.Hq + kvh * G + r % G) * kHeadDim);
#pragma unroll
            for (int u = 0; u < kHeadDim / 8; ++u) qrow[u] = __ldg(src + u);
        }
    }

    if (tid == 0) {
        for (int s = 0; s < NSTAGES; ++s) {
            mbar_init(s32(&bars->k_full[s]), 1);
            mbar_init(s32(&bars->k_empty[s]), 1);
            mbar_init(s32(&bars->v_full[s]), 1);
            mbar_init(s32(&bars->v_empty[s]), 1);
        }
        for (int p = 0; p < NSBUF; ++p) {
            mbar_init(s32(&bars->s_full[p]), 1);
            mbar_init(s32(&bars->p_full[p]), 4);
            mbar_init(s32(&bars->pv_done[p]), 1);
        }
        mbar_init(s32(&bars->drain), 1);
        mbar_init(s32(&bars->q_full), 4);
        bars->abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
        for (const CUtensorMap* m : {&tmap_k, &tmap_v, &tmap_kd, &tmap_vd})
            asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
    }
    if (warp == 1) tmem_alloc(s32(&bars->tmem_slot), TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_slot;

    // ---- Q -> TMEM (softmax warps, one lane = one row) ----
    if (warp >= 4) {
        const uint32_t qaddr = tmem + ((uint32_t)((warp & 3) * 32) << 16) + Q_COL0;
        uint32_t w[32];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const uint4 v = qrow[8 * h + u];
                w[4 * u] = v.x; w[4 * u + 1] = v.y; w[4 * u + 2] = v.z; w[4 * u + 3] = v.w;
            }
            tmem_st32(qaddr + 32 * h, w);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s32(&bars->q_full));
    }

    if (warp == 0 || warp == 2) {
        if (lane == 0) {
            // ---------------- TMA producers: K (warp 0) and V (warp 2) ----------------
            // Ring tiles 0 .. T-1 are the causal tiles, T .. T+ND-1 the diagonal boxes,
            // which so stream in while the last causal tiles are computed.
            const bool isK = warp == 0;
            const CUtensorMap* map = isK ? &tmap_k : &tmap_v;
            const CUtensorMap* dmap = isK ? &tmap_kd : &tmap_vd;
            uint8_t* ring = isK ? sK : sV;
            uint64_t* full = isK ? bars->k_full : bars->v_full;
            uint64_t* empty = isK ? bars->k_empty : bars->v_empty;
            for (int jp = NSTAGES; jp < min(T, NSTAGES + kPrefetch); ++jp) {
                tma_prefetch_3d(map, 0, jp * TBN, kvz);
                tma_prefetch_3d(map, 64, jp * TBN, kvz);
            }
            // round-0 K/V tiles are read by every row tile of the (sequence, kv head):
            // keep them in L2; each diagonal row is read once: let it go first
            const uint64_t keep = l2_policy_evict_last(), once = l2_policy_evict_first();
            for (int t = 0; t < T + ND; ++t) {
                const int st = t % NSTAGES;
                // wait until the MMAs consumed the stage's previous tile
                if (t >= NSTAGES &&
                    !mbar_wait(s32(&empty[st]), (uint32_t)((t - NSTAGES) / NSTAGES) & 1u, abort_flag))
                    break;
                const uint32_t fb = s32(&full[st]);
                uint8_t* dst = ring + st * K_BYTES;
                if (t < T) {
                    if (t >= 1 && t + NSTAGES + kPrefetch - 1 < T) {
                        const int yp = (t + NSTAGES + kPrefetch - 1) * TBN;
                        tma_prefetch_3d(map, 0, yp, kvz);
                        tma_prefetch_3d(map, 64, yp, kvz);
                    }
                    mbar_expect_tx(fb, K_BYTES);
                    tma_load_3d_hint(s32(dst), map, fb, 0, t * TBN, kvz, keep);
                    tma_load_3d_hint(s32(dst + KV_BOX_BYTES), map, fb, 64, t * TBN, kvz, keep);
                } else {
                    mbar_expect_tx(fb, K_BYTES);                  // PB * RB = 128 rows
                    const int u0 = 1 + (t - T) * a.RB;            // first round of the box
                    tma_load_4d_hint(s32(dst), dmap, fb, 0, imin, u0, kvz, once);
                    tma_load_4d_hint(s32(dst + KV_BOX_BYTES), dmap, fb, 64, imin, u0, kvz, once);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer: causal and diagonal tiles ----------------
            attn_common::mma_issue_loop<NSTAGES>(bars, tmem, sK, sV, T + ND, abort_flag);
        }
    } else if (warp >= 4) {
        // ---------------- softmax: one thread per query row ----------------
        const int q4 = warp & 3;                         // TMEM lane quadrant
        const int r = row0 + q4 * 32 + lane;
        const bool valid = r < rows;
        const int i = valid ? r / G : imin;              // position
        const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
        const uint32_t s_addr0 = tmem + lane_base + S_COL0;
        const uint32_t o_addr = tmem + lane_base + O_COL0;
        const float sc = a.scale_log2;
        const int pl = i - imin;                         // position within the diagonal boxes
        float mref = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; ok && j < T + ND; ++j) {
            bool got = mbar_wait(s32(&bars->s_full[j % NSBUF]), ((uint32_t)j / NSBUF) & 1u, abort_flag);
            if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
            tc_fence_after();
            const uint32_t s_addr = s_addr0 + (uint32_t)((j % NSBUF) * TBN);
            float x[TBN];
            attn_common::load_scores(s_addr, x);
            const int key0 = j * TBN;
            if (j >= T) {
                // diagonal tile: key c = (round u0 + c / PB, position imin + c % PB); this
                // row sees its own position in rounds up to r
                const int nr = min(a.RB, a.r - (j - T) * a.RB);
                uint64_t vis[2] = {0ull, 0ull};
                if (valid)
                    for (int ul = 0; ul < nr; ++ul) {
                        const int c = ul * a.PB + pl;
                        vis[c >> 6] |= 1ull << (c & 63);
                    }
#pragma unroll
                for (int c = 0; c < TBN; ++c)
                    if (!((vis[c >> 6] >> (c & 63)) & 1ull)) x[c] = -INFINITY;
            } else if (key0 + TBN - 1 > imin || !valid) {
                // causal mask: key k visible iff k <= i (keys past the sequence arrive as
                // zeros from TMA and are masked too)
                uint64_t vis[2];
#pragma unroll
                for (int w = 0; w < 2; ++w) {
                    const int ne = min(max(i + 1 - (key0 + 64 * w), 0), 64);
                    vis[w] = valid ? (ne >= 64 ? ~0ull : ((1ull << ne) - 1ull)) : 0ull;
                }
#pragma unroll
                for (int c = 0; c < TBN; ++c)
                    if (!((vis[c >> 6] >> (c & 63)) & 1ull)) x[c] = -INFINITY;
            }
            if (!attn_common::softmax_tile(bars, x, sc, mref, l, s_addr, o_addr, j, lane, abort_flag)) {
                ok = false;
                break;
            }
        }
        const int TT = T + ND;
        bool got = ok && TT > 0 ? mbar_wait(s32(&bars->pv_done[(TT - 1) % NSBUF]),
                                            ((uint32_t)(TT - 1) / NSBUF) & 1u, abort_flag)
                                : false;
        got = __all_sync(0xffffffffu, got);
        tc_fence_after();
        const int h = kvh * G + (valid ? r % G : 0);
        uint16_t* dst0 = a.out + (((int64_t)b * S + i) * a.Hq + h) * kHeadDim;
        const float inv = (got && l > 0.f) ? 1.f / l : 0.f;
        for (int cc = 0; cc < kHeadDim / 32; ++cc) {
            uint32_t o[32];
            if (got) tmem_ld32(o_addr + cc * 32, o);
            else
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = 0u;
            if (!valid) continue;
            uint16_t* dst = dst0 + cc * 32;
#pragma unroll
            for (int e = 0; e < 32; e += 8) {
                const uint4 w = make_uint4(
                    pack2(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv),
                    pack2(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv),
                    pack2(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv),
                    pack2(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv));
                *reinterpret_cast<uint4*>(dst + e) = w;
            }
        }
    }
    __syncthreads();
    if (tid == 0 && *abort_flag) flag_error(a.dev_status, EAGLE_DEV_TIMEOUT);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace ttt_tc
}  // namespace eagle
