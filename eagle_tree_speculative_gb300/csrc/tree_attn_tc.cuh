// Tree attention on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Method: see tree_attn.cu (node i attends to the committed rows 0..L_b-1 and
// to the tree rows L_b + j for j = i or an ancestor of i).
//
// One CTA owns 128 query rows (one M-tile) of one (sequence, kv head, KV split):
// the Hq/Hkv query heads that share the kv head are packed as rows (row r =
// node r / G, head kvh * G + r % G); larger groups take several CTAs, adjacent
// in the grid so they share each K/V tile through L2.  Keys come in tiles of
// 128 (the QK^T MMA is N = 128 wide).  Roles:
//   warps 0, 2  lane 0 of warp 0 streams 128-key K tiles and lane 0 of warp 2
//               V tiles by TMA, each into its own 3-stage ring, starting at once,
//               and asks L2 for tiles further on;
//   warp 1      owns TMEM (S: two 128-column fp32 buffers, P written as bf16
//               pairs over the first 64 columns of its S buffer; O: 128 columns;
//               Q: 64 columns of bf16 pairs) and one thread issues the MMAs:
//               S = Q K^T (M=128, N=128, K=16; Q read from TMEM, K a K-major
//               shared-memory operand) and O += P V (P read from TMEM, V an
//               MN-major shared-memory operand), each as soon as its operands
//               are in, so a late K tile never holds back a PV or the reverse;
//   warps 4-7   softmax: one thread per query row; each first parks its row of Q
//               in TMEM, then per tile reads its 128 scores from TMEM, applies the
//               tree mask, keeps a running (reference max, sum) in the exp2
//               domain, and writes P = 2^(s - max) as packed bf16 over the scores,
//               where the PV MMA reads it.
// Keeping Q in TMEM leaves the shared-memory bandwidth to the TMA writes and
// the K / V operand reads.  The output accumulator is rescaled (TMEM load /
// store) only when a row maximum grows by more than 2^8, otherwise the stale
// reference is kept; every P and the final O / l use the same reference, so the
// result is exact up to rounding.  Every wait is bounded.
//
// Barrier protocol: each barrier completes once per tile (or once per two
// tiles when indexed by tile parity); a waiter is never more than one
// completion behind, so a single phase bit identifies the completion it wants.
//   k_full/k_empty[t % 3], v_full/v_empty[t % 3]   TMA rings (32 KB stages)
//   q_full                   Q parked in TMEM      (softmax warps -> MMA)
// and (tile % 2, (tile / 2) & 1) names a completion of the tile-parity barriers:
//   s_full[j%2]              QK^T of tile j done  (MMA -> softmax)
//   p_full[j%2]              P of tile j in TMEM  (softmax -> MMA)
//   pv_done[j%2]             PV of tile j done    (MMA -> MMA, before QK^T of
//                            tile j+2 overwrites that buffer; MMA -> softmax,
//                            before O is rescaled or read)
#pragma once

#include "common.cuh"
#include "tc_common.cuh"
#include "attn_tc_common.cuh"

namespace eagle {
namespace attn_tc {

using attn_common::TBN;
using attn_common::NSBUF;
using attn_common::KV_BOX_BYTES;
using attn_common::K_BYTES;
using attn_common::TMEM_COLS;
using attn_common::S_COL0;
using attn_common::O_COL0;
using attn_common::Q_COL0;

constexpr int KSTAGES = 3;                        // K ring
constexpr int VSTAGES = 3;                        // V ring (the MMA loop takes one depth)
static_assert(KSTAGES == VSTAGES, "one ring depth");
constexpr int kPrefetch = 3;                      // L2 prefetch distance beyond each ring
constexpr int ROWS_PER_CTA = 128;                 // one M-tile
constexpr int SMEM_BYTES = (KSTAGES + VSTAGES) * K_BYTES + 2048;
constexpr int kThreads = 256;                     // warps 0-3 roles, 4-7 softmax

struct Args {
    const uint16_t* q;
    uint16_t* out;
    float* ws_o;
    float* ws_ml;
    const int32_t* kv_len;
    const int32_t* parent;
    int B, n, Hq, Hkv, G, Lmax, splits;
    float scale_log2;
    int32_t* dev_status;
};

struct Bars {
    uint64_t k_full[KSTAGES];
    uint64_t k_empty[KSTAGES];
    uint64_t v_full[VSTAGES];
    uint64_t v_empty[VSTAGES];
    uint64_t s_full[NSBUF];          // [tile parity]
    uint64_t q_full;
    uint64_t p_full[NSBUF];
    uint64_t pv_done[NSBUF];
    uint64_t drain;
    uint32_t tmem_slot;
    int abort_flag;
    int err;
    int pad;
    unsigned long long anc[kMaxNodes];
    int par[kMaxNodes];
};

__global__ void __launch_bounds__(kThreads, 1)
tree_attn_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                    const __grid_constant__ CUtensorMap tmap_v, Args a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* sK = smem;                                   // [KSTAGES][32 KB]
    uint8_t* sV = sK + KSTAGES * K_BYTES;                 // [VSTAGES][32 KB]
    Bars* bars = reinterpret_cast<Bars*>(sV + VSTAGES * K_BYTES);
    volatile int* abort_flag = &bars->abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rg = blockIdx.x;
    const int kvh = blockIdx.y / a.splits, split = blockIdx.y % a.splits;
    const int b = blockIdx.z;
    const int n = a.n, G = a.G, rows = n * G;
    const int row0 = rg * ROWS_PER_CTA;
    const int L = a.kv_len[b];
    // softmax threads: this thread's query row (bf16 pairs), loaded now, parked in TMEM later
    uint4 qrow[kHeadDim / 8];
    if (warp >= 4) {
        const int r = row0 + (warp & 3) * 32 + lane;
#pragma unroll
        for (int u = 0; u < kHeadDim / 8; ++u) qrow[u] = make_uint4(0u, 0u, 0u, 0u);
        if (r < rows) {
            const uint4* src = reinterpret_cast<const uint4*>(
                a.q + (((int64_t)b * n + r / G) * a.Hq + kvh * G + r % G) * kHeadDim);
#pragma unroll
            for (int u = 0; u < kHeadDim / 8; ++u) qrow[u] = __ldg(src + u);
        }
    }

    // the parent array, one node per thread; the ancestor masks are built from it below
    if (tid < n) bars->par[tid] = a.parent[(int64_t)b * n + tid];
    if (tid == 0) {
        bars->err = (L < 0 || (int64_t)L + n > a.Lmax) ? EAGLE_DEV_CAPACITY : 0;
        for (int s = 0; s < KSTAGES; ++s) {
            mbar_init(s32(&bars->k_full[s]), 1);
            mbar_init(s32(&bars->k_empty[s]), 1);
        }
        for (int s = 0; s < VSTAGES; ++s) {
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
        asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&tmap_k)) : "memory");
        asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&tmap_v)) : "memory");
    }
    if (warp == 1) tmem_alloc(s32(&bars->tmem_slot), TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_slot;
    // A0: anc[i] = {i} and its ancestors, one thread per node walking up the parents in
    // shared memory (each step goes to a smaller index, so at most i steps); a parent
    // outside [0, i) (or a root parent other than -1) flags the tree as invalid
    if (tid < n) {
        unsigned long long m = 1ull << tid;
        int e = 0;
        if (tid == 0) {
            if (bars->par[0] != -1) e = EAGLE_DEV_BAD_TREE;
        } else {
            int x = tid;
            while (x > 0) {
                const int p = bars->par[x];
                if (p < 0 || p >= x) { e = EAGLE_DEV_BAD_TREE; break; }
                m |= 1ull << p;
                x = p;
            }
        }
        bars->anc[tid] = m;
        if (e) atomicOr(&bars->err, e);
    }
    __syncthreads();
    if (tid == 0 && bars->err && rg == 0 && blockIdx.y == 0) flag_error(a.dev_status, bars->err);
    const bool err = bars->err != 0;

    // key range of this split: committed keys are chunked, the last split adds the tree
    int chunk = (L + a.splits - 1) / a.splits;
    chunk = (chunk + TBN - 1) / TBN * TBN;
    const int kb = err ? 0 : min(L, split * chunk);
    const int ke = err ? 0 : ((split == a.splits - 1) ? L + n : min(L, kb + chunk));
    const int T = err ? 0 : (ke - kb + TBN - 1) / TBN;
    const int kvz = b * a.Hkv + kvh;                               // (sequence, kv head) slab
    // A partial last tile is loaded ending at the last key (keys ke - TBN .. ke - 1), so it
    // reads no cache row past the keys: rows nobody wrote may hold NaN, and P = 0 does not
    // cancel NaN in the PV product.  Its keys below last_fresh are masked in the softmax:
    // they belong to the tile before, or lie before row 0 and arrive from TMA as zeros.
    const int last_fresh = T > 0 ? kb + (T - 1) * TBN : 0;         // first key the last tile adds
    const int last0 = (T > 0 && ke - last_fresh < TBN) ? ke - TBN : last_fresh;

    // ---- Q -> TMEM (softmax warps, one lane = one row), while K/V already stream ----
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
        if (lane == 0 && T > 0) {
            // ---------------- TMA producers: K (warp 0) and V (warp 2) ----------------
            // Two independent rings, so neither load waits behind the other's stage.
            const bool isK = warp == 0;
            const CUtensorMap* map = isK ? &tmap_k : &tmap_v;
            uint8_t* ring = isK ? sK : sV;
            uint64_t* full = isK ? bars->k_full : bars->v_full;
            uint64_t* empty = isK ? bars->k_empty : bars->v_empty;
            const int NS = isK ? KSTAGES : VSTAGES;
            for (int t = 0; t < T; ++t) {
                const int st = t % NS;
                if (!mbar_wait(s32(&empty[st]), (((uint32_t)t / NS) & 1u) ^ 1u, abort_flag)) break;
                // L2 prefetch kPrefetch tiles beyond the ring, paced with the loads
                if (t == 0) {
                    for (int jp = NS; jp < min(T, NS + kPrefetch); ++jp) {
                        tma_prefetch_3d(map, 0, kb + jp * TBN, kvz);
                        tma_prefetch_3d(map, 64, kb + jp * TBN, kvz);
                    }
                } else if (t + NS + kPrefetch - 1 < T) {
                    const int yp = kb + (t + NS + kPrefetch - 1) * TBN;
                    tma_prefetch_3d(map, 0, yp, kvz);
                    tma_prefetch_3d(map, 64, yp, kvz);
                }
                const uint32_t fb = s32(&full[st]);
                mbar_expect_tx(fb, K_BYTES);
                const int y = t == T - 1 ? last0 : kb + t * TBN;
                tma_load_3d(s32(ring + st * K_BYTES), map, fb, 0, y, kvz);
                tma_load_3d(s32(ring + st * K_BYTES + KV_BOX_BYTES), map, fb, 64, y, kvz);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && T > 0) {
            // ---------------- MMA issuer ----------------
            attn_common::mma_issue_loop<KSTAGES>(bars, tmem, sK, sV, T, abort_flag);
        }
    } else if (warp >= 4) {
        // ---------------- softmax: one thread per query row ----------------
        const int q4 = warp & 3;                         // TMEM lane quadrant
        const int rr = q4 * 32 + lane;
        const int r = row0 + rr;
        const bool valid = r < rows;
        const int i = valid ? r / G : 0;
        const unsigned long long anc = valid ? bars->anc[i] : 0ull;
        const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
        const uint32_t s_addr0 = tmem + lane_base + S_COL0;
        const uint32_t o_addr = tmem + lane_base + O_COL0;
        const float sc = a.scale_log2;
        float mref = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < T; ++j) {
            bool got = mbar_wait(s32(&bars->s_full[j % NSBUF]), ((uint32_t)j / NSBUF) & 1u, abort_flag);
            if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
            tc_fence_after();
            const uint32_t s_addr = s_addr0 + (uint32_t)((j % NSBUF) * TBN);
            float x[TBN];
            attn_common::load_scores(s_addr, x);
            const int key0 = j == T - 1 ? last0 : kb + j * TBN;
            if (key0 + TBN > L || key0 + TBN > ke || !valid || key0 < last_fresh && j == T - 1) {
                // visibility of the tile's keys as a 128-bit map: committed keys below L,
                // tree key L + t visible iff bit t of the ancestor mask, nothing from ke on
                uint64_t vis[2];
#pragma unroll
                for (int w = 0; w < 2; ++w) {
                    const int k0 = key0 + 64 * w;
                    const int nc = min(max(L - k0, 0), 64), ne = min(max(ke - k0, 0), 64);
                    const uint64_t committed = nc >= 64 ? ~0ull : ((1ull << nc) - 1ull);
                    const uint64_t upto = ne >= 64 ? ~0ull : ((1ull << ne) - 1ull);
                    const int sh = L - k0;                     // tree key t sits at bit t + sh
                    const uint64_t tree = (sh >= 64 || sh <= -64) ? 0ull
                                          : (sh >= 0 ? anc << sh : anc >> (-sh));
                    const int seen = last_fresh - k0;                 // keys below were counted
                    const uint64_t fresh = (j < T - 1 || seen <= 0) ? ~0ull
                                           : (seen >= 64 ? 0ull : ~((1ull << seen) - 1ull));
                    vis[w] = valid ? ((committed | tree) & upto & fresh) : 0ull;
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
        bool got = ok && T > 0 ? mbar_wait(s32(&bars->pv_done[(T - 1) % NSBUF]),
                                           ((uint32_t)(T - 1) / NSBUF) & 1u, abort_flag)
                               : false;
        got = __all_sync(0xffffffffu, got);
        tc_fence_after();
        const int h = kvh * G + (valid ? r % G : 0);
        const int64_t orow = ((int64_t)b * n + i) * a.Hq + h;
        const float inv = (got && l > 0.f) ? 1.f / l : 0.f;
        for (int cc = 0; cc < kHeadDim / 32; ++cc) {
            uint32_t o[32];
            if (got) tmem_ld32(o_addr + cc * 32, o);
            else
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = 0u;
            if (!valid) continue;
            if (a.splits == 1) {
                uint16_t* dst = a.out + orow * kHeadDim + cc * 32;
#pragma unroll
                for (int e = 0; e < 32; e += 8) {
                    const uint4 w = make_uint4(
                        pack2(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv),
                        pack2(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv),
                        pack2(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv),
                        pack2(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv));
                    *reinterpret_cast<uint4*>(dst + e) = w;
                }
            } else {
                const int64_t R = (int64_t)a.B * n * a.Hq;
                float* dst = a.ws_o + ((int64_t)split * R + orow) * kHeadDim + cc * 32;
#pragma unroll
                for (int e = 0; e < 32; e += 4)
                    *reinterpret_cast<float4*>(dst + e) =
                        make_float4(__uint_as_float(o[e]), __uint_as_float(o[e + 1]),
                                    __uint_as_float(o[e + 2]), __uint_as_float(o[e + 3]));
            }
        }
        if (valid && a.splits > 1) {
            const int64_t R = (int64_t)a.B * n * a.Hq;
            *reinterpret_cast<float2*>(a.ws_ml + ((int64_t)split * R + orow) * 2) =
                got ? make_float2(mref, l) : make_float2(-INFINITY, 0.f);
        }
    }
    __syncthreads();
    if (tid == 0 && *abort_flag) flag_error(a.dev_status, EAGLE_DEV_TIMEOUT);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace attn_tc
}  // namespace eagle
