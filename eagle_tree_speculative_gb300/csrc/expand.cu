// EAGLE-2 draft-tree expansion and reranking.
//
// Method (Guide "EAGLE-1/2/3 拆解", section "EAGLE-2：草稿树的 Expansion 与
// Reranking"; TTT page, section "EAGLE-3 和 EAGLE-2 动态树如何拼在一起"):
// node value V_i = product of draft confidences on the root path; expansion
// runs the draft forward only on the top-k nodes of the previous level;
// reranking keeps the global top-n nodes by V for verification.
//
// Kernels per level:
//   row_topk_kernel  one CTA per (frontier row, vocabulary segment): the
//                    segment's temperature-1 softmax statistics (max, sum of
//                    exponentials) and its top-k tokens (logit desc, token asc) in
//                    one pass; up to 4 segments per row spread the rows evenly
//                    over the SMs.
//   select_kernel    one CTA per sequence: merges each row's segments into the
//                    row's top-k and confidences c = exp(l - m) / Z, forms the
//                    k_in * k candidates of the level, V_child = V_parent * c in
//                    float32, the next frontier = the k best by (V desc, id asc),
//                    and assigns draft rows.
//   rerank_kernel    one CTA per sequence: bitonic sort of every candidate by
//                    (V desc, depth asc, id asc), keep n-1 plus the root, then
//                    sort those by (depth asc, V desc, id asc) and re-index parents.
// The draft LM-head GEMM (lmhead_gemm.cu) writes the level's logits rows first
// when hidden states are given.
#include <algorithm>
#include <map>
#include <vector>
#include <cstdlib>
#include <mutex>

#include "common.cuh"

namespace eagle {

// Defined in lmhead_gemm.cu.
eagle_status lmhead_gemm_launch(const void* hidden, const void* w, float* out, int M, int K, int N,
                                int64_t ldo, int rows_per_group, int64_t group_stride,
                                int64_t row_offset, int32_t* dev_status, cudaStream_t stream,
                                float* part);
constexpr int kGemmBN = 256;                    // columns per GEMM N-tile (one partial each)

namespace {

constexpr int kKMax = 16;
constexpr int kDepthMax = 16;
constexpr int kSegMax = 4;        // vocabulary segments per draft row

// Per-sequence tree state, 32-bit words:
//   [0..3] reserved
//   value[C] f32, parent[C], token[C], depth[C], row[C], conf[C] f32 (the draft
//   confidence c of each candidate; V of a candidate = V of its parent * c),
//   frontier[kKMax],
//   per (frontier row s < k, segment g < kSegMax), at index s * kSegMax + g:
//   seg_stat[3] (max f32, sum f32, non-finite flag), seg_val[k] f32, seg_tok[k]
struct StateView {
    __host__ __device__ static int cand_count(int k, int D) { return 1 + k + (D - 1) * k * k; }
    __host__ __device__ static int64_t words(int k, int D) {
        return 4 + 6LL * cand_count(k, D) + kKMax + (int64_t)k * kSegMax * (3 + 2LL * k);
    }
};

struct SeqState {
    int* hdr;
    float* value;
    int* parent;
    int* token;
    int* depth;
    int* row;
    float* conf;
    int* frontier;
    int* seg_stat;    // [k * kSegMax][3]
    float* seg_val;   // [k * kSegMax][k]
    int* seg_tok;     // [k * kSegMax][k]
};

__device__ __forceinline__ SeqState seq_state(void* base, int b, int k, int D) {
    const int C = StateView::cand_count(k, D);
    int* p = static_cast<int*>(base) + (int64_t)b * StateView::words(k, D);
    SeqState s;
    s.hdr = p;
    s.value = reinterpret_cast<float*>(p + 4);
    s.parent = p + 4 + C;
    s.token = p + 4 + 2 * C;
    s.depth = p + 4 + 3 * C;
    s.row = p + 4 + 4 * C;
    s.conf = reinterpret_cast<float*>(p + 4 + 5 * C);
    s.frontier = p + 4 + 6 * C;
    s.seg_stat = s.frontier + kKMax;
    s.seg_val = reinterpret_cast<float*>(s.seg_stat + 3 * k * kSegMax);
    s.seg_tok = s.seg_stat + 3 * k * kSegMax + k * k * kSegMax;
    return s;
}

__device__ __forceinline__ bool topk_better(float v, int i, float w, int j) {
    return v > w || (v == w && i < j);
}

// ---------------------------------------------------------------------------
// Segment softmax statistics + top-k in one pass over the segment.
// Statistics: each thread keeps an online (max, sum) with sum = sum
// 2^((l - max) log2 e).  Top-k: each warp keeps ONE sorted list distributed
// over its lanes (lane j holds the j-th best, order: logit desc, token asc).
// Every lane loads 8 float4 chunks before using them.  Before the first chunks
// are used, each warp takes the k-th largest of its 32 lane maxima over them:
// k elements of the segment reach it, so it bounds the segment's k-th best from
// below, and the block keeps the largest such bound in shared memory (raised
// again whenever a warp's own k-th best passes it).  A chunk is tested through
// its maximum against that threshold (one vote per chunk); the rare surviving
// elements are inserted one at a time with a shuffle shift.  At the end every
// entry of the per-warp lists finds its rank among all of them in parallel, and
// the segment's statistics and top-k go to the tree state.
constexpr int kTopkThreads = 256;
constexpr int kTopkWarps = kTopkThreads / 32;

// The k best entries of the kTopkWarps warp lists in s_v / s_i (list w at w * kKMax, each
// sorted best first, empty entries (-inf, 0x7fffffff)) into m_v / m_i in order, merged
// by one warp: lane w < kTopkWarps holds the head of list w, a butterfly over those lanes
// finds the best head (the order is strict, so every lane agrees), and its lane moves on.
__device__ __forceinline__ void merge_warp_lists(const float* s_v, const int* s_i, int k, float* m_v,
                                                 int* m_i) {
    static_assert((kTopkWarps & (kTopkWarps - 1)) == 0 && kTopkWarps <= 32, "butterfly over the lists");
    const int lane = threadIdx.x & 31;
    int p = 0;
    for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int bi = 0x7fffffff, bl = lane;
        if (lane < kTopkWarps && p < k) {
            bv = s_v[lane * kKMax + p];
            bi = s_i[lane * kKMax + p];
        }
#pragma unroll
        for (int o = kTopkWarps / 2; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            const int ol = __shfl_xor_sync(0xffffffffu, bl, o);
            if (topk_better(ov, oi, bv, bi)) { bv = ov; bi = oi; bl = ol; }
        }
        if (lane == bl && bi != 0x7fffffff) ++p;
        if (lane == 0) { m_v[j] = bv; m_i[j] = bi; }
    }
}

constexpr int kTopkUnroll = 8;                 // float4 loads in flight per thread
constexpr int kSegMinElems = 8192;             // shortest segment worth its own CTA
constexpr float kLog2e = 1.4426950408889634f;

// Insert (v, i) into the warp list (lv, li) sorted desc; all lanes call with the
// same (v, i).  Returns nothing; the list keeps its 32 best entries.
__device__ __forceinline__ void warp_list_insert(float& lv, int& li, float v, int i) {
    const int lane = threadIdx.x & 31;
    const bool gt = topk_better(v, i, lv, li);            // candidate beats my entry
    const float pv = __shfl_up_sync(0xffffffffu, lv, 1);
    const int pi = __shfl_up_sync(0xffffffffu, li, 1);
    const bool pgt = __shfl_up_sync(0xffffffffu, gt ? 1 : 0, 1) != 0;
    if (gt) {
        if (lane == 0 || !pgt) { lv = v; li = i; }
        else { lv = pv; li = pi; }
    }
}

// The j-th largest of the warp's 32 values (bitonic sort, descending).
__device__ __forceinline__ float warp_kth_largest(float x, int j) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const float y = __shfl_xor_sync(0xffffffffu, x, stride);
            const bool desc = (lane & size) == 0;               // direction of this block
            const bool lower = (lane & stride) == 0;
            x = (lower == desc) ? fmaxf(x, y) : fminf(x, y);
        }
    return __shfl_sync(0xffffffffu, x, j);
}

// Segments per row: one when the rows alone give every SM two CTAs, otherwise
// enough (at most kSegMax, none shorter than kSegMinElems) to come close.
int topk_segments(int V, int rows, int sms) {
    if (rows >= 2 * sms) return 1;
    int sgs = (2 * sms + rows - 1) / rows;
    const int by_len = (V + kSegMinElems - 1) / kSegMinElems;
    sgs = sgs < by_len ? sgs : by_len;
    return sgs < 1 ? 1 : (sgs > kSegMax ? kSegMax : sgs);
}

__device__ __forceinline__ float ex2f_fast(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

__global__ void __launch_bounds__(kTopkThreads, 5)
row_topk_kernel(const float* __restrict__ logits, int k_in, int R, int off, int V, int k, int D,
                int nseg, void* state) {
    __shared__ float s_v[kTopkWarps * kKMax];
    __shared__ int s_i[kTopkWarps * kKMax];
    __shared__ float s_red[kTopkWarps][2];
    __shared__ int s_bad[kTopkWarps];
    __shared__ float s_thr;                    // a lower bound on the block's k-th best
    __shared__ float s_mv[kKMax];
    __shared__ int s_mi[kKMax];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) s_thr = -INFINITY;
    volatile float* thr_p = &s_thr;
    const int row = blockIdx.x / nseg, seg = blockIdx.x % nseg;
    const int b = row / k_in, s = row % k_in;
    const float* x = logits + ((int64_t)b * R + off + s) * (int64_t)V;
    // segment [e0, e1), a multiple of 4 elements long except at the end of the row
    const int seg_len = ((V + nseg - 1) / nseg + 3) & ~3;
    const int e0 = min(V, seg * seg_len), e1 = min(V, e0 + seg_len);

    float lv = -INFINITY;            // warp list entry of this lane
    int li = 0x7fffffff;
    float tv = -INFINITY;            // the warp's current k-th best (broadcast)
    int ti = 0x7fffffff;
    float m = -INFINITY, sum = 0.f;
    int bad = 0;
    float thr = -INFINITY;

    // lanes whose candidate beats the warp's k-th best and reaches the block's
    // threshold insert it, one at a time
    auto offer = [&](float v, int i, bool mine) {
        unsigned ball = __ballot_sync(0xffffffffu, mine && v >= thr && topk_better(v, i, tv, ti));
        while (ball) {
            const int src = __ffs(ball) - 1;
            ball &= ball - 1;
            const float cv = __shfl_sync(0xffffffffu, v, src);
            const int ci = __shfl_sync(0xffffffffu, i, src);
            if (topk_better(cv, ci, tv, ti)) {
                warp_list_insert(lv, li, cv, ci);
                tv = __shfl_sync(0xffffffffu, lv, k - 1);
                ti = __shfl_sync(0xffffffffu, li, k - 1);
                // publish a raised k-th best (a lost race only leaves a lower bound)
                if (lane == 0 && tv > *thr_p) *thr_p = tv;
            }
        }
    };

    if (((V & 3) == 0) && ((reinterpret_cast<uintptr_t>(logits) & 15) == 0)) {
        const float4* x4 = reinterpret_cast<const float4*>(x + e0);
        const int n4 = (e1 - e0) >> 2;
        // block-uniform trip counts: every lane runs every iteration (votes)
        for (int base = 0; base < n4; base += kTopkUnroll * kTopkThreads) {
            float4 c[kTopkUnroll];
#pragma unroll
            for (int u = 0; u < kTopkUnroll; ++u) {
                const int t = base + u * kTopkThreads + tid;
                c[u] = t < n4 ? __ldg(x4 + t) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            }
            if (base == 0) {
                // seed the threshold: the k-th largest lane maximum of each warp
                float lmax = -INFINITY;
#pragma unroll
                for (int u = 0; u < kTopkUnroll; ++u)
                    lmax = fmaxf(lmax, fmaxf(fmaxf(c[u].x, c[u].y), fmaxf(c[u].z, c[u].w)));
                const float est = warp_kth_largest(lmax, k - 1);
                __syncthreads();                               // s_thr initialised
                if (lane == 0 && est > *thr_p) *thr_p = est;
                __syncthreads();
            }
            thr = fmaxf(tv, *thr_p);
#pragma unroll
            for (int u = 0; u < kTopkUnroll; ++u) {
                const int t = base + u * kTopkThreads + tid;
                const bool valid = t < n4;
                const float4 l4 = c[u];
                const float cm = fmaxf(fmaxf(l4.x, l4.y), fmaxf(l4.z, l4.w));
                if (valid) {
                    // NaN or +inf anywhere in the chunk makes its sum NaN or +inf
                    const float s4 = (l4.x + l4.y) + (l4.z + l4.w);
                    bad |= (s4 != s4) | (s4 == INFINITY);
                    if (cm > m) {
                        sum = (m == -INFINITY) ? 0.f : sum * ex2f_fast((m - cm) * kLog2e);
                        m = cm;
                    }
                    if (m != -INFINITY)
                        sum += ex2f_fast((l4.x - m) * kLog2e) + ex2f_fast((l4.y - m) * kLog2e) +
                               ex2f_fast((l4.z - m) * kLog2e) + ex2f_fast((l4.w - m) * kLog2e);
                }
                // a chunk can only contribute if its maximum reaches the threshold
                if (__any_sync(0xffffffffu, valid && cm >= thr)) {
                    const int i0 = e0 + 4 * t;
                    offer(l4.x, i0, valid);
                    offer(l4.y, i0 + 1, valid);
                    offer(l4.z, i0 + 2, valid);
                    offer(l4.w, i0 + 3, valid);
                    thr = fmaxf(tv, *thr_p);
                }
            }
        }
    } else {
        __syncthreads();                                       // s_thr initialised
        for (int base = e0; base < e1; base += kTopkThreads) {
            const int t = base + tid;
            const bool ok = t < e1;
            const float l = ok ? x[t] : 0.f;
            if (ok) {
                bad |= (l != l) | (l == INFINITY);
                if (l > m) {
                    sum = (m == -INFINITY) ? 0.f : sum * ex2f_fast((m - l) * kLog2e);
                    m = l;
                }
                if (m != -INFINITY) sum += ex2f_fast((l - m) * kLog2e);
            }
            offer(l, t, ok);
        }
    }
    // combine (max, sum) across the warp in the exp2 domain
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, m, o);
        const float os = __shfl_xor_sync(0xffffffffu, sum, o);
        if (om != -INFINITY) {
            if (m == -INFINITY) { m = om; sum = os; }
            else {
                const float nm = fmaxf(m, om);
                sum = sum * ex2f_fast((m - nm) * kLog2e) + os * ex2f_fast((om - nm) * kLog2e);
                m = nm;
            }
        }
    }
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) { s_red[warp][0] = m; s_red[warp][1] = sum; s_bad[warp] = bad; }
    if (lane < k) { s_v[warp * kKMax + lane] = lv; s_i[warp * kKMax + lane] = li; }
    __syncthreads();
    SeqState st = seq_state(state, b, k, D);
    const int slot = s * kSegMax + seg;
    if (warp == 0) {
        // the segment's top-k in order; a segment shorter than k leaves empty entries
        merge_warp_lists(s_v, s_i, k, s_mv, s_mi);
        __syncwarp();
        if (lane < k) {
            const bool has = s_mi[lane] != 0x7fffffff;
            st.seg_val[slot * k + lane] = has ? s_mv[lane] : -INFINITY;
            st.seg_tok[slot * k + lane] = has ? s_mi[lane] : 0x7fffffff;
        }
    }
    if (tid == 0) {
        float M = -INFINITY, S = 0.f;
        int bd = 0;
        for (int w = 0; w < kTopkWarps; ++w) {
            const float wm = s_red[w][0], ws = s_red[w][1];
            bd |= s_bad[w];
            if (wm == -INFINITY) continue;
            if (M == -INFINITY) { M = wm; S = ws; continue; }
            const float nm = fmaxf(M, wm);
            S = S * ex2f_fast((M - nm) * kLog2e) + ws * ex2f_fast((wm - nm) * kLog2e);
            M = nm;
        }
        st.seg_stat[3 * slot] = __float_as_int(M);
        st.seg_stat[3 * slot + 1] = __float_as_int(S);
        st.seg_stat[3 * slot + 2] = bd;
    }
}

// ---------------------------------------------------------------------------
// Top-k of a draft row from the LM-head GEMM's per-tile partials (fused path).
// Each 256-column tile of the row has (max, sum of 2^((l - max) log2 e)) from the
// GEMM's epilogue.  The row's statistics combine those in the exp2 domain.  Its
// top-k: tau = the k-th largest tile maximum bounds the row's k-th best from below
// (k tiles reach it), so every top-k entry lies in a tile whose maximum is >= tau;
// only those tiles (about k of them) are read back from the logits row and fed to
// the same warp lists as row_topk_kernel.  Exact, ties included.  The result goes
// to segment 0 of the row in the tree state.
constexpr int kMergeMaxTiles = 8192;                 // rows up to 2M columns

__global__ void __launch_bounds__(kTopkThreads)
topk_merge_kernel(const float* __restrict__ part, const float* __restrict__ logits, int k_in, int R,
                  int off, int V, int num_n, int k, int D, void* state) {
    __shared__ float s_v[kTopkWarps * kKMax];
    __shared__ int s_i[kTopkWarps * kKMax];
    __shared__ float s_red[kTopkWarps][2];
    __shared__ int s_bad[kTopkWarps];
    __shared__ float s_mv[kKMax];
    __shared__ int s_mi[kKMax];
    __shared__ float s_tau;
    __shared__ int s_nsel;
    __shared__ int s_sel[kMergeMaxTiles];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int row = blockIdx.x, b = row / k_in, s = row % k_in;
    const float2* P = reinterpret_cast<const float2*>(part) + (int64_t)row * num_n;
    const float* x = logits + ((int64_t)b * R + off + s) * (int64_t)V;
    if (tid == 0) s_nsel = 0;

    float lv = -INFINITY, tv = -INFINITY, thr = -INFINITY;
    int li = 0x7fffffff, ti = 0x7fffffff;
    auto offer = [&](float v, int i, bool mine) {
        unsigned ball = __ballot_sync(0xffffffffu, mine && v >= thr && topk_better(v, i, tv, ti));
        while (ball) {
            const int src = __ffs(ball) - 1;
            ball &= ball - 1;
            const float cv = __shfl_sync(0xffffffffu, v, src);
            const int ci = __shfl_sync(0xffffffffu, i, src);
            if (topk_better(cv, ci, tv, ti)) {
                warp_list_insert(lv, li, cv, ci);
                tv = __shfl_sync(0xffffffffu, lv, k - 1);
                ti = __shfl_sync(0xffffffffu, li, k - 1);
            }
        }
    };

    // ---- pass 1: statistics, and the k largest tile maxima ----
    float m = -INFINITY, sum = 0.f;
    int bad = 0;
    for (int base = 0; base < num_n; base += kTopkThreads) {      // block-uniform trip count
        const int t = base + tid;
        const bool ok = t < num_n;
        const float2 pr = ok ? P[t] : make_float2(-INFINITY, 0.f);
        if (ok) {
            bad |= (pr.y != pr.y) | (pr.x == INFINITY);
            if (pr.x != -INFINITY) {
                if (m == -INFINITY) { m = pr.x; sum = pr.y; }
                else {
                    const float nm = fmaxf(m, pr.x);
                    sum = sum * ex2f_fast((m - nm) * kLog2e) + pr.y * ex2f_fast((pr.x - nm) * kLog2e);
                    m = nm;
                }
            }
        }
        offer(pr.x, t, ok);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, m, o);
        const float os = __shfl_xor_sync(0xffffffffu, sum, o);
        if (om != -INFINITY) {
            if (m == -INFINITY) { m = om; sum = os; }
            else {
                const float nm = fmaxf(m, om);
                sum = sum * ex2f_fast((m - nm) * kLog2e) + os * ex2f_fast((om - nm) * kLog2e);
                m = nm;
            }
        }
    }
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) { s_red[warp][0] = m; s_red[warp][1] = sum; s_bad[warp] = bad; }
    if (lane < k) { s_v[warp * kKMax + lane] = lv; s_i[warp * kKMax + lane] = li; }
    __syncthreads();
    if (warp == 0) {
        // the k-th largest tile maximum (fewer tiles: -inf)
        merge_warp_lists(s_v, s_i, k, s_mv, s_mi);
        __syncwarp();
        if (lane == 0) s_tau = s_mi[k - 1] != 0x7fffffff ? s_mv[k - 1] : -INFINITY;
    }
    __syncthreads();
    const float tau = s_tau;
    // ---- the tiles that can hold a top-k entry ----
    for (int t = tid; t < num_n; t += kTopkThreads)
        if (P[t].x >= tau) s_sel[atomicAdd(&s_nsel, 1)] = t;
    __syncthreads();
    const int nsel = s_nsel;
    // ---- pass 2: those tiles' logits, one warp per tile ----
    lv = -INFINITY; tv = -INFINITY; li = 0x7fffffff; ti = 0x7fffffff;
    thr = tau;
    const bool vec4 = ((V & 3) == 0) && ((reinterpret_cast<uintptr_t>(logits) & 15) == 0);
    for (int q = warp; q < nsel; q += kTopkWarps) {                  // warp-uniform
        const int c0 = s_sel[q] * kGemmBN;
        const int c1 = min(V, c0 + kGemmBN);
        if (vec4 && c1 - c0 == kGemmBN) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int c = c0 + 128 * h + 4 * lane;
                const float4 l4 = __ldg(reinterpret_cast<const float4*>(x + c));
                offer(l4.x, c, true);
                offer(l4.y, c + 1, true);
                offer(l4.z, c + 2, true);
                offer(l4.w, c + 3, true);
            }
        } else {
            for (int c = c0 + lane; c < c0 + kGemmBN; c += 32) {
                const bool ok = c < c1;
                offer(ok ? x[c] : -INFINITY, c, ok);
            }
        }
    }
    __syncthreads();                                  // everyone is done with s_v / s_i
    if (lane < k) { s_v[warp * kKMax + lane] = lv; s_i[warp * kKMax + lane] = li; }
    __syncthreads();
    SeqState st = seq_state(state, b, k, D);
    const int slot = s * kSegMax;
    if (warp == 0) {
        // the row's top-k in order; missing entries (a row shorter than k) stay empty
        merge_warp_lists(s_v, s_i, k, s_mv, s_mi);
        __syncwarp();
        if (lane < k) {
            const bool has = s_mi[lane] != 0x7fffffff;
            st.seg_val[slot * k + lane] = has ? s_mv[lane] : -INFINITY;
            st.seg_tok[slot * k + lane] = has ? s_mi[lane] : 0x7fffffff;
        }
    }
    if (tid == 0) {
        float M = -INFINITY, S = 0.f;
        int bd = 0;
        for (int w = 0; w < kTopkWarps; ++w) {
            const float wm = s_red[w][0], ws = s_red[w][1];
            bd |= s_bad[w];
            if (wm == -INFINITY) continue;
            if (M == -INFINITY) { M = wm; S = ws; continue; }
            const float nm = fmaxf(M, wm);
            S = S * ex2f_fast((M - nm) * kLog2e) + ws * ex2f_fast((wm - nm) * kLog2e);
            M = nm;
        }
        st.seg_stat[3 * slot] = __float_as_int(M);
        st.seg_stat[3 * slot + 1] = __float_as_int(S);
        st.seg_stat[3 * slot + 2] = bd;
    }
}

// ---------------------------------------------------------------------------
constexpr int kSelectThreads = 256;

__global__ void __launch_bounds__(kSelectThreads)
select_kernel(int level, int final, int k, int D, int nseg, void* state, int32_t* frontier_tokens,
              const int32_t* d2t, int32_t* dev_status) {
    __shared__ float s_val[kKMax * kKMax];
    __shared__ int s_id[kKMax * kKMax];
    __shared__ float s_conf[kKMax * kKMax];     // [row s][rank j]: confidence of the row's j-th best
    __shared__ int s_tok[kKMax * kKMax];
    __shared__ float s_rowM[kKMax], s_rowS[kKMax];
    const int tid = threadIdx.x, b = blockIdx.x;
    SeqState st = seq_state(state, b, k, D);
    const int k_in = level == 1 ? 1 : k;
    // ---- each row's softmax statistics from its segments ----
    if (tid < k_in) {
        float M = -INFINITY, S = 0.f;
        int bd = 0;
        for (int g = 0; g < nseg; ++g) {
            const int slot = tid * kSegMax + g;
            const float gm = __int_as_float(st.seg_stat[3 * slot]);
            const float gs = __int_as_float(st.seg_stat[3 * slot + 1]);
            bd |= st.seg_stat[3 * slot + 2];
            if (gm == -INFINITY) continue;
            if (M == -INFINITY) { M = gm; S = gs; continue; }
            const float nm = fmaxf(M, gm);
            S = S * exp2f((M - nm) * kLog2e) + gs * exp2f((gm - nm) * kLog2e);
            M = nm;
        }
        if (bd || M == -INFINITY) flag_error(dev_status, EAGLE_DEV_NONFINITE);
        s_rowM[tid] = M;
        s_rowS[tid] = S;
    }
    __syncthreads();
    // ---- each row's top-k: rank of every segment entry among the row's entries (one
    // segment is already in rank order) ----
    for (int e = tid; e < k_in * nseg * k; e += kSelectThreads) {
        const int row = e / (nseg * k), r = e % (nseg * k);
        const int base = row * kSegMax * k;                 // first entry of the row
        const float v = st.seg_val[base + r];
        const int i = st.seg_tok[base + r];
        int rank = r;
        if (nseg > 1) {
            rank = 0;
            for (int f = 0; f < nseg * k; ++f)
                rank += topk_better(st.seg_val[base + f], st.seg_tok[base + f], v, i);
        }
        if (rank < k) {
            s_tok[row * kKMax + rank] = i;
            s_conf[row * kKMax + rank] = exp2f((v - s_rowM[row]) * kLog2e) / s_rowS[row];
        }
    }
    __syncthreads();
    if (level == 1 && tid == 0) {
        st.value[0] = 1.0f;
        st.parent[0] = -1;
        st.token[0] = -1;
        st.depth[0] = 0;
        st.row[0] = 0;
        st.conf[0] = 1.0f;
        st.frontier[0] = 0;
    }
    __syncthreads();
    const int ncand = k_in * k;
    for (int e = tid; e < ncand; e += kSelectThreads) {
        const int s = e / k, j = e % k;
        const int id = level == 1 ? 1 + j : 1 + k + (level - 2) * k * k + s * k + j;
        const int par = st.frontier[s];
        const float c = s_conf[s * kKMax + j];
        const float val = __fmul_rn(st.value[par], c);
        st.value[id] = val;
        st.conf[id] = c;
        st.parent[id] = par;
        const int tk = s_tok[s * kKMax + j];            // id in the logits' vocabulary
        st.token[id] = d2t ? tk + d2t[tk] : tk;         // draft id -> target id
        st.depth[id] = level;
        st.row[id] = -1;
        s_val[e] = val;
        s_id[e] = id;
    }
    __syncthreads();
    // the k best candidates in (V desc, id asc) form the frontier.  Row s's candidates
    // s * k .. s * k + k - 1 are already in that order (V = value[parent] * c with c
    // non-increasing in j, ids increasing), so one warp merges the k_in rows: lane s holds
    // the head of row s, a butterfly finds the best head, and its lane moves on.
    static_assert(kKMax <= 16, "the merge spans 16 lanes");
    if (tid < 32) {
        const int lane = tid;
        int p = 0;
        for (int rank = 0; rank < k; ++rank) {
            float bv = -INFINITY;
            int bi = 0x7fffffff, bl = lane;
            if (lane < k_in && p < k) { bv = s_val[lane * k + p]; bi = s_id[lane * k + p]; }
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                const int ol = __shfl_xor_sync(0xffffffffu, bl, o);
                if (topk_better(ov, oi, bv, bi)) { bv = ov; bi = oi; bl = ol; }
            }
            if (lane == bl && bi != 0x7fffffff) ++p;
            if (lane == 0 && bi != 0x7fffffff) {
                st.frontier[rank] = bi;
                if (level < D && !final) st.row[bi] = 1 + (level - 1) * k + rank;
                if (frontier_tokens) frontier_tokens[(int64_t)b * k + rank] = st.token[bi];
            }
        }
    }
}

// ---------------------------------------------------------------------------
constexpr int kRerankThreads = 512;

__device__ void bitonic_sort(unsigned long long* keys, int n2) {
    for (int size = 2; size <= n2; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = threadIdx.x; i < n2; i += blockDim.x) {
                int j = i ^ stride;
                if (j > i) {
                    bool up = (i & size) == 0;
                    unsigned long long a = keys[i], c = keys[j];
                    if ((a > c) == up) { keys[i] = c; keys[j] = a; }
                }
            }
            __syncthreads();
        }
    }
}

__global__ void __launch_bounds__(kRerankThreads)
rerank_kernel(int k, int D, int level, int n_out, const void* state, int32_t* out_tokens,
              int32_t* out_parent, int32_t* out_row) {
    extern __shared__ unsigned long long s_keys[];
    const int b = blockIdx.x, tid = threadIdx.x;
    const int C = StateView::cand_count(k, level);      // candidates generated so far
    int n2 = 1;
    while (n2 < C - 1) n2 <<= 1;
    int* s_node = reinterpret_cast<int*>(s_keys + n2);     // candidate id -> node index
    __shared__ int s_sel[kMaxNodes];
    SeqState st = seq_state(const_cast<void*>(state), b, k, D);
    // key 1: (V desc, depth asc, id asc); V >= 0 so its bit pattern orders it
    for (int i = tid; i < n2; i += blockDim.x) {
        unsigned long long key = ~0ull;
        if (i < C - 1) {
            const int id = i + 1;
            const unsigned vb = __float_as_uint(st.value[id]);
            key = ((unsigned long long)(0xffffffffu - vb) << 17) |
                  ((unsigned long long)st.depth[id] << 12) | (unsigned long long)id;
        }
        s_keys[i] = key;
    }
    for (int i = tid; i < C; i += blockDim.x) s_node[i] = -1;
    __syncthreads();
    bitonic_sort(s_keys, n2);
    // key 2 over the kept n-1: (depth asc, V desc, id asc); n-1 <= 63 -> 64 slots
    __shared__ unsigned long long s_k2[64];
    if (tid < 64) {
        unsigned long long key = ~0ull;
        if (tid < n_out - 1) {
            const int id = (int)(s_keys[tid] & 0xfffull);
            const unsigned vb = __float_as_uint(st.value[id]);
            key = ((unsigned long long)st.depth[id] << 44) |
                  ((unsigned long long)(0xffffffffu - vb) << 12) | (unsigned long long)id;
        }
        s_k2[tid] = key;
    }
    __syncthreads();
    bitonic_sort(s_k2, 64);
    if (tid == 0) {
        s_sel[0] = 0;
        s_node[0] = 0;
    }
    if (tid < n_out - 1) {
        const int id = (int)(s_k2[tid] & 0xfffull);
        s_sel[tid + 1] = id;
        s_node[id] = tid + 1;
    }
    __syncthreads();
    if (tid < n_out) {
        const int id = s_sel[tid];
        const int64_t o = (int64_t)b * n_out + tid;
        out_tokens[o] = tid == 0 ? -1 : st.token[id];
        out_parent[o] = tid == 0 ? -1 : s_node[st.parent[id]];
        out_row[o] = st.row[id];
    }
}

// ---------------------------------------------------------------------------
// Copy of every candidate's fields out of the tree state, [B, C] per field.
__global__ void tree_candidates_kernel(const void* state, int k, int D, float* value, float* conf,
                                       int32_t* token, int32_t* parent, int32_t* depth,
                                       int32_t* row) {
    const int b = blockIdx.y;
    const int C = StateView::cand_count(k, D);
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= C) return;
    SeqState st = seq_state(const_cast<void*>(state), b, k, D);
    const int64_t o = (int64_t)b * C + i;
    if (value) value[o] = st.value[i];
    if (conf) conf[o] = st.conf[i];
    if (token) token[o] = st.token[i];
    if (parent) parent[o] = st.parent[i];
    if (depth) depth[o] = st.depth[i];
    if (row) row[o] = st.row[i];
}

}  // namespace
}  // namespace eagle

using namespace eagle;

extern "C" size_t eagle2_tree_state_size(int B, int top_k, int depth) {
    if (B < 0 || top_k < 1 || top_k > kKMax || depth < 1 || depth > kDepthMax) return 0;
    return (size_t)B * (size_t)StateView::words(top_k, depth) * 4u;
}

extern "C" size_t eagle2_expand_scratch_size(int B, int V, int top_k) {
    if (B < 0 || V < 1 || top_k < 1 || top_k > kKMax) return 0;
    const size_t tiles = ((size_t)V + kGemmBN - 1) / kGemmBN;
    return (size_t)B * top_k * tiles * 2 * 4u;
}

namespace eagle {
namespace {
// Host checks of one expansion level that do not involve the tree state or the
// partials (shared by the scratch and the fixed-array entry points).
eagle_status expand_validate(int level, int final, const void* hidden, const void* lm_head_w,
                             const float* logits, int B, int H, int V, int top_k, int depth,
                             int n_out, const int32_t* out_tokens, const int32_t* out_parent,
                             const int32_t* out_draft_row) {
    if (B < 0 || V < 1 || top_k < 1 || depth < 1 || level < 1 || level > depth)
        return EAGLE_ERR_INVALID_ARG;
    if (top_k > kKMax || depth > kDepthMax || top_k > V) return EAGLE_ERR_SHAPE;
    if (StateView::cand_count(top_k, depth) > 4096) return EAGLE_ERR_SHAPE;
    if (final) {
        if (n_out < 2 || n_out > kMaxNodes) return EAGLE_ERR_SHAPE;
        const int have = 1 + top_k + (level - 1) * top_k * top_k;
        if (n_out > have) return EAGLE_ERR_SHAPE;
    }
    if (hidden && H < 1) return EAGLE_ERR_INVALID_ARG;
    if (B == 0) return EAGLE_OK;                        // pointers unused: nothing read or written
    if (!logits) return EAGLE_ERR_INVALID_ARG;
    if (final && (!out_tokens || !out_parent || !out_draft_row)) return EAGLE_ERR_INVALID_ARG;
    if (hidden && !lm_head_w) return EAGLE_ERR_INVALID_ARG;
    return EAGLE_OK;
}

eagle_status expand_common(int level, int final, const void* hidden, const void* lm_head_w,
                           float* logits, int B, int H, int V, int top_k, int depth, int n_out,
                           void* tree_state, size_t state_bytes, float* partials,
                           size_t partials_bytes, const int32_t* d2t, int32_t* out_tokens,
                           int32_t* out_parent, int32_t* out_draft_row, int32_t* frontier_tokens,
                           int32_t* dev_status, eagle_stream_t stream) {
    const eagle_status vs = expand_validate(level, final, hidden, lm_head_w, logits, B, H, V,
                                            top_k, depth, n_out, out_tokens, out_parent,
                                            out_draft_row);
    if (vs != EAGLE_OK) return vs;
    if (B == 0) return EAGLE_OK;
    if (!tree_state) return EAGLE_ERR_INVALID_ARG;
    if (state_bytes < eagle2_tree_state_size(B, top_k, depth)) return EAGLE_ERR_CAPACITY;
    // fused top-k: every 256-column tile of a row was (or is now) reduced by the
    // GEMM's epilogue to its statistics and top-k; only those partials are merged
    const bool fused = partials != nullptr;
    if (fused && (partials_bytes < eagle2_expand_scratch_size(B, V, top_k) ||
                  (reinterpret_cast<uintptr_t>(partials) & 7)))
        return EAGLE_ERR_CAPACITY;
    if (fused && (V + kGemmBN - 1) / kGemmBN > kMergeMaxTiles) return EAGLE_ERR_SHAPE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int R = 1 + (depth - 1) * top_k;
    const int k_in = level == 1 ? 1 : top_k;
    const int off = level == 1 ? 0 : 1 + (level - 2) * top_k;
    if (hidden) {
        eagle_status st = lmhead_gemm_launch(hidden, lm_head_w, logits, B * k_in, H, V, V, k_in,
                                             (int64_t)R, off, dev_status, s,
                                             partials);
        if (st != EAGLE_OK) return st;
    }
    int nseg = 1;
    if (fused) {
        const int num_n = (V + kGemmBN - 1) / kGemmBN;
        topk_merge_kernel<<<B * k_in, kTopkThreads, 0, s>>>(partials, logits, k_in, R, off, V,
                                                            num_n, top_k, depth, tree_state);
    } else {
        nseg = topk_segments(V, B * k_in, device_sm_count());
        row_topk_kernel<<<B * k_in * nseg, kTopkThreads, 0, s>>>(logits, k_in, R, off, V, top_k,
                                                                depth, nseg, tree_state);
    }
    EAGLE_CHECK_LAUNCH();
    select_kernel<<<B, kSelectThreads, 0, s>>>(level, final, top_k, depth, nseg, tree_state,
                                                 frontier_tokens, d2t, dev_status);
    EAGLE_CHECK_LAUNCH();
    if (final) {
        const int Cl = StateView::cand_count(top_k, level);
        int n2 = 1;
        while (n2 < Cl - 1) n2 <<= 1;
        const size_t smem = (size_t)n2 * 8 + (size_t)Cl * 4;
        if (smem > 48 * 1024 &&
            cudaFuncSetAttribute(rerank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) != cudaSuccess)
            return EAGLE_ERR_CUDA;
        rerank_kernel<<<B, kRerankThreads, smem, s>>>(top_k, depth, level, n_out, tree_state,
                                                      out_tokens, out_parent, out_draft_row);
        EAGLE_CHECK_LAUNCH();
    }
    return EAGLE_OK;
}

}  // namespace
}  // namespace eagle

extern "C" eagle_status eagle2_expand(int level, int final, const void* hidden, const void* lm_head_w,
                                      float* logits, int B, int H, int V, int top_k, int depth,
                                      int n_out, void* tree_state, size_t state_bytes,
                                      float* partials, size_t partials_bytes, int32_t* out_tokens,
                                      int32_t* out_parent, int32_t* out_draft_row,
                                      int32_t* frontier_tokens, int32_t* dev_status,
                                      eagle_stream_t stream) {
    return expand_common(level, final, hidden, lm_head_w, logits, B, H, V, top_k, depth, n_out,
                         tree_state, state_bytes, partials, partials_bytes, nullptr, out_tokens,
                         out_parent, out_draft_row, frontier_tokens, dev_status, stream);
}

extern "C" eagle_status eagle2_expand_d2t(int level, int final, const void* hidden,
                                          const void* lm_head_w, float* logits, int B, int H, int V,
                                          int top_k, int depth, int n_out, void* tree_state,
                                          size_t state_bytes, float* partials,
                                          size_t partials_bytes, const int32_t* d2t,
                                          int32_t* out_tokens, int32_t* out_parent,
                                          int32_t* out_draft_row, int32_t* frontier_tokens,
                                          int32_t* dev_status, eagle_stream_t stream) {
    if (B != 0 && !d2t) return EAGLE_ERR_INVALID_ARG;
    return expand_common(level, final, hidden, lm_head_w, logits, B, H, V, top_k, depth, n_out,
                         tree_state, state_bytes, partials, partials_bytes, d2t, out_tokens,
                         out_parent, out_draft_row, frontier_tokens, dev_status, stream);
}

extern "C" eagle_status eagle2_tree_candidates(const void* tree_state, size_t state_bytes, int B,
                                               int top_k, int depth, float* value, float* conf,
                                               int32_t* token, int32_t* parent,
                                               int32_t* cand_depth, int32_t* draft_row,
                                               eagle_stream_t stream) {
    if (B < 0 || top_k < 1 || depth < 1) return EAGLE_ERR_INVALID_ARG;
    if (top_k > kKMax || depth > kDepthMax) return EAGLE_ERR_SHAPE;
    if (B == 0) return EAGLE_OK;                        // nothing read or written
    if (!tree_state) return EAGLE_ERR_INVALID_ARG;
    if (state_bytes < eagle2_tree_state_size(B, top_k, depth)) return EAGLE_ERR_CAPACITY;
    const int C = StateView::cand_count(top_k, depth);
    const dim3 grid((C + 255) / 256, B);
    tree_candidates_kernel<<<grid, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        tree_state, top_k, depth, value, conf, token, parent, cand_depth, draft_row);
    EAGLE_CHECK_LAUNCH();
    return EAGLE_OK;
}

// ---------------------------------------------------------------------------
// Allocation-free variant: the tree state lives in a file-scope device array.
// ---------------------------------------------------------------------------
namespace eagle {
namespace {

// Fixed home of the tree state for eagle2_expand_static_state.  It exists on
// every device that loads the library, from load until process exit.
constexpr size_t kStaticStateBytes = size_t(4) << 20;   // 4 MiB
static __device__ __align__(256) unsigned char g_static_tree_state[kStaticStateBytes];

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void* g_static_ptr[kMaxDevices] = {};

// Device address of g_static_tree_state on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device (with that device current) and cached.  The cache is not told about
// cudaDeviceReset: after a reset of a device the cached address is stale.
eagle_status static_state_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return EAGLE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return EAGLE_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (g_static_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_tree_state) != cudaSuccess || p == nullptr)
            return EAGLE_ERR_CUDA;
        g_static_ptr[dev] = p;
    }
    *out = g_static_ptr[dev];
    return EAGLE_OK;
}

}  // namespace
}  // namespace eagle

extern "C" eagle_status eagle2_expand_static_state(int level, int final, const void* hidden,
                                                   const void* lm_head_w, float* logits, int B,
                                                   int H, int V, int top_k, int depth, int n_out,
                                                   int32_t* out_tokens, int32_t* out_parent,
                                                   int32_t* out_draft_row,
                                                   int32_t* frontier_tokens, int32_t* dev_status,
                                                   eagle_stream_t stream) {
    // The same host checks as eagle2_expand, in the same order and before any device
    // call, so both entry points report the same status for the same bad argument.
    const eagle_status vs = expand_validate(level, final, hidden, lm_head_w, logits, B, H, V,
                                            top_k, depth, n_out, out_tokens, out_parent,
                                            out_draft_row);
    if (vs != EAGLE_OK) return vs;
    if (eagle2_tree_state_size(B, top_k, depth) > kStaticStateBytes) return EAGLE_ERR_CAPACITY;
    if (B == 0) return EAGLE_OK;                        // no device call for an empty batch
    void* state = nullptr;
    const eagle_status st = static_state_address(&state);
    if (st != EAGLE_OK) return st;
    // Level 1 writes every field of a sequence's state that later levels read,
    // so the array needs no clearing between trees.
    return eagle2_expand(level, final, hidden, lm_head_w, logits, B, H, V, top_k, depth, n_out,
                         state, kStaticStateBytes, nullptr, 0, out_tokens, out_parent,
                         out_draft_row, frontier_tokens, dev_status, stream);
}

// ---------------------------------------------------------------------------
// Static draft trees (EAGLE-1 / Medusa style): the tree is fixed by a list of
// rank paths ("choices"); node (r_1..r_d) takes the r_d-th best token of its
// parent's draft row.  Guide "EAGLE-2：草稿树的 Expansion 与 Reranking" (the static
// trees that EAGLE-2 replaces add a fixed number of candidates per step).
// ---------------------------------------------------------------------------
namespace eagle {
namespace {

// One CTA per (internal node v at depth level-1, sequence b): the top K = (largest
// child rank + 1) of v's draft row, then each child c of v gets token top[rank[c]].
__global__ void __launch_bounds__(kTopkThreads)
static_tree_level_kernel(int level, const float* __restrict__ logits, const int32_t* parent,
                         const int32_t* rank, const int32_t* depth, const int32_t* draft_row,
                         int n, int R, int V, int32_t* tokens, int32_t* dev_status) {
    __shared__ float s_v[kTopkWarps * kKMax];
    __shared__ int s_i[kTopkWarps * kKMax];
    __shared__ int s_tok[kKMax];
    __shared__ int s_K, s_bad;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int v = blockIdx.x, b = blockIdx.y;
    if (depth[v] != level - 1 || draft_row[v] < 0) return;      // block-uniform
    if (tid == 0) {
        int K = 0;
        for (int c = v + 1; c < n; ++c)
            if (parent[c] == v) K = max(K, rank[c] + 1);
        s_K = K;
        s_bad = 0;
    }
    __syncthreads();
    const int K = s_K;
    if (K == 0) return;
    const int row = draft_row[v];
    if (row >= R || K > kKMax || K > V) {
        if (tid == 0) flag_error(dev_status, EAGLE_DEV_BAD_TREE);
        return;
    }
    const float* x = logits + ((int64_t)b * R + row) * (int64_t)V;
    float lv = -INFINITY, tv = -INFINITY;
    int li = 0x7fffffff, ti = 0x7fffffff, bad = 0;
    for (int base = 0; base < V; base += kTopkThreads) {            // block-uniform trips
        const int t = base + tid;
        const bool ok = t < V;
        const float l = ok ? x[t] : -INFINITY;
        bad |= ok && (l != l || l == INFINITY);
        unsigned ball = __ballot_sync(0xffffffffu, ok && topk_better(l, t, tv, ti));
        while (ball) {
            const int src = __ffs(ball) - 1;
            ball &= ball - 1;
            const float cv = __shfl_sync(0xffffffffu, l, src);
            const int ci = __shfl_sync(0xffffffffu, t, src);
            if (topk_better(cv, ci, tv, ti)) {
                warp_list_insert(lv, li, cv, ci);
                tv = __shfl_sync(0xffffffffu, lv, K - 1);
                ti = __shfl_sync(0xffffffffu, li, K - 1);
            }
        }
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(&s_bad, 1);
    if (lane < K) { s_v[warp * kKMax + lane] = lv; s_i[warp * kKMax + lane] = li; }
    __syncthreads();
    if (tid < kTopkWarps * K) {
        const int w = tid / K, j = tid % K;
        const float val = s_v[w * kKMax + j];
        const int id = s_i[w * kKMax + j];
        int r = 0;
        for (int w2 = 0; w2 < kTopkWarps; ++w2)
            for (int j2 = 0; j2 < K; ++j2)
                r += topk_better(s_v[w2 * kKMax + j2], s_i[w2 * kKMax + j2], val, id);
        if (r < K) s_tok[r] = id;
    }
    __syncthreads();
    if (s_bad) {
        if (tid == 0) flag_error(dev_status, EAGLE_DEV_NONFINITE);
        return;
    }
    for (int c = v + 1 + tid; c < n; c += kTopkThreads)
        if (parent[c] == v) tokens[(int64_t)b * n + c] = s_tok[rank[c]];
}

}  // namespace
}  // namespace eagle

extern "C" eagle_status eagle_static_tree(const int32_t* ranks, const int32_t* lens, int n_choices,
                                          int max_len, int n_max, int32_t* parent, int32_t* rank,
                                          int32_t* depth, int32_t* draft_row, int32_t* n_nodes) {
    if (!ranks || !lens || !parent || !rank || !depth || !draft_row || !n_nodes || n_choices < 0 ||
        max_len < 1)
        return EAGLE_ERR_INVALID_ARG;
    const int n = n_choices + 1;
    if (n > n_max || n > kMaxNodes) return EAGLE_ERR_CAPACITY;
    std::vector<std::vector<int>> paths((size_t)n_choices);
    for (int c = 0; c < n_choices; ++c) {
        const int len = lens[c];
        if (len < 1 || len > max_len) return EAGLE_ERR_SHAPE;
        for (int j = 0; j < len; ++j) {
            const int r = ranks[(size_t)c * max_len + j];
            if (r < 0 || r >= kKMax) return EAGLE_ERR_SHAPE;
            paths[c].push_back(r);
        }
    }
    // node order: (length, lexicographic); the root is node 0
    std::sort(paths.begin(), paths.end(), [](const std::vector<int>& a, const std::vector<int>& b) {
        return a.size() != b.size() ? a.size() < b.size() : a < b;
    });
    std::map<std::vector<int>, int> index;
    index[std::vector<int>()] = 0;
    for (int c = 0; c < n_choices; ++c) {
        if (!index.emplace(paths[c], c + 1).second) return EAGLE_ERR_SHAPE;   // duplicate
    }
    std::vector<int> par(n, -1), rk(n, -1), dep(n, 0);
    for (int c = 0; c < n_choices; ++c) {
        const std::vector<int> pre(paths[c].begin(), paths[c].end() - 1);
        const auto it = index.find(pre);
        if (it == index.end()) return EAGLE_ERR_SHAPE;                         // parent missing
        par[c + 1] = it->second;
        rk[c + 1] = paths[c].back();
        dep[c + 1] = (int)paths[c].size();
    }
    std::vector<char> kids(n, 0);
    for (int i = 1; i < n; ++i) kids[par[i]] = 1;
    int rows = 0;
    for (int i = 0; i < n; ++i) {
        parent[i] = par[i];
        rank[i] = rk[i];
        depth[i] = dep[i];
        draft_row[i] = kids[i] ? rows++ : -1;
    }
    *n_nodes = n;
    return EAGLE_OK;
}

extern "C" eagle_status eagle_static_tree_level(int level, const float* logits, const int32_t* parent,
                                                const int32_t* rank, const int32_t* depth,
                                                const int32_t* draft_row, int n, int B, int R, int V,
                                                int32_t* tokens, int32_t* dev_status,
                                                eagle_stream_t stream) {
    if (level < 1 || B < 0 || R < 1 || V < 1 || n < 1) return EAGLE_ERR_INVALID_ARG;
    if (n > kMaxNodes) return EAGLE_ERR_SHAPE;
    if (B == 0) return EAGLE_OK;                        // nothing read or written
    if (!logits || !parent || !rank || !depth || !draft_row || !tokens) return EAGLE_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    static_tree_level_kernel<<<dim3((unsigned)n, (unsigned)B), kTopkThreads, 0, s>>>(
        level, logits, parent, rank, depth, draft_row, n, R, V, tokens, dev_status);
    EAGLE_CHECK_LAUNCH();
    return EAGLE_OK;
}
