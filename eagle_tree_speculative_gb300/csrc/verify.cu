// Verify-and-accept walk over a draft tree, and per-row softmax statistics.
//
// Method (Lesson "推测解码与 EAGLE-3", sections "不变量：Leviathan 拒绝采样" and
// "动手构建" steps 1-3; Guide "EAGLE-1/2/3 拆解", sections "无损性的来源" and
// "EAGLE-2" on tree acceptance): accept draft x with probability
// min(1, q(x)/p(x)); on rejection resample from norm(max(0, q - p)); walk
// root-to-leaf to the longest accepted path; emit a bonus token when the walk
// ends on a node none of whose children was accepted.
//
// GB300 design: one thread-block cluster walks one sequence.  The walk itself
// is serial, so every CTA of the cluster runs the same control flow and the
// vocabulary-wide passes (row statistics, residual sums, the sampling race,
// the greedy argmax) are split across the CTAs by vocabulary slice; partial
// results meet in distributed shared memory behind one cluster barrier per
// pass.  Row statistics are computed lazily, only for the rows the walk
// visits (the accepted path plus the stopping node), instead of for all
// B x n rows: the walk's HBM traffic is (accept_len + 1) target rows and as
// many draft rows per sequence; residual re-passes hit L2.
#include <cstdlib>

#include "common.cuh"

namespace eagle {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

// Top-k / top-p filter of one row at temperature T > 0 (reading of eagenerate's top_k and
// top_p arguments: rank the row's tokens by probability, lower token first on ties; top-k
// keeps the first k; top-p keeps the shortest prefix of what top-k kept whose probability,
// renormalised over that set, reaches top_p).  The kept set is {t : key(l_t) > key, or
// key(l_t) == key and t <= idx}, key() the order-preserving integer image of a float; S is
// sum 2^((l - lmax) c) over the kept set.  bad != 0: the row holds NaN or +inf.
struct FilterParam {
    float lmax, S;
    uint32_t key;
    int32_t idx;
    int32_t bad, pad0, pad1, pad2;
};

__device__ __forceinline__ uint32_t order_key(float l) {
    const uint32_t u = __float_as_uint(l);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// A filter written by another CTA of the cluster: read at L2, past this SM's L1.
__device__ __forceinline__ FilterParam load_filter(const FilterParam* f) {
    static_assert(sizeof(FilterParam) == 32, "two 16-byte words");
    const uint4 w0 = __ldcg(reinterpret_cast<const uint4*>(f));
    const uint4 w1 = __ldcg(reinterpret_cast<const uint4*>(f) + 1);
    FilterParam r;
    memcpy(&r, &w0, 16);
    memcpy(reinterpret_cast<char*>(&r) + 16, &w1, 16);
    return r;
}

__device__ __forceinline__ bool filter_keeps(const FilterParam& f, int t, float l) {
    const uint32_t k = order_key(l);
    return k > f.key || (k == f.key && t <= f.idx);
}

// Vocabulary shards of a vocab-parallel walk: rank r holds ids [begin[r], begin[r+1])
// of every target and draft row in its own buffers, f32 [B, n, Vr] and [B, R, Vr].
constexpr int kMaxShards = 8;
struct ShardTable {
    const float* tgt[kMaxShards];
    const float* drf[kMaxShards];
    int begin[kMaxShards + 1];
};

struct VerifyArgs {
    const float* target;
    const float* draft;
    const int32_t* draft_row;
    const int32_t* tokens;
    const int32_t* parent;
    int B, n, V, R, D;
    float T;
    float c;          // log2(e) / T
    uint64_t seed;
    int32_t* accept_len;
    int32_t* path;
    int32_t* emit;
    float* row_stats;
    int32_t* dev_status;
    int Vd;                // draft-row length (= V without a draft vocabulary)
    const int32_t* t2d;    // target id -> draft id or -1 (draft vocabulary only)
    FilterParam* fq;       // per target row [B * n], filtered walk only (written on visit)
    FilterParam* fp;       // per draft row [B * R], filtered walk only (written on visit)
    int top_k;             // filtered walk only
    float top_p;
    bool target_in_device; // target rows in device memory (not pinned host memory)
    int S = 0;             // vocab-parallel walk: number of shards (0: whole rows)
    bool shard_vec4 = false;
    ShardTable sh{};
};

// Softmax statistics of a row at temperature T, kept over the raw logits:
// lmax = max l, S = sum 2^((l - lmax) c) with c = log2(e) / T, so that
// softmax(l / T)(x) = 2^((l_x - lmax) c) / S.  (max z = lmax / T, Z = S.)
struct RowStat {
    float lmax, S;
};

__device__ __forceinline__ RowStat rs_combine(RowStat a, RowStat b, float c) {
    if (b.lmax == -INFINITY) return a;
    if (a.lmax == -INFINITY) return b;
    const float M = fmaxf(a.lmax, b.lmax);
    return RowStat{M, a.S * exp2f((a.lmax - M) * c) + b.S * exp2f((b.lmax - M) * c)};
}

__device__ __forceinline__ void rs_push4(RowStat& a, float4 l, float c) {
    const float mx = fmaxf(fmaxf(l.x, l.y), fmaxf(l.z, l.w));
    if (mx == -INFINITY) return;
    if (mx > a.lmax) {
        a.S = (a.lmax == -INFINITY) ? 0.f : a.S * exp2f((a.lmax - mx) * c);
        a.lmax = mx;
    }
    a.S += exp2f((l.x - a.lmax) * c) + exp2f((l.y - a.lmax) * c) + exp2f((l.z - a.lmax) * c) +
           exp2f((l.w - a.lmax) * c);
}

__device__ __forceinline__ void rs_push1(RowStat& a, float l, float c) {
    if (l == -INFINITY) return;
    if (l > a.lmax) {
        a.S = (a.lmax == -INFINITY) ? 0.f : a.S * exp2f((a.lmax - l) * c);
        a.lmax = l;
    }
    a.S += exp2f((l - a.lmax) * c);
}

__device__ __forceinline__ int bad4(float4 l) {
    return isnan(l.x) | isnan(l.y) | isnan(l.z) | isnan(l.w) | (l.x == INFINITY) |
           (l.y == INFINITY) | (l.z == INFINITY) | (l.w == INFINITY);
}

// Probability of a token from its logit: 2^((l - lmax) c) / S, the division
// taken as a product with the precomputed reciprocal inv = 1 / S.
__device__ __forceinline__ float prob_of(float l, float lmax, float inv, float c) {
    return exp2f((l - lmax) * c) * inv;
}

// Weight of token t in q_cur after the rejections so far at the current node.
// The rejection rule r_0 = q, r_j = max(0, r_{j-1} - p) / S_j (kept unchanged when
// S_j == 0) unrolls to r_j(t) = max(0, q(t) - c_j p(t)) / D_j: by induction, with
// c_0 = 0 and D_0 = 1, max(0, r_j - p) = max(0, q - (c_j + D_j) p) / D_j, so a
// rejection pass sums s = sum_t max(0, q - (c_j + D_j) p) and sets
// c_{j+1} = c_j + D_j, D_{j+1} = s (S_{j+1} = s / D_j).  Every pass and the
// final race then cost O(1) per token, however many siblings were rejected.
struct Residual {
    float rc, rD, rinv;   // c_j, D_j, 1 / D_j
};

__device__ __forceinline__ float resid_weight(float lq, float lp, RowStat Q, float iq, RowStat P,
                                              float ip, float c, const Residual& rs) {
    const float q = prob_of(lq, Q.lmax, iq, c);
    if (rs.rc == 0.f) return q;
    return fmaxf(0.f, q - rs.rc * prob_of(lp, P.lmax, ip, c)) * rs.rinv;
}

// The unnormalised weight of the next residual, max(0, q - (c_j + D_j) p).
__device__ __forceinline__ float next_resid(float lq, float lp, RowStat Q, float iq, RowStat P,
                                            float ip, float c, float cnext) {
    return fmaxf(0.f, prob_of(lq, Q.lmax, iq, c) - cnext * prob_of(lp, P.lmax, ip, c));
}

struct Slot {
    float f[4];
    int i;
    int bad;
};

template <int NT>
struct VerifySmem {
    int parent[kMaxNodes];
    int tok[kMaxNodes];
    int row[kMaxNodes];
    int nkids[kMaxNodes];
    int lastkid[kMaxNodes];
    int path[kMaxNodes + 1];
    int emit[kMaxNodes + 1];
    float red[NT / 32][4];
    int redi[NT / 32];
    int redbad[NT / 32];
    Slot x[2];                       // double-buffered exchange slot
    Slot bc;                         // the cluster-wide result, for this CTA's threads
    int err;
};

template <int CS, int NT>
struct Cluster {
    using Smem = VerifySmem<NT>;
    __device__ static void sync() {
        if constexpr (CS > 1) cg::this_cluster().sync();
        else __syncthreads();
    }
    __device__ static const Slot* slot(Smem& sm, int buf, int rank) {
        if constexpr (CS > 1) return cg::this_cluster().map_shared_rank(&sm.x[buf], rank);
        else return &sm.x[buf];
    }
    // Block reduction to thread 0's slot, one cluster barrier, then every thread
    // reads all CS slots in rank order (identical results in every thread).
    __device__ static void stats(Smem& sm, int& buf, RowStat& q, RowStat& p, int& bad, float c) {
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            q = rs_combine(q, RowStat{__shfl_xor_sync(~0u, q.lmax, o), __shfl_xor_sync(~0u, q.S, o)}, c);
            p = rs_combine(p, RowStat{__shfl_xor_sync(~0u, p.lmax, o), __shfl_xor_sync(~0u, p.S, o)}, c);
        }
        bad = __any_sync(~0u, bad);
        if (lane == 0) {
            sm.red[warp][0] = q.lmax; sm.red[warp][1] = q.S;
            sm.red[warp][2] = p.lmax; sm.red[warp][3] = p.S;
            sm.redbad[warp] = bad;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            RowStat a{-INFINITY, 0.f}, b{-INFINITY, 0.f};
            int bd = 0;
            for (int w = 0; w < NT / 32; ++w) {
                a = rs_combine(a, RowStat{sm.red[w][0], sm.red[w][1]}, c);
                b = rs_combine(b, RowStat{sm.red[w][2], sm.red[w][3]}, c);
                bd |= sm.redbad[w];
            }
            sm.x[buf].f[0] = a.lmax; sm.x[buf].f[1] = a.S;
            sm.x[buf].f[2] = b.lmax; sm.x[buf].f[3] = b.S;
            sm.x[buf].bad = bd;
        }
        sync();
        if (warp == 0) {
            // lane r fetches CTA r's slot; lane 0 combines them in rank order
            Slot mine{};
            if (lane < CS) mine = *slot(sm, buf, lane);
            RowStat a{-INFINITY, 0.f}, b{-INFINITY, 0.f};
            int bd = 0;
            for (int r = 0; r < CS; ++r) {       // every lane, same order
                const float f0 = __shfl_sync(0xffffffffu, mine.f[0], r);
                const float f1 = __shfl_sync(0xffffffffu, mine.f[1], r);
                const float f2 = __shfl_sync(0xffffffffu, mine.f[2], r);
                const float f3 = __shfl_sync(0xffffffffu, mine.f[3], r);
                a = rs_combine(a, RowStat{f0, f1}, c);
                b = rs_combine(b, RowStat{f2, f3}, c);
                bd |= __shfl_sync(0xffffffffu, mine.bad, r);
            }
            if (lane == 0) {
                sm.bc.f[0] = a.lmax; sm.bc.f[1] = a.S; sm.bc.f[2] = b.lmax; sm.bc.f[3] = b.S;
                sm.bc.bad = bd;
            }
        }
        __syncthreads();
        q = RowStat{sm.bc.f[0], sm.bc.f[1]};
        p = RowStat{sm.bc.f[2], sm.bc.f[3]};
        bad = sm.bc.bad;
        buf ^= 1;
    }
    __device__ static float sum(Smem& sm, int& buf, float v) {
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        v = warp_sum(v);
        if (lane == 0) sm.red[warp][0] = v;
        __syncthreads();
        if (threadIdx.x == 0) {
            float t = 0.f;
            for (int w = 0; w < NT / 32; ++w) t += sm.red[w][0];
            sm.x[buf].f[0] = t;
        }
        sync();
        if (warp == 0) {
            float mine = 0.f;
            if (lane < CS) mine = slot(sm, buf, lane)->f[0];
            float S = 0.f;
            for (int r = 0; r < CS; ++r) S += __shfl_sync(0xffffffffu, mine, r);   // rank order
            if (lane == 0) sm.bc.f[0] = S;
        }
        __syncthreads();
        const float S = sm.bc.f[0];
        buf ^= 1;
        return S;
    }
    // Two values held by CTA `owner` to every thread of every CTA (one cluster barrier).
    __device__ static void bcast2(Smem& sm, int& buf, int rank, int owner, float& f0, float& f1) {
        if (rank == owner && threadIdx.x == 0) {
            sm.x[buf].f[0] = f0;
            sm.x[buf].f[1] = f1;
        }
        sync();
        if (threadIdx.x == 0) {
            const Slot* o = slot(sm, buf, owner);
            sm.bc.f[0] = o->f[0];
            sm.bc.f[1] = o->f[1];
        }
        __syncthreads();
        f0 = sm.bc.f[0];
        f1 = sm.bc.f[1];
        buf ^= 1;
    }
    __device__ static KeyIdx argmax(Smem& sm, int& buf, KeyIdx v, int& bad) {
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        v = warp_argmax(v);
        bad = __any_sync(~0u, bad);
        if (lane == 0) { sm.red[warp][0] = v.k; sm.redi[warp] = v.i; sm.redbad[warp] = bad; }
        __syncthreads();
        if (threadIdx.x == 0) {
            KeyIdx b{-INFINITY, 0x7fffffff};
            int bd = 0;
            for (int w = 0; w < NT / 32; ++w) {
                KeyIdx c{sm.red[w][0], sm.redi[w]};
                if (ki_better(c, b)) b = c;
                bd |= sm.redbad[w];
            }
            sm.x[buf].f[0] = b.k;
            sm.x[buf].i = b.i;
            sm.x[buf].bad = bd;
        }
        sync();
        if (warp == 0) {
            Slot mine{};
            if (lane < CS) mine = *slot(sm, buf, lane);
            KeyIdx b{-INFINITY, 0x7fffffff};
            int bd = 0;
            for (int r = 0; r < CS; ++r) {       // every lane, same order
                const KeyIdx c{__shfl_sync(0xffffffffu, mine.f[0], r), __shfl_sync(0xffffffffu, mine.i, r)};
                if (ki_better(c, b)) b = c;
                bd |= __shfl_sync(0xffffffffu, mine.bad, r);
            }
            if (lane == 0) {
                sm.bc.f[0] = b.k;
                sm.bc.i = b.i;
                sm.bc.bad = bd;
            }
        }
        __syncthreads();
        const KeyIdx b{sm.bc.f[0], sm.bc.i};
        bad = sm.bc.bad;
        buf ^= 1;
        return b;
    }
};

__device__ __forceinline__ int cta_rank_in_cluster(int cs) {
    if (cs > 1) return (int)cg::this_cluster().block_rank();
    return 0;
}

// The draft logit of target token t.  Without a draft vocabulary the draft row is
// indexed by target id.  With one (the draft head ranks its own Vd ids, and draft id d
// stands for target id d + d2t[d]), t2d[t] is the draft id of t or -1, and a target
// id no draft id maps to has logit -inf: probability 0 under p.
template <bool D2T>
struct PRow {
    const float* p;         // draft row, or nullptr (no draft distribution needed)
    const int32_t* t2d;
    __device__ __forceinline__ float at(int d) const { return d >= 0 ? __ldg(p + d) : -INFINITY; }
    __device__ __forceinline__ float one(int t) const {
        if (!p) return 0.f;
        if constexpr (D2T) return at(__ldg(t2d + t));
        else return __ldg(p + t);
    }
    __device__ __forceinline__ float4 four(int t) const {
        if (!p) return make_float4(0.f, 0.f, 0.f, 0.f);
        if constexpr (D2T) {
            const int4 d = __ldg(reinterpret_cast<const int4*>(t2d + t));
            return make_float4(at(d.x), at(d.y), at(d.z), at(d.w));
        } else {
            return __ldg(reinterpret_cast<const float4*>(p + t));
        }
    }
};

// (max, sum) of row[lo, hi) at c = log2(e) / T into S, non-finite entries into bad;
// 4 float4 in flight per thread on the vector path.
template <int NT>
__device__ __forceinline__ void row_stats_slice(const float* row, int lo, int hi, bool vec4, float c,
                                                RowStat& S, int& bad) {
    if (vec4) {
        int t = lo + 4 * (int)threadIdx.x;
        for (; t + 12 * NT < hi; t += 16 * NT) {
            float4 r4[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) r4[u] = __ldg(reinterpret_cast<const float4*>(row + t + 4 * u * NT));
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                bad |= bad4(r4[u]);
                rs_push4(S, r4[u], c);
            }
        }
        for (; t < hi; t += 4 * NT) {
            const float4 r4 = __ldg(reinterpret_cast<const float4*>(row + t));
            bad |= bad4(r4);
            rs_push4(S, r4, c);
        }
    } else {
        for (int t = lo + (int)threadIdx.x; t < hi; t += NT) {
            const float l = row[t];
            bad |= isnan(l) | (l == INFINITY);
            rs_push1(S, l, c);
        }
    }
}

// E = -ln u' for the race uniform u' = (2 (w >> 9) + 1) 2^-24, as -log1p(-v) of the
// exact complement v = 1 - u' = (2^24 - 2 (w >> 9) - 1) 2^-24 (a float: fewer than
// 24 significant bits).  CUDA's log1pf is within 1 ulp over its whole range, so E
// carries a relative error of at most 2^-23 at every u', including u' near 1 where
// the race is usually won (E small).
__device__ __forceinline__ float race_exponential(uint32_t w) {
    const uint32_t comp = (1u << 24) - (2u * (w >> 9) + 1u);    // in [1, 2^24 - 1]
    return -log1pf(-(float)comp * 0x1p-24f);
}

// Exponential race over the weights w_t (any positive scale): argmax_t w_t / E_t,
// E_t = -ln u'_t.  `weight(lq, lp, t)` gives w_t from the two logits of token t; the
// generator is only run for 4-token blocks with some positive weight.
template <int NT, bool D2T, class Weight>
__device__ __forceinline__ KeyIdx race_slice(const float* qrow, PRow<D2T> prow, int lo, int hi,
                                             bool vec4, uint32_t b, uint32_t k0, uint32_t k1,
                                             Weight weight) {
    KeyIdx best{-1.f, 0x7fffffff};
    auto block4 = [&](float4 a4, float4 b4, int t) {
        const float ax[4] = {a4.x, a4.y, a4.z, a4.w}, bx[4] = {b4.x, b4.y, b4.z, b4.w};
        float rr[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) rr[e] = weight(ax[e], bx[e], t + e);
        if (rr[0] > 0.f || rr[1] > 0.f || rr[2] > 0.f || rr[3] > 0.f) {
            const uint4 w = philox4x32_10(make_uint4((uint32_t)t >> 2, 0u, b, kTagRace), k0, k1);
            const uint32_t wx[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (rr[e] > 0.f) {
                    const KeyIdx cand{rr[e] / race_exponential(wx[e]), t + e};
                    if (ki_better(cand, best)) best = cand;
                }
            }
        }
    };
    if (vec4) {
        int t = lo + 4 * (int)threadIdx.x;
        for (; t + 12 * NT < hi; t += 16 * NT) {          // 4 float4 of each row in flight
            float4 a4[4], b4[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                a4[u] = __ldg(reinterpret_cast<const float4*>(qrow + t + 4 * u * NT));
                b4[u] = prow.four(t + 4 * u * NT);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) block4(a4[u], b4[u], t + 4 * u * NT);
        }
        for (; t < hi; t += 4 * NT) {
            const float4 a4 = __ldg(reinterpret_cast<const float4*>(qrow + t));
            block4(a4, prow.four(t), t);
        }
    } else {
        for (int t = lo + (int)threadIdx.x; t < hi; t += NT) {
            const float rr = weight(qrow[t], prow.one(t), t);
            if (rr > 0.f) {
                const uint4 w = philox4x32_10(make_uint4((uint32_t)t >> 2, 0u, b, kTagRace), k0, k1);
                const uint32_t wx[4] = {w.x, w.y, w.z, w.w};
                const KeyIdx cand{rr / race_exponential(wx[t & 3]), t};
                if (ki_better(cand, best)) best = cand;
            }
        }
    }
    return best;
}

// ---------------------------------------------------------------------------
// Row filters for the filtered walk (top-k, then top-p over what top-k kept) on one CTA:
// the rows that the cluster-wide filter below leaves over.  The cut is
// usually found from a histogram over distance bins and an exact sort of the elements
// up to the cut; otherwise by a radix select over the rows' order keys (11-bit digits,
// most significant first).  Both keep per-bin counts and fixed-point masses
// (2^((l - max) c) scaled by 2^40, integer sums, so the decisions do not depend on the
// order of the atomics); ties at the cut go to the lower token.
// ---------------------------------------------------------------------------
constexpr int kFiltThreads = 256;
constexpr int kFiltBins = 2048;
constexpr int kFiltMaxV = 1 << 22;              // the index select uses two 11-bit digits

constexpr int kCand = 2048;                    // largest bin the sorted path takes
constexpr int kNearBins = 256;                 // the first histogram's bins: 4 log2 units

struct FiltSmem {
    unsigned int cnt[kFiltBins];
    unsigned long long mass[kFiltBins];
    unsigned long long sk[kCand];              // a bin's elements: (key << 32) | ~index, sorted
    int ncand;
    unsigned int wcnt[kFiltThreads / 32];
    unsigned long long wmass[kFiltThreads / 32];
    float redf[kFiltThreads / 32];
    int redi[kFiltThreads / 32];
    int found_bin;
    unsigned int found_cnt;
    unsigned long long found_mass;
    int imax;
    unsigned long long tot;                    // the row's total mass
    unsigned long long near_mass;              // count and mass of the bins below the limit
    unsigned int near_cnt;
};

__device__ __forceinline__ unsigned long long fixed_mass(float l, float lmax, float c) {
    return __float2ull_rz(exp2f((l - lmax) * c) * 0x1p40f);     // exact: <= 2^40, 24-bit mantissa
}

__device__ __forceinline__ float key_float(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Distance bin of a logit: (max - l) c in 1/64 of a log2 unit, the far tail (mass below
// 2^-31.98 of the maximum's) in the last bin.  Monotone: a larger logit never has a
// larger bin, and equal logits share one.
__device__ __forceinline__ int dist_bin(float l, float lmax, float c) {
    const float d = (lmax - l) * c;
    return d < (float)(kFiltBins - 1) / 64.f ? (int)(d * 64.f) : kFiltBins - 1;
}

// Calls f(t, x[t]) for every t in [0, V), spread over the CTA's kFiltThreads threads;
// eight float4 loads in flight per thread when x is 16-byte aligned and V a multiple
// of 4.  The order in which one thread sees its elements is fixed.
template <class F>
__device__ __forceinline__ void row_for_each(const float* __restrict__ x, int V, F&& f) {
    constexpr int DEPTH = 8;
    const int tid = threadIdx.x;
    if ((reinterpret_cast<uintptr_t>(x) & 15) == 0 && (V & 3) == 0) {
        const float4* x4 = reinterpret_cast<const float4*>(x);
        const int V4 = V >> 2;
        int i = tid;
        for (; i + (DEPTH - 1) * kFiltThreads < V4; i += DEPTH * kFiltThreads) {
            float4 w[DEPTH];
#pragma unroll
            for (int u = 0; u < DEPTH; ++u) w[u] = __ldg(x4 + i + u * kFiltThreads);
#pragma unroll
            for (int u = 0; u < DEPTH; ++u) {
                const int t = 4 * (i + u * kFiltThreads);
                f(t, w[u].x);
                f(t + 1, w[u].y);
                f(t + 2, w[u].z);
                f(t + 3, w[u].w);
            }
        }
        for (; i < V4; i += kFiltThreads) {
            const float4 w = __ldg(x4 + i);
            const int t = 4 * i;
            f(t, w.x);
            f(t + 1, w.y);
            f(t + 2, w.z);
            f(t + 3, w.w);
        }
    } else {
        for (int t = tid; t < V; t += kFiltThreads) f(t, x[t]);
    }
}

// Gather the elements of distance bin b (of bins 0 .. b when `upto`; at most kCand of
// them) and sort them by (key desc, index asc) into sm.sk[0 .. ncand).
__device__ void gather_sort(FiltSmem& sm, const float* x, int V, int b, float lmax, float c,
                            bool upto) {
    const int tid = threadIdx.x;
    if (tid == 0) sm.ncand = 0;
    __syncthreads();
    row_for_each(x, V, [&](int t, float l) {
        const int bin = dist_bin(l, lmax, c);
        if (upto ? bin <= b : bin == b) {
            const int pos = atomicAdd(&sm.ncand, 1);
            if (pos < kCand)
                sm.sk[pos] = ((unsigned long long)order_key(l) << 32) | (unsigned long long)(~(uint32_t)t);
        }
    });
    __syncthreads();
    const int n = min(sm.ncand, kCand);
    int n2 = 1;
    while (n2 < n) n2 <<= 1;
    for (int j = n + tid; j < n2; j += kFiltThreads) sm.sk[j] = 0ull;     // sorts last
    __syncthreads();
    for (int size = 2; size <= n2; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = tid; i < n2; i += kFiltThreads) {
                const int j = i ^ stride;
                if (j > i) {
                    const bool desc = (i & size) == 0;
                    const unsigned long long a = sm.sk[i], bb = sm.sk[j];
                    if (desc ? (a < bb) : (a > bb)) { sm.sk[i] = bb; sm.sk[j] = a; }
                }
            }
            __syncthreads();
        }
    }
}

// Adds m to a 64-bit shared-memory counter with 32-bit atomics: the low word first, then
// the high word plus the carry out of that addition (read from the low word's old value).
// Each addition's carry is its own, so once every thread is done the counter holds the
// exact sum, whatever the order.
__device__ __forceinline__ void add_u64_split(unsigned long long* ctr, unsigned long long m) {
    uint32_t* w = reinterpret_cast<uint32_t*>(ctr);      // little endian: w[0] low, w[1] high
    const uint32_t lo = (uint32_t)m, hi = (uint32_t)(m >> 32);
    const uint32_t old = atomicAdd(&w[0], lo);
    const uint32_t up = hi + (old + lo < old ? 1u : 0u);
    if (up) atomicAdd(&w[1], up);
}

// Add one element (count 1, mass m) to bin `bin` of the block histogram; bin < 0 adds
// nothing, and a zero mass skips the mass update.
__device__ __forceinline__ void hist_add(FiltSmem& sm, int bin, unsigned long long m) {
    if (bin < 0) return;
    atomicAdd(&sm.cnt[bin], 1u);
    if (m) add_u64_split(&sm.mass[bin], m);
}

__device__ __forceinline__ bool elig(uint32_t k, int t, uint32_t k0, int i0) {
    return k > k0 || (k == k0 && t <= i0);
}

// Scan the bins in rank order (descending when DESC) for the bin where the running metric
// (count, or mass when MASS) first reaches `remaining` (>= 1, <= the bins' total).  Writes
// found_bin and the count and mass of the bins before it.
template <bool MASS, bool DESC>
__device__ void scan_bins(FiltSmem& sm, int nb, unsigned long long remaining) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = nb / kFiltThreads;
    const int first = DESC ? nb - 1 - tid * per : tid * per;
    if (tid == 0) { sm.found_bin = 0; sm.found_cnt = 0u; sm.found_mass = 0ull; }
    unsigned int lc = 0;
    unsigned long long lm = 0;
    for (int j = 0; j < per; ++j) {
        const int bin = DESC ? first - j : first + j;
        lc += sm.cnt[bin];
        lm += sm.mass[bin];
    }
    unsigned int ic = lc;
    unsigned long long im = lm;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned int yc = __shfl_up_sync(0xffffffffu, ic, o);
        const unsigned long long ym = __shfl_up_sync(0xffffffffu, im, o);
        if (lane >= o) { ic += yc; im += ym; }
    }
    if (lane == 31) { sm.wcnt[warp] = ic; sm.wmass[warp] = im; }
    __syncthreads();
    unsigned int rc = ic - lc;
    unsigned long long rm = im - lm;
    for (int w = 0; w < warp; ++w) { rc += sm.wcnt[w]; rm += sm.wmass[w]; }
    const unsigned long long before = MASS ? rm : rc, mine = MASS ? lm : lc;
    if (before < remaining && before + mine >= remaining) {
        for (int j = 0; j < per; ++j) {
            const int bin = DESC ? first - j : first + j;
            const unsigned long long v = MASS ? sm.mass[bin] : sm.cnt[bin];
            if ((MASS ? rm : rc) + v >= remaining) {
                sm.found_bin = bin;
                sm.found_cnt = rc;
                sm.found_mass = rm;
                break;
            }
            rc += sm.cnt[bin];
            rm += sm.mass[bin];
        }
    }
    __syncthreads();
}

struct Cut {
    uint32_t key;
    int idx;
    unsigned long long mass_upto;     // mass of the elements up to and including the cut
};

// Among the row's elements eligible under (k0, i0), in rank order (key desc, index asc),
// the element at which the running count (MASS false) or fixed-point mass (MASS true)
// first reaches `target` (1 <= target <= the eligible total).
template <bool MASS>
__device__ Cut block_select(FiltSmem& sm, const float* x, int V, float lmax, float c,
                            unsigned long long target, uint32_t k0, int i0) {
    const int tid = threadIdx.x;
    uint32_t prefix = 0u, pmask = 0u;
    unsigned long long mb = 0ull, remaining = target, m_eq_total = 0ull;
    unsigned int n_eq = 0u;
    for (int pass = 0; pass < 3; ++pass) {
        const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
        const int nb = pass == 2 ? 1024 : 2048;
        for (int i = tid; i < nb; i += kFiltThreads) { sm.cnt[i] = 0u; sm.mass[i] = 0ull; }
        __syncthreads();
        for (int base = 0; base < V; base += kFiltThreads) {          // warp-uniform trips
            const int t = base + tid;
            const float l = t < V ? x[t] : -INFINITY;
            const uint32_t k = order_key(l);
            const bool in = t < V && (k & pmask) == prefix && elig(k, t, k0, i0);
            hist_add(sm, in ? (int)((k >> shift) & (uint32_t)(nb - 1)) : -1,
                     in ? fixed_mass(l, lmax, c) : 0ull);
        }
        __syncthreads();
        scan_bins<MASS, true>(sm, nb, remaining);
        const int bin = sm.found_bin;
        remaining -= MASS ? sm.found_mass : (unsigned long long)sm.found_cnt;
        mb += sm.found_mass;
        if (pass == 2) { n_eq = sm.cnt[bin]; m_eq_total = sm.mass[bin]; }
        prefix |= (uint32_t)bin << shift;
        pmask |= (uint32_t)(nb - 1) << shift;
        __syncthreads();
    }
    // the elements whose key is the cut's: they share one value, so one mass each; the
    // cut keeps the first `need` of them by index
    if (n_eq == 0u) n_eq = 1u;                         // (cannot happen: the cut's bin is not empty)
    const unsigned long long m_eq = m_eq_total / n_eq;
    unsigned long long need = MASS ? (remaining + m_eq - 1ull) / m_eq : remaining;
    if (need > n_eq) need = n_eq;
    int idx;
    if (need == n_eq) {
        if (tid == 0) sm.imax = -1;
        __syncthreads();
        for (int t = tid; t < V; t += kFiltThreads)
            if (order_key(x[t]) == prefix && elig(prefix, t, k0, i0)) atomicMax(&sm.imax, t);
        __syncthreads();
        idx = sm.imax;
        __syncthreads();
    } else {
        uint32_t iprefix = 0u, imask = 0u;
        unsigned long long rem = need;
        for (int pass = 0; pass < 2; ++pass) {
            const int shift = pass == 0 ? 11 : 0;
            for (int i = tid; i < kFiltBins; i += kFiltThreads) { sm.cnt[i] = 0u; sm.mass[i] = 0ull; }
            __syncthreads();
            for (int base = 0; base < V; base += kFiltThreads) {      // warp-uniform trips
                const int t = base + tid;
                bool in = t < V && ((uint32_t)t & imask) == iprefix;
                if (in) {
                    const uint32_t k = order_key(x[t]);
                    in = k == prefix && elig(k, t, k0, i0);
                }
                hist_add(sm, in ? (int)(((uint32_t)t >> shift) & (kFiltBins - 1)) : -1, 0ull);
            }
            __syncthreads();
            scan_bins<false, false>(sm, kFiltBins, rem);
            rem -= sm.found_cnt;
            iprefix |= (uint32_t)sm.found_bin << shift;
            imask |= (uint32_t)(kFiltBins - 1) << shift;
            __syncthreads();
        }
        idx = (int)iprefix;
    }
    return Cut{prefix, idx, mb + need * m_eq};
}

// The filter of one row of logits x[0 .. V-1] at c = log2(e) / T, computed by the
// whole CTA (kFiltThreads threads, all of which must call it): the maximum, the cut
// (order key, index) of the kept set and the kept set's sum of exp2((l - max) c).
// Thread 0 writes *out.
__device__ void filter_row(FiltSmem& sm, const float* __restrict__ x, int V, float c, int top_k,
                           float top_p, FilterParam* out, bool l2_prefetch) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // the passes below read the row four or five times: bring it into L2 in one request
    // per 64 KB while the first pass starts (rows in device memory only)
    if (l2_prefetch && (reinterpret_cast<uintptr_t>(x) & 15) == 0) {
        const int64_t bytes = ((int64_t)V * 4) & ~int64_t(15);
        for (int64_t o = (int64_t)tid * 65536; o < bytes; o += (int64_t)kFiltThreads * 65536) {
            const uint32_t n = (uint32_t)(bytes - o < 65536 ? bytes - o : 65536);
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(
                             reinterpret_cast<const char*>(x) + o), "r"(n)
                         : "memory");
        }
    }
    float mx = -INFINITY;
    int bad = 0;
    row_for_each(x, V, [&](int, float l) {
        bad |= (l != l) | (l == INFINITY);
        mx = fmaxf(mx, l);
    });
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) { sm.redf[warp] = mx; sm.redi[warp] = bad; }
    __syncthreads();
    float lmax = -INFINITY;
    int bd = 0;
    for (int w = 0; w < kFiltThreads / 32; ++w) { lmax = fmaxf(lmax, sm.redf[w]); bd |= sm.redi[w]; }
    __syncthreads();
    if (bd || lmax == -INFINITY) {
        if (tid == 0) *out = FilterParam{lmax, 0.f, 0u, 0, 1, 0, 0, 0};
        return;
    }
    uint32_t key = 0u;                 // keep everything
    int idx = 0x7fffffff;
    const bool do_k = top_k > 0 && top_k < V;
    const bool do_p = top_p > 0.f && top_p < 1.f;
    auto fm = [&](unsigned long long e) { return fixed_mass(key_float((uint32_t)(e >> 32)), lmax, c); };
    if (do_k || do_p) {
        // Fast path: a histogram over distance bins (fine where the probability mass is),
        // then an exact sort of the elements the cut falls among.  The radix select takes
        // over when those are in the far tail or more than kCand of them.
        // The histogram first covers only the bins within 4 log2 units of the maximum; it
        // is rebuilt over every bin unless those already hold the cut (top_k elements, or
        // without top-k the top-p mass), so the bins it feeds the scans are always exact.
        unsigned long long total_all = 0ull;      // exact mass of the row (top-p alone)
        for (int limit = kNearBins;; limit = kFiltBins) {
            for (int i = tid; i < kFiltBins; i += kFiltThreads) { sm.cnt[i] = 0u; sm.mass[i] = 0ull; }
            if (tid == 0) { sm.tot = 0ull; sm.near_cnt = 0u; sm.near_mass = 0ull; }
            __syncthreads();
            unsigned long long tm = 0ull;
            const bool need_total = do_p && !do_k;
            if (need_total) {
                row_for_each(x, V, [&](int, float l) {
                    const int bin = dist_bin(l, lmax, c);
                    const unsigned long long m = fixed_mass(l, lmax, c);
                    tm += m;
                    if (bin < limit) hist_add(sm, bin, m);
                });
            } else {
                row_for_each(x, V, [&](int, float l) {
                    const int bin = dist_bin(l, lmax, c);
                    if (bin < limit) hist_add(sm, bin, do_p ? fixed_mass(l, lmax, c) : 0ull);
                });
            }
            if (need_total) add_u64_split(&sm.tot, tm);
            __syncthreads();
            total_all = sm.tot;
            if (limit == kFiltBins) break;
            unsigned int nc = 0u;
            unsigned long long nm = 0ull;
            for (int i = tid; i < limit; i += kFiltThreads) { nc += sm.cnt[i]; nm += sm.mass[i]; }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                nc += __shfl_xor_sync(0xffffffffu, nc, o);
                nm += __shfl_xor_sync(0xffffffffu, nm, o);
            }
            if (lane == 0) {
                atomicAdd(&sm.near_cnt, nc);
                add_u64_split(&sm.near_mass, nm);
            }
            __syncthreads();
            bool enough;
            if (do_k) {
                enough = sm.near_cnt >= (unsigned int)top_k;
            } else {
                unsigned long long tgt = (unsigned long long)ceil((double)top_p * (double)total_all);
                tgt = tgt < 1ull ? 1ull : (tgt > total_all ? total_all : tgt);
                enough = sm.near_mass >= tgt;
            }
            __syncthreads();
            if (enough) break;
        }
        bool hist = true;                 // the histogram is still intact
        int bk = -1, nk = 0;              // top-k cut: its bin, and how many sorted elements stay
        unsigned long long mk = 0ull;     // mass of what precedes sm.sk[0]
        unsigned long long total = 0ull;  // mass of what top-k keeps
        if (do_k) {
            scan_bins<false, false>(sm, kFiltBins, (unsigned long long)top_k);
            const int bin = sm.found_bin;
            const unsigned int cb = sm.found_cnt;
            mk = sm.found_mass;
            if (bin < kFiltBins - 1 && cb + sm.cnt[bin] <= (unsigned int)kCand) {
                // every element up to the cut bin fits: sort them all; the first top_k are
                // the top-k set, and the top-p cut (if any) is among them
                gather_sort(sm, x, V, bin, lmax, c, true);
                nk = top_k;
                mk = 0ull;
                const unsigned long long e = sm.sk[nk - 1];
                key = (uint32_t)(e >> 32);
                idx = (int)(~(uint32_t)e);
                for (int j = 0; j < nk; ++j) total += fm(sm.sk[j]);
                bk = bin;
            } else if (bin < kFiltBins - 1 && sm.cnt[bin] <= (unsigned int)kCand) {
                gather_sort(sm, x, V, bin, lmax, c, false);
                nk = top_k - (int)cb;
                const unsigned long long e = sm.sk[nk - 1];
                key = (uint32_t)(e >> 32);
                idx = (int)(~(uint32_t)e);
                total = mk;
                for (int j = 0; j < nk; ++j) total += fm(sm.sk[j]);
                bk = bin;
            } else {
                const Cut k = block_select<false>(sm, x, V, lmax, c, (unsigned long long)top_k, 0u,
                                                  0x7fffffff);
                key = k.key;
                idx = k.idx;
                total = k.mass_upto;
                hist = false;
            }
        }
        if (do_p) {
            if (!do_k) total = total_all;
            unsigned long long tgt = (unsigned long long)ceil((double)top_p * (double)total);
            tgt = tgt < 1ull ? 1ull : (tgt > total ? total : tgt);
            bool done = false;
            if (hist && bk >= 0 && tgt > mk) {
                // the cut lies among the sorted elements that top-k keeps
                unsigned long long acc = mk;
                int j = 0;
                for (; j < nk - 1; ++j) {
                    acc += fm(sm.sk[j]);
                    if (acc >= tgt) break;
                }
                key = (uint32_t)(sm.sk[j] >> 32);
                idx = (int)(~(uint32_t)sm.sk[j]);
                done = true;
            } else if (hist) {
                if (bk >= 0) {            // only the bins before top-k's cut bin remain eligible
                    __syncthreads();
                    for (int i = bk + tid; i < kFiltBins; i += kFiltThreads) { sm.cnt[i] = 0u; sm.mass[i] = 0ull; }
                    __syncthreads();
                }
                scan_bins<true, false>(sm, kFiltBins, tgt);
                const int bin = sm.found_bin;
                const unsigned long long mb = sm.found_mass;
                if (bin < kFiltBins - 1 && sm.cnt[bin] <= (unsigned int)kCand) {
                    gather_sort(sm, x, V, bin, lmax, c, false);
                    const int n = min(sm.ncand, kCand);
                    unsigned long long acc = mb;
                    int j = 0;
                    for (; j < n - 1; ++j) {
                        acc += fm(sm.sk[j]);
                        if (acc >= tgt) break;
                    }
                    key = (uint32_t)(sm.sk[j] >> 32);
                    idx = (int)(~(uint32_t)sm.sk[j]);
                    done = true;
                }
            }
            if (!done) {
                __syncthreads();
                const Cut pc = block_select<true>(sm, x, V, lmax, c, tgt, key, idx);
                idx = pc.key == key ? min(pc.idx, idx) : pc.idx;
                key = pc.key;
            }
        }
        __syncthreads();
    }
    // S over the kept set; per-thread sums combined in a fixed order
    float s = 0.f;
    row_for_each(x, V, [&](int t, float l) {
        if (elig(order_key(l), t, key, idx)) s += exp2f((l - lmax) * c);
    });
    s = warp_sum(s);
    if (lane == 0) sm.redf[warp] = s;
    __syncthreads();
    if (tid == 0) {
        float S = 0.f;
        for (int w = 0; w < kFiltThreads / 32; ++w) S += sm.redf[w];
        *out = FilterParam{lmax, S, key, idx, 0, 0, 0, 0};
    }
}

// ---------------------------------------------------------------------------
// The filters of the walk's current rows, q(v) and (when v has children) p(v),
// computed by the whole cluster: each CTA reads only its slice [lo, hi) of each row and
// the slices' partial results meet in distributed shared memory.
//   1. the maximum and the non-finite check: one value per CTA and row;
//   2. the counts and fixed-point masses of the distance bins within 4 log2 units of
//      the maximum, merged bin by bin (and, for top-p alone, the row's total mass);
//   3. the bin holding the top-k cut (without top-k, the top-p cut), found by every CTA
//      from the merged histogram;
//   4. the elements of that bin and the bins before it, gathered by each CTA from its
//      slice, copied by every CTA from all of them and sorted (key desc, index asc); the
//      cuts and the kept mass S follow from the sorted list.
// The bins, the integer masses and the order are filter_row's, so the kept sets are the
// same.  A row whose near bins do not reach the cut, or with more than kDCand elements
// up to the cut bin (kDLocal in one slice), is filtered by filter_row on one CTA.
// ---------------------------------------------------------------------------
constexpr int kDBins = kNearBins;
constexpr int kDLocal = 1024;                  // one CTA's candidates of one row
constexpr int kDCand = 1024;                   // all candidates of one row
static_assert(kDBins == kFiltThreads, "one bin per thread in the merge");

struct DFiltSmem {
    unsigned int hc[2][kDBins];                // this CTA's bin counts (read by the cluster)
    unsigned long long hm[2][kDBins];          // and fixed-point masses
    unsigned long long tot[2];                 // this CTA's total mass (top-p alone)
    int lcnt[2];                               // this CTA's candidates
    unsigned long long lk[2][kDLocal];
    unsigned int gc[2][kDBins];                // merged bins
    unsigned long long gm[2][kDBins];
    unsigned long long tot_all[2];
    unsigned long long sk[2][kDCand];          // all candidates, sorted
    int ncand[2];
    int cutbin[2];
    int fb[2];                                 // 1: the row goes to filter_row
    FilterParam res[2];                        // the fast path's results, for every thread
};

__device__ __forceinline__ void hist_add_d(DFiltSmem& ds, int r, int bin, unsigned long long m) {
    atomicAdd(&ds.hc[r][bin], 1u);
    if (m) add_u64_split(&ds.hm[r][bin], m);
}

// One element of row r in the near-bin histogram (and, for top-p alone, the row's mass).
// d = (max - l) c is dist_bin's distance; d * 64 is exact, so bin < kDBins exactly when
// d < kDBins / 64, and only those elements convert d to their bin.
__device__ __forceinline__ void near_hist(DFiltSmem& ds, int r, float l, float lm, float c,
                                          bool need_total, unsigned long long& tm) {
    const float d = (lm - l) * c;
    unsigned long long m = 0ull;
    if (need_total) {
        m = fixed_mass(l, lm, c);
        tm += m;
    }
    if (d < (float)kDBins / 64.f) hist_add_d(ds, r, (int)(d * 64.f), m);   // m = 0 with top-k
}

// Element t of row r into the CTA's candidate list when its bin is at most the cut bin:
// dist_bin(l) <= cbin exactly when d < (cbin + 1) / 64 = dlim.
__device__ __forceinline__ void gather_elem(DFiltSmem& ds, int r, int t, float l, float lm, float c,
                                            float dlim) {
    if ((lm - l) * c < dlim) {
        const int pos = atomicAdd(&ds.lcnt[r], 1);
        if (pos < kDLocal)
            ds.lk[r][pos] = ((unsigned long long)order_key(l) << 32) | (unsigned long long)(~(uint32_t)t);
    }
}

union FiltScratch {
    FiltSmem one;
    DFiltSmem dist;
};

// f0(t, x0[t]) and, when two, f1(t, x1[t]) for t in [lo, hi), NT threads; with vec4 (lo
// and hi multiples of 4, rows 16-byte aligned) four float4 of each row in flight per
// thread.
template <int NT, class F0, class F1>
__device__ __forceinline__ void slice_for_each2(const float* __restrict__ x0, const float* __restrict__ x1,
                                                bool two, int lo, int hi, bool vec4, F0&& f0, F1&& f1) {
    const int tid = threadIdx.x;
    if (vec4) {
        int t = lo + 4 * tid;
        for (; t + 12 * NT < hi; t += 16 * NT) {
            float4 w0[4], w1[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) w0[u] = __ldg(reinterpret_cast<const float4*>(x0 + t + 4 * u * NT));
            if (two) {
#pragma unroll
                for (int u = 0; u < 4; ++u) w1[u] = __ldg(reinterpret_cast<const float4*>(x1 + t + 4 * u * NT));
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int tu = t + 4 * u * NT;
                f0(tu, w0[u].x); f0(tu + 1, w0[u].y); f0(tu + 2, w0[u].z); f0(tu + 3, w0[u].w);
            }
            if (two) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int tu = t + 4 * u * NT;
                    f1(tu, w1[u].x); f1(tu + 1, w1[u].y); f1(tu + 2, w1[u].z); f1(tu + 3, w1[u].w);
                }
            }
        }
        for (; t < hi; t += 4 * NT) {
            const float4 w = __ldg(reinterpret_cast<const float4*>(x0 + t));
            f0(t, w.x); f0(t + 1, w.y); f0(t + 2, w.z); f0(t + 3, w.w);
            if (two) {
                const float4 v = __ldg(reinterpret_cast<const float4*>(x1 + t));
                f1(t, v.x); f1(t + 1, v.y); f1(t + 2, v.z); f1(t + 3, v.w);
            }
        }
    } else {
        for (int t = lo + tid; t < hi; t += NT) {
            f0(t, x0[t]);
            if (two) f1(t, x1[t]);
        }
    }
}

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Sorts s[0 .. n) descending into d[0 .. n) by rank (the keys are distinct): thread
// `first + i` places element i; `count` threads take part, n <= count.
__device__ __forceinline__ void rank_sort(const unsigned long long* s, unsigned long long* d, int n,
                                          int first, int count) {
    const int i = (int)threadIdx.x - first;
    if (i < 0 || i >= count || i >= n) return;
    const unsigned long long e = s[i];
    int r = 0;
    for (int j = 0; j < n; ++j) r += s[j] > e;
    d[r] = e;
}

// Bitonic sort of s[0 .. n) descending (pads to a power of two with zeros, which sort
// last); every thread of the CTA takes part.
template <int NT>
__device__ void sort_desc(unsigned long long* s, int n) {
    const int tid = threadIdx.x;
    int n2 = 1;
    while (n2 < n) n2 <<= 1;
    for (int j = n + tid; j < n2; j += NT) s[j] = 0ull;
    __syncthreads();
    for (int size = 2; size <= n2; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = tid; i < n2; i += NT) {
                const int j = i ^ stride;
                if (j > i) {
                    const bool desc = (i & size) == 0;
                    const unsigned long long x = s[i], y = s[j];
                    if (desc ? (x < y) : (x > y)) { s[i] = y; s[j] = x; }
                }
            }
            __syncthreads();
        }
    }
}

template <int CS, int NT>
__device__ void cluster_filters(VerifySmem<NT>& sm, FiltScratch& fsc, int& buf, int rank,
                                const float* const rows[2], int nr, int lo, int hi, bool vec4, int V,
                                float c, int top_k, float top_p, FilterParam* const slots[2],
                                const bool prefetch[2], FilterParam out[2]) {
    static_assert(NT == kFiltThreads, "the row filter takes the whole CTA");
    using C = Cluster<CS, NT>;
    DFiltSmem& ds = fsc.dist;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool do_k = top_k > 0 && top_k < V;
    const bool do_p = top_p > 0.f && top_p < 1.f;
    const bool need_total = do_p && !do_k;
    const bool two = nr > 1;
    const float* const x0 = rows[0];
    const float* const x1 = two ? rows[1] : rows[0];
    auto remote = [&](int rk) -> const DFiltSmem* {
        if constexpr (CS > 1) return cg::this_cluster().map_shared_rank(&ds, rk);
        else return &ds;
    };

    // ---- 1. maxima and the non-finite check (the slices first go to L2 in bulk) ----
    if (vec4 && tid < 2 && (tid == 0 || two) && prefetch[tid] && hi > lo) {
        const char* base = reinterpret_cast<const char*>(tid == 0 ? x0 : x1) + (int64_t)lo * 4;
        for (int64_t o = 0; o < (int64_t)(hi - lo) * 4; o += 65536) {
            const int64_t left = (int64_t)(hi - lo) * 4 - o;
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(base + o),
                         "r"((uint32_t)(left < 65536 ? left : 65536))
                         : "memory");
        }
    }
    float mx0 = -INFINITY, mx1 = -INFINITY;
    int bd = 0;
    slice_for_each2<NT>(
        x0, x1, two, lo, hi, vec4,
        [&](int, float l) { bd |= (l != l) | (l == INFINITY); mx0 = fmaxf(mx0, l); },
        [&](int, float l) { bd |= ((l != l) | (l == INFINITY)) << 1; mx1 = fmaxf(mx1, l); });
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
        bd |= __shfl_xor_sync(0xffffffffu, bd, o);
    }
    if (lane == 0) { sm.red[warp][0] = mx0; sm.red[warp][1] = mx1; sm.redbad[warp] = bd; }
    __syncthreads();
    if (tid == 0) {
        float a0 = -INFINITY, a1 = -INFINITY;
        int b0 = 0;
        for (int w = 0; w < NT / 32; ++w) {
            a0 = fmaxf(a0, sm.red[w][0]);
            a1 = fmaxf(a1, sm.red[w][1]);
            b0 |= sm.redbad[w];
        }
        sm.x[buf].f[0] = a0;
        sm.x[buf].f[1] = a1;
        sm.x[buf].bad = b0;
    }
    C::sync();
    if (warp == 0) {
        Slot mine{};
        if (lane < CS) mine = *C::slot(sm, buf, lane);
        float a0 = -INFINITY, a1 = -INFINITY;
        int b0 = 0;
        for (int r = 0; r < CS; ++r) {
            a0 = fmaxf(a0, __shfl_sync(0xffffffffu, mine.f[0], r));
            a1 = fmaxf(a1, __shfl_sync(0xffffffffu, mine.f[1], r));
            b0 |= __shfl_sync(0xffffffffu, mine.bad, r);
        }
        if (lane == 0) { sm.bc.f[0] = a0; sm.bc.f[1] = a1; sm.bc.bad = b0; }
    }
    __syncthreads();
    const float lmax0 = sm.bc.f[0], lmax1 = sm.bc.f[1];
    const int bad = sm.bc.bad;
    buf ^= 1;
    bool live[2];
    live[0] = !(bad & 1) && lmax0 != -INFINITY;
    live[1] = two && !(bad & 2) && lmax1 != -INFINITY;
    if (!live[0]) out[0] = FilterParam{lmax0, 0.f, 0u, 0, 1, 0, 0, 0};
    if (two && !live[1]) out[1] = FilterParam{lmax1, 0.f, 0u, 0, 1, 0, 0, 0};
    if (!live[0] && !live[1]) return;

    // ---- 2. near-bin histograms of the slice ----
    for (int i = tid; i < 2 * kDBins; i += NT) {
        (&ds.hc[0][0])[i] = 0u;
        (&ds.hm[0][0])[i] = 0ull;
    }
    if (tid < 2) { ds.tot[tid] = 0ull; ds.lcnt[tid] = 0; }
    __syncthreads();
    unsigned long long tm0 = 0ull, tm1 = 0ull;
    const bool l0 = live[0], l1 = live[1];
    {
        // the first row iterated is q unless only p is live
        const int ra = l0 ? 0 : 1;
        const float lma = l0 ? lmax0 : lmax1;
        slice_for_each2<NT>(
            l0 ? x0 : x1, x1, l0 && l1, lo, hi, vec4,
            [&](int, float l) { near_hist(ds, ra, l, lma, c, need_total, tm0); },
            [&](int, float l) { near_hist(ds, 1, l, lmax1, c, need_total, tm1); });
        if (!l0) { tm1 = tm0; tm0 = 0ull; }
    }
    if (need_total) {
        tm0 = warp_sum_u64(tm0);
        tm1 = warp_sum_u64(tm1);
        if (lane == 0) {
            if (tm0) add_u64_split(&ds.tot[0], tm0);
            if (tm1) add_u64_split(&ds.tot[1], tm1);
        }
    }
    __syncthreads();
    C::sync();
    for (int r = 0; r < 2; ++r) {
        if (!live[r]) continue;
        unsigned int cnt = 0u;
        unsigned long long m = 0ull;
        unsigned int hcs[CS];
#pragma unroll
        for (int rk = 0; rk < CS; ++rk) hcs[rk] = remote(rk)->hc[r][tid];
#pragma unroll
        for (int rk = 0; rk < CS; ++rk) cnt += hcs[rk];
        if (need_total) {
            unsigned long long hms[CS];
#pragma unroll
            for (int rk = 0; rk < CS; ++rk) hms[rk] = remote(rk)->hm[r][tid];
#pragma unroll
            for (int rk = 0; rk < CS; ++rk) m += hms[rk];
        }
        ds.gc[r][tid] = cnt;
        ds.gm[r][tid] = m;
        if (tid == 0 && need_total) {
            unsigned long long t = 0ull;
            for (int rk = 0; rk < CS; ++rk) t += remote(rk)->tot[r];
            ds.tot_all[r] = t;
        }
    }
    __syncthreads();

    // ---- 3. the cut bin: warp r scans row r's bins, eight per lane ----
    if (warp < 2) {
        const int r = warp;
        int fb = 1, cb = 0;
        if (live[r]) {
            unsigned int lc = 0u;
            unsigned long long lm = 0ull;
#pragma unroll
            for (int j = 0; j < kDBins / 32; ++j) {
                lc += ds.gc[r][lane * (kDBins / 32) + j];
                lm += ds.gm[r][lane * (kDBins / 32) + j];
            }
            unsigned int ic = lc;
            unsigned long long im = lm;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned int yc = __shfl_up_sync(0xffffffffu, ic, o);
                const unsigned long long ym = __shfl_up_sync(0xffffffffu, im, o);
                if (lane >= o) { ic += yc; im += ym; }
            }
            const unsigned int near_cnt = __shfl_sync(0xffffffffu, ic, 31);
            const unsigned long long near_mass = __shfl_sync(0xffffffffu, im, 31);
            unsigned long long target;
            bool enough;
            if (do_k) {
                target = (unsigned long long)top_k;
                enough = near_cnt >= (unsigned int)top_k;
            } else {
                const unsigned long long tot = ds.tot_all[r];
                target = (unsigned long long)ceil((double)top_p * (double)tot);
                target = target < 1ull ? 1ull : (target > tot ? tot : target);
                enough = near_mass >= target;
            }
            if (enough) {
                // the lane whose bins the running metric crosses the target in
                const unsigned long long before = do_k ? (unsigned long long)(ic - lc) : im - lm;
                const unsigned long long mine = do_k ? (unsigned long long)lc : lm;
                const bool here = before < target && before + mine >= target;
                const unsigned int who = __ballot_sync(0xffffffffu, here);
                const int src = who ? __ffs(who) - 1 : 0;
                int bin = 0;
                unsigned int cnt_before = 0u;
                if (lane == src) {
                    unsigned long long run = before;
                    unsigned int cbf = ic - lc;
                    for (int j = 0; j < kDBins / 32; ++j) {
                        const int bj = lane * (kDBins / 32) + j;
                        const unsigned long long v = do_k ? (unsigned long long)ds.gc[r][bj] : ds.gm[r][bj];
                        if (run + v >= target) { bin = bj; break; }
                        run += v;
                        cbf += ds.gc[r][bj];
                    }
                    cnt_before = cbf;
                }
                bin = __shfl_sync(0xffffffffu, bin, src);
                cnt_before = __shfl_sync(0xffffffffu, cnt_before, src);
                cb = bin;
                fb = (!who || cnt_before + ds.gc[r][bin] > (unsigned int)kDCand) ? 1 : 0;
            }
        }
        if (lane == 0) { ds.cutbin[r] = cb; ds.fb[r] = live[r] ? fb : 0; }
    }
    __syncthreads();
    bool go[2];
    for (int r = 0; r < 2; ++r) go[r] = live[r] && !ds.fb[r];

    // ---- 4. candidates: every element up to the cut bin, gathered from the slice ----
    // (a few per slice with top-k: one shared atomic each)
    {
        const bool r0 = go[0], r1 = go[1];
        const int ra = r0 ? 0 : 1;
        const float lma = r0 ? lmax0 : lmax1;
        const float dla = (float)(ds.cutbin[ra] + 1) / 64.f, dl1 = (float)(ds.cutbin[1] + 1) / 64.f;
        if (r0 || r1)
            slice_for_each2<NT>(
                r0 ? x0 : x1, x1, r0 && r1, lo, hi, vec4,
                [&](int t, float l) { gather_elem(ds, ra, t, l, lma, c, dla); },
                [&](int t, float l) { gather_elem(ds, 1, t, l, lmax1, c, dl1); });
        __syncthreads();
        C::sync();
    }
    // every CTA copies the elements up to the cut bin from all lists, in rank order
    if (tid < 2) ds.ncand[tid] = 0;
    __syncthreads();
    for (int r = 0; r < 2; ++r) {
        if (!go[r]) continue;
        int ks[CS];
        int total = 0;
        bool over = false;
#pragma unroll
        for (int rk = 0; rk < CS; ++rk) ks[rk] = remote(rk)->lcnt[r];
#pragma unroll
        for (int rk = 0; rk < CS; ++rk) {
            over = over || ks[rk] > kDLocal;
            total += ks[rk];
        }
        if (over || total > kDCand) {              // the same decision in every thread and CTA
            go[r] = false;
            if (tid == 0) ds.fb[r] = 1;
            continue;
        }
        int off = 0;
#pragma unroll
        for (int rk = 0; rk < CS; ++rk) {
            const DFiltSmem* o = remote(rk);
            for (int j = tid; j < ks[rk]; j += NT) ds.sk[r][off + j] = o->lk[r][j];
            off += ks[rk];
        }
        if (tid == 0) ds.ncand[r] = total;
    }
    __syncthreads();
    // short lists: rank sort, half the CTA per row, into the upper half of sk
    int soff[2] = {0, 0};
    const bool small0 = go[0] && ds.ncand[0] <= NT / 2, small1 = go[1] && ds.ncand[1] <= NT / 2;
    if (small0) rank_sort(ds.sk[0], ds.sk[0] + kDCand / 2, ds.ncand[0], 0, NT / 2);
    if (small1) rank_sort(ds.sk[1], ds.sk[1] + kDCand / 2, ds.ncand[1], NT / 2, NT / 2);
    if (small0) soff[0] = kDCand / 2;
    if (small1) soff[1] = kDCand / 2;
    __syncthreads();
    for (int r = 0; r < 2; ++r)
        if (go[r] && !(r == 0 ? small0 : small1)) sort_desc<NT>(ds.sk[r], min(ds.ncand[r], kDCand));

    // ---- cuts and kept mass: warp r for row r ----
    if (warp < 2 && go[warp]) {
        const int r = warp;
        const int nc = min(ds.ncand[r], kDCand);
        const float lm = r == 0 ? lmax0 : lmax1;
        const unsigned long long* s = ds.sk[r] + soff[r];
        auto fm = [&](int j) { return fixed_mass(key_float((uint32_t)(s[j] >> 32)), lm, c); };
        int cut = nc - 1;                          // without top-k everything gathered may stay
        unsigned long long total = ds.tot_all[r];
        if (do_k) {
            cut = top_k - 1;
            unsigned long long t = 0ull;
            for (int j = lane; j < top_k; j += 32) t += fm(j);
            total = warp_sum_u64(t);
        }
        if (do_p) {
            unsigned long long tgt = (unsigned long long)ceil((double)top_p * (double)total);
            tgt = tgt < 1ull ? 1ull : (tgt > total ? total : tgt);
            // the first j (at most cut) whose running mass reaches tgt
            unsigned long long run = 0ull;
            int found = cut;
            for (int base = 0; base < cut; base += 32) {
                const int j = base + lane;
                const unsigned long long m = j < cut ? fm(j) : 0ull;
                unsigned long long inc = m;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const unsigned long long y = __shfl_up_sync(0xffffffffu, inc, o);
                    if (lane >= o) inc += y;
                }
                const unsigned int hit = __ballot_sync(0xffffffffu, j < cut && run + inc >= tgt);
                if (hit) { found = base + __ffs(hit) - 1; break; }
                run += __shfl_sync(0xffffffffu, inc, 31);
            }
            cut = found;
        }
        float S = 0.f;
        for (int j = lane; j <= cut; j += 32) S += exp2f((key_float((uint32_t)(s[j] >> 32)) - lm) * c);
        S = warp_sum(S);
        const unsigned long long e = s[cut];
        if (lane == 0) ds.res[r] = FilterParam{lm, S, (uint32_t)(e >> 32), (int)(~(uint32_t)e), 0, 0, 0, 0};
    }
    __syncthreads();
    for (int r = 0; r < 2; ++r)
        if (go[r]) out[r] = ds.res[r];

    // ---- rows the fast path does not take: filter_row on one CTA each ----
    const bool fb0 = live[0] && ds.fb[0], fb1 = live[1] && ds.fb[1];
    if (fb0 || fb1) {
        C::sync();                                 // nobody reads this CTA's scratch any more
        for (int r = 0; r < 2; ++r) {
            if (!(r == 0 ? fb0 : fb1)) continue;
            if (rank == r % CS) {
                __syncthreads();
                filter_row(fsc.one, rows[r], V, c, top_k, top_p, slots[r], prefetch[r]);
            }
        }
        __threadfence();
        C::sync();
        if (fb0) out[0] = load_filter(slots[0]);
        if (fb1) out[1] = load_filter(slots[1]);
    }
}

// ---------------------------------------------------------------------------
template <int CS, int NT, bool D2T, bool FILT>
__global__ void __launch_bounds__(NT, FILT ? 2 : 4) verify_walk_kernel(VerifyArgs a) {
    using C = Cluster<CS, NT>;
    __shared__ VerifySmem<NT> sm;
    FiltScratch* fsc = nullptr;              // the filtered walk's row-filter scratch
    if constexpr (FILT) {
        static_assert(NT == kFiltThreads, "a row filter takes the whole CTA");
        __shared__ FiltScratch fs;
        fsc = &fs;
    }
    const int tid = threadIdx.x;
    const int rank = cta_rank_in_cluster(CS);
    const int b = blockIdx.x / CS;
    const int n = a.n, V = a.V;
    const float c = a.c;
    int64_t Vl = V;
    int64_t Vdl = D2T ? a.Vd : V;            // draft-row length

    // ---- load and validate the tree (identically in every CTA) ----
    if (tid < n) {
        sm.parent[tid] = a.parent[(int64_t)b * n + tid];
        sm.tok[tid] = a.tokens[(int64_t)b * n + tid];
        sm.row[tid] = a.draft_row ? a.draft_row[(int64_t)b * n + tid] : tid;
        sm.nkids[tid] = 0;
        sm.lastkid[tid] = -1;
    }
    if (tid == 0) sm.err = 0;
    __syncthreads();
    // one thread per node: parent in [0, i) (root: -1), token in range, depth
    // within D (walking up a strictly decreasing chain), children counts
    if (tid < n) {
        int err = 0;
        const int p = sm.parent[tid];
        if (tid == 0) {
            if (p != -1) err |= EAGLE_DEV_BAD_TREE;
        } else if (p < 0 || p >= tid) {
            err |= EAGLE_DEV_BAD_TREE;
        } else {
            if (sm.tok[tid] < 0 || sm.tok[tid] >= V) err |= EAGLE_DEV_BAD_TOKEN;
            int depth = 1, x = p;
            while (x > 0) {
                const int px = sm.parent[x];
                if (px < 0 || px >= x) break;       // flagged by node x itself
                x = px;
                ++depth;
            }
            if (depth > a.D) err |= EAGLE_DEV_DEPTH;
            atomicAdd(&sm.nkids[p], 1);
            atomicMax(&sm.lastkid[p], tid);
        }
        if (err) atomicOr(&sm.err, err);
    }
    __syncthreads();
    if (tid < n && !sm.err && a.T > 0.f && sm.nkids[tid] && (sm.row[tid] < 0 || sm.row[tid] >= a.R))
        atomicOr(&sm.err, EAGLE_DEV_BAD_TOKEN);
    __syncthreads();

    // ---- vocabulary slice of this CTA ----
    const int chunk = (((V + CS - 1) / CS) + 3) & ~3;
    int lo = min(V, rank * chunk), hi = min(V, lo + chunk);
    const float* tgt_b = a.target + (int64_t)b * n * Vl;
    const float* drf_b = a.draft ? a.draft + (int64_t)b * a.R * Vdl : nullptr;
    bool vec4 = ((V & 3) == 0) && ((reinterpret_cast<uintptr_t>(a.target) & 15) == 0) &&
                (a.draft == nullptr || (reinterpret_cast<uintptr_t>(a.draft) & 15) == 0) &&
                (!D2T || (((a.Vd & 3) == 0) && (reinterpret_cast<uintptr_t>(a.t2d) & 15) == 0));
    // Vocab-parallel walk: this CTA stands for rank `rank` and reads only its shard.  Its
    // slice is the shard's id range, its rows are the shard's rows (length hi - lo), and
    // the row bases are moved back by lo so that row[t] is the shard's element t - lo.
    const bool sharded = !D2T && !FILT && a.S > 0;
    int64_t shift = 0;
    if (sharded) {
        // CTAs past the last shard (the cluster is rounded up to a power of two) get an
        // empty slice; their row pointers stay non-null, as "has a draft row" is read from
        // them, and are never dereferenced (the owner of a token is always a real rank).
        const int r = rank < a.S ? rank : 0;
        lo = rank < a.S ? a.sh.begin[rank] : V;
        hi = rank < a.S ? a.sh.begin[rank + 1] : V;
        Vl = Vdl = hi - lo;
        shift = lo;
        tgt_b = a.sh.tgt[r] + (int64_t)b * n * Vl;
        drf_b = a.sh.drf[r] ? a.sh.drf[r] + (int64_t)b * a.R * Vdl : nullptr;
        vec4 = a.shard_vec4;
    }
    // the CTA's slice of the draft row for its statistics (the target slice otherwise)
    const int chunkd = D2T ? ((((a.Vd + CS - 1) / CS) + 3) & ~3) : chunk;
    const int plo = D2T ? min(a.Vd, rank * chunkd) : lo;
    const int phi = D2T ? min(a.Vd, plo + chunkd) : hi;
    const uint32_t k0 = (uint32_t)a.seed, k1 = (uint32_t)(a.seed >> 32);

    int buf = 0;
    int err = sm.err;
    int v = 0, acc_n = 0, y = -1;
    if (tid == 0) sm.path[0] = 0;

    while (!err) {
        const float* qrow = tgt_b + (int64_t)v * Vl - shift;
        const bool kids = sm.nkids[v] > 0;
        if (a.T > 0.f) {
            const float* prow = (kids && drf_b) ? drf_b + (int64_t)sm.row[v] * Vdl - shift : nullptr;
            const PRow<D2T> pr{prow, a.t2d};
            // filtered walk: this node's row filters; logits outside them read as -inf
            FilterParam fqv{}, fpv{};
            if constexpr (FILT) {
                // The rows are filtered when the walk reaches their node, by the whole
                // cluster (each CTA its vocabulary slice); every CTA gets both filters.
                const float* const rws[2] = {qrow, prow};
                FilterParam* const slots[2] = {a.fq + (int64_t)b * n + v,
                                               prow ? a.fp + (int64_t)b * a.R + sm.row[v] : nullptr};
                const bool pf[2] = {a.target_in_device, true};
                FilterParam outs[2];
                cluster_filters<CS, NT>(sm, *fsc, buf, rank, rws, prow ? 2 : 1, lo, hi, vec4, V, c,
                                        a.top_k, a.top_p, slots, pf, outs);
                fqv = outs[0];
                if (prow) fpv = outs[1];
            }
            auto mq = [&](int t, float l) -> float {
                if constexpr (FILT) return filter_keeps(fqv, t, l) ? l : -INFINITY;
                else return l;
            };
            auto mp = [&](int t, float l) -> float {
                if constexpr (FILT) return filter_keeps(fpv, t, l) ? l : -INFINITY;
                else return l;
            };
            // ---------- pass: statistics of q(v) and p(v) ----------
            RowStat Q{-INFINITY, 0.f}, P{-INFINITY, 0.f};
            int bad = 0;
            if constexpr (FILT) {
                // statistics of the filtered rows come with the filters
                Q = RowStat{fqv.lmax, fqv.S};
                bad = fqv.bad;
                if (prow) {
                    P = RowStat{fpv.lmax, fpv.S};
                    bad |= fpv.bad;
                }
            } else if constexpr (D2T) {
                // q over the target slice, p over the draft slice
                row_stats_slice<NT>(qrow, lo, hi, vec4, c, Q, bad);
                if (prow) row_stats_slice<NT>(prow, plo, phi, vec4, c, P, bad);
            } else if (vec4) {
                int t = lo + 4 * tid;
                // 4 float4 of each row in flight per thread
                for (; t + 12 * NT < hi; t += 16 * NT) {
                    float4 q4[4], p4[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        q4[u] = __ldg(reinterpret_cast<const float4*>(qrow + t + 4 * u * NT));
                    if (prow) {
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            p4[u] = __ldg(reinterpret_cast<const float4*>(prow + t + 4 * u * NT));
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            bad |= bad4(p4[u]);
                            rs_push4(P, p4[u], c);
                        }
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        bad |= bad4(q4[u]);
                        rs_push4(Q, q4[u], c);
                    }
                }
                for (; t < hi; t += 4 * NT) {
                    const float4 q0 = __ldg(reinterpret_cast<const float4*>(qrow + t));
                    bad |= bad4(q0);
                    rs_push4(Q, q0, c);
                    if (prow) {
                        const float4 p0 = __ldg(reinterpret_cast<const float4*>(prow + t));
                        bad |= bad4(p0);
                        rs_push4(P, p0, c);
                    }
                }
            } else {
                for (int t = lo + tid; t < hi; t += NT) {
                    const float lq = qrow[t];
                    bad |= isnan(lq) | (lq == INFINITY);
                    rs_push1(Q, lq, c);
                    if (prow) {
                        const float lp = prow[t];
                        bad |= isnan(lp) | (lp == INFINITY);
                        rs_push1(P, lp, c);
                    }
                }
            }
            if constexpr (!FILT) C::stats(sm, buf, Q, P, bad, c);
            if (bad || Q.lmax == -INFINITY || (prow && P.lmax == -INFINITY)) {
                err = EAGLE_DEV_NONFINITE;
                break;
            }
            if (a.row_stats && rank == 0 && tid == 0) {
                float* rs = a.row_stats;
                rs[(((int64_t)0 * a.B + b) * n + v) * 2 + 0] = Q.lmax / a.T;
                rs[(((int64_t)0 * a.B + b) * n + v) * 2 + 1] = Q.S;
                if (prow) {
                    rs[(((int64_t)1 * a.B + b) * n + v) * 2 + 0] = P.lmax / a.T;
                    rs[(((int64_t)1 * a.B + b) * n + v) * 2 + 1] = P.S;
                }
            }
            const float iq = 1.f / Q.S, ip = prow ? 1.f / P.S : 0.f;
            // ---------- children in index order ----------
            Residual rs{0.f, 1.f, 1.f};
            bool moved = false, fused = false;
            for (int ch = v + 1; ch < n && kids; ++ch) {
                if (sm.parent[ch] != v) continue;
                const int x = sm.tok[ch];
                float lq, lp;
                if (sharded) {
                    // q(x) and p(x): only the rank owning x holds them
                    int owner = 0;
                    while (owner + 1 < a.S && x >= a.sh.begin[owner + 1]) ++owner;
                    if (rank == owner) {
                        lq = qrow[x];
                        lp = pr.one(x);
                    }
                    C::bcast2(sm, buf, rank, owner, lq, lp);
                } else {
                    lq = mq(x, qrow[x]);
                    lp = mp(x, pr.one(x));
                }
                const float px = prob_of(lp, P.lmax, ip, c);
                const float r = resid_weight(lq, lp, Q, iq, P, ip, c, rs);
                const float u = accept_uniform(a.seed, (uint32_t)b, (uint32_t)ch);
                if (px <= 0.f || u < r / px) {
                    ++acc_n;
                    if (tid == 0) { sm.path[acc_n] = ch; sm.emit[acc_n - 1] = x; }
                    v = ch;
                    moved = true;
                    break;
                }
                if (ch == sm.lastkid[v]) {
                    // Last child rejected: the final token is drawn from norm(max(0,
                    // r_j - p)); its normaliser is a common factor of the race, so the
                    // race runs directly on the unnormalised weights.
                    fused = true;
                    break;
                }
                // ---------- pass: the next residual's normaliser ----------
                const float cnext = rs.rc + rs.rD;
                auto nr = [&](float lq2, float lp2, int t2) {
                    return next_resid(mq(t2, lq2), mp(t2, lp2), Q, iq, P, ip, c, cnext);
                };
                float s = 0.f;
                if (vec4) {
                    int t = lo + 4 * tid;
                    for (; t + 12 * NT < hi; t += 16 * NT) {      // 4 float4 of each row in flight
                        float4 a4[4], b4[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            a4[u] = __ldg(reinterpret_cast<const float4*>(qrow + t + 4 * u * NT));
                            b4[u] = pr.four(t + 4 * u * NT);
                        }
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            s += nr(a4[u].x, b4[u].x, t + 4 * u * NT) +
                                 nr(a4[u].y, b4[u].y, t + 4 * u * NT + 1) +
                                 nr(a4[u].z, b4[u].z, t + 4 * u * NT + 2) +
                                 nr(a4[u].w, b4[u].w, t + 4 * u * NT + 3);
                    }
                    for (; t < hi; t += 4 * NT) {
                        const float4 a4 = __ldg(reinterpret_cast<const float4*>(qrow + t));
                        const float4 b4 = pr.four(t);
                        s += nr(a4.x, b4.x, t) + nr(a4.y, b4.y, t + 1) + nr(a4.z, b4.z, t + 2) +
                             nr(a4.w, b4.w, t + 3);
                    }
                } else {
                    for (int t = lo + tid; t < hi; t += NT)
                        s += nr(qrow[t], pr.one(t), t);
                }
                const float S = C::sum(sm, buf, s);
                if (S > 0.f) rs = Residual{cnext, S, 1.f / S};   // else q_cur stays as it is
            }
            if (moved) continue;
            // ---------- pass: exponential race for the final token ----------
            int bad2 = 0;
            KeyIdx best;
            if (fused) {
                // weights max(0, r_j - p), up to the positive factor 1 / D_j
                const float cnext = rs.rc + rs.rD;
                best = race_slice<NT>(qrow, pr, lo, hi, vec4, (uint32_t)b, k0, k1,
                                      [&](float lq2, float lp2, int t2) {
                                          return next_resid(mq(t2, lq2), mp(t2, lp2), Q, iq, P, ip,
                                                            c, cnext);
                                      });
                best = C::argmax(sm, buf, best, bad2);
                if (best.i == 0x7fffffff) {
                    // the clamped residual is all zero: keep q_cur (= r_j)
                    best = race_slice<NT>(qrow, pr, lo, hi, vec4, (uint32_t)b, k0, k1,
                                          [&](float lq2, float lp2, int t2) {
                                              return resid_weight(mq(t2, lq2), mp(t2, lp2), Q, iq, P,
                                                                  ip, c, rs);
                                          });
                    best = C::argmax(sm, buf, best, bad2);
                }
            } else {
                best = race_slice<NT>(qrow, pr, lo, hi, vec4, (uint32_t)b, k0, k1,
                                      [&](float lq2, float lp2, int t2) {
                                          return resid_weight(mq(t2, lq2), mp(t2, lp2), Q, iq, P, ip,
                                                              c, rs);
                                      });
                best = C::argmax(sm, buf, best, bad2);
            }
            if (best.i == 0x7fffffff) {
                err = EAGLE_DEV_NONFINITE;
                break;
            }
            y = best.i;
        } else {
            // ---------- greedy: argmax of the target row ----------
            KeyIdx best{-INFINITY, 0x7fffffff};
            int bad = 0;
            if (vec4) {
                for (int t = lo + 4 * tid; t < hi; t += 4 * NT) {
                    const float4 l4 = __ldg(reinterpret_cast<const float4*>(qrow + t));
                    bad |= bad4(l4);
                    const float lx[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const KeyIdx cand{lx[e], t + e};
                        if (ki_better(cand, best)) best = cand;
                    }
                }
            } else {
                for (int t = lo + tid; t < hi; t += NT) {
                    const float l = qrow[t];
                    bad |= isnan(l) | (l == INFINITY);
                    const KeyIdx cand{l, t};
                    if (ki_better(cand, best)) best = cand;
                }
            }
            best = C::argmax(sm, buf, best, bad);
            if (bad || best.k == -INFINITY) {
                err = EAGLE_DEV_NONFINITE;
                break;
            }
            const int g = best.i;
            bool moved = false;
            for (int ch = v + 1; ch < n && kids; ++ch) {
                if (sm.parent[ch] == v && sm.tok[ch] == g) {
                    ++acc_n;
                    if (tid == 0) { sm.path[acc_n] = ch; sm.emit[acc_n - 1] = g; }
                    v = ch;
                    moved = true;
                    break;
                }
            }
            if (moved) continue;
            y = g;
        }
        break;
    }

    // ---- outputs ----
    __syncthreads();
    if (rank == 0) {
        const int Dp1 = a.D + 1;
        int32_t* P = a.path + (int64_t)b * Dp1;
        int32_t* E = a.emit + (int64_t)b * Dp1;
        for (int t = tid; t < Dp1; t += NT) {
            if (err) {
                P[t] = -1;
                E[t] = -1;
            } else {
                P[t] = t <= acc_n ? sm.path[t] : -1;
                E[t] = t < acc_n ? sm.emit[t] : (t == acc_n ? y : -1);
            }
        }
        if (tid == 0) {
            a.accept_len[b] = err ? -1 : acc_n;
            if (err) flag_error(a.dev_status, err);
        }
    }
    // No CTA may leave while a peer can still read its exchange slots.
    C::sync();
}

// ---------------------------------------------------------------------------
// Standalone row statistics: one CTA per row (grid-stride), loads hoisted four
// float4 deep; (max, sum) in the exp2 domain; argmax only when asked.
// ---------------------------------------------------------------------------
constexpr int kStatThreads = 256;

template <bool STATS, bool ARGMAX>
__global__ void __launch_bounds__(kStatThreads)
softmax_stats_kernel(const float* __restrict__ logits, int64_t rows, int V, float T, float c,
                     float* row_max, float* row_sum, int32_t* row_argmax, int32_t* dev_status) {
    __shared__ float red_f[kStatThreads / 32][3];
    __shared__ int red_i[kStatThreads / 32];
    __shared__ int red_bad[kStatThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool vec4 = ((V & 3) == 0) && ((reinterpret_cast<uintptr_t>(logits) & 15) == 0);
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        const float* row = logits + r * (int64_t)V;
        RowStat st{-INFINITY, 0.f};
        KeyIdx best{-INFINITY, 0x7fffffff};
        int bad = 0;
        auto take4 = [&](float4 l4, int t) {
            bad |= bad4(l4);
            if (STATS) rs_push4(st, l4, c);
            if (ARGMAX) {
                const float lx[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const KeyIdx cand{lx[e], t + e};
                    if (ki_better(cand, best)) best = cand;
                }
            }
        };
        if (vec4) {
            const float4* r4 = reinterpret_cast<const float4*>(row);
            const int n4 = V >> 2;
            int t = tid;
            for (; t + 3 * kStatThreads < n4; t += 4 * kStatThreads) {
                const float4 a0 = __ldg(r4 + t), a1 = __ldg(r4 + t + kStatThreads);
                const float4 a2 = __ldg(r4 + t + 2 * kStatThreads), a3 = __ldg(r4 + t + 3 * kStatThreads);
                take4(a0, 4 * t);
                take4(a1, 4 * (t + kStatThreads));
                take4(a2, 4 * (t + 2 * kStatThreads));
                take4(a3, 4 * (t + 3 * kStatThreads));
            }
            for (; t < n4; t += kStatThreads) take4(__ldg(r4 + t), 4 * t);
        } else {
            for (int t = tid; t < V; t += kStatThreads) {
                const float l = row[t];
                bad |= isnan(l) | (l == INFINITY);
                if (STATS) rs_push1(st, l, c);
                if (ARGMAX) {
                    const KeyIdx cand{l, t};
                    if (ki_better(cand, best)) best = cand;
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            st = rs_combine(st, RowStat{__shfl_xor_sync(~0u, st.lmax, o), __shfl_xor_sync(~0u, st.S, o)}, c);
        best = warp_argmax(best);
        bad = __any_sync(0xffffffffu, bad);
        if (lane == 0) {
            red_f[warp][0] = st.lmax; red_f[warp][1] = st.S; red_f[warp][2] = best.k;
            red_i[warp] = best.i;
            red_bad[warp] = bad;
        }
        __syncthreads();
        if (tid == 0) {
            RowStat m{-INFINITY, 0.f};
            KeyIdx bb{-INFINITY, 0x7fffffff};
            int bd = 0;
            for (int w = 0; w < kStatThreads / 32; ++w) {
                m = rs_combine(m, RowStat{red_f[w][0], red_f[w][1]}, c);
                const KeyIdx cand{red_f[w][2], red_i[w]};
                if (ki_better(cand, bb)) bb = cand;
                bd |= red_bad[w];
            }
            if (bd || (STATS && m.lmax == -INFINITY) || (ARGMAX && bb.k == -INFINITY))
                flag_error(dev_status, EAGLE_DEV_NONFINITE);
            if (STATS) {
                row_max[r] = m.lmax / T;
                row_sum[r] = m.S;
            }
            if (ARGMAX) row_argmax[r] = bb.i;
        }
        __syncthreads();
    }
}


// CTAs per sequence: 8 while the clusters fit about four per SM, halved as B grows.
int verify_cluster_size(int B) {
    const int sms = device_sm_count();
    int cs = 8;
    while (cs > 1 && (int64_t)B * cs > 4LL * sms) cs >>= 1;
    return cs;
}

constexpr int kVerifyThreads = 256;

template <bool D2T, bool FILT>
cudaError_t launch_walk(const VerifyArgs& a, cudaStream_t s) {
    constexpr int NT = kVerifyThreads;
    switch (verify_cluster_size(a.B)) {
        case 8: return launch_clustered(verify_walk_kernel<8, NT, D2T, FILT>, a.B, 8, NT, 0, s, a);
        case 4: return launch_clustered(verify_walk_kernel<4, NT, D2T, FILT>, a.B, 4, NT, 0, s, a);
        case 2: return launch_clustered(verify_walk_kernel<2, NT, D2T, FILT>, a.B, 2, NT, 0, s, a);
        default: return launch_clustered(verify_walk_kernel<1, NT, D2T, FILT>, a.B, 1, NT, 0, s, a);
    }
}

// t2d[t] = d for t = d + d2t[d], -1 for target ids no draft id maps to.  A draft id
// mapped outside [0, V) or onto a target id another draft id already holds flags
// EAGLE_DEV_BAD_TOKEN (and is left out of the table).
__global__ void t2d_fill_kernel(int32_t* t2d, int V) {
    for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < V; t += gridDim.x * blockDim.x) t2d[t] = -1;
}
__global__ void t2d_scatter_kernel(const int32_t* d2t, int Vd, int32_t* t2d, int V, int32_t* dev_status) {
    for (int d = blockIdx.x * blockDim.x + threadIdx.x; d < Vd; d += gridDim.x * blockDim.x) {
        const int64_t t = (int64_t)d + d2t[d];
        if (t < 0 || t >= V || atomicCAS(&t2d[t], -1, d) != -1) flag_error(dev_status, EAGLE_DEV_BAD_TOKEN);
    }
}

eagle_status verify_common(const float* target_logits, const float* draft_logits, const int32_t* draft_row,
                           const int32_t* tokens, const int32_t* parent, int B, int n, int V, int R,
                           int Vd, const int32_t* t2d, int max_depth, float temperature, uint64_t seed,
                           int32_t* accept_len, int32_t* path, int32_t* emit, float* row_stats,
                           int32_t* dev_status, eagle_stream_t stream, int top_k = 0,
                           float top_p = 0.f, void* workspace = nullptr, size_t ws_bytes = 0) {
    if (B < 0 || n < 1 || V < 1 || max_depth < 0) return EAGLE_ERR_INVALID_ARG;
    if (n > kMaxNodes || max_depth > kMaxNodes) return EAGLE_ERR_SHAPE;
    if (!(temperature >= 0.f) || !(temperature < INFINITY)) return EAGLE_ERR_INVALID_ARG;
    if (temperature > 0.f && R < 1) return EAGLE_ERR_INVALID_ARG;
    if (B == 0) return EAGLE_OK;                        // nothing read or written
    if (!target_logits || !tokens || !parent || !accept_len || !path || !emit)
        return EAGLE_ERR_INVALID_ARG;
    if (temperature > 0.f) {
        if (!draft_logits) return EAGLE_ERR_INVALID_ARG;
        if (!draft_row && R != n) return EAGLE_ERR_SHAPE;
    }
    const float c = temperature > 0.f ? kLog2e / temperature : 0.f;
    VerifyArgs a{target_logits, draft_logits, draft_row, tokens, parent, B, n, V, R, max_depth,
                 temperature, c, seed, accept_len, path, emit, row_stats, dev_status, Vd, t2d,
                 nullptr, nullptr, 0, 0.f, false};
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool filt = temperature > 0.f && ((top_k > 0 && top_k < V) || (top_p > 0.f && top_p < 1.f));
    cudaError_t e;
    if (filt) {
        if (t2d) return EAGLE_ERR_INVALID_ARG;             // filtering with a draft vocabulary: not offered
        if (V > kFiltMaxV) return EAGLE_ERR_SHAPE;
        const size_t need = (size_t)B * (n + R) * sizeof(FilterParam);
        if (!workspace || ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 15))
            return EAGLE_ERR_CAPACITY;
        FilterParam* fq = static_cast<FilterParam*>(workspace);
        FilterParam* fp = fq + (size_t)B * n;
        a.fq = fq;
        a.fp = fp;
        a.top_k = top_k;
        a.top_p = top_p;
        cudaPointerAttributes pa{};
        const cudaError_t qe = cudaPointerGetAttributes(&pa, target_logits);
        if (qe != cudaSuccess) cudaGetLastError();   // the query's own error, not a launch's
        a.target_in_device = qe == cudaSuccess &&
                             (pa.type == cudaMemoryTypeDevice || pa.type == cudaMemoryTypeManaged);
        e = launch_walk<false, true>(a, s);
    } else {
        e = t2d ? launch_walk<true, false>(a, s) : launch_walk<false, false>(a, s);
    }
    return e == cudaSuccess ? EAGLE_OK : EAGLE_ERR_CUDA;
}

}  // namespace
}  // namespace eagle

using namespace eagle;

extern "C" eagle_status eagle_verify_accept(const float* target_logits, const float* draft_logits,
                                            const int32_t* draft_row, const int32_t* tokens,
                                            const int32_t* parent, int B, int n, int V, int R,
                                            int max_depth, float temperature, uint64_t seed,
                                            int32_t* accept_len, int32_t* path, int32_t* emit,
                                            float* row_stats, int32_t* dev_status,
                                            eagle_stream_t stream) {
    return verify_common(target_logits, draft_logits, draft_row, tokens, parent, B, n, V, R, V,
                         nullptr, max_depth, temperature, seed, accept_len, path, emit, row_stats,
                         dev_status, stream);
}

extern "C" eagle_status eagle_verify_accept_sharded(
    const float* const* target_shards, const float* const* draft_shards, const int32_t* shard_begin,
    int S, const int32_t* draft_row, const int32_t* tokens, const int32_t* parent, int B, int n, int V,
    int R, int max_depth, float temperature, uint64_t seed, int32_t* accept_len, int32_t* path,
    int32_t* emit, float* row_stats, int32_t* dev_status, eagle_stream_t stream) {
    if (!target_shards || !shard_begin || S < 1) return EAGLE_ERR_INVALID_ARG;
    if (S > kMaxShards) return EAGLE_ERR_SHAPE;
    if (B < 0 || n < 1 || V < 1 || max_depth < 0) return EAGLE_ERR_INVALID_ARG;
    if (n > kMaxNodes || max_depth > kMaxNodes) return EAGLE_ERR_SHAPE;
    if (!(temperature >= 0.f) || !(temperature < INFINITY)) return EAGLE_ERR_INVALID_ARG;
    if (shard_begin[0] != 0 || shard_begin[S] != V) return EAGLE_ERR_SHAPE;
    for (int r = 0; r < S; ++r)
        if (shard_begin[r + 1] <= shard_begin[r]) return EAGLE_ERR_SHAPE;     // empty shard
    const bool t_pos = temperature > 0.f;
    if (t_pos && R < 1) return EAGLE_ERR_INVALID_ARG;
    if (B == 0) return EAGLE_OK;                        // nothing read or written
    if (!tokens || !parent || !accept_len || !path || !emit) return EAGLE_ERR_INVALID_ARG;
    if (t_pos) {
        if (!draft_shards) return EAGLE_ERR_INVALID_ARG;
        if (!draft_row && R != n) return EAGLE_ERR_SHAPE;
    }
    VerifyArgs a{};
    bool vec4 = (V & 3) == 0;
    for (int r = 0; r < S; ++r) {
        if (!target_shards[r] || (t_pos && !draft_shards[r])) return EAGLE_ERR_INVALID_ARG;
        a.sh.tgt[r] = target_shards[r];
        a.sh.drf[r] = t_pos ? draft_shards[r] : nullptr;
        a.sh.begin[r] = shard_begin[r];
        vec4 = vec4 && (shard_begin[r] & 3) == 0 &&
               (reinterpret_cast<uintptr_t>(target_shards[r]) & 15) == 0 &&
               (!t_pos || (reinterpret_cast<uintptr_t>(draft_shards[r]) & 15) == 0);
    }
    a.sh.begin[S] = V;
    a.target = target_shards[0];
    a.draft = t_pos ? draft_shards[0] : nullptr;
    a.draft_row = draft_row;
    a.tokens = tokens;
    a.parent = parent;
    a.B = B; a.n = n; a.V = V; a.R = R; a.D = max_depth;
    a.T = temperature;
    a.c = t_pos ? kLog2e / temperature : 0.f;
    a.seed = seed;
    a.accept_len = accept_len; a.path = path; a.emit = emit;
    a.row_stats = row_stats;
    a.dev_status = dev_status;
    a.Vd = V;
    a.S = S;
    a.shard_vec4 = vec4;
    constexpr int NT = kVerifyThreads;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // one CTA per rank; the cluster is the next power of two, extra CTAs hold no shard
    cudaError_t e;
    if (S == 1) e = launch_clustered(verify_walk_kernel<1, NT, false, false>, B, 1, NT, 0, s, a);
    else if (S == 2) e = launch_clustered(verify_walk_kernel<2, NT, false, false>, B, 2, NT, 0, s, a);
    else if (S <= 4) e = launch_clustered(verify_walk_kernel<4, NT, false, false>, B, 4, NT, 0, s, a);
    else e = launch_clustered(verify_walk_kernel<8, NT, false, false>, B, 8, NT, 0, s, a);
    return e == cudaSuccess ? EAGLE_OK : EAGLE_ERR_CUDA;
}

extern "C" eagle_status eagle_verify_accept_d2t(const float* target_logits, const float* draft_logits,
                                                const int32_t* draft_row, const int32_t* tokens,
                                                const int32_t* parent, int B, int n, int V, int R,
                                                int Vd, const int32_t* t2d, int max_depth,
                                                float temperature, uint64_t seed,
                                                int32_t* accept_len, int32_t* path, int32_t* emit,
                                                float* row_stats, int32_t* dev_status,
                                                eagle_stream_t stream) {
    if (Vd < 1 || (B != 0 && !t2d)) return EAGLE_ERR_INVALID_ARG;
    return verify_common(target_logits, draft_logits, draft_row, tokens, parent, B, n, V, R, Vd, t2d,
                         max_depth, temperature, seed, accept_len, path, emit, row_stats, dev_status,
                         stream);
}

extern "C" size_t eagle_verify_filter_workspace_size(int B, int n, int R) {
    if (B < 0 || n < 1 || R < 1) return 0;
    return (size_t)B * (n + R) * sizeof(FilterParam);
}

extern "C" eagle_status eagle_verify_accept_filtered(const float* target_logits,
                                                     const float* draft_logits,
                                                     const int32_t* draft_row, const int32_t* tokens,
                                                     const int32_t* parent, int B, int n, int V,
                                                     int R, int max_depth, float temperature,
                                                     uint64_t seed, int top_k, float top_p,
                                                     int32_t* accept_len, int32_t* path,
                                                     int32_t* emit, float* row_stats,
                                                     void* workspace, size_t ws_bytes,
                                                     int32_t* dev_status, eagle_stream_t stream) {
    if (top_k < 0 || !(top_p >= 0.f) || !(top_p < INFINITY)) return EAGLE_ERR_INVALID_ARG;
    return verify_common(target_logits, draft_logits, draft_row, tokens, parent, B, n, V, R, V,
                         nullptr, max_depth, temperature, seed, accept_len, path, emit, row_stats,
                         dev_status, stream, top_k, top_p, workspace, ws_bytes);
}

extern "C" eagle_status eagle_d2t_inverse(const int32_t* d2t, int Vd, int V, int32_t* t2d,
                                          int32_t* dev_status, eagle_stream_t stream) {
    if (!d2t || !t2d || Vd < 1 || V < 1) return EAGLE_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int grid = device_sm_count() * 4;
    t2d_fill_kernel<<<grid, 256, 0, s>>>(t2d, V);
    EAGLE_CHECK_LAUNCH();
    t2d_scatter_kernel<<<grid, 256, 0, s>>>(d2t, Vd, t2d, V, dev_status);
    EAGLE_CHECK_LAUNCH();
    return EAGLE_OK;
}

namespace eagle {
namespace {
// Resident CTAs per SM of one softmax_stats_kernel variant (looked up once per variant).
template <bool STATS, bool ARGMAX>
int stats_ctas_per_sm() {
    static int cached = 0;
    if (cached == 0) {
        int v = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                &v, softmax_stats_kernel<STATS, ARGMAX>, kStatThreads, 0) != cudaSuccess)
            return 0;
        cached = v;
    }
    return cached;
}
}  // namespace
}  // namespace eagle

extern "C" eagle_status eagle_softmax_stats(const float* logits, int64_t rows, int V,
                                            float temperature, float* row_max, float* row_sum,
                                            int32_t* row_argmax, int32_t* dev_status,
                                            eagle_stream_t stream) {
    if (rows < 0 || V < 1) return EAGLE_ERR_INVALID_ARG;
    if (!(temperature >= 0.f) || !(temperature < INFINITY)) return EAGLE_ERR_INVALID_ARG;
    if (rows == 0) return EAGLE_OK;                     // nothing read or written
    const bool stats = temperature > 0.f;
    if (!logits) return EAGLE_ERR_INVALID_ARG;
    if (stats && (!row_max || !row_sum)) return EAGLE_ERR_INVALID_ARG;
    if (!stats && !row_argmax) return EAGLE_ERR_INVALID_ARG;
    const float c = stats ? kLog2e / temperature : 0.f;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // One resident wave: every CTA of the grid is on an SM from the start (the variants
    // differ in registers, hence in CTAs per SM), and each walks its rows grid-stride.
    auto launch = [&](auto kernel, int per_sm) -> eagle_status {
        if (per_sm < 1) return EAGLE_ERR_CUDA;
        const int64_t cap = (int64_t)device_sm_count() * per_sm;
        const int grid = (int)(rows < cap ? rows : cap);
        kernel<<<grid, kStatThreads, 0, s>>>(logits, rows, V, temperature, c, row_max, row_sum,
                                             row_argmax, dev_status);
        EAGLE_CHECK_LAUNCH();
        return EAGLE_OK;
    };
    if (stats && row_argmax)
        return launch(softmax_stats_kernel<true, true>, stats_ctas_per_sm<true, true>());
    if (stats) return launch(softmax_stats_kernel<true, false>, stats_ctas_per_sm<true, false>());
    return launch(softmax_stats_kernel<false, true>, stats_ctas_per_sm<false, true>());
}
