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

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;

struct VerifyArgs {
    const float* target;
    const float* draft;
    const int32_t* draft_row;
    const int32_t* tokens;
    const int32_t* parent;
    int B, n, V, R, D;
    float T;
    uint64_t seed;
    int32_t* accept_len;
    int32_t* path;
    int32_t* emit;
    float* row_stats;
    int32_t* dev_status;
};

struct Slot {
    float f[4];
    int i;
    int bad;
};

// Per-CTA scratch and the cluster exchange slots.
struct VerifySmem {
    int parent[kMaxNodes];
    int tok[kMaxNodes];
    int row[kMaxNodes];
    int nkids[kMaxNodes];
    float S[kMaxNodes + 1];          // residual normalisers S_1..S_j of the current node
    int path[kMaxNodes + 1];
    int emit[kMaxNodes + 1];
    float red[kWarps][4];
    int redi[kWarps];
    int redbad[kWarps];
    Slot x[2];                       // double-buffered exchange slot
    int err;
};

template <int CS>
struct Sync {
    __device__ static void all() {
        if constexpr (CS > 1) cg::this_cluster().sync();
        else __syncthreads();
    }
    __device__ static const Slot* slot(VerifySmem& sm, int buf, int rank) {
        if constexpr (CS > 1) return cg::this_cluster().map_shared_rank(&sm.x[buf], rank);
        else return &sm.x[buf];
    }
};

__device__ __forceinline__ int cta_rank_in_cluster(int cs) {
    if (cs > 1) return (int)cg::this_cluster().block_rank();
    return 0;
}

// ----- element-wise helpers (z = l / T, IEEE division) ---------------------
__device__ __forceinline__ void ms_push(MaxSum& a, float z) {
    if (z == -INFINITY) return;
    if (z > a.m) {
        a.s = (a.m == -INFINITY) ? 0.f : a.s * expf(a.m - z);
        a.m = z;
    }
    a.s += expf(z - a.m);
}

__device__ __forceinline__ bool not_finite_logit(float l) { return isnan(l) || l == INFINITY; }

// Residual weight of token t after j rejections at the current node:
// r_0 = q(t); r_i = max(0, r_{i-1} - p(t)) / S_i  (unchanged when S_i == 0).
__device__ __forceinline__ float residual_at(float lq, float lp, float T, float mq, float Zq,
                                             float mp, float Zp, const float* S, int j) {
    float r = expf(lq / T - mq) / Zq;
    if (j == 0) return r;
    float pp = expf(lp / T - mp) / Zp;
    for (int i = 1; i <= j; ++i) {
        float s = S[i];
        if (s > 0.f) r = fmaxf(0.f, r - pp) / s;
    }
    return r;
}

// ---------------------------------------------------------------------------
template <int CS>
__global__ void __launch_bounds__(kThreads) verify_walk_kernel(VerifyArgs a) {
    __shared__ VerifySmem sm;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rank = cta_rank_in_cluster(CS);
    const int b = blockIdx.x / CS;
    const int n = a.n, V = a.V;
    const float T = a.T;
    const int64_t Vl = V;

    // ---- load and validate the tree (identically in every CTA) ----
    if (tid < n) {
        sm.parent[tid] = a.parent[(int64_t)b * n + tid];
        sm.tok[tid] = a.tokens[(int64_t)b * n + tid];
        sm.row[tid] = a.draft_row ? a.draft_row[(int64_t)b * n + tid] : tid;
        sm.nkids[tid] = 0;
    }
    __syncthreads();
    if (tid == 0) {
        int err = 0;
        int depth[kMaxNodes];
        if (sm.parent[0] != -1) err |= EAGLE_DEV_BAD_TREE;
        depth[0] = 0;
        for (int i = 1; i < n && !err; ++i) {
            int p = sm.parent[i];
            if (p < 0 || p >= i) { err |= EAGLE_DEV_BAD_TREE; break; }
            depth[i] = depth[p] + 1;
            if (depth[i] > a.D) err |= EAGLE_DEV_DEPTH;
            if (sm.tok[i] < 0 || sm.tok[i] >= V) err |= EAGLE_DEV_BAD_TOKEN;
            sm.nkids[p] += 1;
        }
        if (!err && T > 0.f)
            for (int i = 0; i < n; ++i)
                if (sm.nkids[i] && (sm.row[i] < 0 || sm.row[i] >= a.R)) err |= EAGLE_DEV_BAD_TOKEN;
        sm.err = err;
    }
    __syncthreads();

    // ---- vocabulary slice of this CTA ----
    const int chunk = (((V + CS - 1) / CS) + 3) & ~3;
    const int lo = min(V, rank * chunk), hi = min(V, lo + chunk);
    const float* tgt_b = a.target + (int64_t)b * n * Vl;
    const float* drf_b = a.draft ? a.draft + (int64_t)b * a.R * Vl : nullptr;
    const bool vec4 = ((V & 3) == 0) && ((reinterpret_cast<uintptr_t>(a.target) & 15) == 0) &&
                      (a.draft == nullptr || (reinterpret_cast<uintptr_t>(a.draft) & 15) == 0);
    const uint32_t k0 = (uint32_t)a.seed, k1 = (uint32_t)(a.seed >> 32);

    int buf = 0;
    int err = sm.err;
    int v = 0, acc_n = 0, y = -1;
    if (tid == 0) sm.path[0] = 0;

    while (!err) {
        const float* qrow = tgt_b + (int64_t)v * Vl;
        const bool kids = sm.nkids[v] > 0;
        int moved = 0;
        if (T > 0.f) {
            const float* prow = kids ? drf_b + (int64_t)sm.row[v] * Vl : nullptr;
            // ---------- pass: row statistics of q(v) and p(v) ----------
            MaxSum Q{-INFINITY, 0.f}, P{-INFINITY, 0.f};
            int bad = 0;
            if (vec4) {
#pragma unroll 2
                for (int t = lo + 4 * tid; t < hi; t += 4 * kThreads) {
                    float4 lq = __ldg(reinterpret_cast<const float4*>(qrow + t));
                    float4 lp = prow ? __ldg(reinterpret_cast<const float4*>(prow + t))
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
                    bad |= not_finite_logit(lq.x) | not_finite_logit(lq.y) |
                           not_finite_logit(lq.z) | not_finite_logit(lq.w);
                    ms_push(Q, lq.x / T); ms_push(Q, lq.y / T);
                    ms_push(Q, lq.z / T); ms_push(Q, lq.w / T);
                    if (prow) {
                        bad |= not_finite_logit(lp.x) | not_finite_logit(lp.y) |
                               not_finite_logit(lp.z) | not_finite_logit(lp.w);
                        ms_push(P, lp.x / T); ms_push(P, lp.y / T);
                        ms_push(P, lp.z / T); ms_push(P, lp.w / T);
                    }
                }
            } else {
                for (int t = lo + tid; t < hi; t += kThreads) {
                    float lq = qrow[t];
                    bad |= not_finite_logit(lq);
                    ms_push(Q, lq / T);
                    if (prow) {
                        float lp = prow[t];
                        bad |= not_finite_logit(lp);
                        ms_push(P, lp / T);
                    }
                }
            }
            Q = warp_ms(Q);
            P = warp_ms(P);
            bad = __any_sync(0xffffffffu, bad);
            if (lane == 0) {
                sm.red[warp][0] = Q.m; sm.red[warp][1] = Q.s;
                sm.red[warp][2] = P.m; sm.red[warp][3] = P.s;
                sm.redbad[warp] = bad;
            }
            __syncthreads();
            if (tid == 0) {
                MaxSum q{-INFINITY, 0.f}, p{-INFINITY, 0.f};
                int bd = 0;
                for (int w = 0; w < kWarps; ++w) {
                    q = ms_combine(q, MaxSum{sm.red[w][0], sm.red[w][1]});
                    p = ms_combine(p, MaxSum{sm.red[w][2], sm.red[w][3]});
                    bd |= sm.redbad[w];
                }
                sm.x[buf].f[0] = q.m; sm.x[buf].f[1] = q.s;
                sm.x[buf].f[2] = p.m; sm.x[buf].f[3] = p.s;
                sm.x[buf].bad = bd;
            }
            Sync<CS>::all();
            MaxSum q{-INFINITY, 0.f}, p{-INFINITY, 0.f};
            bad = 0;
#pragma unroll
            for (int r = 0; r < CS; ++r) {
                const Slot* s = Sync<CS>::slot(sm, buf, r);
                q = ms_combine(q, MaxSum{s->f[0], s->f[1]});
                p = ms_combine(p, MaxSum{s->f[2], s->f[3]});
                bad |= s->bad;
            }
            buf ^= 1;
            if (bad || q.m == -INFINITY || (prow && p.m == -INFINITY)) {
                err = EAGLE_DEV_NONFINITE;
                break;
            }
            const float mq = q.m, Zq = q.s, mp = p.m, Zp = p.s;
            if (a.row_stats && rank == 0 && tid == 0) {
                float* rs = a.row_stats;
                rs[(((int64_t)0 * a.B + b) * n + v) * 2 + 0] = mq;
                rs[(((int64_t)0 * a.B + b) * n + v) * 2 + 1] = Zq;
                if (prow) {
                    rs[(((int64_t)1 * a.B + b) * n + v) * 2 + 0] = mp;
                    rs[(((int64_t)1 * a.B + b) * n + v) * 2 + 1] = Zp;
                }
            }
            // ---------- children in index order ----------
            int j = 0;
            for (int c = v + 1; c < n && kids; ++c) {
                if (sm.parent[c] != v) continue;
                const int x = sm.tok[c];
                const float lq = qrow[x], lp = prow[x];
                const float px = expf(lp / T - mp) / Zp;
                const float r = residual_at(lq, lp, T, mq, Zq, mp, Zp, sm.S, j);
                const float u = accept_uniform(a.seed, (uint32_t)b, (uint32_t)c);
                if (px <= 0.f || u < r / px) {
                    ++acc_n;
                    if (tid == 0) { sm.path[acc_n] = c; sm.emit[acc_n - 1] = x; }
                    v = c;
                    moved = 1;
                    break;
                }
                // ---------- pass: residual normaliser S_{j+1} ----------
                float s = 0.f;
                if (vec4) {
#pragma unroll 2
                    for (int t = lo + 4 * tid; t < hi; t += 4 * kThreads) {
                        float4 a4 = __ldg(reinterpret_cast<const float4*>(qrow + t));
                        float4 b4 = __ldg(reinterpret_cast<const float4*>(prow + t));
                        float ax[4] = {a4.x, a4.y, a4.z, a4.w}, bx[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            float rr = residual_at(ax[e], bx[e], T, mq, Zq, mp, Zp, sm.S, j);
                            s += fmaxf(0.f, rr - expf(bx[e] / T - mp) / Zp);
                        }
                    }
                } else {
                    for (int t = lo + tid; t < hi; t += kThreads) {
                        float rr = residual_at(qrow[t], prow[t], T, mq, Zq, mp, Zp, sm.S, j);
                        s += fmaxf(0.f, rr - expf(prow[t] / T - mp) / Zp);
                    }
                }
                s = warp_sum(s);
                if (lane == 0) sm.red[warp][0] = s;
                __syncthreads();
                if (tid == 0) {
                    float t = 0.f;
                    for (int w = 0; w < kWarps; ++w) t += sm.red[w][0];
                    sm.x[buf].f[0] = t;
                }
                Sync<CS>::all();
                float S = 0.f;
#pragma unroll
                for (int r2 = 0; r2 < CS; ++r2) S += Sync<CS>::slot(sm, buf, r2)->f[0];
                buf ^= 1;
                ++j;
                if (tid == 0) sm.S[j] = S;
                __syncthreads();
            }
            if (moved) continue;
            // ---------- pass: exponential race over q_cur ----------
            KeyIdx best{-1.f, 0x7fffffff};
            if (vec4) {
                for (int t = lo + 4 * tid; t < hi; t += 4 * kThreads) {
                    float4 a4 = __ldg(reinterpret_cast<const float4*>(qrow + t));
                    float4 b4 = prow ? __ldg(reinterpret_cast<const float4*>(prow + t))
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
                    uint4 w = philox4x32_10(make_uint4((uint32_t)t >> 2, 0u, (uint32_t)b, kTagRace),
                                            k0, k1);
                    float ax[4] = {a4.x, a4.y, a4.z, a4.w}, bx[4] = {b4.x, b4.y, b4.z, b4.w};
                    uint32_t wx[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        float rr = residual_at(ax[e], bx[e], T, mq, Zq, mp, Zp, sm.S, j);
                        if (rr > 0.f) {
                            float key = rr / -logf(unit_open(wx[e]));
                            KeyIdx cand{key, t + e};
                            if (ki_better(cand, best)) best = cand;
                        }
                    }
                }
            } else {
                for (int t = lo + tid; t < hi; t += kThreads) {
                    float rr = residual_at(qrow[t], prow ? prow[t] : 0.f, T, mq, Zq, mp, Zp, sm.S, j);
                    if (rr > 0.f) {
                        uint4 w = philox4x32_10(
                            make_uint4((uint32_t)t >> 2, 0u, (uint32_t)b, kTagRace), k0, k1);
                        uint32_t wx[4] = {w.x, w.y, w.z, w.w};
                        float key = rr / -logf(unit_open(wx[t & 3]));
                        KeyIdx cand{key, t};
                        if (ki_better(cand, best)) best = cand;
                    }
                }
            }
            best = warp_argmax(best);
            if (lane == 0) { sm.red[warp][0] = best.k; sm.redi[warp] = best.i; }
            __syncthreads();
            if (tid == 0) {
                KeyIdx bb{-1.f, 0x7fffffff};
                for (int w = 0; w < kWarps; ++w) {
                    KeyIdx c{sm.red[w][0], sm.redi[w]};
                    if (ki_better(c, bb)) bb = c;
                }
                sm.x[buf].f[0] = bb.k;
                sm.x[buf].i = bb.i;
            }
            Sync<CS>::all();
            KeyIdx bb{-1.f, 0x7fffffff};
#pragma unroll
            for (int r2 = 0; r2 < CS; ++r2) {
                const Slot* s = Sync<CS>::slot(sm, buf, r2);
                KeyIdx c{s->f[0], s->i};
                if (ki_better(c, bb)) bb = c;
            }
            buf ^= 1;
            y = bb.i;
        } else {
            // ---------- greedy: argmax of the target row ----------
            KeyIdx best{-INFINITY, 0x7fffffff};
            int bad = 0;
            if (vec4) {
                for (int t = lo + 4 * tid; t < hi; t += 4 * kThreads) {
                    float4 l4 = __ldg(reinterpret_cast<const float4*>(qrow + t));
                    float lx[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        bad |= not_finite_logit(lx[e]);
                        KeyIdx c{lx[e], t + e};
                        if (ki_better(c, best)) best = c;
                    }
                }
            } else {
                for (int t = lo + tid; t < hi; t += kThreads) {
                    float l = qrow[t];
                    bad |= not_finite_logit(l);
                    KeyIdx c{l, t};
                    if (ki_better(c, best)) best = c;
                }
            }
            best = warp_argmax(best);
            bad = __any_sync(0xffffffffu, bad);
            if (lane == 0) { sm.red[warp][0] = best.k; sm.redi[warp] = best.i; sm.redbad[warp] = bad; }
            __syncthreads();
            if (tid == 0) {
                KeyIdx bb{-INFINITY, 0x7fffffff};
                int bd = 0;
                for (int w = 0; w < kWarps; ++w) {
                    KeyIdx c{sm.red[w][0], sm.redi[w]};
                    if (ki_better(c, bb)) bb = c;
                    bd |= sm.redbad[w];
                }
                sm.x[buf].f[0] = bb.k;
                sm.x[buf].i = bb.i;
                sm.x[buf].bad = bd;
            }
            Sync<CS>::all();
            KeyIdx bb{-INFINITY, 0x7fffffff};
            int bd = 0;
#pragma unroll
            for (int r2 = 0; r2 < CS; ++r2) {
                const Slot* s = Sync<CS>::slot(sm, buf, r2);
                KeyIdx c{s->f[0], s->i};
                if (ki_better(c, bb)) bb = c;
                bd |= s->bad;
            }
            buf ^= 1;
            if (bd || bb.k == -INFINITY) {
                err = EAGLE_DEV_NONFINITE;
                break;
            }
            const int g = bb.i;
            for (int c = v + 1; c < n && kids; ++c) {
                if (sm.parent[c] == v && sm.tok[c] == g) {
                    ++acc_n;
                    if (tid == 0) { sm.path[acc_n] = c; sm.emit[acc_n - 1] = g; }
                    v = c;
                    moved = 1;
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
        for (int t = tid; t < Dp1; t += kThreads) {
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
    Sync<CS>::all();
}

// ---------------------------------------------------------------------------
// Standalone row statistics: one CTA per row (grid-stride).
// ---------------------------------------------------------------------------
constexpr int kStatThreads = 256;

__global__ void __launch_bounds__(kStatThreads)
softmax_stats_kernel(const float* __restrict__ logits, int64_t rows, int V, float T,
                     float* row_max, float* row_sum, int32_t* row_argmax, int32_t* dev_status) {
    __shared__ float red_f[kStatThreads / 32][2];
    __shared__ int red_i[kStatThreads / 32];
    __shared__ int red_bad[kStatThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool vec4 = ((V & 3) == 0) && ((reinterpret_cast<uintptr_t>(logits) & 15) == 0);
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        const float* row = logits + r * (int64_t)V;
        MaxSum ms{-INFINITY, 0.f};
        KeyIdx best{-INFINITY, 0x7fffffff};
        int bad = 0;
        if (vec4) {
#pragma unroll 4
            for (int t = 4 * tid; t < V; t += 4 * kStatThreads) {
                float4 l4 = __ldg(reinterpret_cast<const float4*>(row + t));
                float lx[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    bad |= not_finite_logit(lx[e]);
                    KeyIdx c{lx[e], t + e};
                    if (ki_better(c, best)) best = c;
                    if (T > 0.f) ms_push(ms, lx[e] / T);
                }
            }
        } else {
            for (int t = tid; t < V; t += kStatThreads) {
                float l = row[t];
                bad |= not_finite_logit(l);
                KeyIdx c{l, t};
                if (ki_better(c, best)) best = c;
                if (T > 0.f) ms_push(ms, l / T);
            }
        }
        ms = warp_ms(ms);
        best = warp_argmax(best);
        bad = __any_sync(0xffffffffu, bad);
        if (lane == 0) {
            red_f[warp][0] = ms.m; red_f[warp][1] = ms.s;
            red_i[warp] = best.i;
            red_bad[warp] = bad;
            // keep the argmax key next to its index
        }
        __shared__ float red_k[kStatThreads / 32];
        if (lane == 0) red_k[warp] = best.k;
        __syncthreads();
        if (tid == 0) {
            MaxSum m{-INFINITY, 0.f};
            KeyIdx bb{-INFINITY, 0x7fffffff};
            int bd = 0;
            for (int w = 0; w < kStatThreads / 32; ++w) {
                m = ms_combine(m, MaxSum{red_f[w][0], red_f[w][1]});
                KeyIdx c{red_k[w], red_i[w]};
                if (ki_better(c, bb)) bb = c;
                bd |= red_bad[w];
            }
            if (bd || bb.k == -INFINITY) flag_error(dev_status, EAGLE_DEV_NONFINITE);
            if (T > 0.f) {
                if (row_max) row_max[r] = m.m;
                if (row_sum) row_sum[r] = m.s;
            }
            if (row_argmax) row_argmax[r] = bb.i;
        }
        __syncthreads();
    }
}

int verify_cluster_size(int B) {
    static int forced = -1;
    if (forced < 0) {
        const char* e = std::getenv("EAGLE_VERIFY_CLUSTER");
        int f = e ? std::atoi(e) : 0;
        forced = (f == 1 || f == 2 || f == 4 || f == 8) ? f : 0;
    }
    if (forced > 0) return forced;
    const int sms = device_sm_count();
    int cs = 8;
    while (cs > 1 && (int64_t)B * cs > 2LL * sms) cs >>= 1;
    return cs;
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
    if (B < 0 || n < 1 || V < 1 || max_depth < 0) return EAGLE_ERR_INVALID_ARG;
    if (n > kMaxNodes || max_depth > kMaxNodes) return EAGLE_ERR_SHAPE;
    if (!(temperature >= 0.f) || !(temperature < INFINITY)) return EAGLE_ERR_INVALID_ARG;
    if (!target_logits || !tokens || !parent || !accept_len || !path || !emit)
        return EAGLE_ERR_INVALID_ARG;
    if (temperature > 0.f) {
        if (!draft_logits || R < 1) return EAGLE_ERR_INVALID_ARG;
        if (!draft_row && R != n) return EAGLE_ERR_SHAPE;
    }
    if (B == 0) return EAGLE_OK;
    VerifyArgs a{target_logits, draft_logits, draft_row, tokens, parent, B, n, V, R, max_depth,
                 temperature, seed, accept_len, path, emit, row_stats, dev_status};
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (verify_cluster_size(B)) {
        case 8: e = launch_clustered(verify_walk_kernel<8>, B, 8, kThreads, 0, s, a); break;
        case 4: e = launch_clustered(verify_walk_kernel<4>, B, 4, kThreads, 0, s, a); break;
        case 2: e = launch_clustered(verify_walk_kernel<2>, B, 2, kThreads, 0, s, a); break;
        default: e = launch_clustered(verify_walk_kernel<1>, B, 1, kThreads, 0, s, a); break;
    }
    return e == cudaSuccess ? EAGLE_OK : EAGLE_ERR_CUDA;
}

extern "C" eagle_status eagle_softmax_stats(const float* logits, int64_t rows, int V,
                                            float temperature, float* row_max, float* row_sum,
                                            int32_t* row_argmax, int32_t* dev_status,
                                            eagle_stream_t stream) {
    if (!logits || rows < 0 || V < 1) return EAGLE_ERR_INVALID_ARG;
    if (!(temperature >= 0.f) || !(temperature < INFINITY)) return EAGLE_ERR_INVALID_ARG;
    if (temperature > 0.f && (!row_max || !row_sum)) return EAGLE_ERR_INVALID_ARG;
    if (temperature == 0.f && !row_argmax) return EAGLE_ERR_INVALID_ARG;
    if (rows == 0) return EAGLE_OK;
    const int64_t cap = (int64_t)device_sm_count() * 8;
    const int grid = (int)(rows < cap ? rows : cap);
    softmax_stats_kernel<<<grid, kStatThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        logits, rows, V, temperature, row_max, row_sum, row_argmax, dev_status);
    EAGLE_CHECK_LAUNCH();
    return EAGLE_OK;
}
