// EAGLE-2 draft-tree expansion and reranking.
//
// Method (Guide "EAGLE-1/2/3 拆解", section "EAGLE-2：草稿树的 Expansion 与
// Reranking"; TTT page, section "EAGLE-3 和 EAGLE-2 动态树如何拼在一起"):
// node value V_i = product of draft confidences on the root path; expansion
// runs the draft forward only on the top-k nodes of the previous level;
// reranking keeps the global top-n nodes by V for verification.
//
// Kernels per level:
//   row_topk_kernel  one CTA per frontier row: temperature-1 softmax statistics
//                    and the row's top-k tokens (logit desc, token asc) in one
//                    pass over the vocabulary; confidences c = exp(l - m) / Z.
//   select_kernel    one CTA per sequence: the k_in * k candidates of the level,
//                    V_child = V_parent * c in float32, the next frontier = the k
//                    best by (V desc, id asc), and draft-row assignment.
//   rerank_kernel    one CTA per sequence: bitonic sort of every candidate by
//                    (V desc, depth asc, id asc), keep n-1 plus the root, then
//                    sort those by (depth asc, V desc, id asc) and re-index parents.
// The draft LM-head GEMM (lmhead_gemm.cu) writes the level's logits rows first
// when hidden states are given.
#include <cstdlib>
#include <mutex>

#include "common.cuh"

namespace eagle {

// Defined in lmhead_gemm.cu.
eagle_status lmhead_gemm_launch(const void* hidden, const void* w, float* out, int M, int K, int N,
                                int64_t ldo, int rows_per_group, int64_t group_stride,
                                int64_t row_offset, int32_t* dev_status, cudaStream_t stream);

namespace {

constexpr int kKMax = 16;
constexpr int kDepthMax = 16;

// Per-sequence tree state, 32-bit words:
//   [0] non-finite flag  [1..3] reserved
//   value[C] f32, parent[C], token[C], depth[C], row[C], frontier[kKMax],
//   row_tok[kKMax * kKMax], row_conf[kKMax * kKMax] f32
struct StateView {
    int C, k;
    int64_t stride;  // words per sequence
    __host__ __device__ static int cand_count(int k, int D) { return 1 + k + (D - 1) * k * k; }
    __host__ __device__ static int64_t words(int k, int D) {
        return 4 + 5LL * cand_count(k, D) + kKMax + 2LL * kKMax * kKMax;
    }
};

struct SeqState {
    int* hdr;
    float* value;
    int* parent;
    int* token;
    int* depth;
    int* row;
    int* frontier;
    int* row_tok;
    float* row_conf;
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
    s.frontier = p + 4 + 5 * C;
    s.row_tok = s.frontier + kKMax;
    s.row_conf = reinterpret_cast<float*>(s.row_tok + kKMax * kKMax);
    return s;
}

__device__ __forceinline__ bool topk_better(float v, int i, float w, int j) {
    return v > w || (v == w && i < j);
}

// ---------------------------------------------------------------------------
// Row softmax statistics + top-k in one pass over the vocabulary.
// Statistics: each thread keeps an online (max, sum) with sum = sum
// 2^((l - max) log2 e).  Top-k: each warp keeps ONE sorted list distributed
// over its lanes (lane j holds the j-th best, order: logit desc, token asc).
// A chunk of 4 logits per lane is filtered against the warp's current k-th
// best (a ballot); the rare survivors are inserted one at a time with a
// shuffle shift.  The block then merges the per-warp lists the same way.
constexpr int kTopkThreads = 256;
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

__global__ void __launch_bounds__(kTopkThreads)
row_topk_kernel(const float* __restrict__ logits, int k_in, int R, int off, int V, int k, int D,
                void* state, int32_t* dev_status) {
    __shared__ float s_v[kTopkThreads / 32][kKMax];
    __shared__ int s_i[kTopkThreads / 32][kKMax];
    __shared__ float s_red[kTopkThreads / 32][2];
    __shared__ int s_bad[kTopkThreads / 32];
    __shared__ float s_pick_v[kKMax];
    __shared__ int s_pick_i[kKMax];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.x / k_in, s = blockIdx.x % k_in;
    const float* x = logits + ((int64_t)b * R + off + s) * (int64_t)V;

    float lv = -INFINITY;            // warp list entry of this lane
    int li = 0x7fffffff;
    float tv = -INFINITY;            // the warp's current k-th best (broadcast)
    int ti = 0x7fffffff;
    float m = -INFINITY, sum = 0.f;
    int bad = 0;

    auto offer = [&](float v, int i, bool mine) {
        // lanes with a surviving candidate insert it, one lane at a time
        unsigned ball = __ballot_sync(0xffffffffu, mine && topk_better(v, i, tv, ti));
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
    auto chunk4 = [&](float4 l4, int t, bool valid) {
        if (valid) {
            bad |= isnan(l4.x) | isnan(l4.y) | isnan(l4.z) | isnan(l4.w) | (l4.x == INFINITY) |
                   (l4.y == INFINITY) | (l4.z == INFINITY) | (l4.w == INFINITY);
            const float mx = fmaxf(fmaxf(l4.x, l4.y), fmaxf(l4.z, l4.w));
            if (mx > m) {
                sum = (m == -INFINITY) ? 0.f : sum * exp2f((m - mx) * kLog2e);
                m = mx;
            }
            if (m != -INFINITY)
                sum += exp2f((l4.x - m) * kLog2e) + exp2f((l4.y - m) * kLog2e) +
                       exp2f((l4.z - m) * kLog2e) + exp2f((l4.w - m) * kLog2e);
        }
        offer(l4.x, t, valid);
        offer(l4.y, t + 1, valid);
        offer(l4.z, t + 2, valid);
        offer(l4.w, t + 3, valid);
    };

    if (((V & 3) == 0) && ((reinterpret_cast<uintptr_t>(logits) & 15) == 0)) {
        const float4* x4 = reinterpret_cast<const float4*>(x);
        const int n4 = V >> 2;
        // warp-uniform trip counts: every lane of a warp runs the same iterations
        int base = warp * 32;
        for (; base + 3 * kTopkThreads < n4; base += 4 * kTopkThreads) {
            const int t = base + lane;
            const float4 a0 = __ldg(x4 + t), a1 = __ldg(x4 + t + kTopkThreads);
            const float4 a2 = __ldg(x4 + t + 2 * kTopkThreads), a3 = __ldg(x4 + t + 3 * kTopkThreads);
            chunk4(a0, 4 * t, true);
            chunk4(a1, 4 * (t + kTopkThreads), true);
            chunk4(a2, 4 * (t + 2 * kTopkThreads), true);
            chunk4(a3, 4 * (t + 3 * kTopkThreads), true);
        }
        for (; base < n4; base += kTopkThreads) {
            const int t = base + lane;
            const bool ok = t < n4;
            chunk4(ok ? __ldg(x4 + t) : make_float4(0.f, 0.f, 0.f, 0.f), 4 * t, ok);
        }
    } else {
        for (int base = warp * 32; base < V; base += kTopkThreads) {
            const int t = base + lane;
            const bool ok = t < V;
            const float l = ok ? x[t] : 0.f;
            if (ok) {
                bad |= isnan(l) | (l == INFINITY);
                if (l > m) { sum = (m == -INFINITY) ? 0.f : sum * exp2f((m - l) * kLog2e); m = l; }
                if (m != -INFINITY) sum += exp2f((l - m) * kLog2e);
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
                sum = sum * exp2f((m - nm) * kLog2e) + os * exp2f((om - nm) * kLog2e);
                m = nm;
            }
        }
    }
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) { s_red[warp][0] = m; s_red[warp][1] = sum; s_bad[warp] = bad; }
    if (lane < kKMax) { s_v[warp][lane] = lv; s_i[warp][lane] = li; }
    __syncthreads();
    if (warp == 0) {
        lv = -INFINITY; li = 0x7fffffff;
        tv = -INFINITY; ti = 0x7fffffff;
        for (int w = 0; w < kTopkThreads / 32; ++w)
            for (int j = 0; j < k; ++j) {
                const float cv = s_v[w][j];
                const int ci = s_i[w][j];
                if (ci != 0x7fffffff && topk_better(cv, ci, tv, ti)) {
                    warp_list_insert(lv, li, cv, ci);
                    tv = __shfl_sync(0xffffffffu, lv, k - 1);
                    ti = __shfl_sync(0xffffffffu, li, k - 1);
                }
            }
        if (lane < k) { s_pick_v[lane] = lv; s_pick_i[lane] = li; }
    }
    __syncthreads();
    if (tid == 0) {
        float M = -INFINITY, S = 0.f;
        int bd = 0;
        for (int w = 0; w < kTopkThreads / 32; ++w) {
            const float wm = s_red[w][0], ws = s_red[w][1];
            bd |= s_bad[w];
            if (wm == -INFINITY) continue;
            if (M == -INFINITY) { M = wm; S = ws; continue; }
            const float nm = fmaxf(M, wm);
            S = S * exp2f((M - nm) * kLog2e) + ws * exp2f((wm - nm) * kLog2e);
            M = nm;
        }
        SeqState st = seq_state(state, b, k, D);
        if (bd || M == -INFINITY) {
            st.hdr[0] = 1;
            flag_error(dev_status, EAGLE_DEV_NONFINITE);
        }
        for (int j = 0; j < k; ++j) {
            st.row_tok[s * kKMax + j] = s_pick_i[j];
            st.row_conf[s * kKMax + j] = exp2f((s_pick_v[j] - M) * kLog2e) / S;
        }
    }
}

// ---------------------------------------------------------------------------
constexpr int kSelectThreads = 256;

__global__ void __launch_bounds__(kSelectThreads)
select_kernel(int level, int final, int k, int D, void* state, int32_t* frontier_tokens) {
    __shared__ float s_val[kKMax * kKMax];
    __shared__ int s_id[kKMax * kKMax];
    const int tid = threadIdx.x, b = blockIdx.x;
    SeqState st = seq_state(state, b, k, D);
    const int k_in = level == 1 ? 1 : k;
    if (level == 1 && tid == 0) {
        st.value[0] = 1.0f;
        st.parent[0] = -1;
        st.token[0] = -1;
        st.depth[0] = 0;
        st.row[0] = 0;
        st.frontier[0] = 0;
    }
    __syncthreads();
    const int ncand = k_in * k;
    for (int e = tid; e < ncand; e += kSelectThreads) {
        const int s = e / k, j = e % k;
        const int id = level == 1 ? 1 + j : 1 + k + (level - 2) * k * k + s * k + j;
        const int par = st.frontier[s];
        const float val = __fmul_rn(st.value[par], st.row_conf[s * kKMax + j]);
        st.value[id] = val;
        st.parent[id] = par;
        st.token[id] = st.row_tok[s * kKMax + j];
        st.depth[id] = level;
        st.row[id] = -1;
        s_val[e] = val;
        s_id[e] = id;
    }
    __syncthreads();
    // rank of each candidate in (V desc, id asc); the k best form the frontier
    for (int e = tid; e < ncand; e += kSelectThreads) {
        const float v = s_val[e];
        const int id = s_id[e];
        int rank = 0;
        for (int f = 0; f < ncand; ++f) rank += topk_better(s_val[f], s_id[f], v, id);
        if (rank < k) {
            st.frontier[rank] = id;
            if (level < D && !final) st.row[id] = 1 + (level - 1) * k + rank;
            if (frontier_tokens) frontier_tokens[(int64_t)b * k + rank] = st.token[id];
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

}  // namespace
}  // namespace eagle

using namespace eagle;

extern "C" size_t eagle2_tree_state_size(int B, int top_k, int depth) {
    if (B < 0 || top_k < 1 || top_k > kKMax || depth < 1 || depth > kDepthMax) return 0;
    return (size_t)B * (size_t)StateView::words(top_k, depth) * 4u;
}

extern "C" eagle_status eagle2_expand(int level, int final, const void* hidden,
                                      const void* lm_head_w, float* logits, int B, int H, int V,
                                      int top_k, int depth, int n_out, void* tree_state,
                                      size_t state_bytes, int32_t* out_tokens, int32_t* out_parent,
                                      int32_t* out_draft_row, int32_t* frontier_tokens,
                                      int32_t* dev_status, eagle_stream_t stream) {
    if (B < 0 || V < 1 || top_k < 1 || depth < 1 || level < 1 || level > depth || !logits ||
        !tree_state)
        return EAGLE_ERR_INVALID_ARG;
    if (top_k > kKMax || depth > kDepthMax || top_k > V) return EAGLE_ERR_SHAPE;
    if (state_bytes < eagle2_tree_state_size(B, top_k, depth)) return EAGLE_ERR_CAPACITY;
    const int C = StateView::cand_count(top_k, depth);
    if (C > 4096) return EAGLE_ERR_SHAPE;
    if (final) {
        if (!out_tokens || !out_parent || !out_draft_row) return EAGLE_ERR_INVALID_ARG;
        if (n_out < 2 || n_out > kMaxNodes) return EAGLE_ERR_SHAPE;
        const int have = 1 + top_k + (level - 1) * top_k * top_k;
        if (n_out > have) return EAGLE_ERR_SHAPE;
    }
    if (hidden && (!lm_head_w || H < 1)) return EAGLE_ERR_INVALID_ARG;
    if (B == 0) return EAGLE_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int R = 1 + (depth - 1) * top_k;
    const int k_in = level == 1 ? 1 : top_k;
    const int off = level == 1 ? 0 : 1 + (level - 2) * top_k;
    if (hidden) {
        eagle_status st = lmhead_gemm_launch(hidden, lm_head_w, logits, B * k_in, H, V, V, k_in,
                                             (int64_t)R, off, dev_status, s);
        if (st != EAGLE_OK) return st;
    }
    row_topk_kernel<<<B * k_in, kTopkThreads, 0, s>>>(logits, k_in, R, off, V, top_k, depth,
                                                     tree_state, dev_status);
    EAGLE_CHECK_LAUNCH();
    select_kernel<<<B, kSelectThreads, 0, s>>>(level, final, top_k, depth, tree_state,
                                                 frontier_tokens);
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
// per device (with that device current) and cached.
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
    const size_t need = eagle2_tree_state_size(B, top_k, depth);
    if (need == 0 && B != 0) return EAGLE_ERR_SHAPE;
    if (need > kStaticStateBytes) return EAGLE_ERR_CAPACITY;
    void* state = nullptr;
    const eagle_status st = static_state_address(&state);
    if (st != EAGLE_OK) return st;
    // Level 1 writes every field of a sequence's state that later levels read,
    // so the array needs no clearing between trees.
    return eagle2_expand(level, final, hidden, lm_head_w, logits, B, H, V, top_k, depth, n_out,
                         state, kStaticStateBytes, out_tokens, out_parent, out_draft_row,
                         frontier_tokens, dev_status, stream);
}
