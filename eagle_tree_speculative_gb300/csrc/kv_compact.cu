// KV compaction of the accepted path and the logical-length update.
//
// Method (Lesson "推测解码与 EAGLE-3", sections "KV cache 回滚" and "第 4 步"):
// keep one physical cache and a logical length; after verification the
// accepted rows become part of the committed prefix.  The tree's rows sit at
// L_b + j; for t = 0..a the row L_b + path[t] moves to L_b + t, then
// kv_len[b] = L_b + a + 1.
//
// In-place safety: the accepted path is strictly increasing with path[0] = 0,
// so path[t] >= t.  Rows are moved in rounds of increasing t; a round first
// loads all its source rows into registers (__syncwarp) and then stores.  A
// store of round k goes to row L + t with t < every source index path[t'] of
// a later round (path[t'] >= t' > t), so no later source is overwritten, and
// no earlier round can have written a source of round k (those destinations
// are below 2k <= t <= path[t]).  Launch: one cluster per sequence; the cluster
// barrier at the end orders every CTA's read of kv_len[b] before its update.
#include <cstdlib>

#include "common.cuh"

namespace eagle {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

struct CompactArgs {
    uint16_t* k;
    uint16_t* v;
    int32_t* kv_len;
    const int32_t* path;
    const int32_t* accept_len;
    int n_layers, B, Hkv, Lmax, D;
    int32_t* dev_status;
};

template <int CS>
__global__ void __launch_bounds__(kThreads) kv_compact_kernel(CompactArgs a) {
    __shared__ int s_path[kMaxNodes + 1];
    __shared__ int s_ok;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rank = CS > 1 ? (int)cg::this_cluster().block_rank() : 0;
    const int b = blockIdx.x / CS;
    const int acc = a.accept_len[b];
    const int L = a.kv_len[b];
    if (tid == 0) {
        int ok = acc >= 0;
        int err = 0;
        if (ok) {
            if (acc > a.D || L < 0 || (int64_t)L + acc + 1 > a.Lmax) { ok = 0; err = EAGLE_DEV_CAPACITY; }
            for (int t = 0; ok && t <= acc; ++t) {
                int p = a.path[(int64_t)b * (a.D + 1) + t];
                s_path[t] = p;
                if ((t == 0 && p != 0) || (t > 0 && p <= s_path[t - 1])) { ok = 0; err = EAGLE_DEV_BAD_TREE; }
                else if ((int64_t)L + p >= a.Lmax) { ok = 0; err = EAGLE_DEV_CAPACITY; }
            }
        }
        if (err && rank == 0) flag_error(a.dev_status, err);
        s_ok = ok;
    }
    __syncthreads();
    if (s_ok) {
        const int units = a.n_layers * 2 * a.Hkv;           // (layer, K|V, kv head)
        const int64_t row_elems = kHeadDim;
        for (int u = rank * kWarps + warp; u < units; u += CS * kWarps) {
            const int h = u % a.Hkv;
            const int kv = (u / a.Hkv) & 1;
            const int layer = u / (2 * a.Hkv);
            uint16_t* base = (kv ? a.v : a.k) +
                             ((((int64_t)layer * a.B + b) * a.Hkv + h) * a.Lmax + L) * row_elems;
            // 32 lanes x 16 bytes = two 256-byte rows per round
            for (int t0 = 0; t0 <= acc; t0 += 2) {
                const int t = t0 + (lane >> 4), c = lane & 15;
                uint4 val = make_uint4(0u, 0u, 0u, 0u);
                const bool active = t <= acc && s_path[t] != t;
                if (active)
                    val = *reinterpret_cast<const uint4*>(base + (int64_t)s_path[t] * row_elems + c * 8);
                __syncwarp();
                if (active) *reinterpret_cast<uint4*>(base + (int64_t)t * row_elems + c * 8) = val;
                __syncwarp();
            }
        }
    }
    if constexpr (CS > 1) cg::this_cluster().sync();
    else __syncthreads();
    if (rank == 0 && tid == 0 && s_ok) a.kv_len[b] = L + acc + 1;
}

int compact_cluster_size(int B) {
    const int sms = device_sm_count();
    int cs = 8;
    while (cs > 1 && (int64_t)B * cs > 4LL * sms) cs >>= 1;
    return cs;
}

}  // namespace
}  // namespace eagle

using namespace eagle;

extern "C" eagle_status eagle_kv_compact(void* k_cache, void* v_cache, int32_t* kv_len,
                                         const int32_t* path, const int32_t* accept_len,
                                         int n_layers, int B, int Hkv, int head_dim, int Lmax,
                                         int max_depth, int32_t* dev_status,
                                         eagle_stream_t stream) {
    if (n_layers < 0 || B < 0 || Hkv < 1 || Lmax < 1 || max_depth < 0) return EAGLE_ERR_INVALID_ARG;
    if (head_dim != kHeadDim || max_depth > kMaxNodes) return EAGLE_ERR_SHAPE;
    if (B == 0 || n_layers == 0) return EAGLE_OK;       // nothing read or written
    if (!k_cache || !v_cache || !kv_len || !path || !accept_len) return EAGLE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(k_cache) & 15) || (reinterpret_cast<uintptr_t>(v_cache) & 15))
        return EAGLE_ERR_INVALID_ARG;
    CompactArgs a{static_cast<uint16_t*>(k_cache), static_cast<uint16_t*>(v_cache), kv_len, path,
                  accept_len, n_layers, B, Hkv, Lmax, max_depth, dev_status};
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (compact_cluster_size(B)) {
        case 8: e = launch_clustered(kv_compact_kernel<8>, B, 8, kThreads, 0, s, a); break;
        case 4: e = launch_clustered(kv_compact_kernel<4>, B, 4, kThreads, 0, s, a); break;
        case 2: e = launch_clustered(kv_compact_kernel<2>, B, 2, kThreads, 0, s, a); break;
        default: e = launch_clustered(kv_compact_kernel<1>, B, 1, kThreads, 0, s, a); break;
    }
    return e == cudaSuccess ? EAGLE_OK : EAGLE_ERR_CUDA;
}
