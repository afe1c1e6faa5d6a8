// Tree-masked GQA attention over the committed KV cache plus the tree rows:
// host side (argument checks, TMA tensor maps, the split-KV decision) and the
// split-KV combine kernel.  The attention kernel itself is tree_attn_tc_kernel
// (tree_attn_tc.cuh, tcgen05 + TMA).
//
// Method (Lesson "推测解码与 EAGLE-3", section "KV cache 回滚": the verifier
// attends with a non-causal mask that follows the tree, one flash-attention
// call with a custom mask; Guide "EAGLE-1/2/3 拆解", section "EAGLE-2": tree
// attention puts every tree token through one forward).  Node i sees the
// committed rows 0..L_b-1 and the tree rows L_b + j for j = i or an ancestor
// of i, encoded as a 64-bit ancestor mask per node built from the parent array.
// When the (sequence, kv head, row tile) units alone leave most SMs idle, the
// committed keys are split across CTAs and the partial (max, sum, O) are merged
// by a log-sum-exp combine kernel.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "tree_attn_tc.cuh"

namespace eagle {
namespace {

constexpr int kMaxSplits = 16;

struct AttnArgs {
    const uint16_t* q;
    const uint16_t* k;
    const uint16_t* v;
    const int32_t* kv_len;
    const int32_t* parent;
    uint16_t* out;
    float* ws_o;    // [splits, B*n*Hq, 128] unnormalised partial outputs
    float* ws_ml;   // [splits, B*n*Hq, 2]  (running max in log2 units, running sum)
    int B, n, Hq, Hkv, G, Lmax, splits;
    float scale_log2;
    int32_t* dev_status;
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// One warp per output row: merge the split partials (log2-domain maxima).
__global__ void __launch_bounds__(256) tree_attn_combine_kernel(AttnArgs a, int64_t rows) {
    const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    float mt = -INFINITY;
    for (int s = 0; s < a.splits; ++s) mt = fmaxf(mt, a.ws_ml[((int64_t)s * rows + row) * 2]);
    const float base = mt == -INFINITY ? 0.f : mt;
    float lt = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < a.splits; ++s) {
        const float2 ml = *reinterpret_cast<const float2*>(a.ws_ml + ((int64_t)s * rows + row) * 2);
        const float w = exp2f(ml.x - base);
        lt += ml.y * w;
        const float4 x = *reinterpret_cast<const float4*>(a.ws_o + ((int64_t)s * rows + row) * kHeadDim + lane * 4);
        acc.x += x.x * w; acc.y += x.y * w; acc.z += x.z * w; acc.w += x.w * w;
    }
    const float inv = lt > 0.f ? 1.f / lt : 0.f;
    uint2 pk = make_uint2(pack_bf16(acc.x * inv, acc.y * inv), pack_bf16(acc.z * inv, acc.w * inv));
    *reinterpret_cast<uint2*>(a.out + row * kHeadDim + lane * 4) = pk;
}

// K or V cache viewed as a 3-D tensor: head_dim (128, innermost), Lmax rows of one
// (sequence, kv head), then B * Hkv of those; 64 x TBN x 1 boxes.  Rows outside 0 .. Lmax - 1
// of a (sequence, head) read as zeros, never as the neighbouring head's rows.
bool kv_map(CUtensorMap* map, const void* base, int Lmax, int64_t heads) {
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)Lmax, (cuuint64_t)heads};
    cuuint64_t strides[2] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)Lmax * kHeadDim * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)attn_tc::TBN, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int tc_row_groups(int n, int G) { return (n * G + attn_tc::ROWS_PER_CTA - 1) / attn_tc::ROWS_PER_CTA; }

int tc_splits(int B, int n, int Hq, int Hkv, int Lmax) {
    const int G = Hq / Hkv;
    const int64_t ctas = (int64_t)B * Hkv * tc_row_groups(n, G);
    const int sms = device_sm_count();
    int splits = (int)((2 * sms + ctas - 1) / ctas);
    const int max_by_len = (Lmax - n) / (4 * attn_tc::TBN);
    splits = splits < max_by_len ? splits : max_by_len;
    splits = splits < kMaxSplits ? splits : kMaxSplits;
    return splits < 1 ? 1 : splits;
}

}  // namespace
}  // namespace eagle

using namespace eagle;

extern "C" size_t eagle_tree_attn_workspace_size(int B, int n, int Hq, int Hkv, int head_dim,
                                                 int Lmax) {
    if (B < 1 || n < 1 || Hkv < 1 || Hq % Hkv != 0 || head_dim != kHeadDim || Lmax < n) return 0;
    const int splits = tc_splits(B, n, Hq, Hkv, Lmax);
    if (splits == 1) return 0;
    return (size_t)splits * B * n * Hq * (kHeadDim + 2) * sizeof(float);
}

extern "C" eagle_status eagle_tree_attn(const void* q, const void* k_cache, const void* v_cache,
                                        const int32_t* kv_len, const int32_t* parent, void* out,
                                        int B, int n, int Hq, int Hkv, int head_dim, int Lmax,
                                        float scale, void* workspace, size_t ws_bytes,
                                        int32_t* dev_status, eagle_stream_t stream) {
    if (B < 0 || n < 1 || Hq < 1 || Hkv < 1 || Lmax < 1 || !(scale > 0.f)) return EAGLE_ERR_INVALID_ARG;
    if (n > kMaxNodes || head_dim != kHeadDim || Hq % Hkv != 0 || Lmax < n) return EAGLE_ERR_SHAPE;
    if (B == 0) return EAGLE_OK;                        // nothing read or written
    if (!q || !k_cache || !v_cache || !kv_len || !parent || !out) return EAGLE_ERR_INVALID_ARG;
    for (const void* p : {q, k_cache, v_cache, (const void*)out})
        if (reinterpret_cast<uintptr_t>(p) & 15) return EAGLE_ERR_INVALID_ARG;
    const int splits = tc_splits(B, n, Hq, Hkv, Lmax);
    const size_t need = splits > 1 ? (size_t)splits * B * n * Hq * (kHeadDim + 2) * sizeof(float) : 0;
    if (need > 0 && (!workspace || ws_bytes < need)) return EAGLE_ERR_CAPACITY;
    const int G = Hq / Hkv;
    AttnArgs a;
    a.q = static_cast<const uint16_t*>(q);
    a.k = static_cast<const uint16_t*>(k_cache);
    a.v = static_cast<const uint16_t*>(v_cache);
    a.kv_len = kv_len;
    a.parent = parent;
    a.out = static_cast<uint16_t*>(out);
    const int64_t rows = (int64_t)B * n * Hq;
    a.ws_o = splits > 1 ? static_cast<float*>(workspace) : nullptr;
    a.ws_ml = splits > 1 ? static_cast<float*>(workspace) + (size_t)splits * rows * kHeadDim : nullptr;
    a.B = B; a.n = n; a.Hq = Hq; a.Hkv = Hkv; a.G = G; a.Lmax = Lmax; a.splits = splits;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.dev_status = dev_status;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    CUtensorMap mk, mv;
    const int64_t heads = (int64_t)B * Hkv;
    if (heads > 0x7fffffffLL) return EAGLE_ERR_SHAPE;
    if (!kv_map(&mk, k_cache, Lmax, heads) || !kv_map(&mv, v_cache, Lmax, heads)) return EAGLE_ERR_CUDA;
    attn_tc::Args t;
    t.q = a.q; t.out = a.out; t.ws_o = a.ws_o; t.ws_ml = a.ws_ml; t.kv_len = kv_len;
    t.parent = parent; t.B = B; t.n = n; t.Hq = Hq; t.Hkv = Hkv; t.G = G; t.Lmax = Lmax;
    t.splits = splits; t.scale_log2 = a.scale_log2; t.dev_status = dev_status;
    if (cudaFuncSetAttribute(attn_tc::tree_attn_tc_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             attn_tc::SMEM_BYTES) != cudaSuccess)
        return EAGLE_ERR_CUDA;
    dim3 grid((unsigned)tc_row_groups(n, G), (unsigned)(Hkv * splits), (unsigned)B);
    attn_tc::tree_attn_tc_kernel<<<grid, attn_tc::kThreads, attn_tc::SMEM_BYTES, s>>>(mk, mv, t);
    EAGLE_CHECK_LAUNCH();
    if (splits > 1) {
        tree_attn_combine_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(a, rows);
        EAGLE_CHECK_LAUNCH();
    }
    return EAGLE_OK;
}
