// Tree-masked GQA attention over the committed KV cache plus the tree rows.
//
// Method (Lesson "推测解码与 EAGLE-3", section "KV cache 回滚": the verifier
// attends with a non-causal mask that follows the tree, one flash-attention
// call with a custom mask; Guide "EAGLE-1/2/3 拆解", section "EAGLE-2": tree
// attention puts every tree token through one forward).  Node i sees the
// committed rows 0..L_b-1 and the tree rows L_b + j for j = i or an ancestor
// of i, encoded as a 64-bit ancestor mask per node built from the parent array.
//
// Kernel: flash-attention style tiling.  One CTA owns a block of 16 * NW query
// rows of one (sequence, kv head): the Hq/Hkv query heads sharing a kv head are
// packed as extra rows (row r = node r / G, head kvh * G + r % G), so each K/V
// tile is loaded once for all of them.  K/V tiles of 64 keys stream through
// shared memory with cp.async double buffering (XOR-swizzled 16-byte chunks so
// ldmatrix is conflict-free); QK^T and PV run on bf16 mma.sync with fp32
// accumulators and an online softmax in registers.  Committed keys may be
// split across CTAs (split-KV) and merged by a log-sum-exp combine kernel.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdlib>

#include "common.cuh"
#include "tree_attn_tc.cuh"

namespace eagle {
namespace {

constexpr int kKeyTile = 64;
constexpr int kTileBytes = kKeyTile * kHeadDim * 2;  // 16 KB
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

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
                 "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// byte offset of 16-byte chunk c of key row j inside a swizzled tile
__device__ __forceinline__ uint32_t swz(int j, int c) { return (uint32_t)(j * 256 + ((c ^ (j & 7)) << 4)); }

template <int NW>
__global__ void __launch_bounds__(NW * 32, 1) tree_attn_kernel(AttnArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ unsigned long long s_anc[kMaxNodes];
    __shared__ int s_err;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rb = blockIdx.x;
    const int kvh = blockIdx.y / a.splits, split = blockIdx.y % a.splits;
    const int b = blockIdx.z;
    const int n = a.n, G = a.G, rows = n * G;
    const int L = a.kv_len[b];

    if (tid == 0) {
        int err = 0;
        const int32_t* par = a.parent + (int64_t)b * n;
        if (par[0] != -1) err = EAGLE_DEV_BAD_TREE;
        s_anc[0] = 1ull;
        for (int i = 1; i < n && !err; ++i) {
            int p = par[i];
            if (p < 0 || p >= i) { err = EAGLE_DEV_BAD_TREE; break; }
            s_anc[i] = s_anc[p] | (1ull << i);
        }
        if (L < 0 || (int64_t)L + n > a.Lmax) err |= EAGLE_DEV_CAPACITY;
        if (err && rb == 0 && blockIdx.y == 0) flag_error(a.dev_status, err);
        s_err = err;
    }
    __syncthreads();

    // key range of this split: committed keys are chunked, the last split adds the tree
    int chunk = (L + a.splits - 1) / a.splits;
    chunk = (chunk + kKeyTile - 1) / kKeyTile * kKeyTile;
    const int kb = min(L, split * chunk);
    const int ke = (split == a.splits - 1) ? L + n : min(L, kb + chunk);
    const bool err = s_err != 0;

    // this thread's two rows (C-fragment rows lane/4 and lane/4 + 8)
    const int r0 = rb * (16 * NW) + warp * 16 + (lane >> 2);
    const int r1 = r0 + 8;
    const int i0 = r0 / G, i1 = r1 / G;
    const bool v0 = r0 < rows, v1 = r1 < rows;
    const unsigned long long anc0 = (!err && v0) ? s_anc[i0] : 0ull;
    const unsigned long long anc1 = (!err && v1) ? s_anc[i1] : 0ull;

    // Q fragments (16 rows x 128 dims of bf16) straight from global memory
    uint32_t qf[8][4];
    {
        const int c0 = (lane & 3) * 2;
        const uint16_t* q0 = a.q + (((int64_t)b * n + i0) * a.Hq + kvh * G + r0 % G) * kHeadDim;
        const uint16_t* q1 = a.q + (((int64_t)b * n + i1) * a.Hq + kvh * G + r1 % G) * kHeadDim;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const int col = kk * 16 + c0;
            qf[kk][0] = v0 ? *reinterpret_cast<const uint32_t*>(q0 + col) : 0u;
            qf[kk][1] = v1 ? *reinterpret_cast<const uint32_t*>(q1 + col) : 0u;
            qf[kk][2] = v0 ? *reinterpret_cast<const uint32_t*>(q0 + col + 8) : 0u;
            qf[kk][3] = v1 ? *reinterpret_cast<const uint32_t*>(q1 + col + 8) : 0u;
        }
    }

    float o[16][4];
#pragma unroll
    for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    const uint16_t* kbase = a.k + ((int64_t)b * a.Hkv + kvh) * a.Lmax * kHeadDim;
    const uint16_t* vbase = a.v + ((int64_t)b * a.Hkv + kvh) * a.Lmax * kHeadDim;
    const int ntiles = err ? 0 : (ke - kb + kKeyTile - 1) / kKeyTile;

    auto load_tile = [&](int t, int stage) {
        uint8_t* ks = smem + stage * 2 * kTileBytes;
        uint8_t* vs = ks + kTileBytes;
        const int key0 = kb + t * kKeyTile;
        for (int c = tid; c < kKeyTile * 16; c += NW * 32) {
            const int j = c >> 4, ch = c & 15;
            const int key = key0 + j;
            const bool in = key < ke;
            const int64_t off = (int64_t)(in ? key : kb) * kHeadDim + ch * 8;
            cp_async16(smem_u32(ks + swz(j, ch)), kbase + off, in ? 16 : 0);
            cp_async16(smem_u32(vs + swz(j, ch)), vbase + off, in ? 16 : 0);
        }
        cp_async_commit();
    };

    if (ntiles > 0) load_tile(0, 0);
    for (int t = 0; t < ntiles; ++t) {
        const int stage = t & 1;
        if (t + 1 < ntiles) {
            load_tile(t + 1, stage ^ 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const uint32_t ks = smem_u32(smem + stage * 2 * kTileBytes);
        const uint32_t vs = ks + kTileBytes;
        const int key0 = kb + t * kKeyTile;

        // ---- S = Q K^T : 16 rows x 64 keys per warp ----
        float s[8][4];
#pragma unroll
        for (int nb = 0; nb < 8; ++nb) s[nb][0] = s[nb][1] = s[nb][2] = s[nb][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                // matrices: keys np*16 + (0..7 | 8..15), dim chunks 2kk, 2kk+1
                const int key = np * 16 + (lane & 7) + ((lane >> 4) << 3);
                const int ch = 2 * kk + ((lane >> 3) & 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(ks + swz(key, ch), b0, b1, b2, b3);
                mma_bf16(s[2 * np], qf[kk], b0, b1);
                mma_bf16(s[2 * np + 1], qf[kk], b2, b3);
            }
        }
        // ---- mask (only tiles reaching the tree rows or the range end) ----
        const bool need_mask = key0 + kKeyTile > L || key0 + kKeyTile > ke;
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int nb = 0; nb < 8; ++nb) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int key = key0 + nb * 8 + (lane & 3) * 2 + e;
                float x0 = s[nb][e] * a.scale_log2, x1 = s[nb][2 + e] * a.scale_log2;
                if (need_mask) {
                    bool ok0 = key < ke, ok1 = key < ke;
                    if (key >= L) {
                        const int j = key - L;
                        ok0 = ok0 && j < n && ((anc0 >> j) & 1ull);
                        ok1 = ok1 && j < n && ((anc1 >> j) & 1ull);
                    }
                    x0 = ok0 ? x0 : -INFINITY;
                    x1 = ok1 ? x1 : -INFINITY;
                }
                s[nb][e] = x0;
                s[nb][2 + e] = x1;
                mx0 = fmaxf(mx0, x0);
                mx1 = fmaxf(mx1, x1);
            }
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float nm0 = fmaxf(m0, mx0), nm1 = fmaxf(m1, mx1);
        const float base0 = nm0 == -INFINITY ? 0.f : nm0, base1 = nm1 == -INFINITY ? 0.f : nm1;
        const float al0 = exp2f(m0 - base0), al1 = exp2f(m1 - base1);   // 0 when m was -inf
        m0 = nm0;
        m1 = nm1;
        float ps0 = 0.f, ps1 = 0.f;
        uint32_t pf[4][4];
#pragma unroll
        for (int nb = 0; nb < 8; ++nb) {
            const float p00 = exp2f(s[nb][0] - base0), p01 = exp2f(s[nb][1] - base0);
            const float p10 = exp2f(s[nb][2] - base1), p11 = exp2f(s[nb][3] - base1);
            ps0 += p00 + p01;
            ps1 += p10 + p11;
            // A fragment of P for key block nb / 2 (16 keys)
            pf[nb >> 1][(nb & 1) * 2 + 0] = pack_bf16(p00, p01);
            pf[nb >> 1][(nb & 1) * 2 + 1] = pack_bf16(p10, p11);
        }
        l0 = l0 * al0 + ps0;
        l1 = l1 * al1 + ps1;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            o[j][0] *= al0; o[j][1] *= al0;
            o[j][2] *= al1; o[j][3] *= al1;
        }
        // ---- O += P V ----
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            // A = P rows x keys kk*16..+15: regs (row, k0-7), (row+8, k0-7), (row, k8-15), (row+8, k8-15)
            const uint32_t af[4] = {pf[kk][0], pf[kk][1], pf[kk][2], pf[kk][3]};
#pragma unroll
            for (int dp = 0; dp < 8; ++dp) {
                // matrices: keys kk*16 + (0..7 | 8..15), dim chunks 2dp, 2dp+1 (transposed)
                const int key = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
                const int ch = 2 * dp + (lane >> 4);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(vs + swz(key, ch), b0, b1, b2, b3);
                mma_bf16(o[2 * dp], af, b0, b1);
                mma_bf16(o[2 * dp + 1], af, b2, b3);
            }
        }
        __syncthreads();
    }

    // ---- epilogue ----
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const int h0 = kvh * G + r0 % G, h1 = kvh * G + r1 % G;
    const int64_t row0 = ((int64_t)b * n + i0) * a.Hq + h0;
    const int64_t row1 = ((int64_t)b * n + i1) * a.Hq + h1;
    const int c0 = (lane & 3) * 2;
    if (a.splits == 1) {
        const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            if (v0) *reinterpret_cast<uint32_t*>(a.out + row0 * kHeadDim + j * 8 + c0) =
                        pack_bf16(o[j][0] * inv0, o[j][1] * inv0);
            if (v1) *reinterpret_cast<uint32_t*>(a.out + row1 * kHeadDim + j * 8 + c0) =
                        pack_bf16(o[j][2] * inv1, o[j][3] * inv1);
        }
    } else {
        const int64_t R = (int64_t)a.B * n * a.Hq;
        float* wo = a.ws_o + (int64_t)split * R * kHeadDim;
        float* wml = a.ws_ml + (int64_t)split * R * 2;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            if (v0) *reinterpret_cast<float2*>(wo + row0 * kHeadDim + j * 8 + c0) = make_float2(o[j][0], o[j][1]);
            if (v1) *reinterpret_cast<float2*>(wo + row1 * kHeadDim + j * 8 + c0) = make_float2(o[j][2], o[j][3]);
        }
        if ((lane & 3) == 0) {
            if (v0) *reinterpret_cast<float2*>(wml + row0 * 2) = make_float2(m0, l0);
            if (v1) *reinterpret_cast<float2*>(wml + row1 * 2) = make_float2(m1, l1);
        }
    }
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

int attn_warps(int n, int G) { return n * G >= 128 ? 8 : 4; }

int attn_splits(int B, int n, int Hq, int Hkv, int Lmax) {
    const int G = Hq / Hkv;
    const int nw = attn_warps(n, G);
    const int rb = (n * G + 16 * nw - 1) / (16 * nw);
    const int64_t ctas = (int64_t)B * Hkv * rb;
    const int target = 2 * device_sm_count();
    int splits = (int)((target + ctas - 1) / ctas);
    const int max_by_len = (Lmax - n) / (4 * kKeyTile);   // at least 4 tiles per split
    splits = splits < max_by_len ? splits : max_by_len;
    splits = splits < kMaxSplits ? splits : kMaxSplits;
    return splits < 1 ? 1 : splits;
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

bool use_mma_sync_kernel() {
    static int v = -1;
    if (v < 0) {
        const char* e = std::getenv("EAGLE_ATTN_MMA_SYNC");
        v = (e && e[0] == '1') ? 1 : 0;
    }
    return v == 1;
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
    const int s1 = attn_splits(B, n, Hq, Hkv, Lmax), s2 = tc_splits(B, n, Hq, Hkv, Lmax);
    const int splits = s1 > s2 ? s1 : s2;
    if (splits == 1) return 0;
    return (size_t)splits * B * n * Hq * (kHeadDim + 2) * sizeof(float);
}

extern "C" eagle_status eagle_tree_attn(const void* q, const void* k_cache, const void* v_cache,
                                        const int32_t* kv_len, const int32_t* parent, void* out,
                                        int B, int n, int Hq, int Hkv, int head_dim, int Lmax,
                                        float scale, void* workspace, size_t ws_bytes,
                                        int32_t* dev_status, eagle_stream_t stream) {
    if (!q || !k_cache || !v_cache || !kv_len || !parent || !out) return EAGLE_ERR_INVALID_ARG;
    if (B < 0 || n < 1 || Hq < 1 || Hkv < 1 || Lmax < 1 || !(scale > 0.f)) return EAGLE_ERR_INVALID_ARG;
    if (n > kMaxNodes || head_dim != kHeadDim || Hq % Hkv != 0 || Lmax < n) return EAGLE_ERR_SHAPE;
    for (const void* p : {q, k_cache, v_cache, (const void*)out})
        if (reinterpret_cast<uintptr_t>(p) & 15) return EAGLE_ERR_INVALID_ARG;
    if (B == 0) return EAGLE_OK;
    const bool v1 = use_mma_sync_kernel();
    const int splits = v1 ? attn_splits(B, n, Hq, Hkv, Lmax) : tc_splits(B, n, Hq, Hkv, Lmax);
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
    if (!v1) {
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
    } else {
        const int nw = attn_warps(n, G);
        const int rb = (n * G + 16 * nw - 1) / (16 * nw);
        const size_t smem = 2 * 2 * kTileBytes;
        dim3 grid((unsigned)rb, (unsigned)(Hkv * splits), (unsigned)B);
        if (nw == 8) {
            if (cudaFuncSetAttribute(tree_attn_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
                return EAGLE_ERR_CUDA;
            tree_attn_kernel<8><<<grid, 256, smem, s>>>(a);
        } else {
            if (cudaFuncSetAttribute(tree_attn_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
                return EAGLE_ERR_CUDA;
            tree_attn_kernel<4><<<grid, 128, smem, s>>>(a);
        }
    }
    EAGLE_CHECK_LAUNCH();
    if (splits > 1) {
        tree_attn_combine_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(a, rows);
        EAGLE_CHECK_LAUNCH();
    }
    return EAGLE_OK;
}
