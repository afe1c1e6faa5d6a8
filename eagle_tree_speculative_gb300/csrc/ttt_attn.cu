// Training-time-test attention: host entry point (the kernel and its method are
// described in ttt_attn_tc.cuh).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"
#include "ttt_attn_tc.cuh"

namespace eagle {
namespace {

// Round 0 of K or V viewed as a 3-D tensor: head_dim (128, innermost), S positions,
// then the B * Hkv (sequence, kv head) slabs, R1 * S rows apart; 64 x 128 x 1 boxes.
// Positions from S on read as zeros.
bool ttt_map(CUtensorMap* map, const void* base, int S, int R1, int64_t slabs) {
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)S, (cuuint64_t)slabs};
    cuuint64_t strides[2] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)R1 * S * kHeadDim * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)ttt_tc::TBN, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Rounds 0 .. nrounds - 1 of K or V as a 4-D tensor (128 dims, S positions, rounds,
// slabs; the slabs R1 rounds apart); boxes of 64 dims x PB positions x RB rounds, PB * RB
// = 128 rows (the diagonal rows of one row tile).  Rounds from nrounds on and positions
// from S on read as zeros.
bool ttt_diag_map(CUtensorMap* map, const void* base, int S, int R1, int nrounds, int64_t slabs,
                  int PB, int RB) {
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    cuuint64_t dims[4] = {(cuuint64_t)kHeadDim, (cuuint64_t)S, (cuuint64_t)nrounds, (cuuint64_t)slabs};
    cuuint64_t strides[3] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)S * kHeadDim * 2,
                             (cuuint64_t)R1 * S * kHeadDim * 2};
    cuuint32_t box[4] = {64, (cuuint32_t)PB, (cuuint32_t)RB, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace eagle

using namespace eagle;

extern "C" eagle_status eagle_ttt_attn(const void* q, const void* k, const void* v, void* out,
                                       int B, int S, int Hq, int Hkv, int head_dim, int R1, int r,
                                       float scale, int32_t* dev_status, eagle_stream_t stream) {
    if (B < 0 || S < 1 || Hq < 1 || Hkv < 1 || R1 < 1 || r < 0 || r >= R1 || !(scale > 0.f))
        return EAGLE_ERR_INVALID_ARG;
    if (head_dim != kHeadDim || Hq % Hkv != 0 || R1 > ttt_tc::kMaxRounds) return EAGLE_ERR_SHAPE;
    if (B == 0) return EAGLE_OK;                        // nothing read or written
    if (!q || !k || !v || !out) return EAGLE_ERR_INVALID_ARG;
    for (const void* p : {q, k, v, (const void*)out})
        if (reinterpret_cast<uintptr_t>(p) & 15) return EAGLE_ERR_INVALID_ARG;
    const int G = Hq / Hkv;
    const int64_t slabs = (int64_t)B * Hkv;
    const int64_t tiles = ((int64_t)S * G + ttt_tc::ROWS_PER_CTA - 1) / ttt_tc::ROWS_PER_CTA;
    if (slabs * tiles > 0x7fffffffLL || (int64_t)S * G > 0x7fffffffLL ||
        (int64_t)R1 * S > 0x7fffffffLL)
        return EAGLE_ERR_SHAPE;
    // A row tile of 128 rows spans at most 127 / G + 1 positions, one more when G
    // does not divide 128.  A diagonal box holds RB rounds (a power of two) of PB =
    // 128 / RB >= that many positions: exactly the 128 rows of a ring stage, so every row
    // the MMAs read was written by the box.  Rounds above r read as zeros.
    const int span = 127 / G + 1 + (128 % G != 0 ? 1 : 0);
    int RB = 1;
    while (2 * RB * span <= 128) RB *= 2;
    const int PB = 128 / RB;
    const int ND = (r + RB - 1) / RB;
    CUtensorMap mk, mv, mkd, mvd;
    if (!ttt_map(&mk, k, S, R1, slabs) || !ttt_map(&mv, v, S, R1, slabs) ||
        !ttt_diag_map(&mkd, k, S, R1, r + 1, slabs, PB, RB) ||
        !ttt_diag_map(&mvd, v, S, R1, r + 1, slabs, PB, RB))
        return EAGLE_ERR_CUDA;
    ttt_tc::Args a;
    a.q = static_cast<const uint16_t*>(q);
    a.out = static_cast<uint16_t*>(out);
    a.B = B; a.S = S; a.Hq = Hq; a.Hkv = Hkv; a.G = G; a.R1 = R1; a.r = r;
    a.PB = PB; a.RB = RB; a.ND = ND;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.dev_status = dev_status;
    if (cudaFuncSetAttribute(ttt_tc::ttt_attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             ttt_tc::SMEM_BYTES) != cudaSuccess)
        return EAGLE_ERR_CUDA;
    a.tiles = (int)tiles;
    // slab-major: the row tiles of one (sequence, kv head) run together, so only a few
    // slabs' round-0 K/V are live in L2 at a time while the diagonal rows stream past
    dim3 grid((unsigned)(slabs * tiles), 1, 1);
    ttt_tc::ttt_attn_tc_kernel<<<grid, ttt_tc::kThreads, ttt_tc::SMEM_BYTES,
                                 reinterpret_cast<cudaStream_t>(stream)>>>(mk, mv, mkd, mvd, a);
    return cudaGetLastError() == cudaSuccess ? EAGLE_OK : EAGLE_ERR_CUDA;
}
