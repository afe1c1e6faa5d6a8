// Shared device helpers of the sm_103a library: status plumbing, the Philox
// generator, reductions and small PTX wrappers.
#pragma once

#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "eagle.h"

namespace eagle {

namespace cg = cooperative_groups;

constexpr int kMaxNodes = 64;
constexpr int kHeadDim = 128;

#define EAGLE_CHECK_LAUNCH()                                   \
    do {                                                       \
        cudaError_t e_ = cudaGetLastError();                   \
        if (e_ != cudaSuccess) return EAGLE_ERR_CUDA;          \
    } while (0)

__device__ __forceinline__ void flag_error(int32_t* dev_status, int bits) {
    if (dev_status) atomicOr(dev_status, bits);
}

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11, section 4.2): ten rounds of
// two 32x32 multiplies whose high halves are XORed with the odd words and the
// round key; the key advances by the Weyl constants between rounds.
// Counter words: (lane block, node/position, sequence, stream tag).
// ---------------------------------------------------------------------------
enum : uint32_t { kTagAccept = 0u, kTagRace = 1u };

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t m0 = 0xD2511F53u, m1 = 0xCD9E8D57u;
        uint32_t h0 = __umulhi(m0, c.x), l0 = m0 * c.x;
        uint32_t h1 = __umulhi(m1, c.z), l1 = m1 * c.z;
        c = make_uint4(h1 ^ c.y ^ k0, l1, h0 ^ c.w ^ k1, l0);
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c;
}

// Uniform on the 2^-24 grid in [0, 1).
__device__ __forceinline__ float unit_closed_open(uint32_t w) {
    return (float)(w >> 8) * 0x1p-24f;
}

__device__ __forceinline__ float accept_uniform(uint64_t seed, uint32_t b, uint32_t node) {
    uint4 w = philox4x32_10(make_uint4(0u, node, b, kTagAccept), (uint32_t)seed,
                            (uint32_t)(seed >> 32));
    return unit_closed_open(w.x);
}

// ---------------------------------------------------------------------------
// Reductions.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Arg-max pair with a deterministic order: larger key first, lower index on ties.
struct KeyIdx {
    float k;
    int i;
};

__device__ __forceinline__ bool ki_better(KeyIdx a, KeyIdx b) {
    return a.k > b.k || (a.k == b.k && a.i < b.i);
}

__device__ __forceinline__ KeyIdx warp_argmax(KeyIdx v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        KeyIdx w{__shfl_xor_sync(0xffffffffu, v.k, o), __shfl_xor_sync(0xffffffffu, v.i, o)};
        if (ki_better(w, v)) v = w;
    }
    return v;
}

// ---------------------------------------------------------------------------
// Launch helper: grid of `clusters` clusters of `cs` CTAs.
// ---------------------------------------------------------------------------
template <typename Kernel, typename... Args>
cudaError_t launch_clustered(Kernel k, int clusters, int cs, int threads, size_t smem,
                             cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(clusters * cs), 1, 1);
    cfg.blockDim = dim3((unsigned)threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, args...);
}

inline int device_sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 148;
    return sms;
}

}  // namespace eagle
