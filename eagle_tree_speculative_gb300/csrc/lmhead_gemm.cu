// Draft LM head on the 5th-generation tensor cores: logits = hidden . W^T.
//
// Method (Guide "EAGLE-1/2/3 拆解", section on EAGLE-3's code changes: the draft
// head carries its own lm_head = Linear(hidden, draft_vocab, bias=False); the
// EAGLE-2 section: every expansion level runs the draft forward, and so this
// projection, on the k frontier nodes).
//
// sm_103a design: a persistent, warp-specialised kernel, one CTA per SM.
//   warp 0      one thread issues TMA loads (128B-swizzled 128x64 A and 256x64 B
//               tiles) into a 4-stage shared-memory ring guarded by mbarriers;
//   warp 1      allocates 512 TMEM columns and one thread issues
//               tcgen05.mma.cta_group::1.kind::f16 (M=128, N=256, K=16, bf16 in,
//               fp32 accumulate in TMEM), releasing each stage with
//               tcgen05.commit; accumulators are double-buffered in TMEM so the
//               epilogue of one tile overlaps the main loop of the next;
//   warps 2-5   the epilogue: tcgen05.ld 32x32b from their TMEM lane quadrant,
//               fp32 stores to the (possibly row-strided) output; optionally each
//               thread also reduces its row of the 256-column tile to a partial
//               softmax statistic (max, sum of 2^((l - max) log2 e)), from which
//               the expansion finds a row's top-k by rescanning only the few
//               tiles whose maximum can hold one.
// Tiles are visited M-fastest so the CTAs working on one 256-column slab of W
// run together and share it through L2: W is read from HBM about once.
// Every mbarrier wait is bounded (about two seconds); on expiry the kernel sets
// EAGLE_DEV_TIMEOUT, stops issuing work, drains its MMAs and frees TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "tc_common.cuh"

namespace eagle {
namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;            // 16 KB
constexpr int B_BYTES = BN * BK * 2;            // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // 48 KB
constexpr uint32_t TMEM_COLS = 2 * BN;          // two fp32 accumulators
constexpr int kThreads = 192;

// Instruction descriptor: M = 128, N = 256, bf16 A and B both K-major, fp32 D.
constexpr uint32_t kIdesc = idesc_bf16(BM, BN, 0, 0);

struct GemmArgs {
    float* out;
    int M, N, K;
    int64_t ldo;
    int rows_per_group;
    int64_t group_stride, row_offset;
    int32_t* dev_status;
    float* part;     // optional: per (row, N-tile) (max, sum) of the tile's columns
};

constexpr float kLog2eG = 1.4426950408889634f;

__device__ __forceinline__ float ex2_fast_g(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

__global__ void __launch_bounds__(kThreads, 1)
lmhead_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                   const __grid_constant__ CUtensorMap tmap_b, GemmArgs g) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * A_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sB + STAGES * B_BYTES);
    uint64_t* full = bars;                 // TMA -> MMA
    uint64_t* empty = bars + STAGES;       // MMA -> TMA
    uint64_t* tfull = bars + 2 * STAGES;   // MMA -> epilogue (2 accumulators)
    uint64_t* tempty = tfull + 2;          // epilogue -> MMA
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int num_m = (g.M + BM - 1) / BM, num_n = (g.N + BN - 1) / BN;
    const int num_tiles = num_m * num_n, num_k = g.K / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(s32(&full[s]), 1);
            mbar_init(s32(&empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(s32(&tfull[a]), 1);
            mbar_init(s32(&tempty[a]), 4);   // one arrival per epilogue warp
        }
        mbar_init(s32(drain), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
        asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&tmap_a)) : "memory");
        asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&tmap_b)) : "memory");
    }
    if (warp == 1) {
        tmem_alloc(s32(tmem_slot), TMEM_COLS);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            int stage = 0;
            uint32_t phase = 0;
            for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
                const int m0 = (t % num_m) * BM, n0 = (t / num_m) * BN;
                for (int kb = 0; kb < num_k; ++kb) {
                    if (!mbar_wait(s32(&empty[stage]), phase ^ 1u, abort_flag)) goto producer_done;
                    const uint32_t fb = s32(&full[stage]);
                    mbar_expect_tx(fb, STAGE_BYTES);
                    tma_load_2d(s32(sA + stage * A_BYTES), &tmap_a, fb, kb * BK, m0);
                    tma_load_2d(s32(sB + stage * B_BYTES), &tmap_b, fb, kb * BK, n0);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
        producer_done:;
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
                if (!mbar_wait(s32(&tempty[acc]), acc_phase ^ 1u, abort_flag)) break;
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(acc * BN);
                bool ok = true;
                for (int kb = 0; kb < num_k; ++kb) {
                    if (!mbar_wait(s32(&full[stage]), phase, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a0 = s32(sA + stage * A_BYTES), b0 = s32(sB + stage * B_BYTES);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)
                        umma_f16(d, sw128_desc(a0 + k * 32), sw128_desc(b0 + k * 32), kIdesc,
                                  (kb | k) != 0 ? 1u : 0u);
                    umma_commit(s32(&empty[stage]));
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                umma_commit(s32(&tfull[acc]));
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            }
            // drain: every MMA issued above has completed once this arrives
            umma_commit(s32(drain));
            mbar_wait(s32(drain), 0u, abort_flag, /*honour_abort=*/false);
        }
    } else {
        // ---------------- epilogue (warps 2..5) ----------------
        const int q = warp & 3;                 // TMEM lane quadrant of this warp
        const int r_in_tile = q * 32 + lane;
        int acc = 0;
        uint32_t acc_phase = 0;
        const bool vec = (g.ldo & 3) == 0 && (reinterpret_cast<uintptr_t>(g.out) & 15) == 0;
        for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
            const bool got = mbar_wait(s32(&tfull[acc]), acc_phase, abort_flag);
            if (!__all_sync(0xffffffffu, got)) break;   // the warp stays converged for tcgen05.ld
            tc_fence_after();
            const int m0 = (t % num_m) * BM, n0 = (t / num_m) * BN;
            const int m = m0 + r_in_tile;
            const bool valid = m < g.M;
            float* orow = g.out;
            if (valid) {
                const int64_t grp = m / g.rows_per_group, within = m % g.rows_per_group;
                orow = g.out + (grp * g.group_stride + g.row_offset + within) * g.ldo;
            }
            // optional partial statistics of this row over the tile's columns
            float pm = -INFINITY, ps = 0.f;
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN + c * 32), r);
                const int col = n0 + c * 32;
                if (g.part && valid) {
                    // online (max, sum of 2^((l - max) log2 e)) over the chunk's columns
                    const int nv = min(32, g.N - col);
                    float cmax = -INFINITY;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (j < nv) cmax = fmaxf(cmax, __uint_as_float(r[j]));
                    if (cmax > pm) {
                        ps = (pm == -INFINITY) ? 0.f : ps * ex2_fast_g((pm - cmax) * kLog2eG);
                        pm = cmax;
                    }
                    if (pm != -INFINITY) {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (j < nv) ps += ex2_fast_g((__uint_as_float(r[j]) - pm) * kLog2eG);
                    }
                }
                if (valid) {
                    if (vec && col + 32 <= g.N) {
#pragma unroll
                        for (int j = 0; j < 32; j += 4)
                            *reinterpret_cast<float4*>(orow + col + j) =
                                make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                                            __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (col + j < g.N) orow[col + j] = __uint_as_float(r[j]);
                    }
                }
            }
            if (g.part && valid)
                *reinterpret_cast<float2*>(g.part + ((int64_t)m * num_n + n0 / BN) * 2) =
                    make_float2(pm, ps);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s32(&tempty[acc]));
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
    }
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) flag_error(g.dev_status, EAGLE_DEV_TIMEOUT);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

bool make_map(CUtensorMap* map, const void* base, int rows, int K, int box_rows) {
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

eagle_status lmhead_gemm_launch(const void* hidden, const void* w, float* out, int M, int K, int N,
                                int64_t ldo, int rows_per_group, int64_t group_stride,
                                int64_t row_offset, int32_t* dev_status, cudaStream_t stream,
                                float* part) {
    if (M < 0 || N < 1 || K < BK || rows_per_group < 1 || ldo < N || group_stride < 0 ||
        row_offset < 0)
        return EAGLE_ERR_INVALID_ARG;
    if (K % BK != 0) return EAGLE_ERR_SHAPE;
    if (M == 0) return EAGLE_OK;                        // nothing read or written
    if (!hidden || !w || !out) return EAGLE_ERR_INVALID_ARG;
    if (part && (reinterpret_cast<uintptr_t>(part) & 7)) return EAGLE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(hidden) & 15) || (reinterpret_cast<uintptr_t>(w) & 15) ||
        (reinterpret_cast<uintptr_t>(out) & 3))
        return EAGLE_ERR_INVALID_ARG;
    CUtensorMap ma, mb;
    if (!make_map(&ma, hidden, M, K, BM) || !make_map(&mb, w, N, K, BN)) return EAGLE_ERR_CUDA;
    GemmArgs g{out, M, N, K, ldo, rows_per_group, group_stride, row_offset, dev_status, part};
    const int tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    const int sms = device_sm_count();
    const int grid = tiles < sms ? tiles : sms;
    const size_t smem = (size_t)STAGES * STAGE_BYTES + 1024 + 256;
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [&] {
        attr_err = cudaFuncSetAttribute(lmhead_gemm_kernel,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    });
    if (attr_err != cudaSuccess) return EAGLE_ERR_CUDA;
    lmhead_gemm_kernel<<<grid, kThreads, smem, stream>>>(ma, mb, g);
    EAGLE_CHECK_LAUNCH();
    return EAGLE_OK;
}

}  // namespace eagle

extern "C" eagle_status eagle_lmhead_gemm(const void* hidden, const void* w, float* out, int M,
                                          int K, int N, int64_t ldo, int rows_per_group,
                                          int64_t group_stride, int64_t row_offset, float* partials,
                                          int32_t* dev_status, eagle_stream_t stream) {
    return eagle::lmhead_gemm_launch(hidden, w, out, M, K, N, ldo, rows_per_group, group_stride,
                                     row_offset, dev_status, reinterpret_cast<cudaStream_t>(stream),
                                     partials);
}

extern "C" const char* eagle_status_str(eagle_status s) {
    switch (s) {
        case EAGLE_OK: return "EAGLE_OK";
        case EAGLE_ERR_INVALID_ARG: return "EAGLE_ERR_INVALID_ARG";
        case EAGLE_ERR_SHAPE: return "EAGLE_ERR_SHAPE";
        case EAGLE_ERR_CAPACITY: return "EAGLE_ERR_CAPACITY";
        case EAGLE_ERR_CUDA: return "EAGLE_ERR_CUDA";
        case EAGLE_ERR_DEVICE_DATA: return "EAGLE_ERR_DEVICE_DATA";
        case EAGLE_ERR_TIMEOUT: return "EAGLE_ERR_TIMEOUT";
    }
    return "EAGLE_ERR_UNKNOWN";
}

extern "C" int eagle_abi_version(void) { return 100; }

// ---------------------------------------------------------------------------
// Self-test of the bounded-wait path: one thread waits on an mbarrier that no
// one completes, the same polling loop as the pipelines' waits but with the
// caller's limit, then reports EAGLE_DEV_TIMEOUT and returns.
namespace eagle {
namespace {

__global__ void wait_selftest_kernel(int32_t* dev_status, long long max_cycles) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(s32(&bar), 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    const long long t0 = clock64();
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(s32(&bar), 0u)) return;            // never: no arrival
        if ((it & 127u) == 127u && clock64() - t0 > max_cycles) break;
    }
    flag_error(dev_status, EAGLE_DEV_TIMEOUT);
}

}  // namespace
}  // namespace eagle

extern "C" eagle_status eagle_wait_selftest(int32_t* dev_status, int64_t max_cycles,
                                            eagle_stream_t stream) {
    if (!dev_status || max_cycles < 1 || max_cycles > eagle::kTimeoutCycles) return EAGLE_ERR_INVALID_ARG;
    eagle::wait_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        dev_status, (long long)max_cycles);
    EAGLE_CHECK_LAUNCH();
    return EAGLE_OK;
}
