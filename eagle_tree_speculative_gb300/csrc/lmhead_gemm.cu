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
//               fp32 stores to the (possibly row-strided) output.
// Tiles are visited M-fastest so the CTAs working on one 256-column slab of W
// run together and share it through L2: W is read from HBM about once.
// Every mbarrier wait is bounded (about two seconds); on expiry the kernel sets
// EAGLE_DEV_TIMEOUT, stops issuing work, drains its MMAs and frees TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace eagle {
namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;            // 16 KB
constexpr int B_BYTES = BN * BK * 2;            // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // 48 KB
constexpr uint32_t TMEM_COLS = 2 * BN;          // two fp32 accumulators
constexpr int kThreads = 192;
constexpr long long kTimeoutCycles = 4000000000LL;

// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A bf16 (7-9 = 1),
// B bf16 (10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 at 17-22,
// M >> 4 at 24-28.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                            ((uint32_t)(BM >> 4) << 24);

struct GemmArgs {
    float* out;
    int M, N, K;
    int64_t ldo;
    int rows_per_group;
    int64_t group_stride, row_offset;
    int32_t* dev_status;
};

__device__ __forceinline__ uint32_t s32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------- mbarrier ----------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ uint32_t mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok;
}
// Bounded wait.  Returns false when the shared abort flag is up or the wait
// exceeded the limit (which raises the flag).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          bool honour_abort = true) {
    const long long t0 = clock64();
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 127u) == 127u) {
            if (honour_abort && *abort_flag) return false;
            if (clock64() - t0 > kTimeoutCycles) {
                *abort_flag = 1;
                return false;
            }
        }
    }
}

// ---------------- TMA ----------------
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
        "%4}], [%2];\n" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}

// ---------------- tcgen05 ----------------
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
                 : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
        "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}

// Shared-memory matrix descriptor, K-major, 128-byte swizzle: start address
// >> 4 (bits 0-13), leading offset 16 B (unused for this layout, bits 16-29),
// stride between 8-row groups 1024 B (bits 32-45), descriptor version 1
// (bits 46-47), layout SWIZZLE_128B = 2 (bits 61-63).  Stepping K by 16 bf16
// inside the 128-byte row adds 32 bytes to the start address.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
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
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                         s32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
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
                        umma_bf16(d, sw128_desc(a0 + k * 32), sw128_desc(b0 + k * 32),
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
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN + c * 32), r);
                const int col = n0 + c * 32;
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
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem_base),
                     "r"(TMEM_COLS)
                     : "memory");
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool make_map(CUtensorMap* map, const void* base, int rows, int K, int box_rows) {
    auto fn = encode_fn();
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
                                int64_t row_offset, int32_t* dev_status, cudaStream_t stream) {
    if (!hidden || !w || !out || M < 1 || N < 1 || K < BK || rows_per_group < 1 || ldo < N ||
        group_stride < 0 || row_offset < 0)
        return EAGLE_ERR_INVALID_ARG;
    if (K % BK != 0) return EAGLE_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(hidden) & 15) || (reinterpret_cast<uintptr_t>(w) & 15) ||
        (reinterpret_cast<uintptr_t>(out) & 3))
        return EAGLE_ERR_INVALID_ARG;
    CUtensorMap ma, mb;
    if (!make_map(&ma, hidden, M, K, BM) || !make_map(&mb, w, N, K, BN)) return EAGLE_ERR_CUDA;
    GemmArgs g{out, M, N, K, ldo, rows_per_group, group_stride, row_offset, dev_status};
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
                                          int64_t group_stride, int64_t row_offset,
                                          int32_t* dev_status, eagle_stream_t stream) {
    return eagle::lmhead_gemm_launch(hidden, w, out, M, K, N, ldo, rows_per_group, group_stride,
                                     row_offset, dev_status, reinterpret_cast<cudaStream_t>(stream));
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
