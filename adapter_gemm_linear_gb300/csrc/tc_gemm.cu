// Base GEMM on the 5th-generation tensor cores (tcgen05, accumulator in
// TMEM, operands staged by TMA) with the LoRA expand fused into the
// epilogue:
//
//   out[m, n] = round( sum_k x[m,k] W[n,k]  +  s_i * sum_j Bt_i[j,n] V[m,j] )
//
// where i is row m's adapter slot (none: no second term), V = A_i x is the
// rank-r intermediate (fp32, produced by the shrink kernel), Bt_i are the
// adapter's B^T rank-rows gathered through the pool's block table, and
// s_i = alpha_i / r_i.  The correction is added to the fp32 accumulator, so
// each output is rounded to bf16 exactly once.
//
// One CTA computes one 128 x BN output tile.  Warp roles:
//   warp 0      TMA producer: x tile [128 x 64] and W tile [BN x 64] per
//               k-block into a STAGES-deep shared-memory ring (128-byte
//               swizzle), completion counted on the stage's `full` barrier;
//   warp 1      TMEM allocator and MMA issuer: 4 tcgen05.mma (K = 16 each)
//               per k-block into a 128 x BN fp32 TMEM accumulator, then
//               tcgen05.commit frees the stage (`empty` barrier);
//   warps 2-5   epilogue: each warp owns one 32-lane quarter of TMEM (= 32
//               output rows), reads 32 columns at a time with tcgen05.ld,
//               adds the row's LoRA correction and stores bf16.
// Every barrier wait is bounded in time; a wait that runs out records
// kDevTimeout in the status word and the CTA unwinds without hanging.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <mutex>

#include "lora_device.cuh"
#include "lora_internal.h"
#include "sm100_ptx.cuh"

namespace lora {

namespace {

constexpr int kBM = 128;               // tile rows (UMMA M)
constexpr int kBK = 64;                // k-block: 64 bf16 = one 128-byte swizzle row
constexpr int kUmmaK = 16;             // K of one tcgen05.mma for 16-bit inputs
constexpr int kThreads = 192;          // 6 warps
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far beyond any legitimate wait

struct TcParams {
    int32_t M, N, K, num_kb;
    __nv_bfloat16 *out;
    int32_t ldo;
    const int32_t *row_slot;
    const __nv_bfloat16 *bt_arena;
    const int32_t *table;
    const int32_t *ranks;
    const float *scales;
    int32_t max_slots, bps, num_blocks;
    const float *V;
    int32_t ldv;
    unsigned long long *status;
};

template <int BN>
__host__ __device__ constexpr uint32_t tmem_cols() {
    return BN <= 32 ? 32 : BN <= 64 ? 64 : BN <= 128 ? 128 : 256;
}

template <int BN, int STAGES>
constexpr size_t smem_bytes() {
    return 1024 /* alignment slack */ + static_cast<size_t>(STAGES) * (kBM + BN) * kBK * 2 +
           (2 * STAGES + 1) * 8 + 16;
}

__device__ __forceinline__ void unpack_bf16x8(const uint4 &q, float *v) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);  // a -> low half, b -> high half
    return *reinterpret_cast<const uint32_t *>(&h);
}

template <int BN, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
tc_gemm_lora_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmw,
                    const TcParams p) {
    using namespace sm100;
    constexpr uint32_t kABytes = kBM * kBK * 2;
    constexpr uint32_t kBBytes = BN * kBK * 2;
    constexpr uint32_t kCols = tmem_cols<BN>();

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + STAGES * kABytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(sB + STAGES * kBBytes);
    uint64_t *empty = full + STAGES;
    uint64_t *tmem_full = empty + STAGES;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tmem_full + 1);
    volatile uint32_t *abort_flag = tmem_slot + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int32_t m0 = blockIdx.x * kBM;
    const int32_t n0 = blockIdx.y * BN;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(tmem_full, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmx);
        prefetch_tensormap(&tmw);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            for (int32_t kb = 0; kb < p.num_kb; ++kb) {
                const int s = kb % STAGES;
                const uint32_t ph = (kb / STAGES) & 1;
                if (!mbar_wait_bounded(&empty[s], ph ^ 1, kWaitLimitNs)) {
                    record_error(p.status, kDevTimeout, 1);
                    *abort_flag = 1;
                    break;
                }
                if (*abort_flag) break;
                mbar_arrive_expect_tx(&full[s], kABytes + kBBytes);
                tma_load_2d(sA + s * kABytes, &tmx, kb * kBK, m0, &full[s]);
                tma_load_2d(sB + s * kBBytes, &tmw, kb * kBK, n0, &full[s]);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(kBM, BN);
            bool ok = true;
            for (int32_t kb = 0; kb < p.num_kb; ++kb) {
                const int s = kb % STAGES;
                const uint32_t ph = (kb / STAGES) & 1;
                if (!mbar_wait_bounded(&full[s], ph, kWaitLimitNs) || *abort_flag) {
                    if (!*abort_flag) record_error(p.status, kDevTimeout, 2);
                    *abort_flag = 1;
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t a_addr = smem_u32(sA + s * kABytes);
                const uint32_t b_addr = smem_u32(sB + s * kBBytes);
#pragma unroll
                for (int k = 0; k < kBK / kUmmaK; ++k) {
                    mma_bf16_f32(tmem_base, desc_kmajor_sw128(a_addr + k * kUmmaK * 2),
                                 desc_kmajor_sw128(b_addr + k * kUmmaK * 2), idesc,
                                 (kb > 0 || k > 0) ? 1u : 0u);
                }
                mma_commit(&empty[s]);
            }
            if (ok)
                mma_commit(tmem_full);
            else
                mbar_arrive(tmem_full);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int32_t m = m0 + q * 32 + lane;
        bool ok = mbar_wait_bounded(tmem_full, 0, kWaitLimitNs);
        if (!ok) record_error(p.status, kDevTimeout, 3);
        ok = __all_sync(0xffffffffu, ok && !*abort_flag);
        tc_fence_after_sync();
        if (ok) {
            int32_t r = 0;
            float s = 0.0f;
            int32_t slot = -1;
            if (m < p.M)
                slot = resolve_slot(p.row_slot[m], m, p.ranks, p.scales, p.max_slots, p.bps, &r, &s,
                                    p.status, false);
            const float *vrow = p.V + static_cast<size_t>(m < p.M ? m : 0) * p.ldv;
            const int32_t *trow = p.table + static_cast<size_t>(slot < 0 ? 0 : slot) * p.bps;
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t raw[32];
                tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + c * 32, raw);
                tmem_ld_wait(raw);
                float acc[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) acc[e] = __uint_as_float(raw[e]);
                const int32_t nc = n0 + c * 32;
                if (slot >= 0 && nc < p.N) {
                    float lo[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) lo[e] = 0.0f;
                    bool bad = false;
#pragma unroll 1
                    for (int32_t jb = 0; jb * LORA_BLOCK_ROWS < r; ++jb) {
                        const int32_t b = trow[jb];
                        if (b < 0 || b >= p.num_blocks) {
                            record_error(p.status, kDevBadBlock, static_cast<uint32_t>(slot));
                            bad = true;
                            break;
                        }
                        const int32_t jn = min(LORA_BLOCK_ROWS, r - jb * LORA_BLOCK_ROWS);
                        const __nv_bfloat16 *bt =
                            p.bt_arena + static_cast<size_t>(b) * LORA_BLOCK_ROWS * p.N + nc;
#pragma unroll 1
                        for (int32_t jj = 0; jj < jn; ++jj) {
                            const float v = vrow[jb * LORA_BLOCK_ROWS + jj];
                            const uint4 *src = reinterpret_cast<const uint4 *>(bt + static_cast<size_t>(jj) * p.N);
#pragma unroll
                            for (int g = 0; g < 4; ++g) {
                                if (nc + g * 8 < p.N) {
                                    float bv[8];
                                    unpack_bf16x8(__ldg(src + g), bv);
#pragma unroll
                                    for (int e = 0; e < 8; ++e) lo[g * 8 + e] = fmaf(bv[e], v, lo[g * 8 + e]);
                                }
                            }
                        }
                    }
                    if (!bad) {
#pragma unroll
                        for (int e = 0; e < 32; ++e) acc[e] = fmaf(s, lo[e], acc[e]);
                    }
                }
                if (m < p.M) {
                    __nv_bfloat16 *dst = p.out + static_cast<size_t>(m) * p.ldo + nc;
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        if (nc + g * 8 < p.N) {
                            uint4 w;
                            w.x = pack_bf16x2(acc[g * 8 + 0], acc[g * 8 + 1]);
                            w.y = pack_bf16x2(acc[g * 8 + 2], acc[g * 8 + 3]);
                            w.z = pack_bf16x2(acc[g * 8 + 4], acc[g * 8 + 5]);
                            w.w = pack_bf16x2(acc[g * 8 + 6], acc[g * 8 + 7]);
                            *reinterpret_cast<uint4 *>(dst + g * 8) = w;
                        }
                    }
                }
                __syncwarp();
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, kCols);
    }
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Row-major bf16 matrix [rows][cols] with row stride `ld` elements, tiled in
// boxes of box_rows x 64 with the 128-byte swizzle; out-of-range elements of
// a box read as zero.
bool make_tmap_bf16(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols, uint64_t ld,
                    uint32_t box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {ld * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
    static int cache[128] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 148;
    if (!cache[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cache[dev] = n > 0 ? n : 148;
    }
    return cache[dev];
}

template <int BN, int STAGES>
cudaError_t launch_tile(const ForwardPlan &plan, const ProjView &v, cudaStream_t stream) {
    auto kernel = tc_gemm_lora_kernel<BN, STAGES>;
    constexpr size_t smem = smem_bytes<BN, STAGES>();
    // the shared-memory opt-in is a per-device function attribute
    static std::mutex mu;
    static bool done[128] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!done[dev]) {
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(smem));
            if (e != cudaSuccess) return e;
            done[dev] = true;
        }
    }
    CUtensorMap tmx, tmw;
    if (!make_tmap_bf16(&tmx, plan.x, plan.M, plan.K, plan.ldx, kBM)) return cudaErrorInvalidValue;
    if (!make_tmap_bf16(&tmw, v.W, v.N, plan.K, plan.K, BN)) return cudaErrorInvalidValue;
    TcParams p;
    p.M = plan.M;
    p.N = v.N;
    p.K = plan.K;
    p.num_kb = (plan.K + kBK - 1) / kBK;
    p.out = static_cast<__nv_bfloat16 *>(v.out);
    p.ldo = v.ldo;
    p.row_slot = plan.row_slot;
    p.bt_arena = static_cast<const __nv_bfloat16 *>(v.bt_arena);
    p.table = v.table;
    p.ranks = v.ranks;
    p.scales = v.scales;
    p.max_slots = v.max_slots;
    p.bps = v.bps;
    p.num_blocks = v.num_blocks;
    p.V = v.V;
    p.ldv = v.max_rank;
    p.status = plan.status;
    dim3 grid((plan.M + kBM - 1) / kBM, (v.N + BN - 1) / BN);
    kernel<<<grid, kThreads, smem, stream>>>(tmx, tmw, p);
    return cudaGetLastError();
}

}  // namespace

// Tile width: fewest waves of CTAs over the SMs, weighting each tile by its
// width plus a fixed per-tile cost.
int choose_tc_bn(int32_t M, int32_t N) {
    const int sms = sm_count();
    const int mt = (M + kBM - 1) / kBM;
    int best = 256;
    long best_cost = -1;
    for (int bn : {256, 128, 64}) {
        const long tiles = static_cast<long>(mt) * ((N + bn - 1) / bn);
        const long waves = (tiles + sms - 1) / sms;
        const long cost = waves * (bn + 32);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = bn;
        }
    }
    return best;
}

cudaError_t launch_gemm_lora_tc(const ForwardPlan &plan, const ProjView &v, cudaStream_t stream) {
    switch (choose_tc_bn(plan.M, v.N)) {
        case 256: return launch_tile<256, 4>(plan, v, stream);
        case 128: return launch_tile<128, 6>(plan, v, stream);
        default: return launch_tile<64, 8>(plan, v, stream);
    }
}

}  // namespace lora
