// Device status word, row-map and pool-copy kernels, and the SIMT
// (CUDA-core) forward path used for fp32 inputs.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "lora_internal.h"
#include "lora_device.cuh"

namespace lora {

// ---------------------------------------------------------------------------
// per-device status word
// ---------------------------------------------------------------------------

__device__ unsigned long long g_lora_status;

namespace {
using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

template <typename F>
F driver_entry(const char *name) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<F>(p);
}
}  // namespace

uint64_t current_context_id() {
    static std::once_flag once;
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    std::call_once(once, [] {
        get_current = driver_entry<CtxGetCurrentFn>("cuCtxGetCurrent");
        get_id = driver_entry<CtxGetIdFn>("cuCtxGetId");
    });
    CUcontext ctx = nullptr;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    unsigned long long id = 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return static_cast<uint64_t>(id) + 1;  // 0 stays "unknown"
}

bool first_use_in_context(uint64_t *slot) {
    const uint64_t id = current_context_id();
    if (id != 0 && *slot == id) return false;
    *slot = id;
    return true;
}

cudaError_t device_status_ptr(unsigned long long **out) {
    static std::mutex mu;
    static unsigned long long *cache[128] = {};
    static uint64_t cache_ctx[128] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    const uint64_t ctx = current_context_id();
    if (!cache[dev] || ctx == 0 || cache_ctx[dev] != ctx) {
        // first use on this device, or its context was replaced (a device
        // reset): the symbol's address is the new context's
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_lora_status);
        if (e != cudaSuccess) return e;
        cache[dev] = static_cast<unsigned long long *>(p);
        cache_ctx[dev] = current_context_id();  // the lookup made the context current
    }
    *out = cache[dev];
    return cudaSuccess;
}

// ---------------------------------------------------------------------------
// segments -> per-row slot ids
// ---------------------------------------------------------------------------

__global__ void segments_to_rows_kernel(int32_t M, const int32_t *__restrict__ off,
                                        const int32_t *__restrict__ seg_adapter,
                                        const int32_t *__restrict__ perm, int32_t S,
                                        int32_t *__restrict__ row_slot,
                                        unsigned long long *status) {
    const int32_t p = blockIdx.x * blockDim.x + threadIdx.x;
    if (p <= S && p < S + 1) {
        // offsets must be non-decreasing within [0, M]
        const int32_t o = off[p];
        const bool bad = o < 0 || o > M || (p > 0 && off[p - 1] > o);
        if (bad) record_error(status, kDevBadSegment, static_cast<uint32_t>(p));
    }
    if (p >= M) return;
    // last segment s with off[s] <= p
    int32_t lo = 0, hi = S;  // search in [0, S]
    if (off[0] > p) return;
    while (lo < hi) {
        const int32_t mid = (lo + hi + 1) >> 1;
        if (off[mid] <= p) lo = mid; else hi = mid - 1;
    }
    const int32_t s = lo;
    if (s >= S || p >= off[s + 1]) return;
    const int32_t row = perm ? perm[p] : p;
    if (row < 0 || row >= M) {
        record_error(status, kDevBadSegment, static_cast<uint32_t>(p));
        return;
    }
    row_slot[row] = seg_adapter[s];
}

cudaError_t launch_segments_to_rows(int32_t M, const int32_t *seg_offsets,
                                    const int32_t *seg_adapter, const int32_t *perm,
                                    int32_t num_segs, int32_t *row_slot,
                                    unsigned long long *status, cudaStream_t stream) {
    const int32_t n = (M > num_segs + 1 ? M : num_segs + 1);
    const int threads = 256;
    segments_to_rows_kernel<<<(n + threads - 1) / threads, threads, 0, stream>>>(
        M, seg_offsets, seg_adapter, perm, num_segs, row_slot, status);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// device-to-device adapter load: A rows and transposed B into pool blocks
// ---------------------------------------------------------------------------

struct ScatterBlocks {
    int32_t b[kMaxBlocksPerSlot];
};

template <typename T>
__global__ void pool_scatter_kernel(const T *__restrict__ A, const T *__restrict__ B, int32_t rank,
                                    int32_t K, int32_t N, T *__restrict__ a_arena,
                                    T *__restrict__ b_arena, ScatterBlocks blocks) {
    const int32_t t = blockIdx.y;
    const int32_t row = blockIdx.z;
    const int32_t j = t * LORA_BLOCK_ROWS + row;
    const size_t b = static_cast<size_t>(blocks.b[t]);
    T *a_dst = a_arena + (b * LORA_BLOCK_ROWS + row) * static_cast<size_t>(K);
    T *b_dst = b_arena + b * static_cast<size_t>(N) * LORA_BLOCK_ROWS + row;
    const int32_t stride = gridDim.x * blockDim.x;
    for (int32_t k = blockIdx.x * blockDim.x + threadIdx.x; k < K; k += stride)
        a_dst[k] = j < rank ? A[static_cast<size_t>(j) * K + k] : from_float<T>(0.0f);
    for (int32_t n = blockIdx.x * blockDim.x + threadIdx.x; n < N; n += stride)
        b_dst[static_cast<size_t>(n) * LORA_BLOCK_ROWS] =
            j < rank ? B[static_cast<size_t>(n) * rank + j] : from_float<T>(0.0f);
}

// The same scatter in 16-byte vectors, for ranks whose B rows are whole
// vectors (rank * element size a multiple of 16): A's rows straight into the
// blocks (zero rows past the rank), and B read a row at a time -- consecutive
// threads take consecutive vectors of a row, so reads are coalesced (also
// over the host link, for page-locked host sources) -- each vector written to
// its block's [N][16] layout; the last block's columns past the rank zeroed.
template <typename T>
__global__ void __launch_bounds__(256)
pool_scatter_vec_kernel(const T *__restrict__ A, const T *__restrict__ B, int32_t rank, int32_t K, int32_t N,
                        T *__restrict__ a_arena, T *__restrict__ b_arena, ScatterBlocks blocks) {
    constexpr int kVec = 16 / sizeof(T);                   // elements per vector
    constexpr int kRowVecs = LORA_BLOCK_ROWS / kVec;       // vectors of a block row of B
    const int32_t nb = (rank + LORA_BLOCK_ROWS - 1) / LORA_BLOCK_ROWS;
    const int64_t kv = K / kVec;                           // vectors of an A row
    const int64_t a_work = static_cast<int64_t>(nb) * LORA_BLOCK_ROWS * kv;
    const int64_t b_row = static_cast<int64_t>(nb) * kRowVecs;  // destination vectors per B row
    const int64_t b_work = static_cast<int64_t>(N) * b_row;
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < a_work + b_work; i += stride) {
        if (i < a_work) {
            const int64_t jrow = i / kv, v = i - jrow * kv;  // block row jrow of the slot (j = jrow)
            const int32_t t = static_cast<int32_t>(jrow / LORA_BLOCK_ROWS), r = static_cast<int32_t>(jrow % LORA_BLOCK_ROWS);
            uint4 *dst = reinterpret_cast<uint4 *>(a_arena + (static_cast<size_t>(blocks.b[t]) * LORA_BLOCK_ROWS + r) * K) + v;
            *dst = jrow < rank ? reinterpret_cast<const uint4 *>(A + jrow * K)[v] : zero;
        } else {
            const int64_t w = i - a_work;
            const int64_t n = w / b_row, c = w - n * b_row;  // c: vector of the slot's (padded) rank
            const int32_t j0 = static_cast<int32_t>(c) * kVec;
            const int32_t t = j0 / LORA_BLOCK_ROWS, jj = j0 % LORA_BLOCK_ROWS;
            uint4 *dst = reinterpret_cast<uint4 *>(b_arena + (static_cast<size_t>(blocks.b[t]) * N + n) * LORA_BLOCK_ROWS + jj);
            *dst = j0 < rank ? *reinterpret_cast<const uint4 *>(B + n * rank + j0) : zero;
        }
    }
}

cudaError_t launch_pool_scatter(const lora_pool *pool, int32_t rank, const int32_t *blocks,
                                const void *A, const void *B, cudaStream_t stream) {
    const int nb = (rank + LORA_BLOCK_ROWS - 1) / LORA_BLOCK_ROWS;
    ScatterBlocks sb;
    for (int t = 0; t < kMaxBlocksPerSlot; ++t) sb.b[t] = t < nb ? blocks[t] : 0;
    count_launches(1);
    const lora_pool_desc_t &dd = pool->d;
    const size_t eb = dd.dtype == LORA_FP32 ? 4 : 2;
    if ((static_cast<size_t>(rank) * eb) % 16 == 0 && (static_cast<size_t>(dd.K) * eb) % 16 == 0) {
        const int64_t work = static_cast<int64_t>(nb) * LORA_BLOCK_ROWS * (dd.K * static_cast<int64_t>(eb) / 16) +
                             static_cast<int64_t>(dd.N) * nb * (LORA_BLOCK_ROWS * static_cast<int64_t>(eb) / 16);
        int64_t grid = (work + 255) / 256;
        const int64_t cap = 4L * device_sm_count();
        grid = grid < 1 ? 1 : grid > cap ? cap : grid;
        if (dd.dtype == LORA_FP32)
            pool_scatter_vec_kernel<float><<<static_cast<unsigned>(grid), 256, 0, stream>>>(
                static_cast<const float *>(A), static_cast<const float *>(B), rank, dd.K, dd.N,
                static_cast<float *>(dd.a_arena), static_cast<float *>(dd.b_arena), sb);
        else
            pool_scatter_vec_kernel<__nv_bfloat16><<<static_cast<unsigned>(grid), 256, 0, stream>>>(
                static_cast<const __nv_bfloat16 *>(A), static_cast<const __nv_bfloat16 *>(B), rank, dd.K, dd.N,
                static_cast<__nv_bfloat16 *>(dd.a_arena), static_cast<__nv_bfloat16 *>(dd.b_arena), sb);
        return cudaGetLastError();
    }
    dim3 grid(8, nb, LORA_BLOCK_ROWS);
    const lora_pool_desc_t &d = pool->d;
    if (d.dtype == LORA_FP32)
        pool_scatter_kernel<float><<<grid, 256, 0, stream>>>(
            static_cast<const float *>(A), static_cast<const float *>(B), rank, d.K, d.N,
            static_cast<float *>(d.a_arena), static_cast<float *>(d.b_arena), sb);
    else
        pool_scatter_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(
            static_cast<const __nv_bfloat16 *>(A), static_cast<const __nv_bfloat16 *>(B), rank,
            d.K, d.N, static_cast<__nv_bfloat16 *>(d.a_arena),
            static_cast<__nv_bfloat16 *>(d.b_arena), sb);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// SIMT shrink: V[m, 16t + j] = sum_k A_i[16t + j, k] x[m, k]
// grid (M, blocks per slot), 128 threads; each CTA one row x one 16-row block
// ---------------------------------------------------------------------------

template <typename T>
__global__ void __launch_bounds__(128)
shrink_simt_kernel(const T *__restrict__ x, int32_t ldx, int32_t K, const int32_t *__restrict__ row_slot,
                   const T *__restrict__ a_arena, const int32_t *__restrict__ table,
                   const int32_t *__restrict__ ranks, int32_t max_slots, int32_t bps,
                   int32_t num_blocks, float *__restrict__ V, int32_t ldv,
                   unsigned long long *status, int32_t *__restrict__ counters, int32_t n_counters) {
    const int32_t m = blockIdx.x;
    const int32_t t = blockIdx.y;
    // the GEMM that follows may launch now: it reads V and the counters only
    // after this grid has completed (griddepcontrol.wait)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // the split-K tile counters of the GEMM that follows start from zero
    if (m == 0 && t == 0)
        for (int32_t c = threadIdx.x; c < n_counters; c += blockDim.x) counters[c] = 0;
    int32_t r;
    float s;
    const int32_t i = resolve_slot(row_slot[m], m, ranks, nullptr, max_slots, bps, &r, &s, status,
                                   t == 0 && threadIdx.x == 0);
    if (i < 0 || t * LORA_BLOCK_ROWS >= r) return;
    const int32_t b = table[i * bps + t];
    if (b < 0 || b >= num_blocks) {
        if (threadIdx.x == 0) record_error(status, kDevBadBlock, static_cast<uint32_t>(i));
        return;
    }
    constexpr int VE = VecTraits<T>::kElems;
    const T *A = a_arena + static_cast<size_t>(b) * LORA_BLOCK_ROWS * K;
    const T *xr = x + static_cast<size_t>(m) * ldx;
    float acc[LORA_BLOCK_ROWS];
#pragma unroll
    for (int j = 0; j < LORA_BLOCK_ROWS; ++j) acc[j] = 0.0f;
    for (int32_t k = threadIdx.x * VE; k < K; k += blockDim.x * VE) {
        float xv[VE];
        VecTraits<T>::load(xr + k, xv);
#pragma unroll
        for (int j = 0; j < LORA_BLOCK_ROWS; ++j) {
            float av[VE];
            VecTraits<T>::load(A + static_cast<size_t>(j) * K + k, av);
#pragma unroll
            for (int e = 0; e < VE; ++e) acc[j] = fmaf(av[e], xv[e], acc[j]);
        }
    }
    __shared__ float red[4][LORA_BLOCK_ROWS];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int j = 0; j < LORA_BLOCK_ROWS; ++j) {
        float v = acc[j];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) red[warp][j] = v;
    }
    __syncthreads();
    if (threadIdx.x < LORA_BLOCK_ROWS) {
        const float v = red[0][threadIdx.x] + red[1][threadIdx.x] + red[2][threadIdx.x] +
                        red[3][threadIdx.x];
        V[static_cast<size_t>(m) * ldv + t * LORA_BLOCK_ROWS + threadIdx.x] = v;
    }
}

// ---------------------------------------------------------------------------
// SIMT GEMM with the expand fused into the epilogue:
// out[m, n] = sum_k x[m,k] W[n,k] + s_i * sum_j B_i[n, j] V[m, j]
// 64x64 tile, 256 threads, 4x4 outputs per thread (rows ty+16a, cols tx+16b)
// ---------------------------------------------------------------------------

template <typename T>
__global__ void __launch_bounds__(256)
gemm_lora_simt_kernel(const T *__restrict__ x, int32_t ldx, const T *__restrict__ W, int32_t M,
                      int32_t N, int32_t K, T *__restrict__ out, int32_t ldo,
                      const int32_t *__restrict__ row_slot, const T *__restrict__ b_arena,
                      const int32_t *__restrict__ table, const int32_t *__restrict__ ranks,
                      const float *__restrict__ scales, int32_t max_slots, int32_t bps,
                      int32_t num_blocks, const float *__restrict__ V, int32_t ldv,
                      unsigned long long *status) {
    constexpr int BM = 64, BN = 64, BK = 16;
    __shared__ float xs[BK][BM + 4];
    __shared__ float wsm[BK][BN + 4];
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int32_t m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
    float acc[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[a][c] = 0.0f;

    const int lr = threadIdx.x >> 2;        // 0..63: tile row loaded by this thread
    const int lk = (threadIdx.x & 3) * 4;   // 0,4,8,12: first k of its 4
    for (int32_t k0 = 0; k0 < K; k0 += BK) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int32_t k = k0 + lk + e;
            const int32_t m = m0 + lr, n = n0 + lr;
            xs[lk + e][lr] = (m < M && k < K) ? to_float(x[static_cast<size_t>(m) * ldx + k]) : 0.0f;
            wsm[lk + e][lr] = (n < N && k < K) ? to_float(W[static_cast<size_t>(n) * K + k]) : 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            float av[4], bv[4];
#pragma unroll
            for (int a = 0; a < 4; ++a) av[a] = xs[kk][ty + 16 * a];
#pragma unroll
            for (int c = 0; c < 4; ++c) bv[c] = wsm[kk][tx + 16 * c];
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[a][c] = fmaf(av[a], bv[c], acc[a][c]);
        }
        __syncthreads();
    }

#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const int32_t m = m0 + ty + 16 * a;
        if (m >= M) continue;
        int32_t r;
        float s;
        const int32_t i = resolve_slot(row_slot[m], m, ranks, scales, max_slots, bps, &r, &s,
                                       status, false);
        float lo[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        if (i >= 0) {
            const float *vr = V + static_cast<size_t>(m) * ldv;
            for (int32_t j = 0; j < r; ++j) {
                const int32_t b = table[i * bps + (j >> 4)];
                if (b < 0 || b >= num_blocks) {
                    record_error(status, kDevBadBlock, static_cast<uint32_t>(i));
                    lo[0] = lo[1] = lo[2] = lo[3] = 0.0f;
                    s = 0.0f;
                    break;
                }
                const T *bb = b_arena + static_cast<size_t>(b) * N * LORA_BLOCK_ROWS + (j & 15);
                const float v = vr[j];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int32_t n = n0 + tx + 16 * c;
                    if (n < N) lo[c] = fmaf(to_float(bb[static_cast<size_t>(n) * LORA_BLOCK_ROWS]), v, lo[c]);
                }
            }
        } else {
            s = 0.0f;
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int32_t n = n0 + tx + 16 * c;
            if (n < N) out[static_cast<size_t>(m) * ldo + n] = from_float<T>(fmaf(s, lo[c], acc[a][c]));
        }
    }
}

template <typename T>
static cudaError_t launch_forward_simt(const ForwardPlan &plan, cudaStream_t stream) {
    for (int p = 0; p < plan.n_proj; ++p) {
        const ProjView &v = plan.proj[p];
        dim3 sgrid(plan.M, v.bps);
        shrink_simt_kernel<T><<<sgrid, 128, 0, stream>>>(
            static_cast<const T *>(plan.x), plan.ldx, plan.K, plan.row_slot,
            static_cast<const T *>(v.a_arena), v.table, v.ranks, v.max_slots, v.bps, v.num_blocks,
            v.V, v.max_rank, plan.status, plan.counters, plan.n_counters);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        if (plan.stage_events) {
            e = cudaEventRecord(static_cast<cudaEvent_t>(plan.stage_events[1 + 2 * p]), stream);
            if (e != cudaSuccess) return e;
        }
        dim3 ggrid((v.N + 63) / 64, (plan.M + 63) / 64);
        gemm_lora_simt_kernel<T><<<ggrid, 256, 0, stream>>>(
            static_cast<const T *>(plan.x), plan.ldx, static_cast<const T *>(v.W), plan.M, v.N,
            plan.K, static_cast<T *>(v.out), v.ldo, plan.row_slot,
            static_cast<const T *>(v.b_arena), v.table, v.ranks, v.scales, v.max_slots, v.bps,
            v.num_blocks, v.V, v.max_rank, plan.status);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        count_launches(2);
        if (plan.stage_events) {
            e = cudaEventRecord(static_cast<cudaEvent_t>(plan.stage_events[2 + 2 * p]), stream);
            if (e != cudaSuccess) return e;
        }
    }
    return cudaSuccess;
}

// Several projections, each's LoRA term by the per-row kernel: one launch of
// it for all of them, then the GEMMs, two projections per launch, each launch
// a programmatic dependent of the kernel before it and with its own split-K
// tile counters (all zeroed by the per-row kernel).  Stage events: the LoRA
// stage of projection 0 covers the per-row kernel, the GEMM stage of the
// first of a pair covers the pair's launch; the other stages are empty.
static cudaError_t launch_forward_fused_rows(const ForwardPlan &plan, cudaStream_t stream) {
    auto record = [&](int i) -> cudaError_t {
        return plan.stage_events ? cudaEventRecord(static_cast<cudaEvent_t>(plan.stage_events[i]), stream)
                                 : cudaSuccess;
    };
    cudaError_t e = launch_lora_rows_all(plan, stream);
    if (e != cudaSuccess) return e;
    count_launches(1);
    if ((e = record(1)) != cudaSuccess) return e;
    int64_t coff = 0;
    for (int i = 0; i < plan.n_proj; i += 2) {
        const bool pair = i + 1 < plan.n_proj;
        if (i > 0 && (e = record(1 + 2 * i)) != cudaSuccess) return e;
        const TcPlan tp = pair ? plan_tc_pair(plan.M, plan.proj[i].N, plan.proj[i + 1].N, plan.K)
                               : plan_tc(plan.M, plan.proj[i].N, plan.K);
        const int64_t ntiles = tp.split_tiles;
        if (coff + ntiles > plan.n_counters) return cudaErrorInvalidValue;
        e = launch_gemm_lora_tc_pair(plan, plan.proj[i], pair ? &plan.proj[i + 1] : nullptr, plan.counters + coff,
                                     plan.n_counters - coff, stream);
        if (e != cudaSuccess) return e;
        count_launches(1);
        coff += ntiles;
        if ((e = record(2 + 2 * i)) != cudaSuccess) return e;
        if (pair && ((e = record(3 + 2 * i)) != cudaSuccess || (e = record(4 + 2 * i)) != cudaSuccess)) return e;
    }
    return cudaSuccess;
}

// Several projections whose LoRA terms go through the pipelined grouped
// kernels: the rows grouped once, one shrink and one expand launch for all of
// them (the SMs split between the projections, each its own ycorr), then the
// GEMMs two projections per launch, each launch a programmatic dependent of
// the kernel before it with its own split-K tile counters (all zeroed by the
// shrink).  Stage events: the LoRA stage of projection 0 covers the LoRA
// launches, the GEMM stage of the second of a pair the pair's launch; the
// other stages are empty.
static cudaError_t launch_forward_piped_pairs(const ForwardPlan &plan, cudaStream_t stream) {
    auto record = [&](int i) -> cudaError_t {
        return plan.stage_events ? cudaEventRecord(static_cast<cudaEvent_t>(plan.stage_events[i]), stream)
                                 : cudaSuccess;
    };
    const ProjView *vs[LORA_MAX_PROJ];
    for (int q = 0; q < plan.n_proj; ++q) vs[q] = &plan.proj[q];
    cudaError_t e = launch_pipe_group(plan, stream);
    if (e == cudaSuccess) e = launch_pipe_shrink(plan, vs, plan.n_proj, stream);
    if (e == cudaSuccess) e = launch_pipe_expand(plan, vs, plan.n_proj, stream);
    if (e != cudaSuccess) return e;
    count_launches(3);
    if ((e = record(1)) != cudaSuccess) return e;
    int64_t coff = 0;
    for (int i = 0; i < plan.n_proj; i += 2) {
        const bool pair = i + 1 < plan.n_proj;
        if (i > 0 && (e = record(1 + 2 * i)) != cudaSuccess) return e;
        if (pair && ((e = record(2 + 2 * i)) != cudaSuccess || (e = record(3 + 2 * i)) != cudaSuccess)) return e;
        const TcPlan tp = pair ? plan_tc_pair(plan.M, plan.proj[i].N, plan.proj[i + 1].N, plan.K)
                               : plan_tc(plan.M, plan.proj[i].N, plan.K);
        const int64_t ntiles = tp.split_tiles;
        if (coff + ntiles > plan.n_counters) return cudaErrorInvalidValue;
        e = launch_gemm_lora_tc_pair(plan, plan.proj[i], pair ? &plan.proj[i + 1] : nullptr, plan.counters + coff,
                                     plan.n_counters - coff, stream);
        if (e != cudaSuccess) return e;
        count_launches(1);
        coff += ntiles;
        if ((e = record(pair ? 4 + 2 * i : 2 + 2 * i)) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// bf16.  Small M (the GEMM's swapped orientation): per projection the LoRA
// term into plan.ycorr (lora_grouped.cu) -- by one per-row kernel when each
// row's A and B are cheap to read, else by the pipelined grouped shrink and
// expand (lora_pipe.cu; for larger pools, the rows' group table and the
// grouped kernels of lora_grouped.cu) -- then the GEMM, which adds it.  Large
// M: the token tiles' block lists and the tensor-core shrink (lora_tiles.cu),
// then the GEMM, which adds the expand as extra MMAs per listed pool block.
// The GEMM is launched as a programmatic dependent of the kernel before it
// (see tc_gemm.cu).
static cudaError_t launch_forward_tc(const ForwardPlan &plan, cudaStream_t stream) {
    const bool swapped = plan_tc(plan.M, plan.proj[0].N, plan.K).swap;
    if (plan.fused_rows) return launch_forward_fused_rows(plan, stream);
    if (plan.piped_pairs) return launch_forward_piped_pairs(plan, stream);
    bool by_row = swapped;
    for (int p = 0; p < plan.n_proj; ++p)
        by_row = by_row && row_lora_preferred(plan.M, plan.K, plan.proj[p].N, plan.proj[p].max_rank);
    // the pipelined grouped kernels read one grouping per projection,
    // made by one launch before them
    bool piped = swapped && !by_row;
    for (int p = 0; p < plan.n_proj; ++p) piped = piped && pipe_grouped_supported(plan.M, plan.proj[p].max_rank);
    GroupTable gt{};
    cudaError_t e = cudaSuccess;
    if (piped) {  // the rows grouped by adapter once, for every projection
        e = launch_pipe_group(plan, stream);
        if (e != cudaSuccess) return e;
        count_launches(1);
    }
    if (swapped && !by_row && !piped) {
        gt = group_table_at(plan.group_table, plan.M);
        e = launch_group_rows(plan, gt, plan.proj[0].max_slots, stream);
        if (e != cudaSuccess) return e;
        count_launches(1);
    }
    for (int p = 0; p < plan.n_proj; ++p) {
        const ProjView &v = plan.proj[p];
        if (by_row) {
            e = launch_lora_rows(plan, v, stream);
            if (e != cudaSuccess) return e;
        } else if (piped) {
            const ProjView *one[1] = {&v};
            e = launch_pipe_shrink(plan, one, 1, stream);
            if (e == cudaSuccess) e = launch_pipe_expand(plan, one, 1, stream);
            if (e != cudaSuccess) return e;
        } else if (swapped) {
            e = launch_shrink_grouped(plan, v, gt, stream);
            if (e == cudaSuccess) e = launch_expand_grouped(plan, v, gt, stream);
            if (e != cudaSuccess) return e;
        } else {
            // large M: the tiles' block lists; then, unless the two-SM GEMM
            // computes it itself, V on the tensor cores and Vt (and the per-row
            // V of tiles whose adapters span too many blocks)
            e = launch_tile_plan(plan, v, stream);
            if (e == cudaSuccess && !pair_gemm_takes(v)) e = launch_tc_shrink(plan, v, stream);
            if (e != cudaSuccess) return e;
        }
        if (plan.stage_events) {
            e = cudaEventRecord(static_cast<cudaEvent_t>(plan.stage_events[1 + 2 * p]), stream);
            if (e != cudaSuccess) return e;
        }
        e = launch_gemm_lora_tc(plan, v, stream);
        if (e != cudaSuccess) return e;
        count_launches(swapped ? (by_row ? 2 : 3) : (pair_gemm_takes(v) ? 2 : 4));
        if (plan.stage_events) {
            e = cudaEventRecord(static_cast<cudaEvent_t>(plan.stage_events[2 + 2 * p]), stream);
            if (e != cudaSuccess) return e;
        }
    }
    return cudaSuccess;
}

cudaError_t launch_forward(const ForwardPlan &plan, cudaStream_t stream) {
    if (plan.dtype == LORA_FP32) return launch_forward_simt<float>(plan, stream);
    return launch_forward_tc(plan, stream);
}

}  // namespace lora
