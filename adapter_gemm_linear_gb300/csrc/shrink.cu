// Shrink for bf16 rows that carry per-row adapter ids:
//
//   V[m, j] = sum_k A_i[j, k] x[m, k]        i = slot of row m, j < 16*ceil(r_i/16)
//
// grouped by adapter, so that each adapter's A rows are read once however
// many rows use it (rows sharing an adapter are gathered together, as in the
// batched operators of "Adapter Residency…", §"Batch composition under many
// adapters", and "S-LoRA…", §"Batched LoRA computation").
//
// Persistent grid, two CTAs per SM.  Every CTA first finds the groups (the
// first row of each adapter present, with a shared-memory first-row table),
// then takes work items (group, 256-wide K slice sl, 128-rank group rg) in
// turn.  For an item it loads the adapter's rank-rows for slice sl (up to
// 128 x 256 bf16) into shared memory in one burst, then the group's x rows 32
// at a time, and computes one dot product per (row, rank-row) in fp32, k
// ascending.
// Each slice writes a partial plane; the last slice of a group to finish
// (per-group counter) adds the planes in slice order and writes V, so the
// result does not depend on scheduling.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "lora_device.cuh"
#include "lora_internal.h"

namespace lora {

namespace {

constexpr int kThreads = 256;
constexpr int kSlice = 256;       // k elements per CTA
constexpr int kPitch = kSlice + 8;
constexpr int kRowsPerPass = 32;  // x rows staged per pass
constexpr int kRankGroup = 128;   // rank rows per CTA (grid.z covers larger ranks)
constexpr int kItems = kRowsPerPass * kRankGroup / kThreads;
constexpr size_t kSmem = static_cast<size_t>(kRankGroup + kRowsPerPass) * kPitch * 2;
constexpr int kMaxRows = 1024;    // rows this kernel serves (kGroupedShrinkMaxRows)
constexpr int kMaxSlots = static_cast<int>(kSmem / 4);  // first-row table in the staging area

__device__ __forceinline__ void unpack8(const uint4 &q, float *v) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

struct ShrinkParams {
    const __nv_bfloat16 *x;
    int32_t ldx, K, M, slices;
    const int32_t *row_slot;
    const __nv_bfloat16 *a_arena;
    const int32_t *table, *ranks;
    int32_t max_slots, bps, num_blocks;
    float *V;          // [M][ldv] final
    int32_t ldv;
    float *part;       // [slices][M][ldv] partial planes
    int32_t *counters; // [M][rank groups], zero on entry
    int32_t rank_groups;
    unsigned long long *status;
};

// Collect, in order, the rows m in [w0, w0 + 256) using `slot`; returns the count.
__device__ __forceinline__ int collect_rows(const ShrinkParams &p, int32_t slot, int32_t w0, int32_t *s_rows,
                                            int32_t *s_warp) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t m = w0 + tid;
    const bool match = m < p.M && p.row_slot[m] == slot;
    const unsigned ballot = __ballot_sync(0xffffffffu, match);
    if (lane == 0) s_warp[warp] = __popc(ballot);
    __syncthreads();
    int before = 0, n = 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) {
        before += (w < warp) ? s_warp[w] : 0;
        n += s_warp[w];
    }
    if (match) s_rows[before + __popc(ballot & ((1u << lane) - 1))] = m;
    __syncthreads();
    return n;
}

__global__ void __launch_bounds__(kThreads)
shrink_grouped_kernel(const ShrinkParams p) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    __nv_bfloat16 (*a_s)[kPitch] = reinterpret_cast<__nv_bfloat16 (*)[kPitch]>(smem_raw);
    __nv_bfloat16 (*x_s)[kPitch] = reinterpret_cast<__nv_bfloat16 (*)[kPitch]>(smem_raw + kRankGroup * kPitch * 2);
    int32_t *first = reinterpret_cast<int32_t *>(smem_raw);  // [max_slots], before staging starts
    __shared__ int32_t s_leaders[kMaxRows];
    __shared__ int32_t s_rows[kThreads];
    __shared__ int32_t s_blk[kRankGroup / LORA_BLOCK_ROWS];
    __shared__ int32_t s_warp[kThreads / 32];
    __shared__ int32_t s_last;
    __shared__ int32_t s_groups;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // ---- groups: the first row of every adapter present (same list in every CTA)
    for (int32_t sl = tid; sl < p.max_slots; sl += kThreads) first[sl] = 0x7fffffff;
    __syncthreads();
    for (int32_t m = tid; m < p.M; m += kThreads) {
        int32_t r;
        float sc;
        const int32_t slot = resolve_slot(p.row_slot[m], m, p.ranks, nullptr, p.max_slots, p.bps, &r, &sc, p.status,
                                          blockIdx.x == 0);
        if (slot >= 0) atomicMin(first + slot, m);
    }
    __syncthreads();
    int32_t groups = 0;
    for (int32_t w0 = 0; w0 < p.M; w0 += kThreads) {
        const int32_t m = w0 + tid;
        bool lead = false;
        if (m < p.M) {
            const int32_t id = p.row_slot[m];
            lead = id >= 0 && id < p.max_slots && first[id] == m;
        }
        const unsigned ballot = __ballot_sync(0xffffffffu, lead);
        if (lane == 0) s_warp[warp] = __popc(ballot);
        __syncthreads();
        int before = 0, n = 0;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) {
            before += (w < warp) ? s_warp[w] : 0;
            n += s_warp[w];
        }
        if (lead) s_leaders[groups + before + __popc(ballot & ((1u << lane) - 1))] = m;
        groups += n;
        __syncthreads();
    }
    if (tid == 0) s_groups = groups;
    __syncthreads();
    groups = s_groups;

    // ---- work items (group, k slice, rank group)
    const int rgroups = p.rank_groups;
    const int32_t items = groups * p.slices * rgroups;
    for (int32_t item = blockIdx.x; item < items; item += gridDim.x) {
        const int32_t gi = item / (p.slices * rgroups);
        const int32_t rem = item % (p.slices * rgroups);
        const int32_t sl = rem / rgroups, rg = rem % rgroups;
        const int32_t g = s_leaders[gi];
        const int32_t slot = p.row_slot[g];
        const int32_t r = p.ranks[slot];
        const int32_t j0 = rg * kRankGroup;
        const int32_t r16 = (r + LORA_BLOCK_ROWS - 1) / LORA_BLOCK_ROWS * LORA_BLOCK_ROWS;
        if (j0 >= r16) continue;  // uniform: same item in every thread
        const int32_t nj = min(kRankGroup, r16 - j0);
        __syncthreads();  // the previous item is done with the shared arrays
        if (tid < nj / LORA_BLOCK_ROWS) {
            const int32_t b = p.table[slot * p.bps + j0 / LORA_BLOCK_ROWS + tid];
            s_blk[tid] = b;
            if (b < 0 || b >= p.num_blocks) record_error(p.status, kDevBadBlock, static_cast<uint32_t>(slot));
        }
        __syncthreads();
        bool bad = false;
        for (int t = 0; t < nj / LORA_BLOCK_ROWS; ++t) bad |= (s_blk[t] < 0 || s_blk[t] >= p.num_blocks);
        if (bad) continue;

        // this slice of the adapter's rank-rows, zero past K
        const int32_t k0 = sl * kSlice;
        for (int idx = tid; idx < nj * (kSlice / 8); idx += kThreads) {
            const int j = idx / (kSlice / 8), c = idx % (kSlice / 8);
            const int32_t k = k0 + c * 8;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (k < p.K)
                v = __ldg(reinterpret_cast<const uint4 *>(
                    p.a_arena +
                    (static_cast<size_t>(s_blk[j / LORA_BLOCK_ROWS]) * LORA_BLOCK_ROWS + j % LORA_BLOCK_ROWS) * p.K + k));
            *reinterpret_cast<uint4 *>(&a_s[j][c * 8]) = v;
        }
        float *plane = p.part + static_cast<size_t>(sl) * p.M * p.ldv;
        for (int32_t w0 = g; w0 < p.M; w0 += kThreads) {
            const int n = collect_rows(p, slot, w0, s_rows, s_warp);
            for (int p0 = 0; p0 < n; p0 += kRowsPerPass) {
                const int np = min(kRowsPerPass, n - p0);
                for (int idx = tid; idx < np * (kSlice / 8); idx += kThreads) {
                    const int i = idx / (kSlice / 8), c = idx % (kSlice / 8);
                    const int32_t k = k0 + c * 8;
                    uint4 v = make_uint4(0, 0, 0, 0);
                    if (k < p.K)
                        v = __ldg(reinterpret_cast<const uint4 *>(p.x + static_cast<size_t>(s_rows[p0 + i]) * p.ldx + k));
                    *reinterpret_cast<uint4 *>(&x_s[i][c * 8]) = v;
                }
                __syncthreads();
#pragma unroll
                for (int q = 0; q < kItems; ++q) {
                    const int it = tid + q * kThreads;
                    if (it < np * nj) {
                        const int i = it / nj, j = it % nj;
                        float a0 = 0.0f, a1 = 0.0f;
#pragma unroll 4
                        for (int c = 0; c < kSlice / 8; c += 2) {
                            float av[8], xv[8], bv[8], yv[8];
                            unpack8(*reinterpret_cast<const uint4 *>(&a_s[j][c * 8]), av);
                            unpack8(*reinterpret_cast<const uint4 *>(&x_s[i][c * 8]), xv);
                            unpack8(*reinterpret_cast<const uint4 *>(&a_s[j][c * 8 + 8]), bv);
                            unpack8(*reinterpret_cast<const uint4 *>(&x_s[i][c * 8 + 8]), yv);
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                a0 = fmaf(av[e], xv[e], a0);
                                a1 = fmaf(bv[e], yv[e], a1);
                            }
                        }
                        plane[static_cast<size_t>(s_rows[p0 + i]) * p.ldv + j0 + j] = a0 + a1;
                    }
                }
                __syncthreads();  // x_s is rewritten by the next pass
            }
        }

        // the last slice to finish adds the planes in slice order
        __threadfence();
        __syncthreads();
        if (tid == 0) {
            const int32_t old = atomicAdd(p.counters + gi * rgroups + rg, 1);
            s_last = (old == p.slices - 1) ? 1 : 0;
        }
        __syncthreads();
        if (!s_last) continue;
        __threadfence();
        for (int32_t w0 = g; w0 < p.M; w0 += kThreads) {
            const int n = collect_rows(p, slot, w0, s_rows, s_warp);
            for (int it = tid; it < n * nj; it += kThreads) {
                const int i = it / nj, j = it % nj;
                const size_t off = static_cast<size_t>(s_rows[i]) * p.ldv + j0 + j;
                float acc = 0.0f;
                for (int32_t s2 = 0; s2 < p.slices; ++s2)
                    acc += __ldcg(p.part + static_cast<size_t>(s2) * p.M * p.ldv + off);
                p.V[off] = acc;
            }
            __syncthreads();
        }
    }
}

}  // namespace

int32_t shrink_slices(int32_t K) { return (K + kSlice - 1) / kSlice; }

size_t shrink_workspace_bytes(int32_t M, int32_t K, int32_t max_rank) {
    const size_t planes = sizeof(float) * static_cast<size_t>(shrink_slices(K)) * M * max_rank;
    const size_t counters = sizeof(int32_t) * static_cast<size_t>(M) * ((max_rank + kRankGroup - 1) / kRankGroup);
    return align_up(planes, 256) + align_up(counters, 256);
}

bool shrink_grouped_supported(int32_t M, int32_t max_slots) { return M <= kMaxRows && max_slots <= kMaxSlots; }

cudaError_t launch_shrink_grouped(const ForwardPlan &plan, const ProjView &v, void *scratch, cudaStream_t stream) {
    static std::mutex mu;
    static bool done[128] = {};
    static int sms[128] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!done[dev]) {
            e = cudaFuncSetAttribute(shrink_grouped_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(kSmem));
            if (e != cudaSuccess) return e;
            e = cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess) return e;
            done[dev] = true;
        }
    }
    ShrinkParams p;
    p.x = static_cast<const __nv_bfloat16 *>(plan.x);
    p.ldx = plan.ldx;
    p.K = plan.K;
    p.M = plan.M;
    p.slices = shrink_slices(plan.K);
    p.row_slot = plan.row_slot;
    p.a_arena = static_cast<const __nv_bfloat16 *>(v.a_arena);
    p.table = v.table;
    p.ranks = v.ranks;
    p.max_slots = v.max_slots;
    p.bps = v.bps;
    p.num_blocks = v.num_blocks;
    p.V = v.V;
    p.ldv = v.max_rank;
    p.rank_groups = (v.max_rank + kRankGroup - 1) / kRankGroup;
    const size_t planes = sizeof(float) * static_cast<size_t>(p.slices) * plan.M * v.max_rank;
    p.part = static_cast<float *>(scratch);
    p.counters = reinterpret_cast<int32_t *>(static_cast<unsigned char *>(scratch) + align_up(planes, 256));
    p.status = plan.status;
    e = cudaMemsetAsync(p.counters, 0, sizeof(int32_t) * static_cast<size_t>(plan.M) * p.rank_groups, stream);
    if (e != cudaSuccess) return e;
    const long max_items = static_cast<long>(plan.M) * p.slices * p.rank_groups;
    const int grid = static_cast<int>(max_items < 2L * sms[dev] ? max_items : 2L * sms[dev]);
    shrink_grouped_kernel<<<grid, kThreads, kSmem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace lora
