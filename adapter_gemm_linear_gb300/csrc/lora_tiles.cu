// The LoRA term of the large-M (prefill) orientation on the tensor cores,
// reading the adapters straight from the paged pool.
//
// A plan tile is 256 tokens (the token tile of the two-SM GEMM).  For each
// plan tile this file builds
//
//   tile_plan_kernel   the tile's block list: the distinct adapter slots its
//                      rows name, in ascending order, and for each the pool
//                      blocks that hold its rank-rows (ceil(r/16) blocks of 16
//                      rank-rows; nothing padded to the pool's maximum rank).
//                      At most kPlanMaxBlocks blocks per tile; a tile that
//                      needs more (rows in no useful order) is marked for the
//                      CUDA-core fallback, whose per-row V this kernel
//                      computes itself.
//   tc_shrink_kernel   V = x_tile A_list^T on tcgen05, per 128-row half of a
//                      plan tile: the MMA's A operand is the half's 128 x
//                      rows, its B operand the plan tile's block
//                      list -- one 16-row TMA box per pool block, stacked in
//                      shared memory -- so N = 16 nb.  The (half tile,
//                      k-block) pairs of all tiles are split into contiguous
//                      ranges of equal length, one per CTA, so every SM
//                      streams the same number of x boxes (halves without
//                      adapter rows are loaded and skipped);
//                      each CTA adds its part of a tile into an fp32
//                      accumulator (zeroed by the plan kernel) with coalesced
//                      reductions, so no CTA waits for another.
//   tile_convert_kernel  Vt from the accumulator: two bf16 parts of s_i V
//                      (hi = bf16(s_i V), lo = bf16(s_i V - hi)), masked to
//                      the row's own slot: column 16e + j of row m holds
//                      rank-row j of block e of the list if that block belongs
//                      to m's slot, else 0.  For tiles marked for the fallback
//                      it computes the per-row V on CUDA cores instead.
//
// The GEMM then adds, for every block e of its token tile's list, the
// products [Vt_hi | Vt_lo](:, 16e:16e+16) x B_block(e)^T as two extra MMAs of
// K = 16, reading the block's 16 rank-columns of B straight from the pool's
// B arena ([N][16] per block: a 32-byte row per output column, a box with
// the 32-byte swizzle).  This is the batched LoRA operator of the S-LoRA
// page (§"Batched LoRA computation: why this requires new CUDA kernels")
// over its paged pool (§"Unified paging"), with the rows grouped by adapter
// as the residency page's segmented GEMM does (§"Batch composition under
// many adapters").
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <climits>
#include <mutex>

#include "lora_device.cuh"
#include "lora_internal.h"
#include "sm100_ptx.cuh"
#include "tensor_map.h"

namespace lora {

namespace {

using namespace sm100;

constexpr int kBK = 64;                 // k-block: 64 bf16, one 128-byte swizzle row
constexpr int kUmmaK = 16;
constexpr int kShrinkThreads = 224;     // x producer warp, MMA warp, A producer warp, four epilogue warps
constexpr int kShrinkEpiThreads = 128;
constexpr int kShrinkEpiBarrier = 1;  // named barrier of the epilogue warps
constexpr int kShrinkXStages = 8;       // x ring: 16 KiB boxes, the DRAM stream
constexpr int kShrinkXGroup = 4;        // x boxes issued together: consecutive k-blocks of the same rows
constexpr int kShrinkMaxAStages = 8;    // A ring: the tile's pool-block boxes of one k-block (mostly L2 hits)
constexpr int kShrinkSmem = 220 * 1024; // rings + bookkeeping (dynamic shared memory)
constexpr int kShrinkMaxSegs = 64;      // segments (tile pieces) one CTA may take
constexpr int kMinPairs = 4;            // fewest (tile, k-block) pairs a CTA takes
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr int kAccCols = 16 * kPlanMaxBlocks;  // 256: TMEM columns of one accumulator
constexpr int kSubRows = 128;           // rows of the shrink's MMA (M): half a plan tile
constexpr uint32_t kXBytes = kSubRows * kBK * 2;  // 16 KiB x box per k-block
constexpr int kConvertSplit = 4;        // CTAs per tile of the convert kernel

static_assert(kPlanRows == 2 * kSubRows, "a plan tile is two shrink tiles");
static_assert(kShrinkXStages % kShrinkXGroup == 0, "x groups tile the ring");
static_assert(kAccCols <= 256, "the MMA's N is at most 256");

struct TilePlanParams {
    int32_t M, T;
    const int32_t *row_slot;
    // sorted segments without a permutation: each row's slot from them,
    // written to row_slot_out (NULL: row_slot holds the slots already)
    const int32_t *seg_offsets, *seg_adapter;
    int32_t num_segs;
    int32_t *row_slot_out;
    const int32_t *table, *ranks;
    int32_t max_slots, bps, num_blocks;
    int32_t *plan;     // [T][kPlanInts]
    float *vacc;       // [T][kAccCols][kPlanRows] fp32, zeroed here for the listed blocks (NULL: none)
    unsigned long long *status;
};

// One CTA per token tile.  Every thread resolves one row's slot (errors are
// recorded here, once per row) and fetches the slot's rank and first
// kPlanPrefetch block-table entries into shared memory, all in parallel.
// Warp 0 then lists the tile's distinct slots -- a repeated warp minimum over
// the slots above the last one listed -- with their pool blocks, read from
// a row of that slot in shared memory (a slot with a block entry out of range
// is reported and left out: its rows get no correction).  More than
// kPlanMaxBlocks blocks mark the tile (-1) for the CUDA-core fallback.  On
// the one-SM path the CTA then zeroes the accumulator columns of the listed
// blocks.
__global__ void __launch_bounds__(256) tile_plan_kernel(const TilePlanParams p) {
    static_assert(kPlanRows == 256, "one thread per row of the plan tile");
    constexpr int kPlanPrefetch = 4;  // table entries fetched per row (ranks up to 64)
    __shared__ int32_t s_nb;
    __shared__ int32_t s_slot[kPlanRows];
    __shared__ int32_t s_rank[kPlanRows];
    __shared__ int32_t s_tbl[kPlanRows][kPlanPrefetch];
    const int32_t t = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int32_t *plan = p.plan + static_cast<size_t>(t) * kPlanInts;
    // the shrink (a programmatic dependent) may launch at once: its x stream
    // needs no plan, and it reads the plan and adds into the accumulator only
    // after this grid has completed
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    {
        // every thread resolves one row's slot (errors recorded here, once per row)
        const int32_t m = t * kPlanRows + threadIdx.x;
        int32_t id = -1;
        if (p.row_slot_out) {
            // segment s covers positions [off[s], off[s+1]); the row's segment is
            // the last one starting at or before it (offsets must not decrease
            // and must lie within [0, M]; the first tile's CTA checks them)
            const int32_t S = p.num_segs;
            if (t == 0)
                for (int32_t i = threadIdx.x; i <= S; i += blockDim.x) {
                    const int32_t o = p.seg_offsets[i];
                    if (o < 0 || o > p.M || (i > 0 && p.seg_offsets[i - 1] > o))
                        record_error(p.status, kDevBadSegment, static_cast<uint32_t>(i));
                }
            if (m < p.M && S > 0 && p.seg_offsets[0] <= m) {
                int32_t lo = 0, hi = S;
                while (lo < hi) {
                    const int32_t mid = (lo + hi + 1) >> 1;
                    if (p.seg_offsets[mid] <= m) lo = mid; else hi = mid - 1;
                }
                if (lo < S && m < p.seg_offsets[lo + 1]) id = p.seg_adapter[lo];
            }
            if (m < p.M) p.row_slot_out[m] = id;
        } else if (m < p.M) {
            id = p.row_slot[m];
        }
        const int32_t rk = (id >= 0 && id < p.max_slots) ? p.ranks[id] : 0;
        int32_t mine = INT_MAX;
        if (id != -1 && m < p.M) {
            if (id < -1 || id >= p.max_slots)
                record_error(p.status, kDevBadAdapter, static_cast<uint32_t>(m));
            else if (rk <= 0)
                record_error(p.status, kDevEmptySlot, static_cast<uint32_t>(m));
            else if (rk > p.bps * LORA_BLOCK_ROWS)
                record_error(p.status, kDevBadBlock, static_cast<uint32_t>(id));
            else
                mine = id;
        }
        s_slot[threadIdx.x] = mine;
        s_rank[threadIdx.x] = mine == INT_MAX ? 0 : rk;
        const int32_t nblk = mine == INT_MAX ? 0 : (rk + LORA_BLOCK_ROWS - 1) / LORA_BLOCK_ROWS;
#pragma unroll
        for (int i = 0; i < kPlanPrefetch; ++i)
            s_tbl[threadIdx.x][i] = i < nblk ? p.table[static_cast<size_t>(mine) * p.bps + i] : 0;
    }
    __syncthreads();
    if (warp == 0) {
        constexpr int kRowsPerLane = kPlanRows / 32;
        int32_t mine[kRowsPerLane];
#pragma unroll
        for (int i = 0; i < kRowsPerLane; ++i) mine[i] = s_slot[i * 32 + lane];
        int32_t last = -1, nb = 0;
        bool overflow = false;
        while (true) {
            int32_t cand = INT_MAX;
#pragma unroll
            for (int i = 0; i < kRowsPerLane; ++i)
                if (mine[i] > last && mine[i] < cand) cand = mine[i];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) cand = min(cand, __shfl_xor_sync(0xffffffffu, cand, o));
            if (cand == INT_MAX) break;
            last = cand;
            // a row of slot cand: its rank and first table entries are in shared memory
            int32_t mrow = -1;
#pragma unroll
            for (int i = kRowsPerLane - 1; i >= 0; --i)
                if (mine[i] == cand) mrow = i * 32 + lane;
            const uint32_t holders = __ballot_sync(0xffffffffu, mrow >= 0);
            const int32_t row = __shfl_sync(0xffffffffu, mrow, __ffs(holders) - 1);
            const int32_t nblk = (s_rank[row] + LORA_BLOCK_ROWS - 1) / LORA_BLOCK_ROWS;
            const int32_t blk = lane < nblk ? (lane < kPlanPrefetch ? s_tbl[row][lane]
                                                                    : p.table[static_cast<size_t>(cand) * p.bps + lane])
                                            : 0;
            if (__any_sync(0xffffffffu, lane < nblk && (blk < 0 || blk >= p.num_blocks))) {
                if (lane == 0) record_error(p.status, kDevBadBlock, static_cast<uint32_t>(cand));
                continue;
            }
            if (nb + nblk > kPlanMaxBlocks) {
                overflow = true;
                break;
            }
            if (lane < nblk) {
                plan[kPlanBlkOff + nb + lane] = blk;
                plan[kPlanSlotOff + nb + lane] = cand;
            }
            nb += nblk;
        }
        if (lane == 0) {
            plan[0] = overflow ? -1 : nb;
            plan[kPlanReadyOff] = 0;
            plan[kPlanPartOff] = 0;
            plan[kPlanPartOff + 1] = 0;
            plan[kPlanQueueOff] = 0;
            s_nb = overflow ? -1 : nb;
        }
    }
    __syncthreads();
    if (!p.vacc) return;  // the two-SM GEMM computes V itself, without the accumulator
    const int32_t n4 = s_nb > 0 ? s_nb * LORA_BLOCK_ROWS * kPlanRows / 4 : 0;
    float4 *acc = reinterpret_cast<float4 *>(p.vacc + static_cast<size_t>(t) * kAccCols * kPlanRows);
    for (int32_t i = threadIdx.x; i < n4; i += blockDim.x) acc[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
}

// ------------------------------------------------------------------ shrink

struct ShrinkParams {
    int32_t M, T, num_kb;  // T: 128-row sub-tiles (two per plan tile)
    const int32_t *plan;
    float *vacc;          // [T][kAccCols][kPlanRows] fp32 accumulator (column-major per tile)
    unsigned long long *status;
};

struct Seg {
    int32_t tile, kb0, kb1;
};

// Shared bookkeeping after the ring.
struct ShrinkShared {
    uint64_t xfull[kShrinkXStages];
    uint64_t xempty[kShrinkXStages];
    uint64_t afull[kShrinkMaxAStages];
    uint64_t aempty[kShrinkMaxAStages];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint32_t tmem_base;
    int32_t nseg;
    volatile uint32_t abort_flag;
    Seg seg[kShrinkMaxSegs];
};

// AND of `v` over the epilogue threads (also a barrier among them), so that
// every epilogue warp takes the same branch at an abort.
__device__ __forceinline__ bool shrink_epi_all(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(v ? 1u : 0u), "n"(kShrinkEpiBarrier), "n"(kShrinkEpiThreads)
        : "memory");
    return r != 0;
}

// The A ring's layout for a CTA's segments, from the plan: stages sized for
// the widest block list among them.  The A producer and the MMA issuer each
// derive it the same way.
__device__ __forceinline__ void a_ring_layout(const Seg *seg, int32_t nseg, const int32_t *plan, int32_t ring_bytes,
                                              int32_t *stages, uint32_t *stage_bytes) {
    int32_t nb_max = 1;
    for (int32_t i = 0; i < nseg; ++i) {
        const int32_t nb = plan[static_cast<size_t>(seg[i].tile >> 1) * kPlanInts];
        nb_max = nb > nb_max ? nb : nb_max;
    }
    const int32_t sb = nb_max * LORA_BLOCK_ROWS * kBK * 2;
    const int32_t st = ring_bytes / sb;
    *stages = st > kShrinkMaxAStages ? kShrinkMaxAStages : st;
    *stage_bytes = static_cast<uint32_t>(sb);
}

__global__ void __launch_bounds__(kShrinkThreads, 1)
tc_shrink_kernel(const __grid_constant__ CUtensorMap tma_x, const __grid_constant__ CUtensorMap tma_a,
                 const ShrinkParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *ring = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    constexpr int kRingBytes = kShrinkSmem - 1024 - static_cast<int>(sizeof(ShrinkShared));
    constexpr int kARingBytes = kRingBytes - kShrinkXStages * static_cast<int>(kXBytes);
    static_assert(kARingBytes >= 2 * kPlanMaxBlocks * LORA_BLOCK_ROWS * kBK * 2, "A ring too small");
    ShrinkShared &sh = *reinterpret_cast<ShrinkShared *>(ring + kRingBytes);
    uint8_t *aring = ring + kShrinkXStages * kXBytes;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kShrinkXStages; ++s) {
            mbar_init(&sh.xfull[s], 1);
            mbar_init(&sh.xempty[s], 1);
        }
        for (int s = 0; s < kShrinkMaxAStages; ++s) {
            mbar_init(&sh.afull[s], 1);
            mbar_init(&sh.aempty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sh.tmem_full[b], 1);
            mbar_init(&sh.tmem_empty[b], 4);  // one arrive per epilogue warp
        }
        sh.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tma_x);
        prefetch_tensormap(&tma_a);
    }
    if (warp == 1) {
        tmem_alloc(&sh.tmem_base, 2 * kAccCols);
        tmem_relinquish();
    }
    if (warp == 2) {
        // This CTA's share of the (tile, k-block) pairs: a contiguous range of
        // equal length over all 128-row sub-tiles (every pair streams one x box from DRAM;
        // the pool blocks mostly hit L2).  It needs no plan, so x streams
        // while the plan kernel before this one is still running; tiles
        // without adapter rows are loaded and skipped.
        const int64_t P = static_cast<int64_t>(p.T) * p.num_kb;
        int64_t G = P / kMinPairs;
        G = G < 1 ? 1 : (G > gridDim.x ? gridDim.x : G);
        const int64_t c = blockIdx.x;
        if (lane == 0) {
            int32_t nseg = 0;
            if (c < G) {
                const int64_t q0 = c * P / G, q1 = (c + 1) * P / G;
                for (int64_t q = q0; q < q1 && nseg < kShrinkMaxSegs;) {
                    const int32_t t = static_cast<int32_t>(q / p.num_kb);
                    const int64_t t_end = static_cast<int64_t>(t + 1) * p.num_kb;
                    const int64_t e = t_end < q1 ? t_end : q1;
                    Seg sg;
                    sg.tile = t;
                    sg.kb0 = static_cast<int32_t>(q - static_cast<int64_t>(t) * p.num_kb);
                    sg.kb1 = static_cast<int32_t>(e - static_cast<int64_t>(t) * p.num_kb);
                    sh.seg[nseg++] = sg;
                    q = e;
                }
                if (nseg == kShrinkMaxSegs && (q1 - q0) > 0 &&
                    sh.seg[nseg - 1].tile * static_cast<int64_t>(p.num_kb) + sh.seg[nseg - 1].kb1 < q1)
                    record_error(p.status, kDevTimeout, 20);  // range too long for the segment list
            }
            sh.nseg = nseg;
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const int32_t nseg = sh.nseg;

    if (warp == 0) {
        // ------------------------------------------------------------ x producer
        if (lane == 0) {
            int32_t it = 0;
            for (int32_t si = 0; si < nseg && !sh.abort_flag; ++si) {
                const Seg sg = sh.seg[si];
                for (int32_t kb = sg.kb0; kb < sg.kb1; ++kb, ++it) {
                    if (it % kShrinkXGroup == 0) {
                        // wait until the next kShrinkXGroup stages are all free, so
                        // that their boxes -- adjacent 128-byte pieces of the
                        // same rows -- reach DRAM together
                        for (int32_t j = 1; j < kShrinkXGroup; ++j) {
                            const int s2 = (it + j) % kShrinkXStages;
                            if (!mbar_wait_bounded(&sh.xempty[s2], (((it + j) / kShrinkXStages) & 1) ^ 1, kWaitNs)) {
                                record_error(p.status, kDevTimeout, 21);
                                sh.abort_flag = 1;
                            }
                        }
                    }
                    const int s = it % kShrinkXStages;
                    if (!mbar_wait_bounded(&sh.xempty[s], ((it / kShrinkXStages) & 1) ^ 1, kWaitNs)) {
                        record_error(p.status, kDevTimeout, 21);
                        sh.abort_flag = 1;
                    }
                    if (sh.abort_flag) break;
                    mbar_arrive_expect_tx(&sh.xfull[s], kXBytes);
                    tma_load_2d(ring + s * kXBytes, &tma_x, kb * kBK, sg.tile * kSubRows, &sh.xfull[s]);
                }
            }
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------ A producer
        if (lane == 0) {
            asm volatile("griddepcontrol.wait;" ::: "memory");  // the plan comes from the kernel before
            int32_t a_stages;
            uint32_t a_stage_bytes;
            a_ring_layout(sh.seg, nseg, p.plan, kARingBytes, &a_stages, &a_stage_bytes);
            int32_t it = 0;
            for (int32_t si = 0; si < nseg && !sh.abort_flag; ++si) {
                const Seg sg = sh.seg[si];
                const int32_t *plan = p.plan + static_cast<size_t>(sg.tile >> 1) * kPlanInts;
                const int32_t nb = plan[0];
                if (nb <= 0) continue;  // no adapter rows (or the fallback): x only
                int32_t blk[kPlanMaxBlocks];
#pragma unroll
                for (int e = 0; e < kPlanMaxBlocks; ++e) blk[e] = e < nb ? plan[kPlanBlkOff + e] : 0;
                for (int32_t kb = sg.kb0; kb < sg.kb1; ++kb, ++it) {
                    const int s = it % a_stages;
                    if (!mbar_wait_bounded(&sh.aempty[s], ((it / a_stages) & 1) ^ 1, kWaitNs)) {
                        record_error(p.status, kDevTimeout, 25);
                        sh.abort_flag = 1;
                        break;
                    }
                    uint8_t *st = aring + static_cast<size_t>(s) * a_stage_bytes;
                    mbar_arrive_expect_tx(&sh.afull[s], nb * LORA_BLOCK_ROWS * kBK * 2);
#pragma unroll
                    for (int e = 0; e < kPlanMaxBlocks; ++e)
                        if (e < nb)
                            tma_load_2d(st + e * LORA_BLOCK_ROWS * kBK * 2, &tma_a, kb * kBK, blk[e] * LORA_BLOCK_ROWS,
                                        &sh.afull[s]);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            asm volatile("griddepcontrol.wait;" ::: "memory");  // the plan comes from the kernel before
            int32_t a_stages;
            uint32_t a_stage_bytes;
            a_ring_layout(sh.seg, nseg, p.plan, kARingBytes, &a_stages, &a_stage_bytes);
            int32_t ix = 0, ia = 0, act = 0;  // x stages, A stages and accumulators used
            bool ok = true;
            for (int32_t si = 0; si < nseg && ok; ++si) {
                const Seg sg = sh.seg[si];
                const int32_t nb = p.plan[static_cast<size_t>(sg.tile >> 1) * kPlanInts];
                if (nb <= 0) {
                    // a tile without blocks: release its x stages unused
                    for (int32_t kb = sg.kb0; kb < sg.kb1; ++kb, ++ix) {
                        const int sx = ix % kShrinkXStages;
                        if (!mbar_wait_bounded(&sh.xfull[sx], (ix / kShrinkXStages) & 1, kWaitNs)) {
                            record_error(p.status, kDevTimeout, 23);
                            ok = false;
                            break;
                        }
                        mbar_arrive(&sh.xempty[sx]);
                    }
                    continue;
                }
                const int b = act & 1;
                ok = mbar_wait_bounded(&sh.tmem_empty[b], ((act >> 1) & 1) ^ 1, kWaitNs);
                if (!ok) record_error(p.status, kDevTimeout, 22);
                tc_fence_after_sync();
                const uint32_t d = sh.tmem_base + b * kAccCols;
                const uint32_t idesc = idesc_bf16_f32(kSubRows, nb * LORA_BLOCK_ROWS);
                for (int32_t kb = sg.kb0; kb < sg.kb1 && ok; ++kb, ++ix, ++ia) {
                    const int sx = ix % kShrinkXStages, sa = ia % a_stages;
                    if (!mbar_wait_bounded(&sh.xfull[sx], (ix / kShrinkXStages) & 1, kWaitNs) ||
                        !mbar_wait_bounded(&sh.afull[sa], (ia / a_stages) & 1, kWaitNs)) {
                        record_error(p.status, kDevTimeout, 23);
                        ok = false;
                        break;
                    }
                    const uint32_t a_addr = smem_u32(ring + sx * kXBytes);
                    const uint32_t b_addr = smem_u32(aring + static_cast<size_t>(sa) * a_stage_bytes);
#pragma unroll
                    for (int k = 0; k < kBK / kUmmaK; ++k)
                        mma_bf16_f32(d, desc_kmajor_sw128(a_addr + k * kUmmaK * 2),
                                     desc_kmajor_sw128(b_addr + k * kUmmaK * 2), idesc,
                                     (kb > sg.kb0 || k > 0) ? 1u : 0u);
                    mma_commit(&sh.xempty[sx]);
                    mma_commit(&sh.aempty[sa]);
                }
                if (!ok || sh.abort_flag) {
                    ok = false;
                    mbar_arrive(&sh.tmem_full[b]);  // wake the epilogue so it can unwind
                    break;
                }
                mma_commit(&sh.tmem_full[b]);
                ++act;
            }
            if (!ok) sh.abort_flag = 1;
        }
    } else {
        // ------------------------------------------------------------ epilogue
        // thread r holds sub-tile row r: its values of column j go to
        // vacc[plan tile][j][row], so each warp's reductions cover 128 contiguous bytes
        const int q = warp & 3;  // TMEM lane quarter of this warp
        const int r = q * 32 + lane;
        const uint32_t lane_addr = sh.tmem_base + (static_cast<uint32_t>(q * 32) << 16);
        // the plan and the zeroed accumulator come from the kernel before
        asm volatile("griddepcontrol.wait;" ::: "memory");
        int32_t act = 0;
        for (int32_t si = 0; si < nseg; ++si) {
            const Seg sg = sh.seg[si];
            const int32_t ncols = p.plan[static_cast<size_t>(sg.tile >> 1) * kPlanInts] * LORA_BLOCK_ROWS;
            if (ncols <= 0) continue;
            const int b = act & 1;
            const bool ok = mbar_wait_bounded(&sh.tmem_full[b], (act >> 1) & 1, kWaitNs);
            ++act;
            if (!ok) {
                record_error(p.status, kDevTimeout, 24);
                sh.abort_flag = 1;
            }
            if (!shrink_epi_all(ok && !sh.abort_flag)) break;  // uniform over the epilogue warps
            tc_fence_after_sync();
            const bool row_ok = sg.tile * kSubRows + r < p.M;
            float *dst = p.vacc + static_cast<size_t>(sg.tile >> 1) * kAccCols * kPlanRows + (sg.tile & 1) * kSubRows + r;
            for (int32_t c0 = 0; c0 < ncols; c0 += 32) {
                uint32_t raw[32];
                tmem_ld_32x32b_x32(lane_addr + b * kAccCols + c0, raw);
                tmem_ld_wait(raw);
                if (row_ok) {
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (c0 + e < ncols) atomicAdd(dst + static_cast<size_t>(c0 + e) * kPlanRows, __uint_as_float(raw[e]));
                }
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.tmem_empty[b]);
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(sh.tmem_base, 2 * kAccCols);
    }
}

// ------------------------------------------------------------------ convert

struct ConvertParams {
    int32_t M, K;
    const int32_t *plan;
    const float *vacc;
    __nv_bfloat16 *vt;    // [T * kPlanRows][kVtCols]: hi parts in columns [0, 256), lo in [256, 512)
    const int32_t *row_slot;
    const int32_t *table, *ranks;
    const float *scales;
    int32_t max_slots, bps, num_blocks, max_rank;
    const __nv_bfloat16 *x;
    int32_t ldx;
    const __nv_bfloat16 *a_arena;
    float *V;             // fallback tiles: fp32 [M][max_rank]
    unsigned long long *status;
};

// grid (T, kConvertSplit): CTA (t, y) takes block entries e = y, y + 4, ...
// of plan tile t (thread: row r of the tile, the entry's 16 columns), or,
// for a tile marked for the fallback, rows y, y + 4, ... (one warp per row,
// lanes over k).
__global__ void __launch_bounds__(256) tile_convert_kernel(const ConvertParams p) {
    // the GEMM (a programmatic dependent) may launch and stream W; it reads Vt
    // and V only after this grid has completed
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the accumulator comes from the shrink
    const int32_t t = blockIdx.x, y = blockIdx.y;
    const int32_t *plan = p.plan + static_cast<size_t>(t) * kPlanInts;
    const int32_t nb = plan[0];
    if (nb > 0) {
        const int r = threadIdx.x;  // row of the plan tile
        const int32_t m = t * kPlanRows + r;
        if (m >= p.M) return;
        int32_t rr;
        float s;
        const int32_t slot = resolve_slot(p.row_slot[m], m, p.ranks, p.scales, p.max_slots, p.bps, &rr, &s, p.status,
                                          false);
        const float *src = p.vacc + static_cast<size_t>(t) * kAccCols * kPlanRows + r;
        __nv_bfloat16 *hi_row = p.vt + static_cast<size_t>(m) * kVtCols;
        for (int32_t e = y; e < nb; e += kConvertSplit) {
            float v[LORA_BLOCK_ROWS];
#pragma unroll
            for (int i = 0; i < LORA_BLOCK_ROWS; ++i)
                v[i] = __ldcg(src + static_cast<size_t>(e * LORA_BLOCK_ROWS + i) * kPlanRows);
            store_vt_entry(hi_row, e, v, slot >= 0 && plan[kPlanSlotOff + e] == slot, s);
        }
        return;
    }
    if (nb == 0) return;
    // fallback tile: V[m][j] = sum_k A_i[j][k] x[m][k], one warp per row, lanes over k
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int32_t i = y + kConvertSplit * warp; i < kPlanRows; i += kConvertSplit * 8) {
        const int32_t m = t * kPlanRows + i;
        if (m >= p.M) break;
        int32_t r;
        float s;
        const int32_t slot = resolve_slot(p.row_slot[m], m, p.ranks, nullptr, p.max_slots, p.bps, &r, &s, p.status,
                                          false);
        if (slot < 0) continue;
        bool blocks_ok = true;
        for (int32_t jb = 0; jb * LORA_BLOCK_ROWS < r; ++jb) {
            const int32_t blk = p.table[static_cast<size_t>(slot) * p.bps + jb];
            blocks_ok &= blk >= 0 && blk < p.num_blocks;
        }
        if (!blocks_ok) continue;  // reported by the plan kernel; the epilogue drops the row's correction
        row_v_by_warp(p.x + static_cast<size_t>(m) * p.ldx, p.K, p.a_arena, p.table + static_cast<size_t>(slot) * p.bps,
                      r, p.V + static_cast<size_t>(m) * p.max_rank, lane);
    }
}

}  // namespace

int tc_shrink_grid(int32_t M, int32_t K) {
    const int64_t T = (M + kSubRows - 1) / kSubRows;
    const int64_t pairs = T * ((K + kBK - 1) / kBK);
    int64_t g = pairs / kMinPairs;
    const int sms = device_sm_count();
    g = g < 1 ? 1 : (g > sms ? sms : g);
    return static_cast<int>(g);
}

size_t tc_shrink_acc_bytes(int32_t M) {
    const size_t T = (static_cast<size_t>(M) + kPlanRows - 1) / kPlanRows;
    return sizeof(float) * T * kAccCols * kPlanRows;
}

namespace {

cudaError_t launch_pdl(const void *fn, dim3 grid, int threads, size_t smem, void **args, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace

cudaError_t launch_tile_plan(const ForwardPlan &plan, const ProjView &v, cudaStream_t stream) {
    TilePlanParams p;
    p.M = plan.M;
    p.T = (plan.M + kPlanRows - 1) / kPlanRows;
    p.row_slot = plan.row_slot;
    p.table = v.table;
    p.ranks = v.ranks;
    p.max_slots = v.max_slots;
    p.bps = v.bps;
    p.num_blocks = v.num_blocks;
    p.plan = v.tile_plan;
    p.vacc = pair_gemm_takes(v) ? nullptr : v.vacc;  // the two-SM GEMM needs no accumulator
    p.status = plan.status;
    p.seg_offsets = plan.seg_offsets;
    p.seg_adapter = plan.seg_adapter;
    p.num_segs = plan.num_segs;
    p.row_slot_out = plan.rows_in_plan ? const_cast<int32_t *>(plan.row_slot) : nullptr;
    if (!p.plan) return cudaErrorInvalidValue;
    tile_plan_kernel<<<p.T, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_tc_shrink(const ForwardPlan &plan, const ProjView &v, cudaStream_t stream) {
    static std::mutex mu;
    static uint64_t done_ctx[128] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(mu);
        uint64_t ctx = done_ctx[dev];
        if (first_use_in_context(&ctx)) {
            e = cudaFuncSetAttribute(tc_shrink_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kShrinkSmem);
            if (e != cudaSuccess) return e;
            done_ctx[dev] = current_context_id();
        }
    }
    if (!v.tile_plan || !v.vacc || !v.vt || v.shrink_grid <= 0) return cudaErrorInvalidValue;
    CUtensorMap tx, ta;
    if (!make_tmap_bf16(&tx, plan.x, plan.M, plan.K, plan.ldx, kSubRows)) return cudaErrorInvalidValue;
    if (!make_tmap_bf16(&ta, v.a_arena, static_cast<uint64_t>(v.num_blocks) * LORA_BLOCK_ROWS, plan.K, plan.K,
                        LORA_BLOCK_ROWS))
        return cudaErrorInvalidValue;
    ShrinkParams p;
    p.M = plan.M;
    p.T = (plan.M + kSubRows - 1) / kSubRows;
    p.num_kb = (plan.K + kBK - 1) / kBK;
    p.plan = v.tile_plan;
    p.vacc = v.vacc;
    p.status = plan.status;
    void *args[] = {&tx, &ta, &p};
    e = launch_pdl(reinterpret_cast<const void *>(tc_shrink_kernel), dim3(v.shrink_grid), kShrinkThreads, kShrinkSmem,
                   args, stream);
    if (e != cudaSuccess) return e;
    ConvertParams c;
    c.M = plan.M;
    c.K = plan.K;
    c.plan = v.tile_plan;
    c.vacc = v.vacc;
    c.vt = static_cast<__nv_bfloat16 *>(v.vt);
    c.row_slot = plan.row_slot;
    c.table = v.table;
    c.ranks = v.ranks;
    c.scales = v.scales;
    c.max_slots = v.max_slots;
    c.bps = v.bps;
    c.num_blocks = v.num_blocks;
    c.max_rank = v.max_rank;
    c.x = static_cast<const __nv_bfloat16 *>(plan.x);
    c.ldx = plan.ldx;
    c.a_arena = static_cast<const __nv_bfloat16 *>(v.a_arena);
    c.V = v.V;
    c.status = plan.status;
    void *cargs[] = {&c};
    return launch_pdl(reinterpret_cast<const void *>(tile_convert_kernel),
                      dim3((plan.M + kPlanRows - 1) / kPlanRows, kConvertSplit), kPlanRows, 0, cargs, stream);
}

}  // namespace lora
