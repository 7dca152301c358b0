// The LoRA term of the large-M (prefill) orientation on the tensor cores,
// reading the adapters straight from the paged pool.
//
// The GEMM of tc_gemm.cu takes 128 tokens per tile.  For each such tile this
// file builds
//
//   tile_plan_kernel   the tile's block list: the distinct adapter slots its
//                      rows name, in ascending order, and for each the pool
//                      blocks that hold its rank-rows (ceil(r/16) blocks of 16
//                      rank-rows; nothing padded to the pool's maximum rank).
//                      At most kPlanMaxBlocks blocks per tile; a tile that
//                      needs more (rows in no useful order) is marked for the
//                      CUDA-core fallback, whose per-row V this kernel
//                      computes itself.
//   tc_shrink_kernel   Vt = x_tile A_list^T on tcgen05: the MMA's A operand is
//                      the tile's 128 x rows, its B operand the tile's block
//                      list -- one 16-row TMA box per pool block, stacked in
//                      shared memory -- so N = 16 nb.  The (tile, k-block)
//                      pairs of all tiles with adapters are split into equal
//                      contiguous ranges, one per CTA, so every SM streams x.
//                      A tile covered by several CTAs is summed from their
//                      fp32 partial results by the CTA that finishes it last
//                      (an atomic count of its k-blocks, no waiting), always
//                      in CTA order, so the result does not depend on timing.
//                      The finished tile is written as two bf16 parts of
//                      s_i V (hi = bf16(s_i V), lo = bf16(s_i V - hi)), masked
//                      to the row's own slot: column 16e + j of row m holds
//                      rank-row j of block e of the list if that block belongs
//                      to m's slot, else 0.
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
constexpr int kShrinkThreads = 192;     // producer warp, MMA warp, four epilogue warps
constexpr int kShrinkEpiThreads = 128;
constexpr int kShrinkEpiBarrier = 1;
constexpr int kShrinkMaxStages = 8;
constexpr int kShrinkSmem = 200 * 1024; // ring + bookkeeping (dynamic shared memory)
constexpr int kShrinkMaxSegs = 64;      // segments (tile pieces) one CTA may take
constexpr int kMinPairs = 4;            // fewest (tile, k-block) pairs a CTA takes
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr int kAccCols = 16 * kPlanMaxBlocks;  // 256: TMEM columns of one accumulator
constexpr uint32_t kXBytes = kPlanRows * kBK * 2;  // 16 KiB x box per k-block

static_assert(kPlanRows == 128, "one MMA M of 128 token rows per plan tile");
static_assert(kAccCols <= 256, "the MMA's N is at most 256");

struct TilePlanParams {
    int32_t M, K, T;
    const int32_t *row_slot;
    const int32_t *table, *ranks;
    int32_t max_slots, bps, num_blocks, max_rank;
    const __nv_bfloat16 *x;
    int32_t ldx;
    const __nv_bfloat16 *a_arena;
    int32_t *plan;     // [T][kPlanInts]
    int32_t *counter;  // [T]
    float *V;          // fallback tiles: fp32 [M][max_rank]
    unsigned long long *status;
};

// Slot of row m for the LoRA term (-1: none); errors are recorded once, here.
__device__ __forceinline__ int32_t plan_row_slot(const TilePlanParams &p, int32_t m, int32_t *rank) {
    int32_t r;
    float s;
    const int32_t slot = resolve_slot(p.row_slot[m], m, p.ranks, nullptr, p.max_slots, p.bps, &r, &s, p.status, true);
    if (slot < 0) return -1;
    for (int32_t jb = 0; jb * LORA_BLOCK_ROWS < r; ++jb) {
        const int32_t blk = p.table[static_cast<size_t>(slot) * p.bps + jb];
        if (blk < 0 || blk >= p.num_blocks) {
            record_error(p.status, kDevBadBlock, static_cast<uint32_t>(slot));
            return -1;
        }
    }
    *rank = r;
    return slot;
}

// One CTA per token tile.  Warp 0 lists the tile's distinct slots (repeated
// warp minimum over the rows' slots above the last one listed) and their
// blocks; if they need more than kPlanMaxBlocks blocks, the tile is marked
// (-1) and all eight warps compute V = A_i x[m] of its rows on CUDA cores
// for the GEMM's per-row epilogue.
__global__ void __launch_bounds__(256) tile_plan_kernel(const TilePlanParams p) {
    __shared__ int32_t s_nb;
    const int32_t t = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int32_t *plan = p.plan + static_cast<size_t>(t) * kPlanInts;
    if (warp == 0) {
        int32_t mine[kPlanRows / 32];
#pragma unroll
        for (int i = 0; i < kPlanRows / 32; ++i) {
            const int32_t m = t * kPlanRows + i * 32 + lane;
            int32_t r = 0;
            const int32_t slot = m < p.M ? plan_row_slot(p, m, &r) : -1;
            mine[i] = slot < 0 ? INT_MAX : slot;
        }
        int32_t last = -1, nb = 0;
        bool overflow = false;
        while (true) {
            int32_t cand = INT_MAX;
#pragma unroll
            for (int i = 0; i < kPlanRows / 32; ++i)
                if (mine[i] > last && mine[i] < cand) cand = mine[i];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) cand = min(cand, __shfl_xor_sync(0xffffffffu, cand, o));
            if (cand == INT_MAX) break;
            const int32_t nblk = (p.ranks[cand] + LORA_BLOCK_ROWS - 1) / LORA_BLOCK_ROWS;
            if (nb + nblk > kPlanMaxBlocks) {
                overflow = true;
                break;
            }
            if (lane < nblk) {
                plan[kPlanBlkOff + nb + lane] = p.table[static_cast<size_t>(cand) * p.bps + lane];
                plan[kPlanSlotOff + nb + lane] = cand;
            }
            nb += nblk;
            last = cand;
        }
        if (lane == 0) {
            plan[0] = overflow ? -1 : nb;
            p.counter[t] = 0;
            s_nb = overflow ? -1 : nb;
        }
    }
    __syncthreads();
    // the shrink kernel (a programmatic dependent) may start once the plan is out
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (s_nb >= 0) return;
    // fallback tile: V[m][j] = sum_k A_i[j][k] x[m][k], one warp per row, lanes over k
    const int32_t K8 = p.K / 8;
    for (int32_t i = warp; i < kPlanRows; i += 8) {
        const int32_t m = t * kPlanRows + i;
        if (m >= p.M) break;
        int32_t r = 0;
        const int32_t slot = plan_row_slot(p, m, &r);
        if (slot < 0) continue;
        const uint4 *xr = reinterpret_cast<const uint4 *>(p.x + static_cast<size_t>(m) * p.ldx);
        for (int32_t jb = 0; jb * LORA_BLOCK_ROWS < r; ++jb) {
            const int32_t blk = p.table[static_cast<size_t>(slot) * p.bps + jb];
            const uint4 *ab = reinterpret_cast<const uint4 *>(p.a_arena + static_cast<size_t>(blk) * LORA_BLOCK_ROWS * p.K);
            float acc[LORA_BLOCK_ROWS];
#pragma unroll
            for (int j = 0; j < LORA_BLOCK_ROWS; ++j) acc[j] = 0.0f;
            for (int32_t k8 = lane; k8 < K8; k8 += 32) {
                float xv[8];
                VecTraits<__nv_bfloat16>::load(reinterpret_cast<const __nv_bfloat16 *>(xr + k8), xv);
#pragma unroll
                for (int j = 0; j < LORA_BLOCK_ROWS; ++j) {
                    float av[8];
                    VecTraits<__nv_bfloat16>::load(reinterpret_cast<const __nv_bfloat16 *>(ab + static_cast<size_t>(j) * K8 + k8), av);
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[j] = fmaf(av[e], xv[e], acc[j]);
                }
            }
#pragma unroll
            for (int j = 0; j < LORA_BLOCK_ROWS; ++j) {
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], o);
            }
            // rank-rows past r are zero in the pool, so every entry of the block is finite
            if (lane < LORA_BLOCK_ROWS) {
                float v = 0.0f;
#pragma unroll
                for (int j = 0; j < LORA_BLOCK_ROWS; ++j) v = lane == j ? acc[j] : v;
                p.V[static_cast<size_t>(m) * p.max_rank + jb * LORA_BLOCK_ROWS + lane] = v;
            }
        }
    }
}

// ------------------------------------------------------------------ shrink

struct ShrinkParams {
    int32_t M, K, T, num_kb;
    const int32_t *plan;
    int32_t *counter;
    const int32_t *row_slot;
    const int32_t *ranks;
    const float *scales;
    int32_t max_slots, bps;
    float *part;          // [gridDim][2][kPlanRows][kAccCols] fp32
    __nv_bfloat16 *vt;    // [T * kPlanRows][kVtCols]: hi parts in columns [0, 256), lo in [256, 512)
    unsigned long long *status;
};

struct Seg {
    int32_t tile, kb0, kb1, part;  // part: -1 whole tile here, else the CTA's partial slot (0 first, 1 last)
};

// Shared bookkeeping after the ring.
struct ShrinkShared {
    uint64_t full[kShrinkMaxStages];
    uint64_t empty[kShrinkMaxStages];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint32_t tmem_base;
    int32_t nseg;
    int32_t nb_max;
    int32_t stage_bytes;
    int32_t stages;
    volatile uint32_t abort_flag;
    volatile int32_t last_flag;
    int32_t g_eff, pairs;
    Seg seg[kShrinkMaxSegs];
};

__device__ __forceinline__ int64_t range_start(int64_t c, int64_t P, int64_t G) { return c * P / G; }
// CTA holding pair q: the largest c with range_start(c) <= q
__device__ __forceinline__ int64_t cta_of_pair(int64_t q, int64_t P, int64_t G) { return ((q + 1) * G - 1) / P; }

__device__ __forceinline__ void shrink_epi_sync() {
    asm volatile("bar.sync %0, %1;" ::"n"(kShrinkEpiBarrier), "n"(kShrinkEpiThreads) : "memory");
}

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

// s V of row m (slot `slot`, scale s) for columns col0 .. col0+31 of the tile's
// accumulator, masked to the row's slot, as hi and lo bf16 parts in Vt.
__device__ __forceinline__ void store_vt(const ShrinkParams &p, const int32_t *plan, int32_t m, int32_t slot, float s,
                                         int32_t col0, int32_t ncols, const float (&v)[32]) {
    __nv_bfloat16 *hi_dst = p.vt + static_cast<size_t>(m) * kVtCols + col0;
    __nv_bfloat16 *lo_dst = hi_dst + kVtCols / 2;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        if (g * 8 >= ncols) break;
        const int32_t e = (col0 + g * 8) / LORA_BLOCK_ROWS;  // the block entry these 8 columns belong to
        const bool own = slot >= 0 && plan[kPlanSlotOff + e] == slot;
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float h2[2], l2[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const float val = own ? s * v[g * 8 + 2 * i + u] : 0.0f;
                const __nv_bfloat16 h = __float2bfloat16_rn(val);
                h2[u] = __bfloat162float(h);
                l2[u] = val - h2[u];
            }
            const __nv_bfloat162 hh = __floats2bfloat162_rn(h2[0], h2[1]);
            const __nv_bfloat162 ll = __floats2bfloat162_rn(l2[0], l2[1]);
            hw[i] = *reinterpret_cast<const uint32_t *>(&hh);
            lw[i] = *reinterpret_cast<const uint32_t *>(&ll);
        }
        *reinterpret_cast<uint4 *>(hi_dst + g * 8) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4 *>(lo_dst + g * 8) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
}

__global__ void __launch_bounds__(kShrinkThreads, 1)
tc_shrink_kernel(const __grid_constant__ CUtensorMap tma_x, const __grid_constant__ CUtensorMap tma_a,
                 const ShrinkParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *ring = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    constexpr int kRingBytes = kShrinkSmem - 1024 - static_cast<int>(sizeof(ShrinkShared));
    ShrinkShared &sh = *reinterpret_cast<ShrinkShared *>(ring + kRingBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kShrinkMaxStages; ++s) {
            mbar_init(&sh.full[s], 1);
            mbar_init(&sh.empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sh.tmem_full[b], 1);
            mbar_init(&sh.tmem_empty[b], 4);  // one arrive per epilogue warp
        }
        sh.abort_flag = 0;
        sh.last_flag = 0;
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
    // the tile plan comes from the kernel before
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (warp == 2) {
        // active tiles (with adapter blocks), this CTA's contiguous range of
        // their (tile, k-block) pairs, and its segments
        int32_t active = 0;
        for (int32_t t0 = 0; t0 < p.T; t0 += 32) {
            const int32_t t = t0 + lane;
            const bool a = t < p.T && p.plan[static_cast<size_t>(t) * kPlanInts] > 0;
            active += __popc(__ballot_sync(0xffffffffu, a));
        }
        const int64_t P = static_cast<int64_t>(active) * p.num_kb;
        int64_t G = P / kMinPairs;
        G = G < 1 ? 1 : (G > gridDim.x ? gridDim.x : G);
        const int64_t c = blockIdx.x;
        int32_t nseg = 0, nb_max = 0;
        if (P > 0 && c < G) {
            const int64_t q0 = range_start(c, P, G), q1 = range_start(c + 1, P, G);
            // walk the active tiles in order up to the range's last pair
            int32_t a_base = 0;  // active tiles before this chunk of 32
            for (int32_t t0 = 0; t0 < p.T && static_cast<int64_t>(a_base) * p.num_kb < q1; t0 += 32) {
                const int32_t t = t0 + lane;
                const int32_t nbt = t < p.T ? p.plan[static_cast<size_t>(t) * kPlanInts] : 0;
                const unsigned act = __ballot_sync(0xffffffffu, nbt > 0);
                for (unsigned bits = act; bits; bits &= bits - 1) {
                    const int j = __ffs(bits) - 1;
                    const int32_t a = a_base + __popc(act & ((1u << j) - 1));
                    const int64_t t_q0 = static_cast<int64_t>(a) * p.num_kb, t_q1 = t_q0 + p.num_kb;
                    const int64_t lo = t_q0 > q0 ? t_q0 : q0, hi = t_q1 < q1 ? t_q1 : q1;
                    if (lo < hi) {
                        const int32_t nbj = __shfl_sync(0xffffffffu, nbt, j);
                        if (lane == 0 && nseg < kShrinkMaxSegs) {
                            Seg sg;
                            sg.tile = t0 + j;
                            sg.kb0 = static_cast<int32_t>(lo - t_q0);
                            sg.kb1 = static_cast<int32_t>(hi - t_q0);
                            sg.part = (sg.kb0 == 0 && sg.kb1 == p.num_kb) ? -1 : (lo == q0 ? 0 : 1);
                            sh.seg[nseg] = sg;
                        }
                        ++nseg;
                        nb_max = nbj > nb_max ? nbj : nb_max;
                    }
                }
                a_base += __popc(act);
            }
        }
        if (lane == 0) {
            if (nseg > kShrinkMaxSegs) {
                record_error(p.status, kDevTimeout, 20);  // range too long for the segment list
                nseg = kShrinkMaxSegs;
            }
            sh.nseg = nseg;
            sh.nb_max = nb_max;
            sh.g_eff = static_cast<int32_t>(G);
            sh.pairs = static_cast<int32_t>(P);
            const int32_t sb = static_cast<int32_t>(kXBytes) + nb_max * LORA_BLOCK_ROWS * kBK * 2;
            int32_t st = kRingBytes / (sb > 0 ? sb : 1);
            sh.stage_bytes = sb;
            sh.stages = st > kShrinkMaxStages ? kShrinkMaxStages : st;
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const int32_t nseg = sh.nseg;
    const int32_t stages = sh.stages;
    const uint32_t stage_bytes = static_cast<uint32_t>(sh.stage_bytes);

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int32_t it = 0;
            for (int32_t si = 0; si < nseg && !sh.abort_flag; ++si) {
                const Seg sg = sh.seg[si];
                const int32_t *plan = p.plan + static_cast<size_t>(sg.tile) * kPlanInts;
                const int32_t nb = plan[0];
                for (int32_t kb = sg.kb0; kb < sg.kb1; ++kb, ++it) {
                    const int s = it % stages;
                    if (!mbar_wait_bounded(&sh.empty[s], ((it / stages) & 1) ^ 1, kWaitNs)) {
                        record_error(p.status, kDevTimeout, 21);
                        sh.abort_flag = 1;
                        break;
                    }
                    uint8_t *st = ring + static_cast<size_t>(s) * stage_bytes;
                    mbar_arrive_expect_tx(&sh.full[s], kXBytes + nb * LORA_BLOCK_ROWS * kBK * 2);
                    tma_load_2d(st, &tma_x, kb * kBK, sg.tile * kPlanRows, &sh.full[s]);
                    for (int32_t e = 0; e < nb; ++e)
                        tma_load_2d(st + kXBytes + e * LORA_BLOCK_ROWS * kBK * 2, &tma_a, kb * kBK,
                                    plan[kPlanBlkOff + e] * LORA_BLOCK_ROWS, &sh.full[s]);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int32_t it = 0;
            for (int32_t si = 0; si < nseg; ++si) {
                const Seg sg = sh.seg[si];
                const int32_t nb = p.plan[static_cast<size_t>(sg.tile) * kPlanInts];
                const int b = si & 1;
                bool ok = mbar_wait_bounded(&sh.tmem_empty[b], ((si >> 1) & 1) ^ 1, kWaitNs);
                if (!ok) record_error(p.status, kDevTimeout, 22);
                tc_fence_after_sync();
                const uint32_t d = sh.tmem_base + b * kAccCols;
                const uint32_t idesc = idesc_bf16_f32(kPlanRows, nb * LORA_BLOCK_ROWS);
                for (int32_t kb = sg.kb0; kb < sg.kb1 && ok; ++kb, ++it) {
                    const int s = it % stages;
                    if (!mbar_wait_bounded(&sh.full[s], (it / stages) & 1, kWaitNs)) {
                        record_error(p.status, kDevTimeout, 23);
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t a_addr = smem_u32(ring + static_cast<size_t>(s) * stage_bytes);
                    const uint32_t b_addr = a_addr + kXBytes;
#pragma unroll
                    for (int k = 0; k < kBK / kUmmaK; ++k)
                        mma_bf16_f32(d, desc_kmajor_sw128(a_addr + k * kUmmaK * 2),
                                     desc_kmajor_sw128(b_addr + k * kUmmaK * 2), idesc,
                                     (kb > sg.kb0 || k > 0) ? 1u : 0u);
                    mma_commit(&sh.empty[s]);
                }
                if (!ok || sh.abort_flag) {
                    sh.abort_flag = 1;
                    mbar_arrive(&sh.tmem_full[b]);  // wake the epilogue so it can unwind
                    break;
                }
                mma_commit(&sh.tmem_full[b]);
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;                 // TMEM lane quarter of this warp
        const int r = q * 32 + lane;            // tile row
        const uint32_t lane_addr = sh.tmem_base + (static_cast<uint32_t>(q * 32) << 16);
        for (int32_t si = 0; si < nseg; ++si) {
            const Seg sg = sh.seg[si];
            const int32_t *plan = p.plan + static_cast<size_t>(sg.tile) * kPlanInts;
            const int32_t nb = plan[0];
            const int32_t ncols = nb * LORA_BLOCK_ROWS;
            const int b = si & 1;
            const bool ok = mbar_wait_bounded(&sh.tmem_full[b], (si >> 1) & 1, kWaitNs);
            if (!ok) {
                record_error(p.status, kDevTimeout, 24);
                sh.abort_flag = 1;
            }
            if (!shrink_epi_all(ok && !sh.abort_flag)) break;  // uniform over the epilogue warps
            tc_fence_after_sync();
            const int32_t m = sg.tile * kPlanRows + r;
            int32_t slot = -1;
            float s = 0.0f;
            if (m < p.M) {
                int32_t rr;
                slot = resolve_slot(p.row_slot[m], m, p.ranks, p.scales, p.max_slots, p.bps, &rr, &s, p.status, false);
            }
            float *mine = sg.part >= 0 ? p.part + ((static_cast<size_t>(blockIdx.x) * 2 + sg.part) * kPlanRows + r) * kAccCols
                                       : nullptr;
            for (int32_t c0 = 0; c0 < ncols; c0 += 32) {
                uint32_t raw[32];
                tmem_ld_32x32b_x32(lane_addr + b * kAccCols + c0, raw);
                tmem_ld_wait(raw);
                float v[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(raw[e]);
                const int32_t nc = ncols - c0 < 32 ? ncols - c0 : 32;
                if (mine) {
#pragma unroll
                    for (int g = 0; g < 8; ++g)
                        if (g * 4 < nc)
                            __stcg(reinterpret_cast<float4 *>(mine + c0) + g,
                                   make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]));
                } else if (m < p.M) {
                    store_vt(p, plan, m, slot, s, c0, nc, v);
                }
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.tmem_empty[b]);
            if (!mine) continue;
            // partial: count the tile's k-blocks; the CTA that completes the
            // count sums every contributor's partial in CTA order
            __threadfence();
            shrink_epi_sync();
            if (threadIdx.x == 64) {
                const int32_t done = atomicAdd(p.counter + sg.tile, sg.kb1 - sg.kb0) + (sg.kb1 - sg.kb0);
                sh.last_flag = done == p.num_kb ? 1 : 0;
            }
            shrink_epi_sync();
            if (!sh.last_flag) continue;
            __threadfence();
            // the tile's active index from the first pair this CTA holds of it
            const int64_t P = sh.pairs, G = sh.g_eff;
            const int64_t my_q0 = range_start(blockIdx.x, P, G);
            const int64_t a = (sg.part == 0 ? my_q0 : range_start(blockIdx.x + 1, P, G) - 1) / p.num_kb;
            const int64_t t_q0 = a * p.num_kb;
            const int64_t c_first = cta_of_pair(t_q0, P, G), c_last = cta_of_pair(t_q0 + p.num_kb - 1, P, G);
            if (m >= p.M) continue;
            for (int32_t c0 = 0; c0 < ncols; c0 += 32) {
                float v[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = 0.0f;
                const int32_t nc = ncols - c0 < 32 ? ncols - c0 : 32;
                for (int64_t cc = c_first; cc <= c_last; ++cc) {
                    const int slot_idx = range_start(cc, P, G) / p.num_kb == a ? 0 : 1;
                    const float4 *src = reinterpret_cast<const float4 *>(
                        p.part + ((static_cast<size_t>(cc) * 2 + slot_idx) * kPlanRows + r) * kAccCols + c0);
#pragma unroll
                    for (int g = 0; g < 8; ++g) {
                        if (g * 4 < nc) {
                            const float4 w = __ldcg(src + g);
                            v[4 * g] += w.x;
                            v[4 * g + 1] += w.y;
                            v[4 * g + 2] += w.z;
                            v[4 * g + 3] += w.w;
                        }
                    }
                }
                store_vt(p, plan, m, slot, s, c0, nc, v);
            }
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(sh.tmem_base, 2 * kAccCols);
    }
}

}  // namespace

int tc_shrink_grid(int32_t M, int32_t K) {
    const int64_t T = (M + kPlanRows - 1) / kPlanRows;
    const int64_t pairs = T * ((K + kBK - 1) / kBK);
    int64_t g = pairs / kMinPairs;
    const int sms = device_sm_count();
    g = g < 1 ? 1 : (g > sms ? sms : g);
    return static_cast<int>(g);
}

size_t tc_shrink_part_bytes(int grid) {
    return sizeof(float) * static_cast<size_t>(grid) * 2 * kPlanRows * kAccCols;
}

cudaError_t launch_tile_plan(const ForwardPlan &plan, const ProjView &v, cudaStream_t stream) {
    TilePlanParams p;
    p.M = plan.M;
    p.K = plan.K;
    p.T = (plan.M + kPlanRows - 1) / kPlanRows;
    p.row_slot = plan.row_slot;
    p.table = v.table;
    p.ranks = v.ranks;
    p.max_slots = v.max_slots;
    p.bps = v.bps;
    p.num_blocks = v.num_blocks;
    p.max_rank = v.max_rank;
    p.x = static_cast<const __nv_bfloat16 *>(plan.x);
    p.ldx = plan.ldx;
    p.a_arena = static_cast<const __nv_bfloat16 *>(v.a_arena);
    p.plan = v.tile_plan;
    p.counter = v.tile_counter;
    p.V = v.V;
    p.status = plan.status;
    if (!p.plan || !p.counter || !p.V) return cudaErrorInvalidValue;
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
    if (!v.tile_plan || !v.tile_counter || !v.shrink_part || !v.vt || v.shrink_grid <= 0) return cudaErrorInvalidValue;
    CUtensorMap tx, ta;
    if (!make_tmap_bf16(&tx, plan.x, plan.M, plan.K, plan.ldx, kPlanRows)) return cudaErrorInvalidValue;
    if (!make_tmap_bf16(&ta, v.a_arena, static_cast<uint64_t>(v.num_blocks) * LORA_BLOCK_ROWS, plan.K, plan.K,
                        LORA_BLOCK_ROWS))
        return cudaErrorInvalidValue;
    ShrinkParams p;
    p.M = plan.M;
    p.K = plan.K;
    p.T = (plan.M + kPlanRows - 1) / kPlanRows;
    p.num_kb = (plan.K + kBK - 1) / kBK;
    p.plan = v.tile_plan;
    p.counter = v.tile_counter;
    p.row_slot = plan.row_slot;
    p.ranks = v.ranks;
    p.scales = v.scales;
    p.max_slots = v.max_slots;
    p.bps = v.bps;
    p.part = v.shrink_part;
    p.vt = static_cast<__nv_bfloat16 *>(v.vt);
    p.status = plan.status;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(v.shrink_grid);
    cfg.blockDim = dim3(kShrinkThreads);
    cfg.dynamicSmemBytes = kShrinkSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tc_shrink_kernel, tx, ta, p);
}

}  // namespace lora
