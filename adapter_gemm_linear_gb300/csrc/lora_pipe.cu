// The small-M LoRA path by adapter group as two pipelined persistent kernels
// (one CTA per SM):
//
//   pipe_shrink_kernel:  V[p][i, 16 jb + j] = sum_{k in slice p} A_s[16 jb + j, k] x[perm[i], k]
//   pipe_expand_kernel:  ycorr[perm[i], n] = scale_s * sum_j B_s[n, j] (sum_p V[p][i, j])
//
// for the sorted positions i of every row group (rows that share adapter slot
// s).  This is the batched shrink/expand of the S-LoRA page's kernel section
// (MBGMV/MBGMM over a paged pool), with the rows sorted by adapter as in the
// Punica SGMV description, laid out for this GPU:
//
//   * One small launch per forward (pipe_group_kernel, a CTA per
//     projection) sorts the rows by (rank blocks descending, slot), a
//     bitonic sort of 512 keys mostly in registers, cuts the groups into
//     chunks of at most 16 positions and writes the chunk table; every CTA
//     of both kernels copies its projection's table into shared memory, so
//     the sort is not repeated per CTA and per projection.
//   * A producer warp streams the adapter data with untiled TMA bulk copies
//     into a ring of shared-memory stages (mbarrier full/empty pairs); eight
//     consumer warps do the arithmetic.  The pool's layouts make every piece
//     contiguous: an A block row of one K slice, a B block's 16 ranks of 1024
//     consecutive output columns (32 KiB).
//   * The per-chunk products are 16 x 16 x 16 tiles on the warp-level MMA
//     (bf16 in, fp32 accumulate).  V enters the expand as bf16 hi and lo
//     parts (hi = bf16(v), lo = bf16(v - hi)), about 16 significant bits,
//     products exact in fp32.  This keeps the instruction count per byte of
//     adapter low enough that the kernels are bound by the bulk copies.
//   * Each CTA takes a contiguous share of the work items balanced by cost:
//     shrink items (chunk, rank block, K slice) cost the same; expand items
//     (chunk, 1024 columns) cost by their rank blocks and rows.
//   * One launch of each kernel serves every projection of the call: the
//     CTAs are split between the projections by the bytes of A (B) a row's
//     adapter brings, and each projection's CTAs share out its items.
//
// Every mbarrier wait is bounded (kDevTimeout), and a CTA that gave up waits,
// again bounded, for its bulk copies in flight before it exits.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

#include "lora_device.cuh"
#include "lora_internal.h"
#include "sm100_ptx.cuh"

namespace lora {

namespace {

using namespace sm100;

constexpr int kPipeConsumerWarps = 8;
constexpr int kPipeConsumers = kPipeConsumerWarps * 32;
constexpr int kPipeThreads = kPipeConsumers + 32;  // + the producer warp
constexpr int kChunkRows = 16;                      // positions per chunk: the MMA's N (two n8 tiles)
constexpr int kPipeMaxBlocks = kPipeMaxRank / LORA_BLOCK_ROWS;
constexpr uint64_t kPipeWaitNs = 2000000000ull;
constexpr uint64_t kPipeDrainNs = 100000000ull;

// shrink stages: 16 A rows and up to 16 x rows of kShrStageK k each (one
// bulk copy of 2 KiB per row: the copy engine's per-request cost makes
// requests under 2 KiB fall well short of the SM's share of HBM bandwidth),
// rows padded by 16 bytes so that ldmatrix's eight row addresses hit
// distinct banks
constexpr int kShrStageK = 1024;
constexpr int kShrPitch = kShrStageK * 2 + 16;
constexpr int kShrStageBytes = (LORA_BLOCK_ROWS + kChunkRows) * kShrPitch;
constexpr int kShrStages = 3;
constexpr int kShrRedBytes = 2 * kPipeConsumerWarps * 32 * 8 * 4;  // two buffers of per-warp partials
constexpr size_t kShrSmem = static_cast<size_t>(kShrStages) * kShrStageBytes + kShrRedBytes;

// expand stages: one rank block's B for 1024 output columns
constexpr int kExpCols = 1024;
constexpr int kExpStageBytes = kExpCols * LORA_BLOCK_ROWS * 2;
constexpr int kExpStages = 4;
constexpr int kExpWarps = 16;                   // consumer warps of the expand
constexpr int kExpThreads = (kExpWarps + 1) * 32;
constexpr int kExpGroups = kExpCols / 16 / kExpWarps;  // 16-column groups a consumer warp owns per range
constexpr int kExpMaxVSlots = 6;  // V slots (an item's V stays until its last stage): the producer's lookahead in items
constexpr int kEpiPitch = 20;  // floats a row of the epilogue's 16 x 16 tile: fragment writes free of bank conflicts

static_assert(kShrStageBytes % 16 == 0 && kShrPitch % 16 == 0, "bulk copy destinations 16-byte aligned");
static_assert(kPipeMaxBlocks <= 32, "one block id per producer lane");

// Rows grouped by adapter in shared memory (identical in every CTA of both
// kernels).  Chunk c covers sorted positions [c_begin[c], c_begin[c+1]);
// c_slot[c] = -1 and c_nblk[c] = 0 for the rows without an adapter (they come
// last).  c_pre is the caller's per-chunk cost prefix.
struct GroupSmem {
    unsigned long long key[kPipeMaxRows];
    int32_t pos_row[kPipeMaxRows];
    int32_t c_begin[kPipeMaxRows + 1];
    int32_t c_slot[kPipeMaxRows];
    int32_t c_nblk[kPipeMaxRows];
    int32_t c_pre[kPipeMaxRows + 1];
    int32_t warp_tot[32];
    int32_t n_chunks;
};

// In-place exclusive prefix sum of a[0, n) in shared memory by the whole CTA
// (every thread calls it); returns the total.
__device__ int32_t cta_scan_inplace(int32_t *a, int32_t n, int32_t *warp_tot) {
    const int T = blockDim.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (n + T - 1) / T;
    const int b = min(n, tid * per), e = min(n, b + per);
    int32_t s = 0;
    for (int i = b; i < e; ++i) s += a[i];
    int32_t incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int32_t before = 0, total = 0;
    for (int w = 0; w < T / 32; ++w) {
        if (w < warp) before += warp_tot[w];
        total += warp_tot[w];
    }
    int32_t run = before + incl - s;
    for (int i = b; i < e; ++i) {
        const int32_t v = a[i];
        a[i] = run;
        run += v;
    }
    __syncthreads();
    return total;
}

// Sort key of row m with slot id `id` of rank `r`: (64 - rank blocks) in
// bits 48..54, the slot in bits 16..47, the row in bits 0..15, so that groups
// of many rank blocks come first and a group keeps its rows in order; rows
// without an adapter get 127 << 48.  Invalid ids, empty slots and ranks above
// the table row are recorded when `report` and treated as no adapter.
__device__ __forceinline__ unsigned long long row_key(int32_t m, int32_t id, int32_t r, int32_t max_slots,
                                                      int32_t bps, unsigned long long *status, bool report) {
    const unsigned long long none = (127ull << 48) | static_cast<unsigned long long>(m);
    if (id == -1) return none;
    if (id < -1 || id >= max_slots) {
        if (report) record_error(status, kDevBadAdapter, static_cast<uint32_t>(m));
        return none;
    }
    if (r <= 0) {
        if (report) record_error(status, kDevEmptySlot, static_cast<uint32_t>(m));
        return none;
    }
    if (r > bps * LORA_BLOCK_ROWS) {
        if (report) record_error(status, kDevBadBlock, static_cast<uint32_t>(id));
        return none;
    }
    const int32_t nblk = (r + LORA_BLOCK_ROWS - 1) / LORA_BLOCK_ROWS;
    return (static_cast<unsigned long long>(64 - nblk) << 48) | (static_cast<unsigned long long>(id) << 16) |
           static_cast<unsigned long long>(m);
}

__device__ __forceinline__ unsigned long long shfl_xor_u64(unsigned long long v, int m) {
    const uint32_t lo = __shfl_xor_sync(0xffffffffu, static_cast<uint32_t>(v), m);
    const uint32_t hi = __shfl_xor_sync(0xffffffffu, static_cast<uint32_t>(v >> 32), m);
    return (static_cast<unsigned long long>(hi) << 32) | lo;
}

// Bitonic sort (ascending) of kPipeMaxRows = 512 keys: thread t < 256 holds
// positions 2t and 2t + 1 in e[0], e[1].  Exchanges between positions less
// than 64 apart stay in a warp (shuffles, or within the thread); only the
// six wider steps go through shared memory `sk`.  Every thread of the CTA
// calls it.
__device__ void bitonic_sort_512(unsigned long long (&e)[2], unsigned long long *sk) {
    static_assert(kPipeMaxRows == 512 && kPipeThreads >= 256, "two keys a thread over the first 256 threads");
    const int t = threadIdx.x;
    const bool act = t < 256;
    for (int k = 2; k <= 512; k <<= 1) {
        int j = k >> 1;
        if (j >= 64) {
            if (act) {
                sk[2 * t] = e[0];
                sk[2 * t + 1] = e[1];
            }
            __syncthreads();
            for (; j >= 64; j >>= 1) {
                if (act) {
                    const int lo = (t / j) * 2 * j + (t % j), hi = lo + j;
                    const unsigned long long a = sk[lo], b = sk[hi];
                    if ((a > b) == ((lo & k) == 0)) {
                        sk[lo] = b;
                        sk[hi] = a;
                    }
                }
                __syncthreads();
            }
            if (act) {
                e[0] = sk[2 * t];
                e[1] = sk[2 * t + 1];
            }
        }
        if (act) {
            for (; j >= 2; j >>= 1) {
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int pos = 2 * t + q;
                    const unsigned long long v = shfl_xor_u64(e[q], j >> 1);
                    const bool lower = (pos & j) == 0, asc = (pos & k) == 0;
                    e[q] = (lower == asc) ? (e[q] < v ? e[q] : v) : (e[q] > v ? e[q] : v);
                }
            }
            const bool asc = ((2 * t) & k) == 0;
            const unsigned long long lo = e[0] < e[1] ? e[0] : e[1], hi = e[0] < e[1] ? e[1] : e[0];
            e[0] = asc ? lo : hi;
            e[1] = asc ? hi : lo;
        }
    }
}

// The rows' chunk table of this CTA (every thread calls it; M <= kPipeMaxRows).
__device__ void group_rows_in_cta(GroupSmem &gs, int32_t M, const int32_t *row_slot, const int32_t *ranks,
                                  int32_t max_slots, int32_t bps, unsigned long long *status, bool report) {
    const int tid = threadIdx.x, T = blockDim.x;
    unsigned long long e[2] = {~0ull, ~0ull};
    if (tid < 256) {
        // both rows' ids, then both ranks: two round trips, not four
        int32_t id[2], r[2] = {0, 0};
#pragma unroll
        for (int q = 0; q < 2; ++q) id[q] = 2 * tid + q < M ? row_slot[2 * tid + q] : -1;
#pragma unroll
        for (int q = 0; q < 2; ++q)
            if (id[q] >= 0 && id[q] < max_slots) r[q] = ranks[id[q]];
#pragma unroll
        for (int q = 0; q < 2; ++q)
            if (2 * tid + q < M) e[q] = row_key(2 * tid + q, id[q], r[q], max_slots, bps, status, report);
    }
    bitonic_sort_512(e, gs.key);
    if (tid < 256) {
        gs.key[2 * tid] = e[0];
        gs.key[2 * tid + 1] = e[1];
    }
    __syncthreads();
    // a chunk starts at a new group and every kChunkRows positions into one
    for (int32_t i = tid; i < M; i += T) {
        const unsigned long long g = gs.key[i] >> 16;
        gs.pos_row[i] = static_cast<int32_t>(gs.key[i] & 0xFFFFull);
        int32_t lo = 0, hi = i;  // first position of the group: lower bound of g << 16
        while (lo < hi) {
            const int32_t mid = (lo + hi) >> 1;
            if ((gs.key[mid] >> 16) < g) lo = mid + 1;
            else hi = mid;
        }
        gs.c_pre[i] = (i - lo) % kChunkRows == 0;
    }
    __syncthreads();
    const int32_t C = cta_scan_inplace(gs.c_pre, M, gs.warp_tot);
    for (int32_t i = tid; i < M; i += T) {
        const bool first = i + 1 == M ? (gs.c_pre[i] < C) : gs.c_pre[i + 1] != gs.c_pre[i];
        if (!first) continue;
        const int32_t c = gs.c_pre[i];
        const unsigned long long key = gs.key[i];
        const int32_t cls = static_cast<int32_t>(key >> 48);
        gs.c_begin[c] = i;
        gs.c_slot[c] = cls == 127 ? -1 : static_cast<int32_t>((key >> 16) & 0xFFFFFFFFull);
        gs.c_nblk[c] = cls == 127 ? 0 : 64 - cls;
    }
    if (tid == 0) {
        gs.c_begin[C] = M;
        gs.n_chunks = C;
    }
    __syncthreads();
}

// One projection's row grouping as pipe_group_kernel leaves it in global
// memory: the fields of GroupSmem that the pipelined kernels read.
struct PipeGroupTable {
    int32_t n_chunks;
    int32_t pos_row[kPipeMaxRows];
    int32_t c_begin[kPipeMaxRows + 1];
    int32_t c_slot[kPipeMaxRows];
    int32_t c_nblk[kPipeMaxRows];
};

// A CTA's copy of a grouping table (every thread calls it).
__device__ void load_group_table(GroupSmem &gs, const PipeGroupTable *t, int32_t M) {
    const int tid = threadIdx.x, T = blockDim.x;
    const int32_t C = t->n_chunks;
    for (int32_t i = tid; i < M; i += T) gs.pos_row[i] = t->pos_row[i];
    for (int32_t i = tid; i <= C; i += T) gs.c_begin[i] = t->c_begin[i];
    for (int32_t i = tid; i < C; i += T) {
        gs.c_slot[i] = t->c_slot[i];
        gs.c_nblk[i] = t->c_nblk[i];
    }
    if (tid == 0) gs.n_chunks = C;
    __syncthreads();
}

struct PipeGroupParams {
    int32_t M;
    const int32_t *row_slot;
    const int32_t *ranks[LORA_MAX_PROJ];
    int32_t max_slots[LORA_MAX_PROJ], bps[LORA_MAX_PROJ];
    PipeGroupTable *tables;  // [projections]
    unsigned long long *status;
};

// CTA q groups the rows for projection q (the ranks come from its pool) and
// writes the table both pipelined kernels of that projection read; invalid
// ids are recorded once, by CTA 0.
__global__ void __launch_bounds__(kPipeThreads, 1) pipe_group_kernel(const PipeGroupParams p) {
    __shared__ GroupSmem gs;
    // the row ids may come from the kernel before (segments to rows)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int q = blockIdx.x;
    group_rows_in_cta(gs, p.M, p.row_slot, p.ranks[q], p.max_slots[q], p.bps[q], p.status, q == 0);
    PipeGroupTable *t = p.tables + q;
    const int tid = threadIdx.x, T = blockDim.x;
    const int32_t C = gs.n_chunks;
    for (int32_t i = tid; i < p.M; i += T) t->pos_row[i] = gs.pos_row[i];
    for (int32_t i = tid; i <= C; i += T) t->c_begin[i] = gs.c_begin[i];
    for (int32_t i = tid; i < C; i += T) {
        t->c_slot[i] = gs.c_slot[i];
        t->c_nblk[i] = gs.c_nblk[i];
    }
    if (tid == 0) t->n_chunks = C;
}

// Lane j's block id of chunk c (its slot's table entry j; 0 past the chunk's
// rank blocks, past the last chunk, or for rows without an adapter).  The
// producers load the next chunk's ids while they stream the current one.
__device__ __forceinline__ int32_t chunk_block_id(const GroupSmem &gs, int32_t c, int32_t C, const int32_t *table,
                                                  int32_t bps, int lane) {
    if (c >= C) return 0;
    const int32_t slot = gs.c_slot[c];
    return slot >= 0 && lane < gs.c_nblk[c] ? table[static_cast<size_t>(slot) * bps + lane] : 0;
}

// Wait for every bulk copy this CTA issued into its stages to land (bounded):
// stage uses [issued - S, issued) may still be in flight after a time-out.
__device__ void drain_stages(uint64_t *full, int S, int64_t issued) {
    for (int64_t i = issued - S > 0 ? issued - S : 0; i < issued; ++i)
        (void)mbar_wait_bounded(&full[i % S], static_cast<uint32_t>((i / S) & 1), kPipeDrainNs);
}

// ---------------------------------------------------------------------------
// shrink
// ---------------------------------------------------------------------------

struct PipeShrinkParams {
    int32_t M, K, ldx;
    const __nv_bfloat16 *x;
    const int32_t *row_slot;
    const __nv_bfloat16 *a_arena;
    const int32_t *table;
    const int32_t *ranks;
    int32_t max_slots, bps, num_blocks;
    float *V;              // [ksplit][M][ldv] fp32, rows in sorted-position order
    int32_t ldv;           // the pool's max_rank
    int32_t ksplit;        // K slices = planes of V
    int32_t kc_len;        // k per slice (a multiple of 8)
    size_t plane_stride;   // elements between planes
    int32_t *counters;     // split-K tile counters of the GEMM that follows, zeroed here
    int32_t n_counters;
    const PipeGroupTable *group;  // the rows grouped by adapter (pipe_group_kernel)
    unsigned long long *status;
};

// One launch of a pipelined kernel over several projections of the same x:
// CTAs [cta_begin[q], cta_begin[q + 1]) serve projection q, each with its own
// parameters (pool, V, ycorr, grouping table).
template <typename P>
struct PipeMulti {
    P proj[LORA_MAX_PROJ];
    int32_t n_proj;
    int32_t cta_begin[LORA_MAX_PROJ + 1];
};

// This CTA's projection, its index among that projection's CTAs and their count.
template <typename P>
__device__ __forceinline__ const P &pipe_projection(const PipeMulti<P> &m, int32_t *cta, int32_t *ncta) {
    int q = 0;
    while (q + 1 < m.n_proj && static_cast<int32_t>(blockIdx.x) >= m.cta_begin[q + 1]) ++q;
    *cta = static_cast<int32_t>(blockIdx.x) - m.cta_begin[q];
    *ncta = m.cta_begin[q + 1] - m.cta_begin[q];
    return m.proj[q];
}

// Work items u = (chunk, rank block jb, K slice kc), kc fastest, each costing
// the row copies of its stages (16 A rows and the chunk's x rows); the CTA
// takes the items whose cost starts in its equal share.  An item is streamed
// in stages of kShrStageK k: the
// block's 16 A rows and the chunk's x rows.  Consumer warp w takes the
// stage's 16-k steps w, w + 8, ...; at the item's last stage the warps' 16 x
// 16 partial tiles are summed through shared memory and stored to plane kc.
__global__ void __launch_bounds__(kPipeThreads, 1)
pipe_shrink_kernel(const __grid_constant__ PipeMulti<PipeShrinkParams> pm) {
    int32_t cta, ncta;
    const PipeShrinkParams p = pipe_projection(pm, &cta, &ncta);  // in registers: read in the hot loops
    extern __shared__ __align__(128) uint8_t pipe_smem[];
    __shared__ GroupSmem gs;
    __shared__ __align__(8) uint64_t full[kShrStages], empty[kShrStages], redbar[2];
    __shared__ int4 meta[kShrStages];
    __shared__ int32_t issued_s;
    uint8_t *stages = pipe_smem;
    float *red = reinterpret_cast<float *>(pipe_smem + static_cast<size_t>(kShrStages) * kShrStageBytes);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // the row ids may come from the kernel before (segments to rows), and the
    // GEMM before may still read the split-K counters zeroed here
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (blockIdx.x == 0)
        for (int32_t c = tid; c < p.n_counters; c += kPipeThreads) p.counters[c] = 0;
    if (tid == 0) {
        for (int s = 0; s < kShrStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kPipeConsumerWarps);
        }
        mbar_init(&redbar[0], kPipeConsumerWarps);
        mbar_init(&redbar[1], kPipeConsumerWarps);
        fence_mbar_init();
        issued_s = 0;
    }
    load_group_table(gs, p.group, p.M);
    const int32_t C = gs.n_chunks;
    // an item's cost: the row copies of its stages, the block's 16 A rows
    // and the chunk's x rows
    for (int32_t c = tid; c < C; c += kPipeThreads)
        gs.c_pre[c] = gs.c_nblk[c] * p.ksplit * (LORA_BLOCK_ROWS + gs.c_begin[c + 1] - gs.c_begin[c]);
    __syncthreads();
    const int32_t total = cta_scan_inplace(gs.c_pre, C, gs.warp_tot);
    if (tid == 0) gs.c_pre[C] = total;
    __syncthreads();
    // this CTA's items: those whose cost starts in [w_lo, w_hi)
    const int64_t w_lo = static_cast<int64_t>(cta) * total / ncta;
    const int64_t w_hi = static_cast<int64_t>(cta + 1) * total / ncta;

    if (warp == kPipeConsumerWarps) {
        // ---- producer warp: lanes 0-15 copy the A rows, lanes 16-31 the x rows
        int32_t ch = 0, i = 0;  // the chunk of the CTA's first item and the item's index in it
        if (C > 0) {
            int32_t lo = 0, hi = C - 1;  // the last chunk whose cost starts at or before w_lo
            while (lo < hi) {
                const int32_t mid = (lo + hi + 1) >> 1;
                if (gs.c_pre[mid] <= w_lo) lo = mid;
                else hi = mid - 1;
            }
            ch = lo;
            const int32_t w = LORA_BLOCK_ROWS + gs.c_begin[ch + 1] - gs.c_begin[ch];
            i = static_cast<int32_t>((w_lo - gs.c_pre[ch] + w - 1) / w);
        }
        int32_t it = 0;
        bool ok = true;
        // blk_next: the block ids of chunk next_ch, loaded one chunk ahead
        int32_t cur_ch = -1, blk_lane = 0, next_ch = ch, blk_next = chunk_block_id(gs, ch, C, p.table, p.bps, lane);
        while (ok && ch < C) {
            const int32_t p0 = gs.c_begin[ch], R = gs.c_begin[ch + 1] - p0;
            if (i >= gs.c_nblk[ch] * p.ksplit) {  // past the chunk's items (none for rows without an adapter)
                ++ch;
                i = 0;
                continue;
            }
            if (gs.c_pre[ch] + static_cast<int64_t>(i) * (LORA_BLOCK_ROWS + R) >= w_hi) break;
            const int32_t local = i++;
            if (ch != cur_ch) {  // a new chunk: its ids were loaded one chunk ago, unless chunks were skipped
                blk_lane = ch == next_ch ? blk_next : chunk_block_id(gs, ch, C, p.table, p.bps, lane);
                cur_ch = ch;
                next_ch = ch + 1;
                blk_next = chunk_block_id(gs, next_ch, C, p.table, p.bps, lane);
            }
            const int32_t jb = local / p.ksplit, kc = local - jb * p.ksplit;
            const int32_t blk = __shfl_sync(0xffffffffu, blk_lane, jb);
            if (blk < 0 || blk >= p.num_blocks) continue;  // reported by the expand, which zeroes these rows
            const int32_t xr = lane - LORA_BLOCK_ROWS;
            const __nv_bfloat16 *src =
                lane < LORA_BLOCK_ROWS
                    ? p.a_arena + (static_cast<size_t>(blk) * LORA_BLOCK_ROWS + lane) * p.K
                    : (xr < R ? p.x + static_cast<size_t>(gs.pos_row[p0 + xr]) * p.ldx : nullptr);
            const int32_t k_begin = kc * p.kc_len, k_end = min(p.K, k_begin + p.kc_len);
            for (int32_t k0 = k_begin; k0 < k_end; k0 += kShrStageK) {
                const int32_t len = min(kShrStageK, k_end - k0);
                const int s = it % kShrStages, use = it / kShrStages;
                bool got = true;
                if (lane == 0 && use > 0) got = mbar_wait_bounded(&empty[s], (use - 1) & 1, kPipeWaitNs);
                if (!__shfl_sync(0xffffffffu, got, 0)) {
                    if (lane == 0) record_error(p.status, kDevTimeout, 20);
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    meta[s] = make_int4(ch, jb, kc, len | (k0 + kShrStageK >= k_end ? 1 << 16 : 0));
                    mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(LORA_BLOCK_ROWS + R) * len * 2);
                }
                __syncwarp();
                if (src) bulk_load(stages + static_cast<size_t>(s) * kShrStageBytes + lane * kShrPitch, src + k0,
                                   static_cast<uint32_t>(len) * 2, &full[s]);
                ++it;
            }
        }
        if (ok) {  // end marker
            const int s = it % kShrStages, use = it / kShrStages;
            bool got = true;
            if (lane == 0 && use > 0) got = mbar_wait_bounded(&empty[s], (use - 1) & 1, kPipeWaitNs);
            if (lane == 0) {
                if (got) {
                    meta[s] = make_int4(-1, 0, 0, 0);
                    mbar_arrive(&full[s]);
                    ++it;
                } else {
                    record_error(p.status, kDevTimeout, 20);
                }
            }
            it = __shfl_sync(0xffffffffu, it, 0);
        }
        if (lane == 0) issued_s = it;
    } else {
        // ---- consumer warps
        const uint32_t a_off = ((lane & 7) + ((lane >> 3) & 1) * 8) * kShrPitch + (lane >> 4) * 16;
        const int32_t xrow = (lane & 7) + (lane >> 4) * 8;
        const uint32_t xk_off = ((lane >> 3) & 1) * 16;
        // four accumulator sets (by 16-k step mod 4) so that consecutive MMAs
        // do not wait on one another; summed at the item's end
        float acc[4][2][4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int q = 0; q < 2; ++q)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[u][q][e] = 0.0f;
        int32_t it = 0, nred = 0;
        while (true) {
            const int s = it % kShrStages;
            if (!mbar_wait_bounded(&full[s], (it / kShrStages) & 1, kPipeWaitNs)) {
                if (lane == 0) record_error(p.status, kDevTimeout, 21);
                break;
            }
            const int4 m = meta[s];
            if (m.x < 0) break;
            const int32_t ch = m.x, jb = m.y, kc = m.z, len = m.w & 0xFFFF;
            const int32_t p0 = gs.c_begin[ch], R = gs.c_begin[ch + 1] - p0;
            const uint32_t sb = smem_u32(stages + static_cast<size_t>(s) * kShrStageBytes);
            const uint32_t a_addr = sb + a_off;
            // x rows past the chunk read row 0 (their columns of the product are dropped)
            const uint32_t x_addr = sb + (LORA_BLOCK_ROWS + (xrow < R ? xrow : 0)) * kShrPitch + xk_off;
            const int32_t steps = (len + 15) >> 4;
            const bool two = R > 8;  // the second 8-row tile only when the chunk has rows there
            for (int32_t st0 = warp; st0 < steps; st0 += 4 * kPipeConsumerWarps) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int32_t st = st0 + u * kPipeConsumerWarps;
                    if (st >= steps) break;
                    uint32_t a[4], b[4];
                    ldmatrix_x4(a, a_addr + st * 32);
                    ldmatrix_x4(b, x_addr + st * 32);
                    if (st * 16 + 16 > len) {  // a ragged slice end: k 8..15 of the step lie past it
                        a[2] = a[3] = 0u;
                        b[1] = b[3] = 0u;
                    }
                    mma_16816_bf16(acc[u][0], a, b[0], b[1]);
                    if (two) mma_16816_bf16(acc[u][1], a, b[2], b[3]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_relaxed(&empty[s]);
            ++it;
            if (m.w >> 16) {
                // the item's last stage: sum the eight warps' partial tiles
                const int buf = nred & 1;
                float t4[2][4];
#pragma unroll
                for (int q = 0; q < 2; ++q)
#pragma unroll
                    for (int e = 0; e < 4; ++e) t4[q][e] = (acc[0][q][e] + acc[1][q][e]) + (acc[2][q][e] + acc[3][q][e]);
                float4 *mine = reinterpret_cast<float4 *>(red + ((buf * kPipeConsumerWarps + warp) * 32 + lane) * 8);
                mine[0] = make_float4(t4[0][0], t4[0][1], t4[0][2], t4[0][3]);
                mine[1] = make_float4(t4[1][0], t4[1][1], t4[1][2], t4[1][3]);
                __syncwarp();
                if (lane == 0) mbar_arrive(&redbar[buf]);
                if (!mbar_wait_bounded(&redbar[buf], (nred >> 1) & 1, kPipeWaitNs)) {
                    if (lane == 0) record_error(p.status, kDevTimeout, 22);
                    break;
                }
                const int e = tid;  // one (lane, register) of the tiles per consumer thread
                float v = 0.0f;
#pragma unroll
                for (int w = 0; w < kPipeConsumerWarps; ++w) v += red[(buf * kPipeConsumerWarps + w) * 256 + e];
                const int le = e >> 3, reg = e & 7, q = reg >> 2, r4 = reg & 3;
                const int j = (le >> 2) + 8 * (r4 >> 1);           // rank row of the block
                const int row = 8 * q + 2 * (le & 3) + (r4 & 1);  // position in the chunk
                if (row < R)
                    p.V[kc * p.plane_stride + static_cast<size_t>(p0 + row) * p.ldv + jb * LORA_BLOCK_ROWS + j] = v;
#pragma unroll
                for (int u = 0; u < 4; ++u)
#pragma unroll
                    for (int q2 = 0; q2 < 2; ++q2)
#pragma unroll
                        for (int e2 = 0; e2 < 4; ++e2) acc[u][q2][e2] = 0.0f;
                ++nred;
            }
        }
    }
    __syncthreads();
    if (tid == 0) drain_stages(full, kShrStages, issued_s);
}

// ---------------------------------------------------------------------------
// expand
// ---------------------------------------------------------------------------

constexpr int kExpVSlotFloatsMax = kChunkRows * kPipeMaxRank;  // one V plane
// dynamic shared memory of the expand: the B stages and as many V slots (2 to
// kExpMaxVSlots) as fit beside them and the static arrays
constexpr size_t kExpSmemMax = 180 * 1024;
static_assert(static_cast<size_t>(kExpStages) * kExpStageBytes + 2 * sizeof(float) * kExpVSlotFloatsMax <= kExpSmemMax,
              "two V slots of the largest size fit");

struct PipeExpandParams {
    int32_t M, N;
    const int32_t *row_slot;
    const __nv_bfloat16 *b_arena;
    const int32_t *table;
    const int32_t *ranks;
    const float *scales;
    int32_t max_slots, bps, num_blocks;
    const float *V;        // [ksplit][M][ldv], rows in sorted-position order
    int32_t ldv, ksplit;
    size_t plane_stride;
    int32_t vslot_floats;  // ksplit * kChunkRows * ldv
    int32_t n_vslots;      // 2 .. kExpMaxVSlots
    float *ycorr;          // [M][N]
    const PipeGroupTable *group;  // the rows grouped by adapter (pipe_group_kernel)
    unsigned long long *status;
};

// v (two adjacent values) as bf16 hi and lo parts, packed for the MMA.
__device__ __forceinline__ void split_bf16x2(float a, float b, uint32_t &hi, uint32_t &lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(a - hf.x, b - hf.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

// Work items (chunk, 1024-column range), ranges fastest, each with a cost
// from its rank blocks and rows; the CTA takes the items whose cost start
// lies in its share.  Stage jb of an item holds rank block jb's B for the range; the
// first stage also brings the chunk's V planes into a V slot (up to four
// slots, so that the producer runs several items ahead), from which every
// consumer thread builds its MMA fragments of block jb (planes summed, hi and
// lo parts).  Consumer warp w owns the 16-column groups w, w +
// 8, ... of the range: out[n, i] += B[n, 16 jb + j] V[i, 16 jb + j] as 16 x 8 x
// 16 tiles for the chunk's two halves of 8 positions.  Items of rows without
// an adapter (or with a corrupt block entry) write zeros.
__global__ void __launch_bounds__(kExpThreads, 1)
pipe_expand_kernel(const __grid_constant__ PipeMulti<PipeExpandParams> pm) {
    int32_t cta, ncta;
    const PipeExpandParams p = pipe_projection(pm, &cta, &ncta);  // in registers: read in the hot loops
    extern __shared__ __align__(128) uint8_t pipe_smem[];
    __shared__ GroupSmem gs;
    __shared__ __align__(8) uint64_t full[kExpStages], empty[kExpStages], vempty[kExpMaxVSlots];
    __shared__ float c_scale[kPipeMaxRows];
    __shared__ int4 meta[kExpStages];
    __shared__ __align__(16) float epi[kExpWarps][16 * kEpiPitch];
    __shared__ int32_t issued_s;
    uint8_t *bstage = pipe_smem;
    float *vslots = reinterpret_cast<float *>(pipe_smem + static_cast<size_t>(kExpStages) * kExpStageBytes);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // the GEMM that follows may launch now; it reads ycorr only after this
    // grid has completed (griddepcontrol.wait)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (tid == 0) {
        for (int s = 0; s < kExpStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kExpWarps);
        }
        for (int v = 0; v < kExpMaxVSlots; ++v) mbar_init(&vempty[v], kExpWarps);
        fence_mbar_init();
        issued_s = 0;
    }
    // the grouping comes from pipe_group_kernel, which completed before the
    // shrink this grid follows passed its own grid-dependency wait
    load_group_table(gs, p.group, p.M);
    const int32_t C = gs.n_chunks;
    const int32_t n_ranges = (p.N + kExpCols - 1) / kExpCols;
    // cost of an item in quarter stages: 4 per rank block (its B copy and
    // MMAs), 2 fixed, and its rows' ycorr stores (16 rows x 4 KiB ~ two stages)
    for (int32_t c = tid; c < C; c += kExpThreads) {
        gs.c_pre[c] = 4 * gs.c_nblk[c] + 2 + (gs.c_begin[c + 1] - gs.c_begin[c] + 1) / 2;
        c_scale[c] = gs.c_slot[c] >= 0 ? p.scales[gs.c_slot[c]] : 0.0f;
    }
    __syncthreads();
    const int32_t wsum = cta_scan_inplace(gs.c_pre, C, gs.warp_tot);
    if (tid == 0) gs.c_pre[C] = wsum;
    __syncthreads();
    const int64_t total = static_cast<int64_t>(n_ranges) * wsum;
    const int64_t c_lo = static_cast<int64_t>(cta) * total / ncta;
    const int64_t c_hi = static_cast<int64_t>(cta + 1) * total / ncta;

    if (warp == kExpWarps) {
        // ---- producer warp
        int32_t ch = 0, nr = 0;
        if (C > 0) {
            int32_t lo = 0, hi = C - 1;  // the last chunk whose first item starts at or before c_lo
            while (lo < hi) {
                const int32_t mid = (lo + hi + 1) >> 1;
                if (static_cast<int64_t>(n_ranges) * gs.c_pre[mid] <= c_lo) lo = mid;
                else hi = mid - 1;
            }
            ch = lo;
            const int32_t w = gs.c_pre[ch + 1] - gs.c_pre[ch];
            const int64_t off = c_lo - static_cast<int64_t>(n_ranges) * gs.c_pre[ch];
            nr = static_cast<int32_t>((off + w - 1) / w);
            if (nr >= n_ranges) {
                ++ch;
                nr = 0;
            }
        }
        bool waited = false, ok = true;
        int32_t it = 0, nv = 0;
        int32_t cur_ch = -1, blk = 0, blk_next = chunk_block_id(gs, ch, C, p.table, p.bps, lane);
        bool blocks_ok = true;
        while (ok && ch < C) {
            const int32_t w = gs.c_pre[ch + 1] - gs.c_pre[ch];
            if (static_cast<int64_t>(n_ranges) * gs.c_pre[ch] + static_cast<int64_t>(nr) * w >= c_hi) break;
            const int32_t slot = gs.c_slot[ch], nblk = gs.c_nblk[ch];
            const int32_t p0 = gs.c_begin[ch], R = gs.c_begin[ch + 1] - p0;
            const int32_t n0 = nr * kExpCols, ncols = min(kExpCols, p.N - n0);
            if (ch != cur_ch) {  // a new chunk: its ids were loaded one chunk ago
                cur_ch = ch;
                blk = blk_next;
                blk_next = chunk_block_id(gs, ch + 1, C, p.table, p.bps, lane);
                blocks_ok = __all_sync(0xffffffffu, lane >= nblk || (blk >= 0 && blk < p.num_blocks));
            }
            const bool valid = slot >= 0 && blocks_ok;
            if (slot >= 0 && !valid && nr == 0 && lane == 0)
                record_error(p.status, kDevBadBlock, static_cast<uint32_t>(slot));
            if (!valid) {
                // rows without a correction: one stage with no copies
                const int s = it % kExpStages, use = it / kExpStages;
                bool got = true;
                if (lane == 0 && use > 0) got = mbar_wait_bounded(&empty[s], (use - 1) & 1, kPipeWaitNs);
                if (!__shfl_sync(0xffffffffu, got, 0)) {
                    if (lane == 0) record_error(p.status, kDevTimeout, 23);
                    ok = false;
                    break;
                }
                if (!waited) {  // the GEMM before may still read ycorr
                    asm volatile("griddepcontrol.wait;" ::: "memory");
                    waited = true;
                }
                if (lane == 0) {
                    meta[s] = make_int4(ch, nr, -1, 0);
                    mbar_arrive(&full[s]);
                }
                __syncwarp();
                ++it;
            } else {
                const int vs = nv % p.n_vslots, vuse = nv / p.n_vslots;
                bool got = true;
                if (lane == 0 && vuse > 0) got = mbar_wait_bounded(&vempty[vs], (vuse - 1) & 1, kPipeWaitNs);
                if (!__shfl_sync(0xffffffffu, got, 0)) {
                    if (lane == 0) record_error(p.status, kDevTimeout, 24);
                    ok = false;
                    break;
                }
                for (int32_t jb = 0; jb < nblk; ++jb) {
                    const int s = it % kExpStages, use = it / kExpStages;
                    got = true;
                    if (lane == 0 && use > 0) got = mbar_wait_bounded(&empty[s], (use - 1) & 1, kPipeWaitNs);
                    if (!__shfl_sync(0xffffffffu, got, 0)) {
                        if (lane == 0) record_error(p.status, kDevTimeout, 23);
                        ok = false;
                        break;
                    }
                    const uint32_t vbytes =
                        jb == 0 ? static_cast<uint32_t>(p.ksplit) * R * p.ldv * static_cast<uint32_t>(sizeof(float)) : 0u;
                    if (lane == 0) {
                        meta[s] = make_int4(ch, nr, jb, vs);
                        mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(ncols) * 32u + vbytes);
                    }
                    __syncwarp();
                    const int32_t b = __shfl_sync(0xffffffffu, blk, jb);
                    if (lane == 0)
                        bulk_load(bstage + static_cast<size_t>(s) * kExpStageBytes,
                                  p.b_arena + (static_cast<size_t>(b) * p.N + n0) * LORA_BLOCK_ROWS,
                                  static_cast<uint32_t>(ncols) * 32u, &full[s]);
                    if (jb == 0) {
                        if (!waited) {  // V comes from the shrink before
                            asm volatile("griddepcontrol.wait;" ::: "memory");
                            waited = true;
                        }
                        if (lane < p.ksplit)
                            bulk_load(vslots + static_cast<size_t>(vs) * p.vslot_floats +
                                          static_cast<size_t>(lane) * kChunkRows * p.ldv,
                                      p.V + lane * p.plane_stride + static_cast<size_t>(p0) * p.ldv,
                                      static_cast<uint32_t>(R) * p.ldv * static_cast<uint32_t>(sizeof(float)),
                                      &full[s]);
                    }
                    ++it;
                }
                ++nv;
            }
            if (++nr == n_ranges) {
                ++ch;
                nr = 0;
            }
        }
        if (ok) {  // end marker
            const int s = it % kExpStages, use = it / kExpStages;
            bool got = true;
            if (lane == 0 && use > 0) got = mbar_wait_bounded(&empty[s], (use - 1) & 1, kPipeWaitNs);
            if (lane == 0) {
                if (got) {
                    meta[s] = make_int4(-1, 0, 0, 0);
                    mbar_arrive(&full[s]);
                    ++it;
                } else {
                    record_error(p.status, kDevTimeout, 23);
                }
            }
            it = __shfl_sync(0xffffffffu, it, 0);
        }
        if (lane == 0) issued_s = it;
    } else {
        // ---- consumer warps
        const int g = lane >> 2, t = lane & 3;
        const uint32_t a_off = ((lane & 7) + ((lane >> 3) & 1) * 8) * 32 + (lane >> 4) * 16;
        const bool vec_out = (p.N & 3) == 0;  // ycorr rows 16-byte aligned
        float acc[kExpGroups][2][4];
        int32_t it = 0, nblk = 0, R = 0, p0 = 0;
        float sc = 0.0f;
        while (true) {
            const int s = it % kExpStages;
            if (!mbar_wait_bounded(&full[s], (it / kExpStages) & 1, kPipeWaitNs)) {
                if (lane == 0) record_error(p.status, kDevTimeout, 25);
                break;
            }
            const int4 m = meta[s];
            if (m.x < 0) break;
            const int32_t ch = m.x, jb = m.z;
            const int32_t n0 = m.y * kExpCols, ncols = min(kExpCols, p.N - n0);
            if (jb < 0) {
                __syncwarp();
                if (lane == 0) mbar_arrive_relaxed(&empty[s]);
                ++it;
                const int32_t z0 = gs.c_begin[ch], zr = gs.c_begin[ch + 1] - z0;
                for (int32_t i = 0; i < zr; ++i) {
                    float *dst = p.ycorr + static_cast<size_t>(gs.pos_row[z0 + i]) * p.N + n0;
                    if (vec_out) {
                        for (int32_t c = 4 * tid; c < ncols; c += 4 * (kExpWarps * 32)) {
                            if (c + 4 <= ncols) *reinterpret_cast<float4 *>(dst + c) = make_float4(0.f, 0.f, 0.f, 0.f);
                            else
                                for (int32_t c2 = c; c2 < ncols; ++c2) dst[c2] = 0.0f;
                        }
                    } else {
                        for (int32_t c = tid; c < ncols; c += (kExpWarps * 32)) dst[c] = 0.0f;
                    }
                }
                continue;
            }
            if (jb == 0) {
                p0 = gs.c_begin[ch];
                R = gs.c_begin[ch + 1] - p0;
                nblk = gs.c_nblk[ch];
                sc = c_scale[ch];
#pragma unroll
                for (int i = 0; i < kExpGroups; ++i)
#pragma unroll
                    for (int q = 0; q < 2; ++q)
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc[i][q][e] = 0.0f;
            }
            // rank block jb of V (planes summed) as hi and lo MMA fragments; the
            // V slot landed with the item's first stage and stays until its last.
            // A chunk of at most 4 rows packs both parts into one 8-wide tile:
            // MMA column n < 4 takes hi of row n, column n >= 4 lo of row n - 4.
            const bool packed = R <= 4;
            uint32_t fh[2][2], fl[2][2];
            {
                const float *vsl = vslots + static_cast<size_t>(m.w) * p.vslot_floats + jb * LORA_BLOCK_ROWS + 2 * t;
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    float f0 = 0.0f, f1 = 0.0f, f2 = 0.0f, f3 = 0.0f;
                    const int row = packed ? (q == 0 ? (g & 3) : kChunkRows) : 8 * q + g;
                    if (row < R) {
                        for (int pl = 0; pl < p.ksplit; ++pl) {
                            const float *src = vsl + (pl * kChunkRows + row) * p.ldv;
                            const float2 lo2 = *reinterpret_cast<const float2 *>(src);
                            const float2 hi2 = *reinterpret_cast<const float2 *>(src + 8);
                            f0 += lo2.x;
                            f1 += lo2.y;
                            f2 += hi2.x;
                            f3 += hi2.y;
                        }
                    }
                    split_bf16x2(f0, f1, fh[q][0], fl[q][0]);
                    split_bf16x2(f2, f3, fh[q][1], fl[q][1]);
                }
                if (packed && g >= 4) {  // lanes of MMA columns 4..7 carry the lo parts
                    fh[0][0] = fl[0][0];
                    fh[0][1] = fl[0][1];
                }
            }
            const uint32_t sb = smem_u32(bstage + static_cast<size_t>(s) * kExpStageBytes) + a_off;
            // the eight column groups' B fragments first, then the MMAs group by
            // group so that consecutive MMAs never share an accumulator
            uint32_t a[kExpGroups][4];
#pragma unroll
            for (int i = 0; i < kExpGroups; ++i) {
                const int32_t nl = (warp + kExpWarps * i) * 16;
                if (nl < ncols) {
                    ldmatrix_x4(a[i], sb + nl * 32);
                } else {  // past a ragged range end: never stored
                    a[i][0] = a[i][1] = a[i][2] = a[i][3] = 0u;
                }
            }
#pragma unroll
            for (int i = 0; i < kExpGroups; ++i) mma_16816_bf16(acc[i][0], a[i], fh[0][0], fh[0][1]);
            if (!packed) {
#pragma unroll
                for (int i = 0; i < kExpGroups; ++i) mma_16816_bf16(acc[i][0], a[i], fl[0][0], fl[0][1]);
            }
            if (R > 8) {  // the second 8-row tile only when the chunk has rows there
#pragma unroll
                for (int i = 0; i < kExpGroups; ++i) mma_16816_bf16(acc[i][1], a[i], fh[1][0], fh[1][1]);
#pragma unroll
                for (int i = 0; i < kExpGroups; ++i) mma_16816_bf16(acc[i][1], a[i], fl[1][0], fl[1][1]);
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive_relaxed(&empty[s]);
                if (jb == nblk - 1) mbar_arrive_relaxed(&vempty[m.w]);
            }
            ++it;
            if (jb == nblk - 1) {
                if (packed) {
                    // hi (columns 0..3, lanes t < 2) plus lo (columns 4..7, lanes t + 2):
                    // lanes t < 2 then hold rows 2t, 2t + 1 at columns g and g + 8
                    int32_t rowoff[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) rowoff[e] = t < 2 && 2 * t + e < R ? gs.pos_row[p0 + 2 * t + e] : -1;
#pragma unroll
                    for (int i = 0; i < kExpGroups; ++i) {
                        const int32_t nl = (warp + kExpWarps * i) * 16;
                        if (nl >= ncols) continue;
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc[i][0][e] += __shfl_xor_sync(0xffffffffu, acc[i][0][e], 2);
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            if (rowoff[e] < 0) continue;
                            float *dst = p.ycorr + static_cast<size_t>(rowoff[e]) * p.N + n0 + nl + g;
                            if (nl + g < ncols) dst[0] = sc * acc[i][0][e];
                            if (nl + g + 8 < ncols) dst[8] = sc * acc[i][0][2 + e];
                        }
                    }
                } else {
                    // each 16-column group through the warp's [16 rows][16 n] tile, so
                    // that a lane stores 4 consecutive columns of a row at once
                    float *tile = epi[warp];
                    const int er = lane >> 2, ec = (lane & 3) * 4;  // the lane's row (of 8) and first column
                    int32_t rowoff[2];
#pragma unroll
                    for (int q = 0; q < 2; ++q) rowoff[q] = 8 * q + er < R ? gs.pos_row[p0 + 8 * q + er] : -1;
#pragma unroll
                    for (int i = 0; i < kExpGroups; ++i) {
                        const int32_t nl = (warp + kExpWarps * i) * 16;
                        if (nl >= ncols) continue;
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            const int r0 = 8 * q + 2 * t;
                            tile[r0 * kEpiPitch + g] = acc[i][q][0];
                            tile[(r0 + 1) * kEpiPitch + g] = acc[i][q][1];
                            tile[r0 * kEpiPitch + g + 8] = acc[i][q][2];
                            tile[(r0 + 1) * kEpiPitch + g + 8] = acc[i][q][3];
                        }
                        __syncwarp();
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            if (rowoff[q] < 0) continue;
                            const float4 v = *reinterpret_cast<const float4 *>(tile + (8 * q + er) * kEpiPitch + ec);
                            const int32_t n = nl + ec;
                            float *dst = p.ycorr + static_cast<size_t>(rowoff[q]) * p.N + n0 + n;
                            if (vec_out && n + 4 <= ncols) {
                                *reinterpret_cast<float4 *>(dst) = make_float4(sc * v.x, sc * v.y, sc * v.z, sc * v.w);
                            } else {
                                const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                                for (int c = 0; c < 4; ++c)
                                    if (n + c < ncols) dst[c] = sc * vv[c];
                            }
                        }
                        __syncwarp();
                    }
                }
            }
        }
    }
    __syncthreads();
    if (tid == 0) drain_stages(full, kExpStages, issued_s);
}

}  // namespace

bool pipe_grouped_supported(int32_t M, int32_t max_rank) { return M <= kPipeMaxRows && max_rank <= kPipeMaxRank; }

bool pipe_pair_projections(int32_t M, int32_t K, int n, const int32_t *N, const int32_t *max_rank, bool any_quant) {
    if (n < 2 || any_quant || M <= 0 || !plan_tc(M, N[0], K).swap) return false;
    bool all_rows = true;
    for (int i = 0; i < n; ++i) {
        if (!pipe_grouped_supported(M, max_rank[i])) return false;
        all_rows = all_rows && row_lora_preferred(M, K, N[i], max_rank[i]);
    }
    return !all_rows;
}

namespace {

// Persistent grid of one CTA per SM, launched as a programmatic dependent of
// the kernel before it on the stream.
template <typename Params>
cudaError_t launch_pipe(void (*kernel)(Params), const Params &p, int threads, size_t smem, size_t smem_max,
                        cudaStream_t stream) {
    static std::mutex mu;
    static uint64_t done_ctx[2][128] = {};  // per kernel and device: the context the opt-in was set in
    const int which = reinterpret_cast<const void *>(kernel) == reinterpret_cast<const void *>(&pipe_shrink_kernel) ? 0 : 1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(mu);
        uint64_t ctx = done_ctx[which][dev];
        if (first_use_in_context(&ctx)) {  // the opt-in is per device; the largest size any call needs
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_max));
            if (e != cudaSuccess) return e;
            done_ctx[which][dev] = current_context_id();
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(device_sm_count());
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

}  // namespace

// K slices of the pipelined shrink: one plane of V each, at most kMaxVPlanes,
// each a multiple of the stage width where that keeps every plane non-empty.
static int32_t pipe_kc_len(int32_t K, int32_t ksplit) {
    int32_t len = ((K + ksplit - 1) / ksplit + kShrStageK - 1) / kShrStageK * kShrStageK;
    if (static_cast<int64_t>(ksplit - 1) * len >= K) len = ((K + ksplit - 1) / ksplit + 7) / 8 * 8;
    return len;
}

size_t pipe_group_bytes() { return sizeof(PipeGroupTable); }

// Projection v's grouping table in plan.pipe_groups (null if v is not one of
// the plan's projections or there is no table region).
static const PipeGroupTable *pipe_group_of(const ForwardPlan &plan, const ProjView &v) {
    const ptrdiff_t q = &v - plan.proj;
    if (!plan.pipe_groups || q < 0 || q >= plan.n_proj) return nullptr;
    return static_cast<const PipeGroupTable *>(plan.pipe_groups) + q;
}

cudaError_t launch_pipe_group(const ForwardPlan &plan, cudaStream_t stream) {
    if (plan.M <= 0) return cudaSuccess;
    if (plan.M > kPipeMaxRows || !plan.pipe_groups || plan.n_proj < 1 || plan.n_proj > LORA_MAX_PROJ)
        return cudaErrorInvalidValue;
    PipeGroupParams p;
    p.M = plan.M;
    p.row_slot = plan.row_slot;
    for (int q = 0; q < plan.n_proj; ++q) {
        p.ranks[q] = plan.proj[q].ranks;
        p.max_slots[q] = plan.proj[q].max_slots;
        p.bps[q] = plan.proj[q].bps;
    }
    p.tables = static_cast<PipeGroupTable *>(plan.pipe_groups);
    p.status = plan.status;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.n_proj);
    cfg.blockDim = dim3(kPipeThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, pipe_group_kernel, p);
}

// Split the grid's CTAs between n projections by their weights (each gets
// at least one; largest remainders take the rest).
static bool split_ctas(const double *w, int n, int32_t ctas, int32_t *begin) {
    if (n < 1 || n > LORA_MAX_PROJ || ctas < n) return false;
    double total = 0.0;
    for (int q = 0; q < n; ++q) total += w[q] > 0.0 ? w[q] : 0.0;
    int32_t cnt[LORA_MAX_PROJ];
    double rem[LORA_MAX_PROJ];
    int32_t used = 0;
    for (int q = 0; q < n; ++q) {
        const double share = total > 0.0 ? (ctas - n) * (w[q] > 0.0 ? w[q] : 0.0) / total : 0.0;
        cnt[q] = 1 + static_cast<int32_t>(share);
        rem[q] = share - static_cast<int32_t>(share);
        used += cnt[q];
    }
    while (used < ctas) {
        int best = 0;
        for (int q = 1; q < n; ++q)
            if (rem[q] > rem[best]) best = q;
        ++cnt[best];
        rem[best] = -1.0;
        ++used;
    }
    begin[0] = 0;
    for (int q = 0; q < n; ++q) begin[q + 1] = begin[q] + cnt[q];
    return begin[n] == ctas;
}

cudaError_t launch_pipe_shrink(const ForwardPlan &plan, const ProjView *const *vs, int n, cudaStream_t stream) {
    if (plan.M <= 0) return cudaSuccess;
    if (n < 1 || n > LORA_MAX_PROJ || plan.v_parts < 1 || plan.v_parts > kMaxVPlanes) return cudaErrorInvalidValue;
    PipeMulti<PipeShrinkParams> m = {};
    m.n_proj = n;
    double w[LORA_MAX_PROJ];
    for (int q = 0; q < n; ++q) {
        const ProjView &v = *vs[q];
        if (!pipe_grouped_supported(plan.M, v.max_rank)) return cudaErrorInvalidValue;
        PipeShrinkParams &p = m.proj[q];
        p.M = plan.M;
        p.K = plan.K;
        p.ldx = plan.ldx;
        p.x = static_cast<const __nv_bfloat16 *>(plan.x);
        p.row_slot = plan.row_slot;
        p.a_arena = static_cast<const __nv_bfloat16 *>(v.a_arena);
        p.table = v.table;
        p.ranks = v.ranks;
        p.max_slots = v.max_slots;
        p.bps = v.bps;
        p.num_blocks = v.num_blocks;
        p.V = v.V;
        p.ldv = v.max_rank;
        // one item covers all of K (in kShrStageK stages), so V is one plane:
        // the expand then fetches one V piece per item instead of one per slice
        p.ksplit = 1;
        p.kc_len = pipe_kc_len(plan.K, 1);
        p.plane_stride = static_cast<size_t>(plan.M) * v.max_rank;
        p.counters = plan.counters;
        p.n_counters = plan.n_counters;
        p.group = pipe_group_of(plan, v);
        if (!p.group) return cudaErrorInvalidValue;
        p.status = plan.status;
        w[q] = static_cast<double>(v.max_rank);  // the A bytes a row's adapter brings, at most
    }
    if (!split_ctas(w, n, device_sm_count(), m.cta_begin)) return cudaErrorInvalidValue;
    return launch_pipe(pipe_shrink_kernel, m, kPipeThreads, kShrSmem, kShrSmem, stream);
}

cudaError_t launch_pipe_expand(const ForwardPlan &plan, const ProjView *const *vs, int n, cudaStream_t stream) {
    if (plan.M <= 0) return cudaSuccess;
    if (n < 1 || n > LORA_MAX_PROJ || plan.v_parts < 1 || plan.v_parts > kMaxVPlanes) return cudaErrorInvalidValue;
    PipeMulti<PipeExpandParams> m = {};
    m.n_proj = n;
    double w[LORA_MAX_PROJ];
    size_t smem = 0;
    const size_t room = kExpSmemMax - static_cast<size_t>(kExpStages) * kExpStageBytes;
    for (int q = 0; q < n; ++q) {
        const ProjView &v = *vs[q];
        if (!pipe_grouped_supported(plan.M, v.max_rank)) return cudaErrorInvalidValue;
        PipeExpandParams &p = m.proj[q];
        p.M = plan.M;
        p.N = v.N;
        p.row_slot = plan.row_slot;
        p.b_arena = static_cast<const __nv_bfloat16 *>(v.b_arena);
        p.table = v.table;
        p.ranks = v.ranks;
        p.scales = v.scales;
        p.max_slots = v.max_slots;
        p.bps = v.bps;
        p.num_blocks = v.num_blocks;
        p.V = v.V;
        p.ldv = v.max_rank;
        p.ksplit = 1;  // as the shrink writes it
        p.plane_stride = static_cast<size_t>(plan.M) * v.max_rank;
        p.vslot_floats = kChunkRows * v.max_rank;
        p.ycorr = v.ycorr;
        p.group = pipe_group_of(plan, v);
        if (!p.group) return cudaErrorInvalidValue;
        p.status = plan.status;
        const size_t vbytes = sizeof(float) * static_cast<size_t>(p.vslot_floats);
        p.n_vslots = static_cast<int32_t>(room / vbytes < kExpMaxVSlots ? room / vbytes : kExpMaxVSlots);
        if (p.n_vslots < 2) return cudaErrorInvalidValue;
        const size_t need = static_cast<size_t>(kExpStages) * kExpStageBytes + p.n_vslots * vbytes;
        smem = need > smem ? need : smem;
        w[q] = static_cast<double>(v.N) * v.max_rank;  // the B bytes a row's adapter brings, at most
    }
    if (!split_ctas(w, n, device_sm_count(), m.cta_begin)) return cudaErrorInvalidValue;
    return launch_pipe(pipe_expand_kernel, m, kExpThreads, smem, kExpSmemMax, stream);
}

}  // namespace lora
