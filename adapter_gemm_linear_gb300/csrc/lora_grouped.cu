// The LoRA path of the small-M (swapped) GEMM orientation, organised by
// adapter group:
//
//   1. group_rows_kernel: the rows sorted by adapter id on the device (a stable
//      counting of keys), giving a group table: group g holds the sorted
//      positions [start[g], start[g+1]) of rows with adapter slot[g]; rows
//      without an adapter (id -1, or an id outside the pool) follow the
//      groups.  This is the segmenter's job (rows sorted by adapter) done where
//      the ids live.
//   2. shrink_grouped_kernel:  V[p][m, 16 jb + j] = sum_{k in slice p} A_i[16 jb + j, k] x[m, k]
//      one work item per (group, rank block, K slice): the block's 16 A rows
//      of the slice are read once and applied to every row of the group.  The
//      slices' partial sums are separate planes p of V (no atomics); the
//      expand adds them.
//   3. expand_grouped_kernel:  ycorr[m, n] = s_i * sum_j B_i[n, j] V[m, j]
//      one work item per (group, 1024 output columns): the group's B pieces
//      for those columns are read once and applied to every row of the group;
//      rows without an adapter get zeros.
//
// The GEMM that follows adds ycorr to its fp32 accumulator before the single
// rounding to bf16.  All three kernels use persistent grids that walk their
// work items, since the number of groups is known only on the device.
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

constexpr int kSegThreads = 1024;
constexpr int kShrThreads = 256;
constexpr int kShrStep = kShrThreads * 8;   // k covered by one pass of the CTA (8 bf16 per thread)
constexpr int kShrRows = 2;                 // rows of a group per pass
constexpr int kExpThreads = 256;
constexpr int kExpColsPerThread = 4;
constexpr int kExpCols = kExpThreads * kExpColsPerThread;  // output columns per expand item
constexpr int kExpRows = 8;                 // rows of a group per pass
constexpr int kExpBlkChunk = 1;             // rank blocks whose B pieces are in flight together
static_assert(kExpRows * kMaxRankLimit * 4 <= 48 * 1024, "expand stage within the default shared memory");

__device__ __forceinline__ void unpack_bf16x8(const uint4 &q, float *v) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// ---------------------------------------------------------------------------
// 1. group table
// ---------------------------------------------------------------------------

// Exclusive prefix sum of one value per thread over the whole CTA, in a
// pass over kSegThreads consecutive items; *total gets the pass's sum.
__device__ __forceinline__ int32_t cta_exclusive_scan(int32_t v, int32_t *warp_tot, int32_t *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int32_t before = 0, sum = 0;
    for (int w = 0; w < kSegThreads / 32; ++w) {
        before += w < warp ? warp_tot[w] : 0;
        sum += warp_tot[w];
    }
    __syncthreads();  // warp_tot is rewritten by the next pass
    *total = sum;
    return before + incl - v;
}

// One CTA.  key[m] = the row's slot id, or INT_MAX for rows without an adapter
// (an id outside [-1, max_slots) is reported and treated as none); the rank of
// (key, m) among all rows is the row's sorted position, so rows of one slot
// keep their order.  Then the group table and its chunk list.
__global__ void __launch_bounds__(kSegThreads)
group_rows_kernel(int32_t M, const int32_t *__restrict__ row_slot, int32_t max_slots, GroupTable gt,
                  unsigned long long *status) {
    extern __shared__ __align__(16) int32_t seg_smem[];
    int32_t *key = seg_smem;              // [M]
    int32_t *pos_row = key + M;           // [M] sorted position -> row
    int32_t *gs = pos_row + M;            // [M + 1] group -> first sorted position
    __shared__ int32_t warp_tot[kSegThreads / 32];
    __shared__ int32_t n_adapted;
    const int tid = threadIdx.x;
    if (tid == 0) n_adapted = 0;
    __syncthreads();
    for (int32_t base = 0; base < M; base += kSegThreads) {
        const int32_t m = base + tid;
        bool adapted = false;
        if (m < M) {
            const int32_t id = row_slot[m];
            int32_t k = 0x7fffffff;
            if (id >= 0 && id < max_slots) {
                k = id;
                adapted = true;
            } else if (id != -1) {
                record_error(status, kDevBadAdapter, static_cast<uint32_t>(m));
            }
            key[m] = k;
        }
        const unsigned ballot = __ballot_sync(0xffffffffu, adapted);  // one shared atomic per warp
        if ((tid & 31) == 0 && ballot) atomicAdd(&n_adapted, __popc(ballot));
    }
    __syncthreads();
    for (int32_t m = tid; m < M; m += kSegThreads) {
        const int32_t k = key[m];
        int32_t rnk = 0;
        int32_t m2 = 0;
        for (; m2 + 4 <= M; m2 += 4) {
            const int4 k4 = *reinterpret_cast<const int4 *>(key + m2);
            rnk += (k4.x < k) || (k4.x == k && m2 < m);
            rnk += (k4.y < k) || (k4.y == k && m2 + 1 < m);
            rnk += (k4.z < k) || (k4.z == k && m2 + 2 < m);
            rnk += (k4.w < k) || (k4.w == k && m2 + 3 < m);
        }
        for (; m2 < M; ++m2) rnk += (key[m2] < k) || (key[m2] == k && m2 < m);
        pos_row[rnk] = m;
    }
    __syncthreads();
    const int32_t na = n_adapted;
    // groups: a new one starts at every adapted position whose slot differs
    // from the one before
    int32_t G = 0;
    for (int32_t base = 0; base < M; base += kSegThreads) {
        const int32_t i = base + tid;
        const int32_t f = i < na && (i == 0 || key[pos_row[i]] != key[pos_row[i - 1]]);
        if (i < M) gt.perm[i] = pos_row[i];
        int32_t tot;
        const int32_t g = G + cta_exclusive_scan(f, warp_tot, &tot);
        if (f) {
            gs[g] = i;
            gt.start[g] = i;
            gt.slot[g] = key[pos_row[i]];
        }
        G += tot;
    }
    if (tid == 0) {
        gs[G] = na;
        gt.start[G] = na;  // end of the last group; rows without an adapter follow
    }
    __syncthreads();
    // chunk lists (see GroupTable): the groups' chunks, then the rows without
    // an adapter
#pragma unroll 1
    for (int L = 0; L < 2; ++L) {
        const int32_t R = L == 0 ? kGroupChunkRowsShrink : kGroupChunkRowsExpand;
        int32_t C = 0;
        for (int32_t base = 0; base <= G; base += kSegThreads) {
            const int32_t g = base + tid;
            int32_t rows = 0;
            if (g < G) rows = gs[g + 1] - gs[g];
            else if (g == G) rows = M - na;
            const int32_t nch = (rows + R - 1) / R;
            int32_t tot;
            const int32_t c0 = C + cta_exclusive_scan(nch, warp_tot, &tot);
            for (int32_t c = 0; c < nch; ++c) {
                gt.chunk_group[L][c0 + c] = g;
                gt.chunk_begin[L][c0 + c] = (g < G ? gs[g] : na) + c * R;
            }
            if (g == G) {
                gt.count[1 + 2 * L] = c0;  // chunks of the groups
                gt.count[2 + 2 * L] = c0 + nch;
                gt.chunk_begin[L][c0 + nch] = M;
            }
            C += tot;
        }
    }
    if (tid == 0) gt.count[0] = G;
}

// ---------------------------------------------------------------------------
// 2. shrink by group
// ---------------------------------------------------------------------------

struct GroupedShrinkParams {
    int32_t M, K, ldx;
    const __nv_bfloat16 *x;
    GroupTable gt;
    const __nv_bfloat16 *a_arena;
    const int32_t *table;
    const int32_t *ranks;
    int32_t max_slots, bps, num_blocks;
    float *V;              // [ksplit][M][ldv]
    int32_t ldv;
    int32_t ksplit;        // K slices = planes of V
    int32_t kc_len;        // k per slice (a multiple of 8)
    size_t plane_stride;   // elements between planes
    int32_t *counters;     // split-K tile counters of the GEMM that follows, zeroed here
    int32_t n_counters;
    unsigned long long *status;
};

// Persistent grid over items u = ((c * bps) + jb) * ksplit + kc over the
// groups' row chunks c; items past the group's rank blocks are skipped.  Each
// pass handles kShrRows rows of the chunk: every thread takes 8 consecutive k
// of the slice per step, keeps the 16 A values of each of those k in
// registers and applies them to the pass's rows; the CTA then sums the
// per-thread partial dot products.
__global__ void __launch_bounds__(kShrThreads, 2)
shrink_grouped_kernel(const GroupedShrinkParams p) {
    __shared__ float red[kShrThreads / 32][kShrRows * LORA_BLOCK_ROWS];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (blockIdx.x == 0)
        for (int32_t c = tid; c < p.n_counters; c += kShrThreads) p.counters[c] = 0;
    const int32_t chunks = p.gt.count[1];  // list 0
    const int32_t items = chunks * p.bps * p.ksplit;
    const int32_t K8 = p.K / 8;
    for (int32_t u = blockIdx.x; u < items; u += gridDim.x) {
        const int32_t kc = u % p.ksplit;
        const int32_t t = u / p.ksplit;
        const int32_t jb = t % p.bps;
        const int32_t ch = t / p.bps;
        const int32_t g = p.gt.chunk_group[0][ch];
        const int32_t slot = p.gt.slot[g];
        const int32_t r = p.ranks[slot];
        if (r <= 0 || r > p.bps * LORA_BLOCK_ROWS) continue;  // reported by the expand
        if (jb * LORA_BLOCK_ROWS >= r) continue;
        const int32_t blk = p.table[static_cast<size_t>(slot) * p.bps + jb];
        if (blk < 0 || blk >= p.num_blocks) continue;        // reported by the expand
        const int32_t p0 = p.gt.chunk_begin[0][ch], p1 = p.gt.chunk_begin[0][ch + 1];
        const int32_t k8_0 = kc * (p.kc_len / 8);
        const int32_t k8_1 = min(K8, k8_0 + p.kc_len / 8);
        const uint4 *A = reinterpret_cast<const uint4 *>(p.a_arena + static_cast<size_t>(blk) * LORA_BLOCK_ROWS * p.K);
#pragma unroll 1
        for (int32_t pc = p0; pc < p1; pc += kShrRows) {
            int32_t rows[kShrRows];
#pragma unroll
            for (int rr = 0; rr < kShrRows; ++rr) rows[rr] = pc + rr < p1 ? p.gt.perm[pc + rr] : -1;
            float acc[kShrRows][LORA_BLOCK_ROWS];
#pragma unroll
            for (int rr = 0; rr < kShrRows; ++rr)
#pragma unroll
                for (int j = 0; j < LORA_BLOCK_ROWS; ++j) acc[rr][j] = 0.0f;
#pragma unroll 1
            for (int32_t k8 = k8_0 + tid; k8 < k8_1; k8 += kShrThreads) {
                uint4 aq[LORA_BLOCK_ROWS];
#pragma unroll
                for (int j = 0; j < LORA_BLOCK_ROWS; ++j) aq[j] = __ldg(A + static_cast<size_t>(j) * K8 + k8);
                uint4 xq[kShrRows];
#pragma unroll
                for (int rr = 0; rr < kShrRows; ++rr)
                    if (rows[rr] >= 0)
                        xq[rr] = __ldg(reinterpret_cast<const uint4 *>(p.x + static_cast<size_t>(rows[rr]) * p.ldx) + k8);
#pragma unroll
                for (int rr = 0; rr < kShrRows; ++rr) {
                    if (rows[rr] < 0) continue;
                    float xv[8];
                    unpack_bf16x8(xq[rr], xv);
#pragma unroll
                    for (int j = 0; j < LORA_BLOCK_ROWS; ++j) {
                        float av[8];
                        unpack_bf16x8(aq[j], av);
                        float a = acc[rr][j];
#pragma unroll
                        for (int q = 0; q < 8; ++q) a = fmaf(av[q], xv[q], a);
                        acc[rr][j] = a;
                    }
                }
            }
            // CTA sum of the partial dot products
#pragma unroll
            for (int rr = 0; rr < kShrRows; ++rr)
#pragma unroll
                for (int j = 0; j < LORA_BLOCK_ROWS; ++j) {
                    float v = acc[rr][j];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                    if (lane == 0) red[warp][rr * LORA_BLOCK_ROWS + j] = v;
                }
            __syncthreads();
            if (tid < kShrRows * LORA_BLOCK_ROWS) {
                const int rr = tid / LORA_BLOCK_ROWS, j = tid % LORA_BLOCK_ROWS;
                if (rows[rr] >= 0) {
                    float v = 0.0f;
#pragma unroll
                    for (int w = 0; w < kShrThreads / 32; ++w) v += red[w][tid];
                    p.V[kc * p.plane_stride + static_cast<size_t>(rows[rr]) * p.ldv + jb * LORA_BLOCK_ROWS + j] = v;
                }
            }
            __syncthreads();  // red is rewritten by the next pass
        }
    }
}

// ---------------------------------------------------------------------------
// 3. expand by group
// ---------------------------------------------------------------------------

struct GroupedExpandParams {
    int32_t M, N;
    GroupTable gt;
    const __nv_bfloat16 *b_arena;
    const int32_t *table;
    const int32_t *ranks;
    const float *scales;
    int32_t max_slots, bps, num_blocks;
    const float *V;        // [ksplit][M][ldv]
    int32_t ldv;
    int32_t ksplit;
    size_t plane_stride;
    float *ycorr;          // [M][N]
    unsigned long long *status;
};

// Persistent grid over items u = c * n_ranges + nr over all row chunks c (a
// chunk of group G holds rows without an adapter, which get zeros).  A thread owns kExpColsPerThread
// columns n = nr * kExpCols + tid + kExpThreads c.  Per pass of kExpRows rows
// of the group the rows' V (planes summed) are staged in shared memory while
// the first kExpBlkChunk blocks' B pieces are in flight; every B piece then
// serves all rows of the pass.
__global__ void __launch_bounds__(kExpThreads, 2)
expand_grouped_kernel(const GroupedExpandParams p) {
    extern __shared__ __align__(16) float vs[];  // [kExpRows][ldv]
    // the GEMM that follows may launch now; it reads ycorr only after this
    // grid has completed (griddepcontrol.wait)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int tid = threadIdx.x;
    const int32_t G = p.gt.count[0];
    const int32_t n_ranges = (p.N + kExpCols - 1) / kExpCols;
    const int32_t items = p.gt.count[4] * n_ranges;  // list 1
    for (int32_t u = blockIdx.x; u < items; u += gridDim.x) {
        const int32_t ch = u / n_ranges;
        const int32_t nr = u % n_ranges;
        const int32_t g = p.gt.chunk_group[1][ch];
        const int32_t p0 = p.gt.chunk_begin[1][ch];
        const int32_t p1 = p.gt.chunk_begin[1][ch + 1];
        int32_t nblk = 0, slot = -1;
        float sc = 0.0f;
        if (g < G) {
            slot = p.gt.slot[g];
            const int32_t r = p.ranks[slot];
            bool ok = r > 0 && r <= p.bps * LORA_BLOCK_ROWS;
            if (ok) {
                nblk = (r + LORA_BLOCK_ROWS - 1) / LORA_BLOCK_ROWS;
                for (int32_t jb = 0; jb < nblk; ++jb) {
                    const int32_t blk = p.table[static_cast<size_t>(slot) * p.bps + jb];
                    ok &= blk >= 0 && blk < p.num_blocks;
                }
                sc = p.scales[slot];
            }
            if (!ok) {
                // empty slot or corrupt block entry: these rows get no correction
                if (nr == 0 && tid == 0 && p0 == p.gt.start[g])
                    record_error(p.status, r <= 0 ? kDevEmptySlot : kDevBadBlock,
                                 static_cast<uint32_t>(r <= 0 ? p.gt.perm[p0] : slot));
                nblk = 0;
            }
        }
        int32_t cols[kExpColsPerThread];
#pragma unroll
        for (int c = 0; c < kExpColsPerThread; ++c) cols[c] = nr * kExpCols + tid + c * kExpThreads;
        if (nblk == 0) {
            for (int32_t i = p0; i < p1; ++i) {
                float *dst = p.ycorr + static_cast<size_t>(p.gt.perm[i]) * p.N;
#pragma unroll
                for (int c = 0; c < kExpColsPerThread; ++c)
                    if (cols[c] < p.N) dst[cols[c]] = 0.0f;
            }
            continue;
        }
        const int32_t *trow = p.table + static_cast<size_t>(slot) * p.bps;
#pragma unroll 1
        for (int32_t pc = p0; pc < p1; pc += kExpRows) {
            const int nrows = min(kExpRows, p1 - pc);
            float acc[kExpRows][kExpColsPerThread];
#pragma unroll
            for (int rr = 0; rr < kExpRows; ++rr)
#pragma unroll
                for (int c = 0; c < kExpColsPerThread; ++c) acc[rr][c] = 0.0f;
#pragma unroll 1
            for (int32_t jb0 = 0; jb0 < nblk; jb0 += kExpBlkChunk) {
                // this chunk's B pieces: 16 ranks of each owned column
                uint4 q[kExpBlkChunk][kExpColsPerThread][2];
#pragma unroll
                for (int b = 0; b < kExpBlkChunk; ++b) {
                    if (jb0 + b >= nblk) continue;
                    const __nv_bfloat16 *base = p.b_arena + static_cast<size_t>(trow[jb0 + b]) * p.N * LORA_BLOCK_ROWS;
#pragma unroll
                    for (int c = 0; c < kExpColsPerThread; ++c) {
                        if (cols[c] >= p.N) continue;
                        const uint4 *src = reinterpret_cast<const uint4 *>(base + static_cast<size_t>(cols[c]) * LORA_BLOCK_ROWS);
                        q[b][c][0] = __ldg(src);
                        q[b][c][1] = __ldg(src + 1);
                    }
                }
                if (jb0 == 0) {
                    // stage the pass's V rows (all rank blocks, planes summed)
                    __syncthreads();  // the previous pass is done with vs
                    const int q4 = nblk * (LORA_BLOCK_ROWS / 4);
                    for (int i4 = tid; i4 < nrows * q4; i4 += kExpThreads) {
                        const int rr = i4 / q4, c4 = i4 - rr * q4;
                        const float4 *src =
                            reinterpret_cast<const float4 *>(p.V + static_cast<size_t>(p.gt.perm[pc + rr]) * p.ldv) + c4;
                        float4 v = *src;
                        for (int pl = 1; pl < p.ksplit; ++pl) {
                            const float4 w = src[pl * (p.plane_stride / 4)];
                            v.x += w.x;
                            v.y += w.y;
                            v.z += w.z;
                            v.w += w.w;
                        }
                        reinterpret_cast<float4 *>(vs)[rr * (p.ldv / 4) + c4] = v;
                    }
                    __syncthreads();
                }
#pragma unroll
                for (int b = 0; b < kExpBlkChunk; ++b) {
                    if (jb0 + b >= nblk) continue;
#pragma unroll
                    for (int c = 0; c < kExpColsPerThread; ++c) {
                        if (cols[c] >= p.N) continue;
                        float bv[16];
                        unpack_bf16x8(q[b][c][0], bv);
                        unpack_bf16x8(q[b][c][1], bv + 8);
#pragma unroll
                        for (int rr = 0; rr < kExpRows; ++rr) {
                            if (rr >= nrows) break;
                            const float4 *vr = reinterpret_cast<const float4 *>(vs + rr * p.ldv + (jb0 + b) * LORA_BLOCK_ROWS);
                            const float4 v0 = vr[0], v1 = vr[1], v2 = vr[2], v3 = vr[3];
                            float a0 = bv[0] * v0.x, a1 = bv[1] * v0.y, a2 = bv[2] * v0.z, a3 = bv[3] * v0.w;
                            a0 = fmaf(bv[4], v1.x, a0);
                            a1 = fmaf(bv[5], v1.y, a1);
                            a2 = fmaf(bv[6], v1.z, a2);
                            a3 = fmaf(bv[7], v1.w, a3);
                            a0 = fmaf(bv[8], v2.x, a0);
                            a1 = fmaf(bv[9], v2.y, a1);
                            a2 = fmaf(bv[10], v2.z, a2);
                            a3 = fmaf(bv[11], v2.w, a3);
                            a0 = fmaf(bv[12], v3.x, a0);
                            a1 = fmaf(bv[13], v3.y, a1);
                            a2 = fmaf(bv[14], v3.z, a2);
                            a3 = fmaf(bv[15], v3.w, a3);
                            acc[rr][c] += (a0 + a1) + (a2 + a3);
                        }
                    }
                }
            }
#pragma unroll
            for (int rr = 0; rr < kExpRows; ++rr) {
                if (rr >= nrows) break;
                float *dst = p.ycorr + static_cast<size_t>(p.gt.perm[pc + rr]) * p.N;
#pragma unroll
                for (int c = 0; c < kExpColsPerThread; ++c)
                    if (cols[c] < p.N) dst[cols[c]] = sc * acc[rr][c];
            }
        }
    }
}

// ---------------------------------------------------------------------------
// 4. the whole LoRA term of one row (rows few enough that reading the row's
//    A and B per row is cheap)
// ---------------------------------------------------------------------------

// One projection (its pool and correction array) of the per-row kernel.
struct RowProj {
    int32_t N;
    const __nv_bfloat16 *a_arena;
    const __nv_bfloat16 *b_arena;
    const int32_t *table;
    const int32_t *ranks;
    const float *scales;
    int32_t max_slots, bps, num_blocks;
    int32_t cols_per_cta;  // output columns per CTA (a multiple of kRowThreads)
    int32_t splits;        // column ranges: CTAs of blockIdx.y >= splits have no work
    float *ycorr;          // [M][N]
};

struct RowLoraParams {
    int32_t M, K, ldx;
    const __nv_bfloat16 *x;
    const int32_t *row_slot;
    int32_t *counters;     // split-K tile counters of the GEMMs that follow, zeroed here
    int32_t n_counters;
    unsigned long long *status;
    RowProj proj[LORA_MAX_PROJ];  // blockIdx.z selects one
};

// Four warps of at most 152 registers: a CTA fits on an SM beside a CTA of
// the swapped GEMM (ten warps, allocated as twelve, of 120 registers), so the
// GEMM that follows as a programmatic dependent streams W while this kernel
// runs.
constexpr int kRowThreads = 128;
constexpr int kRowMaxRegs = 152;
constexpr int kRowBatch = 1;  // k steps of A loads in flight per thread
constexpr int kRowCols = 8;   // output columns per thread whose B pieces are in flight together

// grid (M, column splits, projections).  The CTA resolves its row's adapter
// in the pool of projection blockIdx.z, computes
// v = A_i x[m] (all rank blocks; per block every thread takes 8 consecutive k
// per step and the CTA sums the partial dot products) into shared memory, then
// writes ycorr[m, n] = s_i <B_i[n, :], v> for its columns (zeros for a row
// without an adapter).
__global__ void __maxnreg__(kRowMaxRegs) lora_rows_kernel(const __grid_constant__ RowLoraParams p) {
    __shared__ float red[kRowThreads / 32][LORA_BLOCK_ROWS];
    extern __shared__ __align__(16) float v[];  // [max_rank]
    // the GEMM that follows may launch now; it reads ycorr only after this
    // grid has completed (griddepcontrol.wait)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t m = blockIdx.x;
    if (m == 0 && blockIdx.y == 0 && blockIdx.z == 0)
        for (int32_t c = tid; c < p.n_counters; c += kRowThreads) p.counters[c] = 0;
    const RowProj &q = p.proj[blockIdx.z];
    if (static_cast<int32_t>(blockIdx.y) >= q.splits) return;
    const int32_t n_begin = blockIdx.y * q.cols_per_cta;
    const int32_t n_end = min(q.N, n_begin + q.cols_per_cta);
    int32_t r = 0;
    float sc = 0.0f;
    int32_t slot = resolve_slot(p.row_slot[m], m, q.ranks, q.scales, q.max_slots, q.bps, &r, &sc, p.status,
                                blockIdx.y == 0 && tid == 0);
    const int32_t nblk = (r + LORA_BLOCK_ROWS - 1) / LORA_BLOCK_ROWS;
    const int32_t *trow = q.table + static_cast<size_t>(slot < 0 ? 0 : slot) * q.bps;
    if (slot >= 0) {
        bool ok = true;
        for (int32_t jb = 0; jb < nblk; ++jb) ok &= trow[jb] >= 0 && trow[jb] < q.num_blocks;
        if (!ok) {
            if (blockIdx.y == 0 && tid == 0) record_error(p.status, kDevBadBlock, static_cast<uint32_t>(slot));
            slot = -1;
        }
    }
    if (slot >= 0 && tid == 0) {
        // the row's A blocks (16 rows x K, contiguous) and this CTA's columns
        // of its B blocks head for L2 now, so that the loads below, issued a
        // few at a time, mostly hit it
        for (int32_t jb = 0; jb < nblk; ++jb) {
            sm100::bulk_prefetch_l2(q.a_arena + static_cast<size_t>(trow[jb]) * LORA_BLOCK_ROWS * p.K,
                                    static_cast<uint32_t>(LORA_BLOCK_ROWS) * p.K * 2u);
            if (n_end > n_begin)
                sm100::bulk_prefetch_l2(
                    q.b_arena + (static_cast<size_t>(trow[jb]) * q.N + n_begin) * LORA_BLOCK_ROWS,
                    static_cast<uint32_t>(n_end - n_begin) * LORA_BLOCK_ROWS * 2u);
        }
        sm100::bulk_prefetch_l2(p.x + static_cast<size_t>(m) * p.ldx, static_cast<uint32_t>(p.K) * 2u);
    }
    float *dst = q.ycorr + static_cast<size_t>(m) * q.N;
    if (slot < 0) {
        for (int32_t n = n_begin + tid; n < n_end; n += kRowThreads) dst[n] = 0.0f;
        return;
    }
    // v = A_i x[m], one rank block at a time
    const uint4 *xr = reinterpret_cast<const uint4 *>(p.x + static_cast<size_t>(m) * p.ldx);
    const int32_t K8 = p.K / 8;
#pragma unroll 1
    for (int32_t jb = 0; jb < nblk; ++jb) {
        const uint4 *A = reinterpret_cast<const uint4 *>(q.a_arena + static_cast<size_t>(trow[jb]) * LORA_BLOCK_ROWS * p.K);
        float acc[LORA_BLOCK_ROWS];
#pragma unroll
        for (int j = 0; j < LORA_BLOCK_ROWS; ++j) acc[j] = 0.0f;
#pragma unroll 1
        for (int32_t k0 = tid; k0 < K8; k0 += kRowBatch * kRowThreads) {
            uint4 xq[kRowBatch];
            uint4 aq[kRowBatch][LORA_BLOCK_ROWS];
#pragma unroll
            for (int u = 0; u < kRowBatch; ++u) {
                const int32_t k = k0 + u * kRowThreads;
                if (k < K8) {
                    xq[u] = __ldg(xr + k);
#pragma unroll
                    for (int j = 0; j < LORA_BLOCK_ROWS; ++j) aq[u][j] = __ldg(A + static_cast<size_t>(j) * K8 + k);
                }
            }
#pragma unroll
            for (int u = 0; u < kRowBatch; ++u) {
                if (k0 + u * kRowThreads >= K8) continue;
                float xv[8];
                unpack_bf16x8(xq[u], xv);
#pragma unroll
                for (int j = 0; j < LORA_BLOCK_ROWS; ++j) {
                    float av[8];
                    unpack_bf16x8(aq[u][j], av);
                    float a = acc[j];
#pragma unroll
                    for (int q = 0; q < 8; ++q) a = fmaf(av[q], xv[q], a);
                    acc[j] = a;
                }
            }
        }
#pragma unroll
        for (int j = 0; j < LORA_BLOCK_ROWS; ++j) {
            float t = acc[j];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
            if (lane == 0) red[warp][j] = t;
        }
        __syncthreads();
        if (tid < LORA_BLOCK_ROWS) {
            float t = 0.0f;
#pragma unroll
            for (int w = 0; w < kRowThreads / 32; ++w) t += red[w][tid];
            v[jb * LORA_BLOCK_ROWS + tid] = t;
        }
        __syncthreads();
    }
    // ycorr[m, n] for this CTA's columns, kRowCols columns per thread at a
    // time with their B pieces (16 ranks per block) all in flight
    const float4 *vv = reinterpret_cast<const float4 *>(v);
#pragma unroll 1
    for (int32_t n0 = n_begin + tid; n0 < n_end; n0 += kRowCols * kRowThreads) {
        float acc[kRowCols];
#pragma unroll
        for (int c = 0; c < kRowCols; ++c) acc[c] = 0.0f;
#pragma unroll 1
        for (int32_t jb = 0; jb < nblk; ++jb) {
            const __nv_bfloat16 *bb = q.b_arena + static_cast<size_t>(trow[jb]) * q.N * LORA_BLOCK_ROWS;
            uint4 q[kRowCols][2];
#pragma unroll
            for (int c = 0; c < kRowCols; ++c) {
                const int32_t n = n0 + c * kRowThreads;
                if (n < n_end) {
                    const uint4 *src = reinterpret_cast<const uint4 *>(bb + static_cast<size_t>(n) * LORA_BLOCK_ROWS);
                    q[c][0] = __ldg(src);
                    q[c][1] = __ldg(src + 1);
                }
            }
            const float4 v0 = vv[jb * 4], v1 = vv[jb * 4 + 1], v2 = vv[jb * 4 + 2], v3 = vv[jb * 4 + 3];
#pragma unroll
            for (int c = 0; c < kRowCols; ++c) {
                if (n0 + c * kRowThreads >= n_end) continue;
                float bv[16];
                unpack_bf16x8(q[c][0], bv);
                unpack_bf16x8(q[c][1], bv + 8);
                float a0 = bv[0] * v0.x, a1 = bv[1] * v0.y, a2 = bv[2] * v0.z, a3 = bv[3] * v0.w;
                a0 = fmaf(bv[4], v1.x, a0);
                a1 = fmaf(bv[5], v1.y, a1);
                a2 = fmaf(bv[6], v1.z, a2);
                a3 = fmaf(bv[7], v1.w, a3);
                a0 = fmaf(bv[8], v2.x, a0);
                a1 = fmaf(bv[9], v2.y, a1);
                a2 = fmaf(bv[10], v2.z, a2);
                a3 = fmaf(bv[11], v2.w, a3);
                a0 = fmaf(bv[12], v3.x, a0);
                a1 = fmaf(bv[13], v3.y, a1);
                a2 = fmaf(bv[14], v3.z, a2);
                a3 = fmaf(bv[15], v3.w, a3);
                acc[c] += (a0 + a1) + (a2 + a3);
            }
        }
#pragma unroll
        for (int c = 0; c < kRowCols; ++c) {
            const int32_t n = n0 + c * kRowThreads;
            if (n < n_end) dst[n] = sc * acc[c];
        }
    }
}

int split_k_slices(int32_t K) {
    const int s = (K + kShrStep - 1) / kShrStep;
    return s < 1 ? 1 : s > kMaxVPlanes ? kMaxVPlanes : s;
}

}  // namespace

int grouped_v_planes(int32_t K) { return split_k_slices(K); }

bool row_lora_preferred(int32_t M, int32_t K, int32_t N, int32_t max_rank) {
    // bytes of A and B the per-row kernel reads (every row its own adapter
    // at the largest rank): small enough to come from L2 in a few microseconds
    const double bytes = static_cast<double>(M) * max_rank * (static_cast<double>(K) + N) * 2.0;
    return bytes <= 256.0 * 1024 * 1024;
}

bool fuse_row_projections(int32_t M, int32_t K, int n, const int32_t *N, const int32_t *max_rank) {
    // the paired GEMM launches take token tiles of 128 or 256 (M > 64)
    if (n < 2 || M <= 64 || !plan_tc(M, N[0], K).swap) return false;
    for (int i = 0; i < n; ++i)
        if (!row_lora_preferred(M, K, N[i], max_rank[i])) return false;
    return true;
}

// The per-row kernel over projections vs[0..n): grid (M, column splits, n).
static cudaError_t launch_rows(const ForwardPlan &plan, const ProjView *const *vs, int n, cudaStream_t stream) {
    if (plan.M <= 0) return cudaSuccess;
    if (n < 1 || n > LORA_MAX_PROJ) return cudaErrorInvalidValue;
    RowLoraParams p = {};
    p.M = plan.M;
    p.K = plan.K;
    p.ldx = plan.ldx;
    p.x = static_cast<const __nv_bfloat16 *>(plan.x);
    p.row_slot = plan.row_slot;
    p.counters = plan.counters;
    p.n_counters = plan.n_counters;
    p.status = plan.status;
    const int sms = device_sm_count();
    int max_splits = 1, max_rank = 0;
    for (int i = 0; i < n; ++i) {
        const ProjView &v = *vs[i];
        RowProj &q = p.proj[i];
        q.N = v.N;
        q.a_arena = static_cast<const __nv_bfloat16 *>(v.a_arena);
        q.b_arena = static_cast<const __nv_bfloat16 *>(v.b_arena);
        q.table = v.table;
        q.ranks = v.ranks;
        q.scales = v.scales;
        q.max_slots = v.max_slots;
        q.bps = v.bps;
        q.num_blocks = v.num_blocks;
        q.ycorr = v.ycorr;
        // column splits: about one CTA per SM (each fits beside a GEMM CTA),
        // at least kRowThreads columns per CTA
        int splits = sms / plan.M;
        const int most = (v.N + kRowThreads - 1) / kRowThreads;
        splits = splits < 1 ? 1 : splits > most ? most : splits;
        q.cols_per_cta = ((v.N + splits - 1) / splits + kRowThreads - 1) / kRowThreads * kRowThreads;
        q.splits = (v.N + q.cols_per_cta - 1) / q.cols_per_cta;
        max_splits = q.splits > max_splits ? q.splits : max_splits;
        max_rank = v.max_rank > max_rank ? v.max_rank : max_rank;
    }
    {
        // run with the shared-memory carveout the GEMM needs, so that its CTAs
        // can be placed beside this kernel's (an SM changes its carveout only
        // when idle)
        static std::mutex mu;
        static uint64_t done_ctx[128] = {};  // per device: the context the attribute was set in
        int dev = 0;
        if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < 128) {
            std::lock_guard<std::mutex> lock(mu);
            uint64_t ctx = done_ctx[dev];
            if (first_use_in_context(&ctx)) {
                const cudaError_t e = cudaFuncSetAttribute(lora_rows_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                                           static_cast<int>(cudaSharedmemCarveoutMaxShared));
                if (e != cudaSuccess) return e;
                done_ctx[dev] = current_context_id();
            }
        }
    }
    lora_rows_kernel<<<dim3(plan.M, max_splits, n), kRowThreads, sizeof(float) * max_rank, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_lora_rows(const ForwardPlan &plan, const ProjView &v, cudaStream_t stream) {
    const ProjView *vs[1] = {&v};
    return launch_rows(plan, vs, 1, stream);
}

cudaError_t launch_lora_rows_all(const ForwardPlan &plan, cudaStream_t stream) {
    const ProjView *vs[LORA_MAX_PROJ];
    for (int i = 0; i < plan.n_proj && i < LORA_MAX_PROJ; ++i) vs[i] = &plan.proj[i];
    return launch_rows(plan, vs, plan.n_proj, stream);
}

size_t group_table_ints(int32_t M) { return 7 * static_cast<size_t>(M) + 16; }

GroupTable group_table_at(int32_t *base, int32_t M) {
    GroupTable gt;
    gt.count = base;                                // [5]
    gt.start = base + 5;                            // [M + 1]
    gt.slot = gt.start + (M + 1);                   // [M]
    gt.perm = gt.slot + M;                          // [M]
    gt.chunk_group[0] = gt.perm + M;                // [M + 1]
    gt.chunk_begin[0] = gt.chunk_group[0] + M + 1;  // [M + 2]
    gt.chunk_group[1] = gt.chunk_begin[0] + M + 2;  // [M + 1]
    gt.chunk_begin[1] = gt.chunk_group[1] + M + 1;  // [M + 2]
    return gt;
}

cudaError_t launch_group_rows(const ForwardPlan &plan, const GroupTable &gt, int32_t max_slots, cudaStream_t stream) {
    if (plan.M <= 0) return cudaSuccess;
    if (plan.M > kGroupedMaxRows) return cudaErrorInvalidValue;
    const size_t smem = sizeof(int32_t) * (3 * static_cast<size_t>(plan.M) + 1);
    group_rows_kernel<<<1, kSegThreads, smem, stream>>>(plan.M, plan.row_slot, max_slots, gt, plan.status);
    return cudaGetLastError();
}

cudaError_t launch_shrink_grouped(const ForwardPlan &plan, const ProjView &v, const GroupTable &gt,
                                  cudaStream_t stream) {
    if (plan.M <= 0) return cudaSuccess;
    GroupedShrinkParams p;
    p.M = plan.M;
    p.K = plan.K;
    p.ldx = plan.ldx;
    p.x = static_cast<const __nv_bfloat16 *>(plan.x);
    p.gt = gt;
    p.a_arena = static_cast<const __nv_bfloat16 *>(v.a_arena);
    p.table = v.table;
    p.ranks = v.ranks;
    p.max_slots = v.max_slots;
    p.bps = v.bps;
    p.num_blocks = v.num_blocks;
    p.V = v.V;
    p.ldv = v.max_rank;
    p.ksplit = plan.v_parts;
    p.kc_len = ((plan.K + p.ksplit - 1) / p.ksplit + 7) / 8 * 8;
    p.plane_stride = static_cast<size_t>(plan.M) * v.max_rank;
    p.counters = plan.counters;
    p.n_counters = plan.n_counters;
    p.status = plan.status;
    // upper bound of the items: chunks <= groups + rows / chunk rows
    const long groups = plan.M < v.max_slots ? plan.M : v.max_slots;
    const long items = (groups + plan.M / kGroupChunkRowsShrink + 1) * v.bps * p.ksplit;
    const long cap = 4L * device_sm_count();  // two CTAs per SM, two waves of items
    const int grid = static_cast<int>(items < cap ? items : cap);
    shrink_grouped_kernel<<<grid > 0 ? grid : 1, kShrThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_expand_grouped(const ForwardPlan &plan, const ProjView &v, const GroupTable &gt,
                                  cudaStream_t stream) {
    if (plan.M <= 0) return cudaSuccess;
    GroupedExpandParams p;
    p.M = plan.M;
    p.N = v.N;
    p.gt = gt;
    p.b_arena = static_cast<const __nv_bfloat16 *>(v.b_arena);
    p.table = v.table;
    p.ranks = v.ranks;
    p.scales = v.scales;
    p.max_slots = v.max_slots;
    p.bps = v.bps;
    p.num_blocks = v.num_blocks;
    p.V = v.V;
    p.ldv = v.max_rank;
    p.ksplit = plan.v_parts;
    p.plane_stride = static_cast<size_t>(plan.M) * v.max_rank;
    p.ycorr = v.ycorr;
    p.status = plan.status;
    // at most kExpRows * 1024 fp32 = 32 KiB: within the default dynamic shared memory
    const size_t smem = sizeof(float) * kExpRows * static_cast<size_t>(v.max_rank);
    const long groups = plan.M < v.max_slots ? plan.M : v.max_slots;
    const long items = (groups + plan.M / kGroupChunkRowsExpand + 2) * ((v.N + kExpCols - 1) / kExpCols);
    const long cap = 8L * device_sm_count();
    const int grid = static_cast<int>(items < cap ? items : cap);
    expand_grouped_kernel<<<grid > 0 ? grid : 1, kExpThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace lora
