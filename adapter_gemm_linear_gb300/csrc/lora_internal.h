// Internal declarations shared by the host library and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "lora.h"

// Host-side pool metadata.  Device state (table, ranks, scales, arenas) lives
// in caller memory; the vectors here mirror it so that loads and unloads can
// be validated without reading the device.
struct lora_pool {
    lora_pool_desc_t d;
    int bps;                       // blocks per slot = max_rank / 16
    int device;                    // CUDA device the pool was created on
    std::vector<int32_t> free_list;  // stack: back() is handed out next
    std::vector<int32_t> rank;       // [max_slots], 0 = empty
    std::vector<float> scale;        // [max_slots]
    std::vector<int32_t> table;      // [max_slots * bps], -1 = unused
    std::vector<int64_t> last_use;   // [max_slots] use clock at the last load or touch, 0 = empty
    std::vector<int32_t> pins;       // [max_slots] in-flight uses (never evicted while > 0)
    int64_t use_clock = 0;
};

namespace lora {

constexpr int kMaxRankLimit = 1024;               // largest pool max_rank
constexpr int kMaxBlocksPerSlot = kMaxRankLimit / LORA_BLOCK_ROWS;

// Codes kernels record in the per-device status word (first error wins).
enum DeviceError : uint32_t {
    kDevOk = 0,
    kDevBadAdapter = 1,   // id outside [-1, max_slots); detail = row
    kDevEmptySlot = 2,    // row names a slot with rank 0; detail = row
    kDevBadBlock = 3,     // table entry outside [0, num_blocks) or bad rank; detail = slot
    kDevBadSegment = 4,   // segment offsets out of order / range, or perm row out of range
    kDevTimeout = 5,      // a bounded mbarrier wait ran out; detail = kernel site
};

// Device address of this device's status word (a 64-bit word holding
// code << 32 | detail).  Looked up once per CUDA context of each device.
cudaError_t device_status_ptr(unsigned long long **out);

// Process-unique id of the calling thread's current CUDA context (the
// driver's cuCtxGetId), or 0 when there is none or the driver cannot say.
// Per-device caches of device addresses and function attributes key on it,
// so that a device reset (a new primary context) invalidates them.
uint64_t current_context_id();

// Whether the per-device entry *slot records a context other than the
// current one (or none); if so it records the current one.  For one-time
// set-up per context (a function attribute, a symbol address).  A zero
// context id (unknown) always counts as new.
bool first_use_in_context(uint64_t *slot);

// Element size of a dtype.
inline size_t dtype_bytes(lora_dtype_t t) { return t == LORA_FP32 ? 4 : 2; }

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Per-projection view handed to the kernel launchers.
struct ProjView {
    const void *W;
    const float *w_scale;  // NULL, or W is quantized with these per-row scales
    int32_t w_bits;        // with w_scale: 8 (int8) or 4 (packed int4)
    void *out;
    int32_t N, ldo;
    const void *a_arena, *b_arena;
    const int32_t *table;
    const int32_t *ranks;
    const float *scales;
    int32_t max_slots, bps, num_blocks, max_rank;
    float *V;              // workspace: [v_parts][M][max_rank] fp32
    float *ycorr;          // workspace: fp32 [M][N] LoRA correction of the small-M orientation
    // large M in bf16: the LoRA term on the tensor cores (lora_tiles.cu).  Per
    // 128-token tile, the pool blocks of the slots its rows use (tile_plan);
    // Vt holds s_i V of each row as bf16 hi and lo parts per block entry; the
    // GEMM adds them times the blocks' B as extra MMAs.
    int32_t lora_tiles;    // 1: this path (tile_plan, vacc, vt set)
    int32_t *tile_plan;    // workspace: int32 [tiles][kPlanInts]
    float *vacc;           // workspace: fp32 V accumulator, [plan tiles][256 columns][kPlanRows] (column-major per tile)
    void *vt;              // workspace: bf16 [tiles * kPlanRows][kVtCols]
    int32_t shrink_grid;   // CTAs of the tensor-core shrink
};

// Large-M LoRA term (lora_tiles.cu).  A plan tile is 256 tokens: the token
// tile of the two-SM GEMM, two tiles of the one-SM GEMM and of the shrink;
// its record: [0] = nb, the pool blocks it lists (-1: more than
// kPlanMaxBlocks, rows take the CUDA-core fallback), [kPlanReadyOff] = how
// many CTAs of the two-SM GEMM have written the tile's Vt (or fallback V),
// [kPlanPartOff + r] = how many K-slices of the tile's V the GEMM's CTAs of
// rank r have stored, and in tile 0's record [kPlanQueueOff] = the main
// units the two-SM GEMM has handed out past its first round (all zeroed by
// the plan kernel),
// [kPlanBlkOff + e] = block id and [kPlanSlotOff + e] = slot of entry e.
constexpr int kPlanRows = 256;
constexpr int kPlanMaxBlocks = 16;
constexpr int kPlanInts = 48;
constexpr int kPlanReadyOff = 1;
constexpr int kPlanPartOff = 2;  // two entries, one per CTA rank of a pair
constexpr int kPlanQueueOff = 4;
constexpr int kPlanBlkOff = 16;
constexpr int kPlanSlotOff = 32;
constexpr int kVtCols = 2 * LORA_BLOCK_ROWS * kPlanMaxBlocks;  // hi parts, then lo parts

// Rows grouped by adapter slot (device int32 arrays in the workspace):
// count[0] = G groups; group g holds the sorted positions [start[g],
// start[g+1]) and slot[g]; perm[i] = the row at sorted position i; positions
// start[G] .. M-1 are the rows without an adapter.  The groups are cut into
// two lists of chunks, the grouped kernels' work items: list L cuts every
// group into chunks of at most kGroupChunkRowsShrink (L = 0) or
// kGroupChunkRowsExpand (L = 1) positions; chunk c covers
// positions [chunk_begin[L][c], chunk_begin[L][c+1]) of group chunk_group[L][c].
// count[1 + 2L] chunks belong to groups, count[2 + 2L] >= count[1 + 2L] also
// cover the rows without an adapter (chunk_group = G).  List 0 feeds the
// shrink (short chunks: many items), list 1 the expand (long chunks: each B
// piece serves more rows).
constexpr int kGroupChunkRowsShrink = 8;   // list 0
constexpr int kGroupChunkRowsExpand = 32;  // list 1
struct GroupTable {
    int32_t *count;           // [5]
    int32_t *start;           // [M + 1]
    int32_t *slot;            // [M]
    int32_t *perm;            // [M]
    int32_t *chunk_group[2];  // [M + 1] each
    int32_t *chunk_begin[2];  // [M + 2] each
};
constexpr int kGroupedMaxRows = 2048;  // rows the group table is built for (shared memory of its kernel)
constexpr int kMaxVPlanes = 4;         // K slices of the grouped shrink
constexpr int kPipeMaxRows = 512;      // rows the pipelined grouped kernels sort in shared memory
constexpr int kPipeMaxRank = 128;      // pool max_rank of the pipelined grouped kernels
constexpr int kQuantMaxRows = 64;      // int8 base weights: rows of x (token tiles of 32 or 64)

struct ForwardPlan {
    lora_dtype_t dtype;
    int32_t M, K, ldx;
    const void *x;
    const int32_t *row_slot;  // per-row slot ids (device)
    int n_proj;
    ProjView proj[LORA_MAX_PROJ];
    unsigned long long *status;
    void *const *stage_events;  // NULL or 1 + 2*n_proj cudaEvent_t
    float *part;                // workspace: split-K partial tiles
    float *ycorr;               // workspace: fp32 [M][N] LoRA correction (small-M orientation)
    int32_t *group_table;       // workspace: GroupTable storage (small-M orientation)
    void *pipe_groups;          // workspace: one row grouping per projection for the pipelined kernels
    int32_t *counters;          // workspace: split-K tile counters, zeroed by the shrink
    int32_t n_counters;         // entries of `counters`
    int v_parts;                // K-slice planes of V the shrink writes
    // small M, every projection's LoRA term by the per-row kernel: one launch
    // of it for all projections (each its own ycorr), then the GEMMs two
    // projections per launch (each launch its own split-K counters)
    bool fused_rows;
    // small M, every projection's LoRA term by the pipelined grouped kernels:
    // one shrink and one expand launch for all projections (each its own
    // ycorr), then the GEMMs two projections per launch (each launch its own
    // split-K counters)
    bool piped_pairs;
    // lora_test_arm_wait_timeout: 0, or the time limit of this call's split-K
    // counter waits, which then wait for one arrival more than any launch makes
    uint64_t test_wait_limit_ns;
    // sorted segments without a permutation on the large-M path: the tile plan
    // kernel derives every row's slot from them and writes row_slot itself
    const int32_t *seg_offsets, *seg_adapter;
    int32_t num_segs;
    bool rows_in_plan;
};

// Count of kernels launched by the library (lora_kernel_launches).
void count_launches(int n);

// Workspace layout of one forward call.
struct WorkspaceLayout {
    size_t row_slot_off;          // int32[M] (segment mode only)
    size_t v_off[LORA_MAX_PROJ];  // fp32[M][max_rank]
    size_t part_off;              // fp32 split-K partial tiles (largest projection)
    size_t ycorr_off;             // fp32 [M][N] correction of the small-M orientation (largest projection)
    size_t group_off;             // int32 group table (small-M orientation)
    size_t pipe_group_off;        // the pipelined kernels' row groupings, one per projection
    size_t plan_off, vacc_off, vt_off;  // large-M tensor-core LoRA term
    size_t counter_off;           // int32 per output tile (split-K)
    size_t total;
};

// Tensor-core GEMM launch plan (tc_gemm.cu): orientation, tile width, split-K.
struct TcPlan {
    bool swap;            // W rows on the TMEM lanes, tokens as the MMA's N
    int bn;               // MMA N (tokens when swapped, output columns otherwise)
    int num_kb, kb_per_split, splits;
    int full_units;       // units that are whole tiles (the rest: split_tiles tiles in `splits` K ranges)
    int split_tiles;
    int tiles_a, tiles_b, units, grid;
    size_t part_bytes, counter_bytes;  // split-K partial tiles and tile counters
};

// Launchers (lora_kernels.cu).
cudaError_t launch_segments_to_rows(int32_t M, const int32_t *seg_offsets,
                                    const int32_t *seg_adapter, const int32_t *perm,
                                    int32_t num_segs, int32_t *row_slot,
                                    unsigned long long *status, cudaStream_t stream);
// Copy a device-resident adapter (A [rank][K], B [N][rank]) into the blocks
// `blocks` (host array of ceil(rank/16) ids) in the arena layouts of
// lora_pool_desc_t, zeroing the entries past `rank` in the last block.
cudaError_t launch_pool_scatter(const lora_pool *pool, int32_t rank, const int32_t *blocks,
                                const void *A, const void *B, cudaStream_t stream);
cudaError_t launch_forward(const ForwardPlan &plan, cudaStream_t stream);

// Multiprocessors of the current device (cached per device; 148 if unknown).
int device_sm_count();

// Large M with the LoRA term on the tensor cores (lora_tiles.cu): the tile
// plan (block lists; per-row V of fallback tiles), then the tensor-core
// shrink into Vt; the main GEMM adds Vt x B_block^T per listed block.
int tc_shrink_grid(int32_t M, int32_t K);
size_t tc_shrink_acc_bytes(int32_t M);
cudaError_t launch_tile_plan(const ForwardPlan &plan, const ProjView &v, cudaStream_t stream);
// The shrink and the convert kernel after it (Vt, and V of fallback tiles).
cudaError_t launch_tc_shrink(const ForwardPlan &plan, const ProjView &v, cudaStream_t stream);

// The small-M LoRA path by adapter group (lora_grouped.cu): the rows' group
// table (rows sorted by slot), then per projection the grouped shrink into
// plan.v_parts K-slice planes of V and the grouped expand into plan.ycorr
// ([M][N] fp32, zero for rows without an adapter).
int grouped_v_planes(int32_t K);
// Rows few and ranks small enough for the per-row LoRA kernel (one kernel:
// v = A_i x[m] in shared memory, then ycorr[m, :]); otherwise the grouped path.
bool row_lora_preferred(int32_t M, int32_t K, int32_t N, int32_t max_rank);
cudaError_t launch_lora_rows(const ForwardPlan &plan, const ProjView &v, cudaStream_t stream);
// Whether a call of n projections (widths N, pool max ranks max_rank) takes
// the fused per-row path (ForwardPlan::fused_rows).
bool fuse_row_projections(int32_t M, int32_t K, int n, const int32_t *N, const int32_t *max_rank);
// The per-row kernel over every projection of the plan in one launch.
cudaError_t launch_lora_rows_all(const ForwardPlan &plan, cudaStream_t stream);
size_t group_table_ints(int32_t M);
GroupTable group_table_at(int32_t *base, int32_t M);
cudaError_t launch_group_rows(const ForwardPlan &plan, const GroupTable &gt, int32_t max_slots, cudaStream_t stream);
cudaError_t launch_shrink_grouped(const ForwardPlan &plan, const ProjView &v, const GroupTable &gt,
                                  cudaStream_t stream);
cudaError_t launch_expand_grouped(const ForwardPlan &plan, const ProjView &v, const GroupTable &gt,
                                  cudaStream_t stream);
// The same path as two pipelined persistent kernels (lora_pipe.cu), each of
// which groups the rows itself: the shrink writes plan.v_parts K-slice planes
// of V with rows in sorted order, the expand plan.ycorr.  For M <=
// kPipeMaxRows and pools of max_rank <= kPipeMaxRank.
bool pipe_grouped_supported(int32_t M, int32_t max_rank);
// Whether a call of n projections takes the pipelined kernels with the GEMMs
// two projections per launch (ForwardPlan::piped_pairs): small M, LoRA terms
// not all for the per-row kernel, every pool within the pipelined kernels'
// rank limit, no quantized base weights.
bool pipe_pair_projections(int32_t M, int32_t K, int n, const int32_t *N, const int32_t *max_rank, bool any_quant);
// The rows grouped by adapter once per forward for every projection (one CTA
// each, into plan.pipe_groups), read by both pipelined kernels.
size_t pipe_group_bytes();
cudaError_t launch_pipe_group(const ForwardPlan &plan, cudaStream_t stream);
// The pipelined shrink (expand) of projections vs[0..n) (elements of
// plan.proj) in one launch, the SMs split between them by the bytes of A (B)
// a row's adapter brings at most.
cudaError_t launch_pipe_shrink(const ForwardPlan &plan, const ProjView *const *vs, int n, cudaStream_t stream);
cudaError_t launch_pipe_expand(const ForwardPlan &plan, const ProjView *const *vs, int n, cudaStream_t stream);

// Tensor-core base GEMM with the fused expand epilogue (tc_gemm.cu), bf16.
TcPlan plan_tc(int32_t M, int32_t N, int32_t K);
cudaError_t launch_gemm_lora_tc(const ForwardPlan &plan, const ProjView &v, cudaStream_t stream);
// Large M: whether the projection's GEMM is the two-SM kernel, which also
// computes the LoRA term's V itself (only the plan kernel runs before it);
// otherwise the shrink and convert kernels of lora_tiles.cu run first.
bool pair_gemm_takes(const ProjView &v);
// Its fp32 scratch for the K-slices of V (in ProjView::vacc): bytes for M rows.
size_t pair_vpart_bytes(int32_t M);
// Swapped orientation: projections v0 and (if not NULL) v1 of the same x in
// one launch, with its own split-K tile counters.
TcPlan plan_tc_pair(int32_t M, int32_t N0, int32_t N1, int32_t K);
cudaError_t launch_gemm_lora_tc_pair(const ForwardPlan &plan, const ProjView &v0, const ProjView *v1,
                                     int32_t *counters, int64_t n_counters, cudaStream_t stream);

}  // namespace lora
