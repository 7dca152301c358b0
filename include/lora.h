/*
 * lora.h — C ABI of the GB300 multi-adapter LoRA linear layer.
 *
 * The layer computes, for every row m of a mixed batch,
 *
 *     out[m,:] = W x[m,:] + (alpha_i / r_i) * B_i (A_i x[m,:])
 *
 * where i is the adapter slot of row m, or no adapter at all (-1): one dense
 * base projection shared by every row plus a rank-r_i correction of the
 * row's own adapter ("Your LoRA Adapters Are Thrashing Your GPUs", §02 "The
 * full decomposition with scaling factor"; "Adapter Residency When One
 * Replica Serves Many Fine-Tunes", §"What the forward pass has to do
 * differently"; "LoRA Adapters: Many Models in One", §"A picture" and
 * §"The model runner's part").  Shapes follow the pages: W is d x k (here
 * N x K, nn.Linear layout), A_i is r_i x K, B_i is N x r_i.
 *
 * Adapters live in a paged pool in the spirit of S-LoRA's unified paging
 * ("S-LoRA: what the paper actually says…", §"Unified paging"): fixed-size
 * blocks of LORA_BLOCK_ROWS rank-rows, addressed through a block table, so a
 * rank-r adapter holds ceil(r/16) blocks and is never padded to the maximum
 * rank ("LoRA Adapters: Many Models in One", §"Using it" describes the
 * padding this avoids).
 *
 * Conventions for every entry point
 *  - Plain C: no exceptions cross the ABI; every call returns a status.
 *  - Memory: the CALLER owns and allocates all device memory (x, W, out,
 *    arenas, block table, ranks, scales, workspace).  The library owns only
 *    host-side pool metadata.  No entry point allocates device memory.
 *  - Streams: `stream` is a cudaStream_t passed as void* (NULL = legacy
 *    default stream).  All device work is stream-ordered on it.
 *  - Alignment: every device pointer must be 16-byte aligned; K and N must
 *    be multiples of 8 (bf16) or 4 (fp32), and so must leading dimensions.
 *  - Errors detected on the host leave all state unchanged.  Errors detected
 *    by kernels (bad adapter id, unloaded slot, corrupt block-table entry,
 *    bad segment bounds, a bounded wait that ran out) skip the offending
 *    work and are recorded in a per-device status word; read it with
 *    lora_get_device_status().
 */
#ifndef LORA_H
#define LORA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LORA_ABI_VERSION 5  /* 3: lora_proj_t.w_scale (int8 base weights); 4: w_bits (int4);
                               5: lora_forward_args_t.scales (per-call scales) */
#define LORA_BLOCK_ROWS 16
#define LORA_MAX_PROJ 4

typedef enum lora_status {
    LORA_OK = 0,
    LORA_ERR_INVALID_ARG = 1,    /* NULL pointer, bad size or count */
    LORA_ERR_ALIGNMENT = 2,      /* pointer or dimension misaligned */
    LORA_ERR_DTYPE = 3,          /* dtype mismatch between call and pool */
    LORA_ERR_RANK = 4,           /* rank <= 0 or > pool max_rank */
    LORA_ERR_SLOT = 5,           /* slot out of range, or (un)loaded twice */
    LORA_ERR_OUT_OF_BLOCKS = 6,  /* pool has too few free blocks */
    LORA_ERR_ADAPTER_ID = 7,     /* a row named an id outside [-1, slots) or an empty slot */
    LORA_ERR_SEGMENTS = 8,       /* segment offsets not within [0, M] or decreasing */
    LORA_ERR_CUDA = 9,           /* a CUDA runtime call failed */
    LORA_ERR_DEVICE_TIMEOUT = 10,/* a kernel's bounded wait ran out */
    LORA_ERR_DEVICE_INDEX = 11,  /* a block-table entry outside [0, num_blocks) */
    LORA_ERR_WORKSPACE = 12,     /* workspace NULL or smaller than required */
    LORA_ERR_UNSUPPORTED = 13    /* shape or device the kernels do not support */
} lora_status_t;

typedef enum lora_dtype {
    LORA_BF16 = 0, /* bf16 inputs and outputs, fp32 accumulation */
    LORA_FP32 = 1  /* fp32 inputs and outputs, fp32 accumulation */
} lora_dtype_t;

/* ---------------------------------------------------------------------- */
/* Adapter pool                                                            */
/* ---------------------------------------------------------------------- */

/*
 * Description of one projection's adapter pool.  Block b holds 16 rank
 * indices j (16t <= j < 16t+16) of one adapter in both arenas, in `dtype`:
 *   a_arena[(b*16 + jj)*K + k]  = A_i[16t + jj][k]   (16 rows of A, width K)
 *   b_arena[(b*N + n)*16 + jj]  = B_i[n][16t + jj]   (N rows of 16 B values)
 * Slot s of rank r uses blocks block_table[s*(max_rank/16) + t] for
 * t < ceil(r/16).  Entries of a slot's last block beyond its rank are zero.
 * ranks[s] = 0 marks an empty slot, and scales[s] = alpha/r (fp32).  Unused
 * table entries are -1.
 */
typedef struct lora_pool_desc {
    lora_dtype_t dtype;
    int32_t K;            /* in-features: width of A rows; multiple of 8 (bf16) / 4 (fp32) */
    int32_t N;            /* out-features: rows of B; same rule */
    int32_t max_slots;    /* adapters that can be resident at once (>= 1) */
    int32_t max_rank;     /* largest rank accepted; multiple of 16, <= 1024 */
    int32_t num_blocks;   /* blocks in each arena (>= 1) */
    void *a_arena;        /* device, num_blocks*16*K elements */
    void *b_arena;        /* device, num_blocks*N*16 elements */
    int32_t *block_table; /* device, max_slots*(max_rank/16) int32 */
    int32_t *ranks;       /* device, max_slots int32 */
    float *scales;        /* device, max_slots fp32 */
    uint64_t free_list_seed; /* 0: blocks handed out in ascending order;
                                otherwise a seeded shuffle of the free list */
} lora_pool_desc_t;

typedef struct lora_pool lora_pool_t; /* opaque; host metadata */

/*
 * Create a pool over caller-allocated device memory.  Writes the empty
 * state (table -1, ranks 0, scales 0) on `stream` and waits for it.
 * Errors: INVALID_ARG (NULL, non-positive sizes), ALIGNMENT, RANK
 * (max_rank not a multiple of 16), CUDA.
 */
lora_status_t lora_pool_create(const lora_pool_desc_t *desc, void *stream,
                               lora_pool_t **out);

/* Free the host metadata.  Device memory stays the caller's. */
lora_status_t lora_pool_destroy(lora_pool_t *pool);

/*
 * Load adapter (A [rank][K] row-major, B [N][rank] row-major, both in the
 * pool dtype) into empty slot `slot` with scale alpha/rank.  Takes
 * ceil(rank/16) blocks from the free list, copies A's rank-rows and B's
 * columns into them (16 of each per block), zeroes the unused tail of the
 * last block, and writes the slot's table row, rank and scale.  The pages call
 * this activating an adapter into a GPU slot ("LoRA Adapters: Many Models
 * in One", §"Three tiers of storage"; "S-LoRA…", §"Unified paging").
 * src_on_device = LORA_SRC_HOST (0): A and B are host memory; the call
 *   returns once the copies are done (A/B may be freed after it returns).
 *   Where the device can address them (page-locked memory, or any memory on
 *   a Grace system), the scatter kernel below reads them directly; else they
 *   are staged block by block.
 * src_on_device = LORA_SRC_DEVICE (1): A and B are device memory; the copy
 *   is a kernel on `stream`, so A/B must stay valid until `stream` reaches
 *   that point.
 * src_on_device = LORA_SRC_MAPPED_HOST (2): A and B are page-locked host
 *   memory mapped into the device address space (cudaHostAlloc, or
 *   cudaHostRegister with cudaHostRegisterMapped; on a 64-bit system every
 *   page-locked allocation is mapped).  The same kernel reads them straight
 *   over the host link (NVLink-C2C on Grace systems), asynchronously on
 *   `stream`: A/B must stay valid and unchanged until `stream` reaches it.
 *   This is the application of adapter weights from host memory of "Adapter
 *   Residency When One Replica Serves Many Fine-Tunes" (§"Residency: which
 *   adapters stay loaded"), into the pool without a staging copy.  Host
 *   memory the device cannot address is refused (INVALID_ARG) before any
 *   access: page-locked memory always qualifies; where the GPU can address
 *   pageable memory (address translation over NVLink-C2C on Grace), any
 *   host memory does.
 * A load counts as a use of the slot for lora_pool_evict_lru.
 * Errors: SLOT (out of range or already loaded), RANK, OUT_OF_BLOCKS,
 * INVALID_ARG, ALIGNMENT (device and mapped sources must be 16-byte
 * aligned), CUDA.
 */
lora_status_t lora_pool_load_slot(lora_pool_t *pool, int32_t slot, int32_t rank,
                                  float alpha, const void *A, const void *B,
                                  int32_t src_on_device, void *stream);

#define LORA_SRC_HOST 0
#define LORA_SRC_DEVICE 1
#define LORA_SRC_MAPPED_HOST 2

/*
 * Empty slot `slot` and return its blocks to the free list.  The device
 * table/rank/scale updates are ordered on `stream`: forwards queued earlier
 * on the same stream still see the adapter, so a slot in use by queued work
 * is never torn out from under it.  Errors: SLOT (out of range or empty).
 */
lora_status_t lora_pool_unload_slot(lora_pool_t *pool, int32_t slot, void *stream);

/*
 * Residency bookkeeping for a slot cache: LRU eviction ("Your LoRA Adapters
 * Are Thrashing Your GPUs", §"Eviction: LRU by default, but routing makes it
 * rare") that never evicts an adapter in use by in-flight requests ("Multi-
 * LoRA Adapter Caching in Production…", §"Data Plane: Managing 'Where the
 * Adapter Currently Is'").  All host-side:
 * the library cannot see which slots a queued forward's row ids name, so the
 * caller pins the slots of a batch before launching its forward and unpins
 * them once the stream has passed it.
 * lora_pool_touch: marks a loaded slot as used now (recency for LRU).
 * lora_pool_pin / lora_pool_unpin: count in-flight uses of a loaded slot.
 *   A pinned slot is never evicted, and lora_pool_unload_slot refuses it
 *   (SLOT).  Unpinning a slot with no pins is an error (SLOT).
 * lora_pool_evict_lru: unloads (as lora_pool_unload_slot, ordered on
 *   `stream`) the loaded, unpinned slot used least recently, and returns it
 *   in *slot (may be NULL).  SLOT if every loaded slot is pinned or none is
 *   loaded.
 * lora_pool_slot_use: *last_use (a pool-wide use counter, 0 if empty) and
 *   *pins of a slot (either may be NULL).
 */
lora_status_t lora_pool_touch(lora_pool_t *pool, int32_t slot);
lora_status_t lora_pool_pin(lora_pool_t *pool, int32_t slot);
lora_status_t lora_pool_unpin(lora_pool_t *pool, int32_t slot);
lora_status_t lora_pool_evict_lru(lora_pool_t *pool, void *stream, int32_t *slot);
lora_status_t lora_pool_slot_use(const lora_pool_t *pool, int32_t slot, int64_t *last_use,
                                 int32_t *pins);

/* Host view of a slot: rank (0 if empty), scale, and its block ids
 * (`blocks` receives max_rank/16 entries, -1 where unused; may be NULL). */
lora_status_t lora_pool_slot_info(const lora_pool_t *pool, int32_t slot,
                                  int32_t *rank, float *scale, int32_t *blocks);

/* Blocks currently on the free list (-1 if pool is NULL). */
int32_t lora_pool_free_blocks(const lora_pool_t *pool);

/* The descriptor the pool was created with (0 on success). */
lora_status_t lora_pool_get_desc(const lora_pool_t *pool, lora_pool_desc_t *out);

/*
 * Bytes of one adapted projection's adapter, rank*(K+N)*element size: the
 * r(d+k) parameter count of "Adapter Residency…" (second paragraph) and the
 * (d_in+d_out) x rank x bytes_per_param estimate of "Multi-LoRA Adapter
 * Caching in Production…", §"Adapter Capacity Planning…".  0 on bad input.
 */
size_t lora_pool_slot_bytes(int32_t K, int32_t N, int32_t rank, lora_dtype_t dtype);

/* Device bytes a pool of this shape needs for its two arenas. */
size_t lora_pool_arena_bytes(int32_t K, int32_t N, int32_t num_blocks, lora_dtype_t dtype);

/* ---------------------------------------------------------------------- */
/* Host segmenter                                                          */
/* ---------------------------------------------------------------------- */

/*
 * Sort rows by adapter so each adapter's rows are contiguous ("Adapter
 * Residency…", §"Batch composition under many adapters"; "S-LoRA…",
 * §"Batched LoRA computation").  Stable counting sort of host ids[M] with
 * base-only rows (-1) first, then ascending slot; ties keep input order.
 * Outputs (host, caller-allocated): perm[M] (sorted position -> input row),
 * seg_offsets[num_segs+1], seg_adapter[num_segs] (-1 for the base-only
 * segment), *num_segs.  Capacity needed: M for perm and seg_adapter, M+1
 * for seg_offsets.  Empty segments are omitted.  Errors: INVALID_ARG,
 * ADAPTER_ID (an id outside [-1, num_slots)); outputs untouched on error.
 */
lora_status_t lora_segment_rows(const int32_t *ids, int32_t M, int32_t num_slots,
                                int32_t *perm, int32_t *seg_offsets,
                                int32_t *seg_adapter, int32_t *num_segs);

/* ---------------------------------------------------------------------- */
/* Forward                                                                 */
/* ---------------------------------------------------------------------- */

/*
 * One adapted projection sharing x and the row->adapter map.
 *
 * Quantized base ("Your LoRA Adapters Are Thrashing Your GPUs", §02
 * "Numerical precision: FP16 adapters on INT4 base models": the base weights
 * are stored quantized and dequantized on the fly inside the matrix
 * multiply, the adapters stay 16-bit).  With w_scale non-NULL the base
 * weight is q[n][k] * w_scale[n] (symmetric, one fp32 scale per output
 * channel) and W holds q:
 *  - w_bits 8 (or 0): int8 [N][K] row-major, K a multiple of 16;
 *  - w_bits 4: int4 in [-8, 7] packed two per byte, [N][K/2] bytes row-major,
 *    element 2j in the low nibble of byte j, 2j+1 in the high nibble; K a
 *    multiple of 32.
 * The adapters keep the pool's dtype.  Supported for bf16 x with M <= 64
 * (the decode orientation of the GEMM); other shapes return
 * LORA_ERR_UNSUPPORTED, a misaligned K LORA_ERR_ALIGNMENT, another w_bits
 * LORA_ERR_INVALID_ARG.  w_scale: device fp32 [N], 16-byte aligned.  NULL:
 * W has the pool dtype and w_bits is ignored.
 */
typedef struct lora_proj {
    const void *W;            /* device [N][K] row-major, pool dtype (int8 with w_scale) */
    const lora_pool_t *pool;  /* adapters of this projection (N, K from it) */
    void *out;                /* device [M][ldo], overwritten (not accumulated) */
    int32_t ldo;              /* row stride of out in elements, >= N */
    const float *w_scale;     /* NULL, or the quantized W's per-row scales (see above) */
    int32_t w_bits;           /* with w_scale: 8 (0 means 8) or 4 */
} lora_proj_t;

/*
 * Arguments of lora_linear_forward.  Rows reach adapters in one of two
 * forms (exactly one must be given):
 *  - per-row ids (decode, BGMV-style): row_adapter, device int32[M], each
 *    in [-1, max_slots); "LoRA Adapters…", §"The model runner's part";
 *  - sorted segments (prefill, SGMV-style): seg_offsets device int32
 *    [num_segs+1] non-decreasing within [0, M], seg_adapter device int32
 *    [num_segs], perm device int32[M] mapping sorted position -> row (NULL:
 *    identity, rows already sorted).  Positions outside every segment are
 *    base-only.  These are lora_segment_rows' outputs, copied to the device.
 * Slot ids refer to the same slot index in every projection's pool.
 */
typedef struct lora_forward_args {
    lora_dtype_t dtype;
    int32_t M;                /* rows (>= 0; 0 is a no-op) */
    int32_t K;                /* in-features */
    const void *x;            /* device [M][ldx] */
    int32_t ldx;              /* row stride of x in elements, >= K */
    int32_t n_proj;           /* 1..LORA_MAX_PROJ */
    const lora_proj_t *proj;  /* host array of n_proj projections */
    const int32_t *row_adapter;
    const int32_t *seg_offsets;
    const int32_t *seg_adapter;
    const int32_t *perm;
    int32_t num_segs;
    void *workspace;          /* device scratch, >= lora_forward_workspace_bytes */
    size_t workspace_bytes;
    /* Optional profiling hook: NULL, or 1 + 2*n_proj cudaEvent_t handles
     * (created by the caller).  The forward records event 0 on `stream`
     * before its first kernel, event 1+2p after projection p's shrink kernel
     * and event 2+2p after its GEMM, so elapsed times between them are the
     * stage durations on the launching stream. */
    void *const *stage_events;
    int32_t num_stage_events; /* 0, or exactly 1 + 2*n_proj */
    /* Optional per-call adapter scales: NULL, or device fp32 [max_slots]
     * (16-byte aligned) used for this call in place of every projection's
     * pool scales, so that row m of slot i gets scales[i] * B_i (A_i x[m]).
     * The scale belongs with the adapter ("Adapter Residency When One
     * Replica Serves Many Fine-Tunes", §"What the forward pass has to do
     * differently"); this lets a caller change an adapter's strength per
     * call without reloading it.  There is no per-call rank: a slot's rank
     * is fixed by the blocks it was loaded into, whose rank-rows past that
     * rank are zero; load the adapter again to change it. */
    const float *scales;
} lora_forward_args_t;

/* Scratch bytes lora_linear_forward needs for these arguments, 0 on invalid
 * input.  It depends on M, K, every projection's N and pool shape, the form
 * of the row map and the kernels the call will take, so this function is the
 * only exact measure of the need: size workspaces (and check calls against
 * LORA_NOALLOC_SCRATCH_BYTES) with it, not with a formula. */
size_t lora_forward_workspace_bytes(const lora_forward_args_t *args);

/*
 * out_p = x W_p^T + per-row (alpha_i/r_i) B_i (A_i x) for every projection
 * p: the two-pass structure of "S-LoRA…", §"Batched LoRA computation" (one
 * dense base GEMM over the full batch plus a batched LoRA operator over all
 * rows in one pass), with the per-adapter scale of "Adapter Residency…".
 * The rank-r intermediate (A_i x) is kept in fp32, the correction is added
 * to the fp32 accumulator, and each output is rounded once to the dtype.
 * Asynchronous on `stream`.  Host-detected errors: INVALID_ARG, ALIGNMENT,
 * DTYPE, WORKSPACE, UNSUPPORTED, CUDA.  Device-detected errors (bad ids,
 * empty slots, bad segments, corrupt table entries) skip that row's
 * correction and are reported by lora_get_device_status.
 */
lora_status_t lora_linear_forward(const lora_forward_args_t *args, void *stream);

/*
 * Size of the scratch array behind lora_linear_forward_noalloc: 16 MiB.
 */
#define LORA_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

/*
 * lora_linear_forward for callers that cannot allocate device memory.
 * (The pages have no counterpart of this entry point; it exists for
 * integration.)  Some callers have no way to obtain scratch memory: a
 * plugin inside a host framework that owns the whole device memory budget
 * and hands out none, a process that reserves all of its memory at start-up
 * under a fixed cap, or a latency-critical loop that must not call
 * cudaMalloc because an allocation can stall or synchronise the device.
 * This entry point takes the same arguments as lora_linear_forward; the
 * caller still provides x, W, the pools, the row ids or segments and the
 * outputs, but `workspace` and `workspace_bytes` are ignored.  Instead the
 * forward uses a scratch array of LORA_NOALLOC_SCRATCH_BYTES that the
 * library keeps in the memory of every device that loads it, for the life
 * of the process.  Nothing is allocated: no cudaMalloc, no cudaFree, no
 * allocating library routine.
 * Limits and rules:
 *  - Returns LORA_ERR_WORKSPACE, launching nothing, when the call needs more
 *    scratch than LORA_NOALLOC_SCRATCH_BYTES.  lora_forward_workspace_bytes
 *    on the same arguments gives the need exactly (it includes the kernels'
 *    intermediates, split-K partial tiles and counters, not only the rank-r
 *    intermediate).
 *  - The first call on a device looks up that device's copy of the array
 *    (with the device current), so make that first call before starting
 *    any stream capture on the device.  The address is kept per CUDA
 *    context: after a device reset the next call looks it up again.
 *  - Every call on a device shares the one array, and the array keeps
 *    whatever the last call left in it; the forward itself resets what must
 *    start from a known value.  Calls whose work overlaps on the GPU (for
 *    example on two streams without ordering between them) race on the
 *    array and may corrupt each other's results: order them on one stream.
 * Other errors are those of lora_linear_forward.
 */
lora_status_t lora_linear_forward_noalloc(const lora_forward_args_t *args, void *stream);

/*
 * Wait for `stream`, then read and clear this device's status word.
 * Returns LORA_OK when no kernel recorded an error, else ADAPTER_ID,
 * SEGMENTS, DEVICE_INDEX or DEVICE_TIMEOUT; *detail (may be NULL) receives
 * the row, segment or block index the first error concerned.
 */
lora_status_t lora_get_device_status(void *stream, int32_t *detail);

/*
 * Testing hook for the failure path of the kernels' bounded waits (no
 * counterpart in the pages).  Arms the next lora_linear_forward call on any
 * thread: in that call every split-K tile-counter wait of the tensor-core
 * GEMM (small M), and every wait of the large-M two-SM GEMM for a token
 * tile's LoRA intermediate, waits for one arrival more than the launch makes,
 * giving up after limit_ns (1 ms .. 2 s) instead of the normal 2 s.  The
 * waits then run out: the GEMM records LORA_ERR_DEVICE_TIMEOUT in the status
 * word, writes no output for the tiles it could not finish, releases its
 * tensor memory and ends normally (after its other bounded waits, up to a
 * few seconds), so the context stays usable.  The arming is taken by the
 * next call that passes validation and reaches the device; calls with
 * neither kind of wait take it without effect.  limit_ns = 0 disarms.
 * Errors: INVALID_ARG (limit out of range).
 */
lora_status_t lora_test_arm_wait_timeout(uint64_t limit_ns);

/* Static, human-readable name of a status code. */
const char *lora_status_string(lora_status_t status);

/* The CUDA runtime error behind the calling thread's most recent
 * LORA_ERR_CUDA from lora_linear_forward (a cudaError_t value; 0 when that
 * call saw none), and the runtime's static name for such a code. */
int32_t lora_last_cuda_error(void);
const char *lora_cuda_error_name(int32_t code);

/* LORA_ABI_VERSION of the library. */
int32_t lora_abi_version(void);

/* Kernels this library has launched in this process (all devices), for
 * accounting in benchmarks. */
uint64_t lora_kernel_launches(void);

#ifdef __cplusplus
}
#endif

#endif /* LORA_H */
