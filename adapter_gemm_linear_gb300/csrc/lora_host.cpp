// Host side of the C ABI: adapter pool management, the row segmenter,
// argument validation and forward dispatch.  No entry point here allocates
// device memory; every device buffer is the caller's.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <new>
#include <vector>

#include "lora_internal.h"

static std::atomic<uint64_t> g_kernel_launches{0};
static std::atomic<uint64_t> g_test_wait_limit_ns{0};  // lora_test_arm_wait_timeout: armed limit, 0 = off
static thread_local int32_t g_last_cuda_error = 0;  // behind this thread's last forward LORA_ERR_CUDA

void lora::count_launches(int n) { g_kernel_launches.fetch_add(static_cast<uint64_t>(n), std::memory_order_relaxed); }

using lora::align_up;
using lora::dtype_bytes;

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int vec_elems(lora_dtype_t t) { return t == LORA_FP32 ? 4 : 8; }  // elements per 16 bytes

bool valid_dtype(lora_dtype_t t) { return t == LORA_BF16 || t == LORA_FP32; }

// splitmix64: the free-list shuffle's generator (Steele, Lea, Flood 2014).
uint64_t splitmix64(uint64_t *state) {
    uint64_t z = (*state += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

// Push the host mirror of one slot (table row, rank, scale) to the device.
lora_status_t push_slot(lora_pool *p, int32_t slot, cudaStream_t st) {
    const size_t bps = static_cast<size_t>(p->bps);
    cudaError_t e = cudaMemcpyAsync(p->d.block_table + slot * bps, p->table.data() + slot * bps,
                                    bps * sizeof(int32_t), cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(p->d.ranks + slot, p->rank.data() + slot, sizeof(int32_t),
                            cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(p->d.scales + slot, p->scale.data() + slot, sizeof(float),
                            cudaMemcpyHostToDevice, st);
    return e == cudaSuccess ? LORA_OK : LORA_ERR_CUDA;
}

}  // namespace

extern "C" {

int32_t lora_abi_version(void) { return LORA_ABI_VERSION; }

int32_t lora_last_cuda_error(void) { return g_last_cuda_error; }

const char *lora_cuda_error_name(int32_t code) { return cudaGetErrorName(static_cast<cudaError_t>(code)); }

uint64_t lora_kernel_launches(void) { return g_kernel_launches.load(std::memory_order_relaxed); }

const char *lora_status_string(lora_status_t s) {
    switch (s) {
        case LORA_OK: return "ok";
        case LORA_ERR_INVALID_ARG: return "invalid argument";
        case LORA_ERR_ALIGNMENT: return "misaligned pointer or dimension";
        case LORA_ERR_DTYPE: return "dtype mismatch";
        case LORA_ERR_RANK: return "rank out of range";
        case LORA_ERR_SLOT: return "slot out of range or in the wrong state";
        case LORA_ERR_OUT_OF_BLOCKS: return "adapter pool out of free blocks";
        case LORA_ERR_ADAPTER_ID: return "row names an invalid or empty adapter slot";
        case LORA_ERR_SEGMENTS: return "invalid segment offsets or permutation";
        case LORA_ERR_CUDA: return "CUDA runtime error";
        case LORA_ERR_DEVICE_TIMEOUT: return "kernel wait timed out";
        case LORA_ERR_DEVICE_INDEX: return "block table entry out of range";
        case LORA_ERR_WORKSPACE: return "workspace missing or too small";
        case LORA_ERR_UNSUPPORTED: return "unsupported shape or device";
    }
    return "unknown status";
}

size_t lora_pool_slot_bytes(int32_t K, int32_t N, int32_t rank, lora_dtype_t dtype) {
    if (K <= 0 || N <= 0 || rank <= 0 || !valid_dtype(dtype)) return 0;
    return static_cast<size_t>(rank) * (static_cast<size_t>(K) + static_cast<size_t>(N)) *
           dtype_bytes(dtype);
}

size_t lora_pool_arena_bytes(int32_t K, int32_t N, int32_t num_blocks, lora_dtype_t dtype) {
    if (K <= 0 || N <= 0 || num_blocks <= 0 || !valid_dtype(dtype)) return 0;
    return static_cast<size_t>(num_blocks) * LORA_BLOCK_ROWS *
           (static_cast<size_t>(K) + static_cast<size_t>(N)) * dtype_bytes(dtype);
}

lora_status_t lora_pool_create(const lora_pool_desc_t *desc, void *stream, lora_pool_t **out) {
    if (!desc || !out) return LORA_ERR_INVALID_ARG;
    const lora_pool_desc_t &d = *desc;
    if (!valid_dtype(d.dtype)) return LORA_ERR_DTYPE;
    if (d.K <= 0 || d.N <= 0 || d.max_slots <= 0 || d.num_blocks <= 0 || d.max_rank <= 0)
        return LORA_ERR_INVALID_ARG;
    if (d.max_rank % LORA_BLOCK_ROWS != 0 || d.max_rank > lora::kMaxRankLimit)
        return LORA_ERR_RANK;
    if (!d.a_arena || !d.b_arena || !d.block_table || !d.ranks || !d.scales)
        return LORA_ERR_INVALID_ARG;
    if (!aligned16(d.a_arena) || !aligned16(d.b_arena) || !aligned16(d.block_table) ||
        !aligned16(d.ranks) || !aligned16(d.scales))
        return LORA_ERR_ALIGNMENT;
    if (d.K % vec_elems(d.dtype) || d.N % vec_elems(d.dtype)) return LORA_ERR_ALIGNMENT;

    lora_pool *p = new (std::nothrow) lora_pool();
    if (!p) return LORA_ERR_INVALID_ARG;
    try {
        p->d = d;
        p->bps = d.max_rank / LORA_BLOCK_ROWS;
        p->rank.assign(d.max_slots, 0);
        p->scale.assign(d.max_slots, 0.0f);
        p->table.assign(static_cast<size_t>(d.max_slots) * p->bps, -1);
        p->last_use.assign(d.max_slots, 0);
        p->pins.assign(d.max_slots, 0);
        // free list as a stack: back() is handed out first
        p->free_list.resize(d.num_blocks);
        for (int32_t b = 0; b < d.num_blocks; ++b) p->free_list[b] = d.num_blocks - 1 - b;
        if (d.free_list_seed != 0) {
            uint64_t st = d.free_list_seed;
            for (int32_t i = d.num_blocks - 1; i > 0; --i) {
                int32_t j = static_cast<int32_t>(splitmix64(&st) % static_cast<uint64_t>(i + 1));
                std::swap(p->free_list[i], p->free_list[j]);
            }
        }
    } catch (...) {
        delete p;
        return LORA_ERR_INVALID_ARG;
    }
    if (cudaGetDevice(&p->device) != cudaSuccess) {
        delete p;
        return LORA_ERR_CUDA;
    }
    cudaStream_t st = as_stream(stream);
    cudaError_t e = cudaMemcpyAsync(d.block_table, p->table.data(), p->table.size() * sizeof(int32_t),
                                    cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess)
        e = cudaMemsetAsync(d.ranks, 0, sizeof(int32_t) * d.max_slots, st);
    if (e == cudaSuccess)
        e = cudaMemsetAsync(d.scales, 0, sizeof(float) * d.max_slots, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) {
        delete p;
        return LORA_ERR_CUDA;
    }
    *out = p;
    return LORA_OK;
}

lora_status_t lora_pool_destroy(lora_pool_t *pool) {
    if (!pool) return LORA_ERR_INVALID_ARG;
    delete pool;
    return LORA_OK;
}

int32_t lora_pool_free_blocks(const lora_pool_t *pool) {
    return pool ? static_cast<int32_t>(pool->free_list.size()) : -1;
}

lora_status_t lora_pool_get_desc(const lora_pool_t *pool, lora_pool_desc_t *out) {
    if (!pool || !out) return LORA_ERR_INVALID_ARG;
    *out = pool->d;
    return LORA_OK;
}

lora_status_t lora_pool_slot_info(const lora_pool_t *pool, int32_t slot, int32_t *rank,
                                  float *scale, int32_t *blocks) {
    if (!pool) return LORA_ERR_INVALID_ARG;
    if (slot < 0 || slot >= pool->d.max_slots) return LORA_ERR_SLOT;
    if (rank) *rank = pool->rank[slot];
    if (scale) *scale = pool->scale[slot];
    if (blocks)
        memcpy(blocks, pool->table.data() + static_cast<size_t>(slot) * pool->bps,
               sizeof(int32_t) * pool->bps);
    return LORA_OK;
}

lora_status_t lora_pool_load_slot(lora_pool_t *pool, int32_t slot, int32_t rank, float alpha,
                                  const void *A, const void *B, int32_t src_on_device,
                                  void *stream) {
    if (!pool || !A || !B) return LORA_ERR_INVALID_ARG;
    lora_pool *p = pool;
    if (slot < 0 || slot >= p->d.max_slots) return LORA_ERR_SLOT;
    if (p->rank[slot] != 0) return LORA_ERR_SLOT;
    if (rank <= 0 || rank > p->d.max_rank) return LORA_ERR_RANK;
    const int nb = (rank + LORA_BLOCK_ROWS - 1) / LORA_BLOCK_ROWS;
    if (static_cast<int>(p->free_list.size()) < nb) return LORA_ERR_OUT_OF_BLOCKS;
    if (src_on_device < LORA_SRC_HOST || src_on_device > LORA_SRC_MAPPED_HOST) return LORA_ERR_INVALID_ARG;
    if (src_on_device != LORA_SRC_HOST && (!aligned16(A) || !aligned16(B))) return LORA_ERR_ALIGNMENT;
    if (src_on_device == LORA_SRC_MAPPED_HOST) {
        // the device's view of page-locked host memory; anything else is refused
        void *dA = nullptr, *dB = nullptr;
        if (cudaHostGetDevicePointer(&dA, const_cast<void *>(A), 0) != cudaSuccess ||
            cudaHostGetDevicePointer(&dB, const_cast<void *>(B), 0) != cudaSuccess || !dA || !dB) {
            (void)cudaGetLastError();  // not a sticky error: leave no trace for later calls
            return LORA_ERR_INVALID_ARG;
        }
        if (!aligned16(dA) || !aligned16(dB)) return LORA_ERR_ALIGNMENT;
        A = dA;
        B = dB;
    }

    std::vector<int32_t> blocks(nb);
    for (int t = 0; t < nb; ++t) blocks[t] = p->free_list[p->free_list.size() - 1 - t];

    cudaStream_t st = as_stream(stream);
    const size_t eb = dtype_bytes(p->d.dtype);
    const size_t K = static_cast<size_t>(p->d.K), N = static_cast<size_t>(p->d.N);
    cudaError_t e = cudaSuccess;
    bool direct = src_on_device != LORA_SRC_HOST;
    if (!direct) {
        // host memory the device can address (page-locked, or any memory where
        // the GPU translates host addresses, as over NVLink-C2C on Grace): the
        // scatter kernel reads it directly, and the call waits for it below
        void *dA = nullptr, *dB = nullptr;
        if (cudaHostGetDevicePointer(&dA, const_cast<void *>(A), 0) == cudaSuccess &&
            cudaHostGetDevicePointer(&dB, const_cast<void *>(B), 0) == cudaSuccess && dA && dB && aligned16(dA) &&
            aligned16(dB)) {
            A = dA;
            B = dB;
            direct = true;
        } else {
            (void)cudaGetLastError();  // not a sticky error: the staged copies follow
        }
    }
    if (direct) {
        e = lora::launch_pool_scatter(p, rank, blocks.data(), A, B, st);
    } else {
        // per block t: A rows 16t.. (contiguous) and B columns 16t..16t+15
        // gathered on the host into the block's [N][16] layout
        std::vector<unsigned char> bblk;
        try {
            bblk.resize(N * LORA_BLOCK_ROWS * eb);
        } catch (...) {
            return LORA_ERR_INVALID_ARG;
        }
        const unsigned char *a_src = static_cast<const unsigned char *>(A);
        const unsigned char *b_src = static_cast<const unsigned char *>(B);
        unsigned char *a_arena = static_cast<unsigned char *>(p->d.a_arena);
        unsigned char *b_arena = static_cast<unsigned char *>(p->d.b_arena);
        for (int t = 0; t < nb && e == cudaSuccess; ++t) {
            const size_t b = static_cast<size_t>(blocks[t]);
            const size_t j0 = static_cast<size_t>(t) * LORA_BLOCK_ROWS;
            const size_t rows = std::min<size_t>(LORA_BLOCK_ROWS, rank - j0);
            unsigned char *a_dst = a_arena + b * LORA_BLOCK_ROWS * K * eb;
            e = cudaMemcpyAsync(a_dst, a_src + j0 * K * eb, rows * K * eb, cudaMemcpyHostToDevice, st);
            if (e == cudaSuccess && rows < LORA_BLOCK_ROWS)
                e = cudaMemsetAsync(a_dst + rows * K * eb, 0, (LORA_BLOCK_ROWS - rows) * K * eb, st);
            if (e != cudaSuccess) break;
            // the previous block's copy must finish before the staging buffer is reused
            e = cudaStreamSynchronize(st);
            if (e != cudaSuccess) break;
            memset(bblk.data(), 0, bblk.size());
            for (size_t n = 0; n < N; ++n)
                memcpy(&bblk[n * LORA_BLOCK_ROWS * eb], b_src + (n * rank + j0) * eb, rows * eb);
            e = cudaMemcpyAsync(b_arena + b * N * LORA_BLOCK_ROWS * eb, bblk.data(), bblk.size(),
                                cudaMemcpyHostToDevice, st);
        }
        // the host staging buffer dies with this scope
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    }
    if (e != cudaSuccess) return LORA_ERR_CUDA;

    // commit: host mirror first, then the device copy of this slot's metadata
    p->free_list.resize(p->free_list.size() - nb);
    for (int t = 0; t < nb; ++t) p->table[static_cast<size_t>(slot) * p->bps + t] = blocks[t];
    p->rank[slot] = rank;
    p->scale[slot] = alpha / static_cast<float>(rank);
    p->last_use[slot] = ++p->use_clock;
    p->pins[slot] = 0;
    lora_status_t s = push_slot(p, slot, st);
    if (s == LORA_OK && src_on_device == LORA_SRC_HOST && cudaStreamSynchronize(st) != cudaSuccess)
        s = LORA_ERR_CUDA;
    return s;
}

lora_status_t lora_pool_unload_slot(lora_pool_t *pool, int32_t slot, void *stream) {
    if (!pool) return LORA_ERR_INVALID_ARG;
    lora_pool *p = pool;
    if (slot < 0 || slot >= p->d.max_slots) return LORA_ERR_SLOT;
    if (p->rank[slot] == 0) return LORA_ERR_SLOT;
    if (p->pins[slot] > 0) return LORA_ERR_SLOT;  // in use by in-flight work
    const int nb = (p->rank[slot] + LORA_BLOCK_ROWS - 1) / LORA_BLOCK_ROWS;
    int32_t *row = p->table.data() + static_cast<size_t>(slot) * p->bps;
    // blocks go back so that the most recently freed is handed out last
    for (int t = nb - 1; t >= 0; --t) {
        p->free_list.insert(p->free_list.begin(), row[t]);
        row[t] = -1;
    }
    p->rank[slot] = 0;
    p->scale[slot] = 0.0f;
    p->last_use[slot] = 0;
    return push_slot(p, slot, as_stream(stream));
}

lora_status_t lora_pool_touch(lora_pool_t *pool, int32_t slot) {
    if (!pool) return LORA_ERR_INVALID_ARG;
    if (slot < 0 || slot >= pool->d.max_slots || pool->rank[slot] == 0) return LORA_ERR_SLOT;
    pool->last_use[slot] = ++pool->use_clock;
    return LORA_OK;
}

lora_status_t lora_pool_pin(lora_pool_t *pool, int32_t slot) {
    if (!pool) return LORA_ERR_INVALID_ARG;
    if (slot < 0 || slot >= pool->d.max_slots || pool->rank[slot] == 0) return LORA_ERR_SLOT;
    ++pool->pins[slot];
    pool->last_use[slot] = ++pool->use_clock;
    return LORA_OK;
}

lora_status_t lora_pool_unpin(lora_pool_t *pool, int32_t slot) {
    if (!pool) return LORA_ERR_INVALID_ARG;
    if (slot < 0 || slot >= pool->d.max_slots || pool->rank[slot] == 0 || pool->pins[slot] <= 0)
        return LORA_ERR_SLOT;
    --pool->pins[slot];
    return LORA_OK;
}

lora_status_t lora_pool_evict_lru(lora_pool_t *pool, void *stream, int32_t *slot) {
    if (!pool) return LORA_ERR_INVALID_ARG;
    int32_t victim = -1;
    for (int32_t s = 0; s < pool->d.max_slots; ++s)
        if (pool->rank[s] != 0 && pool->pins[s] == 0 &&
            (victim < 0 || pool->last_use[s] < pool->last_use[victim]))
            victim = s;
    if (victim < 0) return LORA_ERR_SLOT;
    const lora_status_t st = lora_pool_unload_slot(pool, victim, stream);
    if (st == LORA_OK && slot) *slot = victim;
    return st;
}

lora_status_t lora_pool_slot_use(const lora_pool_t *pool, int32_t slot, int64_t *last_use, int32_t *pins) {
    if (!pool) return LORA_ERR_INVALID_ARG;
    if (slot < 0 || slot >= pool->d.max_slots) return LORA_ERR_SLOT;
    if (last_use) *last_use = pool->last_use[slot];
    if (pins) *pins = pool->pins[slot];
    return LORA_OK;
}

lora_status_t lora_segment_rows(const int32_t *ids, int32_t M, int32_t num_slots, int32_t *perm,
                                int32_t *seg_offsets, int32_t *seg_adapter, int32_t *num_segs) {
    if (M < 0 || num_slots < 0 || !seg_offsets || !num_segs) return LORA_ERR_INVALID_ARG;
    if (M > 0 && (!ids || !perm || !seg_adapter)) return LORA_ERR_INVALID_ARG;
    for (int32_t m = 0; m < M; ++m)
        if (ids[m] < -1 || ids[m] >= num_slots) return LORA_ERR_ADAPTER_ID;
    // counting sort over keys id+1 in [0, num_slots]
    std::vector<int32_t> count;
    try {
        count.assign(static_cast<size_t>(num_slots) + 2, 0);
    } catch (...) {
        return LORA_ERR_INVALID_ARG;
    }
    for (int32_t m = 0; m < M; ++m) ++count[ids[m] + 2];
    for (size_t k = 1; k < count.size(); ++k) count[k] += count[k - 1];
    // count[key+1] is now the first sorted position of key (key = id + 1)
    int32_t S = 0;
    seg_offsets[0] = 0;
    for (int32_t key = 0; key <= num_slots; ++key) {
        int32_t begin = count[key], end = count[key + 1];
        if (end > begin) {
            seg_adapter[S] = key - 1;
            seg_offsets[++S] = end;
        }
    }
    for (int32_t m = 0; m < M; ++m) perm[count[ids[m] + 1]++] = m;
    *num_segs = S;
    return LORA_OK;
}

// ---------------------------------------------------------------------------
// forward
// ---------------------------------------------------------------------------

static lora_status_t plan_forward(const lora_forward_args_t *a, lora::ForwardPlan *plan,
                                  lora::WorkspaceLayout *ws) {
    if (!a) return LORA_ERR_INVALID_ARG;
    if (!valid_dtype(a->dtype)) return LORA_ERR_DTYPE;
    if (a->M < 0 || a->K <= 0 || a->n_proj < 1 || a->n_proj > LORA_MAX_PROJ || !a->proj)
        return LORA_ERR_INVALID_ARG;
    if (a->ldx < a->K) return LORA_ERR_INVALID_ARG;
    const int ve = vec_elems(a->dtype);
    if (a->K % ve || a->ldx % ve) return LORA_ERR_ALIGNMENT;
    const bool seg_mode = a->row_adapter == nullptr;
    if (a->M > 0) {
        if (!a->x) return LORA_ERR_INVALID_ARG;
        if (!aligned16(a->x)) return LORA_ERR_ALIGNMENT;
        if (seg_mode) {
            if (a->num_segs < 0) return LORA_ERR_SEGMENTS;
            if (a->num_segs > 0 && (!a->seg_offsets || !a->seg_adapter)) return LORA_ERR_INVALID_ARG;
            if (a->seg_offsets && !aligned16(a->seg_offsets)) return LORA_ERR_ALIGNMENT;
        } else {
            if (a->seg_offsets || a->seg_adapter || a->num_segs) return LORA_ERR_INVALID_ARG;
        }
    }
    if (a->num_stage_events != 0 &&
        (a->num_stage_events != 1 + 2 * a->n_proj || !a->stage_events))
        return LORA_ERR_INVALID_ARG;
    if (a->num_stage_events == 0 && a->stage_events) return LORA_ERR_INVALID_ARG;
    if (a->scales && !aligned16(a->scales)) return LORA_ERR_ALIGNMENT;
    plan->test_wait_limit_ns = 0;
    plan->stage_events = a->stage_events;
    plan->dtype = a->dtype;
    // the small-M orientation's grouped shrink writes one V plane per K slice
    plan->v_parts = (a->dtype == LORA_BF16 && a->M > 0 && lora::plan_tc(a->M, 128, a->K).swap)
                        ? lora::grouped_v_planes(a->K)
                        : 1;
    plan->M = a->M;
    plan->K = a->K;
    plan->ldx = a->ldx;
    plan->x = a->x;
    plan->n_proj = a->n_proj;
    size_t off = 0;
    ws->row_slot_off = 0;
    if (seg_mode) off = align_up(sizeof(int32_t) * static_cast<size_t>(a->M), 256);
    for (int i = 0; i < a->n_proj; ++i) {
        const lora_proj_t &pj = a->proj[i];
        if (!pj.pool) return LORA_ERR_INVALID_ARG;
        const lora_pool_desc_t &d = pj.pool->d;
        if (d.dtype != a->dtype) return LORA_ERR_DTYPE;
        if (d.K != a->K) return LORA_ERR_INVALID_ARG;
        if (pj.ldo < d.N) return LORA_ERR_INVALID_ARG;
        if (pj.ldo % ve) return LORA_ERR_ALIGNMENT;
        if (a->M > 0) {
            if (!pj.W || !pj.out) return LORA_ERR_INVALID_ARG;
            if (!aligned16(pj.W) || !aligned16(pj.out)) return LORA_ERR_ALIGNMENT;
        }
        if (pj.w_scale) {  // quantized base weights: bf16 x, the decode orientation
            if (pj.w_bits != 0 && pj.w_bits != 8 && pj.w_bits != 4) return LORA_ERR_INVALID_ARG;
            if (a->dtype != LORA_BF16 || a->M > lora::kQuantMaxRows) return LORA_ERR_UNSUPPORTED;
            if (a->K % (pj.w_bits == 4 ? 32 : 16)) return LORA_ERR_ALIGNMENT;  // 16-byte rows
            if (!aligned16(pj.w_scale)) return LORA_ERR_ALIGNMENT;
        }
        lora::ProjView &v = plan->proj[i];
        v.W = pj.W;
        v.w_scale = pj.w_scale;
        v.w_bits = pj.w_scale ? (pj.w_bits == 4 ? 4 : 8) : 0;
        v.out = pj.out;
        v.N = d.N;
        v.ldo = pj.ldo;
        v.a_arena = d.a_arena;
        v.b_arena = d.b_arena;
        v.table = d.block_table;
        v.ranks = d.ranks;
        v.scales = a->scales ? a->scales : d.scales;  // the call's own scales, if given
        v.max_slots = d.max_slots;
        v.bps = pj.pool->bps;
        v.num_blocks = d.num_blocks;
        v.max_rank = d.max_rank;
        v.V = nullptr;
        // large M in bf16: the LoRA term on the tensor cores, per token tile
        // over the pool blocks its rows use (lora_tiles.cu); V (below) then
        // serves only tiles that take the CUDA-core fallback
        v.lora_tiles = (a->dtype == LORA_BF16 && a->M > 0 && !lora::plan_tc(a->M, d.N, a->K).swap) ? 1 : 0;
        v.tile_plan = nullptr;
        v.vacc = nullptr;
        v.vt = nullptr;
        v.shrink_grid = 0;
        ws->v_off[i] = off;
        off += align_up(sizeof(float) * static_cast<size_t>(a->M) * d.max_rank * plan->v_parts, 256);
    }
    // slot ids of every pool must mean the same adapters
    for (int i = 1; i < a->n_proj; ++i)
        if (a->proj[i].pool->d.max_slots != a->proj[0].pool->d.max_slots) return LORA_ERR_INVALID_ARG;
    // split-K scratch and the small-M orientation's correction array of the
    // tensor-core GEMM, shared by the projections (their kernels run one
    // after the other on the stream)
    // With the fused per-row path every projection keeps its own correction
    // array and each GEMM launch (two projections) its own tile counters.
    // So does the pipelined path with several projections (one LoRA launch
    // for all of them, then the GEMMs two projections per launch).
    size_t part = 0, cnt = 0, ycorr = 0;
    plan->fused_rows = false;
    plan->piped_pairs = false;
    if (a->dtype == LORA_BF16 && a->M > 0) {
        int32_t Ns[LORA_MAX_PROJ], ranks[LORA_MAX_PROJ];
        bool any_quant = false;
        for (int i = 0; i < a->n_proj; ++i) {
            Ns[i] = a->proj[i].pool->d.N;
            ranks[i] = a->proj[i].pool->d.max_rank;
            any_quant = any_quant || a->proj[i].w_scale != nullptr;
        }
        plan->fused_rows = lora::fuse_row_projections(a->M, a->K, a->n_proj, Ns, ranks);
        plan->piped_pairs =
            !plan->fused_rows && lora::pipe_pair_projections(a->M, a->K, a->n_proj, Ns, ranks, any_quant);
        if (plan->fused_rows || plan->piped_pairs) {
            for (int i = 0; i < a->n_proj; i += 2) {
                const lora::TcPlan tp = i + 1 < a->n_proj ? lora::plan_tc_pair(a->M, Ns[i], Ns[i + 1], a->K)
                                                          : lora::plan_tc(a->M, Ns[i], a->K);
                part = std::max(part, tp.part_bytes);
                cnt += tp.counter_bytes;
            }
            for (int i = 0; i < a->n_proj; ++i)
                ycorr += align_up(sizeof(float) * static_cast<size_t>(a->M) * Ns[i], 256);
        } else {
            for (int i = 0; i < a->n_proj; ++i) {
                const lora::TcPlan tp = lora::plan_tc(a->M, Ns[i], a->K);
                part = std::max(part, tp.part_bytes);
                cnt = std::max(cnt, tp.counter_bytes);
                if (tp.swap) ycorr = std::max(ycorr, sizeof(float) * static_cast<size_t>(a->M) * Ns[i]);
            }
        }
    }
    ws->part_off = off;
    off += align_up(part, 256);
    ws->ycorr_off = off;
    off += align_up(ycorr, 256);
    ws->group_off = off;
    if (ycorr) off += align_up(sizeof(int32_t) * lora::group_table_ints(a->M), 256);
    ws->pipe_group_off = off;
    if (ycorr && a->M <= lora::kPipeMaxRows) off += align_up(lora::pipe_group_bytes() * a->n_proj, 256);
    // the tensor-core LoRA term of large M: tile plans, the V accumulator and
    // Vt, shared by the projections (their kernels run one after the other
    // on the stream)
    // (the fp32 region: the shrink's accumulator for projections whose GEMM
    // is the one-SM kernel, the K-slices of V for the two-SM kernel, which
    // computes V itself)
    size_t plan_b = 0, vacc_b = 0, vt_b = 0;
    int sgrid = 0;
    if (a->n_proj > 0 && plan->proj[0].lora_tiles) {
        const size_t T = (static_cast<size_t>(a->M) + lora::kPlanRows - 1) / lora::kPlanRows;
        plan_b = sizeof(int32_t) * T * lora::kPlanInts;
        vt_b = sizeof(uint16_t) * T * lora::kPlanRows * lora::kVtCols;
        bool shrink = false, pair = false;
        for (int i = 0; i < a->n_proj; ++i) {
            const bool pg = lora::pair_gemm_takes(plan->proj[i]);
            shrink = shrink || !pg;
            pair = pair || pg;
        }
        if (shrink) {
            sgrid = lora::tc_shrink_grid(a->M, a->K);
            vacc_b = lora::tc_shrink_acc_bytes(a->M);
        }
        if (pair) vacc_b = std::max(vacc_b, lora::pair_vpart_bytes(a->M));  // the same region, used in turn
    }
    for (int i = 0; i < a->n_proj; ++i)
        plan->proj[i].shrink_grid = plan->proj[i].lora_tiles && !lora::pair_gemm_takes(plan->proj[i]) ? sgrid : 0;
    ws->plan_off = off;
    off += align_up(plan_b, 256);
    ws->vacc_off = off;
    off += align_up(vacc_b, 256);
    ws->vt_off = off;
    off += align_up(vt_b, 256);
    ws->counter_off = off;  // last: the counters run to the end of the workspace
    off += align_up(cnt, 256);
    ws->total = off;
    return LORA_OK;
}

size_t lora_forward_workspace_bytes(const lora_forward_args_t *args) {
    lora::ForwardPlan plan;
    lora::WorkspaceLayout ws;
    if (plan_forward(args, &plan, &ws) != LORA_OK) return 0;
    return ws.total > 0 ? ws.total : 256;
}

static lora_status_t linear_forward(const lora_forward_args_t *args, void *stream);

lora_status_t lora_linear_forward(const lora_forward_args_t *args, void *stream) {
    g_last_cuda_error = 0;
    const lora_status_t s = linear_forward(args, stream);
    if (s == LORA_ERR_CUDA && g_last_cuda_error == 0) g_last_cuda_error = static_cast<int32_t>(cudaGetLastError());
    return s;
}

static lora_status_t linear_forward(const lora_forward_args_t *args, void *stream) {
    lora::ForwardPlan plan;
    lora::WorkspaceLayout ws;
    lora_status_t s = plan_forward(args, &plan, &ws);
    if (s != LORA_OK) return s;
    if (args->M == 0) return LORA_OK;
    if (!args->workspace || args->workspace_bytes < ws.total) return LORA_ERR_WORKSPACE;
    if (!aligned16(args->workspace)) return LORA_ERR_ALIGNMENT;
    unsigned char *base = static_cast<unsigned char *>(args->workspace);
    if (lora::device_status_ptr(&plan.status) != cudaSuccess) return LORA_ERR_CUDA;
    for (int i = 0; i < plan.n_proj; ++i) plan.proj[i].V = reinterpret_cast<float *>(base + ws.v_off[i]);
    plan.part = reinterpret_cast<float *>(base + ws.part_off);
    plan.ycorr = reinterpret_cast<float *>(base + ws.ycorr_off);
    {
        size_t yoff = ws.ycorr_off;
        for (int i = 0; i < plan.n_proj; ++i) {
            plan.proj[i].ycorr =
                reinterpret_cast<float *>(base + (plan.fused_rows || plan.piped_pairs ? yoff : ws.ycorr_off));
            yoff += align_up(sizeof(float) * static_cast<size_t>(plan.M) * plan.proj[i].N, 256);
        }
    }
    plan.group_table = reinterpret_cast<int32_t *>(base + ws.group_off);
    plan.pipe_groups = base + ws.pipe_group_off;
    for (int i = 0; i < plan.n_proj; ++i) {
        if (!plan.proj[i].lora_tiles) continue;
        plan.proj[i].tile_plan = reinterpret_cast<int32_t *>(base + ws.plan_off);
        plan.proj[i].vacc = ws.vt_off > ws.vacc_off ? reinterpret_cast<float *>(base + ws.vacc_off) : nullptr;
        plan.proj[i].vt = base + ws.vt_off;
    }
    plan.counters = reinterpret_cast<int32_t *>(base + ws.counter_off);
    plan.n_counters = static_cast<int32_t>((ws.total - ws.counter_off) / sizeof(int32_t));
    cudaStream_t st = as_stream(stream);
    plan.test_wait_limit_ns = g_test_wait_limit_ns.exchange(0);
    plan.seg_offsets = plan.seg_adapter = nullptr;
    plan.num_segs = 0;
    plan.rows_in_plan = false;
    if (plan.stage_events &&
        cudaEventRecord(static_cast<cudaEvent_t>(plan.stage_events[0]), st) != cudaSuccess)
        return LORA_ERR_CUDA;
    if (args->row_adapter) {
        if (!aligned16(args->row_adapter)) return LORA_ERR_ALIGNMENT;
        plan.row_slot = args->row_adapter;
    } else if (!args->perm && plan.proj[0].lora_tiles) {
        // the large-M path's plan kernel turns the segments into row slots itself
        plan.row_slot = reinterpret_cast<int32_t *>(base + ws.row_slot_off);
        plan.seg_offsets = args->seg_offsets;
        plan.seg_adapter = args->seg_adapter;
        plan.num_segs = args->num_segs;
        plan.rows_in_plan = true;
    } else {
        int32_t *row_slot = reinterpret_cast<int32_t *>(base + ws.row_slot_off);
        if (cudaMemsetAsync(row_slot, 0xFF, sizeof(int32_t) * plan.M, st) != cudaSuccess)
            return LORA_ERR_CUDA;
        if (args->num_segs > 0) {
            if (lora::launch_segments_to_rows(plan.M, args->seg_offsets, args->seg_adapter, args->perm,
                                              args->num_segs, row_slot, plan.status, st) != cudaSuccess)
                return LORA_ERR_CUDA;
            lora::count_launches(1);
        }
        plan.row_slot = row_slot;
    }
    const cudaError_t e = lora::launch_forward(plan, st);
    g_last_cuda_error = static_cast<int32_t>(e);
    return e == cudaSuccess ? LORA_OK : LORA_ERR_CUDA;
}

lora_status_t lora_test_arm_wait_timeout(uint64_t limit_ns) {
    if (limit_ns != 0 && (limit_ns < 1000000ull || limit_ns > 2000000000ull)) return LORA_ERR_INVALID_ARG;
    g_test_wait_limit_ns.store(limit_ns);
    return LORA_OK;
}

lora_status_t lora_get_device_status(void *stream, int32_t *detail) {
    unsigned long long *ptr = nullptr;
    if (lora::device_status_ptr(&ptr) != cudaSuccess) return LORA_ERR_CUDA;
    cudaStream_t st = as_stream(stream);
    unsigned long long word = 0, zero = 0;
    if (cudaStreamSynchronize(st) != cudaSuccess) return LORA_ERR_CUDA;
    if (cudaMemcpyAsync(&word, ptr, sizeof(word), cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return LORA_ERR_CUDA;
    if (cudaMemcpyAsync(ptr, &zero, sizeof(zero), cudaMemcpyHostToDevice, st) != cudaSuccess)
        return LORA_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return LORA_ERR_CUDA;
    const uint32_t code = static_cast<uint32_t>(word >> 32);
    if (detail) *detail = static_cast<int32_t>(word & 0xFFFFFFFFu);
    switch (code) {
        case lora::kDevOk: return LORA_OK;
        case lora::kDevBadAdapter:
        case lora::kDevEmptySlot: return LORA_ERR_ADAPTER_ID;
        case lora::kDevBadBlock: return LORA_ERR_DEVICE_INDEX;
        case lora::kDevBadSegment: return LORA_ERR_SEGMENTS;
        case lora::kDevTimeout: return LORA_ERR_DEVICE_TIMEOUT;
    }
    return LORA_ERR_DEVICE_INDEX;
}

}  // extern "C"
