// Base GEMM on the 5th-generation tensor cores (tcgen05, fp32 accumulators in
// TMEM, operands staged by TMA) with the LoRA term added before the rounding:
//
//   out[m, n] = round( sum_k x[m,k] W[n,k]  +  s_i * sum_j B_i[n,j] V[m,j] )
//
// where i is row m's adapter slot (none: no second term), V = A_i x is the
// rank-r intermediate and s_i = alpha_i / r_i.  The correction is added to
// the fp32 accumulator, so each output is rounded to bf16 exactly once.
//
// Where the LoRA term comes from:
//   small M (swapped orientation)  the LoRA kernels before this one write the
//                whole correction as an fp32 [M][N] array (ycorr), added in
//                the epilogue;
//   large M (non-swapped)          the tensor cores add it: after a unit's
//                main k-blocks come one step per pool block of its token
//                tile's plan (lora_tiles.cu), two MMAs of K = 16 each, with
//                A = the tile's s_i V as bf16 hi and lo parts (Vt, from the
//                tensor-core shrink) and B = the block's 16 rank-columns of B
//                for the unit's output columns, loaded straight from the
//                pool's B arena; tiles whose adapters span more blocks than a
//                plan lists take a CUDA-core expand in the epilogue (V per row
//                from the plan kernel, B gathered through the block table).
//
// Persistent kernel: one CTA per SM walks a list of work units; a unit is an
// output tile (and, for split-K, one K range of it).  Two orientations:
//   non-swapped  (large M): the MMA's M = 128 token rows of x, its N = BN
//                columns of W; TMEM lane = token, TMEM column = output column.
//   swapped      (small M): the MMA's M = 128 rows of W (output columns), its
//                N = BN tokens (up to 256: one tile for up to 256 tokens, so
//                each MMA instruction does the most work); TMEM lane = output
//                column, column = token.  With few tokens this puts W's rows on
//                the 128 lanes, and split-K spreads each tile's K range over
//                several CTAs so that ~all SMs stream W; with more tiles than
//                SMs only the last round's tiles are split, over all of them.
//                The correction comes precomputed from the LoRA kernels as an
//                fp32 [M][N] array (ycorr) and is added before the rounding.
//                Under split-K each split stores its fp32 partial tile to an
//                L2-resident slice and bumps a per-tile counter; when the count
//                is complete every split sums the slices and ycorr over its own
//                range of tokens (four columns per thread, several tokens'
//                loads in flight) and stores bf16.
// Warp roles:
//   warp 0      TMA producer: A tile [128 x 64] and B tile [BN x 64] per
//               k-block into a shared-memory ring (128-byte swizzle);
//   warp 1      TMEM allocator and MMA issuer: 4 tcgen05.mma (K = 16 each)
//               per k-block into one of two TMEM accumulators, so the next
//               unit's MMAs overlap the previous unit's epilogue;
//   warps 2-9   epilogue: each warp may read one 32-lane quarter of TMEM
//               (two warps per quarter, alternating 32-column chunks), reads
//               32 columns at a time with tcgen05.ld, adds the correction and
//               stores bf16 (or the fp32 partial tile under split-K).
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
#include "tensor_map.h"

namespace lora {

namespace {

constexpr int kBM = 128;               // rows of the A operand per tile (UMMA M)
constexpr int kBK = 64;                // k-block: 64 bf16 = one 128-byte swizzle row
constexpr int kUmmaK = 16;             // K of one tcgen05.mma for 16-bit inputs
constexpr int kEpiWarps = 8;   // two per TMEM lane quarter
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kThreads = 64 + kEpiThreads;
constexpr int kSmemLimit = 226 * 1024;   // dynamic shared memory per CTA (227 KiB opt-in maximum)
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far beyond any legitimate wait
constexpr int kEpiBarrier = 1;         // named barrier of the epilogue warps
constexpr uint32_t kVtBoxBytes = kBM * LORA_BLOCK_ROWS * 2;  // a [128 x 16] bf16 box of Vt
constexpr int kTaBand = 8;             // non-swapped unit order: token tiles per band

struct TcParams {
    int32_t M, N, K;
    int32_t num_kb, kb_per_split, splits;
    // units [0, full_units) are whole tiles over all of K; the rest are the
    // split_tiles tiles after them, each in `splits` K ranges (split-K)
    int32_t full_units, split_tiles;
    int32_t tiles_a, tiles_b, num_units;
    __nv_bfloat16 *out;
    int32_t ldo;
    const int32_t *row_slot;
    const __nv_bfloat16 *b_arena;
    const int32_t *table;
    const int32_t *ranks;
    const float *scales;
    int32_t max_slots, bps, num_blocks;
    const float *V;
    int32_t ldv;
    int32_t v_parts;        // K-slice planes of V, summed here
    size_t v_part_stride;   // elements between the planes
    float *part;        // split-K partial tiles [splits][tiles][BN][128] fp32 (splits > 1)
    const float *ycorr; // swapped orientation: fp32 [M][N] LoRA correction from the expand kernel
    // non-swapped orientation, LoRA term on the tensor cores: after the main
    // k-blocks, one step per pool block e listed in the token tile's plan,
    // two MMAs of K = 16: [Vt_hi | Vt_lo](tile rows, 16e:16e+16) (tma_va) times
    // the block's 16 rank-columns of B for the tile's output columns (tma_vb,
    // straight from the pool's B arena).  Tiles whose plan is -1 take the
    // CUDA-core expand in the epilogue instead (V from the plan kernel).
    int32_t lora_tiles;
    const int32_t *tile_plan;  // [token tiles][kPlanInts]
    int32_t *counters;  // per tile, zero on entry (splits > 1)
    unsigned long long *status;
    // swapped orientation, two projections of the same x in one launch: W
    // tiles [0, tiles_a0) are the first projection's (tma_a; N, out, ldo,
    // ycorr above), the rest the second's (tma_va; the fields below).  With
    // one projection tiles_a0 = tiles_a.
    int32_t tiles_a0;
    int32_t N1, ldo1;
    __nv_bfloat16 *out1;
    const float *ycorr1;
    // quantized base weights (QUANT variants): W[n][k] = q[n][k] * w_scale[n],
    // q int8 (w_bits 8) or packed int4, two per byte, low nibble first (4)
    const float *w_scale;
    int32_t w_bits;
    // split-K tile-counter waits (and the two-SM kernel's Vt ready waits):
    // the arrivals expected beyond the real ones (1 only when armed for a
    // test, so that the waits run out) and their limit
    int32_t counter_extra;
    uint64_t counter_wait_ns;
    // two-SM kernel: V items, kVSplit per token tile (v_units tiles), each
    // computes one K-slice of the tile's V = x A_list^T into v_part; the last
    // slice of a CTA's rows to finish writes their Vt (vt_out), or for a
    // fallback tile the slices write the per-row V (v_rows, from x and the A
    // arena); then the plan's ready entry (plan_rw) counts the CTA
    int32_t v_units;
    __nv_bfloat16 *vt_out;
    float *v_rows;
    float *v_part;  // fp32 [v_units][kVSplit][256 rows][256 columns]: the K-slices of V
    int32_t *queue;  // main units handed out past the first round (zero on entry)
    int32_t *plan_rw;
    const __nv_bfloat16 *x;
    int32_t ldx;
    const __nv_bfloat16 *a_arena;
};

// The projection of a swapped W tile (second: the launch's second
// projection) and its fields; with one projection per launch (PAIR false)
// these are the parameters themselves.
template <bool PAIR>
struct ProjTile {
    const TcParams &p;
    bool second;
    int32_t ta;  // the tile's index within its projection
    __device__ __forceinline__ ProjTile(const TcParams &p_, int32_t ta_)
        : p(p_), second(PAIR && ta_ >= p_.tiles_a0), ta(PAIR && ta_ >= p_.tiles_a0 ? ta_ - p_.tiles_a0 : ta_) {}
    __device__ __forceinline__ int32_t N() const { return PAIR && second ? p.N1 : p.N; }
    __device__ __forceinline__ int32_t ldo() const { return PAIR && second ? p.ldo1 : p.ldo; }
    __device__ __forceinline__ __nv_bfloat16 *out() const { return PAIR && second ? p.out1 : p.out; }
    __device__ __forceinline__ const float *ycorr() const { return PAIR && second ? p.ycorr1 : p.ycorr; }
};

// QUANT (swapped only): W arrives as int8 in a staging tile of its own and
// is converted to the bf16 A tile in shared memory before the MMAs read it.
template <bool SWAP, int BN, bool QUANT = false>
struct Cfg {
    static constexpr uint32_t kABytes = kBM * kBK * 2;
    static constexpr uint32_t kBBytes = BN * kBK * 2;
    static constexpr uint32_t kQBytes = QUANT ? kBM * kBK : 0;  // int8 W staging
    // ring + barriers + TMEM address + flags + alignment slack
    static constexpr int kFixed = 1024 + (3 * 12 + 4) * 8 + 16;
    static constexpr int kStages0 = (kSmemLimit - kFixed) / static_cast<int>(kABytes + kBBytes + kQBytes);
    static constexpr int kStages = kStages0 > 12 ? 12 : kStages0;
    static constexpr uint32_t kTmemCols = 2 * BN <= 32 ? 32 : 2 * BN <= 64 ? 64 : 2 * BN <= 128 ? 128
                                        : 2 * BN <= 256 ? 256 : 512;
    static constexpr size_t kSmem = 1024 + static_cast<size_t>(kStages) * (kABytes + kBBytes + kQBytes) +
                                    ((QUANT ? 3 : 2) * kStages + 4) * 8 + 16;
    static_assert(kSmem <= kSmemLimit, "shared memory over budget");
    static_assert(kStages >= 2, "ring too small");
    // swapped with a deep ring (narrow token tiles): k-blocks whose loads are
    // issued together
    static constexpr int kLoadGroup = SWAP && kStages >= 8 ? 2 : 1;
};

struct Unit {
    int32_t ta, tb, ks;
    int32_t st;  // split-K: the tile's index among the split tiles; -1: the unit is the whole tile
};

// Units are numbered with the split fastest; for the swapped orientation the
// token tiles of one W tile come next (so they run at the same time and share
// the W tile through L2), for the non-swapped one the x tiles of one W tile
// within a band of kTaBand token tiles.  The first full_units units are whole
// tiles; the split tiles follow them.
template <bool SWAP>
__device__ __forceinline__ Unit decode_unit(int32_t u, const TcParams &p) {
    Unit w;
    int32_t r = u;
    w.ks = 0;
    w.st = -1;
    if (u >= p.full_units) {
        const int32_t v = u - p.full_units;
        w.ks = v % p.splits;
        r = p.full_units + v / p.splits;
        if (p.splits > 1) w.st = v / p.splits;
    }
    if (SWAP) {
        w.tb = r % p.tiles_b;
        w.ta = r / p.tiles_b;
    } else if (p.tiles_a > kTaBand) {
        // bands of kTaBand token tiles, each over all W tiles: a wave of CTAs
        // then streams a few MB of x (read from DRAM about once) while the W
        // tiles it shares stay in L2
        const int32_t per = kTaBand * p.tiles_b;
        const int32_t band = r / per, q = r % per;
        const int32_t rows = min(kTaBand, p.tiles_a - band * kTaBand);
        w.ta = band * kTaBand + q % rows;
        w.tb = q / rows;
    } else {
        w.ta = r % p.tiles_a;
        w.tb = r / p.tiles_a;
    }
    return w;
}

// The k-blocks [kb0, kb1) of unit w.
__device__ __forceinline__ void unit_kblocks(const TcParams &p, const Unit &w, int32_t *kb0, int32_t *kb1) {
    *kb0 = w.st < 0 ? 0 : w.ks * p.kb_per_split;
    *kb1 = w.st < 0 ? p.num_kb : min(*kb0 + p.kb_per_split, p.num_kb);
}

// Byte `j` of w as two signed int4 (low nibble first), converted exactly to
// a bf16 pair.
__device__ __forceinline__ uint32_t int4x2_to_bf16x2(uint32_t w, int j) {
    const uint32_t b = (w >> (8 * j)) & 0xFFu;
    const int lo = static_cast<int>((b & 0xFu) ^ 8u) - 8;
    const int hi = static_cast<int>((b >> 4) ^ 8u) - 8;
    return (__float_as_uint(static_cast<float>(lo)) >> 16) | (__float_as_uint(static_cast<float>(hi)) & 0xFFFF0000u);
}

// Bytes `sh` and `sh` + 1 of w as signed int8, converted exactly to a bf16
// pair (the low half takes byte sh): |v| <= 128 fits bf16's 8-bit mantissa,
// so the upper half of the float is the value.
__device__ __forceinline__ uint32_t int8x2_to_bf16x2(uint32_t w, int sh) {
    const int lo = static_cast<int8_t>(static_cast<uint8_t>(w >> (8 * sh)));
    const int hi = static_cast<int8_t>(static_cast<uint8_t>(w >> (8 * sh + 8)));
    return (__float_as_uint(static_cast<float>(lo)) >> 16) | (__float_as_uint(static_cast<float>(hi)) & 0xFFFF0000u);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);  // a -> low half, b -> high half
    return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ void epi_sync() {
    asm volatile("bar.sync %0, %1;" ::"n"(kEpiBarrier), "n"(kEpiThreads) : "memory");
}

// --------------------------------------------------------------- producer

// Extension steps of token tile ta: the pool blocks the plan of its 256-row
// plan tile lists (0 when that has no adapter rows or takes the CUDA-core
// expand).
__device__ __forceinline__ int32_t tile_ext_steps(const TcParams &p, int32_t ta) {
    const int32_t nb = p.tile_plan[static_cast<size_t>(ta / (kPlanRows / kBM)) * kPlanInts];
    return nb > 0 ? nb : 0;
}

// The idx-th work unit of this CTA (every gridDim.x-th unit), or -1.
__device__ __forceinline__ int32_t next_unit(const TcParams &p, int32_t idx) {
    const int32_t u = blockIdx.x + idx * static_cast<int32_t>(gridDim.x);
    return u < p.num_units ? u : -1;
}

// The kernel is launched as a programmatic dependent of the LoRA kernel before it:
// wait until that grid has completed and its writes are visible.  Returns at
// once when the launch had no programmatic dependency (or after the first
// call).
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <bool SWAP, int BN, bool PAIR = false, bool QUANT = false>
__device__ __forceinline__ void run_producer(const CUtensorMap *tma_a, const CUtensorMap *tma_b,
                                             const CUtensorMap *tma_va, const CUtensorMap *tma_vb,
                                             const TcParams &p, uint8_t *sA, uint8_t *sB, uint8_t *sQ,
                                             uint64_t *full, uint64_t *empty,
                                             volatile uint32_t *abort_flag) {
    using namespace sm100;
    using C = Cfg<SWAP, BN, QUANT>;
    int32_t it = 0;
    for (int32_t idx = 0;; ++idx) {
        const int32_t u = next_unit(p, idx);
        if (u < 0) break;
        const Unit w = decode_unit<SWAP>(u, p);
        int32_t kb0, kb1;
        unit_kblocks(p, w, &kb0, &kb1);
        const int32_t nmain = kb1 - kb0;
        int32_t total = nmain;
        // swapped: the W tile's projection (its tensor map) and row
        const bool second = SWAP && PAIR && w.ta >= p.tiles_a0;
        const CUtensorMap *map_a = second ? tma_va : tma_a;
        const int32_t row_a = (second ? w.ta - p.tiles_a0 : w.ta) * kBM;
        for (int32_t i = 0; i < total; ++i, ++it) {
            if (!SWAP && p.lora_tiles && i == nmain - 1) {
                // with the unit's last main k-block next: the plan and Vt
                // come from the kernels before
                grid_dependency_wait();
                total = nmain + tile_ext_steps(p, w.ta);
            }
            if (C::kLoadGroup > 1 && i % C::kLoadGroup == 0) {
                // wait until the next kLoadGroup stages are all free,
                // so that their W boxes (adjacent 128-byte pieces of the same
                // 128 rows) reach memory together
                for (int32_t j = 1; j < C::kLoadGroup && i + j < total; ++j) {
                    const int s2 = (it + j) % C::kStages;
                    if (!mbar_wait_bounded(&empty[s2], (((it + j) / C::kStages) & 1) ^ 1, kWaitLimitNs)) {
                        record_error(p.status, kDevTimeout, 1);
                        *abort_flag = 1;
                    }
                }
            }
            const int s = it % C::kStages;
            const uint32_t ph = (it / C::kStages) & 1;
            if (!mbar_wait_bounded(&empty[s], ph ^ 1, kWaitLimitNs)) {
                record_error(p.status, kDevTimeout, 1);
                *abort_flag = 1;
            }
            if (*abort_flag) return;
            if (i < nmain) {
                mbar_arrive_expect_tx(&full[s], (QUANT ? (p.w_bits == 4 ? C::kQBytes / 2 : C::kQBytes) : C::kABytes) +
                                                    C::kBBytes);
                const int32_t kb = kb0 + i;
                if (QUANT)  // int8 (or packed int4) W into the staging tile; the epilogue warps convert it
                    tma_load_2d(sQ + s * C::kQBytes, map_a, p.w_bits == 4 ? kb * (kBK / 2) : kb * kBK, row_a,
                                &full[s]);
                else
                    tma_load_2d(sA + s * C::kABytes, map_a, kb * kBK, row_a, &full[s]);
                tma_load_2d(sB + s * C::kBBytes, tma_b, kb * kBK, w.tb * BN, &full[s]);
            } else {
                // LoRA step e: the tile's Vt hi and lo columns of block entry
                // e (32-byte swizzle, side by side in the A area) and the
                // block's B rows of this unit's output columns
                const int32_t e = i - nmain;
                const int32_t blk = p.tile_plan[static_cast<size_t>(w.ta / (kPlanRows / kBM)) * kPlanInts + kPlanBlkOff + e];
                mbar_arrive_expect_tx(&full[s], 2 * kVtBoxBytes + BN * LORA_BLOCK_ROWS * 2);
                tma_load_2d(sA + s * C::kABytes, tma_va, e * LORA_BLOCK_ROWS, w.ta * kBM, &full[s]);
                tma_load_2d(sA + s * C::kABytes + kVtBoxBytes, tma_va, kVtCols / 2 + e * LORA_BLOCK_ROWS, w.ta * kBM,
                            &full[s]);
                tma_load_2d(sB + s * C::kBBytes, tma_vb, 0, blk * p.N + w.tb * BN, &full[s]);
            }
        }
    }
}

// --------------------------------------------------------------- MMA issuer

template <bool SWAP, int BN, bool QUANT = false>
__device__ __forceinline__ void run_mma(const TcParams &p, uint8_t *sA, uint8_t *sB, uint64_t *full,
                                        uint64_t *empty, uint64_t *tmem_full, uint64_t *tmem_empty,
                                        uint32_t tmem_base, volatile uint32_t *abort_flag) {
    using namespace sm100;
    using C = Cfg<SWAP, BN, QUANT>;
    constexpr uint32_t idesc = idesc_bf16_f32(kBM, BN);
    int32_t it = 0, t = 0;
    for (int32_t idx = 0;; ++idx) {
        const int32_t u = next_unit(p, idx);
        if (u < 0) break;
        const Unit w = decode_unit<SWAP>(u, p);
        int32_t kb0, kb_main;
        unit_kblocks(p, w, &kb0, &kb_main);
        int32_t kb1 = kb_main;
        const int b = t & 1;
        bool ok = mbar_wait_bounded(&tmem_empty[b], ((t >> 1) & 1) ^ 1, kWaitLimitNs);
        if (!ok) record_error(p.status, kDevTimeout, 2);
        tc_fence_after_sync();
        const uint32_t d = tmem_base + b * BN;
        for (int32_t kb = kb0; kb < kb1 && ok; ++kb, ++it) {
            if (!SWAP && p.lora_tiles && kb == kb_main - 1) {
                // the LoRA steps follow the main k-blocks in the ring (the
                // plan comes from the kernels before)
                grid_dependency_wait();
                kb1 = kb_main + tile_ext_steps(p, w.ta);
            }
            const int s = it % C::kStages;
            const uint32_t ph = (it / C::kStages) & 1;
            if (!mbar_wait_bounded(&full[s], ph, kWaitLimitNs)) {
                record_error(p.status, kDevTimeout, 3);
                ok = false;
                break;
            }
            // a tile converted by the epilogue threads (QUANT) was written through
            // the generic proxy; TMA-filled stages need no fence
            if (QUANT) tc_fence_after_sync();
            const uint32_t a_addr = smem_u32(sA + s * C::kABytes);
            const uint32_t b_addr = smem_u32(sB + s * C::kBBytes);
            if (kb < kb_main) {
#pragma unroll
                for (int k = 0; k < kBK / kUmmaK; ++k)
                    mma_bf16_f32(d, desc_kmajor_sw128(a_addr + k * kUmmaK * 2),
                                 desc_kmajor_sw128(b_addr + k * kUmmaK * 2), idesc,
                                 (kb > kb0 || k > 0) ? 1u : 0u);
            } else {  // LoRA step: Vt_hi and Vt_lo times the block's B, K = 16 each
                mma_bf16_f32(d, desc_kmajor_sw32(a_addr), desc_kmajor_sw32(b_addr), idesc, 1u);
                mma_bf16_f32(d, desc_kmajor_sw32(a_addr + kVtBoxBytes), desc_kmajor_sw32(b_addr), idesc, 1u);
            }
            mma_commit(&empty[s]);
        }
        if (!ok || *abort_flag) {
            *abort_flag = 1;
            mbar_arrive(&tmem_full[b]);  // wake the epilogue so it can unwind
            return;
        }
        mma_commit(&tmem_full[b]);
        ++t;
    }
}

// --------------------------------------------------------------- epilogue

// AND of `v` over the epilogue threads, also a barrier among them.
__device__ __forceinline__ bool epi_all(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(v ? 1u : 0u), "n"(kEpiBarrier), "n"(kEpiThreads)
        : "memory");
    return r != 0;
}

// Non-swapped orientation: this thread owns token row m (adapter slot, rank
// r, scale s); the 32 values in acc are output columns n0 .. n0+31.  The
// correction for 8 columns at a time keeps 8 independent accumulators.
__device__ __forceinline__ void rows_finish_chunk(const TcParams &p, int32_t slot, int32_t r, float s,
                                                  int32_t m, int32_t n0, float (&acc)[32]) {
    if (slot < 0 || n0 >= p.N) return;
    const float *vrow = p.V + static_cast<size_t>(m) * p.ldv;
    const int32_t *trow = p.table + static_cast<size_t>(slot) * p.bps;
    float lo[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) lo[e] = 0.0f;
#pragma unroll 1
    for (int32_t jb = 0; jb * LORA_BLOCK_ROWS < r; ++jb) {
        const int32_t blk = trow[jb];
        if (blk < 0 || blk >= p.num_blocks) {
            record_error(p.status, kDevBadBlock, static_cast<uint32_t>(slot));
            return;
        }
        float v[16];
        const float4 *vsrc = reinterpret_cast<const float4 *>(vrow + jb * LORA_BLOCK_ROWS);
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            float4 q = vsrc[g];
            for (int32_t pl = 1; pl < p.v_parts; ++pl) {  // K-slice planes of the shrink
                const float4 w2 = vsrc[g + pl * (p.v_part_stride / 4)];
                q.x += w2.x; q.y += w2.y; q.z += w2.z; q.w += w2.w;
            }
            v[4 * g] = q.x;
            v[4 * g + 1] = q.y;
            v[4 * g + 2] = q.z;
            v[4 * g + 3] = q.w;
        }
        const uint4 *bsrc = reinterpret_cast<const uint4 *>(
            p.b_arena + (static_cast<size_t>(blk) * p.N + n0) * LORA_BLOCK_ROWS);
        const int valid = min(32, p.N - n0);  // a multiple of 8
#pragma unroll
        for (int eg = 0; eg < 4; ++eg) {
            if (eg * 8 >= valid) break;
            // columns n0 + 8eg .. +7: 16 B values each, as 2 x 16 bytes
            uint4 q[8][2];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                q[e][0] = __ldg(bsrc + 2 * (eg * 8 + e));
                q[e][1] = __ldg(bsrc + 2 * (eg * 8 + e) + 1);
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
                for (int w = 0; w < 4; ++w) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const uint32_t word = w == 0 ? q[e][h].x : w == 1 ? q[e][h].y : w == 2 ? q[e][h].z : q[e][h].w;
                        lo[eg * 8 + e] = fmaf(__uint_as_float(word << 16), v[h * 8 + 2 * w], lo[eg * 8 + e]);
                        lo[eg * 8 + e] = fmaf(__uint_as_float(word & 0xFFFF0000u), v[h * 8 + 2 * w + 1],
                                              lo[eg * 8 + e]);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int e = 0; e < 32; ++e) acc[e] = fmaf(s, lo[e], acc[e]);
}

__device__ __forceinline__ void load_tmem_chunk(uint32_t taddr, float (&acc)[32]) {
    uint32_t raw[32];
    sm100::tmem_ld_32x32b_x32(taddr, raw);
    sm100::tmem_ld_wait(raw);
#pragma unroll
    for (int e = 0; e < 32; ++e) acc[e] = __uint_as_float(raw[e]);
}

// Split-K finish of the swapped orientation: each thread sums four adjacent
// output columns (16-byte loads of the tile's partial slices and of the
// correction; N and ldo are multiples of 8, which the host checks), the
// eight token lanes of the epilogue step through this split's share of the
// tokens [e_begin, e_end), and every load of a batch of kR tokens is in
// flight before the sums.
template <int BN, bool PAIR, bool QUANT>
__device__ __forceinline__ void finish_split_vec4(const TcParams &p, const ProjTile<PAIR> &pt, int32_t tb,
                                                  const float *tile_part, size_t split_stride, int32_t e_begin,
                                                  int32_t e_end, int et) {
    constexpr int kR = BN <= 64 ? 2 : 4;  // within the narrow variants' register cap
    constexpr int kLanes = kEpiThreads / (kBM / 4);  // token lanes: 8
    const int cq = et % (kBM / 4), tr = et / (kBM / 4);
    const int32_t nn0 = pt.ta * kBM + 4 * cq;
    if (nn0 >= pt.N()) return;  // N % 4 == 0: the group is wholly inside or outside
    const float *col = tile_part + 4 * cq;
    const float4 wsc = QUANT ? __ldg(reinterpret_cast<const float4 *>(p.w_scale + nn0)) : make_float4(1.f, 1.f, 1.f, 1.f);
#pragma unroll 1
    for (int32_t e0 = e_begin + tr; e0 < e_end; e0 += kLanes * kR) {
        float4 a[kR], sp[kR];
#pragma unroll
        for (int r = 0; r < kR; ++r) {
            const int32_t e = e0 + kLanes * r, m = tb * BN + e;
            a[r] = (e < e_end && m < p.M)
                       ? __ldcg(reinterpret_cast<const float4 *>(pt.ycorr() + static_cast<size_t>(m) * pt.N() + nn0))
                       : make_float4(0.f, 0.f, 0.f, 0.f);
            sp[r] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll 2
        for (int32_t ks = 0; ks < p.splits; ++ks) {
#pragma unroll
            for (int r = 0; r < kR; ++r) {
                const int32_t e = e0 + kLanes * r;
                if (e < e_end) {
                    const float4 v = __ldcg(reinterpret_cast<const float4 *>(col + ks * split_stride +
                                                                            static_cast<size_t>(e) * kBM));
                    sp[r].x += v.x;
                    sp[r].y += v.y;
                    sp[r].z += v.z;
                    sp[r].w += v.w;
                }
            }
        }
#pragma unroll
        for (int r = 0; r < kR; ++r) {
            const int32_t e = e0 + kLanes * r, m = tb * BN + e;
            if (e >= e_end || m >= p.M) continue;
            // the int8 W row's scale multiplies the base sum only
            uint2 o;
            o.x = pack_bf16x2(QUANT ? fmaf(sp[r].x, wsc.x, a[r].x) : a[r].x + sp[r].x,
                              QUANT ? fmaf(sp[r].y, wsc.y, a[r].y) : a[r].y + sp[r].y);
            o.y = pack_bf16x2(QUANT ? fmaf(sp[r].z, wsc.z, a[r].z) : a[r].z + sp[r].z,
                              QUANT ? fmaf(sp[r].w, wsc.w, a[r].w) : a[r].w + sp[r].w);
            *reinterpret_cast<uint2 *>(pt.out() + static_cast<size_t>(m) * pt.ldo() + nn0) = o;
        }
    }
}

// Epilogue warps: warp w (2..2+kEpiWarps-1) may access TMEM lane quarter
// w % 4; the kEpiWarps / 4 warps sharing a quarter take turns over the
// 32-column chunks.
template <bool SWAP, int BN, bool PAIR = false, bool QUANT = false>
__device__ __forceinline__ void run_epilogue(const TcParams &p, uint8_t *sA, const uint8_t *sQ, uint64_t *full,
                                             uint64_t *conv, uint64_t *tmem_full, uint64_t *tmem_empty,
                                             uint32_t tmem_base, volatile uint32_t *abort_flag,
                                             volatile uint32_t *last_flag) {
    using namespace sm100;
    using C = Cfg<SWAP, BN, QUANT>;
    constexpr int kGroups = kEpiWarps / 4;
    constexpr int kChunks = BN / 32;
    const int et = threadIdx.x - 64;  // 0 .. kEpiThreads-1
    const int warp = threadIdx.x >> 5;
    const int q = warp & 3;           // TMEM lane quarter this warp may access
    const int grp = (warp - 2) >> 2;  // which of the warps sharing the quarter
    const int lane = threadIdx.x & 31;
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    int32_t t = 0, cit = 0;
    for (int32_t idx = 0;; ++idx) {
        const int32_t u = next_unit(p, idx);
        if (u < 0) break;
        const Unit w = decode_unit<SWAP>(u, p);
        if (QUANT) {
            // the unit's k-blocks as they land: the int8 W staging tile into
            // the bf16 A tile, laid out as a TMA load with the 128-byte
            // swizzle leaves it (16-byte chunk c of row r at chunk c ^ (r % 8)).
            // Thread et converts half hh of row r's 64 values.
            int32_t kb0, kb1;
            unit_kblocks(p, w, &kb0, &kb1);
            const int32_t nk = kb1 - kb0;
            const int r = et >> 1, hh = et & 1;
            for (int32_t i = 0; i < nk; ++i, ++cit) {
                const int s = cit % C::kStages;
                if (!mbar_wait_bounded(&full[s], (cit / C::kStages) & 1, kWaitLimitNs)) {
                    record_error(p.status, kDevTimeout, 6);
                    *abort_flag = 1;
                    break;  // without arriving: the MMA gives up too
                }
                uint8_t *row = sA + s * C::kABytes + r * (kBK * 2);
                if (p.w_bits == 4) {  // the row's 32 bytes staged; this half's 16 hold 32 values
                    const uint4 qv = *reinterpret_cast<const uint4 *>(sQ + s * C::kQBytes + r * (kBK / 2) + hh * 16);
                    const uint32_t wd[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint4 o;
                        o.x = int4x2_to_bf16x2(wd[c], 0);
                        o.y = int4x2_to_bf16x2(wd[c], 1);
                        o.z = int4x2_to_bf16x2(wd[c], 2);
                        o.w = int4x2_to_bf16x2(wd[c], 3);
                        *reinterpret_cast<uint4 *>(row + (((4 * hh + c) ^ (r & 7)) << 4)) = o;
                    }
                } else {
                    const uint4 *src = reinterpret_cast<const uint4 *>(sQ + s * C::kQBytes + r * kBK + hh * 32);
                    const uint4 q0 = src[0], q1 = src[1];
                    const uint32_t wd[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint4 o;
                        o.x = int8x2_to_bf16x2(wd[2 * c], 0);
                        o.y = int8x2_to_bf16x2(wd[2 * c], 2);
                        o.z = int8x2_to_bf16x2(wd[2 * c + 1], 0);
                        o.w = int8x2_to_bf16x2(wd[2 * c + 1], 2);
                        *reinterpret_cast<uint4 *>(row + (((4 * hh + c) ^ (r & 7)) << 4)) = o;
                    }
                }
                fence_proxy_async_shared();  // the MMAs read the tile through the async proxy
                __syncwarp();
                if (lane == 0) mbar_arrive(&conv[s]);
            }
        }
        const int b = t & 1;
        // swapped, one split: this thread's correction values (rows of its
        // 32-token chunks, its column) are fetched while the MMAs finish --
        // the first kPre chunks; each later chunk's into the slot its
        // predecessor kPre back has just used
        constexpr int kMyChunks = (kChunks + kGroups - 1) / kGroups;
        constexpr int kPre = kMyChunks <= 2 ? kMyChunks : 1;  // four chunks: one slot (registers)
        float yc[SWAP ? kPre : 1][32];
        const ProjTile<PAIR> pt(p, w.ta);
        const int32_t n_sw = pt.ta * kBM + q * 32 + lane;
        if (SWAP && w.st < 0) {
            grid_dependency_wait();  // ycorr comes from the expand kernel
#pragma unroll
            for (int ci = 0; ci < kPre; ++ci) {
                const int32_t m0 = w.tb * BN + (grp + ci * kGroups) * 32;
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    yc[ci][e] = (n_sw < pt.N() && m0 + e < p.M && grp + ci * kGroups < kChunks)
                                    ? __ldcg(pt.ycorr() + static_cast<size_t>(m0 + e) * pt.N() + n_sw)
                                    : 0.0f;
            }
        }
        bool ok = mbar_wait_bounded(&tmem_full[b], (t >> 1) & 1, kWaitLimitNs);
        if (!ok) {
            record_error(p.status, kDevTimeout, 4);
            *abort_flag = 1;
        }
        if (!epi_all(ok && !*abort_flag)) return;  // uniform over the epilogue warps
        tc_fence_after_sync();
        const uint32_t col0 = lane_addr + b * BN;

        if (SWAP) {
            const int32_t n = pt.ta * kBM + q * 32 + lane;
            const bool n_ok = n < pt.N();
            if (w.st < 0) {
#pragma unroll
                for (int ci = 0; ci < kMyChunks; ++ci) {
                    const int c = grp + ci * kGroups;
                    if (c >= kChunks) break;
                    float acc[32];
                    load_tmem_chunk(col0 + c * 32, acc);
                    const int32_t m0 = w.tb * BN + c * 32;
                    if (QUANT) {  // the int8 W row's scale
                        const float wsc = n_ok ? __ldg(p.w_scale + n) : 0.0f;
#pragma unroll
                        for (int e = 0; e < 32; ++e) acc[e] = fmaf(acc[e], wsc, yc[ci % kPre][e]);
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e) acc[e] += yc[ci % kPre][e];
                    }
                    if (ci + kPre < kMyChunks) {
                        const int c2 = grp + (ci + kPre) * kGroups;
                        const int32_t m2 = w.tb * BN + c2 * 32;
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            yc[ci % kPre][e] = (n_sw < pt.N() && m2 + e < p.M && c2 < kChunks)
                                                   ? __ldcg(pt.ycorr() + static_cast<size_t>(m2 + e) * pt.N() + n_sw)
                                                   : 0.0f;
                    }
                    if (n_ok) {
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (m0 + e < p.M)
                                pt.out()[static_cast<size_t>(m0 + e) * pt.ldo() + n] = __float2bfloat16_rn(acc[e]);
                    }
                    __syncwarp();
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tmem_empty[b]);
            } else {
                // partial tile to this split's slice; once every split of the
                // tile has stored its slice, each sums the slices and the
                // correction over its own range of the tile's tokens.  All
                // splits of a tile run at once: the split units are the last
                // round of the grid, one per CTA at most.
                const size_t tile = static_cast<size_t>(w.st);
                const size_t tiles = static_cast<size_t>(p.split_tiles);
                constexpr size_t kTileElems = static_cast<size_t>(BN) * kBM;
                float *mine = p.part + (w.ks * tiles + tile) * kTileElems + q * 32 + lane;
#pragma unroll 1
                for (int c = grp; c < kChunks; c += kGroups) {
                    float acc[32];
                    load_tmem_chunk(col0 + c * 32, acc);
#pragma unroll
                    for (int e = 0; e < 32; ++e) __stcg(mine + (c * 32 + e) * kBM, acc[e]);
                    __syncwarp();
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tmem_empty[b]);
                grid_dependency_wait();  // the counters' zeroing and ycorr precede this kernel
                __threadfence();
                epi_sync();
                if (et == 0) {
                    atomicAdd(p.counters + tile, 1);
                    const bool all =
                        wait_counter_at_least(p.counters + tile, p.splits + p.counter_extra, p.counter_wait_ns);
                    if (!all) record_error(p.status, kDevTimeout, 5);
                    *last_flag = all ? 1u : 0u;
                }
                epi_sync();
                if (*last_flag) {
                    __threadfence();
                    const int32_t per = (BN + p.splits - 1) / p.splits;
                    const int32_t e_begin = w.ks * per;
                    const int32_t e_end = min(BN, e_begin + per);
                    finish_split_vec4<BN, PAIR, QUANT>(p, pt, w.tb, p.part + tile * kTileElems, tiles * kTileElems,
                                                       e_begin, e_end, et);
                }
            }
        } else {
            grid_dependency_wait();  // the plan and V come from the kernels before
            const int32_t m = w.ta * kBM + q * 32 + lane;
            // the CUDA-core expand for rows of tiles whose adapters span too
            // many pool blocks for the LoRA steps (or without the steps at all)
            const bool per_row = !p.lora_tiles || p.tile_plan[static_cast<size_t>(w.ta / (kPlanRows / kBM)) * kPlanInts] < 0;
            int32_t r = 0, slot = -1;
            float s = 0.0f;
            if (per_row && m < p.M)
                slot = resolve_slot(p.row_slot[m], m, p.ranks, p.scales, p.max_slots, p.bps, &r, &s, p.status,
                                    false);
#pragma unroll 1
            for (int c = grp; c < kChunks; c += kGroups) {
                float acc[32];
                load_tmem_chunk(col0 + c * 32, acc);
                const int32_t n0 = w.tb * BN + c * 32;
                if (per_row) rows_finish_chunk(p, slot, r, s, m, n0, acc);
                if (m < p.M) {
                    __nv_bfloat16 *dst = p.out + static_cast<size_t>(m) * p.ldo + n0;
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        if (n0 + g * 8 < p.N) {
                            uint4 v;
                            v.x = pack_bf16x2(acc[g * 8 + 0], acc[g * 8 + 1]);
                            v.y = pack_bf16x2(acc[g * 8 + 2], acc[g * 8 + 3]);
                            v.z = pack_bf16x2(acc[g * 8 + 4], acc[g * 8 + 5]);
                            v.w = pack_bf16x2(acc[g * 8 + 6], acc[g * 8 + 7]);
                            *reinterpret_cast<uint4 *>(dst + g * 8) = v;
                        }
                    }
                }
                __syncwarp();
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tmem_empty[b]);
        }
        epi_sync();  // last_flag is rewritten by the next unit
        ++t;
    }
}

// --------------------------------------------------------------- kernel

template <bool SWAP, int BN, bool PAIR = false, bool QUANT = false>
__global__ void __maxnreg__(SWAP && BN <= 64 ? 120 : 168)
tc_gemm_lora_kernel(const __grid_constant__ CUtensorMap tma_a, const __grid_constant__ CUtensorMap tma_b,
                    const __grid_constant__ CUtensorMap tma_va, const __grid_constant__ CUtensorMap tma_vb,
                    const TcParams p) {
    using namespace sm100;
    using C = Cfg<SWAP, BN, QUANT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + C::kStages * C::kABytes;
    uint8_t *sQ = sB + C::kStages * C::kBBytes;  // QUANT: int8 W staging
    uint64_t *full = reinterpret_cast<uint64_t *>(sQ + C::kStages * C::kQBytes);
    uint64_t *empty = full + C::kStages;
    uint64_t *conv = empty + C::kStages;        // QUANT: the A tile is converted
    uint64_t *tmem_full = conv + (QUANT ? C::kStages : 0);   // [2]
    uint64_t *tmem_empty = tmem_full + 2;       // [2]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tmem_empty + 2);
    volatile uint32_t *abort_flag = tmem_slot + 1;
    volatile uint32_t *last_flag = tmem_slot + 2;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            if (QUANT) mbar_init(&conv[s], kEpiWarps);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tmem_full[b], 1);
            mbar_init(&tmem_empty[b], kEpiWarps);
        }
        *abort_flag = 0;
        *last_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tma_a);
        prefetch_tensormap(&tma_b);
        if (!SWAP && p.lora_tiles) {
            prefetch_tensormap(&tma_va);
            prefetch_tensormap(&tma_vb);
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0)
            run_producer<SWAP, BN, PAIR, QUANT>(&tma_a, &tma_b, &tma_va, &tma_vb, p, sA, sB, sQ, full, empty,
                                                abort_flag);
    } else if (warp == 1) {
        if (lane == 0)
            // with int8 W the MMAs wait for the converted tile, not the load
            run_mma<SWAP, BN, QUANT>(p, sA, sB, QUANT ? conv : full, empty, tmem_full, tmem_empty, tmem_base,
                                     abort_flag);
    } else {
        run_epilogue<SWAP, BN, PAIR, QUANT>(p, sA, sQ, full, conv, tmem_full, tmem_empty, tmem_base, abort_flag,
                                            last_flag);
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, C::kTmemCols);
    }
}


// --------------------------------------------------------------- two-SM kernel (large M)
//
// Large M in bf16 with at least 256 output columns: one MMA over a pair of
// CTAs (a cluster of two, tcgen05 cta_group::2).  A main unit is a pair tile
// of 256 tokens x kPairBN output columns; CTA r of the pair loads its 128
// token rows of x and its kPairBN/2 rows of W per k-block (32 KiB instead of
// the 48 KiB a 128 x 256 tile takes on one SM), the even CTA issues the MMAs
// (M = 256, N = kPairBN) over both CTAs' shared memory, and each CTA's
// Tensor Memory holds the accumulator rows of its 128 tokens.  Both CTAs'
// loads signal the even CTA's `full` barrier; its MMA completions signal its
// `empty` barrier (its producer passes each release on to the odd CTA) and
// both CTAs' `tmem_full`; both CTAs' epilogues signal its `tmem_empty`.
// After the main k-blocks come the LoRA steps of the pair tile's plan, in
// the same split (Vt rows per CTA, half of the block's B rows per CTA), two
// pool blocks per ring stage.
//
// The LoRA term's V is computed here too, by V items: kVSplit per token
// tile, each V = x_tile A_list^T over one K-slice with the same pair MMA (M
// = 256 tokens, N = 32 ceil(nb/2): CTA r stacks blocks [r h, r h + h) of the
// tile's list, h = ceil(nb/2), from 16-row boxes of the pool's A arena).
// Every slice of a CTA's rows stores its fp32 sums and then counts itself (a
// per-tile, per-rank counter in the plan); the last to count adds the others
// to its own, writes the rows' Vt -- hi and lo bf16 parts of s_i V masked to
// each row's own slot -- and counts the CTA in the plan's ready entry; a
// main unit's producer waits for both CTAs' counts before it loads Vt for
// the LoRA steps.  Tiles whose plan overflowed get the per-row V on CUDA
// cores from their V items' epilogues instead (rows split between the
// slices), which the main units' epilogues wait for.
//
// Order of work: a pair takes its V items first (dealt one at a time from the
// last pair down), then its main units, handed out on demand (fetch_main_unit)
// so that the pairs' work evens out; the first two main units of a pair run
// both main loops before their LoRA steps (for_each_main_phase).  V items
// wait for nothing but their own loads and precede every main unit, so every
// wait points to work that never waits, and all pairs are resident at once
// (the grid is at most the resident cluster count): every wait ends.

constexpr int kPairM = 2 * kBM;   // tokens per pair tile
constexpr int kPairBN = 256;      // output columns per pair tile of the large-M path (the MMA's N)
constexpr int kPairAcc = 256;     // Tensor Memory columns of one accumulator
constexpr int kPairBand = 4;      // unit order: pair tiles per band (as kTaBand for one SM)
constexpr uint32_t kBlockBoxBytes = LORA_BLOCK_ROWS * kBK * 2;  // one pool block's 16 A rows of a k-block
constexpr int kVSplit = 2;        // K-slices of a token tile's V (V items per tile)
constexpr int kLoraPerStage = 2;  // pool blocks of a main unit's LoRA steps per ring stage
constexpr int kUnitRing = 4;      // main-unit ids in flight from the even CTA's producer to the other roles
constexpr int kUnitReaders = 2 + 2 * kEpiWarps;  // MMA warp, the odd CTA's producer, both CTAs' epilogue warps
static_assert(kPairM == kPlanRows, "a pair tile is a plan tile");

template <int BN>
struct PairCfg {
    // the V items stack a CTA's half of a tile's block list in the B area,
    // which takes the 128 W rows of a 256-column tile
    static_assert(BN == 256, "pair tiles of 256 output columns");
    static constexpr uint32_t kABytes = kBM * kBK * 2;              // this CTA's 128 rows of x
    static constexpr uint32_t kBBytes = (BN / 2) * kBK * 2;         // this CTA's half of the W tile
    static constexpr uint32_t kOutBytes = kBM * kBK * 2;            // an output staging buffer: 128 rows x 64 columns
    static constexpr int kOutBufs = 2;
    static constexpr int kBarBytes = (2 * 12 + 4 + 2 * kUnitRing) * 8 + 16 + 4 * kUnitRing;
    static constexpr int kFixed = 1024 + kOutBufs * static_cast<int>(kOutBytes) + kBarBytes;
    static constexpr int kStages0 = (kSmemLimit - kFixed) / static_cast<int>(kABytes + kBBytes);
    static constexpr int kStages = kStages0 > 12 ? 12 : kStages0;
    static constexpr uint32_t kTmemCols = 2 * kPairAcc;             // two accumulators (V items use up to 256 columns)
    static constexpr size_t kSmem = 1024 + static_cast<size_t>(kStages) * (kABytes + kBBytes) +
                                    kOutBufs * kOutBytes + (2 * kStages + 4 + 2 * kUnitRing) * 8 + 16 + 4 * kUnitRing;
    static_assert(kSmem <= kSmemLimit, "shared memory over budget");
    static_assert(kTmemCols <= 512, "two accumulators in Tensor Memory");
    static constexpr uint32_t kLoraBBytes = (BN / 2) * LORA_BLOCK_ROWS * 2;  // a block's B box of this CTA
    static_assert(kABytes >= kLoraPerStage * 2 * kVtBoxBytes, "a stage's Vt boxes fit the A area");
    static_assert(kBBytes >= kLoraPerStage * kLoraBBytes, "a stage's B boxes fit the B area");
    static_assert(kBBytes >= ((kPlanMaxBlocks + 1) / 2) * kBlockBoxBytes,
                  "a CTA's half of a V item's block list fits the B area");
};

__device__ __forceinline__ Unit decode_pair_unit(int32_t u, const TcParams &p) {
    Unit w;
    w.ks = 0;
    if (p.tiles_a > kPairBand) {
        const int32_t per = kPairBand * p.tiles_b;
        const int32_t band = u / per, q = u % per;
        const int32_t rows = min(kPairBand, p.tiles_a - band * kPairBand);
        w.ta = band * kPairBand + q % rows;
        w.tb = q / rows;
    } else {
        w.ta = u % p.tiles_a;
        w.tb = u / p.tiles_a;
    }
    return w;
}

// V item idx of this pair (token tile v / kVSplit, K-slice v % kVSplit), or
// -1 after its last.  A pair takes its V items before its main units; they
// are dealt one at a time from the last pair down (the main units, handed
// out on demand, even out the rest).
__device__ __forceinline__ int32_t pair_v_item(const TcParams &p, int32_t idx) {
    const int32_t G = static_cast<int32_t>(gridDim.x >> 1), P = static_cast<int32_t>(blockIdx.x >> 1);
    const int32_t v = (G - 1 - P) + idx * G;
    return v < p.v_units * kVSplit ? v : -1;
}

// The main units of a pair: unit k of its sequence is P for k = 0 (every
// pair's first, fixed), then units G, G + 1, ... in band order, handed out
// one at a time from the queue counter to whichever pair asks first, so that
// a pair slowed by its V items takes fewer; -1 ends the sequence.  The even
// CTA's producer fetches them and passes them to the other roles of both
// CTAs through a ring of kUnitRing ids in shared memory.
__device__ __forceinline__ int32_t fetch_main_unit(const TcParams &p, int32_t k) {
    const int32_t G = static_cast<int32_t>(gridDim.x >> 1), P = static_cast<int32_t>(blockIdx.x >> 1);
    if (k == 0) return P < p.num_units ? P : -1;
    grid_dependency_wait();  // the counter is zeroed by the kernel before
    const int32_t u = G + atomicAdd(p.queue, 1);
    return u < p.num_units ? u : -1;
}

struct UnitRing {
    volatile int32_t *ids;  // [kUnitRing]
    uint64_t *full;         // [kUnitRing]: an id is there (count 1)
    uint64_t *empty;        // [kUnitRing], the even CTA's: every reader has it (count kUnitReaders)
};

// The even CTA's producer: put main unit k's id into both CTAs' rings.
__device__ __forceinline__ bool ring_publish(const TcParams &p, const UnitRing &r, int32_t k, int32_t u) {
    using namespace sm100;
    const int slot = k % kUnitRing;
    if (!mbar_wait_cluster_bounded(&r.empty[slot], ((k / kUnitRing) & 1) ^ 1, kWaitLimitNs)) {
        record_error(p.status, kDevTimeout, 19);
        return false;
    }
    r.ids[slot] = u;
    st_shared_cluster_u32(mapa_shared(smem_u32(const_cast<int32_t *>(&r.ids[slot])), 1), static_cast<uint32_t>(u));
    mbar_arrive_cluster(mapa_shared(smem_u32(&r.full[slot]), 0));
    mbar_arrive_cluster(mapa_shared(smem_u32(&r.full[slot]), 1));
    return true;
}

// Every other role: main unit k's id (-1 at the end, or when the wait gives
// up).  Each reading warp then tells the even CTA's producer once
// (ring_done), after all of its threads have read it.
__device__ __forceinline__ int32_t ring_read(const TcParams &p, const UnitRing &r, int32_t k) {
    using namespace sm100;
    const int slot = k % kUnitRing;
    if (!mbar_wait_cluster_bounded(&r.full[slot], (k / kUnitRing) & 1, kWaitLimitNs)) {
        record_error(p.status, kDevTimeout, 20);
        return -1;
    }
    return r.ids[slot];
}

__device__ __forceinline__ void ring_done(const UnitRing &r, int32_t k) {
    using namespace sm100;
    mbar_arrive_cluster(mapa_shared(smem_u32(&r.empty[k % kUnitRing]), 0));
}

// The phases (0: main k-blocks, 1: LoRA steps) of main units k = 0, 1, ... in
// the order every role takes them: both phase-0s of the first two units
// before their phase-1s (the LoRA steps, which wait for the tiles' V, start
// one unit later; the two accumulators hold both units meanwhile), then each
// unit's two phases in turn.  get(k) gives unit k's id (-1: none), phase(u, k,
// ph) runs a phase and returns false when the pair gives up.
template <typename Get, typename Phase>
__device__ __forceinline__ void for_each_main_phase(Get &&get, Phase &&phase) {
    const int32_t u0 = get(0);
    if (u0 < 0 || !phase(u0, 0, 0)) return;
    const int32_t u1 = get(1);
    if (u1 < 0) {
        phase(u0, 0, 1);
        return;
    }
    if (!phase(u1, 1, 0) || !phase(u0, 0, 1) || !phase(u1, 1, 1)) return;
    for (int32_t k = 2;; ++k) {
        const int32_t u = get(k);
        if (u < 0 || !phase(u, k, 0) || !phase(u, k, 1)) return;
    }
}

// K-slice s of a V item: k-blocks [kb0, kb1) (empty when num_kb < kVSplit).
__device__ __forceinline__ void vslice_kblocks(const TcParams &p, int32_t s, int32_t *kb0, int32_t *kb1) {
    *kb0 = s * p.num_kb / kVSplit;
    *kb1 = (s + 1) * p.num_kb / kVSplit;
}

// LoRA steps of a main unit of token tile ta (none without the tile plans).
__device__ __forceinline__ int32_t pair_ext_steps(const TcParams &p, int32_t ta) {
    if (!p.lora_tiles) return 0;
    const int32_t nb = p.tile_plan[static_cast<size_t>(ta) * kPlanInts];
    return nb > 0 ? nb : 0;
}

template <int BN>
__device__ __forceinline__ void run_pair_producer(const CUtensorMap *tma_x, const CUtensorMap *tma_w,
                                                  const CUtensorMap *tma_vt, const CUtensorMap *tma_bb,
                                                  const CUtensorMap *tma_pa, const TcParams &p, uint32_t rank,
                                                  uint8_t *sA, uint8_t *sB, uint64_t *full, uint64_t *empty,
                                                  const UnitRing &ring, volatile uint32_t *abort_flag) {
    using namespace sm100;
    using C = PairCfg<BN>;
    int32_t it = 0, idx = 0;
    // Wait for stage `it` to be free in both CTAs (the even CTA's MMAs have
    // read it: that CTA's producer, which has just waited for it, tells the
    // other); false when the pair gives up.
    auto acquire_stage = [&](int32_t site) -> bool {
        const int s = it % C::kStages;
        if (!mbar_wait_bounded(&empty[s], ((it / C::kStages) & 1) ^ 1, kWaitLimitNs)) {
            record_error(p.status, kDevTimeout, site);
            *abort_flag = 1;
        }
        if (*abort_flag) return false;
        if (rank == 0 && it >= C::kStages) mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(&empty[s]), 1));
        return true;
    };
    for (;; ++idx) {  // V items: x and this CTA's half of the tile's block list, one K-slice
        const int32_t v = pair_v_item(p, idx);
        if (v < 0) break;
        const int32_t ta = v / kVSplit;
        int32_t kb0, kb1;
        vslice_kblocks(p, v % kVSplit, &kb0, &kb1);
        grid_dependency_wait();  // the plan comes from the kernel before
        const int32_t *plan = p.tile_plan + static_cast<size_t>(ta) * kPlanInts;
        const int32_t nb = plan[0];
        if (nb <= 0) continue;  // nothing for the tensor cores
        const int32_t h = (nb + 1) >> 1;
        const int32_t e0 = static_cast<int32_t>(rank) * h, e1 = min(nb, e0 + h);
        const int32_t row = ta * kPairM + static_cast<int32_t>(rank) * kBM;
        for (int32_t i = kb0; i < kb1; ++i, ++it) {
            if (!acquire_stage(15)) return;
            const int s = it % C::kStages;
            const uint32_t fb = mapa_shared(smem_u32(&full[s]), 0);  // the even CTA's barrier
            if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * C::kABytes + static_cast<uint32_t>(nb) * kBlockBoxBytes);
            tma_load_2d_pair(sA + s * C::kABytes, tma_x, i * kBK, row, fb);
            for (int32_t e = e0; e < e1; ++e)
                tma_load_2d_pair(sB + s * C::kBBytes + (e - e0) * kBlockBoxBytes, tma_pa, i * kBK,
                                 plan[kPlanBlkOff + e] * LORA_BLOCK_ROWS, fb);
        }
    }
    auto get = [&](int32_t k) -> int32_t {
        if (rank == 1) {
            const int32_t u = ring_read(p, ring, k);
            ring_done(ring, k);
            return u;
        }
        const int32_t u = fetch_main_unit(p, k);
        return ring_publish(p, ring, k, u) ? u : -1;
    };
    auto phase = [&](int32_t u, int32_t, int32_t ph) -> bool {
        const Unit w = decode_pair_unit(u, p);
        const int32_t row = w.ta * kPairM + static_cast<int32_t>(rank) * kBM;
        const int32_t n0 = w.tb * BN + static_cast<int32_t>(rank) * (BN / 2);  // this CTA's W rows
        if (ph == 0) {
            for (int32_t i = 0; i < p.num_kb; ++i, ++it) {
                if (!acquire_stage(11)) return false;
                const int s = it % C::kStages;
                const uint32_t fb = mapa_shared(smem_u32(&full[s]), 0);
                if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * (C::kABytes + C::kBBytes));
                tma_load_2d_pair(sA + s * C::kABytes, tma_x, i * kBK, row, fb);
                tma_load_2d_pair(sB + s * C::kBBytes, tma_w, i * kBK, n0, fb);
            }
            return true;
        }
        grid_dependency_wait();  // the plan comes from the kernel before
        const int32_t ext = pair_ext_steps(p, w.ta);
        if (ext == 0) return true;
        // the tile's Vt comes from its V items (both CTAs of some pair)
        if (!wait_counter_at_least(p.tile_plan + static_cast<size_t>(w.ta) * kPlanInts + kPlanReadyOff,
                                   2 + p.counter_extra, p.counter_wait_ns)) {
            record_error(p.status, kDevTimeout, 16);
            *abort_flag = 1;
            return false;
        }
        fence_proxy_async_global();  // the TMA loads below read what generic stores wrote
        // kLoraPerStage pool blocks per stage: their Vt hi and lo boxes side by
        // side in the A area, their B boxes in the B area
        for (int32_t e = 0; e < ext; e += kLoraPerStage, ++it) {
            if (!acquire_stage(11)) return false;
            const int s = it % C::kStages;
            const uint32_t fb = mapa_shared(smem_u32(&full[s]), 0);
            const int32_t eb = min(kLoraPerStage, ext - e);
            if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * eb * (2 * kVtBoxBytes + C::kLoraBBytes));
            for (int32_t j = 0; j < eb; ++j) {
                const int32_t blk = p.tile_plan[static_cast<size_t>(w.ta) * kPlanInts + kPlanBlkOff + e + j];
                uint8_t *va = sA + s * C::kABytes + j * 2 * kVtBoxBytes;
                tma_load_2d_pair(va, tma_vt, (e + j) * LORA_BLOCK_ROWS, row, fb);
                tma_load_2d_pair(va + kVtBoxBytes, tma_vt, kVtCols / 2 + (e + j) * LORA_BLOCK_ROWS, row, fb);
                tma_load_2d_pair(sB + s * C::kBBytes + j * C::kLoraBBytes, tma_bb, 0, blk * p.N + n0, fb);
            }
        }
        return true;
    };
    for_each_main_phase(get, phase);
}

// The even CTA's MMA issuer: the V items, then the phases of the main units
// in the order of for_each_main_phase (the same stage order as the
// producers').
// Unit number t (V items and main units in their sequence order) uses
// accumulator t & 1.
template <int BN>
__device__ __forceinline__ void run_pair_mma(const TcParams &p, uint8_t *sA, uint8_t *sB, uint64_t *full,
                                             uint64_t *empty, uint64_t *tmem_full, uint64_t *tmem_empty,
                                             const UnitRing &ring, uint32_t tmem_base,
                                             volatile uint32_t *abort_flag) {
    using namespace sm100;
    using C = PairCfg<BN>;
    constexpr uint32_t idesc_main = idesc_bf16_f32(kPairM, BN);
    int32_t it = 0, idx = 0;
    // wake both epilogues for accumulator b so they can unwind
    auto give_up = [&](int b) {
        *abort_flag = 1;
        mbar_arrive_cluster(mapa_shared(smem_u32(&tmem_full[b]), 0));
        mbar_arrive_cluster(mapa_shared(smem_u32(&tmem_full[b]), 1));
    };
    auto claim_accumulator = [&](int32_t t) -> bool {
        const bool ok = mbar_wait_bounded(&tmem_empty[t & 1], ((t >> 1) & 1) ^ 1, kWaitLimitNs);
        if (!ok) record_error(p.status, kDevTimeout, 12);
        tc_fence_after_sync();
        return ok;
    };
    auto wait_stage = [&]() -> bool {
        const int s = it % C::kStages;
        if (!mbar_wait_bounded(&full[s], (it / C::kStages) & 1, kWaitLimitNs)) {
            record_error(p.status, kDevTimeout, 13);
            return false;
        }
        return true;
    };
    // the stage is free once these MMAs have read it (the producer of this
    // CTA passes that on to the other CTA's)
    auto release_stage = [&]() { mma_commit_pair(mapa_shared(smem_u32(&empty[it % C::kStages]), 0)); };
    auto finish_unit = [&](int b) {
        mma_commit_pair(mapa_shared(smem_u32(&tmem_full[b]), 0));
        mma_commit_pair(mapa_shared(smem_u32(&tmem_full[b]), 1));
    };
    for (;; ++idx) {  // V items: N = 32 ceil(nb / 2), one K-slice, no LoRA steps
        const int32_t v = pair_v_item(p, idx);
        if (v < 0) break;
        const int32_t t = idx, b = t & 1;
        const int32_t ta = v / kVSplit;
        int32_t kb0, kb1;
        vslice_kblocks(p, v % kVSplit, &kb0, &kb1);
        grid_dependency_wait();
        const int32_t nb = p.tile_plan[static_cast<size_t>(ta) * kPlanInts];
        const int32_t total = nb > 0 ? kb1 - kb0 : 0;
        const uint32_t idesc = idesc_bf16_f32(kPairM, nb > 0 ? 32 * ((nb + 1) >> 1) : 32);
        if (!claim_accumulator(t)) return give_up(b);
        const uint32_t d = tmem_base + b * kPairAcc;
        for (int32_t i = 0; i < total; ++i, ++it) {
            if (!wait_stage()) return give_up(b);
            const uint32_t a_addr = smem_u32(sA + (it % C::kStages) * C::kABytes);
            const uint32_t b_addr = smem_u32(sB + (it % C::kStages) * C::kBBytes);
#pragma unroll
            for (int k = 0; k < kBK / kUmmaK; ++k)
                mma_bf16_f32_pair(d, desc_kmajor_sw128(a_addr + k * kUmmaK * 2), desc_kmajor_sw128(b_addr + k * kUmmaK * 2),
                                  idesc, (i > 0 || k > 0) ? 1u : 0u);
            release_stage();
        }
        if (*abort_flag) return give_up(b);
        finish_unit(b);
    }
    const int32_t nv = idx;
    auto get = [&](int32_t k) -> int32_t {
        const int32_t u = ring_read(p, ring, k);
        ring_done(ring, k);
        return u;
    };
    auto phase = [&](int32_t u, int32_t k, int32_t ph) -> bool {
        const int32_t t = nv + k, b = t & 1;
        const uint32_t d = tmem_base + b * kPairAcc;
        if (ph == 0) {
            if (!claim_accumulator(t)) {
                give_up(b);
                return false;
            }
            for (int32_t i = 0; i < p.num_kb; ++i, ++it) {
                if (!wait_stage()) {
                    give_up(b);
                    return false;
                }
                const uint32_t a_addr = smem_u32(sA + (it % C::kStages) * C::kABytes);
                const uint32_t b_addr = smem_u32(sB + (it % C::kStages) * C::kBBytes);
#pragma unroll
                for (int kk = 0; kk < kBK / kUmmaK; ++kk)
                    mma_bf16_f32_pair(d, desc_kmajor_sw128(a_addr + kk * kUmmaK * 2),
                                      desc_kmajor_sw128(b_addr + kk * kUmmaK * 2), idesc_main, (i > 0 || kk > 0) ? 1u : 0u);
                release_stage();
            }
            return true;
        }
        const Unit w = decode_pair_unit(u, p);
        grid_dependency_wait();
        const int32_t ext = pair_ext_steps(p, w.ta);
        // LoRA steps, kLoraPerStage pool blocks per stage: Vt_hi and Vt_lo
        // times the block's B, K = 16 each
        for (int32_t e = 0; e < ext; e += kLoraPerStage, ++it) {
            if (!wait_stage()) {
                give_up(b);
                return false;
            }
            const uint32_t a_addr = smem_u32(sA + (it % C::kStages) * C::kABytes);
            const uint32_t b_addr = smem_u32(sB + (it % C::kStages) * C::kBBytes);
            const int32_t eb = min(kLoraPerStage, ext - e);
            for (int32_t j = 0; j < eb; ++j) {
                const uint32_t va = a_addr + j * 2 * kVtBoxBytes, vb = b_addr + j * C::kLoraBBytes;
                mma_bf16_f32_pair(d, desc_kmajor_sw32(va), desc_kmajor_sw32(vb), idesc_main, 1u);
                mma_bf16_f32_pair(d, desc_kmajor_sw32(va + kVtBoxBytes), desc_kmajor_sw32(vb), idesc_main, 1u);
            }
            release_stage();
        }
        if (*abort_flag) {
            give_up(b);
            return false;
        }
        finish_unit(b);
        return true;
    };
    for_each_main_phase(get, phase);
}

// Epilogue of V item v in CTA `rank` (row: this thread's row of the CTA's
// 128, warp_e: its index among the eight epilogue warps, grp: which half of
// the 32-column chunks it reads).  Accumulator column 16e + j holds rank-row
// j of block e of the tile's list (CTA 0's B rows first).  Every slice of a
// CTA's rows stores its fp32 sums (row-major, [256 rows][256 columns] per
// slice) and then counts itself; the last to count adds the others' sums to
// its own, still in Tensor Memory, writes the rows' Vt and publishes.  No
// slice waits for another pair, so a V item never holds its accumulator
// for longer than its own work.  For a fallback tile the slices compute
// their share of the rows' per-row V instead.
__device__ __forceinline__ void run_pair_v_epilogue(const TcParams &p, int32_t v, uint32_t rank, uint32_t col0,
                                                    int row, int warp_e, int grp, int lane,
                                                    volatile uint32_t *v_last) {
    using namespace sm100;
    const int32_t ta = v / kVSplit, sl = v % kVSplit;
    const int32_t *plan = p.tile_plan + static_cast<size_t>(ta) * kPlanInts;
    int32_t *counts = p.plan_rw + static_cast<size_t>(ta) * kPlanInts;
    const int32_t nb = plan[0];
    const int32_t m0 = ta * kPairM + static_cast<int32_t>(rank) * kBM;
    const int32_t m = m0 + row;
    const int32_t prow = static_cast<int32_t>(rank) * kBM + row;  // row of the 256-row slice
    const size_t slice_elems = static_cast<size_t>(kPlanRows) * kPlanRows;
    float *tile_part = p.v_part + static_cast<size_t>(ta) * kVSplit * slice_elems;
    int32_t kb0, kb1;
    vslice_kblocks(p, sl, &kb0, &kb1);
    const bool own_slice = kb1 > kb0;  // this item accumulated something
    const int32_t h = (nb + 1) >> 1;
    // the row's slot and scale now, while nothing waits on them
    int32_t r = 0, slot = -1;
    float sc = 0.0f;
    if (nb > 0 && m < p.M)
        slot = resolve_slot(p.row_slot[m], m, p.ranks, p.scales, p.max_slots, p.bps, &r, &sc, p.status, false);
    if (nb < 0) {
        // rows in no useful order: V of each row on CUDA cores, one warp per
        // row, this slice's share of the CTA's rows
        const int32_t lo = sl * kBM / kVSplit, hi = (sl + 1) * kBM / kVSplit;
#pragma unroll 1
        for (int32_t i = lo + warp_e; i < hi; i += kEpiWarps) {
            const int32_t mi = m0 + i;
            if (mi >= p.M) break;
            int32_t ri = 0;
            float si = 0.0f;
            const int32_t slot_i =
                resolve_slot(p.row_slot[mi], mi, p.ranks, nullptr, p.max_slots, p.bps, &ri, &si, p.status, false);
            if (slot_i < 0) continue;
            const int32_t *blocks = p.table + static_cast<size_t>(slot_i) * p.bps;
            bool blocks_ok = true;
            for (int32_t jb = 0; jb * LORA_BLOCK_ROWS < ri; ++jb) blocks_ok &= blocks[jb] >= 0 && blocks[jb] < p.num_blocks;
            if (!blocks_ok) continue;  // reported by the plan kernel; the epilogue drops the row's correction
            row_v_by_warp(p.x + static_cast<size_t>(mi) * p.ldx, p.K, p.a_arena, blocks, ri,
                          p.v_rows + static_cast<size_t>(mi) * p.ldv, lane);
        }
    }
    if (nb > 0 && own_slice) {
        float *dst_row = tile_part + sl * slice_elems + static_cast<size_t>(prow) * kPlanRows;
#pragma unroll 1
        for (int32_t c = grp; c < h; c += 2) {
            float acc[32];
            load_tmem_chunk(col0 + c * 32, acc);
            float4 *dst = reinterpret_cast<float4 *>(dst_row + c * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                __stcg(dst + i, make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]));
        }
    }
    // count this slice (every writer fences, one thread counts); the last
    // one goes on after an acquiring fence
    __threadfence();
    epi_sync();
    if (threadIdx.x == 64) {
        const bool last = atomicAdd(counts + kPlanPartOff + rank, 1) == kVSplit - 1;
        __threadfence();
        *v_last = last ? 1u : 0u;
    }
    epi_sync();
    if (!*v_last) return;
    if (nb > 0) {
        __nv_bfloat16 *vt_row = p.vt_out + static_cast<size_t>(m) * kVtCols;
#pragma unroll 1
        for (int32_t c = grp; c < h; c += 2) {  // 32 columns: blocks 2c and 2c + 1
            float acc[32];
            if (own_slice) {
                load_tmem_chunk(col0 + c * 32, acc);
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) acc[i] = 0.0f;
            }
            if (m < p.M) {
#pragma unroll
                for (int q = 0; q < kVSplit; ++q) {
                    int32_t q0, q1;
                    vslice_kblocks(p, q, &q0, &q1);
                    if (q == sl || q1 <= q0) continue;
                    const float4 *src = reinterpret_cast<const float4 *>(
                        tile_part + q * slice_elems + static_cast<size_t>(prow) * kPlanRows + c * 32);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float4 f = __ldcg(src + i);
                        acc[4 * i] += f.x;
                        acc[4 * i + 1] += f.y;
                        acc[4 * i + 2] += f.z;
                        acc[4 * i + 3] += f.w;
                    }
                }
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int32_t e = 2 * c + u;
                    if (e < nb) store_vt_entry(vt_row, e, acc + 16 * u, slot >= 0 && plan[kPlanSlotOff + e] == slot, sc);
                }
            }
        }
    }
    // publish: this CTA's rows are written (the main units read Vt through
    // TMA loads, V through plain loads)
    fence_proxy_async_global();
    __threadfence();
    epi_sync();
    if (threadIdx.x == 64) atomicAdd(counts + kPlanReadyOff, 1);
}

// Epilogue of both CTAs: for each unit, the 256 accumulator columns in four
// chunks of 64: every warp reads 32 of them for its 32 rows from TMEM, adds
// the CUDA-core expand where the tile needs it, and writes bf16 into a
// shared-memory staging buffer laid out as a 128-byte-swizzled [128 x 64]
// box; one thread then stores the box with TMA (rows past M and columns past
// N are clipped).  Two staging buffers alternate.
template <int BN>
__device__ __forceinline__ void run_pair_epilogue(const TcParams &p, const CUtensorMap *tma_out, uint32_t rank,
                                                  uint8_t *sOut, uint64_t *tmem_full, uint64_t *tmem_empty,
                                                  const UnitRing &ring, uint32_t tmem_base,
                                                  volatile uint32_t *abort_flag, volatile uint32_t *v_last) {
    using namespace sm100;
    using C = PairCfg<BN>;
    const int warp = threadIdx.x >> 5;
    const int q = warp & 3;
    const int grp = (warp - 2) >> 2;  // which 32 of a chunk's 64 columns
    const int lane = threadIdx.x & 31;
    const int et = threadIdx.x - 64;
    const int row = q * 32 + lane;    // row of this CTA's 128
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    grid_dependency_wait();  // the plan comes from the kernel before
    int32_t t = 0, chunk_no = 0, nv = 0;
    while (pair_v_item(p, nv) >= 0) ++nv;
    for (int32_t idx = 0;; ++idx) {
        // V items first, then the main units from the ring
        int32_t u;
        if (idx < nv) {
            u = p.num_units + pair_v_item(p, idx);
        } else {
            u = ring_read(p, ring, idx - nv);
            __syncwarp();
            if (lane == 0) ring_done(ring, idx - nv);
        }
        if (u < 0) break;
        const int b = t & 1;
        bool ok = mbar_wait_bounded(&tmem_full[b], (t >> 1) & 1, kWaitLimitNs);
        if (!ok) {
            record_error(p.status, kDevTimeout, 14);
            *abort_flag = 1;
        }
        if (!epi_all(ok && !*abort_flag)) break;  // uniform over the epilogue warps
        tc_fence_after_sync();
        const uint32_t col0 = lane_addr + b * kPairAcc;
        if (u >= p.num_units) {
            run_pair_v_epilogue(p, u - p.num_units, rank, col0, row, warp - 2, grp, lane, v_last);
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tmem_empty[b]), 0));
            ++t;
            continue;
        }
        const Unit w = decode_pair_unit(u, p);
        const int32_t m0 = w.ta * kPairM + static_cast<int32_t>(rank) * kBM;
        const int32_t m = m0 + row;
        // the CUDA-core expand for tiles whose plan overflowed (with ycorr the
        // LoRA term is already in it)
        const bool per_row = p.lora_tiles && p.tile_plan[static_cast<size_t>(w.ta) * kPlanInts] < 0;
        if (per_row && p.v_units > 0) {
            // the rows' V comes from the tile's V unit
            const bool ready = wait_counter_at_least(p.tile_plan + static_cast<size_t>(w.ta) * kPlanInts + kPlanReadyOff,
                                                     2 + p.counter_extra, p.counter_wait_ns);
            if (!ready) {
                record_error(p.status, kDevTimeout, 17);
                *abort_flag = 1;
            }
            if (!epi_all(ready && !*abort_flag)) break;
        }
        int32_t r = 0, slot = -1;
        float s = 0.0f;
        if (per_row && m < p.M)
            slot = resolve_slot(p.row_slot[m], m, p.ranks, p.scales, p.max_slots, p.bps, &r, &s, p.status, false);
#pragma unroll 1
        for (int j = 0; j < BN / kBK; ++j, ++chunk_no) {
            float acc[32];
            load_tmem_chunk(col0 + j * kBK + grp * 32, acc);
            const int32_t n0 = w.tb * BN + j * kBK;
            if (per_row) rows_finish_chunk(p, slot, r, s, m, n0 + grp * 32, acc);
            uint8_t *buf = sOut + (chunk_no & 1) * C::kOutBytes;
            // the store that last read this buffer (two chunks back) must be done
            if (et == 0) bulk_wait_group_read<C::kOutBufs - 1>();
            epi_sync();
            uint8_t *dst_row = buf + row * (kBK * 2);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint4 v;
                v.x = pack_bf16x2(acc[i * 8 + 0], acc[i * 8 + 1]);
                v.y = pack_bf16x2(acc[i * 8 + 2], acc[i * 8 + 3]);
                v.z = pack_bf16x2(acc[i * 8 + 4], acc[i * 8 + 5]);
                v.w = pack_bf16x2(acc[i * 8 + 6], acc[i * 8 + 7]);
                // 16-byte piece c of the row lands at c ^ (row % 8): the 128-byte swizzle
                const int c = grp * 4 + i;
                *reinterpret_cast<uint4 *>(dst_row + ((c ^ (row & 7)) << 4)) = v;
            }
            fence_proxy_async_shared();  // the TMA store reads the buffer through the async proxy
            epi_sync();
            if (et == 0) {
                tma_store_2d(tma_out, n0, m0, buf);
                bulk_commit_group();
            }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tmem_empty[b]), 0));  // the even CTA's barrier
        ++t;
    }
    if (et == 0) bulk_wait_group_all();  // the staging buffers must outlive the stores
}

template <int BN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
tc_gemm_pair_kernel(const __grid_constant__ CUtensorMap tma_x, const __grid_constant__ CUtensorMap tma_w,
                    const __grid_constant__ CUtensorMap tma_vt, const __grid_constant__ CUtensorMap tma_bb,
                    const __grid_constant__ CUtensorMap tma_pa, const __grid_constant__ CUtensorMap tma_out,
                    const TcParams p) {
    using namespace sm100;
    using C = PairCfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + C::kStages * C::kABytes;
    uint8_t *sOut = sB + C::kStages * C::kBBytes;  // output staging, 1024-byte aligned
    uint64_t *full = reinterpret_cast<uint64_t *>(sOut + C::kOutBufs * C::kOutBytes);
    uint64_t *empty = full + C::kStages;
    uint64_t *tmem_full = empty + C::kStages;  // [2]
    uint64_t *tmem_empty = tmem_full + 2;      // [2]
    UnitRing ring;
    ring.full = tmem_empty + 2;                // [kUnitRing]
    ring.empty = ring.full + kUnitRing;        // [kUnitRing]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(ring.empty + kUnitRing);
    volatile uint32_t *abort_flag = tmem_slot + 1;
    volatile uint32_t *v_last = tmem_slot + 2;  // a V item's epilogue: this slice was the last
    ring.ids = reinterpret_cast<volatile int32_t *>(tmem_slot + 4);  // [kUnitRing]
    const uint32_t rank = cluster_ctarank();
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tmem_full[b], 1);
            mbar_init(&tmem_empty[b], 2 * kEpiWarps);  // the epilogue warps of both CTAs
        }
        for (int i = 0; i < kUnitRing; ++i) {
            mbar_init(&ring.full[i], 1);
            mbar_init(&ring.empty[i], kUnitReaders);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tma_x);
        prefetch_tensormap(&tma_w);
        prefetch_tensormap(&tma_out);
        if (p.lora_tiles) {
            prefetch_tensormap(&tma_vt);
            prefetch_tensormap(&tma_bb);
            prefetch_tensormap(&tma_pa);
        }
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, C::kTmemCols);
        tmem_relinquish_pair();
    }
    // both CTAs' barriers initialised and Tensor Memory allocated before any
    // signal crosses the pair
    tc_fence_before_sync();
    cluster_sync();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0)
            run_pair_producer<BN>(&tma_x, &tma_w, &tma_vt, &tma_bb, &tma_pa, p, rank, sA, sB, full, empty, ring,
                                  abort_flag);
    } else if (warp == 1) {
        if (lane == 0 && rank == 0)
            run_pair_mma<BN>(p, sA, sB, full, empty, tmem_full, tmem_empty, ring, tmem_base, abort_flag);
    } else {
        run_pair_epilogue<BN>(p, &tma_out, rank, sOut, tmem_full, tmem_empty, ring, tmem_base, abort_flag, v_last);
    }

    // no CTA leaves while the other may still signal its barriers or read its
    // shared memory through the pair MMA
    tc_fence_before_sync();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem_base, C::kTmemCols);
    }
}

// ---------------------------------------------------------------- host side

// v1: a second projection of the same x in the same launch (swapped
// orientation only; tp plans both).  counters: the split-K tile counters of
// this launch (NULL: the plan's).
template <bool SWAP, int BN, bool PAIR = false, bool QUANT = false>
cudaError_t launch_variant(const ForwardPlan &plan, const ProjView &v, const TcPlan &tp, cudaStream_t stream,
                           const ProjView *v1 = nullptr, int32_t *counters = nullptr,
                           int64_t n_counters = 0) {
    using C = Cfg<SWAP, BN, QUANT>;
    auto kernel = tc_gemm_lora_kernel<SWAP, BN, PAIR, QUANT>;
    static std::mutex mu;
    static uint64_t done_ctx[128] = {};  // per device: the context the opt-in was set in
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(mu);
        uint64_t ctx = done_ctx[dev];
        if (first_use_in_context(&ctx)) {  // the shared-memory opt-in is a per-device function attribute
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(C::kSmem));
            if (e != cudaSuccess) return e;
            done_ctx[dev] = current_context_id();
        }
    }
    CUtensorMap tx, tw;
    if (!make_tmap_bf16(&tx, plan.x, plan.M, plan.K, plan.ldx, SWAP ? BN : kBM)) return cudaErrorInvalidValue;
    if (QUANT != (v.w_scale != nullptr) || (QUANT && (!SWAP || PAIR))) return cudaErrorInvalidValue;
    if (QUANT) {  // int8 [N][K] bytes, or packed int4 [N][K/2]: 64 values of a row per box
        const bool i4 = v.w_bits == 4;
        if (!make_tmap_u8(&tw, v.W, v.N, i4 ? plan.K / 2 : plan.K, kBM, i4 ? kBK / 2 : kBK))
            return cudaErrorInvalidValue;
    } else if (!make_tmap_bf16(&tw, v.W, v.N, plan.K, plan.K, SWAP ? kBM : BN)) {
        return cudaErrorInvalidValue;
    }
    // LoRA steps (non-swapped orientation): Vt beside x, the pool's B arena
    // ([num_blocks * N][16]) beside W, both in [rows x 16] boxes with the
    // 32-byte swizzle; unused maps are copies of the main ones
    CUtensorMap tva = tx, tvb = tw;
    const bool tiles = !SWAP && v.lora_tiles;
    if (PAIR != (v1 != nullptr)) return cudaErrorInvalidValue;
    if (v1) {  // the second projection's W in the slot of the LoRA steps' A-side map
        if (!SWAP || !make_tmap_bf16(&tva, v1->W, v1->N, plan.K, plan.K, kBM)) return cudaErrorInvalidValue;
    }
    if (tiles) {
        const uint64_t tiles_m = static_cast<uint64_t>((plan.M + kPlanRows - 1) / kPlanRows) * kPlanRows;
        if (!v.vt || !v.tile_plan ||
            !make_tmap_bf16(&tva, v.vt, tiles_m, kVtCols, kVtCols, kBM, LORA_BLOCK_ROWS, 32) ||
            !make_tmap_bf16(&tvb, v.b_arena, static_cast<uint64_t>(v.num_blocks) * v.N, LORA_BLOCK_ROWS,
                            LORA_BLOCK_ROWS, BN, LORA_BLOCK_ROWS, 32))
            return cudaErrorInvalidValue;
    }
    TcParams p;
    p.M = plan.M;
    p.N = v.N;
    p.K = plan.K;
    p.num_kb = tp.num_kb;
    p.kb_per_split = tp.kb_per_split;
    p.splits = tp.splits;
    p.full_units = tp.full_units;
    p.split_tiles = tp.split_tiles;
    p.tiles_a = tp.tiles_a;
    p.tiles_b = tp.tiles_b;
    p.num_units = tp.units;
    p.out = static_cast<__nv_bfloat16 *>(v.out);
    p.ldo = v.ldo;
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
    p.v_parts = plan.v_parts;
    p.v_part_stride = static_cast<size_t>(plan.M) * v.max_rank;
    p.part = plan.part;
    p.ycorr = v.ycorr;
    p.lora_tiles = tiles ? 1 : 0;
    p.tile_plan = v.tile_plan;
    p.counters = counters ? counters : plan.counters;
    if (!counters) n_counters = plan.n_counters;
    p.status = plan.status;
    p.w_scale = v.w_scale;
    p.w_bits = v.w_scale ? (v.w_bits == 4 ? 4 : 8) : 0;
    p.counter_extra = plan.test_wait_limit_ns ? 1 : 0;
    p.counter_wait_ns = plan.test_wait_limit_ns ? plan.test_wait_limit_ns : kWaitLimitNs;
    p.tiles_a0 = tp.tiles_a;
    p.N1 = 0;
    p.ldo1 = 0;
    p.out1 = nullptr;
    p.ycorr1 = nullptr;
    if (v1) {
        p.tiles_a0 = (v.N + kBM - 1) / kBM;
        if (p.tiles_a0 + (v1->N + kBM - 1) / kBM != tp.tiles_a) return cudaErrorInvalidValue;
        p.N1 = v1->N;
        p.ldo1 = v1->ldo;
        p.out1 = static_cast<__nv_bfloat16 *>(v1->out);
        p.ycorr1 = v1->ycorr;
    }
    // the splits of a tile wait for one another, so they must all be resident:
    // the split units form the grid's last round (whole rounds of whole
    // tiles before them), at most one per CTA
    if (tp.splits > 1 && (!plan.part || !p.counters || tp.full_units % tp.grid != 0 ||
                          tp.units - tp.full_units > tp.grid || n_counters < tp.split_tiles))
        return cudaErrorInvalidValue;
    // programmatic dependent of the shrink kernel before it on the stream:
    // the CTAs may start (and stream W and x) while the shrink finishes; the
    // epilogue waits for the shrink's grid before it reads V or the counters
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(tp.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (SWAP) return cudaLaunchKernelEx(&cfg, kernel, tw, tx, tva, tvb, p);
    return cudaLaunchKernelEx(&cfg, kernel, tx, tw, tva, tvb, p);
}


// The two-SM GEMM of the large-M orientation (see tc_gemm_pair_kernel): as
// many pairs as can be resident at once (a cluster needs two SMs of one
// GPC).
template <int BN>
cudaError_t launch_pair_gemm(const ForwardPlan &plan, const ProjView &v, cudaStream_t stream) {
    using C = PairCfg<BN>;
    auto kernel = tc_gemm_pair_kernel<BN>;
    static std::mutex mu;
    static uint64_t done_ctx[128] = {};
    static int max_pairs[128] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    int pairs_cap = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        uint64_t ctx = done_ctx[dev];
        if (first_use_in_context(&ctx)) {
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::kSmem));
            if (e != cudaSuccess) return e;
            cudaLaunchConfig_t oc = {};
            oc.gridDim = dim3(2 * 128);
            oc.blockDim = dim3(kThreads);
            oc.dynamicSmemBytes = C::kSmem;
            int n = 0;
            e = cudaOccupancyMaxActiveClusters(&n, kernel, &oc);
            if (e != cudaSuccess || n < 1) return e != cudaSuccess ? e : cudaErrorInvalidConfiguration;
            max_pairs[dev] = n;
            done_ctx[dev] = current_context_id();
        }
        pairs_cap = max_pairs[dev];
    }
    if (!v.lora_tiles || !v.vt || !v.tile_plan || !v.V || !v.vacc) return cudaErrorInvalidValue;
    CUtensorMap tx, tw, tvt, tbb, tpa, tout;
    const uint64_t tiles_m = static_cast<uint64_t>((plan.M + kPlanRows - 1) / kPlanRows) * kPlanRows;
    if (!make_tmap_bf16(&tx, plan.x, plan.M, plan.K, plan.ldx, kBM) ||
        !make_tmap_bf16(&tout, v.out, plan.M, v.N, v.ldo, kBM) ||
        !make_tmap_bf16(&tw, v.W, v.N, plan.K, plan.K, BN / 2) ||
        !make_tmap_bf16(&tvt, v.vt, tiles_m, kVtCols, kVtCols, kBM, LORA_BLOCK_ROWS, 32) ||
        !make_tmap_bf16(&tbb, v.b_arena, static_cast<uint64_t>(v.num_blocks) * v.N, LORA_BLOCK_ROWS,
                        LORA_BLOCK_ROWS, BN / 2, LORA_BLOCK_ROWS, 32) ||
        !make_tmap_bf16(&tpa, v.a_arena, static_cast<uint64_t>(v.num_blocks) * LORA_BLOCK_ROWS, plan.K, plan.K,
                        LORA_BLOCK_ROWS))
        return cudaErrorInvalidValue;
    TcParams p = {};
    p.M = plan.M;
    p.N = v.N;
    p.K = plan.K;
    p.num_kb = (plan.K + kBK - 1) / kBK;
    p.kb_per_split = p.num_kb;
    p.splits = 1;
    p.full_units = 0;
    p.split_tiles = 0;
    p.tiles_a = (plan.M + kPairM - 1) / kPairM;
    p.tiles_b = (v.N + BN - 1) / BN;
    p.num_units = p.tiles_a * p.tiles_b;
    p.out = static_cast<__nv_bfloat16 *>(v.out);
    p.ldo = v.ldo;
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
    p.v_parts = 1;
    p.v_part_stride = static_cast<size_t>(plan.M) * v.max_rank;
    p.status = plan.status;
    p.tiles_a0 = p.tiles_a;
    p.lora_tiles = 1;
    p.tile_plan = v.tile_plan;
    p.v_units = p.tiles_a;
    p.vt_out = static_cast<__nv_bfloat16 *>(v.vt);
    p.v_rows = v.V;
    p.v_part = v.vacc;
    p.queue = v.tile_plan + kPlanQueueOff;
    p.plan_rw = v.tile_plan;
    // armed for a test: the Vt ready waits expect one count more than comes
    p.counter_extra = plan.test_wait_limit_ns ? 1 : 0;
    p.counter_wait_ns = plan.test_wait_limit_ns ? plan.test_wait_limit_ns : kWaitLimitNs;
    p.x = static_cast<const __nv_bfloat16 *>(plan.x);
    p.ldx = plan.ldx;
    p.a_arena = static_cast<const __nv_bfloat16 *>(v.a_arena);
    const int total_units = p.num_units + p.v_units * kVSplit;
    const int pairs = total_units < pairs_cap ? total_units : pairs_cap;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * pairs);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, tx, tw, tvt, tbb, tpa, tout, p);
}

}  // namespace

int device_sm_count() {
    static int cache[128] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 148;
    if (!cache[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cache[dev] = n;
    }
    return cache[dev];
}

// Split-K of the swapped orientation, each split at least four k-blocks
// long, at most 16: with fewer tiles than SMs, enough splits to give every
// SM a unit; with more, whole rounds of whole tiles and then, when the last
// round would leave at least half of the SMs idle, its tiles split along K
// over all of them (every CTA takes at most one split unit, so the splits of
// a tile are resident together).
static void swapped_splits(TcPlan *t, int sms) {
    const int tiles = t->tiles_a * t->tiles_b;
    const int left = tiles % sms;
    int s = 1;
    t->full_units = 0;
    if (tiles < sms) {
        s = sms / tiles;
    } else if (left != 0 && 2 * left <= sms) {
        s = sms / left;
        t->full_units = tiles - left;
    }
    const int max_s = t->num_kb / 4 > 0 ? t->num_kb / 4 : 1;
    if (s > max_s) s = max_s;
    if (s > 16) s = 16;
    if (s < 1) s = 1;
    t->kb_per_split = (t->num_kb + s - 1) / s;
    t->splits = (t->num_kb + t->kb_per_split - 1) / t->kb_per_split;
    if (t->splits == 1) t->full_units = 0;
}

static void finish_plan(TcPlan *t, int sms) {
    const int tiles = t->tiles_a * t->tiles_b;
    t->split_tiles = t->splits > 1 ? tiles - t->full_units : 0;
    t->units = t->full_units + (tiles - t->full_units) * t->splits;
    t->grid = t->units < sms ? t->units : sms;
    t->part_bytes = sizeof(float) * static_cast<size_t>(t->splits) * t->split_tiles * t->bn * kBM;
    t->counter_bytes = sizeof(int32_t) * static_cast<size_t>(t->split_tiles);
}

// Orientation, tile width and split-K factor for an M x N x K problem.
TcPlan plan_tc(int32_t M, int32_t N, int32_t K) {
    TcPlan t{};
    const int sms = device_sm_count();
    t.num_kb = (K + kBK - 1) / kBK;
    t.swap = M <= 512;
    if (t.swap) {
        // tokens per tile: 256 above 128 tokens.  An MMA of 128 W rows x 256
        // tokens issues half the instructions per flop of 128 x 128 (the MMA
        // warp, not the loads, sets the pace of 128 x 128 tiles), and one
        // token tile reads each W row once: the 70B q+v call (256 tokens,
        // 8192 -> 9216, split-K 2) went 78.3 -> 74.1 us per step once the
        // split-K finish kept several loads in flight per thread
        t.bn = M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : 256;
        t.tiles_a = (N + kBM - 1) / kBM;
        t.tiles_b = (M + t.bn - 1) / t.bn;
        swapped_splits(&t, sms);
    } else {
        t.tiles_a = (M + kBM - 1) / kBM;
        const long u256 = static_cast<long>(t.tiles_a) * ((N + 255) / 256);
        const long u128 = static_cast<long>(t.tiles_a) * ((N + 127) / 128);
        const long c256 = ((u256 + sms - 1) / sms) * (256 + 32);
        const long c128 = ((u128 + sms - 1) / sms) * (128 + 32);
        t.bn = c256 <= c128 ? 256 : 128;
        t.tiles_b = (N + t.bn - 1) / t.bn;
        t.splits = 1;
        t.kb_per_split = t.num_kb;
    }
    finish_plan(&t, sms);
    return t;
}

// Two projections of one x in one swapped launch: their W tiles side by
// side (M <= 512 only; swap is false otherwise).
TcPlan plan_tc_pair(int32_t M, int32_t N0, int32_t N1, int32_t K) {
    TcPlan t = plan_tc(M, N0, K);
    if (!t.swap) return t;
    const int sms = device_sm_count();
    t.tiles_a = (N0 + kBM - 1) / kBM + (N1 + kBM - 1) / kBM;
    swapped_splits(&t, sms);
    finish_plan(&t, sms);
    return t;
}

cudaError_t launch_gemm_lora_tc_pair(const ForwardPlan &plan, const ProjView &v0, const ProjView *v1,
                                     int32_t *counters, int64_t n_counters, cudaStream_t stream) {
    const TcPlan tp = v1 ? plan_tc_pair(plan.M, v0.N, v1->N, plan.K) : plan_tc(plan.M, v0.N, plan.K);
    if (!tp.swap) return cudaErrorInvalidValue;
    if (v0.w_scale || (v1 && v1->w_scale)) {  // int8 W: one projection, token tiles of 32 or 64
        if (v1) return cudaErrorInvalidValue;
        if (tp.bn == 32)
            return launch_variant<true, 32, false, true>(plan, v0, tp, stream, nullptr, counters, n_counters);
        if (tp.bn == 64)
            return launch_variant<true, 64, false, true>(plan, v0, tp, stream, nullptr, counters, n_counters);
        return cudaErrorInvalidValue;
    }
    // pairs: tiles of at least 128 tokens (the narrower variants keep their
    // register count low enough to share an SM with the per-row kernel)
    if (v1) {
        if (tp.bn == 128) return launch_variant<true, 128, true>(plan, v0, tp, stream, v1, counters, n_counters);
        if (tp.bn == 256) return launch_variant<true, 256, true>(plan, v0, tp, stream, v1, counters, n_counters);
        return cudaErrorInvalidValue;
    }
    switch (tp.bn) {
        case 32: return launch_variant<true, 32>(plan, v0, tp, stream, nullptr, counters, n_counters);
        case 64: return launch_variant<true, 64>(plan, v0, tp, stream, nullptr, counters, n_counters);
        case 128: return launch_variant<true, 128>(plan, v0, tp, stream, nullptr, counters, n_counters);
        default: return launch_variant<true, 256>(plan, v0, tp, stream, nullptr, counters, n_counters);
    }
}

bool pair_gemm_takes(const ProjView &v) { return v.lora_tiles && !v.w_scale && v.N >= kPairBN; }

size_t pair_vpart_bytes(int32_t M) {
    const size_t T = (static_cast<size_t>(M) + kPairM - 1) / kPairM;
    return sizeof(float) * T * kVSplit * kPlanRows * kPlanRows;
}

cudaError_t launch_gemm_lora_tc(const ForwardPlan &plan, const ProjView &v, cudaStream_t stream) {
    if (v.w_scale) return launch_gemm_lora_tc_pair(plan, v, nullptr, nullptr, 0, stream);
    const TcPlan tp = plan_tc(plan.M, v.N, plan.K);
    if (tp.swap) {
        switch (tp.bn) {
            case 32: return launch_variant<true, 32>(plan, v, tp, stream);
            case 64: return launch_variant<true, 64>(plan, v, tp, stream);
            case 128: return launch_variant<true, 128>(plan, v, tp, stream);
            default: return launch_variant<true, 256>(plan, v, tp, stream);
        }
    }
    // large M with at least one full pair tile of columns: the two-SM kernel
    if (pair_gemm_takes(v)) return launch_pair_gemm<kPairBN>(plan, v, stream);
    if (tp.bn == 128) return launch_variant<false, 128>(plan, v, tp, stream);
    return launch_variant<false, 256>(plan, v, tp, stream);
}

}  // namespace lora
