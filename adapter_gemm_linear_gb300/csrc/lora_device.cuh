// Small device helpers shared by the kernel files.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "lora_internal.h"

namespace lora {

// First error wins: the word goes from 0 to (code << 32 | detail) once.
__device__ __forceinline__ void record_error(unsigned long long *status, uint32_t code,
                                             uint32_t detail) {
    const unsigned long long w = (static_cast<unsigned long long>(code) << 32) | detail;
    atomicCAS(status, 0ull, w);
}

// Map a row's slot id to (slot, rank, scale); -1 when the row gets no
// correction.  Ids outside [-1, max_slots), empty slots and ranks larger than
// the table row are recorded (when `report`) and treated as no correction.
__device__ __forceinline__ int32_t resolve_slot(int32_t id, int32_t m, const int32_t *ranks,
                                                const float *scales, int32_t max_slots,
                                                int32_t bps, int32_t *r, float *s,
                                                unsigned long long *status, bool report) {
    *r = 0;
    *s = 0.0f;
    if (id == -1) return -1;
    if (id < -1 || id >= max_slots) {
        if (report) record_error(status, kDevBadAdapter, static_cast<uint32_t>(m));
        return -1;
    }
    const int32_t rr = ranks[id];
    if (rr <= 0) {
        if (report) record_error(status, kDevEmptySlot, static_cast<uint32_t>(m));
        return -1;
    }
    if (rr > bps * LORA_BLOCK_ROWS) {
        if (report) record_error(status, kDevBadBlock, static_cast<uint32_t>(id));
        return -1;
    }
    *r = rr;
    if (scales) *s = scales[id];
    return id;
}

__device__ __forceinline__ float to_float(float v) { return v; }
__device__ __forceinline__ float to_float(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T>
__device__ __forceinline__ T from_float(float v);
template <>
__device__ __forceinline__ float from_float<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// 16-byte vector loads widened to fp32.
template <typename T>
struct VecTraits;

template <>
struct VecTraits<float> {
    static constexpr int kElems = 4;
    __device__ __forceinline__ static void load(const float *p, float *v) {
        const float4 q = *reinterpret_cast<const float4 *>(p);
        v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
    }
};

template <>
struct VecTraits<__nv_bfloat16> {
    static constexpr int kElems = 8;
    __device__ __forceinline__ static void load(const __nv_bfloat16 *p, float *v) {
        const uint4 q = *reinterpret_cast<const uint4 *>(p);
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            // bf16 -> fp32 is exact: the bf16 bits are the high half of the fp32
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
};

// Vt entry e of one row (the large-M LoRA path): the block's 16 values
// s * v[j] as bf16 hi parts at columns [16e, 16e + 16) and the bf16 of what
// each hi part leaves (lo) at [kVtCols / 2 + 16e, ...), or zeros when the
// block is not the row's own adapter's (own false).
__device__ __forceinline__ void store_vt_entry(__nv_bfloat16 *vt_row, int32_t e, const float *v, bool own, float s) {
    uint32_t hw[8], lw[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float h2[2], l2[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const float val = own ? s * v[2 * i + u] : 0.0f;
            h2[u] = __bfloat162float(__float2bfloat16_rn(val));
            l2[u] = val - h2[u];
        }
        const __nv_bfloat162 hh = __floats2bfloat162_rn(h2[0], h2[1]);
        const __nv_bfloat162 ll = __floats2bfloat162_rn(l2[0], l2[1]);
        hw[i] = *reinterpret_cast<const uint32_t *>(&hh);
        lw[i] = *reinterpret_cast<const uint32_t *>(&ll);
    }
    uint4 *hd = reinterpret_cast<uint4 *>(vt_row + e * LORA_BLOCK_ROWS);
    uint4 *ld = reinterpret_cast<uint4 *>(vt_row + kVtCols / 2 + e * LORA_BLOCK_ROWS);
    hd[0] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    hd[1] = make_uint4(hw[4], hw[5], hw[6], hw[7]);
    ld[0] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    ld[1] = make_uint4(lw[4], lw[5], lw[6], lw[7]);
}

// V[m][0, r) = A_slot x[m] for one row on CUDA cores, by one warp (lanes
// over k in 8-wide pieces, then a butterfly sum): the fallback of the
// large-M path for tiles whose adapters span too many pool blocks.  The
// slot's table entries must already be checked to lie in [0, num_blocks).
// K must be a multiple of 8.  Rank-rows past r are zero in the pool, so the
// whole last block is computed and written.
__device__ __forceinline__ void row_v_by_warp(const __nv_bfloat16 *x_row, int32_t K, const __nv_bfloat16 *a_arena,
                                              const int32_t *slot_blocks, int32_t r, float *v_row, int lane) {
    const int32_t K8 = K / 8;
    const uint4 *xr = reinterpret_cast<const uint4 *>(x_row);
    for (int32_t jb = 0; jb * LORA_BLOCK_ROWS < r; ++jb) {
        const int32_t blk = slot_blocks[jb];
        const uint4 *ab = reinterpret_cast<const uint4 *>(a_arena + static_cast<size_t>(blk) * LORA_BLOCK_ROWS * K);
        float acc[LORA_BLOCK_ROWS];
#pragma unroll
        for (int j = 0; j < LORA_BLOCK_ROWS; ++j) acc[j] = 0.0f;
        for (int32_t k8 = lane; k8 < K8; k8 += 32) {
            float xv[8];
            VecTraits<__nv_bfloat16>::load(reinterpret_cast<const __nv_bfloat16 *>(xr + k8), xv);
#pragma unroll
            for (int j = 0; j < LORA_BLOCK_ROWS; ++j) {
                float av[8];
                VecTraits<__nv_bfloat16>::load(reinterpret_cast<const __nv_bfloat16 *>(ab + static_cast<size_t>(j) * K8 + k8),
                                               av);
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[j] = fmaf(av[e], xv[e], acc[j]);
            }
        }
#pragma unroll
        for (int j = 0; j < LORA_BLOCK_ROWS; ++j) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], o);
        }
        if (lane < LORA_BLOCK_ROWS) {
            float v = 0.0f;
#pragma unroll
            for (int j = 0; j < LORA_BLOCK_ROWS; ++j) v = lane == j ? acc[j] : v;
            v_row[jb * LORA_BLOCK_ROWS + lane] = v;
        }
    }
}

}  // namespace lora
