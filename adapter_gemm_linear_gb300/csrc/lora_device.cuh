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

}  // namespace lora
