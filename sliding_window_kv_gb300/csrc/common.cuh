// common.cuh -- device helpers shared by every kernel: the RoPE rotation (one definition, so
// a key rotated by the append kernel and by the fused decode kernel is the same bf16 value),
// bf16 packing, and the 128-byte swizzle used by TMA tiles and tcgen05 operands.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

namespace vst {

// NEOX rotation of the pair (x1, x2) = (x[i], x[i + D/2]) by the angle whose (cos, sin) is
// cs (family doc "Voxtral Realtime", Architecture: NEOX RoPE; rotate-half convention
// y = x cos + rotate_half(x) sin). The rounding is pinned with explicit _rn intrinsics so
// that every kernel produces identical bits for the same (x, position).
__device__ __forceinline__ void rope_pair(float x1, float x2, float2 cs, float& y1, float& y2)
{
    y1 = __fmaf_rn(x1, cs.x, __fmul_rn(-x2, cs.y));
    y2 = __fmaf_rn(x2, cs.x, __fmul_rn(x1, cs.y));
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Round two floats to bf16 (nearest even) and pack: a in the low half.
__device__ __forceinline__ uint32_t pack_bf16(float a, float b)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` in a 128-byte-swizzled tile whose
// rows are 128 bytes (the layout TMA writes with CU_TENSOR_MAP_SWIZZLE_128B and tcgen05
// reads with a SWIZZLE_128B descriptor; tile base 1024-byte aligned).
__device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t chunk)
{
    return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

}  // namespace vst
