// Encoding of one binary32 value into an 8-bit KV-cache code with the
// (block, head) scale s, shared by the store and quantize kernels and by the
// decode kernel's fused append.
//
// "Block-Paged KV Cache" (Hurray format documentation), Quantization
// compatibility: per-block-affine scales, one per page slot.  A stored value
// is s * decode(code).  E4M3: x / s in binary32, rounded to the nearest even
// OCP E4M3 code, saturating at +-448.  int8: x / s rounded to the nearest
// integer (ties to even), NaN -> 0, clamped to +-127.  A zero scale stores
// code 0 in both formats.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace pkv {
namespace {

// binary32 -> int8 code: nearest integer, ties to even (cvt.rni); NaN -> 0
// (the conversion's rule for NaN), then clamped to +-127.
__device__ __forceinline__ uint32_t q8_int8_code(float y) {
    const int r = min(max(__float2int_rn(y), -127), 127);
    return static_cast<uint32_t>(r) & 0xFFu;
}

// Two binary32 -> two codes (lo in the low byte) of x / s; a zero scale gives 0.
template <bool INT8> __device__ __forceinline__ uint32_t q8_encode2(float lo, float hi, float s) {
    if (s == 0.f) return 0u;
    const float a = __fdiv_rn(lo, s), b = __fdiv_rn(hi, s);
    if constexpr (INT8) {
        return q8_int8_code(a) | q8_int8_code(b) << 8;
    } else {
        uint16_t d;
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(b), "f"(a));
        return d;
    }
}

}  // namespace
}  // namespace pkv
