// mx_rule.cuh -- the OCP MX conversion rule on the device, shared by the
// quantizer (quantize.cu) and the GEMM epilogue that writes C as an MX tensor
// (gemm.cu):
//   amax = max |x| over a block of 32; e = floor(log2 amax) from the fp32
//   exponent field; X = 2^clamp(e - emax, -127, 127); the scale code is
//   log2(X) + 127 (0 for an all-zero block, 0xFF when the block holds a NaN
//   or an infinity); each element is x / X rounded to nearest-even and
//   saturated to the element format.
#pragma once
#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"

namespace mxk {

__device__ __forceinline__ uint32_t abs_bits(float x) {
  return __float_as_uint(x) & 0x7FFFFFFFu;
}

template <int FMT>
__host__ __device__ constexpr int emax_of() {
  return FMT == FMT_E4M3 ? 8 : FMT == FMT_E5M2 ? 15 : 2;
}

// Two scaled values -> two 8-bit codes (lo in the low byte).
template <int FMT>
__device__ __forceinline__ uint32_t cvt8x2(float lo, float hi) {
  return FMT == FMT_E5M2 ? cvt_e5m2x2(lo, hi) : cvt_e4m3x2(lo, hi);
}

// Scale code and the multiplier 1/X for a block whose largest |x| has the bit
// pattern amax (sign cleared).  emax: 8 for E4M3, 15 for E5M2, 2 for E2M1.
__device__ __forceinline__ void block_scale(uint32_t amax, int emax,
                                            uint32_t& code, float& inv_x) {
  if (amax >= 0x7F800000u) {          // Inf or NaN somewhere in the block
    code = 0xFFu;
    inv_x = 1.0f;
    return;
  }
  int es;
  if (amax == 0u) {
    es = -127;
  } else {
    const int E = static_cast<int>(amax >> 23);
    const int e = E ? (E - 127) : ((31 - __clz(static_cast<int>(amax))) - 149);
    es = e - emax;
    es = es < -127 ? -127 : (es > 127 ? 127 : es);
  }
  code = static_cast<uint32_t>(es + 127);
  // 2^-es as an fp32: biased exponent 127 - es lies in [2, 254] because
  // e <= 127 bounds es above by 119 (E4M3) / 112 (E5M2) / 125 (E2M1).
  inv_x = __uint_as_float(static_cast<uint32_t>(127 - es) << 23);
}

// Runtime form of emax_of.
__host__ __device__ __forceinline__ int emax_of_fmt(int fmt) {
  return fmt == FMT_E4M3 ? 8 : fmt == FMT_E5M2 ? 15 : 2;
}

}  // namespace mxk
