// mx_rule.cuh -- the OCP MX conversion rule on the device, shared by the
// quantizer (quantize.cu) and the GEMM epilogue that writes C as an MX tensor
// (gemm.cu):
//   amax = max |x| over a block of 32; e = floor(log2 amax) from the fp32
//   exponent field; X = 2^clamp(e - emax, -127, 127); the scale code is
//   log2(X) + 127 (0 for an all-zero block, 0xFF when the block holds a NaN
//   or an infinity); each element is x / X rounded to nearest-even and
//   saturated to the element format.  Integer formats (int8 / int4 / int2,
//   two's complement) use emax = bits - 2, the largest power of two they
//   hold, and round x / X to the nearest integer, ties to even, saturated to
//   their range (WWDC26 session 330, "Quantized data types": 8-, 4- and
//   2-bit integer elements under E8M0 block scales; for int8 this is the OCP
//   MXINT8 rule with its implicit 2^-6 folded into X).
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
  return FMT == FMT_E4M3 ? 8 : FMT == FMT_E5M2 ? 15 : FMT == FMT_INT8 ? 6 : FMT == FMT_INT2 ? 0 : 2;
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
  // 2^-es as an fp32: biased exponent 127 - es, in [1, 254] for every format
  // but int2 (emax 0), whose es reaches 127 when the block maximum is near
  // 2^127: then 2^-127 is the fp32 subnormal 0x00400000 (a block maximum of
  // that size times it is still a normal number, exactly).
  inv_x = es >= 127 ? __uint_as_float(0x00400000u)
                    : __uint_as_float(static_cast<uint32_t>(127 - es) << 23);
}

// Runtime form of emax_of.
__host__ __device__ __forceinline__ int emax_of_fmt(int fmt) {
  return fmt == FMT_E4M3 ? 8 : fmt == FMT_E5M2 ? 15 : fmt == FMT_INT8 ? 6 : fmt == FMT_INT2 ? 0 : 2;
}

// One scaled value -> an integer code of `bits` bits: nearest integer, ties
// to even (cvt.rni), saturated to the two's-complement range.
template <int BITS>
__device__ __forceinline__ uint32_t int_code(float v) {
  constexpr int lo = -(1 << (BITS - 1)), hi = (1 << (BITS - 1)) - 1;
  int q = __float2int_rn(v);
  q = q < lo ? lo : (q > hi ? hi : q);
  return static_cast<uint32_t>(q) & ((1u << BITS) - 1u);
}

// Four consecutive elements x0..x3 (already multiplied by 1/X) -> their codes
// packed in element order: 32 bits (8-bit formats), 16 (E2M1, int4) or 8
// (int2); element 0 in the lowest bits.
template <int FMT>
__device__ __forceinline__ uint32_t codes4(float x0, float x1, float x2, float x3) {
  if (FMT == FMT_E4M3 || FMT == FMT_E5M2) return cvt8x2<FMT>(x0, x1) | (cvt8x2<FMT>(x2, x3) << 16);
  if (FMT == FMT_E2M1) return cvt_e2m1x2(x0, x1) | (cvt_e2m1x2(x2, x3) << 8);
  if (FMT == FMT_INT8)
    return int_code<8>(x0) | (int_code<8>(x1) << 8) | (int_code<8>(x2) << 16) |
           (int_code<8>(x3) << 24);
  if (FMT == FMT_INT4)
    return int_code<4>(x0) | (int_code<4>(x1) << 4) | (int_code<4>(x2) << 8) |
           (int_code<4>(x3) << 12);
  return int_code<2>(x0) | (int_code<2>(x1) << 2) | (int_code<2>(x2) << 4) | (int_code<2>(x3) << 6);
}

}  // namespace mxk
