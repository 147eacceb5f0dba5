// dq_common.cuh -- dequantization of MX codes to 16-bit values, shared by
// the GEMMs that dequantize an operand before the tensor core reads it
// (dqgemm.cu: into swizzled shared-memory tiles; dqdec.cu: into tensor
// memory).  What is computed follows WWDC26 session 330, "Quantized matrix
// multiplication" (custom formats: dequantize to f16, then matmul) and
// "Quantized data types" (8-, 4- and 2-bit integers with E8M0 scales): one
// 32-element block's codes times the block's scale 2^(c - 127), rounded
// once to fp16 or bf16.
#pragma once
#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"

namespace mxk {
namespace dq {

// The block scale X = 2^(c - 127) as an fp32 (c = 0: the subnormal 2^-127;
// c = 0xFF: NaN).
__device__ __forceinline__ float scale_value(uint32_t c) {
  const uint32_t bits = c == 0 ? 0x00400000u : c == 0xFFu ? 0x7FC00000u : (c << 23);
  return __uint_as_float(bits);
}

// Eight values of one B row (codes already in registers) -> four 16-bit
// pairs.  Integers: a code's biased value u = q + 2^(bits-1) becomes the float
// 2^23 + u (OR into the bit pattern of 2^23), and fma(2^23 + u, X,
// -(2^23 + 2^(bits-1)) X) = q X exactly, rounded once.  That constant
// overflows fp32 for X >= 2^105; with SAFE the code is first turned into the
// exact float q = (2^23 + u) - (2^23 + 2^(bits-1)) and then multiplied by X
// (exact, or +-inf when q X itself is out of range).
template <int FMT, bool SAFE = false>
__device__ __forceinline__ void dq8(const uint32_t* w, int i, float X, bool bf16, uint32_t (&o)[4]) {
  float y[8];
  // m: the bit pattern of 2^23 + u
  auto from_magic = [&](uint32_t m, float bias_magic, float c) {
    return SAFE ? (__uint_as_float(m) - bias_magic) * X : fmaf(__uint_as_float(m), X, c);
  };
  if (FMT == FMT_INT8) {
    const float c = -8388736.0f * X;                     // -(2^23 + 128) X
    const uint32_t v0 = w[2 * i] ^ 0x80808080u, v1 = w[2 * i + 1] ^ 0x80808080u;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      y[e] = from_magic(__byte_perm(v0, 0x4B000000u, 0x7650 | e), 8388736.0f, c);
      y[4 + e] = from_magic(__byte_perm(v1, 0x4B000000u, 0x7650 | e), 8388736.0f, c);
    }
  } else if (FMT == FMT_INT4) {
    const float c = -8388616.0f * X;                     // -(2^23 + 8) X
    const uint32_t v = w[i] ^ 0x88888888u;
#pragma unroll
    for (int e = 0; e < 8; ++e)
      y[e] = from_magic(((v >> (4 * e)) & 0xFu) | 0x4B000000u, 8388616.0f, c);
  } else if (FMT == FMT_INT2) {
    const float c = -8388610.0f * X;                     // -(2^23 + 2) X
    const uint32_t v = (w[i >> 1] >> (16 * (i & 1))) ^ 0xAAAAu;
#pragma unroll
    for (int e = 0; e < 8; ++e)
      y[e] = from_magic(((v >> (2 * e)) & 0x3u) | 0x4B000000u, 8388610.0f, c);
  } else if (FMT == FMT_E2M1) {
    const uint32_t v = w[i];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float lo, hi;
      f16x2_to_f32(cvt_f16x2_e2m1x2((v >> (8 * e)) & 0xFFu), lo, hi);
      y[2 * e] = lo * X;
      y[2 * e + 1] = hi * X;
    }
  } else {                                               // E4M3 / E5M2
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t pair = (w[2 * i + (e >> 1)] >> (16 * (e & 1))) & 0xFFFFu;
      const uint32_t h = (FMT == FMT_E5M2) ? cvt_f16x2_e5m2x2(pair) : cvt_f16x2_e4m3x2(pair);
      float lo, hi;
      f16x2_to_f32(h, lo, hi);
      y[2 * e] = lo * X;
      y[2 * e + 1] = hi * X;
    }
  }
#pragma unroll
  for (int e = 0; e < 4; ++e)
    o[e] = bf16 ? cvt_bf16x2(y[2 * e], y[2 * e + 1]) : cvt_f16x2(y[2 * e], y[2 * e + 1]);
}

// bf16 pairs of integer codes, the packed path for a bf16 A: the biased code
// u = q + 2^(bits-1) (< 128) as the low byte under the high byte 0x43 is the
// bf16 value 128 + u, exactly; fma(128 + u, X, -(128 + 2^(bits-1)) X) = q X,
// one rounding of an exact bf16 value (X a power of two, so every product
// here is exact): two elements per instruction, no conversions.  The biased
// codes are spread one per byte with masks, paired with byte permutes, and
// the 0x43 bytes are spliced in with a last permute.
constexpr uint32_t kBf16Hi = 0x43434343u;

// 8 int4 codes (element e at bits 4e) -> four bf16 pairs (128 + u).
__device__ __forceinline__ void int4_pairs(uint32_t v, uint32_t (&o)[4]) {
  const uint32_t L = (v & 0x0F0F0F0Fu) ^ 0x08080808u;          // u0 u2 u4 u6
  const uint32_t H = ((v >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;   // u1 u3 u5 u7
  const uint32_t t0 = __byte_perm(L, H, 0x5140);               // u0 u1 u2 u3
  const uint32_t t1 = __byte_perm(L, H, 0x7362);               // u4 u5 u6 u7
  o[0] = __byte_perm(t0, kBf16Hi, 0x4140);
  o[1] = __byte_perm(t0, kBf16Hi, 0x4342);
  o[2] = __byte_perm(t1, kBf16Hi, 0x4140);
  o[3] = __byte_perm(t1, kBf16Hi, 0x4342);
}

// 16 int2 codes (element e at bits 2e) -> eight bf16 pairs (128 + u),
// elements 0..7 in o[0..3], 8..15 in o[4..7].
__device__ __forceinline__ void int2_pairs(uint32_t v, uint32_t (&o)[8]) {
  const uint32_t E0 = (v & 0x03030303u) ^ 0x02020202u;         // e0 e4 e8 e12
  const uint32_t E1 = ((v >> 2) & 0x03030303u) ^ 0x02020202u;  // e1 e5 e9 e13
  const uint32_t E2 = ((v >> 4) & 0x03030303u) ^ 0x02020202u;  // e2 e6 e10 e14
  const uint32_t E3 = ((v >> 6) & 0x03030303u) ^ 0x02020202u;  // e3 e7 e11 e15
  const uint32_t a = __byte_perm(E0, E1, 0x5140);              // e0 e1 e4 e5
  const uint32_t b = __byte_perm(E2, E3, 0x5140);              // e2 e3 e6 e7
  const uint32_t c = __byte_perm(E0, E1, 0x7362);              // e8 e9 e12 e13
  const uint32_t d = __byte_perm(E2, E3, 0x7362);              // e10 e11 e14 e15
  o[0] = __byte_perm(a, kBf16Hi, 0x4140);
  o[1] = __byte_perm(b, kBf16Hi, 0x4140);
  o[2] = __byte_perm(a, kBf16Hi, 0x4342);
  o[3] = __byte_perm(b, kBf16Hi, 0x4342);
  o[4] = __byte_perm(c, kBf16Hi, 0x4140);
  o[5] = __byte_perm(d, kBf16Hi, 0x4140);
  o[6] = __byte_perm(c, kBf16Hi, 0x4342);
  o[7] = __byte_perm(d, kBf16Hi, 0x4342);
}

// Bytes of one 32-element block of codes.
template <int FMT>
__host__ __device__ constexpr int block_code_bytes() {
  return (FMT == FMT_INT8 || FMT == FMT_E4M3 || FMT == FMT_E5M2) ? 32
         : (FMT == FMT_INT2)                                    ? 8
                                                                : 16;
}

// One 32-element block's codes (block_code_bytes<FMT>() bytes, 8-byte
// aligned, 16-byte aligned unless int2) into words w[0 ..).
template <int FMT>
__device__ __forceinline__ void load_block_codes(const uint8_t* codes, uint32_t (&w)[8]) {
  constexpr int BB = block_code_bytes<FMT>();
  if (BB == 8) {
    const uint2 q = *reinterpret_cast<const uint2*>(codes);
    w[0] = q.x;
    w[1] = q.y;
  } else {
#pragma unroll
    for (int v = 0; v < BB / 16; ++v) {
      const uint4 q = reinterpret_cast<const uint4*>(codes)[v];
      w[4 * v] = q.x;
      w[4 * v + 1] = q.y;
      w[4 * v + 2] = q.z;
      w[4 * v + 3] = q.w;
    }
  }
}

// One 32-element block (codes in w, scale code sc) -> sixteen 16-bit pairs
// o[0 .. 15], element 2 i in the low half of o[i].
template <int FMT>
__device__ __forceinline__ void dq_block_regs(const uint32_t (&w)[8], uint32_t sc, bool bf16,
                                              uint32_t (&o)[16]) {
  const float X = scale_value(sc);
  constexpr bool INT = (FMT == FMT_INT8 || FMT == FMT_INT4 || FMT == FMT_INT2);
  // -(128 + 2^(bits-1)) X is a finite bf16 up to X = 2^120 (scale code 247)
  if ((FMT == FMT_INT4 || FMT == FMT_INT2) && bf16 && sc <= 247u) {
    constexpr int BITS = (FMT == FMT_INT4) ? 4 : 2;
    const uint32_t xb = __float_as_uint(X) >> 16;                      // exact
    const uint32_t cb = __float_as_uint(-(128.0f + (1 << (BITS - 1))) * X) >> 16;
    const uint32_t x2 = xb | (xb << 16), c2 = cb | (cb << 16);
    if (BITS == 4) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t p[4];
        int4_pairs(w[j], p);
#pragma unroll
        for (int e = 0; e < 4; ++e) o[4 * j + e] = fma_bf16x2(p[e], x2, c2);
      }
    } else {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        uint32_t p[8];
        int2_pairs(w[k], p);
#pragma unroll
        for (int e = 0; e < 8; ++e) o[8 * k + e] = fma_bf16x2(p[e], x2, c2);
      }
    }
    return;
  }
  // the fp32 magic constant -(2^23 + 2^(bits-1)) X is finite up to X = 2^104
  // (scale code 231); larger scales of integer codes take the exact two-step
  if (INT && sc > 231u) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t p[4];
      dq8<FMT, true>(w, j, X, bf16, p);
#pragma unroll
      for (int e = 0; e < 4; ++e) o[4 * j + e] = p[e];
    }
    return;
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t p[4];
    dq8<FMT>(w, j, X, bf16, p);
#pragma unroll
    for (int e = 0; e < 4; ++e) o[4 * j + e] = p[e];
  }
}

}  // namespace dq
}  // namespace mxk
