// gemm_common.cuh -- pieces shared by the GEMM kernels (gemm.cu: the
// tensor-core GEMM on MX and 16-bit operands; dqgemm.cu: the GEMM that
// dequantizes its B operand in shared memory): tile geometry, the raster
// order of tiles, and the epilogue (bias, activation, the MX quantization of
// C) applied to accumulator rows held in registers.
#pragma once
#include <cstdint>

#include "common.cuh"
#include "mx_rule.cuh"
#include "ptx.cuh"

namespace mxk {

constexpr int BM = 128;              // rows of A per CTA
constexpr int BN = 256;              // columns of C per tile
constexpr int GROUP_M = 8;           // raster group height in M tiles

// the form in which the epilogue stores C
enum Out : int { OUT_F32 = 0, OUT_BF16 = 1, OUT_MX8 = 2, OUT_MX4 = 3 };

// Tiles walked in groups of `group` tile rows, column by column inside a
// group, so that the clusters running at the same time share A and B tiles
// in L2, and a group's rows of A stay in L2 while all of B streams past them
// once: B is read from DRAM once per group.  Odd groups walk the columns
// backwards, so a group starts on the columns of B its predecessor read last
// (still in L2).
struct TileSched {
  int num_m, num_n, total;   // in tiles
  int group = GROUP_M;       // tile rows per raster group
  __host__ __device__ __forceinline__ void tile(int t, int& mb, int& nb) const {
    const int per_group = group * num_n;
    const int g = t / per_group;
    const int first_m = g * group;
    const int gsz = min(num_m - first_m, group);
    const int r = t - g * per_group;
    mb = first_m + r % gsz;
    nb = (g & 1) ? num_n - 1 - r / gsz : r / gsz;
  }
};


// Kernel-side form of Epilogue (plus the geometry of an MX output's scale
// plane).
struct EpiArgs {
  const float* bias;
  int act;
  int q_fmt;
  uint8_t* q_sf;
  int64_t q_k_atoms;     // atoms along the columns of C
  int64_t q_row_atoms;   // atoms along the rows of C
};

// GELU(x) = x * Phi(x) = x (1 + erf(x / sqrt 2)) / 2.  Inlined, so that the
// 128 evaluations of one thread interleave.  Where 1 + erf cancels (x below
// about -4) the result keeps an absolute error near 2^-24 |x| instead of its
// relative accuracy, far below the product's own accumulation error.
__device__ __forceinline__ float gelu_exact(float x) {
  return 0.5f * x * (1.0f + erff(x * 0.7071067811865476f));
}

// The tanh approximation: 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))),
// evaluated as x / (1 + e^(-2u)), the same function (1 + tanh u =
// 2 / (1 + e^(-2u))) in three instructions on the special-function unit
// instead of a tanh: 2^-2u log2 e by ex2.approx, then one fast division.
// Both ends are exact limits: u -> +inf gives x, u -> -inf gives x / inf = 0.
// 0.331 -> 0.261 ms for a 16384 x 8192 x 2048 MXFP8 product with bias +
// GELU-tanh against tanhf.
__device__ __forceinline__ float gelu_tanh(float x) {
  const float u = 0.7978845608028654f * (x + 0.044715f * x * x * x);
  return __fdividef(x, 1.0f + ex2_approx(-2.8853900817779268f * u));
}

// Bias and activation on one thread's EPI_COLS accumulator values of one row
// of C, columns col0 .. col0 + EPI_COLS - 1 (bias is read below N only).
template <int NC>
__device__ __forceinline__ void apply_bias_act(uint32_t (&r)[NC], const EpiArgs& e, int col0,
                                               int N) {
  if (e.bias != nullptr) {
#pragma unroll
    for (int v = 0; v < NC / 4; ++v) {
      const int c = col0 + 4 * v;
      float4 b = make_float4(0.f, 0.f, 0.f, 0.f);
      if (c + 3 < N) {
        b = __ldg(reinterpret_cast<const float4*>(e.bias + c));
      } else {
        if (c < N) b.x = __ldg(e.bias + c);
        if (c + 1 < N) b.y = __ldg(e.bias + c + 1);
        if (c + 2 < N) b.z = __ldg(e.bias + c + 2);
      }
      r[4 * v + 0] = __float_as_uint(__uint_as_float(r[4 * v + 0]) + b.x);
      r[4 * v + 1] = __float_as_uint(__uint_as_float(r[4 * v + 1]) + b.y);
      r[4 * v + 2] = __float_as_uint(__uint_as_float(r[4 * v + 2]) + b.z);
      r[4 * v + 3] = __float_as_uint(__uint_as_float(r[4 * v + 3]) + b.w);
    }
  }
  if (e.act == ACT_GELU) {
#pragma unroll
    for (int i = 0; i < NC; ++i) r[i] = __float_as_uint(gelu_exact(__uint_as_float(r[i])));
  } else if (e.act == ACT_GELU_TANH) {
#pragma unroll
    for (int i = 0; i < NC; ++i) r[i] = __float_as_uint(gelu_tanh(__uint_as_float(r[i])));
  }
}

// 32 bytes to p (16-byte aligned): one 256-bit store where p is 32-byte
// aligned, else two 16-byte stores.
__device__ __forceinline__ void store_32B(void* p, const uint32_t (&w)[8], bool wide) {
  if (wide) {
    st_global_v8(p, w);
  } else {
    uint4* q = reinterpret_cast<uint4*>(p);
    q[0] = make_uint4(w[0], w[1], w[2], w[3]);
    q[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

// Quantize one row's 32 values of C (one block: columns c .. c + 31, c < N,
// N a multiple of 32) by the OCP rule: codes to the MX data plane (row stride
// N codes), the block's scale code returned.
template <int OUT>
__device__ __forceinline__ uint32_t quantize_block_row(const uint32_t (&x)[32], const EpiArgs& e,
                                                       uint8_t* data, int64_t row, int c, int N) {
  uint32_t a = 0;
#pragma unroll
  for (int i = 0; i < 32; ++i) a = max(a, x[i] & 0x7FFFFFFFu);
  uint32_t code;
  float s;
  block_scale(a, emax_of_fmt(e.q_fmt), code, s);
  if (OUT == OUT_MX8) {
    const bool e5 = (e.q_fmt == FMT_E5M2);
    uint32_t q[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float x0 = __uint_as_float(x[4 * i]) * s, x1 = __uint_as_float(x[4 * i + 1]) * s;
      const float x2 = __uint_as_float(x[4 * i + 2]) * s, x3 = __uint_as_float(x[4 * i + 3]) * s;
      q[i] = e5 ? (cvt_e5m2x2(x0, x1) | (cvt_e5m2x2(x2, x3) << 16))
                : (cvt_e4m3x2(x0, x1) | (cvt_e4m3x2(x2, x3) << 16));
    }
    uint8_t* dst = data + row * N + c;
    store_32B(dst, q, (reinterpret_cast<uintptr_t>(dst) & 31u) == 0);
  } else {
    uint32_t q[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t* y = x + 8 * i;
      q[i] = cvt_e2m1x2(__uint_as_float(y[0]) * s, __uint_as_float(y[1]) * s) |
             (cvt_e2m1x2(__uint_as_float(y[2]) * s, __uint_as_float(y[3]) * s) << 8) |
             (cvt_e2m1x2(__uint_as_float(y[4]) * s, __uint_as_float(y[5]) * s) << 16) |
             (cvt_e2m1x2(__uint_as_float(y[6]) * s, __uint_as_float(y[7]) * s) << 24);
    }
    *reinterpret_cast<uint4*>(data + (row * N + c) / 2) = make_uint4(q[0], q[1], q[2], q[3]);
  }
  return code;
}

// One row's four scale codes for columns col0 .. col0 + 127 (col0 a multiple
// of 128: one 32-bit word of the scale plane).  Rows beyond M inside the last
// row atom and blocks beyond N carry code 0, the plane's padding.
__device__ __forceinline__ void store_mx_scales(uint32_t sf_word, const EpiArgs& e, int64_t row,
                                                int col0, int N) {
  if (col0 >= N || (row >> 7) >= e.q_row_atoms) return;
  *reinterpret_cast<uint32_t*>(e.q_sf + ((row >> 7) * e.q_k_atoms + (col0 >> 7)) * SF_ATOM_BYTES +
                               sf_in_atom(static_cast<int>(row & 127), 0)) = sf_word;
}

// Store one row's 128 values of C (columns col0 .. col0 + 127) as an MX
// tensor: four blocks of 32, then the row's scale word.
template <int OUT, int NC>
__device__ __forceinline__ void store_mx_row(const uint32_t (&r)[NC], const EpiArgs& e,
                                             uint8_t* data, int64_t row, int col0, int M,
                                             int N) {
  static_assert(NC == 4 * 32, "one thread stores four whole blocks");
  uint32_t sf = 0;
  if (row < M) {
#pragma unroll
    for (int b = 0; b < NC / 32; ++b) {
      const int c = col0 + 32 * b;
      if (c < N)
        sf |= quantize_block_row<OUT>(*reinterpret_cast<const uint32_t(*)[32]>(r + 32 * b), e,
                                      data, row, c, N)
              << (8 * b);
    }
  }
  store_mx_scales(sf, e, row, col0, N);
}

// One thread's segment of one row of a plain C: NV fp32 accumulator values
// for columns c0 .. c0 + NV - 1 (c0 a multiple of 16), stored as fp32 or as
// bf16 (RNE), clipped at N.  Each thread writes its own row, so the warp's
// stores hit 32 different rows: 32 bytes per store fill whole L2 sectors,
// where 16-byte stores left a stream of half-sector writes that slowed the
// GEMMs' operand loads (measured, 8192^3 with bf16 C: MXFP4 9 %, MXFP8 2 %;
// 16384 x 8192 x 2048 MXFP8 18 %).
template <int OUT, int NV>
__device__ __forceinline__ void store_row_segment(const uint32_t (&r)[NV], void* C, int64_t ldc,
                                                  int64_t row, int c0, int N) {
  if (OUT == OUT_BF16) {
    static_assert(NV % 16 == 0, "16 bf16 columns per store");
    uint16_t* crow = reinterpret_cast<uint16_t*>(C) + row * ldc;
    const bool wide = (reinterpret_cast<uintptr_t>(crow) & 31u) == 0;
#pragma unroll
    for (int v = 0; v < NV / 16; ++v) {
      const int c = c0 + 16 * v;
      uint32_t w[8];
#pragma unroll
      for (int e = 0; e < 8; ++e)
        w[e] = cvt_bf16x2(__uint_as_float(r[16 * v + 2 * e]),
                          __uint_as_float(r[16 * v + 2 * e + 1]));
      if (c + 15 < N) {
        store_32B(crow + c, w, wide);
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e)
          if (c + e < N) crow[c + e] = static_cast<uint16_t>(w[e >> 1] >> (16 * (e & 1)));
      }
    }
  } else {
    static_assert(NV % 8 == 0, "8 fp32 columns per store");
    float* crow = reinterpret_cast<float*>(C) + row * ldc;
    const bool wide = (reinterpret_cast<uintptr_t>(crow) & 31u) == 0;
#pragma unroll
    for (int v = 0; v < NV / 8; ++v) {
      const int c = c0 + 8 * v;
      if (c + 7 < N) {
        store_32B(crow + c, *reinterpret_cast<const uint32_t(*)[8]>(r + 8 * v), wide);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (c + e < N) crow[c + e] = __uint_as_float(r[8 * v + e]);
      }
    }
  }
}

// Tensor maps (cuTensorMapEncodeTiled, through the driver entry point):
// a rows x cols matrix of elem_bytes elements, leading dimension ld_elems, a
// box of box_cols x box_rows.  Returns false when the driver rejects it.
bool make_tmap(CUtensorMap* m, const void* ptr, CUtensorMapDataType dt, int elem_bytes,
               uint64_t cols, uint64_t rows, uint64_t ld_elems, uint32_t box_cols,
               uint32_t box_rows, CUtensorMapSwizzle swz);

// Any rank: dims / box / element strides innermost first, strides in bytes
// for dimensions 1 .. rank-1.
bool encode_tiled(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* ptr,
                  const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                  const cuuint32_t* estr, CUtensorMapSwizzle swz);

}  // namespace mxk
