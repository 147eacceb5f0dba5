// quantize.cu -- OCP MX quantization, fp32 -> an E4M3 / E5M2 / E2M1 / int8 /
// int4 / int2 data plane plus a UE8M0 scale plane in the tensor-core
// scale-factor layout.
//
// The rule (OCP Microscaling v1.0 conversion; block of 32 along the
// innermost / K axis as in the WWDC26 session 330 "Multi-plane tensors"
// chapter and its 4:48 listing, block factors {32, 1}):
//   amax = max |x| over the 32 values of the block
//   e    = floor(log2 amax), read off the fp32 exponent field (for a subnormal
//          amax, from the position of its leading one) -- never via a log
//          function, which can round up just below a power of two
//   X    = 2^clamp(e - emax, -127, 127), emax = 8 (E4M3) / 15 (E5M2) / 2 (E2M1)
//          / bits - 2 (int8 6, int4 2, int2 0)
//   code = e_s + 127 (UE8M0); all-zero block -> 0; NaN/Inf in block -> 0xFF
//   q_i  = RNE-saturate(x_i / X) to the element format (for the integers: the
//          nearest integer, ties to even, saturated to the two's-complement
//          range).
// x / X is a multiplication by a power of two in fp32; it is exact except when
// the product is an fp32 subnormal, which every element format rounds to +-0
// anyway (the smallest E5M2 subnormal is 2^-16).
//
// Both kernels are HBM-streaming passes: each CTA owns one 128-row x 128-K
// region, i.e. exactly one 512-byte scale atom, which it assembles in shared
// memory and writes out as one coalesced 512-byte store.
#include "common.cuh"
#include "mx_rule.cuh"
#include "ptx.cuh"

namespace mxk {

namespace {

__device__ unsigned int g_status_quantize = 0;

constexpr int QT_THREADS = 256;   // 8 warps per CTA

// ---------------------------------------------------------------------------
// Source outer x K, K contiguous.  CTA = (K chunk kc, row group rg); each warp
// owns 16 rows; for one row a warp reads the chunk's 128 floats as 32 float4,
// lane l covering k = 4l..4l+3 of block l/8.  The block amax is a max over 8
// lanes (shuffles), the 4 codes of a lane are one 32-bit (8-bit formats) or
// 16-bit (E2M1) store, so a warp stores 128 (64) contiguous bytes per row.
template <int FMT>
__global__ void __launch_bounds__(QT_THREADS)
quantize_kcontig(const float* __restrict__ src, int64_t ld, int64_t outer,
                 int64_t K, uint8_t* __restrict__ data, uint8_t* __restrict__ sf) {
  constexpr int EMAX = emax_of<FMT>();
  constexpr int ROWS_PER_WARP = 16;
  // Rows whose loads are in flight together.  Fewer registers (40 at 4, 64
  // at 8, 80 at 16) keep more CTAs resident, which pays more than deeper
  // batches: 8192 x 8192 E4M3 took 0.054 / 0.056 / 0.061 ms at 4 / 8 / 16.
  constexpr int BATCH = 4;
  __shared__ __align__(16) uint8_t atom[SF_ATOM_BYTES];

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int64_t kc = blockIdx.x;
  const int64_t rg = blockIdx.y;
  const int64_t k_atoms = sf_k_atoms(K);

  for (int i = threadIdx.x; i < SF_ATOM_BYTES / 16; i += QT_THREADS)
    reinterpret_cast<uint4*>(atom)[i] = make_uint4(0, 0, 0, 0);
  __syncthreads();

  const int64_t k = kc * 128 + 4 * lane;
  const bool kvalid = (kc * 128 + 32 * (lane >> 3)) < K;   // K % 32 == 0
  const int j = lane >> 3;

#pragma unroll
  for (int b0 = 0; b0 < ROWS_PER_WARP; b0 += BATCH) {
    float4 v[BATCH];
#pragma unroll
    for (int i = 0; i < BATCH; ++i) {
      const int64_t r = rg * 128 + warp * ROWS_PER_WARP + b0 + i;
      if (kvalid && r < outer)
        v[i] = __ldcs(reinterpret_cast<const float4*>(src + r * ld + k));
      else
        v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int i = 0; i < BATCH; ++i) {
      const int rl = warp * ROWS_PER_WARP + b0 + i;     // row inside group
      const int64_t r = rg * 128 + rl;
      uint32_t a = max(max(abs_bits(v[i].x), abs_bits(v[i].y)),
                       max(abs_bits(v[i].z), abs_bits(v[i].w)));
      a = max(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
      a = max(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
      a = max(a, __shfl_xor_sync(0xFFFFFFFFu, a, 4));
      uint32_t code;
      float s;
      block_scale(a, EMAX, code, s);
      if (r < outer && kvalid) {
        if ((lane & 7) == 0) atom[sf_in_atom(rl, j)] = static_cast<uint8_t>(code);
        const uint32_t c4 = codes4<FMT>(v[i].x * s, v[i].y * s, v[i].z * s, v[i].w * s);
        constexpr int BITS = (FMT == FMT_INT2) ? 2 : (FMT == FMT_E2M1 || FMT == FMT_INT4) ? 4 : 8;
        if (BITS == 8)
          *reinterpret_cast<uint32_t*>(data + r * K + k) = c4;
        else if (BITS == 4)
          *reinterpret_cast<uint16_t*>(data + (r * K + k) / 2) = static_cast<uint16_t>(c4);
        else
          data[(r * K + k) / 4] = static_cast<uint8_t>(c4);
      }
    }
  }
  __syncthreads();
  if (threadIdx.x < SF_ATOM_BYTES / 16) {
    uint4* dst = reinterpret_cast<uint4*>(sf + (rg * k_atoms + kc) * SF_ATOM_BYTES);
    dst[threadIdx.x] = reinterpret_cast<const uint4*>(atom)[threadIdx.x];
  }
}

// ---------------------------------------------------------------------------
// Source K x outer, outer contiguous (a row-major K x N operand); output is
// outer x K (K-major).  CTA = (row group rg of 128 outputs, K chunk kc of 128),
// 4 warps; warp w owns block j = w (32 consecutive K) and lane l owns the four
// output rows n = 128*rg + 4l .. 4l+3.  For i = 0..31 the warp loads source
// row k = 128*kc + 32*w + i at columns 128*rg + 4l.. as one float4 per lane --
// 512 contiguous bytes per warp instruction -- so each lane ends up holding the
// complete 32-element block of each of its four output rows in registers: the
// transpose costs no shared-memory pass and the amax no shuffles.
template <int FMT>
__global__ void __launch_bounds__(128)
quantize_kstrided(const float* __restrict__ src, int64_t ld, int64_t outer,
                  int64_t K, uint8_t* __restrict__ data, uint8_t* __restrict__ sf) {
  constexpr int EMAX = emax_of<FMT>();
  __shared__ __align__(16) uint8_t atom[SF_ATOM_BYTES];

  const int lane = threadIdx.x & 31;
  const int w = threadIdx.x >> 5;
  const int64_t rg = blockIdx.x;
  const int64_t kc = blockIdx.y;
  const int64_t k_atoms = sf_k_atoms(K);

  reinterpret_cast<uint32_t*>(atom)[threadIdx.x] = 0u;   // 128 threads x 4 B
  __syncthreads();

  const int64_t kb = kc * 128 + 32 * w;            // first K of this warp's block
  const int64_t n = rg * 128 + 4 * lane;           // first of the lane's 4 rows
  if (kb < K) {                                    // K % 32 == 0: whole block valid
    float4 v[32];
    const float* p = src + kb * ld + n;
    if (n + 3 < outer) {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = __ldcs(reinterpret_cast<const float4*>(p + i * ld));
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (n + 0 < outer) v[i].x = __ldcs(p + i * ld + 0);
        if (n + 1 < outer) v[i].y = __ldcs(p + i * ld + 1);
        if (n + 2 < outer) v[i].z = __ldcs(p + i * ld + 2);
      }
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      if (n + c >= outer) break;
      float x[32];
#pragma unroll
      for (int i = 0; i < 32; ++i)
        x[i] = (c == 0) ? v[i].x : (c == 1) ? v[i].y : (c == 2) ? v[i].z : v[i].w;
      uint32_t a = 0;
#pragma unroll
      for (int i = 0; i < 32; ++i) a = max(a, abs_bits(x[i]));
      uint32_t code;
      float s;
      block_scale(a, EMAX, code, s);
      atom[sf_in_atom(4 * lane + c, w)] = static_cast<uint8_t>(code);
      uint32_t c4[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        c4[i] = codes4<FMT>(x[4 * i] * s, x[4 * i + 1] * s, x[4 * i + 2] * s, x[4 * i + 3] * s);
      constexpr int BITS = (FMT == FMT_INT2) ? 2 : (FMT == FMT_E2M1 || FMT == FMT_INT4) ? 4 : 8;
      if (BITS == 8) {
        // the lanes write 32 different rows: one 32-byte store per lane
        // fills a whole L2 sector (the plane is 32-byte aligned unless the
        // caller placed it otherwise)
        uint8_t* dst = data + (n + c) * K + kb;
        if ((reinterpret_cast<uintptr_t>(dst) & 31u) == 0) {
          st_global_v8(dst, c4);
        } else {
          uint4* d4 = reinterpret_cast<uint4*>(dst);
          d4[0] = make_uint4(c4[0], c4[1], c4[2], c4[3]);
          d4[1] = make_uint4(c4[4], c4[5], c4[6], c4[7]);
        }
      } else if (BITS == 4) {
        *reinterpret_cast<uint4*>(data + ((n + c) * K + kb) / 2) =
            make_uint4(c4[0] | (c4[1] << 16), c4[2] | (c4[3] << 16), c4[4] | (c4[5] << 16),
                       c4[6] | (c4[7] << 16));
      } else {
        *reinterpret_cast<uint2*>(data + ((n + c) * K + kb) / 4) =
            make_uint2(c4[0] | (c4[1] << 8) | (c4[2] << 16) | (c4[3] << 24),
                       c4[4] | (c4[5] << 8) | (c4[6] << 16) | (c4[7] << 24));
      }
    }
  }
  __syncthreads();
  if (threadIdx.x < SF_ATOM_BYTES / 16) {
    uint4* dst = reinterpret_cast<uint4*>(sf + (rg * k_atoms + kc) * SF_ATOM_BYTES);
    dst[threadIdx.x] = reinterpret_cast<const uint4*>(atom)[threadIdx.x];
  }
}

template <int FMT>
cudaError_t launch_fmt(const float* src, int64_t ld, int k_strided, int64_t outer,
                       int64_t K, uint8_t* data, uint8_t* sf, cudaStream_t st) {
  const int64_t ra = sf_row_atoms(outer), ka = sf_k_atoms(K);
  if (!k_strided) {
    dim3 grid(static_cast<unsigned>(ka), static_cast<unsigned>(ra));
    quantize_kcontig<FMT><<<grid, QT_THREADS, 0, st>>>(src, ld, outer, K, data, sf);
  } else {
    dim3 grid(static_cast<unsigned>(ra), static_cast<unsigned>(ka));
    quantize_kstrided<FMT><<<grid, 128, 0, st>>>(src, ld, outer, K, data, sf);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quantize(const float* src, int64_t ld, int k_strided, int fmt,
                            int64_t outer, int64_t K, void* data, uint8_t* scales,
                            cudaStream_t st) {
  if (outer == 0 || K == 0) return cudaSuccess;
  uint8_t* d = static_cast<uint8_t*>(data);
  switch (fmt) {
    case FMT_E4M3: return launch_fmt<FMT_E4M3>(src, ld, k_strided, outer, K, d, scales, st);
    case FMT_E5M2: return launch_fmt<FMT_E5M2>(src, ld, k_strided, outer, K, d, scales, st);
    case FMT_INT8: return launch_fmt<FMT_INT8>(src, ld, k_strided, outer, K, d, scales, st);
    case FMT_INT4: return launch_fmt<FMT_INT4>(src, ld, k_strided, outer, K, d, scales, st);
    case FMT_INT2: return launch_fmt<FMT_INT2>(src, ld, k_strided, outer, K, d, scales, st);
    default: return launch_fmt<FMT_E2M1>(src, ld, k_strided, outer, K, d, scales, st);
  }
}

// ---------------------------------------------------------------------------
// Small utility kernels that share this translation unit.

namespace {

__global__ void zero_fill_kernel(uint8_t* C, int64_t rows, int64_t row_bytes,
                                 int64_t ld_bytes) {
  const int64_t total = rows * row_bytes;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / row_bytes, c = i - r * row_bytes;
    C[r * ld_bytes + c] = 0;
  }
}

// Waits on an mbarrier that nothing arrives at; the bound always runs out.
__global__ void selftest_timeout_kernel(long long limit) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const long long t0 = clock64();
    bool done = false;
    while (!done) {
      done = mbar_try_wait(b, 0);
      if (clock64() - t0 > limit) break;
    }
    if (!done) atomicOr(&g_status_quantize, STATUS_TIMEOUT | 0xEEu);
  }
}

}  // namespace

cudaError_t launch_zero_fill(void* C, int64_t rows, int64_t cols, int64_t ldc,
                             int elem_bytes, cudaStream_t st) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  const int64_t total = rows * cols * elem_bytes;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  zero_fill_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(
      static_cast<uint8_t*>(C), rows, cols * elem_bytes, ldc * elem_bytes);
  return cudaGetLastError();
}

cudaError_t launch_selftest_timeout(long long limit_cycles, cudaStream_t st) {
  selftest_timeout_kernel<<<1, 32, 0, st>>>(limit_cycles);
  return cudaGetLastError();
}

unsigned fetch_and_clear_status_quantize(cudaError_t* err) {
  unsigned v = 0, z = 0;
  *err = cudaMemcpyFromSymbol(&v, g_status_quantize, sizeof(v));
  if (*err == cudaSuccess) *err = cudaMemcpyToSymbol(g_status_quantize, &z, sizeof(z));
  return v;
}

}  // namespace mxk
