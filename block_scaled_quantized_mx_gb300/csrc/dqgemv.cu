// dqgemv.cu -- gemm_dequant for a single row of a bf16 A (decoding one
// token) and 4- or 2-bit weights: c = a * dequant(B)^T on the CUDA cores,
// streaming B's codes once.
//
// What is computed follows WWDC26 session 330, "Quantized matrix
// multiplication" and "Quantized data types": each 32-element block of B's
// codes times its scale 2^(c - 127), rounded once to bf16 (A's type, as in
// the tensor-core kernels), multiplied by a and summed over K in fp32.  With
// one token each weight element is used once, so the product is a stream of
// B from HBM; the tensor-core decode kernel (dqdec.cu) pads the token to 64
// rows and spends its time converting codes into tensor memory, the wrong
// trade for so little arithmetic.
//
// Layout: a CTA of eight warps owns DQV_ROWS weight rows (columns of c); its
// warps take the 1024-K chunks of K in turn, each lane one whole 32-element
// block of a chunk (one scale per lane and row).  A lane loads its 32 values
// of a once per chunk (64 bytes, from L1 / L2: a is small) and reuses them
// for every row; every code load of a step (one 16-byte block of 4-bit codes
// per row) is issued before any arithmetic, so that a CTA's whole share of
// the stream is in flight at once.  The lane sums, the warp sums (a fixed
// butterfly) and the warps' sums (in warp order) give the same bits every
// run.
#include <cstdint>

#include "common.cuh"
#include "dq_common.cuh"
#include "gemm_common.cuh"
#include "ptx.cuh"

namespace mxk {
namespace {

constexpr int DQV_WARPS = 8;
constexpr int DQV_ROWS = 8;        // weight rows per CTA
constexpr int DQV_CHUNK = 1024;    // K per warp step: 32 lanes x one block

struct GemvArgs {
  const uint16_t* a;      // bf16, K values
  const uint8_t* codes;   // N x K codes, rows back to back
  const uint8_t* sf;      // scale plane, tensor-core atom layout
  void* C;
  int N, K;
  EpiArgs epi;
};

template <int FMT, int OUT>
__global__ void __launch_bounds__(DQV_WARPS * 32, 2) dqgemv_kernel(const GemvArgs g) {
  constexpr int BITS = (FMT == FMT_INT2) ? 2 : 4;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * DQV_ROWS;
  const int64_t row_bytes = static_cast<int64_t>(g.K) * BITS / 8;
  const int64_t k_atoms = sf_k_atoms(g.K);
  const int nchunks = (g.K + DQV_CHUNK - 1) / DQV_CHUNK;
  const int rows = min(DQV_ROWS, g.N - n0);

  float acc[DQV_ROWS];
#pragma unroll
  for (int r = 0; r < DQV_ROWS; ++r) acc[r] = 0.0f;

  for (int c = warp; c < nchunks; c += DQV_WARPS) {
    const int k = c * DQV_CHUNK + 32 * lane;   // the lane's block; K % 32 == 0
    if (k < g.K) {
      // every load of the step first: the rows' code blocks and scales, a
      // (loads past N read the last row, which is never stored)
      uint32_t w[DQV_ROWS][8];
      uint32_t sc[DQV_ROWS];
#pragma unroll
      for (int r = 0; r < DQV_ROWS; ++r) {
        const int n = min(n0 + r, g.N - 1);
        dq::load_block_codes<FMT>(g.codes + n * row_bytes + static_cast<int64_t>(k) * BITS / 8,
                                  w[r]);
        sc[r] = __ldg(g.sf + sf_offset(n, k >> 5, k_atoms));
      }
      uint4 av[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = __ldg(reinterpret_cast<const uint4*>(g.a + k) + i);
      float a[32];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t v[4] = {av[i].x, av[i].y, av[i].z, av[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          a[8 * i + 2 * j] = __uint_as_float(v[j] << 16);
          a[8 * i + 2 * j + 1] = __uint_as_float(v[j] & 0xFFFF0000u);
        }
      }
#pragma unroll
      for (int r = 0; r < DQV_ROWS; ++r) {
        // the block as 16 bf16 pairs (element 2 i in the low half of o[i]),
        // exactly the other kernels' dequantized operand
        uint32_t o[16];
        dq::dq_block_regs<FMT>(w[r], sc[r], true, o);
        float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          s0 = fmaf(a[2 * i], __uint_as_float(o[i] << 16), s0);
          s1 = fmaf(a[2 * i + 1], __uint_as_float(o[i] & 0xFFFF0000u), s1);
        }
        acc[r] += s0 + s1;
      }
    }
  }

  // over the lanes (a fixed butterfly), then over the warps in order
  __shared__ float red[DQV_WARPS][DQV_ROWS];
#pragma unroll
  for (int r = 0; r < DQV_ROWS; ++r) {
    float v = acc[r];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    if (lane == 0) red[warp][r] = v;
  }
  __syncthreads();
  const int r = threadIdx.x;
  if (r < rows) {
    const int n = n0 + r;
    float v = red[0][r];
#pragma unroll
    for (int w = 1; w < DQV_WARPS; ++w) v += red[w][r];
    if (g.epi.bias != nullptr) v += __ldg(g.epi.bias + n);
    if (g.epi.act == ACT_GELU) v = gelu_exact(v);
    else if (g.epi.act == ACT_GELU_TANH) v = gelu_tanh(v);
    if (OUT == OUT_BF16)
      reinterpret_cast<uint16_t*>(g.C)[n] = static_cast<uint16_t>(cvt_bf16x2(v, 0.0f) & 0xFFFFu);
    else
      reinterpret_cast<float*>(g.C)[n] = v;
  }
}

template <int FMT>
cudaError_t dqv_run(const GemvArgs& g, int out_bf16, cudaStream_t st) {
  const dim3 grid(static_cast<unsigned>((g.N + DQV_ROWS - 1) / DQV_ROWS));
  if (out_bf16)
    dqgemv_kernel<FMT, OUT_BF16><<<grid, DQV_WARPS * 32, 0, st>>>(g);
  else
    dqgemv_kernel<FMT, OUT_F32><<<grid, DQV_WARPS * 32, 0, st>>>(g);
  return cudaGetLastError();
}

}  // namespace

bool dequant_gemv_applies(int64_t M, int a_dtype, int fmt_b, const Epilogue& epi) {
  return M == 1 && a_dtype == DT_BF16 && epi.q_fmt == 0 &&
         (fmt_b == FMT_INT4 || fmt_b == FMT_INT2 || fmt_b == FMT_E2M1);
}

cudaError_t launch_gemm_dequant_gemv(const void* A, int fmt_b, const void* b_data,
                                     const uint8_t* b_sf, void* C, int c_dtype, int64_t N,
                                     int64_t K, const Epilogue& epi, cudaStream_t st) {
  if (K % 64 != 0 || N >= (int64_t{1} << 31) || K >= (int64_t{1} << 31))
    return cudaErrorInvalidValue;
  GemvArgs g{};
  g.a = static_cast<const uint16_t*>(A);
  g.codes = static_cast<const uint8_t*>(b_data);
  g.sf = b_sf;
  g.C = C;
  g.N = static_cast<int>(N);
  g.K = static_cast<int>(K);
  g.epi.bias = epi.bias;
  g.epi.act = epi.act;
  const int ob = (c_dtype == DT_BF16) ? 1 : 0;
  switch (fmt_b) {
    case FMT_INT4: return dqv_run<FMT_INT4>(g, ob, st);
    case FMT_INT2: return dqv_run<FMT_INT2>(g, ob, st);
    case FMT_E2M1: return dqv_run<FMT_E2M1>(g, ob, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mxk
