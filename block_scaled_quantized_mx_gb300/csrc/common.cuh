// common.cuh -- definitions shared by the library's kernels and host code:
// the scale-plane layout (one definition, used by the quantizer that writes it
// and by the GEMM loaders that read it), format codes and launch entry points.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace mxk {

enum Format : int {
  FMT_E4M3 = 1, FMT_E2M1 = 2, FMT_E5M2 = 3,
  FMT_INT8 = 4, FMT_INT4 = 5, FMT_INT2 = 6   // two's-complement integer codes
};

// Bits of one element code.
__host__ __device__ __forceinline__ int code_bits(int fmt) {
  return fmt == FMT_INT2 ? 2 : (fmt == FMT_E2M1 || fmt == FMT_INT4) ? 4 : 8;
}
enum DType : int { DT_F32 = 0, DT_BF16 = 1, DT_F16 = 2 };
enum Act : int { ACT_NONE = 0, ACT_GELU = 1, ACT_GELU_TANH = 2 };

// What the GEMM epilogue does between the fp32 accumulator and the store of
// C: add bias[j] to column j (bias may be null), apply the activation, and
// store C plain (q_fmt = 0: fp32 or bf16 by c_dtype) or as an MX tensor of
// element format q_fmt whose blocks of 32 run along the columns of C (C is
// then the data plane and q_sf its scale plane).
struct Epilogue {
  const float* bias = nullptr;
  int act = ACT_NONE;
  int q_fmt = 0;
  uint8_t* q_sf = nullptr;
};

// Status word bits recorded by kernels (the host maps any non-zero word to
// MX_ERR_TIMEOUT; the low byte says which wait gave up).
constexpr unsigned STATUS_TIMEOUT = 0x100u;

// ---------------------------------------------------------------- scale plane
// Scales are grouped in atoms of 128 rows x 4 blocks (128 K elements): 512
// contiguous bytes, the byte of (row r, block j) at 16*(r%32) + 4*((r/32)%4)
// + j%4.  This is the arrangement in which one 32-lane x 16-byte tensor-memory
// copy, replicated to the four lane quarters, hands each accumulator row its
// four scales.  Atoms are ordered K-chunk fastest.
constexpr int SF_ATOM_ROWS = 128;
constexpr int SF_ATOM_BLOCKS = 4;
constexpr int SF_ATOM_BYTES = 512;

__host__ __device__ __forceinline__ int64_t sf_k_atoms(int64_t K) {
  return (K + 127) / 128;
}
__host__ __device__ __forceinline__ int64_t sf_row_atoms(int64_t outer) {
  return (outer + 127) / 128;
}
__host__ __device__ __forceinline__ int sf_in_atom(int r, int j) {
  return (r & 31) * 16 + ((r >> 5) & 3) * 4 + (j & 3);
}
__host__ __device__ __forceinline__ int64_t sf_offset(int64_t r, int64_t j,
                                                      int64_t k_atoms) {
  return ((r >> 7) * k_atoms + (j >> 2)) * SF_ATOM_BYTES +
         sf_in_atom(static_cast<int>(r & 127), static_cast<int>(j & 3));
}

// ---------------------------------------------------------------- launches
cudaError_t launch_quantize(const float* src, int64_t ld, int k_strided, int fmt,
                            int64_t outer, int64_t K, void* data, uint8_t* scales,
                            cudaStream_t st);

// mx GEMM: A data outer=M, B data outer=N, both K-major; C row-major.
// ws: workspace for the fp32 partials of K-split tiles (nullptr, or fewer
// than gemm_workspace_bytes() bytes: no splitting).
// fmt_a / fmt_b: the element formats of A and B (FMT_*).
cudaError_t launch_gemm_mx(int fmt_a, int fmt_b, const void* a_data, const uint8_t* a_sf,
                           const void* b_data, const uint8_t* b_sf, void* C,
                           int c_dtype, int64_t ldc, int64_t M, int64_t N,
                           int64_t K, void* ws, size_t ws_bytes, const Epilogue& epi,
                           cudaStream_t st);

cudaError_t launch_gemm_f16(int ab_dtype, const void* A, const void* B, float* C,
                            int64_t M, int64_t N, int64_t K, int64_t lda,
                            int64_t ldb, int64_t ldc, void* ws, size_t ws_bytes,
                            const Epilogue& epi, cudaStream_t st);

// C = A * dequant(B)^T for a row-major 16-bit A (a_dtype DT_F16 / DT_BF16,
// M x K, leading dimension lda) and an MX tensor B of any format (N x K);
// K a multiple of 64.  With a workspace of at least dequant_workspace_bytes
// the tiles' K ranges are split over otherwise idle SMs (plain outputs).
cudaError_t launch_gemm_dequant(int a_dtype, const void* A, int64_t lda, int fmt_b,
                                const void* b_data, const uint8_t* b_sf, void* C, int c_dtype,
                                int64_t ldc, int64_t M, int64_t N, int64_t K, const Epilogue& epi,
                                void* ws, size_t ws_bytes, cudaStream_t st);
size_t dequant_workspace_bytes(int64_t M, int64_t N, int64_t K);

// The decode-shaped dequantizing GEMM (dqdec.cu): M <= 128 tokens, a plain or
// bias / activation output; K a multiple of 64.  Its K split stays inside
// thread-block clusters: no workspace (dequant_decode_workspace_bytes is 0).
bool dequant_decode_applies(int64_t M, const Epilogue& epi);
size_t dequant_decode_workspace_bytes(int64_t M, int64_t N, int64_t K);
cudaError_t launch_gemm_dequant_decode(int a_dtype, const void* A, int64_t lda, int fmt_b,
                                       const void* b_data, const uint8_t* b_sf, void* C,
                                       int c_dtype, int64_t ldc, int64_t M, int64_t N, int64_t K,
                                       const Epilogue& epi, cudaStream_t st);
unsigned fetch_and_clear_status_dqd(cudaError_t* err);

// A single row of a bf16 A and 4- or 2-bit weights (dqgemv.cu): CUDA-core
// dot products streaming B once, for a plain or bias / activation output; K
// a multiple of 64.  No workspace, no waits.
bool dequant_gemv_applies(int64_t M, int a_dtype, int fmt_b, const Epilogue& epi);
cudaError_t launch_gemm_dequant_gemv(const void* A, int fmt_b, const void* b_data,
                                     const uint8_t* b_sf, void* C, int c_dtype, int64_t N,
                                     int64_t K, const Epilogue& epi, cudaStream_t st);

// O = softmax(Q K^T * scale) V for BH heads: Q BH x Lq x d, K and V
// BH x Lk x d, row-major, dtype DT_F16 / DT_BF16; d 64 or 128; O BH x Lq x d
// of o_dtype (DT_F32, DT_BF16 or DT_F16).
// ws / ws_bytes: scratch for the parts of split units (nullptr: no split).
cudaError_t launch_attention(int dtype, const void* Q, const void* K, const void* V, void* O,
                             int o_dtype, int64_t BH, int64_t Lq, int64_t Lk, int64_t d,
                             float scale, void* ws, size_t ws_bytes, cudaStream_t st);
size_t attention_workspace_bytes(int64_t BH, int64_t Lq, int64_t Lk, int64_t d);

// Workspace bytes the K-split needs (0: the problem is not split).
// kind: FMT_E4M3 / FMT_E5M2 (the FP8-rate kernel, also for mixed formats),
// FMT_E2M1 (both operands E2M1), or 0 for the 16-bit GEMM.
size_t gemm_workspace_bytes(int kind, int64_t M, int64_t N, int64_t K);

// Tile width of the GEMMs' configuration: 0 picks it per shape, 128 or 256
// fixes it (128 only for plain or bias/activation outputs).
void gemm_force_tile_width(int tbn);

cudaError_t launch_zero_fill(void* C, int64_t rows, int64_t cols, int64_t ldc,
                             int elem_bytes, cudaStream_t st);

cudaError_t launch_selftest_timeout(long long limit_cycles, cudaStream_t st);

// Read and clear the device status word of each translation unit.
unsigned fetch_and_clear_status_quantize(cudaError_t* err);
unsigned fetch_and_clear_status_gemm(cudaError_t* err);
unsigned fetch_and_clear_status_dq(cudaError_t* err);
unsigned fetch_and_clear_status_attn(cudaError_t* err);

}  // namespace mxk
