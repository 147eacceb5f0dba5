// api.cu -- the C ABI of include/mx.h: argument, shape and alignment checks
// on the host, then one asynchronous launch on the caller's stream.
//
// The pages' interface (WWDC26 session 330, 3:53 / 4:48 listings): a quantized
// tensor is one object carrying a data plane and a scale plane, and creating
// one reports failure through a status rather than by crashing; the matmul
// takes two such tensors and a plain output with no transposes.  Here that is
// the mx_tensor struct plus mx_status codes.
#include <cstdint>
#include <cstring>

#include "mx.h"
#include "common.cuh"

namespace {

constexpr int64_t kMaxDim = (int64_t{1} << 31) - 1;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The library ships sm_103a code only: require compute capability 10.3.
mx_status check_device() {
  static int ok_cache[64] = {};   // 0 unknown, 1 ok, 2 unsupported
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MX_ERR_CUDA;
  if (dev < 64 && ok_cache[dev]) return ok_cache[dev] == 1 ? MX_OK : MX_ERR_UNSUPPORTED;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return MX_ERR_CUDA;
  const bool ok = (major == 10 && minor == 3);
  if (dev < 64) ok_cache[dev] = ok ? 1 : 2;
  return ok ? MX_OK : MX_ERR_UNSUPPORTED;
}

mx_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MX_OK : MX_ERR_CUDA; }

bool is_int_fmt(int32_t fmt) {
  return fmt == MX_FMT_INT8 || fmt == MX_FMT_INT4 || fmt == MX_FMT_INT2;
}

// A and B of one product: equal K; an E2M1 operand beside an 8-bit one is
// unpacked by TMA, which needs K % 128 == 0 and a 32-byte aligned plane.
mx_status check_pair(const mx_tensor* A, const mx_tensor* B) {
  // the tensor cores have no block-scaled integer kind: integer tensors are
  // B operands of gemm_dequant only
  if (is_int_fmt(A->fmt) || is_int_fmt(B->fmt)) return MX_ERR_INVALID_ARG;
  if (A->K != B->K) return MX_ERR_SHAPE;
  if ((A->fmt == MX_FMT_E2M1) == (B->fmt == MX_FMT_E2M1)) return MX_OK;
  if (A->outer == 0 || B->outer == 0 || A->K == 0) return MX_OK;
  if (A->K % 128) return MX_ERR_SHAPE;
  const mx_tensor* f4 = (A->fmt == MX_FMT_E2M1) ? A : B;
  if (reinterpret_cast<uintptr_t>(f4->data) % 32) return MX_ERR_ALIGN;
  return MX_OK;
}

mx_status check_tensor(const mx_tensor* t) {
  if (!t) return MX_ERR_INVALID_ARG;
  if (t->fmt < MX_FMT_E4M3 || t->fmt > MX_FMT_INT2) return MX_ERR_INVALID_ARG;
  if (t->outer < 0 || t->K < 0 || t->outer > kMaxDim || t->K > kMaxDim) return MX_ERR_SHAPE;
  if (t->K % 32) return MX_ERR_SHAPE;
  if (t->outer > 0 && t->K > 0) {
    if (!t->data || !t->scales) return MX_ERR_INVALID_ARG;
    if (!aligned16(t->data) || !aligned16(t->scales)) return MX_ERR_ALIGN;
  }
  return MX_OK;
}

// The optional epilogue argument: NULL means none.  The bias must be
// 16-byte aligned (it is read as float4).
mx_status epilogue_from(const mx_epilogue* epi, mxk::Epilogue* out) {
  *out = mxk::Epilogue{};
  if (!epi) return MX_OK;
  if (epi->act != MX_ACT_NONE && epi->act != MX_ACT_GELU && epi->act != MX_ACT_GELU_TANH)
    return MX_ERR_INVALID_ARG;
  if (epi->bias && !aligned16(epi->bias)) return MX_ERR_ALIGN;
  out->bias = epi->bias;
  out->act = epi->act;
  return MX_OK;
}

bool has_work(const mxk::Epilogue& e) { return e.bias != nullptr || e.act != MX_ACT_NONE; }

// mx_gemm, mx_gemm_splitk and mx_gemm_fused: checks, then one launch.
mx_status mx_product(const mx_tensor* A, const mx_tensor* B, const mx_epilogue* epi, void* C,
                     int32_t c_dtype, int64_t ldc, void* ws, size_t ws_bytes, void* stream) {
  mx_status s;
  if ((s = check_tensor(A)) != MX_OK) return s;
  if ((s = check_tensor(B)) != MX_OK) return s;
  if ((s = check_pair(A, B)) != MX_OK) return s;
  if (c_dtype != MX_DT_F32 && c_dtype != MX_DT_BF16) return MX_ERR_INVALID_ARG;
  mxk::Epilogue e;
  if ((s = epilogue_from(epi, &e)) != MX_OK) return s;
  const int64_t M = A->outer, N = B->outer, K = A->K;
  if (M == 0 || N == 0) return MX_OK;
  if (!C) return MX_ERR_INVALID_ARG;
  const int64_t eb = (c_dtype == MX_DT_BF16) ? 2 : 4;
  if (ldc < N || (ldc * eb) % 16) return MX_ERR_SHAPE;
  if (!aligned16(C)) return MX_ERR_ALIGN;
  if (K == 0 && has_work(e)) return MX_ERR_SHAPE;
  if ((s = check_device()) != MX_OK) return s;
  return from_cuda(mxk::launch_gemm_mx(A->fmt, B->fmt, A->data, A->scales, B->data, B->scales,
                                       C, c_dtype, ldc, M, N, K, ws, ws_bytes, e,
                                       static_cast<cudaStream_t>(stream)));
}

// gemm_f16, gemm_f16_splitk and gemm_f16_fused.
mx_status f16_product(const void* A, const void* B, const mx_epilogue* epi, float* C,
                      int32_t ab_dtype, int64_t M, int64_t N, int64_t K, int64_t lda,
                      int64_t ldb, int64_t ldc, void* ws, size_t ws_bytes, void* stream) {
  if (ab_dtype != MX_DT_F16 && ab_dtype != MX_DT_BF16) return MX_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
    return MX_ERR_SHAPE;
  mxk::Epilogue e;
  mx_status s = epilogue_from(epi, &e);
  if (s != MX_OK) return s;
  if (M == 0 || N == 0) return MX_OK;
  if (!C) return MX_ERR_INVALID_ARG;
  if (ldc < N || ldc % 4) return MX_ERR_SHAPE;
  if (!aligned16(C)) return MX_ERR_ALIGN;
  if (K > 0) {
    if (!A || !B) return MX_ERR_INVALID_ARG;
    if (lda < K || ldb < N || lda % 8 || ldb % 8) return MX_ERR_SHAPE;
    if (!aligned16(A) || !aligned16(B)) return MX_ERR_ALIGN;
  } else if (has_work(e)) {
    return MX_ERR_SHAPE;
  }
  if ((s = check_device()) != MX_OK) return s;
  return from_cuda(mxk::launch_gemm_f16(ab_dtype, A, B, C, M, N, K, lda, ldb, ldc, ws,
                                        ws_bytes, e, static_cast<cudaStream_t>(stream)));
}

}  // namespace

#pragma GCC visibility push(default)
extern "C" {

size_t mx_data_bytes(int32_t fmt, int64_t outer, int64_t K) {
  if (outer < 0 || K < 0 || K % 32) return 0;
  if (fmt < MX_FMT_E4M3 || fmt > MX_FMT_INT2) return 0;
  return static_cast<size_t>(outer) * static_cast<size_t>(K) *
         static_cast<size_t>(mxk::code_bits(fmt)) / 8;
}

size_t mx_scale_bytes(int64_t outer, int64_t K) {
  if (outer < 0 || K < 0 || K % 32) return 0;
  return static_cast<size_t>(mxk::sf_row_atoms(outer)) *
         static_cast<size_t>(mxk::sf_k_atoms(K)) * mxk::SF_ATOM_BYTES;
}

mx_status mx_quantize(const float* src, int64_t ld, int32_t src_layout, const mx_tensor* out,
                      void* stream) {
  mx_status s = check_tensor(out);
  if (s != MX_OK) return s;
  if (src_layout != MX_SRC_K_CONTIGUOUS && src_layout != MX_SRC_K_STRIDED)
    return MX_ERR_INVALID_ARG;
  if (out->outer == 0 || out->K == 0) return MX_OK;
  if (!src) return MX_ERR_INVALID_ARG;
  const int64_t inner = (src_layout == MX_SRC_K_CONTIGUOUS) ? out->K : out->outer;
  if (ld < inner || ld % 4) return MX_ERR_SHAPE;
  if (!aligned16(src)) return MX_ERR_ALIGN;
  // grid limits: 65535 CTAs along the second grid dimension
  const int64_t ra = mxk::sf_row_atoms(out->outer), ka = mxk::sf_k_atoms(out->K);
  if ((src_layout == MX_SRC_K_CONTIGUOUS ? ra : ka) > 65535) return MX_ERR_SHAPE;
  if ((s = check_device()) != MX_OK) return s;
  return from_cuda(mxk::launch_quantize(src, ld, src_layout == MX_SRC_K_STRIDED, out->fmt,
                                        out->outer, out->K, out->data, out->scales,
                                        static_cast<cudaStream_t>(stream)));
}

mx_status mx_gemm(const mx_tensor* A, const mx_tensor* B, void* C, int32_t c_dtype,
                  int64_t ldc, void* stream) {
  return mx_product(A, B, nullptr, C, c_dtype, ldc, nullptr, 0, stream);
}

size_t mx_gemm_workspace_bytes(int32_t fmt, int64_t M, int64_t N, int64_t K) {
  if (fmt != MX_FMT_E4M3 && fmt != MX_FMT_E5M2 && fmt != MX_FMT_E2M1) return 0;
  if (M <= 0 || N <= 0 || K <= 0 || K % 32 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
    return 0;
  if (check_device() != MX_OK) return 0;
  return mxk::gemm_workspace_bytes(fmt, M, N, K);
}

mx_status mx_gemm_splitk(const mx_tensor* A, const mx_tensor* B, void* C, int32_t c_dtype,
                         int64_t ldc, void* workspace, size_t workspace_bytes, void* stream) {
  if (workspace && !aligned16(workspace)) return MX_ERR_ALIGN;
  return mx_product(A, B, nullptr, C, c_dtype, ldc, workspace, workspace_bytes, stream);
}

mx_status mx_gemm_fused(const mx_tensor* A, const mx_tensor* B, const mx_epilogue* epi,
                        void* C, int32_t c_dtype, int64_t ldc, void* stream) {
  return mx_product(A, B, epi, C, c_dtype, ldc, nullptr, 0, stream);
}

mx_status mx_gemm_fused_quantize(const mx_tensor* A, const mx_tensor* B,
                                 const mx_epilogue* epi, const mx_tensor* C, void* stream) {
  mx_status s;
  if ((s = check_tensor(A)) != MX_OK) return s;
  if ((s = check_tensor(B)) != MX_OK) return s;
  if ((s = check_pair(A, B)) != MX_OK) return s;
  if ((s = check_tensor(C)) != MX_OK) return s;
  if (is_int_fmt(C->fmt)) return MX_ERR_INVALID_ARG;
  const int64_t M = A->outer, N = B->outer, K = A->K;
  if (C->outer != M || C->K != N) return MX_ERR_SHAPE;
  mxk::Epilogue e;
  if ((s = epilogue_from(epi, &e)) != MX_OK) return s;
  if (M == 0 || N == 0) return MX_OK;
  if (K == 0) return MX_ERR_SHAPE;
  if ((s = check_device()) != MX_OK) return s;
  e.q_fmt = C->fmt;
  e.q_sf = C->scales;
  return from_cuda(mxk::launch_gemm_mx(A->fmt, B->fmt, A->data, A->scales, B->data, B->scales,
                                       C->data, MX_DT_F32, N, M, N, K, nullptr, 0, e,
                                       static_cast<cudaStream_t>(stream)));
}

mx_status gemm_dequant_splitk(const void* A, int32_t a_dtype, int64_t M, int64_t lda,
                              const mx_tensor* B, const mx_epilogue* epi, void* C,
                              int32_t c_dtype, int64_t ldc, void* workspace,
                              size_t workspace_bytes, void* stream) {
  mx_status s;
  if (a_dtype != MX_DT_F16 && a_dtype != MX_DT_BF16) return MX_ERR_INVALID_ARG;
  if (c_dtype != MX_DT_F32 && c_dtype != MX_DT_BF16) return MX_ERR_INVALID_ARG;
  if ((s = check_tensor(B)) != MX_OK) return s;
  mxk::Epilogue e;
  if ((s = epilogue_from(epi, &e)) != MX_OK) return s;
  if (M < 0 || M > kMaxDim) return MX_ERR_SHAPE;
  const int64_t N = B->outer, K = B->K;
  if (M == 0 || N == 0) return MX_OK;
  if (K == 0 || K % 64) return MX_ERR_SHAPE;
  if (!A || !C) return MX_ERR_INVALID_ARG;
  if (lda < K || lda % 8) return MX_ERR_SHAPE;
  const int64_t eb = (c_dtype == MX_DT_BF16) ? 2 : 4;
  if (ldc < N || (ldc * eb) % 16) return MX_ERR_SHAPE;
  if (!aligned16(A) || !aligned16(C) || (workspace && !aligned16(workspace)))
    return MX_ERR_ALIGN;
  if ((s = check_device()) != MX_OK) return s;
  return from_cuda(mxk::launch_gemm_dequant(a_dtype, A, lda, B->fmt, B->data, B->scales, C,
                                            c_dtype, ldc, M, N, K, e, workspace,
                                            workspace_bytes,
                                            static_cast<cudaStream_t>(stream)));
}

mx_status gemm_dequant(const void* A, int32_t a_dtype, int64_t M, int64_t lda,
                       const mx_tensor* B, const mx_epilogue* epi, void* C, int32_t c_dtype,
                       int64_t ldc, void* stream) {
  return gemm_dequant_splitk(A, a_dtype, M, lda, B, epi, C, c_dtype, ldc, nullptr, 0, stream);
}

size_t gemm_dequant_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || N <= 0 || K <= 0 || K % 64 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
    return 0;
  if (check_device() != MX_OK) return 0;
  return mxk::dequant_workspace_bytes(M, N, K);
}

namespace {

mx_status attention(const void* Q, const void* K, const void* V, void* O, int32_t dtype,
                    int32_t o_dtype, int64_t BH, int64_t Lq, int64_t Lk, int64_t d, float scale,
                    void* workspace, size_t workspace_bytes, void* stream) {
  if (dtype != MX_DT_F16 && dtype != MX_DT_BF16) return MX_ERR_INVALID_ARG;
  if (o_dtype != MX_DT_F32 && o_dtype != MX_DT_BF16 && o_dtype != MX_DT_F16)
    return MX_ERR_INVALID_ARG;
  if (!(scale == scale) || scale > 3.0e38f || scale < -3.0e38f) return MX_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return MX_ERR_SHAPE;
  if (BH < 0 || Lq < 0 || Lk < 0 || BH > 65535 || Lq > kMaxDim || Lk > kMaxDim)
    return MX_ERR_SHAPE;
  if (BH == 0 || Lq == 0) return MX_OK;
  if (Lk == 0) return MX_ERR_SHAPE;
  if (!Q || !K || !V || !O) return MX_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O)) return MX_ERR_ALIGN;
  mx_status s = check_device();
  if (s != MX_OK) return s;
  if (workspace && !aligned16(workspace)) return MX_ERR_ALIGN;
  return from_cuda(mxk::launch_attention(dtype, Q, K, V, O, o_dtype, BH, Lq, Lk, d, scale,
                                         workspace, workspace_bytes,
                                         static_cast<cudaStream_t>(stream)));
}

}  // namespace

mx_status flash_attention(const void* Q, const void* K, const void* V, void* O, int32_t dtype,
                          int32_t o_dtype, int64_t BH, int64_t Lq, int64_t Lk, int64_t d,
                          float scale, void* stream) {
  return attention(Q, K, V, O, dtype, o_dtype, BH, Lq, Lk, d, scale, nullptr, 0, stream);
}

size_t flash_attention_workspace_bytes(int64_t BH, int64_t Lq, int64_t Lk, int64_t d) {
  if (BH <= 0 || Lq <= 0 || Lk <= 0 || BH > 65535 || Lq > kMaxDim || Lk > kMaxDim) return 0;
  if (d != 64 && d != 128) return 0;
  if (check_device() != MX_OK) return 0;
  return mxk::attention_workspace_bytes(BH, Lq, Lk, d);
}

mx_status flash_attention_splitkv(const void* Q, const void* K, const void* V, void* O,
                                  int32_t dtype, int32_t o_dtype, int64_t BH, int64_t Lq,
                                  int64_t Lk, int64_t d, float scale, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  return attention(Q, K, V, O, dtype, o_dtype, BH, Lq, Lk, d, scale, workspace, workspace_bytes,
                   stream);
}

mx_status gemm_f16(const void* A, const void* B, float* C, int32_t ab_dtype, int64_t M,
                   int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                   void* stream) {
  return f16_product(A, B, nullptr, C, ab_dtype, M, N, K, lda, ldb, ldc, nullptr, 0, stream);
}

size_t gemm_f16_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || N <= 0 || K <= 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return 0;
  if (check_device() != MX_OK) return 0;
  return mxk::gemm_workspace_bytes(0, M, N, K);
}

mx_status gemm_f16_splitk(const void* A, const void* B, float* C, int32_t ab_dtype, int64_t M,
                          int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                          void* workspace, size_t workspace_bytes, void* stream) {
  if (workspace && !aligned16(workspace)) return MX_ERR_ALIGN;
  return f16_product(A, B, nullptr, C, ab_dtype, M, N, K, lda, ldb, ldc, workspace,
                     workspace_bytes, stream);
}

mx_status gemm_f16_fused(const void* A, const void* B, const mx_epilogue* epi, float* C,
                         int32_t ab_dtype, int64_t M, int64_t N, int64_t K, int64_t lda,
                         int64_t ldb, int64_t ldc, void* stream) {
  return f16_product(A, B, epi, C, ab_dtype, M, N, K, lda, ldb, ldc, nullptr, 0, stream);
}

mx_status mx_last_error(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MX_ERR_CUDA;
  cudaError_t e1 = cudaSuccess, e2 = cudaSuccess;
  const unsigned a = mxk::fetch_and_clear_status_quantize(&e1);
  const unsigned b = mxk::fetch_and_clear_status_gemm(&e2);
  cudaError_t e3 = cudaSuccess, e4 = cudaSuccess;
  const unsigned c = mxk::fetch_and_clear_status_dq(&e3);
  const unsigned d = mxk::fetch_and_clear_status_attn(&e4);
  cudaError_t e5 = cudaSuccess;
  const unsigned f = mxk::fetch_and_clear_status_dqd(&e5);
  if (e1 != cudaSuccess || e2 != cudaSuccess || e3 != cudaSuccess || e4 != cudaSuccess ||
      e5 != cudaSuccess)
    return MX_ERR_CUDA;
  if ((a | b | c | d | f) & mxk::STATUS_TIMEOUT) return MX_ERR_TIMEOUT;
  return MX_OK;
}

mx_status mx_selftest_wait_timeout(int64_t limit_cycles, void* stream) {
  if (limit_cycles < 1 || limit_cycles > (int64_t{1} << 40)) return MX_ERR_INVALID_ARG;
  mx_status s = check_device();
  if (s != MX_OK) return s;
  return from_cuda(
      mxk::launch_selftest_timeout(limit_cycles, static_cast<cudaStream_t>(stream)));
}

mx_status mx_scales_to_rowmajor(const uint8_t* tiled, uint8_t* rowmajor, int64_t outer,
                                int64_t K) {
  if (outer < 0 || K < 0 || K % 32) return MX_ERR_SHAPE;
  if ((outer > 0 && K > 0) && (!tiled || !rowmajor)) return MX_ERR_INVALID_ARG;
  const int64_t nb = K / 32, ka = mxk::sf_k_atoms(K);
  for (int64_t r = 0; r < outer; ++r)
    for (int64_t j = 0; j < nb; ++j) rowmajor[r * nb + j] = tiled[mxk::sf_offset(r, j, ka)];
  return MX_OK;
}

const char* mx_status_string(int32_t status) {
  switch (status) {
    case MX_OK: return "MX_OK";
    case MX_ERR_INVALID_ARG: return "MX_ERR_INVALID_ARG";
    case MX_ERR_SHAPE: return "MX_ERR_SHAPE";
    case MX_ERR_ALIGN: return "MX_ERR_ALIGN";
    case MX_ERR_UNSUPPORTED: return "MX_ERR_UNSUPPORTED";
    case MX_ERR_CUDA: return "MX_ERR_CUDA";
    case MX_ERR_TIMEOUT: return "MX_ERR_TIMEOUT";
    default: return "MX_ERR_UNKNOWN";
  }
}

int32_t mx_version(void) { return 200; }

mx_status mx_set_tile_width(int32_t tbn) {
  if (tbn != 0 && tbn != 128 && tbn != 256) return MX_ERR_INVALID_ARG;
  mxk::gemm_force_tile_width(tbn);
  return MX_OK;
}

}  // extern "C"
#pragma GCC visibility pop
