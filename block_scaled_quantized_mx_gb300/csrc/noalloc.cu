// noalloc.cu -- mx_gemm_splitk_noalloc: the K-split MX GEMM for callers that
// cannot allocate device memory.
//
// mx_gemm_splitk needs a scratch buffer for the fp32 partial tiles of the
// split.  Some callers cannot hand one over: code that owns only the operand
// and result pointers (a plugin or operator interface with no workspace
// argument), and processes whose device memory is all reserved up front by a
// framework's caching allocator or by a fixed memory budget, where a call to
// cudaMalloc would fail or would bypass that allocator's accounting.  This
// entry point takes its scratch from a fixed array in the library's own
// device memory instead, so it allocates nothing.
//
// The array lives as long as the process: every GPU on which this module has
// been loaded (at the latest on the first call there) keeps its 24 MiB until
// exit.  All calls share it.
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "mx.h"

namespace {

// 24 MiB.  The split never needs more than one fp32 partial of 256 x 128
// per cluster of two SMs, plus its counters (76 x 128 KiB ~ 10 MiB on a
// 152-SM GB300); a problem that would need more is rejected with
// MX_ERR_SHAPE.
constexpr size_t kScratchBytes = size_t{24} << 20;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;

// The cached device address of g_scratch, per device ordinal, with the
// unique id (cuCtxGetId) of the context it was looked up in.  A device reset
// or a new primary context reloads the module, possibly at another address,
// and comes with a new id, so the address is looked up again.
struct Slot {
  unsigned long long ctx = 0;
  void* ptr = nullptr;
};
Slot g_slot[64];

// The unique id of the context current on this thread, through the driver
// entry points; false when there is none yet (or no driver support).
bool current_context_id(unsigned long long* id) {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (!get_current) {
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return false;
    get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
  }
  if (!get_id) {
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return false;
    get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
  }
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

// The device address of g_scratch on the current device.  The host-side name
// g_scratch is only a stand-in and must never reach a kernel; the address is
// looked up with the device current (cudaGetSymbolAddress) the first time a
// context of that device calls, and cached for that context.
mx_status scratch_on_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MX_ERR_CUDA;
  if (dev < 0 || dev >= 64) return MX_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  unsigned long long ctx = 0;
  const bool have_id = current_context_id(&ctx);
  Slot& slot = g_slot[dev];
  if (have_id && slot.ptr != nullptr && slot.ctx == ctx) {
    *out = slot.ptr;
    return MX_OK;
  }
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
  if (e != cudaSuccess || p == nullptr) return MX_ERR_CUDA;
  // the lookup initialises the device's context if no call had yet
  if (have_id || current_context_id(&ctx)) {
    slot.ctx = ctx;
    slot.ptr = p;
  } else {
    slot = Slot{};   // no id to key the cache on: look up again next time
  }
  *out = p;
  return MX_OK;
}

}  // namespace

#pragma GCC visibility push(default)
extern "C" {

mx_status mx_gemm_splitk_noalloc(const mx_tensor* A, const mx_tensor* B, void* C,
                                 int32_t c_dtype, int64_t ldc, void* stream) {
  if (!A || !B) return MX_ERR_INVALID_ARG;
  if (A->K == B->K && A->outer > 0 && B->outer > 0 && A->K > 0) {
    // the FP8-rate kernel unless both operands are E2M1
    const int32_t kind = (A->fmt == MX_FMT_E2M1 && B->fmt == MX_FMT_E2M1) ? MX_FMT_E2M1
                                                                          : MX_FMT_E4M3;
    const size_t need = mx_gemm_workspace_bytes(kind, A->outer, B->outer, A->K);
    if (need > kScratchBytes) return MX_ERR_SHAPE;
  }
  void* scratch = nullptr;
  const mx_status s = scratch_on_current_device(&scratch);
  if (s != MX_OK) return s;
  // The partial tiles are written in full before they are read, within this
  // call, and the split's counters count only this launch's tagged arrivals
  // (and are left at zero by every completed launch), so nothing in the
  // scratch has to start at zero.
  return mx_gemm_splitk(A, B, C, c_dtype, ldc, scratch, kScratchBytes, stream);
}

}  // extern "C"
#pragma GCC visibility pop
