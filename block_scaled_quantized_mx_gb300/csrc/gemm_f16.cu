// gemm_f16.cu -- the GEMM kernel (gemm_kernel.cuh) instantiated for
// kind::f16: fp16 or bf16 operands, fp32 C, for every configuration.
#include "gemm_kernel.cuh"

namespace mxk {
namespace gemm {

cudaError_t launch_f16(int kind, int cg, int tbn, const Launch& l) {
  if (kind == KIND_BF16) return launch_cfg<KIND_BF16, OUT_F32>(cg, tbn, l);
  return launch_cfg<KIND_F16, OUT_F32>(cg, tbn, l);
}

unsigned fetch_and_clear_status_f16(cudaError_t* err) { return fetch_and_clear_status_tu(err); }

}  // namespace gemm
}  // namespace mxk
