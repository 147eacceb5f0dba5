// gemm_mxf8.cu -- the GEMM kernel (gemm_kernel.cuh) instantiated for
// kind::mxf8f6f4: E4M3 / E5M2 operands, and pairs of an 8-bit format with
// E2M1 (unpacked by TMA), for every configuration and output form.
#include "gemm_kernel.cuh"

namespace mxk {
namespace gemm {

cudaError_t launch_mxf8(int cg, int tbn, int out, const Launch& l) {
  switch (out) {
    case OUT_BF16:
      return launch_cfg<KIND_MXF8, OUT_BF16>(cg, tbn, l);
    case OUT_MX8:
      return launch_cfg<KIND_MXF8, OUT_MX8>(cg, tbn, l);
    case OUT_MX4:
      return launch_cfg<KIND_MXF8, OUT_MX4>(cg, tbn, l);
    default:
      return launch_cfg<KIND_MXF8, OUT_F32>(cg, tbn, l);
  }
}

unsigned fetch_and_clear_status_mxf8(cudaError_t* err) { return fetch_and_clear_status_tu(err); }

}  // namespace gemm
}  // namespace mxk
