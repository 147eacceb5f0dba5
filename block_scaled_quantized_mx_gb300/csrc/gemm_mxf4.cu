// gemm_mxf4.cu -- the GEMM kernel (gemm_kernel.cuh) instantiated for
// kind::mxf4: packed E2M1 on both sides, for every configuration and output
// form.
#include "gemm_kernel.cuh"

namespace mxk {
namespace gemm {

cudaError_t launch_mxf4(int cg, int tbn, int out, const Launch& l) {
  switch (out) {
    case OUT_BF16:
      return launch_cfg<KIND_MXF4, OUT_BF16>(cg, tbn, l);
    case OUT_MX8:
      return launch_cfg<KIND_MXF4, OUT_MX8>(cg, tbn, l);
    case OUT_MX4:
      return launch_cfg<KIND_MXF4, OUT_MX4>(cg, tbn, l);
    default:
      return launch_cfg<KIND_MXF4, OUT_F32>(cg, tbn, l);
  }
}

unsigned fetch_and_clear_status_mxf4(cudaError_t* err) { return fetch_and_clear_status_tu(err); }

}  // namespace gemm
}  // namespace mxk
