// gma_tc.cu -- bf16 I/O path.  Placeholder that routes to the CUDA-core kernels until the
// tcgen05 kernels land.
#include "gma_internal.h"

namespace gma {

TcPlan tc_plan(const gma_problem_t& p, gma_op_t op) {
  TcPlan t{};
  t.total = simt_plan(p, op).total;
  return t;
}

gma_status_t tc_run(const gma_problem_t& p, gma_op_t op, const void* Q, const void* K, const void* V,
                    const float* mu, const float* sigma2, const float* log_pi, void* out, void* ws,
                    cudaStream_t stream) {
  return simt_run(p, op, Q, K, V, mu, sigma2, log_pi, out, ws, stream);
}

bool tc_available() { return false; }

}  // namespace gma
