// The decode kernel (gemm_dec.cuh) instantiated for bf16 activations, scales and outputs: one
// translation unit per value type, so that the two build in parallel.
#include "gemm_dec.cuh"

namespace w4 {
namespace detail {

cudaError_t launch_gemm_dec_bf16(const DecParams &p, int nb8, int clusters, int cluster, cudaStream_t stream) {
  return launch_dec_dt<kDtypeBf16>(p, nb8, clusters, cluster, stream);
}

}  // namespace detail
}  // namespace w4
