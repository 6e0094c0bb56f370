// prefill_cluster.cu -- thread-block-cluster variant of the tensor-core prefill (not yet enabled:
// every workload runs the fused kernel of prefill_tc.cu).
#include "tc_common.cuh"

namespace gdr {
namespace tc {

int cluster_size_for(const gdr_shape&) { return 1; }

cudaError_t launch_prefill_cluster(const gdr_shape&, const PrefillArgs&, const TcMaps&, int,
                                   cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace tc
}  // namespace gdr
