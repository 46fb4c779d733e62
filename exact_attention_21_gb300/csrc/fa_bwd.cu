// Backward kernels (placeholder until the tcgen05 backward lands).
#include "fa_common.cuh"

namespace fa {
int launch_bwd(int, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
               const BwdParams&, cudaStream_t) {
  return -1;
}
}  // namespace fa
