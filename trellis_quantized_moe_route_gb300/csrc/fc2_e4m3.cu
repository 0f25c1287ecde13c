// FC2 instantiations, e4m3 operands (see fc.cuh).
#include "fc.cuh"

namespace tmoe {

cudaError_t launch_fc2_e4m3(const FcArgs& a, int bn, int uniform_k, int max_blocks, cudaStream_t st) {
#define TM_FC2(KB, BN) \
  if (bn == BN) return launch_fc_t<true, 2, KB, 128, BN>(a, max_blocks, st);
  if (uniform_k == 4) {
    TM_FC2(4, 64) TM_FC2(4, 8)
  }
  TM_FC2(0, 64) TM_FC2(0, 8)
#undef TM_FC2
  return cudaErrorInvalidValue;
}

}  // namespace tmoe
