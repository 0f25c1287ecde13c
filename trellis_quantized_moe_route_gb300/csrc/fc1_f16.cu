// FC1 instantiations, f16 operands (see fc.cuh).
#include "fc.cuh"

namespace tmoe {

cudaError_t launch_fc1_f16(const FcArgs& a, int bi, int bn, int uniform_k, int max_blocks, cudaStream_t st) {
#define TM_FC1(KB, BI, BN) \
  if (uniform_k == (KB == 0 ? uniform_k : KB) && bi == BI && bn == BN) \
    return launch_fc_t<false, 1, KB, 2 * BI, BN>(a, max_blocks, st);
  if (uniform_k == 4) {
    TM_FC1(4, 128, 64) TM_FC1(4, 128, 8) TM_FC1(4, 64, 64) TM_FC1(4, 64, 8)
  }
  TM_FC1(0, 128, 64) TM_FC1(0, 128, 8) TM_FC1(0, 64, 64) TM_FC1(0, 64, 8)
#undef TM_FC1
  return cudaErrorInvalidValue;
}

}  // namespace tmoe
