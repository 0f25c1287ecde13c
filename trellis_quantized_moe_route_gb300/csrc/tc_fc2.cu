// Tensor-core kernel variants of one projection: FC2 (256 output columns per unit, 128 when H % 256 != 0).
// One translation unit per projection, so that the variants compile in
// parallel; the launcher with the tensor maps is in tc.cu.
#include "tc_kernel.cuh"

namespace tmoe {

cudaError_t launch_tc_fc2(const TcArgs& args, int uniform_k, int max_blocks, cudaStream_t st) {
  return (args.f.H % 256 == 0) ? tc_pick<2, 256, false>(args, uniform_k, max_blocks, st)
                               : tc_pick<2, 128, false>(args, uniform_k, max_blocks, st);
}

}  // namespace tmoe
