// Tensor-core kernel variants of one projection: FC1 (gate and up rows, N = 2 bi; separate gate / up operands as a variant of their own).
// One translation unit per projection, so that the variants compile in
// parallel; the launcher with the tensor maps is in tc.cu.
#include "tc_kernel.cuh"

namespace tmoe {

cudaError_t launch_tc_fc1(const TcArgs& args, int uniform_k, int max_blocks, cudaStream_t st) {
  const bool split = args.act2 != nullptr;
  if (args.bi == 128)
    return split ? tc_pick<1, 256, true>(args, uniform_k, max_blocks, st)
                 : tc_pick<1, 256, false>(args, uniform_k, max_blocks, st);
  return split ? tc_pick<1, 128, true>(args, uniform_k, max_blocks, st)
               : tc_pick<1, 128, false>(args, uniform_k, max_blocks, st);
}

}  // namespace tmoe
