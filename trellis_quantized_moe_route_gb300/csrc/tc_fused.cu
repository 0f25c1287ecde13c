// Tensor-core kernel variants of one projection: FC1 and FC2 in one launch (both with 256-row units).
// One translation unit per projection, so that the variants compile in
// parallel; the launcher with the tensor maps is in tc.cu.
#include "tc_kernel.cuh"

namespace tmoe {

cudaError_t launch_tc_fused(const TcArgs& args, int uniform_k, int max_blocks, cudaStream_t st) {
  return tc_pick<3, 256, false>(args, uniform_k, max_blocks, st);
}

}  // namespace tmoe
