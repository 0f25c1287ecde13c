// Tensor-core FC launches (sm_103a): the activation tensor maps and the
// dispatch to the per-projection kernel variants (tc_kernel.cuh).
#include "tc_kernel.cuh"

namespace tmoe {

int tc_route_block() { return kTcBN; }

bool tc_fused_supported(int H, int bi, bool split) { return bi == 128 && H % 256 == 0 && !split; }

bool tc_supported(int H, int I, int bi, int rot_h, int rot_i) {
  // (512-point output rotations: the FC2 epilogue takes the levels inside
  // 64 columns, the combine the rest)
  return H % 128 == 0 && I % 64 == 0 && (bi == 64 || bi == 128) && I % bi == 0 &&
         (rot_h <= 128 || (rot_h == 512 && H % 512 == 0)) && rot_i <= bi;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

cudaError_t launch_tc_fc(const TcArgs& args_in, int proj, int uniform_k, int max_blocks, cudaStream_t st) {
  TcArgs args = args_in;
  {
    // the activation operand [act_rows][K] fp16 in boxes of 64 columns (128
    // bytes, the swizzle span) x 128 rows
    const int kdim = (proj == 2) ? args.f.I : args.f.H;
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {(cuuint64_t)kdim, (cuuint64_t)args.act_rows};
    cuuint64_t strides[1] = {(cuuint64_t)kdim * 2};
    cuuint32_t box[2] = {(cuuint32_t)kTcKS, 128};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(&args.amap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(args.f.act), dims, strides,
                           box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (proj == 3) {
      // FC2's operand: z~ [act_rows][I]
      if (!tc_fused_supported(args.f.H, args.bi, args.act2 != nullptr) || args.dep == nullptr)
        return cudaErrorInvalidValue;
      cuuint64_t dz[2] = {(cuuint64_t)args.f.I, (cuuint64_t)args.act_rows};
      cuuint64_t sz[1] = {(cuuint64_t)args.f.I * 2};
      const CUresult rz = enc(&args.amapz, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(args.f2.act), dz, sz,
                              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (rz != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    if (args.act2 != nullptr) {
      // separate gate / up operands: FC1 only, one 128-route accumulator per unit
      if (proj != 1 || args.route_block != 128) return cudaErrorInvalidValue;
      const CUresult r2 = enc(&args.amap2, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(args.act2), dims,
                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r2 != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    if (args.route_block != 128 && args.route_block != kTcBN) return cudaErrorInvalidValue;
  }
  switch (proj) {
    case 1: return launch_tc_fc1(args, uniform_k, max_blocks, st);
    case 2: return launch_tc_fc2(args, uniform_k, max_blocks, st);
    default: return launch_tc_fused(args, uniform_k, max_blocks, st);
  }
}

}  // namespace tmoe
