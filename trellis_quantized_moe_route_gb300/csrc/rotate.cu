// Fused input rotation + quantisation (sm_103a): x~ = H_b(suh * x) / sqrt(b)
// per block of b entries of H (b = 1, 64, 128 or 512), then fp16 (W4A16) or MXFP8 (W4A8) in the same
// kernel (b12x PR #129 "feat(moe): serve canonical Fruit QSRT atoms", Hot
// path: FC1 input rotation and MXFP8 quantization in one fixed CUDA kernel).
#include "rotate_dev.cuh"

namespace tmoe {

template <bool W4A8, int PER>
__global__ void __launch_bounds__(256) k_rotate_quant(const uint16_t* __restrict__ x, const uint16_t* __restrict__ suh,
                                                      int T, int H, int rot_b, void* __restrict__ xq,
                                                      uint8_t* __restrict__ xs, const int32_t* __restrict__ slot_of_route,
                                                      int topk) {
  rotate_quant_warp<W4A8, PER>(x, suh, T, H, rot_b, xq, xs, (blockIdx.x * blockDim.x + threadIdx.x) >> 5,
                               slot_of_route, topk);
}

cudaError_t launch_rotate_quant(const uint16_t* x, const uint16_t* suh, int T, int H, int rot_b, bool w4a8,
                                void* xq, uint8_t* xs, cudaStream_t st, const int32_t* slot_of_route, int topk) {
  if (T == 0) return cudaSuccess;
  if (w4a8 && slot_of_route != nullptr) return cudaErrorInvalidValue;  // slot order is the fp16 (W4A16) form
  const int per = rot_per(rot_b);
  const long warps = (long)T * (H / (32 * per));
  const int blocks = (int)((warps * 32 + 255) / 256);
  if (per == 16) {
    if (w4a8)
      k_rotate_quant<true, 16><<<blocks, 256, 0, st>>>(x, suh, T, H, rot_b, xq, xs, slot_of_route, topk);
    else
      k_rotate_quant<false, 16><<<blocks, 256, 0, st>>>(x, suh, T, H, rot_b, xq, xs, slot_of_route, topk);
  } else if (w4a8) {
    k_rotate_quant<true, 4><<<blocks, 256, 0, st>>>(x, suh, T, H, rot_b, xq, xs, slot_of_route, topk);
  } else {
    k_rotate_quant<false, 4><<<blocks, 256, 0, st>>>(x, suh, T, H, rot_b, xq, xs, slot_of_route, topk);
  }
  return cudaGetLastError();
}

template <bool W4A8, int PER>
__global__ void __launch_bounds__(256) k_rotate_routes(const RouteRotArgs a) {
  rotate_routes_warp<W4A8, PER>(a, (blockIdx.x * blockDim.x + threadIdx.x) >> 5);
}

cudaError_t launch_rotate_routes(const RouteRotArgs& a, bool w4a8, cudaStream_t st) {
  if (a.T == 0) return cudaSuccess;
  const int per = rot_per(a.rot_b);
  const long warps = (long)a.T * (a.H / (32 * per));
  const int blocks = (int)((warps * 32 + 255) / 256);
  if (per == 16) {
    if (w4a8)
      k_rotate_routes<true, 16><<<blocks, 256, 0, st>>>(a);
    else
      k_rotate_routes<false, 16><<<blocks, 256, 0, st>>>(a);
  } else if (w4a8) {
    k_rotate_routes<true, 4><<<blocks, 256, 0, st>>>(a);
  } else {
    k_rotate_routes<false, 4><<<blocks, 256, 0, st>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace tmoe
