// Deterministic top-k combine (sm_103a): y_t = sum_{j=0..k-1} w_{t,j} * row(slot(t, j)),
// FP32, in ascending j for every token (sparkinfer PR #90 "moe: integrate
// EXL3 Trellis into the fused W4A16 API", walkthrough: FP32 routed output;
// b12x PR #129 "feat(moe): serve canonical Fruit QSRT atoms", Hot path: FC2
// preserves exact top-k weighting). The rows already carry H and down_svh.
#include "launch.h"

namespace tmoe {

__global__ void __launch_bounds__(256) k_combine(const float* __restrict__ rows, const int32_t* __restrict__ slot_of_route,
                                                 const float* __restrict__ w, int T, int H, int k,
                                                 float* __restrict__ out) {
  const int vec_per_row = H >> 2;
  const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long)T * vec_per_row) return;
  const int t = (int)(i / vec_per_row), c = (int)(i % vec_per_row);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = 0; j < k; ++j) {
    const int slot = slot_of_route[t * k + j];
    if (slot < 0) continue;  // dropped (out-of-range) expert id
    const float wj = w[t * k + j];
    const float4 v = __ldg(reinterpret_cast<const float4*>(rows + (size_t)slot * H) + c);
    acc.x = fmaf(wj, v.x, acc.x);
    acc.y = fmaf(wj, v.y, acc.y);
    acc.z = fmaf(wj, v.z, acc.z);
    acc.w = fmaf(wj, v.w, acc.w);
  }
  reinterpret_cast<float4*>(out + (size_t)t * H)[c] = acc;
}

cudaError_t launch_combine(const float* rows, const int32_t* slot_of_route, const float* w, int T, int H, int k,
                           float* out, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const long n = (long)T * (H / 4);
  k_combine<<<(int)((n + 255) / 256), 256, 0, st>>>(rows, slot_of_route, w, T, H, k, out);
  return cudaGetLastError();
}

}  // namespace tmoe
