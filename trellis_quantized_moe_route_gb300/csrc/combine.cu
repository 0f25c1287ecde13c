// Deterministic top-k combine (sm_103a): y_t = sum_{j=0..k-1} w_{t,j} * row(slot(t, j)),
// FP32, in ascending j for every token (sparkinfer PR #90 "moe: integrate
// EXL3 Trellis into the fused W4A16 API", walkthrough: FP32 routed output;
// b12x PR #129 "feat(moe): serve canonical Fruit QSRT atoms", Hot path: FC2
// preserves exact top-k weighting). k_combine takes rows that already carry
// H and down_svh; k_combine_unrot applies them itself.
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

// Combine of partly unrotated per-slot rows (the tensor-core FC2 stores, per
// 128-column block, the scaled accumulator after the Hadamard levels inside
// each 64-column half): for each route in ascending j, the level across the
// halves (rotation blocks of 128), hs * down_svh_e, then w * that into the
// FP32 sum -- the same steps and roundings an FC2 epilogue would take. A warp
// covers 256 output channels; lane l holds channels 4i..4i+3 and 64+4i..
// 64+4i+3 of block l/16 (i = l%16), so the remaining level is in registers.
__device__ __forceinline__ float4 h4_to_f4(uint2 p) {
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&p.x));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&p.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

constexpr int kCombineMaxK = 32;

__global__ void __launch_bounds__(256, 3) k_combine_unrot(CombineUnrotArgs a) {
  const int lane = threadIdx.x & 31;
  const int chunks = (a.H + 255) >> 8;
  const long wid = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (wid >= (long)a.T * chunks) return;
  const int t = (int)(wid / chunks);
  const int c0 = (int)(wid % chunks) * 256 + (lane >> 4) * 128 + 4 * (lane & 15);
  const bool live = c0 < a.H;  // (H % 256 == 128: the last warp's upper half idles)
  const bool across = a.rot_b > 64;
  // the token's slots, experts and weights, one route per lane
  int my_slot = -1, my_e = 0;
  float my_w = 0.0f;
  if (lane < a.k) {
    my_slot = a.slot_of_route[(size_t)t * a.k + lane];
    my_w = a.w[(size_t)t * a.k + lane];
    if (my_slot >= 0) my_e = a.block_expert[my_slot / a.bn];
  }
  const float hs = hadamard_scale(a.rot_b);
  float4 lo = make_float4(0.f, 0.f, 0.f, 0.f), hi = lo;
  // four routes at a time: their loads are issued before any is used
  for (int j0 = 0; j0 < a.k; j0 += 4) {
    float4 va[4], vb[4];
    uint2 ga[4], gb[4];
    int slot[4];
    float wj[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int j = j0 + u;
      slot[u] = __shfl_sync(0xFFFFFFFFu, my_slot, j & 31);
      wj[u] = __shfl_sync(0xFFFFFFFFu, my_w, j & 31);
      const int e = __shfl_sync(0xFFFFFFFFu, my_e, j & 31);
      if (j >= a.k) slot[u] = -1;
      va[u] = vb[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      ga[u] = gb[u] = make_uint2(0u, 0u);
      if (slot[u] >= 0 && live) {  // (a dropped, out-of-range expert id has no slot)
        const float* r = a.rows + (size_t)slot[u] * a.H + c0;
        const uint16_t* g = a.svh + (size_t)e * a.H + c0;
        va[u] = __ldcs(reinterpret_cast<const float4*>(r));
        vb[u] = __ldcs(reinterpret_cast<const float4*>(r + 64));
        ga[u] = __ldg(reinterpret_cast<const uint2*>(g));
        gb[u] = __ldg(reinterpret_cast<const uint2*>(g + 64));
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (slot[u] < 0) continue;  // warp-uniform
      const float4 fa = h4_to_f4(ga[u]), fb = h4_to_f4(gb[u]);
      float4 x = va[u], y = vb[u];
      if (across) {
        x = make_float4(va[u].x + vb[u].x, va[u].y + vb[u].y, va[u].z + vb[u].z, va[u].w + vb[u].w);
        y = make_float4(va[u].x - vb[u].x, va[u].y - vb[u].y, va[u].z - vb[u].z, va[u].w - vb[u].w);
      }
      x = make_float4(x.x * (hs * fa.x), x.y * (hs * fa.y), x.z * (hs * fa.z), x.w * (hs * fa.w));
      y = make_float4(y.x * (hs * fb.x), y.y * (hs * fb.y), y.z * (hs * fb.z), y.w * (hs * fb.w));
      lo = make_float4(fmaf(wj[u], x.x, lo.x), fmaf(wj[u], x.y, lo.y), fmaf(wj[u], x.z, lo.z), fmaf(wj[u], x.w, lo.w));
      hi = make_float4(fmaf(wj[u], y.x, hi.x), fmaf(wj[u], y.y, hi.y), fmaf(wj[u], y.z, hi.z), fmaf(wj[u], y.w, hi.w));
    }
  }
  if (live) {
    float* o = a.out + (size_t)t * a.H + c0;
    *reinterpret_cast<float4*>(o) = lo;
    *reinterpret_cast<float4*>(o + 64) = hi;
  }
}

// The same for 512-point output rotation blocks (the coupled H512 boundary
// of TrellisMX-style layers: flashinfer PR #69 "b12x fused MoE: TrellisMX
// ...", Description): one warp per (token, 512 output channels); lane l (h =
// l / 16, i = l % 16) holds, for each 128-column quarter b of the block,
// channels 128 b + 64 h + 4 i .. +3. The remaining levels: across the halves
// (64) with the partner lane l ^ 16, across quarters (128 and 256) in
// registers; then hs * down_svh and w * that into the FP32 sum, routes in
// ascending j.
__global__ void __launch_bounds__(256) k_combine_unrot512(CombineUnrotArgs a) {
  const int lane = threadIdx.x & 31;
  const int chunks = a.H >> 9;
  const long wid = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (wid >= (long)a.T * chunks) return;
  const int t = (int)(wid / chunks);
  const int hb = lane >> 4;
  const int c0 = (int)(wid % chunks) * 512 + 64 * hb + 4 * (lane & 15);
  int my_slot = -1, my_e = 0;
  float my_w = 0.0f;
  if (lane < a.k) {
    my_slot = a.slot_of_route[(size_t)t * a.k + lane];
    my_w = a.w[(size_t)t * a.k + lane];
    if (my_slot >= 0) my_e = a.block_expert[my_slot / a.bn];
  }
  const float hs = hadamard_scale(512);
  float4 acc[4];
#pragma unroll
  for (int b = 0; b < 4; ++b) acc[b] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = 0; j < a.k; ++j) {
    const int slot = __shfl_sync(0xFFFFFFFFu, my_slot, j);
    const float wj = __shfl_sync(0xFFFFFFFFu, my_w, j);
    const int e = __shfl_sync(0xFFFFFFFFu, my_e, j);
    if (slot < 0) continue;  // warp-uniform: a dropped (out-of-range) expert id has no slot
    float4 v[4];
    uint2 g[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      v[b] = __ldcs(reinterpret_cast<const float4*>(a.rows + (size_t)slot * a.H + c0 + 128 * b));
      g[b] = __ldg(reinterpret_cast<const uint2*>(a.svh + (size_t)e * a.H + c0 + 128 * b));
    }
#pragma unroll
    for (int b = 0; b < 4; ++b) {  // level 64: the lower half keeps x + x', the upper x' - x
      const float4 o = make_float4(__shfl_xor_sync(0xFFFFFFFFu, v[b].x, 16), __shfl_xor_sync(0xFFFFFFFFu, v[b].y, 16),
                                   __shfl_xor_sync(0xFFFFFFFFu, v[b].z, 16), __shfl_xor_sync(0xFFFFFFFFu, v[b].w, 16));
      v[b] = hb ? make_float4(o.x - v[b].x, o.y - v[b].y, o.z - v[b].z, o.w - v[b].w)
                : make_float4(v[b].x + o.x, v[b].y + o.y, v[b].z + o.z, v[b].w + o.w);
    }
#pragma unroll
    for (int d = 1; d <= 2; d <<= 1) {  // levels 128 and 256 across the quarters
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        if (b & d) continue;
        const float4 x = v[b], y = v[b + d];
        v[b] = make_float4(x.x + y.x, x.y + y.y, x.z + y.z, x.w + y.w);
        v[b + d] = make_float4(x.x - y.x, x.y - y.y, x.z - y.z, x.w - y.w);
      }
    }
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const float4 f = h4_to_f4(g[b]);
      acc[b] = make_float4(fmaf(wj, v[b].x * (hs * f.x), acc[b].x), fmaf(wj, v[b].y * (hs * f.y), acc[b].y),
                           fmaf(wj, v[b].z * (hs * f.z), acc[b].z), fmaf(wj, v[b].w * (hs * f.w), acc[b].w));
    }
  }
#pragma unroll
  for (int b = 0; b < 4; ++b) *reinterpret_cast<float4*>(a.out + (size_t)t * a.H + c0 + 128 * b) = acc[b];
}

cudaError_t launch_combine_unrot(const CombineUnrotArgs& a, cudaStream_t st) {
  if (a.T == 0) return cudaSuccess;
  if (a.rot_b == 512) {
    if (a.H % 512 != 0 || a.k > kCombineMaxK) return cudaErrorInvalidValue;
    const long warps = (long)a.T * (a.H / 512);
    k_combine_unrot512<<<(int)((warps + 7) / 8), 256, 0, st>>>(a);
    return cudaGetLastError();
  }
  if (a.H % 128 != 0 || a.k > kCombineMaxK || a.rot_b > 128) return cudaErrorInvalidValue;
  const long warps = (long)a.T * ((a.H + 255) / 256);
  k_combine_unrot<<<(int)((warps + 7) / 8), 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_combine(const float* rows, const int32_t* slot_of_route, const float* w, int T, int H, int k,
                           float* out, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const long n = (long)T * (H / 4);
  k_combine<<<(int)((n + 255) / 256), 256, 0, st>>>(rows, slot_of_route, w, T, H, k, out);
  return cudaGetLastError();
}

}  // namespace tmoe
