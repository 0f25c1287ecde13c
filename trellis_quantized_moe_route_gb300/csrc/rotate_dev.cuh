// Device body of the fused rotate + quantize step, shared by the stand-alone
// kernel (rotate.cu) and the fused decode prologue (dec.cu).
#pragma once

#include "launch.h"

namespace tmoe {

// One warp per (token, 128-wide chunk of H); lane l holds entries 4l..4l+3.
// Outputs: fp16 x~ [T][H] (W4A16), E4M3 codes [T][H] + E8M0 scales (W4A8;
// with `f16_codes` each code is stored as the fp16 number it encodes, and
// `xq_scaled`, if given, receives code * 2^e as fp16, exact for e in [-15, 7]).
// With `slot_of_route` the row is stored as fp16 once per route of the token,
// at the route's slot (x~ in slot order, [slots][H]); W4A8 then stores the
// exact dequantized MXFP8 values code * 2^e.
template <bool W4A8>
static __device__ __forceinline__ void rotate_quant_warp(const uint16_t* __restrict__ x,
                                                         const uint16_t* __restrict__ suh, int T, int H, int rot_b,
                                                         void* __restrict__ xq, uint8_t* __restrict__ xs, int gw,
                                                         const int32_t* __restrict__ slot_of_route = nullptr,
                                                         int topk = 0, bool f16_codes = false,
                                                         uint16_t* __restrict__ xq_scaled = nullptr) {
  const int lane = threadIdx.x & 31;
  const int chunks = H >> 7;
  if (gw >= T * chunks) return;
  const int t = gw / chunks, c = gw % chunks;
  const size_t base = (size_t)t * H + (size_t)c * 128 + 4 * lane;
  const uint2 xr = __ldg(reinterpret_cast<const uint2*>(x + base));
  const uint2 sr = __ldg(reinterpret_cast<const uint2*>(suh + (size_t)c * 128 + 4 * lane));
  // the token's slots (topk <= 32), one per lane, fetched with x
  const int my_slot = (slot_of_route != nullptr && lane < topk) ? slot_of_route[(size_t)t * topk + lane] : -1;
  float v[4];
  const uint32_t xw[2] = {xr.x, xr.y};
  const uint32_t sw[2] = {sr.x, sr.y};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t xb = (xw[i >> 1] >> (16 * (i & 1))) & 0xFFFFu;
    const uint32_t sb = (sw[i >> 1] >> (16 * (i & 1))) & 0xFFFFu;
    v[i] = __uint_as_float(xb << 16) * __half2float(__ushort_as_half((unsigned short)sb));
  }
  warp_fwht<4>(v, rot_b);
  const float sc = hadamard_scale(rot_b);
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] *= sc;
  if (W4A8 && slot_of_route != nullptr) {
    // MXFP8 rounding kept as the dequantized values (32-element block = 8 lanes)
    float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    const int e = e8m0_exponent(amax);
    const float inv = exp2_int(-e), sc = exp2_int(e);
#pragma unroll
    for (int i = 0; i < 4; i += 2) {
      const uint32_t q = e4m3x2_to_f16x2(e4m3x2_from_float2(v[i] * inv, v[i + 1] * inv));
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&q));
      v[i] = f.x * sc;
      v[i + 1] = f.y * sc;
    }
  }
  if (!W4A8 || slot_of_route != nullptr) {
    __half2 a = __floats2half2_rn(v[0], v[1]);
    __half2 b = __floats2half2_rn(v[2], v[3]);
    uint2 o;
    o.x = *reinterpret_cast<uint32_t*>(&a);
    o.y = *reinterpret_cast<uint32_t*>(&b);
    if (slot_of_route == nullptr) {
      *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(xq) + base) = o;
    } else {
      for (int k = 0; k < topk; ++k) {
        const int slot = __shfl_sync(0xFFFFFFFFu, my_slot, k);
        if (slot >= 0)
          *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(xq) + (size_t)slot * H + (size_t)c * 128 + 4 * lane) = o;
      }
    }
  } else {
    // 32-element block = 8 lanes
    float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    const int e = e8m0_exponent(amax);
    const float inv = exp2_int(-e);
    const uint32_t q0 = e4m3x2_from_float2(v[0] * inv, v[1] * inv), q1 = e4m3x2_from_float2(v[2] * inv, v[3] * inv);
    if (f16_codes) {  // the E4M3 codes held exactly as fp16
      const uint2 c = make_uint2(e4m3x2_to_f16x2(q0), e4m3x2_to_f16x2(q1));
      *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(xq) + base) = c;
      if (xq_scaled) *reinterpret_cast<uint2*>(xq_scaled + base) = f16x4_times_exp2(c, e);
    } else
      *reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(xq) + base) = q0 | (q1 << 16);
    if ((lane & 7) == 0) xs[(size_t)t * (H >> 5) + (size_t)c * 4 + (lane >> 3)] = (uint8_t)(e + 127);
  }
}

}  // namespace tmoe
