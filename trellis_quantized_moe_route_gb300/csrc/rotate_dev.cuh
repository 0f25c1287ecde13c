// Device body of the fused rotate + quantize step, shared by the stand-alone
// kernel (rotate.cu) and the fused decode prologue (dec.cu).
#pragma once

#include "launch.h"
#include "route_dev.cuh"

namespace tmoe {

// One warp per (token, 128-wide chunk of H); lane l holds entries 4l..4l+3.
// Outputs: fp16 x~ [T][H] (W4A16), E4M3 codes [T][H] + E8M0 scales (W4A8;
// with `f16_codes` each code is stored as the fp16 number it encodes, and
// `xq_scaled`, if given, receives code * 2^e as fp16, exact for e in [-15, 7]).
// With `slot_of_route` (W4A16 only) the row is stored as fp16 once per route
// of the token, at the route's slot (x~ in slot order, [slots][H]).
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
  if (W4A8) {
    // fp64 butterflies, one rounding to fp32 (see warp_fwht_f64)
    double dv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) dv[i] = (double)v[i];
    warp_fwht_f64<4>(dv, rot_b);
    const double sc = hadamard_scale_f64(rot_b);
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = __double2float_rn(dv[i] * sc);
  } else {
    warp_fwht<4>(v, rot_b);
    const float sc = hadamard_scale(rot_b);
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] *= sc;
  }
  if (!W4A8) {
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

// This lane's 4 values (entries 4l..4l+3 of 128-chunk c) of row `row`:
// W4A16 as fp16 into out; W4A8 as MXFP8 over 32-blocks (8 lanes): the E4M3
// codes held exactly as fp16 into out, code * 2^e as fp16 into `scaled` (exact
// for e in [-15, 7]) and the E8M0 byte into xs.
template <bool W4A8>
static __device__ __forceinline__ void store_rot_chunk(const float (&v)[4], size_t row, int H, int c,
                                                       uint16_t* __restrict__ out, uint16_t* __restrict__ scaled,
                                                       uint8_t* __restrict__ xs) {
  const int lane = threadIdx.x & 31;
  const size_t base = row * H + (size_t)c * 128 + 4 * lane;
  if (!W4A8) {
    __half2 a = __floats2half2_rn(v[0], v[1]);
    __half2 b = __floats2half2_rn(v[2], v[3]);
    *reinterpret_cast<uint2*>(out + base) = make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
    return;
  }
  float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
  const int e = e8m0_exponent(amax);
  const float inv = exp2_int(-e);
  const uint2 cd = make_uint2(e4m3x2_to_f16x2(e4m3x2_from_float2(v[0] * inv, v[1] * inv)),
                              e4m3x2_to_f16x2(e4m3x2_from_float2(v[2] * inv, v[3] * inv)));
  *reinterpret_cast<uint2*>(out + base) = cd;
  *reinterpret_cast<uint2*>(scaled + base) = f16x4_times_exp2(cd, e);
  if ((lane & 7) == 0) xs[row * (H >> 5) + (size_t)c * 4 + (lane >> 3)] = (uint8_t)(e + 127);
}

// One warp per (token, 128-wide chunk of H), lane l holding entries 4l..4l+3:
// for each of the token's routes with a valid expert, both rotations of the
// chunk (computed once per token when the sign rows are shared), stored at
// the route's row. Routes with an out-of-range id are skipped (the FC kernels
// drop them).
template <bool W4A8>
static __device__ __forceinline__ void rotate_routes_warp(const RouteRotArgs& a, int gw) {
  const int lane = threadIdx.x & 31;
  const int chunks = a.H >> 7;
  if (gw >= a.T * chunks) return;
  const int t = gw / chunks, c = gw % chunks;
  const size_t xb = (size_t)t * a.H + (size_t)c * 128 + 4 * lane;
  const uint2 xr = __ldg(reinterpret_cast<const uint2*>(a.x + xb));
  float xv[4];
  const uint32_t xw[2] = {xr.x, xr.y};
#pragma unroll
  for (int i = 0; i < 4; ++i) xv[i] = __uint_as_float(((xw[i >> 1] >> (16 * (i & 1))) & 0xFFFFu) << 16);
  int my_e = -1;
  if (a.ids != nullptr) {
    if (lane < a.topk) my_e = a.ids[(size_t)t * a.topk + lane];
  } else {
    float w_, ws_;
    route_token_select(a.logits + (size_t)t * a.E, a.E, a.topk, my_e, w_, ws_);
  }
  long my_row = -1;
  if (lane < a.topk && my_e >= 0 && my_e < a.E)
    my_row = a.slot_of_route ? (long)a.slot_of_route[(size_t)t * a.topk + lane] : (long)t * a.topk + lane;
  const float hs = hadamard_scale(a.rot_b);
  float vg[4], vu[4];
  int have = -1;  // sign row of the rotations held in vg / vu
  for (int j = 0; j < a.topk; ++j) {
    const long row = __shfl_sync(0xFFFFFFFFu, my_row, j);
    const int e = __shfl_sync(0xFFFFFFFFu, my_e, j);
    if (row < 0) continue;  // warp-uniform
    const int sr = (a.sign_rows == 1) ? 0 : e;
    if (sr != have) {
      const uint2 gr = __ldg(reinterpret_cast<const uint2*>(a.gsuh + (size_t)sr * a.H + (size_t)c * 128 + 4 * lane));
      const uint2 ur = __ldg(reinterpret_cast<const uint2*>(a.usuh + (size_t)sr * a.H + (size_t)c * 128 + 4 * lane));
      const uint32_t gw2[2] = {gr.x, gr.y}, uw2[2] = {ur.x, ur.y};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        vg[i] = xv[i] * __half2float(__ushort_as_half((unsigned short)((gw2[i >> 1] >> (16 * (i & 1))) & 0xFFFFu)));
        vu[i] = xv[i] * __half2float(__ushort_as_half((unsigned short)((uw2[i >> 1] >> (16 * (i & 1))) & 0xFFFFu)));
      }
      if (W4A8) {
        // fp64 butterflies, one rounding to fp32 (see warp_fwht_f64)
        double dg[4], du[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          dg[i] = (double)vg[i];
          du[i] = (double)vu[i];
        }
        warp_fwht_f64<4>(dg, a.rot_b);
        warp_fwht_f64<4>(du, a.rot_b);
        const double hs64 = hadamard_scale_f64(a.rot_b);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          vg[i] = __double2float_rn(dg[i] * hs64);
          vu[i] = __double2float_rn(du[i] * hs64);
        }
      } else {
        warp_fwht<4>(vg, a.rot_b);
        warp_fwht<4>(vu, a.rot_b);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          vg[i] *= hs;
          vu[i] *= hs;
        }
      }
      have = sr;
    }
    store_rot_chunk<W4A8>(vg, (size_t)row, a.H, c, a.out_g, a.scaled_g, a.xs_g);
    store_rot_chunk<W4A8>(vu, (size_t)row, a.H, c, a.out_u, a.scaled_u, a.xs_u);
  }
}

}  // namespace tmoe
