// Device body of the fused rotate + quantize step, shared by the stand-alone
// kernels (rotate.cu) and the fused decode prologue (dec.cu).
//
// One warp per (token, chunk of 32 * PER entries of H); lane l holds entries
// PER*l .. PER*l + PER-1 of the chunk. PER = 4 for rotation blocks of up to
// 128 entries, PER = 16 for blocks of 512 (the coupled H512 boundary of
// TrellisMX-style layers: flashinfer PR #69 "b12x fused MoE: TrellisMX ...",
// Description), so that a whole rotation block sits in one warp.
#pragma once

#include "launch.h"
#include "route_dev.cuh"

namespace tmoe {

// Values per lane for a rotation block of rot_b entries on H.
__host__ __device__ constexpr int rot_per(int rot_b) { return rot_b > 128 ? 16 : 4; }

// PER consecutive 16-bit words at p (8-byte aligned: the inputs' contract) as
// PER floats of bf16 (BF = true) or fp16 bit patterns.
template <int PER, bool BF>
static __device__ __forceinline__ void load16(const uint16_t* __restrict__ p, float (&v)[PER]) {
  uint32_t w[PER / 2];
#pragma unroll
  for (int i = 0; i < PER / 4; ++i) {
    const uint2 q = __ldg(reinterpret_cast<const uint2*>(p) + i);
    w[2 * i] = q.x;
    w[2 * i + 1] = q.y;
  }
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const uint32_t b = (w[i >> 1] >> (16 * (i & 1))) & 0xFFFFu;
    v[i] = BF ? __uint_as_float(b << 16) : __half2float(__ushort_as_half((unsigned short)b));
  }
}

// The block rotation of v (in place) scaled by 1/sqrt(rot_b). W4A8 runs the
// butterflies in fp64 and rounds once to fp32 (see warp_fwht_f64).
template <bool W4A8, int PER>
static __device__ __forceinline__ void rotate_values(float (&v)[PER], int rot_b) {
  if (W4A8) {
    double dv[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) dv[i] = (double)v[i];
    warp_fwht_f64<PER>(dv, rot_b);
    const double sc = hadamard_scale_f64(rot_b);
#pragma unroll
    for (int i = 0; i < PER; ++i) v[i] = __double2float_rn(dv[i] * sc);
  } else {
    warp_fwht<PER>(v, rot_b);
    const float sc = hadamard_scale(rot_b);
#pragma unroll
    for (int i = 0; i < PER; ++i) v[i] *= sc;
  }
}

// PER floats as fp16 at p (8-byte aligned).
template <int PER>
static __device__ __forceinline__ void store_f16(uint16_t* p, const float (&v)[PER]) {
  uint32_t w[PER / 2];
#pragma unroll
  for (int i = 0; i < PER / 2; ++i) {
    __half2 h = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t*>(&h);
  }
#pragma unroll
  for (int i = 0; i < PER / 4; ++i) reinterpret_cast<uint2*>(p)[i] = make_uint2(w[2 * i], w[2 * i + 1]);
}

// MXFP8 of this lane's PER values: the block exponent over 32 entries (32 /
// PER lanes), then the E4M3 codes as 2 bytes per 32-bit word.
template <int PER>
static __device__ __forceinline__ int mxfp8_codes(const float (&v)[PER], uint32_t (&q)[PER / 2]) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < PER; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
  for (int o = 1; o < 32 / PER; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
  const int e = e8m0_exponent(amax);
  const float inv = exp2_int(-e);
#pragma unroll
  for (int i = 0; i < PER / 2; ++i) q[i] = e4m3x2_from_float2(v[2 * i] * inv, v[2 * i + 1] * inv);
  return e;
}

// This lane's PER values (entries PER*l.. of chunk c) of row `row`: W4A16 as
// fp16 into out; W4A8 as MXFP8 over 32-blocks: the E4M3 codes held exactly as
// fp16 into out, code * 2^e as fp16 into `scaled` (exact for e in [-15, 7])
// and the E8M0 byte into xs.
template <bool W4A8, int PER>
static __device__ __forceinline__ void store_rot_chunk(const float (&v)[PER], size_t row, int H, int c,
                                                       uint16_t* __restrict__ out, uint16_t* __restrict__ scaled,
                                                       uint8_t* __restrict__ xs) {
  const int lane = threadIdx.x & 31;
  const size_t base = row * H + (size_t)c * (32 * PER) + PER * lane;
  if (!W4A8) {
    store_f16<PER>(out + base, v);
    return;
  }
  uint32_t q[PER / 2];
  const int e = mxfp8_codes<PER>(v, q);
  uint32_t cd[PER / 2], sc[PER / 2];
#pragma unroll
  for (int i = 0; i < PER / 2; ++i) {
    cd[i] = e4m3x2_to_f16x2(q[i]);
    sc[i] = f16x2_times_exp2(cd[i], e);
  }
#pragma unroll
  for (int i = 0; i < PER / 4; ++i) {
    *reinterpret_cast<uint2*>(out + base + 4 * i) = make_uint2(cd[2 * i], cd[2 * i + 1]);
    *reinterpret_cast<uint2*>(scaled + base + 4 * i) = make_uint2(sc[2 * i], sc[2 * i + 1]);
  }
  if ((lane & (32 / PER - 1)) == 0) xs[row * (H >> 5) + ((size_t)c * (32 * PER) + PER * lane) / 32] = (uint8_t)(e + 127);
}

// Outputs: fp16 x~ [T][H] (W4A16), E4M3 codes [T][H] + E8M0 scales (W4A8;
// with `f16_codes` each code is stored as the fp16 number it encodes, and
// `xq_scaled`, if given, receives code * 2^e as fp16, exact for e in [-15, 7]).
// With `slot_of_route` (W4A16 only) the row is stored as fp16 once per route
// of the token, at the route's slot (x~ in slot order, [slots][H]).
template <bool W4A8, int PER>
static __device__ __forceinline__ void rotate_quant_warp(const uint16_t* __restrict__ x,
                                                         const uint16_t* __restrict__ suh, int T, int H, int rot_b,
                                                         void* __restrict__ xq, uint8_t* __restrict__ xs, int gw,
                                                         const int32_t* __restrict__ slot_of_route = nullptr,
                                                         int topk = 0, bool f16_codes = false,
                                                         uint16_t* __restrict__ xq_scaled = nullptr) {
  constexpr int CH = 32 * PER;
  const int lane = threadIdx.x & 31;
  const int chunks = H / CH;
  if (gw >= T * chunks) return;
  const int t = gw / chunks, c = gw % chunks;
  const size_t base = (size_t)t * H + (size_t)c * CH + PER * lane;
  // the token's slots (topk <= 32), one per lane, fetched with x
  const int my_slot = (slot_of_route != nullptr && lane < topk) ? slot_of_route[(size_t)t * topk + lane] : -1;
  float v[PER], s[PER];
  load16<PER, true>(x + base, v);
  load16<PER, false>(suh + (size_t)c * CH + PER * lane, s);
#pragma unroll
  for (int i = 0; i < PER; ++i) v[i] *= s[i];
  rotate_values<W4A8, PER>(v, rot_b);
  if (!W4A8) {
    if (slot_of_route == nullptr) {
      store_f16<PER>(reinterpret_cast<uint16_t*>(xq) + base, v);
    } else {
      for (int k = 0; k < topk; ++k) {
        const int slot = __shfl_sync(0xFFFFFFFFu, my_slot, k);
        if (slot >= 0) store_f16<PER>(reinterpret_cast<uint16_t*>(xq) + (size_t)slot * H + (size_t)c * CH + PER * lane, v);
      }
    }
  } else if (f16_codes) {
    store_rot_chunk<true, PER>(v, (size_t)t, H, c, reinterpret_cast<uint16_t*>(xq), xq_scaled, xs);
  } else {
    uint32_t q[PER / 2];
    const int e = mxfp8_codes<PER>(v, q);
    uint8_t* qb = reinterpret_cast<uint8_t*>(xq) + base;
#pragma unroll
    for (int i = 0; i < PER / 4; ++i) reinterpret_cast<uint32_t*>(qb)[i] = q[2 * i] | (q[2 * i + 1] << 16);
    if ((lane & (32 / PER - 1)) == 0) xs[(size_t)t * (H >> 5) + ((size_t)c * CH + PER * lane) / 32] = (uint8_t)(e + 127);
  }
}

// One warp per (token, chunk of H), separate gate / up input signs: for each
// of the token's routes with a valid expert, both rotations of the chunk
// (computed once per token when the sign rows are shared), stored at the
// route's row. Routes with an out-of-range id are skipped (the FC kernels
// drop them).
template <bool W4A8, int PER>
static __device__ __forceinline__ void rotate_routes_warp(const RouteRotArgs& a, int gw) {
  constexpr int CH = 32 * PER;
  const int lane = threadIdx.x & 31;
  const int chunks = a.H / CH;
  if (gw >= a.T * chunks) return;
  const int t = gw / chunks, c = gw % chunks;
  float xv[PER];
  load16<PER, true>(a.x + (size_t)t * a.H + (size_t)c * CH + PER * lane, xv);
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
  float vg[PER], vu[PER];
  int have = -1;  // sign row of the rotations held in vg / vu
  for (int j = 0; j < a.topk; ++j) {
    const long row = __shfl_sync(0xFFFFFFFFu, my_row, j);
    const int e = __shfl_sync(0xFFFFFFFFu, my_e, j);
    if (row < 0) continue;  // warp-uniform
    const int sr = (a.sign_rows == 1) ? 0 : e;
    if (sr != have) {
      float gs[PER], us[PER];
      load16<PER, false>(a.gsuh + (size_t)sr * a.H + (size_t)c * CH + PER * lane, gs);
      load16<PER, false>(a.usuh + (size_t)sr * a.H + (size_t)c * CH + PER * lane, us);
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        vg[i] = xv[i] * gs[i];
        vu[i] = xv[i] * us[i];
      }
      rotate_values<W4A8, PER>(vg, a.rot_b);
      rotate_values<W4A8, PER>(vu, a.rot_b);
      have = sr;
    }
    store_rot_chunk<W4A8, PER>(vg, (size_t)row, a.H, c, a.out_g, a.scaled_g, a.xs_g);
    store_rot_chunk<W4A8, PER>(vu, (size_t)row, a.H, c, a.out_u, a.scaled_u, a.xs_u);
  }
}

}  // namespace tmoe
