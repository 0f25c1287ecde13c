// Device helpers shared by the trellis-MoE kernels (sm_103a).
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace tmoe {

// ---------------------------------------------------------------------------
// MCG codebook (sparkinfer PR #90 "moe: integrate EXL3 Trellis into the fused
// W4A16 API", review of intrinsics.py: multiplier 0xCBAC1FED, mask 0x8fff8fff,
// third constant 0x3b603b60). A 16-bit state s maps to
//   y = ((s * 0xCBAC1FED) & 0x8fff8fff) ^ 0x3b603b60,
// whose two 16-bit halves are fp16 numbers; the weight is their fp16 sum.
// ---------------------------------------------------------------------------
constexpr uint32_t kMcgMult = 0xCBAC1FEDu;
constexpr uint32_t kMcgMask = 0x8FFF8FFFu;
constexpr uint32_t kMcgXor = 0x3B603B60u;

__device__ __forceinline__ uint32_t mcg_raw(uint32_t s) {
  return ((s * kMcgMult) & kMcgMask) ^ kMcgXor;
}

// Two weights from the raw codebook words of two states: (cb(a), cb(b)) as a
// half2 with cb(a) in the low half. One fp16x2 add rounds each sum to nearest.
__device__ __forceinline__ uint32_t cb_pair_from_raw(uint32_t ya, uint32_t yb) {
  uint32_t lo = __byte_perm(ya, yb, 0x5410);
  uint32_t hi = __byte_perm(ya, yb, 0x7632);
  __half2 r = __hadd2(*reinterpret_cast<__half2*>(&lo), *reinterpret_cast<__half2*>(&hi));
  return *reinterpret_cast<uint32_t*>(&r);
}

// fp16x2 -> two E4M3 bytes (round to nearest even, saturate to +-448), low byte
// from the low half.
__device__ __forceinline__ uint32_t e4m3x2_from_half2(uint32_t h2) {
  __half2_raw r;
  r.x = (unsigned short)(h2 & 0xFFFF);
  r.y = (unsigned short)(h2 >> 16);
  return (uint32_t)__nv_cvt_halfraw2_to_fp8x2(r, __NV_SATFINITE, __NV_E4M3);
}

__device__ __forceinline__ uint32_t e4m3x2_from_float2(float lo, float hi) {
  float2 v = make_float2(lo, hi);
  return (uint32_t)__nv_cvt_float2_to_fp8x2(v, __NV_SATFINITE, __NV_E4M3);
}

// Swap the two 16-bit words of a little-endian 32-bit load so that the first
// stored word is the most significant (tile streams are MSB first, words in
// storage order).
__device__ __forceinline__ uint32_t swap_words(uint32_t v) { return __byte_perm(v, 0, 0x1032); }

// ---------------------------------------------------------------------------
// Trellis states. Bit p of a tile's stream is bit (15 - p%16) of word p/16;
// the state of weight j is the 16 bits starting at stream bit (j+1)K-16
// (mod 256K), first bit most significant. A "run" is 8 consecutive states
// j0..j0+7 with j0 % 8 == 0 (half a tile row).
// ---------------------------------------------------------------------------

// Raw words for a run, any K in 2..6: the 64 stream bits starting at the word
// holding bit q0 = (j0+1)K-16 (mod 256K). Returns the window as hi:lo and the
// bit offset of state j0 inside it.
template <int K>
__device__ __forceinline__ void run_window_generic(const uint16_t* __restrict__ tile, int j0,
                                                   uint32_t& hi, uint32_t& lo, int& off) {
  constexpr int NB = 256 * K;
  constexpr int NW = 16 * K;
  int q0 = (j0 + 1) * K - 16;
  if (q0 < 0) q0 += NB;
  const int w = q0 >> 4;
  off = q0 & 15;
  const uint32_t w0 = __ldg(tile + w);
  const uint32_t w1 = __ldg(tile + (w + 1) % NW);
  const uint32_t w2 = __ldg(tile + (w + 2) % NW);
  const uint32_t w3 = __ldg(tile + (w + 3) % NW);
  hi = (w0 << 16) | w1;
  lo = (w2 << 16) | w3;
}

// States of a run from its window (off + 7K <= 48 holds for every run start
// j0 % 8 == 0 and K in 2..6).
template <int K>
__device__ __forceinline__ void run_states_generic(uint32_t hi, uint32_t lo, int off, uint32_t (&s)[8]) {
  const uint64_t v = ((uint64_t)hi << 32) | lo;
#pragma unroll
  for (int i = 0; i < 8; ++i) s[i] = (uint32_t)(v >> (48 - off - i * K)) & 0xFFFFu;
}

// K = 4 fast path. Row r of a tile is words 4r..4r+3; the run (r, h) needs
// the 32-bit word pair starting at word 4r+2h (cur) and the pair before it
// (prev, wrapping around the tile). Both are 4-byte aligned loads.
__device__ __forceinline__ void run_load_k4(const uint16_t* __restrict__ tile, int row, int h,
                                            uint32_t& prev, uint32_t& cur) {
  const uint32_t* t32 = reinterpret_cast<const uint32_t*>(tile);
  const int c = 2 * row + h;          // 32-bit word index of cur, 0..31
  cur = __ldg(t32 + c);
  prev = __ldg(t32 + ((c + 31) & 31));
}

// States of a K = 4 run: with V = prev:cur (as stream-order 64 bits), state i
// sits at V >> (28 - 4i). Only the high word of prev and both words of cur
// are needed: A = (prev.hi << 16) | cur.lo holds stream bits 16..47 of V, and
// the 32-bit window at shift n of A:cur (n >= 16, so cur.lo is shifted out)
// holds states m (high half) and m+4 (low half) for n = 28 - 4m.
__device__ __forceinline__ void run_states_k4(uint32_t prev_raw, uint32_t cur_raw, uint32_t (&s)[8]) {
  const uint32_t A = __byte_perm(prev_raw, cur_raw, 0x3254);
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const uint32_t q = __funnelshift_r(cur_raw, A, 28 - 4 * m);
    s[m] = q >> 16;
    s[m + 4] = q & 0xFFFFu;
  }
}

// Raw codebook words y[i] = mcg_raw(state i) of a K = 4 run, with the state
// split done by the integer multiply unit instead of the ALU:
// for a window q = [s_hi : s_lo], s_hi = umulhi(q, 2^16), x_hi = s_hi * M and
// x_lo = q * M - x_hi * 2^16 = s_lo * M (mod 2^32). `k16` must be 65536 and
// `nk16` 0xFFFF0000, passed at run time so they stay multiplies.
__device__ __forceinline__ void run_mcg_k4(uint32_t prev_raw, uint32_t cur_raw, uint32_t k16, uint32_t nk16,
                                           uint32_t (&y)[8]) {
  const uint32_t A = __byte_perm(prev_raw, cur_raw, 0x3254);
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const uint32_t q = __funnelshift_r(cur_raw, A, 28 - 4 * m);
    const uint32_t sh = __umulhi(q, k16);
    const uint32_t xh = sh * kMcgMult;
    const uint32_t xl = q * kMcgMult + xh * nk16;
    y[m] = (xh & kMcgMask) ^ kMcgXor;
    y[m + 4] = (xl & kMcgMask) ^ kMcgXor;
  }
}

// Weights from raw codebook words: fp16 pairs (w0,w1) .. (w6,w7). Each
// word's halves are summed by one fp16x2 add of its low and high halves
// (both lanes hold the sum), and one byte permute joins two such sums; on
// sm_103 this costs fewer integer-pipe instructions than permuting the
// words' halves first (measured).
__device__ __forceinline__ void raw_to_f16(const uint32_t (&y)[8], uint32_t (&w)[4]) {
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const __half2 va = *reinterpret_cast<const __half2*>(&y[2 * p]);
    const __half2 vb = *reinterpret_cast<const __half2*>(&y[2 * p + 1]);
    __half2 da = __hadd2(__low2half2(va), __high2half2(va));
    __half2 db = __hadd2(__low2half2(vb), __high2half2(vb));
    w[p] = __byte_perm(*reinterpret_cast<uint32_t*>(&da), *reinterpret_cast<uint32_t*>(&db), 0x5410);
  }
}

// fp16x2 -> two E4M3 bytes with the native conversion instruction.
__device__ __forceinline__ uint32_t cvt_e4m3x2(uint32_t h2) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(r) : "r"(h2));
  return r;
}

// E4M3 bytes from raw codebook words: (w0..w3), (w4..w7). Each weight is the
// fp16 sum of its word's halves (one fp16 add with half selectors), paired
// and converted two at a time.
__device__ __forceinline__ void raw_to_e4m3(const uint32_t (&y)[8], uint32_t (&q)[2]) {
  __half hw[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const __half2 v = *reinterpret_cast<const __half2*>(&y[i]);
    hw[i] = __hadd(__low2half(v), __high2half(v));
  }
  uint32_t c[4];
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    __half2 t = __halves2half2(hw[2 * p], hw[2 * p + 1]);
    c[p] = cvt_e4m3x2(*reinterpret_cast<uint32_t*>(&t));
  }
  q[0] = __byte_perm(c[0], c[1], 0x5410);
  q[1] = __byte_perm(c[2], c[3], 0x5410);
}

// Two E4M3 bytes (low byte first) -> fp16x2, exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t b2) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((uint16_t)b2));
  return r;
}

// W4A8 weights for the fp16 tensor path: each weight is the E4M3 rounding of
// its fp16 codebook value, returned as the (exactly representable) fp16 value;
// pairs (w0,w1) .. (w6,w7). Products of such weights with E4M3 activations
// held in fp16 are exact, so an fp16 MMA with fp32 accumulation computes the
// same sums as an E4M3 MMA (up to summation order).
__device__ __forceinline__ void raw_to_e4m3_f16(const uint32_t (&y)[8], uint32_t (&w)[4]) {
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const __half2 va = *reinterpret_cast<const __half2*>(&y[2 * p]);
    const __half2 vb = *reinterpret_cast<const __half2*>(&y[2 * p + 1]);
    __half2 t = __halves2half2(__hadd(__low2half(va), __high2half(va)), __hadd(__low2half(vb), __high2half(vb)));
    w[p] = e4m3x2_to_f16x2(cvt_e4m3x2(*reinterpret_cast<uint32_t*>(&t)));
  }
}

// Decoded fp16 weights of a run as 4 half2 registers: (w0,w1), (w2,w3), (w4,w5), (w6,w7).
__device__ __forceinline__ void run_weights_f16(const uint32_t (&s)[8], uint32_t (&w)[4]) {
  uint32_t y[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) y[i] = mcg_raw(s[i]);
#pragma unroll
  for (int p = 0; p < 4; ++p) w[p] = cb_pair_from_raw(y[2 * p], y[2 * p + 1]);
}

// E4M3 weights of a run as 2 registers of 4 bytes: (w0..w3), (w4..w7).
__device__ __forceinline__ void run_weights_e4m3(const uint32_t (&s)[8], uint32_t (&q)[2]) {
  uint32_t w[4];
  run_weights_f16(s, w);
  q[0] = __byte_perm(cvt_e4m3x2(w[0]), cvt_e4m3x2(w[1]), 0x5410);
  q[1] = __byte_perm(cvt_e4m3x2(w[2]), cvt_e4m3x2(w[3]), 0x5410);
}

// ---------------------------------------------------------------------------
// Warp Walsh-Hadamard transform (Sylvester order) of a vector spread over the
// warp, PER consecutive values per lane (lane l holds v[PER*l .. PER*l+PER-1]),
// applied independently to blocks of B entries (B a power of two, B <= 32*PER).
// Butterfly: for h = 1, 2, 4, ...: (x[i], x[i+h]) <- (x[i] + x[i+h], x[i] - x[i+h]).
// ---------------------------------------------------------------------------
template <int PER>
__device__ __forceinline__ void warp_fwht(float (&v)[PER], int B) {
  // in-register stages
#pragma unroll
  for (int h = 1; h < PER; h <<= 1) {
    if (h < B) {
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        if ((i & h) == 0) {
          const float a = v[i], b = v[i + h];
          v[i] = a + b;
          v[i + h] = a - b;
        }
      }
    }
  }
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int lh = 1; lh < 32; lh <<= 1) {
    if (lh * PER < B) {
      const bool upper = (lane & lh) != 0;
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const float o = __shfl_xor_sync(0xFFFFFFFFu, v[i], lh);
        v[i] = upper ? (o - v[i]) : (v[i] + o);
      }
    }
  }
}

// The same transform in fp64. The W4A8 input rotation runs in it: the block
// sums of bf16 x fp16 products are then exact for ordinary data, and their
// one rounding to fp32 matches a float64 evaluation, so the MXFP8 codes
// (decided on those fp32 values) do not depend on the butterfly order.
template <int PER>
__device__ __forceinline__ void warp_fwht_f64(double (&v)[PER], int B) {
#pragma unroll
  for (int h = 1; h < PER; h <<= 1) {
    if (h < B) {
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        if ((i & h) == 0) {
          const double a = v[i], b = v[i + h];
          v[i] = a + b;
          v[i + h] = a - b;
        }
      }
    }
  }
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int lh = 1; lh < 32; lh <<= 1) {
    if (lh * PER < B) {
      const bool upper = (lane & lh) != 0;
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const double o = __shfl_xor_sync(0xFFFFFFFFu, v[i], lh);
        v[i] = upper ? (o - v[i]) : (v[i] + o);
      }
    }
  }
}

// 1/sqrt(B) in fp64, as 1 / fp64(sqrt(B)) rounds (0.08838834764831843 for
// B = 128, the rotation matrix's entries in a float64 evaluation).
__device__ __forceinline__ double hadamard_scale_f64(int B) {
  return B == 128 ? 0.08838834764831843
                  : (B == 64 ? 0.125 : (B == 512 ? 0.04419417382415922 : (B == 32 ? 0.17677669529663687 : 1.0)));
}

__device__ __forceinline__ float hadamard_scale(int B) {
  // 1/sqrt(B) rounded to fp32 (B = 128: 0.088388347648...)
  return B == 128 ? 0.08838834764831845f
                  : (B == 64 ? 0.125f : (B == 512 ? 0.044194173824159216f : (B == 32 ? 0.17677669529663687f : 1.0f)));
}

// UE8M0 exponent of a block from its max |v|: e = ceil(log2(fp32(amax/448))),
// clamped to [-127, 127]; amax == 0 gives -127 (flashinfer PR #69 "b12x fused
// MoE: TrellisMX (procedural NPK) source format with an in-tree P8 runtime",
// Evidence, precision notes: exponent from the exact FP32 bits of amax/448).
__device__ __forceinline__ int e8m0_exponent(float amax) {
  const float q = __fdiv_rn(amax, 448.0f);
  const uint32_t b = __float_as_uint(q) & 0x7FFFFFFFu;
  if (b == 0) return -127;
  const int ex = (int)(b >> 23);
  const uint32_t man = b & 0x7FFFFFu;
  int e;
  if (ex == 0) {
    e = (32 - __clz(man - 1)) - 149;  // ceil(log2(man)) - 149
  } else {
    e = ex - 127 + (man != 0 ? 1 : 0);
  }
  return max(-127, min(127, e));
}

// MXFP8 blocks whose E8M0 exponent e lies in [-15, 7] can be held as fp16
// values code * 2^e exactly (448 * 2^7 < 65504; the smallest code step
// 2^-9 * 2^-15 is the fp16 subnormal step).
constexpr int kE8m0PreLo = 127 - 15, kE8m0PreHi = 127 + 7;

// 2^e as a float, exact for e in [-149, 127].
__device__ __forceinline__ float exp2_int(int e) {
  if (e >= -126) return __uint_as_float((uint32_t)(e + 127) << 23);
  return __uint_as_float(1u << (e + 149));
}

// Four fp16 values (two half2 words) times 2^e, rounded to fp16 (exact when
// the result is representable).
__device__ __forceinline__ uint32_t f16x2_times_exp2(uint32_t c, int e) {
  const float sc = exp2_int(max(-149, min(127, e)));
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&c));
  __half2 r = __floats2half2_rn(a.x * sc, a.y * sc);
  return *reinterpret_cast<uint32_t*>(&r);
}
__device__ __forceinline__ uint2 f16x4_times_exp2(uint2 c, int e) {
  const float sc = exp2_int(max(-149, min(127, e)));
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&c.x));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&c.y));
  __half2 ra = __floats2half2_rn(a.x * sc, a.y * sc), rb = __floats2half2_rn(b.x * sc, b.y * sc);
  return make_uint2(*reinterpret_cast<uint32_t*>(&ra), *reinterpret_cast<uint32_t*>(&rb));
}


// ---------------------------------------------------------------------------
// Warp-level MMA (legacy mma.sync) wrappers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_e4m3_16832(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%10,%10,%10};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.0f));
}

// cp.async 16 bytes global -> shared; src_bytes = 0 zero-fills.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, int src_bytes) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

}  // namespace tmoe
