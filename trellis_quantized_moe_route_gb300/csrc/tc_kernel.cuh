// The tensor-core FC kernel (sm_103a): roles, kernel and launch template.
// Included by one translation unit per projection (tc_fc1.cu, tc_fc2.cu,
// tc_fused.cu) so that the variants compile in parallel; tc.cu holds the
// tensor maps and the dispatch.
//
// FC1 / FC2 on the 5th-generation tensor cores (sm_103a) outside the decode
// regime, W4A16: fp16 activations x fp16 trellis weights -> fp32 (W4A8 is the
// bounded-decode-rows mode, b12x PR #129 "feat(moe): serve canonical Fruit
// QSRT atoms", Hot path, and runs on the decode-rows kernels).
//
// A persistent, warp-specialised kernel; one CTA per SM takes work units
// (route block rb of up to 256 routes of one expert) x (block mb of N weight
// rows: FC1 takes bi gate rows and the bi matching up rows, N = 2 bi; FC2
// takes N output columns). The contraction runs in stages of 64 columns:
//
//   warp 16     (payload)   claims units from a device counter, publishes them
//                           to the other roles through a small ring, and
//                           streams each stage's trellis payload (4 tiles per
//                           tile row) into a 4-deep ring with bulk copies;
//   warp 17     (activation) one thread loads a stage's activation rows (slot
//                           order, one 128-row box per accumulator) into a
//                           128-byte swizzled operand with TMA;
//   warps 0-7   (expanders) decode the stage's N x 64 weights from the payload
//                           into a second swizzled operand, each codebook value
//                           the fp16 sum of its word's two halves as the
//                           codebook defines it;
//   warp 18     (issuer)    one thread issues tcgen05.mma with the routes as M
//                           (one or two accumulators of 128 routes) and the
//                           weight rows as N, and commits each stage to the
//                           mbarriers that free its operand slots;
//   warps 8-15  (epilogue)  one TMEM lane (route) per thread and two warps per
//                           lane quarter, each taking half of every column
//                           block, so the block Hadamard transforms run inside
//                           registers plus one exchange level across the pair
//                           (FC1: H -> svh -> SiLU(gate)*up -> suh_down -> H, as
//                           in sparkinfer PR #90 "moe: integrate EXL3 Trellis
//                           into the fused W4A16 API", review of kernel.py;
//                           FC2: scale, H, down_svh).
//
// Where FC1 and FC2 both take 256-row units the two run as one launch: the
// unit order holds every FC1 unit, then every FC2 unit; an FC2 unit's
// activation loader waits (bounded) until the epilogue warps of its route
// block's FC1 units have counted their z~ rows in a per-block counter, so the
// FC2 units fill the SMs that the last wave of FC1 units leaves idle.
//
// Tensor memory holds two 256-column accumulator buffers: a unit of up to 128
// routes takes one (alternating), a unit of up to 256 routes takes both, so
// the epilogue of one unit overlaps the contraction of the next. Every
// hand-off is an mbarrier (full/empty rings of 2 activation, 3 decoded and 4
// payload stages, full/empty per accumulator buffer); no role waits on a
// block-wide barrier. Waits are bounded in wall time; on a timeout the CTA
// raises the error word, drains its copies and MMAs and releases its tensor
// memory.
#pragma once

#include <cudaTypedefs.h>

#include <algorithm>

#include "launch.h"
#include "tc.cuh"

namespace tmoe {

constexpr int kTcThreads = 640;        // warpgroups: 2 expander, 2 epilogue, 1 loader/issuer
// Registers per thread after the split: the expander and loader/issuer
// warpgroups give registers up, the epilogue warpgroups take them (sum x 128
// threads <= 640 x 96, the launch budget: the kernel must be compiled at 96
// registers, which the launcher checks, or setmaxnreg.inc could wait for
// registers never freed). With the K=4 expansion the expanders fit in 56 and
// the FC1 epilogue needs 168 to run without spilling; the general-K
// expanders keep the launch count.
constexpr int kRegAux = 32, kRegLaunch = 96;
template <int KB>
struct TcRegs {
  static constexpr int exp = KB > 0 ? 56 : 96;
  static constexpr int epi = KB > 0 ? 168 : 128;
  static_assert(128 * (2 * exp + 2 * epi + kRegAux) <= kTcThreads * kRegLaunch, "register split over budget");
};
constexpr int kTcExp = 256;            // expander threads
constexpr int kTcEpiWarps = 8;         // two per TMEM lane quarter, one per column half
constexpr int kEvecBytes = 1024;       // per epilogue warp: its half of the unit's folded vectors (fp32)
constexpr int kStageWords = 20;        // per epilogue warp: 32 rows x 16 words of output staging, stride 20 words
constexpr int kStageBytes = 32 * kStageWords * 4;
constexpr int kTcBN = 256;             // routes per route block (128 with split gate / up operands)
constexpr int kTcKS = 64;              // contraction columns per stage
// Stage barriers: full[g % SB] completes when stage g's activation box has
// landed and every expander warp has stored its decoded rows (one wait for
// the MMA issuer); empty[g % SB] when the stage's MMAs have completed (one
// commit), which frees both the decoded buffer and the activation slot.
// Every barrier operation costs the issuer a shared-memory round trip while
// the tensor core streams its operands, so it waits and commits once per
// stage. The activation ring is no deeper than the decoded ring (kSA <= SB),
// so a phase of empty[] is never overtaken before the loader has seen it.
constexpr int kSA = 2, kSW = 4, kSBMax = 3;
// decoded-operand ring depth: 3 for the 4-bit payload, 2 for the general
// case, whose larger payload slots leave no room for a third
__host__ __device__ constexpr int tc_sb(int KB) { return KB > 0 ? 3 : 2; }
constexpr int kABytes = 256 * 128;     // activation operand: 256 routes x 128 bytes
constexpr int kBBytes = 256 * 128;     // decoded operand: 256 weight rows x 128 bytes
constexpr uint64_t kTcWaitNs = 2000000000ull;   // default limit of a pipeline wait
constexpr uint64_t kTcDrainNs = kTcWaitNs / 4;   // limit of a wait for copies in flight after an abort

// Limit (ns) of every pipeline wait of this CTA, from the launch arguments.
static __shared__ uint64_t tc_wait_limit;

// Payload of one stage: 16 tile rows x 4 tiles of 32K bytes.
__host__ __device__ constexpr int tc_wslot_bytes(int kmax) { return 16 * 4 * 32 * kmax; }
// Dynamic shared memory: activation ring, decoded ring, payload ring, the
// epilogue warps' vectors and output staging (plus 1024 bytes to align the base).
__host__ __device__ constexpr int tc_smem_total(int kmax, int sb) {
  return 1024 + kSA * kABytes + sb * kBBytes + kSW * tc_wslot_bytes(kmax) + kTcEpiWarps * (kEvecBytes + kStageBytes);
}

struct TcBars {
  uint64_t full[kSBMax], empty[kSBMax], fullW[kSW], emptyW[kSW], accFull[2], accEmpty[2];
  uint64_t pair[4];  // epilogue warp pairs, one per TMEM lane quarter
  uint64_t never;    // nothing arrives here: the issuer's wait on it runs out (stall_issuer test)
  uint64_t fullU[4], emptyU[4];  // unit ring: the scheduler's picks, read by every role in order
};

// Work unit geometry shared by every role.
template <int PROJ, int NR>
struct TcGeom {
  int mblocks, kdim, nst, tiles_k, bi;
  __device__ __forceinline__ explicit TcGeom(const TcArgs& args) {
    const FcArgs& a = args.f;
    bi = (PROJ == 1) ? NR / 2 : 0;
    mblocks = (PROJ == 1) ? a.I / bi : a.H / NR;
    kdim = (PROJ == 1) ? a.H : a.I;
    nst = kdim / kTcKS;
    tiles_k = kdim >> 4;
  }
  // first weight row of tile row tr of block mb
  __device__ __forceinline__ int tile_row0(const FcArgs& a, int mb, int tr) const {
    if (PROJ == 1) {
      const int m = 16 * tr;
      return (m < bi) ? mb * bi + m : a.I + mb * bi + (m - bi);
    }
    return mb * NR + 16 * tr;
  }
};

// Window of a run for any K from a tile in shared memory (see run_window_generic).
template <int K>
__device__ __forceinline__ void run_window_smem(const uint16_t* tile, int j0, uint32_t& hi, uint32_t& lo, int& off) {
  constexpr int NB = 256 * K;
  constexpr int NW = 16 * K;
  int q0 = (j0 + 1) * K - 16;
  if (q0 < 0) q0 += NB;
  const int w = q0 >> 4;
  off = q0 & 15;
  const uint32_t w0 = tile[w], w1 = tile[(w + 1) % NW], w2 = tile[(w + 2) % NW], w3 = tile[(w + 3) % NW];
  hi = (w0 << 16) | w1;
  lo = (w2 << 16) | w3;
}

// 2^(u - 127) as an fp16 pair for a UE8M0 byte u with u - 127 in [-15, 13]
// (the prepared layer guarantees the range; 2^-15 is an fp16 subnormal).
__device__ __forceinline__ uint32_t ue8m0_half2(uint32_t u) {
  const int k = (int)u - 127;
  const uint32_t h = (k >= -14) ? ((uint32_t)(k + 15) << 10) : 0x0200u;
  return h | (h << 16);
}

// TrellisMX-style weights for the fp16 contraction: each codebook value
// rounded to E4M3, times its block's power of two. Both steps are exact in
// fp16 (E4M3 values carry 4 significant bits, |E4M3(cb)| <= 4 and the
// exponent lies in [-15, 13]).
__device__ __forceinline__ void mx_scale(uint32_t (&w)[4], uint32_t f2) {
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const uint32_t q = e4m3x2_to_f16x2(cvt_e4m3x2(w[p]));
    __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&q), *reinterpret_cast<const __half2*>(&f2));
    w[p] = *reinterpret_cast<uint32_t*>(&r);
  }
}

__device__ __forceinline__ void sts128(unsigned char* p, const uint32_t (&w)[4]) {
  *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}

// Expand one stage: NR weight rows x 64 columns from the payload slot `wsl`
// (tile row tr of the stage at tr * 4 * 32K bytes, its 4 tiles contiguous)
// into the swizzled operand `bsl`. Thread t takes row t % NR and 8 * NR / 256
// of the row's 8 chunks of 8 columns; chunk c of a row is run (tile c / 2,
// half c % 2) of the row's trellis tiles.
// MX: `ws` points at the thread's weight row's UE8M0 bytes for this stage
// (two 32-column blocks).
template <int NR, int K, bool MX>
__device__ __forceinline__ void tc_expand_stage(const unsigned char* wsl, unsigned char* bsl, int tid,
                                                uint32_t k16, uint32_t nk16, const uint8_t* ws) {
  constexpr int CPT = 8 * NR / 256;
  const int n = tid % NR;
  const int c0 = (tid / NR) * CPT;
  const int rr = n & 15;
  const unsigned char* trow = wsl + (n >> 4) * 4 * 32 * K;
  unsigned char* brow = bsl + (n >> 3) * 1024 + (n & 7) * 128;
  const uint32_t sw = (uint32_t)(n & 7);
  uint32_t f2[2] = {0u, 0u};
  if (MX) {
    const uint32_t sb = __ldg(reinterpret_cast<const uint16_t*>(ws));
    f2[0] = ue8m0_half2(sb & 0xFFu);
    f2[1] = ue8m0_half2(sb >> 8);
  }
  if (K == 4) {
    // A K=4 tile row rr is the 32-bit words 2rr (first 8 weights) and 2rr+1;
    // a run also needs the word before it, which for the first half is the
    // previous row's second word (row 15's for row 0), held by lane-1 (lane+15).
    const int lane = tid & 31;
    const int src = (lane & 16) | ((lane + 15) & 15);
#pragma unroll
    for (int tt = 0; tt < CPT / 2; ++tt) {
      const int t = c0 / 2 + tt;
      const uint2 cw = *reinterpret_cast<const uint2*>(trow + t * 128 + 8 * rr);
      const uint32_t pw = __shfl_sync(0xFFFFFFFFu, cw.y, src);
      uint32_t y[8], w[4];
      run_mcg_k4(pw, cw.x, k16, nk16, y);
      raw_to_f16(y, w);
      if (MX) mx_scale(w, f2[t >> 1]);
      sts128(brow + (((uint32_t)(2 * t) ^ sw) << 4), w);
      run_mcg_k4(cw.x, cw.y, k16, nk16, y);
      raw_to_f16(y, w);
      if (MX) mx_scale(w, f2[t >> 1]);
      sts128(brow + (((uint32_t)(2 * t + 1) ^ sw) << 4), w);
    }
  } else {
#pragma unroll
    for (int cc = 0; cc < CPT; ++cc) {
      const int c = c0 + cc;
      uint32_t hi, lo, s8[8], y[8], w[4];
      int off;
      run_window_smem<K>(reinterpret_cast<const uint16_t*>(trow + (c >> 1) * 32 * K), 16 * rr + 8 * (c & 1), hi, lo,
                         off);
      run_states_generic<K>(hi, lo, off, s8);
#pragma unroll
      for (int q = 0; q < 8; ++q) y[q] = mcg_raw(s8[q]);
      raw_to_f16(y, w);
      if (MX) mx_scale(w, f2[c >> 2]);
      sts128(brow + (((uint32_t)c ^ sw) << 4), w);
    }
  }
}

// Bounded wait used while draining after an abort (ignores the abort flag).
__device__ __forceinline__ void mbar_wait_drain(uint64_t* mbar, uint32_t parity) {
  const uint32_t a = smem_u32(mbar);
  const uint64_t t0 = global_ns();
  while (!mbar_try(a, parity) && global_ns() - t0 < kTcDrainNs) {
  }
}

// ---------------------------------------------------------------------------
// Epilogues: the calling thread owns one route (one TMEM lane) and the unit's
// N accumulator columns. All TMEM accesses are warp-collective; only threads
// of valid routes store.
// ---------------------------------------------------------------------------
// L (a multiple of 32) accumulator columns of this thread's TMEM lane into
// column pairs (warp-collective): every load in flight before the one wait.
template <int L>
__device__ __forceinline__ void ld_cols2(uint32_t taddr, float2 (&w)[L / 2]) {
  uint32_t r[L / 32][32];
#pragma unroll
  for (int j = 0; j < L / 32; ++j) tmem_ld32(taddr + 32 * j, r[j]);
  tmem_ld_wait();
#pragma unroll
  for (int j = 0; j < L / 32; ++j) {
    reg_fence32(r[j]);
#pragma unroll
    for (int i = 0; i < 16; ++i) w[16 * j + i] = make_float2(__uint_as_float(r[j][2 * i]), __uint_as_float(r[j][2 * i + 1]));
  }
}
template <int L>
__device__ __forceinline__ void st_cols2(uint32_t taddr, const float2 (&w)[L / 2]) {
#pragma unroll
  for (int j = 0; j < L / 32; ++j) {
    uint32_t r[32];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      r[2 * i] = __float_as_uint(w[16 * j + i].x);
      r[2 * i + 1] = __float_as_uint(w[16 * j + i].y);
    }
    tmem_st32(taddr + 32 * j, r);
  }
  tmem_st_wait();
}

// Block FWHT (blocks of B <= L, natural order, unnormalised) on L values held
// as pairs: the distance-1 level inside each pair, every wider level on whole
// pairs with packed fp32 adds.
template <int L>
__device__ __forceinline__ void fwht2(float2 (&w)[L / 2], int B) {
  if (B > 1) {
#pragma unroll
    for (int j = 0; j < L / 2; ++j) w[j] = make_float2(w[j].x + w[j].y, w[j].x - w[j].y);
  }
  const float2 m1 = make_float2(-1.0f, -1.0f);
#pragma unroll
  for (int h = 1; h < L / 2; h <<= 1) {  // pair distance h = element distance 2h
    if (2 * h < B) {
#pragma unroll
      for (int j = 0; j < L / 2; ++j) {
        if ((j & h) == 0) {
          const float2 x = w[j], y = w[j + h];
          w[j] = __fadd2_rn(x, y);
          w[j + h] = __ffma2_rn(y, m1, x);
        }
      }
    }
  }
}

// w[j] *= f[j] for L fp32 factors in shared memory (16-byte aligned).
template <int L>
__device__ __forceinline__ void scale2(float2 (&w)[L / 2], const float* f) {
#pragma unroll
  for (int j = 0; j < L / 2; j += 2) {
    const float4 q = *reinterpret_cast<const float4*>(f + 2 * j);
    w[j] = __fmul2_rn(w[j], make_float2(q.x, q.y));
    w[j + 1] = __fmul2_rn(w[j + 1], make_float2(q.z, q.w));
  }
}

__device__ __forceinline__ float tanh_fast(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// SiLU(g) = g * sigmoid(g) = h * (1 + tanh(h)) with h = g / 2.
__device__ __forceinline__ float2 silu2(float2 g) {
  const float2 h = __fmul2_rn(g, make_float2(0.5f, 0.5f));
  return __ffma2_rn(h, make_float2(tanh_fast(h.x), tanh_fast(h.y)), h);
}

// Coalesced row stores through the warp's staging area: lane l holds 16
// words of row l (destination base + row_l * stride words, row_l < 0: not
// stored); each store instruction then writes 64 contiguous bytes of 8 rows.
// The 20-word row stride keeps the 16-byte writes conflict-free; reading rows
// r and r + 4 in each group of 8 lanes keeps the reads conflict-free.
__device__ __forceinline__ void stage_store16(uint32_t* stg, const uint32_t (&v)[16], uint32_t* base, size_t stride,
                                              int row) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 0; j < 16; j += 4)
    *reinterpret_cast<uint4*>(stg + lane * kStageWords + j) = make_uint4(v[j], v[j + 1], v[j + 2], v[j + 3]);
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = 8 * i + ((lane >> 2) & 1) * 4 + (lane >> 3), qd = lane & 3;
    const int rw = __shfl_sync(0xFFFFFFFFu, row, r);
    const uint4 x = *reinterpret_cast<const uint4*>(stg + r * kStageWords + 4 * qd);
    if (rw >= 0) *reinterpret_cast<uint4*>(base + (size_t)rw * stride + 4 * qd) = x;
  }
  __syncwarp();
}

// The two epilogue warps of a TMEM lane quarter split every block of columns
// in halves; a rotation block wider than a half needs its last butterfly
// level across the pair, exchanged through tensor memory around a bounded
// two-warp barrier.
struct PairSync {
  uint64_t* bar;
  int phase;
};
__device__ __forceinline__ bool pair_sync(PairSync& p, volatile int* abort) {
  tmem_st_wait();  // this warp's tensor-memory stores are complete
  tc_fence_before();
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(p.bar);
  const bool ok = mbar_wait_abort_lim(p.bar, p.phase & 1, abort, &tc_wait_limit);
  ++p.phase;
  tc_fence_after();
  return __all_sync(0xFFFFFFFFu, ok);
}

// Last butterfly level with the partner's half at `theirs` (TMEM columns):
// the lower warp keeps mine + theirs, the upper theirs - mine.
template <int HF>
__device__ __forceinline__ void combine_half(float2 (&w)[HF / 2], uint32_t theirs, int h) {
  const float2 m1 = make_float2(-1.0f, -1.0f);
#pragma unroll
  for (int c = 0; c < HF; c += 32) {
    float2 t[16];
    ld_cols2<32>(theirs + c, t);
#pragma unroll
    for (int j = 0; j < 16; ++j)
      w[c / 2 + j] = (h == 0) ? __fadd2_rn(w[c / 2 + j], t[j]) : __ffma2_rn(w[c / 2 + j], m1, t[j]);
  }
}

// FC1, half h of the route's gate and up columns (HF = BI / 2 each). Gate ->
// scale, H, hs * svh, SiLU; up -> scale, H, hs * svh * suh_down, times
// SiLU(gate); H; hs; this half of the z~ row (fp16). Tensor-memory plan for
// the exchange case: each warp publishes its half in place, reads the
// partner's, then parks SiLU(gate) in the partner's gate half (which only it
// reads from then on) and later publishes its final half there too.
// ev (fp32, HF each): gate scale, hs * gate svh, up scale, hs * up svh * down suh.
template <int BI>
__device__ __forceinline__ bool tc_epi_fc1(const FcArgs& a, const float* ev, uint32_t* stg, int mb, int slot, bool valid,
                                           uint32_t tg, int h, PairSync& ps, volatile int* abort) {
  constexpr int HF = BI / 2;
  const bool xch = a.rot_b > HF;
  const uint32_t mine = h * HF, other = (1 - h) * HF;
  const uint32_t tu = tg + BI;
  const uint32_t park = xch ? other : mine;
  float2 w[HF / 2];
  ld_cols2<HF>(tg + mine, w);
  scale2<HF>(w, ev);
  fwht2<HF>(w, a.rot_b);
  if (xch) {
    st_cols2<HF>(tg + mine, w);
    if (!pair_sync(ps, abort)) return false;
    combine_half<HF>(w, tg + other, h);
  }
  scale2<HF>(w, ev + HF);
#pragma unroll
  for (int j = 0; j < HF / 2; ++j) w[j] = silu2(w[j]);
  st_cols2<HF>(tg + park, w);
  ld_cols2<HF>(tu + mine, w);
  scale2<HF>(w, ev + 2 * HF);
  fwht2<HF>(w, a.rot_b);
  if (xch) {
    st_cols2<HF>(tu + mine, w);
    if (!pair_sync(ps, abort)) return false;
    combine_half<HF>(w, tu + other, h);
  }
  scale2<HF>(w, ev + 3 * HF);
#pragma unroll
  for (int c = 0; c < HF; c += 32) {
    float2 g[16];
    ld_cols2<32>(tg + park + c, g);
#pragma unroll
    for (int j = 0; j < 16; ++j) w[c / 2 + j] = __fmul2_rn(w[c / 2 + j], g[j]);
  }
  fwht2<HF>(w, a.rot_b);
  if (xch) {
    st_cols2<HF>(tg + park, w);
    if (!pair_sync(ps, abort)) return false;
    combine_half<HF>(w, tg + mine, h);
  }
  {
    const float hs = hadamard_scale(a.rot_b);
    const float2 h2s = make_float2(hs, hs);
#pragma unroll
    for (int j = 0; j < HF / 2; ++j) w[j] = __fmul2_rn(w[j], h2s);
    // this half of the z~ row, 32 fp16 (16 words) at a time
    uint32_t* zb = reinterpret_cast<uint32_t*>(reinterpret_cast<uint16_t*>(a.out_act) + mb * BI + h * HF);
#pragma unroll
    for (int c = 0; c < HF / 2; c += 16) {
      uint32_t pk[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        __half2 h2 = __float22half2_rn(w[c + i]);
        pk[i] = *reinterpret_cast<uint32_t*>(&h2);
      }
      stage_store16(stg, pk, zb + c, (size_t)a.I / 2, valid ? slot : -1);
    }
  }
  return true;
}

// FC2, half h of each 128-column block of the route's NR output columns:
// scale and the Hadamard levels within the half into the slot's fp32 row
// (raw_rows: the combine finishes the route), or scale, H, hs * down_svh,
// then the fp32 row of the slot or weighted atomics into the token's output row.
// ev (fp32): per block, 64 output scales then 64 values hs * down_svh.
template <int NR>
__device__ __forceinline__ bool tc_epi_fc2(const FcArgs& a, const float* ev, uint32_t* stg, int mb, int slot, int route,
                                           bool valid, uint32_t tb, int h, PairSync& ps, volatile int* abort) {
  const float wr = (valid && a.atomic) ? a.route_w[route] : 0.0f;
  const uint32_t mine = h * 64, other = (1 - h) * 64;
  if (a.raw_rows) {
    // this half of each 128-column block: scale, then the Hadamard levels
    // inside the half (all of them for blocks of 64); the combine applies the
    // level across halves and hs * down_svh
#pragma unroll 1
    for (int blk = 0; blk < NR / 128; ++blk) {
      float2 w[32];
      ld_cols2<64>(tb + blk * 128 + mine, w);
      scale2<64>(w, ev + blk * 128);
      fwht2<64>(w, a.rot_b > 64 ? 64 : a.rot_b);
      uint32_t* ob = reinterpret_cast<uint32_t*>(a.out_f32) + mb * NR + blk * 128 + h * 64;
#pragma unroll
      for (int c = 0; c < 32; c += 8) {
        uint32_t v16[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          v16[2 * i] = __float_as_uint(w[c + i].x);
          v16[2 * i + 1] = __float_as_uint(w[c + i].y);
        }
        stage_store16(stg, v16, ob + 2 * c, (size_t)a.H, valid ? slot : -1);
      }
    }
    return true;
  }
#pragma unroll 1
  for (int blk = 0; blk < NR / 128; ++blk) {
    const uint32_t t0 = tb + blk * 128;
    float2 w[32];
    ld_cols2<64>(t0 + mine, w);
    scale2<64>(w, ev + blk * 128);
    fwht2<64>(w, a.rot_b);
    if (a.rot_b > 64) {
      st_cols2<64>(t0 + mine, w);
      if (!pair_sync(ps, abort)) return false;
      combine_half<64>(w, t0 + other, h);
    }
    scale2<64>(w, ev + blk * 128 + 64);
    const int col0 = mb * NR + blk * 128 + h * 64;
    if (!a.atomic) {
      // the slot's fp32 row, 16 values at a time through the staging area
      uint32_t* ob = reinterpret_cast<uint32_t*>(a.out_f32) + col0;
#pragma unroll
      for (int c = 0; c < 32; c += 8) {
        uint32_t v16[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          v16[2 * i] = __float_as_uint(w[c + i].x);
          v16[2 * i + 1] = __float_as_uint(w[c + i].y);
        }
        stage_store16(stg, v16, ob + 2 * c, (size_t)a.H, valid ? slot : -1);
      }
    } else if (valid) {
      float* o = a.out_f32 + (size_t)(route / a.topk) * a.H + col0;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        atomicAdd(o + 2 * j, wr * w[j].x);
        atomicAdd(o + 2 * j + 1, wr * w[j].y);
      }
    }
  }
  return true;
}

// ---------------------------------------------------------------------------
// Roles. Every role walks the same unit sequence u = blockIdx.x, +gridDim.x, ...
// and the same global stage counter g, so ring slots and phases agree.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int tc_macc(const TcArgs& args, int slot0) {
  // valid routes are a prefix of the block: a second accumulator iff route 128 exists
  return (args.route_block > 128 && args.f.route_of_slot[slot0 + 128] >= 0) ? 2 : 1;
}

// Unit ring. The payload warp, the first role to need a unit, claims units
// from a device counter (so a CTA that drew cheap units draws more; the claim
// for the next unit is issued one unit early to hide its latency) and
// publishes each pick, -1 when none is left; every other role reads the picks
// in order and frees an entry once read.
constexpr int kUnitRing = 4;
constexpr int kUnitConsumers = 8 + kTcEpiWarps + 2;  // expander warps, epilogue warps, act and issuer threads

// Next unit for a consumer warp (all lanes) or a single consumer thread;
// -1 when the units are done or a wait gave up (then *ok = false).
__device__ __forceinline__ int pop_unit_warp(TcBars& B, volatile int* uring, int& i, volatile int* abort, bool* ok) {
  const int slot = i % kUnitRing;
  const bool w = mbar_wait_abort_lim(&B.fullU[slot], (i / kUnitRing) & 1, abort, &tc_wait_limit);
  if (!__all_sync(0xFFFFFFFFu, w)) {
    *ok = false;
    return -1;
  }
  const int u = uring[slot];
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&B.emptyU[slot]);
  ++i;
  return u;
}
__device__ __forceinline__ int pop_unit_thread(TcBars& B, volatile int* uring, int& i, volatile int* abort, bool* ok) {
  const int slot = i % kUnitRing;
  if (!mbar_wait_abort_lim(&B.fullU[slot], (i / kUnitRing) & 1, abort, &tc_wait_limit)) {
    *ok = false;
    return -1;
  }
  const int u = uring[slot];
  mbar_arrive(&B.emptyU[slot]);
  ++i;
  return u;
}

// Accumulator buffers of a unit: one alternating buffer for <= 128 routes,
// both (acc 0 in buffer 0, acc 1 in buffer 1) for more.
struct TcAccPlan {
  int nb = 0;          // buffer of the next one-accumulator unit
  int uses[2] = {0, 0};
  __device__ __forceinline__ int buf(int macc, int acc) const { return macc == 2 ? acc : nb; }
  __device__ __forceinline__ void advance(int macc) { nb = (macc == 2) ? 0 : (nb ^ 1); }
};

// Fused launch (proj 3): the FC1 units of every route block come first in
// the unit order, then the FC2 units. An FC2 unit's activations are the z~
// rows of its route block, complete once every epilogue warp of each of the
// block's FC1 units has counted itself in dep[rb] (after a device-scope fence
// over its stores). Only FC2 units wait, and only on FC1 units claimed before
// them, whose pipelines wait on nothing outside their CTA: no cycle.
template <int PROJ>
struct TcProj {
  static constexpr int first = PROJ == 3 ? 1 : PROJ;  // projection of the launch's first units
  static constexpr bool fused = PROJ == 3;
};

// Waits (bounded) until *cnt >= target, then orders the acquired z~ rows
// before this thread's later bulk-tensor (async proxy) reads.
__device__ __forceinline__ bool tc_dep_wait(const uint32_t* cnt, uint32_t target, volatile int* abort) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];\n" : "=r"(v) : "l"(cnt) : "memory");
  if (v < target) {
    const uint64_t t0 = global_ns();
    for (;;) {
      __nanosleep(128);
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];\n" : "=r"(v) : "l"(cnt) : "memory");
      if (v >= target) break;
      if (*abort) return false;
      if (global_ns() - t0 > tc_wait_limit) {
        *abort = 1;
        return false;
      }
    }
  }
  asm volatile("fence.proxy.async.global;\n" ::: "memory");
  return true;
}

// One unit's stages on the expander warps; false when a wait gave up.
template <int P, int KB, int NR, bool MX>
__device__ __forceinline__ bool tc_expand_unit(const FcArgs& a, const TcGeom<P, NR>& G, int u, TcBars& B,
                                               const unsigned char* wring, unsigned char* bring, int& g, int& ready,
                                               volatile int* abort) {
  const int tid = threadIdx.x, lane = tid & 31;
  const uint32_t k16 = 0x10000u + (uint32_t)((unsigned)G.nst >> 30), nk16 = 0u - k16;
  const int wsz = tc_wslot_bytes(KB > 0 ? KB : 6);
  constexpr int SB = tc_sb(KB);
  const int rb = u / G.mblocks;
  const int K = (KB > 0) ? KB : a.bits[a.block_expert[rb]];
  // MX: the UE8M0 bytes of this thread's weight row (tc_expand_stage: row tid % NR)
  const uint8_t* wsr = nullptr;
  if (MX) {
    const int mb = u - rb * G.mblocks, n = tid % NR;
    const int row = G.tile_row0(a, mb, n >> 4) + (n & 15);
    wsr = a.wscale + ((size_t)a.block_expert[rb] * a.wrows + row) * a.wcols;
  }
  for (int s = 0; s < G.nst; ++s, ++g) {
    const int ws = g % kSW, bs = g % SB;
    if (g > ready) {
      // the stage's payload slot full and decoded buffer free, tested
      // together; with three decoded buffers also the next stage's (its
      // buffer was released by the MMAs of the stage before this one)
      const bool two = SB >= 3 && s + 1 < G.nst;
      const int g1 = two ? g + 1 : g;
      const uint32_t fw0 = smem_u32(&B.fullW[ws]), fw1 = smem_u32(&B.fullW[g1 % kSW]);
      const uint32_t eb0 = (g >= SB) ? smem_u32(&B.empty[bs]) : fw0;
      const uint32_t eb1 = (g1 >= SB) ? smem_u32(&B.empty[g1 % SB]) : fw1;
      const uint32_t pw0 = (g / kSW) & 1, pw1 = (g1 / kSW) & 1;
      const uint32_t pb0 = (g >= SB) ? ((g / SB) - 1) & 1 : pw0, pb1 = (g1 >= SB) ? ((g1 / SB) - 1) & 1 : pw1;
      if (mbar_test4(fw0, pw0, eb0, pb0, fw1, pw1, eb1, pb1)) {
        ready = g1;
      } else {
        bool okw = mbar_wait_abort_lim(&B.fullW[ws], pw0, abort, &tc_wait_limit);
        if (okw && g >= SB) okw = mbar_wait_abort_lim(&B.empty[bs], pb0, abort, &tc_wait_limit);
        if (!__all_sync(0xFFFFFFFFu, okw)) return false;
        ready = g;
      }
    }
    const unsigned char* wsl = wring + ws * wsz;
    unsigned char* bsl = bring + bs * kBBytes;
    const uint8_t* wss = MX ? wsr + 2 * s : nullptr;
    if (KB > 0) {
      tc_expand_stage<NR, (KB > 0 ? KB : 4), MX>(wsl, bsl, tid, k16, nk16, wss);
    } else {
      switch (K) {
        case 2: tc_expand_stage<NR, 2, MX>(wsl, bsl, tid, k16, nk16, wss); break;
        case 3: tc_expand_stage<NR, 3, MX>(wsl, bsl, tid, k16, nk16, wss); break;
        case 4: tc_expand_stage<NR, 4, MX>(wsl, bsl, tid, k16, nk16, wss); break;
        case 5: tc_expand_stage<NR, 5, MX>(wsl, bsl, tid, k16, nk16, wss); break;
        default: tc_expand_stage<NR, 6, MX>(wsl, bsl, tid, k16, nk16, wss); break;
      }
    }
    fence_proxy_async();  // generic-proxy stores -> visible to the tensor core
    __syncwarp();
    if (lane == 0) {      // one arrival per warp
      mbar_arrive(&B.full[bs]);
      mbar_arrive(&B.emptyW[ws]);
    }
  }
  return true;
}

template <int PROJ, int KB, int NR, bool MX>
__device__ __forceinline__ void tc_expanders(const TcArgs& args, const TcGeom<TcProj<PROJ>::first, NR>& G,
                                             const TcGeom<2, NR>& G2, int U1, volatile int* uring, TcBars& B,
                                             const unsigned char* wring, unsigned char* bring, volatile int* abort) {
  int g = 0, iu = 0, ready = -1;  // stages up to `ready` have their inputs
  bool ok = true;
  // a CTA's units ascend: (fused) its FC1 units, then its FC2 units
  int u = pop_unit_warp(B, uring, iu, abort, &ok);
  for (; u >= 0 && (!TcProj<PROJ>::fused || u < U1); u = pop_unit_warp(B, uring, iu, abort, &ok))
    if (!tc_expand_unit<TcProj<PROJ>::first, KB, NR, MX>(args.f, G, u, B, wring, bring, g, ready, abort)) return;
  if constexpr (TcProj<PROJ>::fused)
    for (; u >= 0; u = pop_unit_warp(B, uring, iu, abort, &ok))
      if (!tc_expand_unit<2, KB, NR, MX>(args.f2, G2, u - U1, B, wring, bring, g, ready, abort)) return;
}

// One unit on an epilogue warp: its vectors, then each accumulator once the
// MMAs have filled it; false when a wait gave up.
template <int P, int KB, int NR>
__device__ __forceinline__ bool tc_epi_unit(const TcArgs& args, const FcArgs& a, const TcGeom<P, NR>& G, int u,
                                            TcBars& B, float* ev, uint32_t* stg, uint32_t tmem, PairSync& ps,
                                            TcAccPlan& plan, volatile int* abort) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = warp & 3;           // TMEM lane quarter
  const int h = (warp - 8) >> 2;    // column half
  const int rb = u / G.mblocks, mb = u - rb * G.mblocks;
  const int e = a.block_expert[rb];
  const int slot0 = rb * args.route_block;
  const int macc = tc_macc(args, slot0);
  // this warp's half of the unit's vectors, converted to fp32 and folded
  // (its reads of the last unit are done)
  __syncwarp();
  {
    const float hs = hadamard_scale(a.rot_b);
    if (P == 1) {
      const int bi = NR / 2, hf = bi / 2, c0 = mb * bi + h * hf;
      const uint16_t* s1 = a.scale + (size_t)e * 2 * a.I + c0;
      const uint16_t* rt = a.rot_tab + (size_t)e * 3 * a.I + c0;
      for (int c = lane; c < hf; c += 32) {
        ev[c] = __half2float(__ushort_as_half(s1[c]));
        ev[hf + c] = hs * __half2float(__ushort_as_half(rt[c]));
        ev[2 * hf + c] = __half2float(__ushort_as_half(s1[a.I + c]));
        ev[3 * hf + c] = hs * __half2float(__ushort_as_half(rt[a.I + c])) * __half2float(__ushort_as_half(rt[2 * a.I + c]));
      }
    } else {
      const uint16_t* s2 = a.scale + (size_t)e * a.H + mb * NR;
      const uint16_t* sv = a.rot_tab + (size_t)e * a.H + mb * NR;
      for (int i = lane; i < NR / 2; i += 32) {
        const int blk = i >> 6, c = blk * 128 + h * 64 + (i & 63);
        ev[blk * 128 + (i & 63)] = __half2float(__ushort_as_half(s2[c]));
        ev[blk * 128 + 64 + (i & 63)] = hs * __half2float(__ushort_as_half(sv[c]));
      }
    }
  }
  __syncwarp();
  for (int acc = 0; acc < macc; ++acc) {
    const int b = plan.buf(macc, acc);
    const bool ok = mbar_wait_abort_lim(&B.accFull[b], plan.uses[b] & 1, abort, &tc_wait_limit);
    if (!__all_sync(0xFFFFFFFFu, ok)) return false;
    tc_fence_after();
    const int n = acc * 128 + 32 * q + lane;
    const int route = a.route_of_slot[slot0 + n];
    const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(b * 256);
    // a lane quarter without valid routes has nothing to store (both warps
    // of the pair see the same lanes, so they skip together)
    if (__any_sync(0xFFFFFFFFu, route >= 0)) {
      const bool done = (P == 1) ? tc_epi_fc1<NR / 2>(a, ev, stg, mb, slot0 + n, route >= 0, taddr, h, ps, abort)
                                 : tc_epi_fc2<NR>(a, ev, stg, mb, slot0 + n, route, route >= 0, taddr, h, ps, abort);
      if (!done) return false;
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&B.accEmpty[b]);
    plan.uses[b]++;
  }
  plan.advance(macc);
  return true;
}

template <int PROJ, int KB, int NR>
__device__ __forceinline__ void tc_epilogue(const TcArgs& args, const TcGeom<TcProj<PROJ>::first, NR>& G,
                                            const TcGeom<2, NR>& G2, int U1, volatile int* uring, TcBars& B, float* ev,
                                            uint32_t* stg, uint32_t tmem, volatile int* abort) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  PairSync ps{&B.pair[warp & 3], 0};
  TcAccPlan plan;
  int iu = 0;
  bool ok = true;
  // a CTA's units ascend: (fused) its FC1 units, then its FC2 units
  int u = pop_unit_warp(B, uring, iu, abort, &ok);
  for (; u >= 0 && (!TcProj<PROJ>::fused || u < U1); u = pop_unit_warp(B, uring, iu, abort, &ok)) {
    if (!tc_epi_unit<TcProj<PROJ>::first, KB, NR>(args, args.f, G, u, B, ev, stg, tmem, ps, plan, abort)) return;
    if constexpr (TcProj<PROJ>::fused) {
      // this warp's z~ rows of the unit are stored: count it for the route block
      __threadfence();
      asm volatile("fence.proxy.async.global;\n" ::: "memory");
      __syncwarp();
      if (lane == 0) asm volatile("red.release.gpu.global.add.u32 [%0], 1;\n" ::"l"(args.dep + u / G.mblocks) : "memory");
    }
  }
  if constexpr (TcProj<PROJ>::fused)
    for (; u >= 0; u = pop_unit_warp(B, uring, iu, abort, &ok))
      if (!tc_epi_unit<2, KB, NR>(args, args.f2, G2, u - U1, B, ev, stg, tmem, ps, plan, abort)) return;
}

// One unit's payload stages (payload warp); false when a wait gave up.
template <int P, int KB, int NR>
__device__ __forceinline__ bool tc_payload_unit(const FcArgs& a, const TcGeom<P, NR>& G, int u, TcBars& B,
                                                unsigned char* wring, int& g, int& gw, volatile int* abort) {
  const int lane = threadIdx.x & 31;
  const int wsz = tc_wslot_bytes(KB > 0 ? KB : 6);
  const int rb = u / G.mblocks, mb = u - rb * G.mblocks;
  const int e = a.block_expert[rb];
  const int K = (KB > 0) ? KB : a.bits[e];
  const uint32_t wbytes = 4 * 32 * K;  // one tile row of a stage
  const uint16_t* wsrc = reinterpret_cast<const uint16_t*>(a.payload);
  if (lane < NR / 16) wsrc += a.word_off[e] + (size_t)(G.tile_row0(a, mb, lane) >> 4) * G.tiles_k * 16 * K;
  for (int s = 0; s < G.nst; ++s, ++g) {
    const int ws = g % kSW;
    const bool okw = (g < kSW) || mbar_wait_abort_lim(&B.emptyW[ws], ((g / kSW) - 1) & 1, abort, &tc_wait_limit);
    if (!__all_sync(0xFFFFFFFFu, okw)) return false;
    if (lane == 0) mbar_arrive_expect_tx(&B.fullW[ws], (NR / 16) * wbytes);
    __syncwarp();
    if (lane < NR / 16) bulk_g2s(wring + ws * wsz + lane * wbytes, wsrc + (size_t)s * 4 * 16 * K, wbytes, &B.fullW[ws]);
    gw = g + 1;
  }
  return true;
}

template <int PROJ, int KB, int NR>
__device__ __forceinline__ void tc_payload_loader(const TcArgs& args, const TcGeom<TcProj<PROJ>::first, NR>& G,
                                                  const TcGeom<2, NR>& G2, int U1, int units, volatile int* uring,
                                                  TcBars& B, unsigned char* wring, volatile int* abort) {
  const int lane = threadIdx.x & 31;
  int g = 0, gw = 0;
  bool ok = true;
  uint32_t next = (lane == 0) ? atomicAdd(args.sched, 1u) : 0u;
  for (int iu = 0;; ++iu) {
    const int slot = iu % kUnitRing;
    if (iu >= kUnitRing) {
      const bool okr = mbar_wait_abort_lim(&B.emptyU[slot], ((iu / kUnitRing) - 1) & 1, abort, &tc_wait_limit);
      if (!__all_sync(0xFFFFFFFFu, okr)) {
        ok = false;
        break;
      }
    }
    const uint32_t claimed = __shfl_sync(0xFFFFFFFFu, next, 0);
    const int u = (claimed < (uint32_t)units) ? (int)claimed : -1;
    if (lane == 0) {
      uring[slot] = u;
      mbar_arrive(&B.fullU[slot]);  // release: the pick is visible to the waiters
      if (u >= 0) next = atomicAdd(args.sched, 1u);
    }
    if (u < 0) break;
    if constexpr (TcProj<PROJ>::fused) {
      if (u >= U1) {
        ok = tc_payload_unit<2, KB, NR>(args.f2, G2, u - U1, B, wring, g, gw, abort);
        if (!ok) break;
        continue;
      }
    }
    ok = tc_payload_unit<TcProj<PROJ>::first, KB, NR>(args.f, G, u, B, wring, g, gw, abort);
    if (!ok) break;
  }
  if (!ok && lane == 0)  // copies in flight land before the CTA exits
    for (int gg = (gw > kSW ? gw - kSW : 0); gg < gw; ++gg) mbar_wait_drain(&B.fullW[gg % kSW], (gg / kSW) & 1);
}

// TMA load of a 64-column x 128-row box of the activations (slot order) into
// the swizzled operand.
__device__ __forceinline__ void tma_tile2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* mbar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n"
      ::"r"(smem_u32(dst)), "l"(map), "r"(x), "r"(y), "r"(smem_u32(mbar))
      : "memory");
}

// One unit's activation stages (lane 0 of the activation warp): one box per
// 128 routes. Rows of padding routes hold whatever the slot holds; they only
// reach accumulator rows that no epilogue stores. False when a wait gave up.
template <int P, int KB, int NR, bool SPLIT>
__device__ __forceinline__ bool tc_act_unit(const TcArgs& args, const CUtensorMap* map, const TcGeom<P, NR>& G, int u,
                                            TcBars& B, unsigned char* aring, int& g, int& ga, volatile int* abort) {
  constexpr int SB = tc_sb(KB);
  static_assert(kSA <= SB, "the activation ring must not be deeper than the decoded ring");
  const int slot0 = (u / G.mblocks) * args.route_block;
  const int macc = tc_macc(args, slot0);
  constexpr bool split = SPLIT;  // separate gate / up operands (route blocks of 128: one accumulator)
  for (int s = 0; s < G.nst; ++s, ++g) {
    const int as = g % kSA;
    uint64_t* fb = &B.full[g % SB];
    // the slot's previous stage, g - kSA, has completed its MMAs
    if (g >= kSA && !mbar_wait_abort_lim(&B.empty[(g - kSA) % SB], ((g - kSA) / SB) & 1, abort, &tc_wait_limit))
      return false;
    mbar_arrive_expect_tx(fb, (uint32_t)(split ? 2 : macc) * 128 * 128);
    unsigned char* dst = aring + as * kABytes;
    tma_tile2d(dst, map, s * kTcKS, slot0, fb);
    if constexpr (split)  // the up rows' operand in the second half
      tma_tile2d(dst + 128 * 128, &args.amap2, s * kTcKS, slot0, fb);
    else if (macc == 2)
      tma_tile2d(dst + 128 * 128, map, s * kTcKS, slot0 + 128, fb);
    ga = g + 1;
  }
  return true;
}

template <int PROJ, int KB, int NR, bool SPLIT>
__device__ __forceinline__ void tc_act_loader(const TcArgs& args, const TcGeom<TcProj<PROJ>::first, NR>& G,
                                              const TcGeom<2, NR>& G2, int U1, volatile int* uring, TcBars& B,
                                              unsigned char* aring, volatile int* abort) {
  constexpr int SB = tc_sb(KB);
  int g = 0, ga = 0, iu = 0;
  bool ok = true;
  // a CTA's units ascend: (fused) its FC1 units, then its FC2 units
  int u = pop_unit_thread(B, uring, iu, abort, &ok);
  while (ok && u >= 0 && (!TcProj<PROJ>::fused || u < U1)) {
    ok = tc_act_unit<TcProj<PROJ>::first, KB, NR, SPLIT>(args, &args.amap, G, u, B, aring, g, ga, abort);
    if (ok) u = pop_unit_thread(B, uring, iu, abort, &ok);
  }
  if constexpr (TcProj<PROJ>::fused) {
    while (ok && u >= 0) {
      const int v = u - U1;
      // the route block's z~ rows: every epilogue warp of its FC1 units
      ok = tc_dep_wait(args.dep + v / G2.mblocks, (uint32_t)(G.mblocks * kTcEpiWarps), abort) &&
           tc_act_unit<2, KB, NR, false>(args, &args.amapz, G2, v, B, aring, g, ga, abort);
      if (ok) u = pop_unit_thread(B, uring, iu, abort, &ok);
    }
  }
  // copies in flight land before the CTA exits (their stage barrier also
  // counts the expanders' arrivals, so after an abort elsewhere this wait
  // can run to its limit)
  if (!ok)
    for (int gg = (ga > kSA ? ga - kSA : 0); gg < ga; ++gg) mbar_wait_drain(&B.full[gg % SB], (gg / SB) & 1);
}

template <int PROJ, int KB, int NR, bool SPLIT>
__device__ __forceinline__ void tc_issuer(const TcArgs& args, const TcGeom<TcProj<PROJ>::first, NR>& G,
                                          const TcGeom<2, NR>& G2, int U1, volatile int* uring, TcBars& B,
                                          const unsigned char* aring, const unsigned char* bring, uint32_t tmem,
                                          volatile int* abort) {
  const uint32_t idesc = idesc_f16(128, NR);
  const uint32_t idesc_half = idesc_f16(128, NR / 2);
  constexpr bool split = SPLIT;
  const uint64_t adesc0 = smem_desc_sw128(smem_u32(aring));
  const uint64_t bdesc0 = smem_desc_sw128(smem_u32(bring));
  TcAccPlan plan;
  int g = 0, glast = -1, iu = 0;
  bool ok = true;
  // test of the bounded waits: a wait that nothing ends, before any MMA is
  // issued, so that the CTA aborts with only completed copies behind it
  if (args.stall_issuer && !mbar_wait_abort_lim(&B.never, 0, abort, &tc_wait_limit)) return;
  for (int u; ok && (u = pop_unit_thread(B, uring, iu, abort, &ok)) >= 0;) {
    int rb = u / G.mblocks, nst = G.nst;
    if (TcProj<PROJ>::fused && u >= U1) {
      rb = (u - U1) / G2.mblocks;
      nst = G2.nst;
    }
    const int macc = tc_macc(args, rb * args.route_block);
    for (int acc = 0; acc < macc && ok; ++acc) {  // the unit's buffers drained by the epilogue
      const int b = plan.buf(macc, acc);
      if (plan.uses[b] > 0) ok = mbar_wait_abort_lim(&B.accEmpty[b], (plan.uses[b] - 1) & 1, abort, &tc_wait_limit);
    }
    if (!ok) break;
    tc_fence_after();
    const uint32_t d0 = tmem + (uint32_t)(plan.buf(macc, 0) * 256);
    for (int s = 0; s < nst; ++s, ++g) {
      const int as = g % kSA, bs = g % tc_sb(KB);
      if (!mbar_wait_abort_lim(&B.full[bs], (g / tc_sb(KB)) & 1, abort, &tc_wait_limit)) {
        ok = false;
        break;
      }
      // (each expander warp fenced its stores to the async proxy before arriving)
      tc_fence_after();
      const uint64_t ad = adesc0 + (uint64_t)(as * (kABytes >> 4));
      const uint64_t bd = bdesc0 + (uint64_t)(bs * (kBBytes >> 4));
      if constexpr (split) {
        // gate rows (decoded rows 0..NR/2-1) x the gate operand into columns
        // 0..NR/2-1, up rows x the up operand (second half of the A slot)
        // into columns NR/2..NR-1
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint32_t accum = (s > 0 || kk > 0) ? 1u : 0u;
          tc_mma_f16(d0, ad + 2 * kk, bd + 2 * kk, idesc_half, accum);
          tc_mma_f16(d0 + NR / 2, ad + 1024 + 2 * kk, bd + (uint64_t)(NR / 2 * 128 >> 4) + 2 * kk, idesc_half,
                     accum);
        }
      } else {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint32_t accum = (s > 0 || kk > 0) ? 1u : 0u;
          tc_mma_f16(d0, ad + 2 * kk, bd + 2 * kk, idesc, accum);
          if (macc == 2) tc_mma_f16(tmem + 256, ad + 1024 + 2 * kk, bd + 2 * kk, idesc, accum);
        }
      }
      tc_commit(&B.empty[bs]);
      glast = g;
    }
    if (!ok) break;
    for (int acc = 0; acc < macc; ++acc) {
      const int b = plan.buf(macc, acc);
      tc_commit(&B.accFull[b]);
      plan.uses[b]++;
    }
    plan.advance(macc);
  }
  if (*abort && glast >= 0) mbar_wait_drain(&B.empty[glast % tc_sb(KB)], (glast / tc_sb(KB)) & 1);
}

template <int N>
__device__ __forceinline__ void regs_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(N)); }
template <int N>
__device__ __forceinline__ void regs_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(N)); }

template <int PROJ, int KB, int NR, bool MX, bool SPLIT>
__global__ void __launch_bounds__(kTcThreads, 1) k_tc_fc(const __grid_constant__ TcArgs args) {
  extern __shared__ unsigned char tc_smem_raw[];
  __shared__ __align__(8) TcBars bars;
  __shared__ uint32_t tmem_slot;
  __shared__ int s_abort;
  __shared__ int s_uring[kUnitRing];
  constexpr int kmax = KB > 0 ? KB : 6;
  static_assert(tc_smem_total(kmax, tc_sb(KB)) + 1024 <= 232448, "dynamic + static shared memory over the per-block limit");
  unsigned char* smem = tc_smem_raw + ((1024u - (smem_u32(tc_smem_raw) & 1023u)) & 1023u);
  unsigned char* aring = smem;
  unsigned char* bring = aring + kSA * kABytes;
  unsigned char* wring = bring + tc_sb(KB) * kBBytes;
  unsigned char* evec = wring + kSW * tc_wslot_bytes(kmax);
  const int tid = threadIdx.x, warp = tid >> 5;
  const TcGeom<TcProj<PROJ>::first, NR> G(args);
  const TcGeom<2, NR> G2(args);  // (fused launch: the FC2 units)
  if (tid == 0) {
    for (int i = 0; i < tc_sb(KB); ++i) {
      mbar_init(&bars.full[i], kTcExp / 32 + 1);  // expander warps + the activation loader's expect_tx
      mbar_init(&bars.empty[i], 1);
    }
    for (int i = 0; i < kSW; ++i) {
      mbar_init(&bars.fullW[i], 1);
      mbar_init(&bars.emptyW[i], kTcExp / 32);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.accFull[i], 1);
      mbar_init(&bars.accEmpty[i], kTcEpiWarps);
    }
    for (int i = 0; i < 4; ++i) mbar_init(&bars.pair[i], 2);
    mbar_init(&bars.never, 1);
    tc_wait_limit = args.wait_ns ? args.wait_ns : kTcWaitNs;
    for (int i = 0; i < kUnitRing; ++i) {
      mbar_init(&bars.fullU[i], 1);
      mbar_init(&bars.emptyU[i], kUnitConsumers);
    }
    s_abort = 0;
    mbar_fence_init();
  }
  if (warp == 0) tmem_alloc(&tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const int U1 = *args.f.nblocks * G.mblocks;  // (fused launch: the FC1 units, then the FC2 units)
  const int units = TcProj<PROJ>::fused ? U1 + *args.f.nblocks * G2.mblocks : U1;
  const uint32_t tmem = tmem_slot;
  volatile int* abort = &s_abort;
  volatile int* uring = s_uring;
  if (warp < 8) {
    if (TcRegs<KB>::exp < kRegLaunch) regs_dec<TcRegs<KB>::exp>();
    tc_expanders<PROJ, KB, NR, MX>(args, G, G2, U1, uring, bars, wring, bring, abort);
  } else if (warp < 16) {
    regs_inc<TcRegs<KB>::epi>();
    tc_epilogue<PROJ, KB, NR>(args, G, G2, U1, uring, bars, reinterpret_cast<float*>(evec + (warp - 8) * kEvecBytes),
                              reinterpret_cast<uint32_t*>(evec + kTcEpiWarps * kEvecBytes + (warp - 8) * kStageBytes),
                              tmem, abort);
  } else {
    regs_dec<kRegAux>();
    if (warp == 16)
      tc_payload_loader<PROJ, KB, NR>(args, G, G2, U1, units, uring, bars, wring, abort);
    else if (warp == 17 && (tid & 31) == 0)
      tc_act_loader<PROJ, KB, NR, SPLIT>(args, G, G2, U1, uring, bars, aring, abort);
    else if (warp == 18 && (tid & 31) == 0)
      tc_issuer<PROJ, KB, NR, SPLIT>(args, G, G2, U1, uring, bars, aring, bring, tmem, abort);
  }
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort) atomicOr(args.err, 2u);
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

template <int PROJ, int KB, int NR, bool MX = false, bool SPLIT = false>
static cudaError_t launch_tc_t(const TcArgs& args, int max_blocks, cudaStream_t st) {
  auto kern = k_tc_fc<PROJ, KB, NR, MX, SPLIT>;
  constexpr int kmax = KB > 0 ? KB : 6;
  static_assert(tc_smem_total(kmax, tc_sb(KB)) + 1024 <= 232448, "dynamic + static shared memory over the per-block limit");
  static bool attr_done = false;  // first forward call, before any capture
  if (!attr_done) {
    cudaFuncAttributes fa;
    cudaError_t err = cudaFuncGetAttributes(&fa, kern);
    if (err != cudaSuccess) return err;
    if (fa.numRegs != kRegLaunch) return cudaErrorInvalidConfiguration;  // the register split assumes 128
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, tc_smem_total(kmax, tc_sb(KB)));
    if (err != cudaSuccess) return err;
    attr_done = true;
  }
  int dev = 0, sms = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err == cudaSuccess) err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return err;
  const int mblocks = (PROJ == 1) ? args.f.I / args.bi : (PROJ == 2) ? args.f.H / NR : args.f.I / args.bi + args.f.H / NR;
  const long units = (long)max_blocks * mblocks;
  const int grid = (int)std::max<long>(1, std::min<long>(units, sms));
  kern<<<grid, kTcThreads, tc_smem_total(kmax, tc_sb(KB)), st>>>(args);
  return cudaGetLastError();
}

// One launch of the variant for the layer: TrellisMX-style weights take the
// general-K kernel with the scale step, else the K=4 or the general-K kernel.
template <int PROJ, int NR, bool SPLIT>
static cudaError_t tc_pick(const TcArgs& args, int uniform_k, int max_blocks, cudaStream_t st) {
  if (args.f.wscale) return launch_tc_t<PROJ, 0, NR, true, SPLIT>(args, max_blocks, st);
  if (uniform_k == 4) return launch_tc_t<PROJ, 4, NR, false, SPLIT>(args, max_blocks, st);
  return launch_tc_t<PROJ, 0, NR, false, SPLIT>(args, max_blocks, st);
}

}  // namespace tmoe
