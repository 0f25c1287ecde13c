// Decode-rows FC1 / FC2 (sm_103a): persistent, warp-granular kernels for the
// few-token regime, where every touched expert serves a handful of routes and
// the layer is bound by expanding the touched trellis payload (b12x PR #129
// "feat(moe): serve canonical Fruit QSRT atoms", Hot path: W4A8 only for
// bounded decode rows; the payload is expanded straight into MMA operands).
//
// Work item = (route block rb of 8 slots, 16-row strip, segment of 256
// contraction columns, or of 512 for K=4 layers from kDecWideRoutes routes
// on, where fewer and longer items halve the per-item bookkeeping). Warp w of
// the grid takes items w, w + W, w + 2W, ... (W warps in all; items cost the
// same, so no claiming is needed). It copies each item's 16 (32) payload
// tiles (one K-bit trellis tile holds 16x16 weights) into a private two-slot
// shared ring with cp.async -- the copy of the next item overlaps the
// expansion of this one -- expands the tiles in registers into fp16 mma.sync
// operands and multiplies them with the block's activation fragments, read
// straight from L2. W4A8: weights are rounded to E4M3 and activations are
// E4M3 codes held exactly in fp16, so each 32-column MMA result is exact up
// to summation order and is scaled by the route's E8M0 block exponent
// (mma.sync of E4M3 operands is not a native tensor instruction on sm_103).
// The 16x8 partial sums of an item go to the workspace.
//
// The epilogue kernels that follow sum each item's partials in segment order
// (deterministic). FC1, one warp per (epilogue unit, slot): the activation
// H -> svh -> SiLU(gate)*up -> suh_down -> H into z~ (sparkinfer PR #90,
// review of kernel.py: _run_activation). FC2, one CTA per (token, 128
// columns), a warp per route: the unrotation (H, down_svh) times the route
// weight into shared memory, then the top-k combine in route order. No CTA
// waits on another.
//
// Two expansion variants: the codebook hash in registers (several four-warp
// CTAs per SM; the default), or one shared-memory table lookup per weight
// (the full-codeword lookup table that b12x PR #129's commit notes split out
// for separate review; one CTA per SM whose warps share the 128 KB table,
// copied from the layer's device copy at kernel start). The table trades the
// hash's integer, fp16-add and E4M3-conversion instructions for one shared
// load, whose random bank conflicts make it the slower of the two here.
#include <algorithm>

#include "launch.h"

namespace tmoe {

constexpr int kDwThreads = 128;          // four independent warps
constexpr int kDwWarps = kDwThreads / 32;
constexpr int kDwSteps = kDecSeg / 32;   // k-steps (two tiles each) per kDecSeg columns
constexpr int kDwTiles = kDecSeg / 16;   // payload tiles per kDecSeg columns
constexpr int kDwRing = 2;

__device__ __forceinline__ void dw_griddep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void dw_griddep_launch() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

// Per-warp metadata of one route block: lanes 0..7 load the slots' routes,
// lane 8 the block's expert | bits << 16 | valid slots << 24, lane 9 the byte
// offset of the expert's payload; dw_meta_final broadcasts them. Issued two
// items ahead of use so that the loads overlap an item's expansion.
struct DwRaw {
  int v;
  long long o;
};
struct DwMetaW {
  int row;  // lane n < 8: activation row of slot n (FC1 token, or route with split signs; FC2 slot), -1 if empty
  int ek;
  long long off;
};

__device__ __forceinline__ DwRaw dw_meta_issue(const DecArgs& d, int rb, int lane) {
  DwRaw r{-1, 0};
  if (lane < kDecBlock)
    r.v = d.f.route_of_slot[rb * kDecBlock + lane];
  else if (lane == kDecBlock)
    r.v = d.blk_meta[rb];
  else if (lane == kDecBlock + 1)
    r.o = d.blk_off[rb];
  return r;
}

template <int PROJ>
__device__ __forceinline__ DwMetaW dw_meta_final(const DwRaw& r, int rb, int lane, int topk, int split) {
  DwMetaW m;
  m.ek = __shfl_sync(0xFFFFFFFFu, r.v, kDecBlock);
  m.off = __shfl_sync(0xFFFFFFFFu, r.o, kDecBlock + 1);
  // FC1: the token's x~ row (the route's own rows with separate gate / up
  // signs); FC2: the slot's z~ row
  m.row = (lane < kDecBlock && r.v >= 0) ? ((PROJ == 1) ? (split ? r.v : r.v / topk) : rb * kDecBlock + lane) : -1;
  return m;
}

__host__ __device__ inline int dw_slot_bytes(int kmax, int segs) { return segs * kDwTiles * 32 * kmax; }

// Codebook lookup table: the fp16 weight of each of the 65,536 trellis states
// (W4A8: of its E4M3 rounding), 128 KB. The lookup variant runs one CTA per
// SM whose warps share the table in shared memory; the procedural variant
// runs several four-warp CTAs per SM.
constexpr int kDwLutEntries = 65536;
constexpr int kDwLutBytes = kDwLutEntries * 2;
// (lookup variant with two-piece items: half the warps, so that the table and
// their rings still fit in one CTA's shared memory)
__host__ __device__ constexpr int dw_cta_warps(int kb, bool lut, int segs = 1) {
  return lut ? (kb > 0 ? 24 : 16) / segs : kDwWarps;
}
__host__ __device__ inline int dw_smem_bytes(int kmax, bool lut, int warps, int segs) {
  return (lut ? kDwLutBytes : 0) + warps * kDwRing * dw_slot_bytes(kmax, segs);
}

// Window of a run for any K, read from shared memory: the 64 stream bits
// starting at the word holding bit q0 = (j0+1)K-16 (mod 256K), and the bit
// offset of state j0 inside them.
template <int K>
__device__ __forceinline__ void dw_window(const uint16_t* tile, int j0, uint32_t& hi, uint32_t& lo, int& off) {
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

// An item's payload tiles (32K bytes each) into a ring slot, one cp.async
// group per item. K = 4: the 64-byte halves of odd tiles are swapped so that
// the two tiles a warp reads in one k-step fall on different banks.
template <int K>
__device__ __forceinline__ void dw_copy(unsigned char* dst, const unsigned char* src, int ntiles, int lane) {
  const int chunks = ntiles * 2 * K;
  for (int c = lane; c < chunks; c += 32) {
    int off = c * 16;
    if (K == 4) {
      const int t = c >> 3, cc = c & 7;
      off = t * 128 + ((cc ^ ((t & 1) << 2)) << 4);
    }
    cp_async16(dst + off, src + (size_t)c * 16, 16);
  }
}

__device__ __forceinline__ void dw_copy_any(int k, unsigned char* dst, const unsigned char* src, int ntiles, int lane) {
  switch (k) {
    case 2: dw_copy<2>(dst, src, ntiles, lane); break;
    case 3: dw_copy<3>(dst, src, ntiles, lane); break;
    case 4: dw_copy<4>(dst, src, ntiles, lane); break;
    case 5: dw_copy<5>(dst, src, ntiles, lane); break;
    default: dw_copy<6>(dst, src, ntiles, lane); break;
  }
}

// Item geometry shared by the copy and the compute.
struct DwItem {
  int rb, sg, strip;
  int e, k, nvalid;
  int ncols;  // columns of this segment (a multiple of 32)
};

__device__ __forceinline__ DwItem dw_item(const DecArgs& d, uint32_t id, uint32_t nstrips, int kdim, int seg) {
  DwItem it;
  const uint32_t t = id / nstrips;
  it.strip = (int)(id - t * nstrips);
  const uint32_t rb = t / (uint32_t)d.nseg;
  it.sg = (int)(t - rb * (uint32_t)d.nseg);
  it.rb = (int)rb;
  it.ncols = min(seg, kdim - it.sg * seg);
  return it;
}

__device__ __forceinline__ void dw_item_meta(DwItem& it, const DwMetaW& m) {
  it.e = m.ek & 0xFFFF;
  it.k = (m.ek >> 16) & 0xFF;
  it.nvalid = m.ek >> 24;
}

// The item's activation operand: the up rows' own with separate gate / up
// input signs (FC1 strips at or past row I), else the shared one.
struct DwAct {
  const uint16_t* codes;   // fp16 rows (W4A8: the E4M3 codes as fp16)
  const uint16_t* scaled;  // W4A8: code * 2^e rows
  const uint8_t* scale;    // W4A8: E8M0 rows
};
__device__ __forceinline__ DwAct dw_act(const DecArgs& d, const DwItem& it) {
  if (d.split && it.strip * 16 >= d.f.I)
    return {reinterpret_cast<const uint16_t*>(d.act2), d.act_scaled2, d.act_scale2};
  return {reinterpret_cast<const uint16_t*>(d.f.act), d.act_scaled, d.f.act_scale};
}

__device__ __forceinline__ const unsigned char* dw_src(const DecArgs& d, const DwMetaW& m, const DwItem& it, int kdim,
                                                     int seg) {
  const int tiles_k = kdim >> 4;
  return reinterpret_cast<const unsigned char*>(d.f.payload) + m.off +
         ((size_t)it.strip * tiles_k + (size_t)it.sg * (seg >> 4)) * 32 * it.k;
}

// One 8-weight run of a tile (tile row r, half h; K = 4: the 32-bit words at
// byte offsets oc and op of the row's run and of the word before it) as fp16
// pairs, either by the codebook hash (W4A8: rounded to E4M3) ...
template <bool W4A8, int K>
__device__ __forceinline__ void dw_run_hash(const unsigned char* tile, int r, int h, int oc, int op, uint32_t k16,
                                            uint32_t nk16, uint32_t (&w)[4]) {
  uint32_t y[8];
  if (K == 4) {
    run_mcg_k4(*reinterpret_cast<const uint32_t*>(tile + op), *reinterpret_cast<const uint32_t*>(tile + oc), k16, nk16, y);
  } else {
    uint32_t hi, lo, s8[8];
    int off;
    dw_window<K>(reinterpret_cast<const uint16_t*>(tile), 16 * r + 8 * h, hi, lo, off);
    run_states_generic<K>(hi, lo, off, s8);
#pragma unroll
    for (int i = 0; i < 8; ++i) y[i] = mcg_raw(s8[i]);
  }
  if (W4A8)
    raw_to_e4m3_f16(y, w);
  else
    raw_to_f16(y, w);
}

// ... or by one lookup per weight in the shared-memory codebook table.
template <int K>
__device__ __forceinline__ void dw_run_lut(const unsigned char* tile, const uint16_t* lut, int r, int h, int oc, int op,
                                           uint32_t (&w)[4]) {
  uint32_t s[8];
  if (K == 4) {
    run_states_k4(*reinterpret_cast<const uint32_t*>(tile + op), *reinterpret_cast<const uint32_t*>(tile + oc), s);
  } else {
    uint32_t hi, lo;
    int off;
    dw_window<K>(reinterpret_cast<const uint16_t*>(tile), 16 * r + 8 * h, hi, lo, off);
    run_states_generic<K>(hi, lo, off, s);
  }
#pragma unroll
  for (int p = 0; p < 4; ++p) w[p] = __byte_perm((uint32_t)lut[s[2 * p]], (uint32_t)lut[s[2 * p + 1]], 0x5410);
}

// With the table, how many of a lane's two runs per tile take it (the other
// takes the hash, so that the shared-memory pipe and the integer / fp16 pipes
// could share the work). Lookups of random states meet bank conflicts: on
// sm_103 both the full table and the one-run split are slower than the hash
// alone, which is why the hash is the default.
constexpr int kDwLutRuns = 2;

// Expansion and MMAs of one item: acc (this lane's D fragment, rows g, g+8 of
// the strip, slots 2q, 2q+1) over the item's k-steps.
// PRE (W4A8): the activations are read as code * 2^e, so the MMAs accumulate
// straight into acc with no per-block scaling (every block of the item has
// its exponent in [-15, 7]; see dw_pre_issue).
// MX (TrellisMX-style weights): the weights are E4M3-rounded in both modes
// and every 32-column block of a weight row carries a UE8M0 scale, applied
// to that k-step's MMA result per row (exact powers of two in fp32).
template <bool W4A8, bool PRE, int K, bool LUT, bool MX, int SEGS>
__device__ __forceinline__ void dw_compute(const DecArgs& d, const DwItem& it, int row,
                                           const unsigned char* wt, const uint16_t* lut, int kdim, float (&acc)[4]) {
  const FcArgs& a = d.f;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3, h = q & 1, tsel = q >> 1;
  const int steps = it.ncols >> 5;
  const int col0 = it.sg * (SEGS * kDecSeg);
  // activation fragment source: slot g's row, columns 32 ks + 16 tsel + 8 h
  const int arow = __shfl_sync(0xFFFFFFFFu, row, g);
  const DwAct src = dw_act(d, it);
  const uint16_t* ap = (PRE ? src.scaled : src.codes) + (size_t)(arow < 0 ? 0 : arow) * kdim + col0 +
                       16 * tsel + 8 * h;
  // W4A8: E8M0 block exponents of slots 2q and 2q+1 for this segment
  const int r0 = (W4A8 && !PRE) ? __shfl_sync(0xFFFFFFFFu, row, 2 * q) : -1;
  const int r1 = (W4A8 && !PRE) ? __shfl_sync(0xFFFFFFFFu, row, 2 * q + 1) : -1;
  const uint8_t* sp0 = src.scale + (size_t)(r0 < 0 ? 0 : r0) * (kdim >> 5) + (col0 >> 5);
  const uint8_t* sp1 = src.scale + (size_t)(r1 < 0 ? 0 : r1) * (kdim >> 5) + (col0 >> 5);
  const uint32_t k16 = 0x10000u + (uint32_t)(d.T >> 30);  // 65536, opaque to the compiler
  const uint32_t nk16 = 0u - k16;
  // MX: the UE8M0 bytes of weight rows 16 strip + g and + 8 for this segment
  const uint8_t* wsg = nullptr;
  if (MX) wsg = a.wscale + ((size_t)it.e * a.wrows + 16 * it.strip + g) * a.wcols + (col0 >> 5);
  const int swz = 64 * tsel;
  const int oc0 = (4 * (2 * g + h)) ^ swz, op0 = (4 * ((2 * g + h + 31) & 31)) ^ swz;
  const int oc1 = (4 * (2 * g + 16 + h)) ^ swz, op1 = (4 * (2 * g + 15 + h)) ^ swz;
#pragma unroll
  for (int ks = 0; ks < SEGS * kDwSteps; ++ks) {
    if (ks < steps) {
      const uint4 bv = (arow >= 0) ? __ldg(reinterpret_cast<const uint4*>(ap + 32 * ks)) : make_uint4(0u, 0u, 0u, 0u);
      const unsigned char* tile = wt + (2 * ks + tsel) * 32 * K;
      uint32_t wa[4], wb[4];
      if (LUT)
        dw_run_lut<K>(tile, lut, g, h, oc0, op0, wa);
      else
        dw_run_hash<W4A8 || MX, K>(tile, g, h, oc0, op0, k16, nk16, wa);
      if (LUT && kDwLutRuns == 2)
        dw_run_lut<K>(tile, lut, g + 8, h, oc1, op1, wb);
      else
        dw_run_hash<W4A8 || MX, K>(tile, g + 8, h, oc1, op1, k16, nk16, wb);
      const uint32_t a0[4] = {wa[0], wb[0], wa[1], wb[1]};
      const uint32_t a1[4] = {wa[2], wb[2], wa[3], wb[3]};
      if (MX) {
        const float s0 = (W4A8 && !PRE) ? ((r0 >= 0) ? exp2_int((int)__ldg(sp0 + ks) - 127) : 0.0f) : 1.0f;
        const float s1 = (W4A8 && !PRE) ? ((r1 >= 0) ? exp2_int((int)__ldg(sp1 + ks) - 127) : 0.0f) : 1.0f;
        const float wg = exp2_int((int)__ldg(wsg + ks) - 127);
        const float wg8 = exp2_int((int)__ldg(wsg + 8 * a.wcols + ks) - 127);
        float dd[4] = {0.f, 0.f, 0.f, 0.f};
        mma_f16_16816(dd, a0, bv.x, bv.y);
        mma_f16_16816(dd, a1, bv.z, bv.w);
        acc[0] = fmaf(dd[0], wg * s0, acc[0]);
        acc[1] = fmaf(dd[1], wg * s1, acc[1]);
        acc[2] = fmaf(dd[2], wg8 * s0, acc[2]);
        acc[3] = fmaf(dd[3], wg8 * s1, acc[3]);
      } else if (W4A8 && !PRE) {
        const float s0 = (r0 >= 0) ? exp2_int((int)__ldg(sp0 + ks) - 127) : 0.0f;
        const float s1 = (r1 >= 0) ? exp2_int((int)__ldg(sp1 + ks) - 127) : 0.0f;
        float dd[4] = {0.f, 0.f, 0.f, 0.f};
        mma_f16_16816(dd, a0, bv.x, bv.y);
        mma_f16_16816(dd, a1, bv.z, bv.w);
        acc[0] = fmaf(dd[0], s0, acc[0]);
        acc[1] = fmaf(dd[1], s1, acc[1]);
        acc[2] = fmaf(dd[2], s0, acc[2]);
        acc[3] = fmaf(dd[3], s1, acc[3]);
      } else {
        mma_f16_16816(acc, a0, bv.x, bv.y);
        mma_f16_16816(acc, a1, bv.z, bv.w);
      }
    }
  }
}

template <bool W4A8, bool PRE, int KB, bool LUT, bool MX, int SEGS>
__device__ __forceinline__ void dw_compute_k(const DecArgs& d, const DwItem& it, int row, const unsigned char* wt,
                                             const uint16_t* lut, int kdim, float (&acc)[4]) {
  if (KB > 0) {
    dw_compute<W4A8, PRE, (KB > 0 ? KB : 4), LUT, MX, SEGS>(d, it, row, wt, lut, kdim, acc);
    return;
  }
  switch (it.k) {
    case 2: dw_compute<W4A8, PRE, 2, LUT, MX, SEGS>(d, it, row, wt, lut, kdim, acc); break;
    case 3: dw_compute<W4A8, PRE, 3, LUT, MX, SEGS>(d, it, row, wt, lut, kdim, acc); break;
    case 4: dw_compute<W4A8, PRE, 4, LUT, MX, SEGS>(d, it, row, wt, lut, kdim, acc); break;
    case 5: dw_compute<W4A8, PRE, 5, LUT, MX, SEGS>(d, it, row, wt, lut, kdim, acc); break;
    default: dw_compute<W4A8, PRE, 6, LUT, MX, SEGS>(d, it, row, wt, lut, kdim, acc); break;
  }
}

template <bool W4A8, int KB, bool LUT, bool MX, int SEGS>
__device__ __forceinline__ void dw_compute_any(const DecArgs& d, const DwItem& it, bool pre, int row,
                                               const unsigned char* wt, const uint16_t* lut, int kdim,
                                               float (&acc)[4]) {
  if (W4A8 && pre)
    dw_compute_k<W4A8, true, KB, LUT, MX, SEGS>(d, it, row, wt, lut, kdim, acc);
  else
    dw_compute_k<W4A8, false, KB, LUT, MX, SEGS>(d, it, row, wt, lut, kdim, acc);
}

// W4A8: the E8M0 exponents an item reads (its valid slots x its 32-column
// blocks), 2 * SEGS per lane (lane l: slot l/4, blocks 2 SEGS (l%4) on, one
// byte each of the result), loaded one item ahead; dw_pre_final says whether
// all lie in [-15, 7] (absent blocks count as 0 = 127 - 127).
template <int SEGS>
__device__ __forceinline__ uint32_t dw_pre_issue(const DecArgs& d, const DwItem& it, int row, int kdim, int lane) {
  const int n = lane >> 2, b0 = 2 * SEGS * (lane & 3);
  const int r = __shfl_sync(0xFFFFFFFFu, row, n);
  const int nb = it.ncols >> 5;
  uint32_t v = 0x7F7F7F7Fu;
  if (r >= 0) {
    const uint8_t* sp = dw_act(d, it).scale + (size_t)r * (kdim >> 5) + it.sg * (SEGS * kDwSteps) + b0;
#pragma unroll
    for (int j = 0; j < 2 * SEGS; ++j)
      if (b0 + j < nb) v = (v & ~(0xFFu << (8 * j))) | ((uint32_t)__ldg(sp + j) << (8 * j));
  }
  return v;
}
__device__ __forceinline__ bool dw_pre_final(uint32_t v) {
  bool ok = true;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t b = (v >> (8 * j)) & 0xFFu;
    ok = ok && b >= (uint32_t)kE8m0PreLo && b <= (uint32_t)kE8m0PreHi;
  }
  return __all_sync(0xFFFFFFFFu, ok);
}

// ---------------------------------------------------------------------------
// Epilogues, one warp for one slot n of one unit of route block rb. Partial
// sums of an item sit at partial[item * 128 + slot * 16 + row16], item = (rb *
// nseg + sg) * nstrips + strip. dw_sum_parts adds those of one strip in
// segment order, four loads in flight at a time.
// ---------------------------------------------------------------------------
template <int V>
__device__ __forceinline__ void dw_sum_parts(const DecArgs& d, int rb, int strip, int nstrips, int n, int r16,
                                             float (&v)[V]) {
#pragma unroll
  for (int i = 0; i < V; ++i) v[i] = 0.0f;
  for (int s0 = 0; s0 < d.nseg; s0 += 4) {
    float x[4][V];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const bool ok = s0 + u < d.nseg;
      const float* p = d.partial + ((size_t)(rb * d.nseg + (ok ? s0 + u : 0)) * nstrips + strip) * 128 + n * 16 + r16;
      if (V == 4) {
        const float4 q = ok ? __ldcg(reinterpret_cast<const float4*>(p)) : make_float4(0.f, 0.f, 0.f, 0.f);
        x[u][0] = q.x; x[u][1] = q.y; x[u][V > 2 ? 2 : 0] = q.z; x[u][V > 3 ? 3 : 0] = q.w;
      } else {
        const float2 q = ok ? __ldcg(reinterpret_cast<const float2*>(p)) : make_float2(0.f, 0.f);
        x[u][0] = q.x; x[u][1] = q.y;
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (s0 + u < d.nseg) {
#pragma unroll
        for (int i = 0; i < V; ++i) v[i] += x[u][i];
      }
  }
}

// The same for two strips at once (gate and up), all loads of four segments
// in flight together.
template <int V>
__device__ __forceinline__ void dw_sum_parts2(const DecArgs& d, int rb, int strip_a, int strip_b, int nstrips, int n,
                                              int r16, float (&va)[V], float (&vb)[V]) {
#pragma unroll
  for (int i = 0; i < V; ++i) va[i] = vb[i] = 0.0f;
  for (int s0 = 0; s0 < d.nseg; s0 += 4) {
    float xa[4][V], xb[4][V];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const bool ok = s0 + u < d.nseg;
      const size_t base = (size_t)(rb * d.nseg + (ok ? s0 + u : 0)) * nstrips;
      const float* pa = d.partial + (base + strip_a) * 128 + n * 16 + r16;
      const float* pb = d.partial + (base + strip_b) * 128 + n * 16 + r16;
      if (V == 4) {
        const float4 qa = ok ? __ldcg(reinterpret_cast<const float4*>(pa)) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 qb = ok ? __ldcg(reinterpret_cast<const float4*>(pb)) : make_float4(0.f, 0.f, 0.f, 0.f);
        xa[u][0] = qa.x; xa[u][1] = qa.y; xa[u][V > 2 ? 2 : 0] = qa.z; xa[u][V > 3 ? 3 : 0] = qa.w;
        xb[u][0] = qb.x; xb[u][1] = qb.y; xb[u][V > 2 ? 2 : 0] = qb.z; xb[u][V > 3 ? 3 : 0] = qb.w;
      } else {
        const float2 qa = ok ? __ldcg(reinterpret_cast<const float2*>(pa)) : make_float2(0.f, 0.f);
        const float2 qb = ok ? __ldcg(reinterpret_cast<const float2*>(pb)) : make_float2(0.f, 0.f);
        xa[u][0] = qa.x; xa[u][1] = qa.y;
        xb[u][0] = qb.x; xb[u][1] = qb.y;
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (s0 + u < d.nseg) {
#pragma unroll
        for (int i = 0; i < V; ++i) {
          va[i] += xa[u][i];
          vb[i] += xb[u][i];
        }
      }
  }
}

// PER consecutive fp16 values as floats (PER = 2 or 4, 4- or 8-byte aligned).
template <int PER>
__device__ __forceinline__ void dw_ld_h(const uint16_t* p, float (&v)[PER]) {
  if (PER == 4) {
    const uint2 q = __ldg(reinterpret_cast<const uint2*>(p));
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&q.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&q.y));
    v[0] = a.x; v[1] = a.y; v[PER > 2 ? 2 : 0] = b.x; v[PER > 3 ? 3 : 0] = b.y;
  } else {
    const uint32_t q = __ldg(reinterpret_cast<const uint32_t*>(p));
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&q));
    v[0] = a.x; v[1] = a.y;
  }
}

// FC1 unit mb: gate channels mb*BI .. +BI-1 and the matching up channels.
template <int PER, bool W4A8>
__device__ __forceinline__ void dw_epilogue_fc1(const DecArgs& d, int rb, int mb, int e, int n, int nstrips) {
  constexpr int BI = 32 * PER;
  const FcArgs& a = d.f;
  const int lane = threadIdx.x & 31;
  const uint16_t* s1 = a.scale + (size_t)e * 2 * a.I;
  const uint16_t* rt = a.rot_tab + (size_t)e * 3 * a.I;
  const int c0 = mb * BI + lane * PER;  // this lane's first channel (PER consecutive, one strip)
  const int strip_g = c0 >> 4, strip_u = (a.I + c0) >> 4, r16 = c0 & 15;
  const float hs = hadamard_scale(a.rot_b);
  {
    const int slot = rb * kDecBlock + n;
    float gv[PER], uv[PER], av[PER];
    // the channel vectors first, then the partial sums: both in flight together
    float sg_[PER], su_[PER], vg_[PER], vu_[PER], vd_[PER];
    dw_ld_h<PER>(s1 + c0, sg_);
    dw_ld_h<PER>(s1 + a.I + c0, su_);
    dw_ld_h<PER>(rt + c0, vg_);
    dw_ld_h<PER>(rt + a.I + c0, vu_);
    dw_ld_h<PER>(rt + 2 * a.I + c0, vd_);
    dw_griddep_wait();  // the partial sums come from the predecessor
    dw_sum_parts2<PER>(d, rb, strip_g, strip_u, nstrips, n, r16, gv, uv);
#pragma unroll
    for (int p = 0; p < PER; ++p) {
      gv[p] *= sg_[p];
      uv[p] *= su_[p];
    }
    warp_fwht<PER>(gv, a.rot_b);
    warp_fwht<PER>(uv, a.rot_b);
#pragma unroll
    for (int p = 0; p < PER; ++p) {
      const float gg = gv[p] * hs * vg_[p];
      const float uu = uv[p] * hs * vu_[p];
      av[p] = (gg / (1.0f + __expf(-gg))) * uu * vd_[p];
    }
    warp_fwht<PER>(av, a.rot_b);
#pragma unroll
    for (int p = 0; p < PER; ++p) av[p] *= hs;
    uint16_t* z = reinterpret_cast<uint16_t*>(a.out_act) + (size_t)slot * a.I + c0;
    if (!W4A8) {
#pragma unroll
      for (int p = 0; p < PER; p += 2) {
        __half2 v2 = __floats2half2_rn(av[p], av[p + 1]);
        *reinterpret_cast<__half2*>(z + p) = v2;
      }
    } else {
      // MXFP8 of z~ per 32 channels: E4M3 codes kept as fp16, E8M0 exponent apart
      constexpr int LPB = 32 / PER;  // lanes per 32-channel block
      float amax = 0.0f;
#pragma unroll
      for (int p = 0; p < PER; ++p) amax = fmaxf(amax, fabsf(av[p]));
#pragma unroll
      for (int o = 1; o < LPB; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
      const int ex = e8m0_exponent(amax);
      const float inv = exp2_int(-ex);
      uint16_t* zs = d.out_act_scaled + (size_t)slot * a.I + c0;
#pragma unroll
      for (int p = 0; p < PER; p += 2) {
        const uint32_t c = e4m3x2_to_f16x2(e4m3x2_from_float2(av[p] * inv, av[p + 1] * inv));
        *reinterpret_cast<uint32_t*>(z + p) = c;
        *reinterpret_cast<uint32_t*>(zs + p) = f16x2_times_exp2(c, ex);
      }
      if ((lane % LPB) == 0) a.out_scale[(size_t)slot * (a.I >> 5) + (c0 >> 5)] = (uint8_t)(ex + 127);
    }
  }
}

// FC2 epilogue and top-k combine, one CTA of kDwEpiWarps warps per (token t,
// 128 output columns mb): warp u takes the token's routes j = u, u + 8, ...;
// for each, the route's summed partials, output scale, H, hs * down_svh and
// the route weight w_j, into a shared row per route; then one warp adds the
// rows in route order j = 0..k-1 (the deterministic FP32 combine). A route
// whose expert id was dropped contributes zeros.
constexpr int kDwEpiWarps = 8;
__device__ __forceinline__ void dw_epilogue_fc2(const DecArgs& d, int t, int mb, int nstrips, float4* rows) {
  const FcArgs& a = d.f;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h0 = mb * 128 + lane * 4;
  const int strip = h0 >> 4, r16 = h0 & 15;
  const float hs = hadamard_scale(a.rot_b);
  const int k = a.topk;
  for (int j = warp; j < k; j += kDwEpiWarps) {
    // (route map, weights and tables come from the prologue or the layer,
    // complete before this grid could start)
    const int slot = d.slot_of_route[t * k + j];
    const bool ok = slot >= 0;  // warp-uniform
    const int e = ok ? d.ids[t * k + j] : 0;
    float sc[4], sv[4], v[4];
    dw_ld_h<4>(a.scale + (size_t)e * a.H + h0, sc);
    dw_ld_h<4>(a.rot_tab + (size_t)e * a.H + h0, sv);
    if (j == warp) dw_griddep_wait();  // the partial sums come from the predecessor
    float4 y4 = make_float4(0.f, 0.f, 0.f, 0.f);
    if (ok) {
      const float wj = d.route_w[t * k + j];
      dw_sum_parts<4>(d, slot / kDecBlock, strip, nstrips, slot % kDecBlock, r16, v);
      float y[4];
#pragma unroll
      for (int p = 0; p < 4; ++p) y[p] = v[p] * sc[p];
      warp_fwht<4>(y, a.rot_b);
      y4 = make_float4(wj * (y[0] * hs * sv[0]), wj * (y[1] * hs * sv[1]), wj * (y[2] * hs * sv[2]),
                       wj * (y[3] * hs * sv[3]));
    }
    rows[j * 32 + lane] = y4;
  }
  __syncthreads();
  if (warp == 0) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
      const float4 r = rows[j * 32 + lane];
      acc.x += r.x;
      acc.y += r.y;
      acc.z += r.z;
      acc.w += r.w;
    }
    *reinterpret_cast<float4*>(d.out + (size_t)t * a.H + h0) = acc;
  }
}

// The same for 512-point output rotation blocks (the coupled H512 boundary of
// TrellisMX-style layers: flashinfer PR #69 "b12x fused MoE: TrellisMX ...",
// Description): one CTA of kDwEpiWarps warps per (token t, 512 output columns
// mb); lane l holds the 16 columns of strip (mb * 512 + 16 l) / 16; the
// routes' rows sit in dynamic shared memory, [k][32 lanes][16] fp32.
__device__ __forceinline__ void dw_epilogue_fc2_512(const DecArgs& d, int t, int mb, int nstrips, float* rows) {
  const FcArgs& a = d.f;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h0 = mb * 512 + lane * 16;
  const int strip = h0 >> 4;
  const float hs = hadamard_scale(a.rot_b);
  const int k = a.topk;
  for (int j = warp; j < k; j += kDwEpiWarps) {
    const int slot = d.slot_of_route[t * k + j];
    const bool ok = slot >= 0;  // warp-uniform
    const int e = ok ? d.ids[t * k + j] : 0;
    float sc[16], sv[16], y[16];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float f[4];
      dw_ld_h<4>(a.scale + (size_t)e * a.H + h0 + 4 * q, f);
#pragma unroll
      for (int p = 0; p < 4; ++p) sc[4 * q + p] = f[p];
      dw_ld_h<4>(a.rot_tab + (size_t)e * a.H + h0 + 4 * q, f);
#pragma unroll
      for (int p = 0; p < 4; ++p) sv[4 * q + p] = f[p];
    }
    if (j == warp) dw_griddep_wait();  // the partial sums come from the predecessor
#pragma unroll
    for (int p = 0; p < 16; ++p) y[p] = 0.0f;
    if (ok) {
      const float wj = d.route_w[t * k + j];
      const int rb = slot / kDecBlock, n = slot % kDecBlock;
      for (int sg = 0; sg < d.nseg; ++sg) {  // the item's partial sums in segment order
        const float4* p4 = reinterpret_cast<const float4*>(d.partial + ((size_t)(rb * d.nseg + sg) * nstrips + strip) * 128 + n * 16);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 v = __ldcg(p4 + q);
          y[4 * q] += v.x;
          y[4 * q + 1] += v.y;
          y[4 * q + 2] += v.z;
          y[4 * q + 3] += v.w;
        }
      }
#pragma unroll
      for (int p = 0; p < 16; ++p) y[p] *= sc[p];
      warp_fwht<16>(y, a.rot_b);
#pragma unroll
      for (int p = 0; p < 16; ++p) y[p] = wj * (y[p] * hs * sv[p]);
    }
    float4* r4 = reinterpret_cast<float4*>(rows + ((size_t)j * 32 + lane) * 16);
#pragma unroll
    for (int q = 0; q < 4; ++q) r4[q] = make_float4(y[4 * q], y[4 * q + 1], y[4 * q + 2], y[4 * q + 3]);
  }
  __syncthreads();
  if (warp == 0) {
    float acc[16];
#pragma unroll
    for (int p = 0; p < 16; ++p) acc[p] = 0.0f;
    for (int j = 0; j < k; ++j) {
      const float4* r4 = reinterpret_cast<const float4*>(rows + ((size_t)j * 32 + lane) * 16);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 r = r4[q];
        acc[4 * q] += r.x;
        acc[4 * q + 1] += r.y;
        acc[4 * q + 2] += r.z;
        acc[4 * q + 3] += r.w;
      }
    }
    float4* o4 = reinterpret_cast<float4*>(d.out + (size_t)t * a.H + h0);
#pragma unroll
    for (int q = 0; q < 4; ++q) o4[q] = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
  }
}

// ---------------------------------------------------------------------------
// The kernel. Warp w of W takes items w, w + W, ..., so that the warps work
// through the payload together, one window of W consecutive items at a time
// (measured faster than giving each warp a contiguous range, which balances
// the last window better but scatters the concurrent reads). The metadata of
// an item's route block is loaded two items ahead, its payload one item
// ahead. FC2 reads only prologue outputs (route map, block table) and
// constant weights before it waits for its predecessor, so its first payload
// copy overlaps the FC1 epilogue. Partial sums: per item, [slot][16 rows] fp32.
// ---------------------------------------------------------------------------
template <bool W4A8, int PROJ, int KB, bool LUT, bool MX, int SEGS>
__global__ void __launch_bounds__(dw_cta_warps(KB, LUT, SEGS) * 32, LUT ? 1 : (KB > 0 ? 6 : 4)) k_dec_warp(const DecArgs d) {
  extern __shared__ __align__(128) unsigned char dw_smem[];
  constexpr int NW = dw_cta_warps(KB, LUT, SEGS);
  const FcArgs& a = d.f;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int KMAX = KB > 0 ? KB : 6;
  const int slot_bytes = dw_slot_bytes(KMAX, SEGS);
  constexpr int SEG = SEGS * kDecSeg;  // contraction columns per item
  unsigned char* ring = dw_smem + (LUT ? kDwLutBytes : 0) + warp * kDwRing * slot_bytes;
  const uint16_t* lut = reinterpret_cast<const uint16_t*>(dw_smem);
  const int kdim = PROJ == 1 ? a.H : a.I;
  const uint32_t nstrips = (uint32_t)((PROJ == 1 ? 2 * a.I : a.H) >> 4);
  const uint32_t per_block = (uint32_t)d.nseg * nstrips;
  const uint32_t nwarps = gridDim.x * NW;

  if (LUT) {
    // the codebook table (fixed since the layer was prepared) into shared
    // memory, overlapping the predecessor's tail
    const uint4* src = reinterpret_cast<const uint4*>(d.lut);
    uint4* dst = reinterpret_cast<uint4*>(dw_smem);
    for (int i = threadIdx.x; i < kDwLutBytes / 16; i += NW * 32) dst[i] = __ldg(src + i);
    __syncthreads();
  }
  if (PROJ == 1) dw_griddep_wait();  // the route map and x~ come from the prologue
  const int nb = min(*a.nblocks, d.max_blocks);
  const uint32_t h1 = (uint32_t)nb * per_block;  // items
  uint32_t h = blockIdx.x * NW + warp;           // next item of this warp
  const bool any = h < h1;
  uint32_t pc = 0, pn = 0, pn2 = 0;
  DwItem it{}, nit{};
  DwMetaW m{}, nm{};
  DwRaw raw1{-1, 0}, raw2{-1, 0};
  bool has1 = false, has2 = false;
  uint32_t pre_cur = 0, pre_next = 0;
  if (any) {
    pc = h;
    h += nwarps;
    const DwRaw raw0 = dw_meta_issue(d, (int)(pc / per_block), lane);
    has1 = h < h1;
    if (has1) {
      pn = h;
      h += nwarps;
      raw1 = dw_meta_issue(d, (int)(pn / per_block), lane);
    }
    it = dw_item(d, pc, nstrips, kdim, SEG);
    m = dw_meta_final<PROJ>(raw0, it.rb, lane, a.topk, d.split);
    dw_item_meta(it, m);
    dw_copy_any(KB > 0 ? KB : it.k, ring, dw_src(d, m, it, kdim, SEG), it.ncols >> 4, lane);
  }
  cp_async_commit();
  if (PROJ == 2) dw_griddep_wait();  // z~, its exponents and the partial buffer belong to the predecessors until now
  dw_griddep_launch();
  if (!any) return;
  if (W4A8) pre_cur = dw_pre_issue<SEGS>(d, it, m.row, kdim, lane);
  if (has1) {
    nit = dw_item(d, pn, nstrips, kdim, SEG);
    nm = dw_meta_final<PROJ>(raw1, nit.rb, lane, a.topk, d.split);
    dw_item_meta(nit, nm);
    if (W4A8) pre_next = dw_pre_issue<SEGS>(d, nit, nm.row, kdim, lane);
    has2 = h < h1;
    if (has2) {
      pn2 = h;
      h += nwarps;
      raw2 = dw_meta_issue(d, (int)(pn2 / per_block), lane);
    }
  }
  for (int n = 0;; ++n) {
    if (has1)
      dw_copy_any(KB > 0 ? KB : nit.k, ring + ((n + 1) & 1) * slot_bytes, dw_src(d, nm, nit, kdim, SEG), nit.ncols >> 4, lane);
    cp_async_commit();
    cp_async_wait<1>();
    __syncwarp();

    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    const bool pre = W4A8 && dw_pre_final(pre_cur);
    dw_compute_any<W4A8, KB, LUT, MX, SEGS>(d, it, pre, m.row, ring + (n & 1) * slot_bytes, lut, kdim, acc);

    // partial sums of the valid slots, [slot][16 rows]
    const int g = lane >> 2, c = 2 * (lane & 3);
    float* pb = d.partial + (size_t)pc * 128;
    if (c < it.nvalid) {
      pb[c * 16 + g] = acc[0];
      pb[c * 16 + g + 8] = acc[2];
    }
    if (c + 1 < it.nvalid) {
      pb[(c + 1) * 16 + g] = acc[1];
      pb[(c + 1) * 16 + g + 8] = acc[3];
    }
    __syncwarp();  // this ring slot is refilled two pieces on
    if (!has1) break;
    pc = pn;
    it = nit;
    m = nm;
    pre_cur = pre_next;
    has1 = has2;
    if (has1) {
      pn = pn2;
      nit = dw_item(d, pn, nstrips, kdim, SEG);
      nm = dw_meta_final<PROJ>(raw2, nit.rb, lane, a.topk, d.split);
      dw_item_meta(nit, nm);
      if (W4A8) pre_next = dw_pre_issue<SEGS>(d, nit, nm.row, kdim, lane);
      has2 = h < h1;
      if (has2) {
        pn2 = h;
      h += nwarps;
        raw2 = dw_meta_issue(d, (int)(pn2 / per_block), lane);
      }
    }
  }
  cp_async_wait<0>();
}

// The epilogue kernels: FC1 one warp per (route block, unit of BI
// intermediate channels, slot), FC2 one CTA per (token, 128 output channels).
template <bool W4A8, int PROJ>
__global__ void __launch_bounds__(256) k_dec_epi(const DecArgs d) {
  // (the route map and block table come from the prologue, complete before
  // this grid could start; each epilogue waits for its predecessor only
  // before it reads the partial sums)
  dw_griddep_launch();
  const FcArgs& a = d.f;
  const int gw = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  if (PROJ == 1) {
    const int n = gw % kDecBlock;
    const int um = gw / kDecBlock;
    const int mb = um % d.units_m;
    const int rb = um / d.units_m;
    if (rb >= d.max_blocks) return;
    const int meta = d.blk_meta[rb];  // (0 past the last block)
    if (n >= (meta >> 24)) return;    // padding slot
    const int e = meta & 0xFFFF;
    const int nstrips = (2 * a.I) >> 4;
    if (d.bi == 128)
      dw_epilogue_fc1<4, W4A8>(d, rb, mb, e, n, nstrips);
    else
      dw_epilogue_fc1<2, W4A8>(d, rb, mb, e, n, nstrips);
  } else {
    __shared__ float4 rows[32 * 32];  // one 128-column row per route (top-k <= 32)
    const int mb = blockIdx.x % d.units_m;
    const int t = blockIdx.x / d.units_m;
    if (t >= d.T) return;  // (whole CTA)
    dw_epilogue_fc2(d, t, mb, a.H >> 4, rows);
  }
}

template <bool W4A8, int PROJ, int KB, bool LUT, bool MX = false, int SEGS = 1>
static cudaError_t dw_warps_t(int* warps) {
  // attributes and the resident-CTA count are fixed on the first call (before any capture)
  constexpr int NW = dw_cta_warps(KB, LUT, SEGS);
  static int resident = 0;
  if (resident == 0) {
    auto kern = k_dec_warp<W4A8, PROJ, KB, LUT, MX, SEGS>;
    const int smem = dw_smem_bytes(KB > 0 ? KB : 6, LUT, NW, SEGS);
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    int per_sm = 0;
    if ((err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NW * 32, smem)) != cudaSuccess) return err;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    int dev = 0, sms = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
    resident = per_sm * sms;
  }
  *warps = resident * NW;
  return cudaSuccess;
}

template <bool W4A8, int PROJ, int KB, bool LUT, bool MX = false, int SEGS = 1>
static cudaError_t launch_dw_t(const DecArgs& d, cudaStream_t st) {
  constexpr int NW = dw_cta_warps(KB, LUT, SEGS);
  if (d.fc_warps <= 0 || d.fc_warps % NW || d.segs != SEGS) return cudaErrorInvalidValue;
  if (LUT && (!d.lut || ((uintptr_t)d.lut) % 16)) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(d.fc_warps / NW);
  cfg.blockDim = dim3(NW * 32);
  cfg.dynamicSmemBytes = dw_smem_bytes(KB > 0 ? KB : 6, LUT, NW, SEGS);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_dec_warp<W4A8, PROJ, KB, LUT, MX, SEGS>, d);
}

// FC2 epilogue for 512-point output rotation blocks: one CTA per (token,
// 512 columns), the routes' rows in topk * 2 KB of dynamic shared memory.
__global__ void __launch_bounds__(256) k_dec_epi512(const DecArgs d) {
  extern __shared__ __align__(16) float dw_rows512[];
  dw_griddep_launch();
  const int mb = blockIdx.x % d.units_m;
  const int t = blockIdx.x / d.units_m;
  if (t >= d.T) return;  // (whole CTA)
  dw_epilogue_fc2_512(d, t, mb, d.f.H >> 4, dw_rows512);
}

static cudaError_t launch_epi512(const DecArgs& d, cudaStream_t st) {
  const int smem = d.f.topk * 32 * 16 * 4;
  static bool attr_done = false;  // first call, before any capture
  if (!attr_done) {
    const cudaError_t err = cudaFuncSetAttribute(k_dec_epi512, cudaFuncAttributeMaxDynamicSharedMemorySize, 32 * 32 * 16 * 4);
    if (err != cudaSuccess) return err;
    attr_done = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((long)d.T * d.units_m));
  cfg.blockDim = dim3(32 * kDwEpiWarps);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_dec_epi512, d);
}

template <bool W4A8, int PROJ>
static cudaError_t launch_epi_t(const DecArgs& d, cudaStream_t st) {
  // FC1: one warp per (block, unit, slot); FC2: one CTA per (token, unit)
  const long warps = (PROJ == 1) ? (long)d.max_blocks * d.units_m * kDecBlock : (long)d.T * d.units_m * 8;
  static_assert(kDwEpiWarps == 8, "the FC2 epilogue CTA is the launch's 256 threads");
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((warps + 7) / 8));
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_dec_epi<W4A8, PROJ>, d);
}

// TrellisMX-style weights (scales present): the general-K, hash-expansion
// kernels only.
static cudaError_t dec_fc_warps_mx(int proj, bool w4a8, int* warps) {
  if (proj == 1) return w4a8 ? dw_warps_t<true, 1, 0, false, true>(warps) : dw_warps_t<false, 1, 0, false, true>(warps);
  return w4a8 ? dw_warps_t<true, 2, 0, false, true>(warps) : dw_warps_t<false, 2, 0, false, true>(warps);
}

template <bool LUT>
static cudaError_t dec_fc_warps_t(int proj, bool w4a8, int uniform_k, int segs, int* warps) {
  const bool k4 = uniform_k == 4;
  if (k4 && segs == 2) {
    if (proj == 1) return w4a8 ? dw_warps_t<true, 1, 4, LUT, false, 2>(warps) : dw_warps_t<false, 1, 4, LUT, false, 2>(warps);
    return w4a8 ? dw_warps_t<true, 2, 4, LUT, false, 2>(warps) : dw_warps_t<false, 2, 4, LUT, false, 2>(warps);
  }
  if (proj == 1) {
    if (w4a8) return k4 ? dw_warps_t<true, 1, 4, LUT>(warps) : dw_warps_t<true, 1, 0, LUT>(warps);
    return k4 ? dw_warps_t<false, 1, 4, LUT>(warps) : dw_warps_t<false, 1, 0, LUT>(warps);
  }
  if (w4a8) return k4 ? dw_warps_t<true, 2, 4, LUT>(warps) : dw_warps_t<true, 2, 0, LUT>(warps);
  return k4 ? dw_warps_t<false, 2, 4, LUT>(warps) : dw_warps_t<false, 2, 0, LUT>(warps);
}

cudaError_t dec_fc_warps(int proj, bool w4a8, int uniform_k, bool lut, bool mx, int segs, int* warps) {
  if (mx) return dec_fc_warps_mx(proj, w4a8, warps);
  return lut ? dec_fc_warps_t<true>(proj, w4a8, uniform_k, segs, warps)
             : dec_fc_warps_t<false>(proj, w4a8, uniform_k, segs, warps);
}

cudaError_t launch_dec_epilogue(const DecArgs& d, int proj, bool w4a8, cudaStream_t st) {
  if (proj == 1) return w4a8 ? launch_epi_t<true, 1>(d, st) : launch_epi_t<false, 1>(d, st);
  if (d.f.rot_b > 128) return launch_epi512(d, st);  // (units_m = H / 512)
  return w4a8 ? launch_epi_t<true, 2>(d, st) : launch_epi_t<false, 2>(d, st);
}

template <bool LUT>
static cudaError_t launch_dec_fc_t(const DecArgs& d, int proj, bool w4a8, int uniform_k, cudaStream_t st) {
  const bool k4 = uniform_k == 4;
  if (k4 && d.segs == 2) {
    if (proj == 1) return w4a8 ? launch_dw_t<true, 1, 4, LUT, false, 2>(d, st) : launch_dw_t<false, 1, 4, LUT, false, 2>(d, st);
    return w4a8 ? launch_dw_t<true, 2, 4, LUT, false, 2>(d, st) : launch_dw_t<false, 2, 4, LUT, false, 2>(d, st);
  }
  if (proj == 1) {
    if (w4a8) return k4 ? launch_dw_t<true, 1, 4, LUT>(d, st) : launch_dw_t<true, 1, 0, LUT>(d, st);
    return k4 ? launch_dw_t<false, 1, 4, LUT>(d, st) : launch_dw_t<false, 1, 0, LUT>(d, st);
  }
  if (w4a8) return k4 ? launch_dw_t<true, 2, 4, LUT>(d, st) : launch_dw_t<true, 2, 0, LUT>(d, st);
  return k4 ? launch_dw_t<false, 2, 4, LUT>(d, st) : launch_dw_t<false, 2, 0, LUT>(d, st);
}

cudaError_t launch_dec_fc(const DecArgs& d, int proj, bool w4a8, int uniform_k, cudaStream_t st) {
  if (d.f.wscale) {
    if (proj == 1) return w4a8 ? launch_dw_t<true, 1, 0, false, true>(d, st) : launch_dw_t<false, 1, 0, false, true>(d, st);
    return w4a8 ? launch_dw_t<true, 2, 0, false, true>(d, st) : launch_dw_t<false, 2, 0, false, true>(d, st);
  }
  return d.lut ? launch_dec_fc_t<true>(d, proj, w4a8, uniform_k, st) : launch_dec_fc_t<false>(d, proj, w4a8, uniform_k, st);
}

// The codebook tables of a layer: [0, 65536) the fp16 weight of each state,
// [65536, 131072) the fp16 value of its E4M3 rounding, computed by the same
// expansion functions as the procedural path (8 states per thread).
__global__ void k_build_decode_lut(uint16_t* lut) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= kDwLutEntries / 8) return;
  uint32_t y[8], w[4], we[4];
#pragma unroll
  for (int i = 0; i < 8; ++i) y[i] = mcg_raw((uint32_t)(8 * t + i));
  raw_to_f16(y, w);
  raw_to_e4m3_f16(y, we);
  reinterpret_cast<uint4*>(lut)[t] = make_uint4(w[0], w[1], w[2], w[3]);
  reinterpret_cast<uint4*>(lut + kDwLutEntries)[t] = make_uint4(we[0], we[1], we[2], we[3]);
}

size_t decode_lut_bytes() { return 2 * (size_t)kDwLutBytes; }

cudaError_t build_decode_lut(uint16_t* lut, cudaStream_t st) {
  k_build_decode_lut<<<kDwLutEntries / 8 / 256, 256, 0, st>>>(lut);
  return cudaGetLastError();
}

}  // namespace tmoe
