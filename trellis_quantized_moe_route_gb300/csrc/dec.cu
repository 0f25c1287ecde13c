// Decode-rows path (sm_103a): the layer for a few tokens (T * topk <= 1024),
// where every expert is touched by a handful of routes and the layer is bound
// by streaming and decoding the touched trellis payload (b12x PR #129 "feat(moe):
// serve canonical Fruit QSRT atoms", Hot path: W4A8 only for bounded decode
// rows; the decode expands the payload directly into E4M3 MMA operands).
//
// Three kernels on one stream:
//   1. prologue: router (optional), route map and the fused rotate+quantize
//      in one launch; it also clears the counters and the output.
//   2. FC1: CTA = (route block of 8 routes, 128 weight rows, column split).
//      Weight tiles and activations are staged through a 3-deep cp.async ring;
//      each warp expands 16 rows x 32 columns per k-step into fp16 mma.sync
//      operands (W4A8: E4M3-rounded weights and E4M3 activations, both held
//      exactly in fp16, since the E4M3 form of mma.sync is not a native
//      tensor instruction on sm_103). Partial sums go to the workspace; the last CTA of a unit
//      (gate + up rows of one intermediate block) reduces them in fixed split
//      order and runs the activation epilogue.
//   3. FC2: the same with the unrotation epilogue; the last unit finishing a
//      (token, 128-column block) performs that block's top-k combine in fixed
//      slot order.
// FC1 and FC2 are launched with programmatic dependent launch, so each can be
// scheduled while its predecessor drains; they wait (griddepcontrol.wait)
// before reading anything the predecessor writes. No kernel spins.
#include <algorithm>

#include "rotate_dev.cuh"
#include "route_dev.cuh"

namespace tmoe {

constexpr int kDecThreads = 256;    // 8 warps, one 16-row m-tile each
constexpr int kDecRows = 128;       // weight rows per CTA
constexpr int kDecBN = 8;           // routes per route block
constexpr int kDecTargetCtas = 608; // 4 x 152 SMs
constexpr int kDecMaxChunk = 2560;  // most columns one split covers

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

// ---------------------------------------------------------------------------
// Prologue. CTA 0: router (when logits are given) and the route map; the
// other CTAs: rotate+quantize (one warp per token x 128 columns), clearing
// of counters and output.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) k_dec_prologue(const DecPrologueArgs a) {
  const int tid = threadIdx.x, warp = tid >> 5;
  if (blockIdx.x == 0) {
    __shared__ RankScratch sm;
    if (tid == 0) *a.rm.err = 0;  // ordered before tile_rank's flags by its barriers
    if (a.logits) {
      for (int t = warp; t < a.T; t += 32) route_token_warp(a.logits, t, a.rm.E, a.topk, a.ids_out, a.w_out);
      __syncthreads();
    }
    const RouteMapArgs& r = a.rm;
    tile_rank(r.ids, r.R, r.E, 0, sm, r.rank, r.tile_counts, r.err);
    __syncthreads();
    scan_experts(r.E, 1, r.block, r.tile_counts, r.counts, r.offsets, r.block_expert, r.nblocks);
    __syncthreads();
    pack_routes(r.ids, r.R, r.E, r.block, tid, blockDim.x, r.rank, r.tile_counts, r.counts, r.offsets,
                r.route_of_slot, r.slot_of_route);
    return;
  }
  const int nrot = gridDim.x - 1;
  const int cta = blockIdx.x - 1;
  const int gw = cta * 32 + warp;
  if (a.w4a8)
    rotate_quant_warp<true>(a.x, a.suh, a.T, a.H, a.rot_b, a.xq, a.xs, gw);
  else
    rotate_quant_warp<false>(a.x, a.suh, a.T, a.H, a.rot_b, a.xq, a.xs, gw);
  const long gtid = (long)cta * blockDim.x + tid, gstride = (long)nrot * blockDim.x;
  for (long i = gtid; i < a.n_zero_i32; i += gstride) a.zero_i32[i] = 0;
  for (long i = gtid; i < a.out_n / 4; i += gstride) reinterpret_cast<float4*>(a.out)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

cudaError_t launch_dec_prologue(const DecPrologueArgs& a, cudaStream_t st) {
  const long warps = (long)a.T * (a.H / 128);
  const int nrot = (int)std::max<long>(1, (warps + 31) / 32);
  k_dec_prologue<<<1 + nrot, 1024, 0, st>>>(a);
  return cudaGetLastError();
}

// Window of a run for any K, read from shared memory (see run_window_generic).
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

// ---------------------------------------------------------------------------
// Epilogues, run by the last CTA of a unit on C[unit_rows][9] (fp32 sums of
// the unit's rows for the 8 routes of the block; columns of padding slots 0).
// One warp per route column.
// ---------------------------------------------------------------------------

// FC1: rows 0..BI-1 gate, BI..2BI-1 up of intermediate block mb.
// z~ = H(suh_d * SiLU(svh_g * H(s1g * gate)) * svh_u * H(s1u * up)), then fp16
// or MXFP8 into the slot's z~ row (sparkinfer PR #90, review of kernel.py:
// _run_activation: H128 -> svh -> SiLU -> suh_down -> H128).
template <int PER, bool W4A8>
__device__ __forceinline__ void dec_epilogue_fc1(const FcArgs& a, int e, int mb, int slot0, const float* C,
                                                 const int* row_slot) {
  constexpr int BI = 32 * PER;
  constexpr int CS = kDecBN + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int col = warp;
  const uint16_t* s1 = a.scale + (size_t)e * 2 * a.I;
  const uint16_t* rt = a.rot_tab + (size_t)e * 3 * a.I;
  const int c0 = mb * BI + lane * PER;
  const bool valid = row_slot[col] >= 0;
  const float hs = hadamard_scale(a.rot_b);
  float gv[PER], uv[PER], av[PER];
#pragma unroll
  for (int p = 0; p < PER; ++p) {
    gv[p] = C[(lane * PER + p) * CS + col] * __half2float(__ushort_as_half(s1[c0 + p]));
    uv[p] = C[(BI + lane * PER + p) * CS + col] * __half2float(__ushort_as_half(s1[a.I + c0 + p]));
  }
  warp_fwht<PER>(gv, a.rot_b);
  warp_fwht<PER>(uv, a.rot_b);
#pragma unroll
  for (int p = 0; p < PER; ++p) {
    const float gg = gv[p] * hs * __half2float(__ushort_as_half(rt[c0 + p]));
    const float uu = uv[p] * hs * __half2float(__ushort_as_half(rt[a.I + c0 + p]));
    av[p] = (gg / (1.0f + __expf(-gg))) * uu * __half2float(__ushort_as_half(rt[2 * a.I + c0 + p]));
  }
  warp_fwht<PER>(av, a.rot_b);
#pragma unroll
  for (int p = 0; p < PER; ++p) av[p] = valid ? av[p] * hs : 0.0f;
  const int slot = slot0 + col;
  if (!W4A8) {
    uint16_t* z = reinterpret_cast<uint16_t*>(a.out_act) + (size_t)slot * a.I + c0;
#pragma unroll
    for (int p = 0; p < PER; p += 2) {
      __half2 v2 = __floats2half2_rn(av[p], av[p + 1]);
      *reinterpret_cast<__half2*>(z + p) = v2;
    }
  } else {
    constexpr int LPB = 32 / PER;  // lanes per 32-channel block
    float amax = 0.0f;
#pragma unroll
    for (int p = 0; p < PER; ++p) amax = fmaxf(amax, fabsf(av[p]));
#pragma unroll
    for (int o = 1; o < LPB; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    const int ex = e8m0_exponent(amax);
    const float inv = exp2_int(-ex);
    uint8_t* z = reinterpret_cast<uint8_t*>(a.out_act) + (size_t)slot * a.I + c0;
#pragma unroll
    for (int p = 0; p < PER; p += 2)
      *reinterpret_cast<uint16_t*>(z + p) = (uint16_t)e4m3x2_from_float2(av[p] * inv, av[p + 1] * inv);
    if ((lane % LPB) == 0) a.out_scale[(size_t)slot * (a.I >> 5) + (c0 >> 5)] = valid ? (uint8_t)(ex + 127) : (uint8_t)0;
  }
}

// FC2: rows = output columns mb*128 .. +127. Unrotate (H, down_svh), then
// either store the slot's row and combine finished tokens, or add w * row into
// the output with FP32 atomics.
__device__ __forceinline__ void dec_epilogue_fc2(const DecArgs& d, int e, int mb, int slot0, const float* C,
                                                 const int* row_slot) {
  constexpr int CS = kDecBN + 1;
  const FcArgs& a = d.f;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int col = warp;
  const int r = row_slot[col];
  if (r < 0) return;  // padding slot
  const int h0 = mb * 128 + lane * 4;
  const uint16_t* s2 = a.scale + (size_t)e * a.H;
  const uint16_t* sv = a.rot_tab + (size_t)e * a.H;
  float v[4];
#pragma unroll
  for (int p = 0; p < 4; ++p) v[p] = C[(lane * 4 + p) * CS + col] * __half2float(__ushort_as_half(s2[h0 + p]));
  warp_fwht<4>(v, a.rot_b);
  const float hs = hadamard_scale(a.rot_b);
#pragma unroll
  for (int p = 0; p < 4; ++p) v[p] = v[p] * hs * __half2float(__ushort_as_half(sv[h0 + p]));
  const int t = r / a.topk;
  if (a.atomic) {
    const float wr = d.route_w[r];
    float* dst = d.out + (size_t)t * a.H + h0;
#pragma unroll
    for (int p = 0; p < 4; ++p) atomicAdd(dst + p, wr * v[p]);
    return;
  }
  __stcg(reinterpret_cast<float4*>(a.out_f32 + (size_t)(slot0 + col) * a.H + h0), make_float4(v[0], v[1], v[2], v[3]));
  // Completion count of (token t, column block mb); the route that completes
  // it combines the block in slot order j = 0..k-1.
  const int k = a.topk;
  const int my_slot = (lane < k) ? d.slot_of_route[t * k + lane] : -1;
  const int nvalid = __popc(__ballot_sync(0xFFFFFFFFu, my_slot >= 0));
  __threadfence();
  __syncwarp();
  int last = 0;
  if (lane == 0) last = (atomicAdd(&d.tok_cnt[t * d.units_m + mb], 1) == nvalid - 1);
  last = __shfl_sync(0xFFFFFFFFu, last, 0);
  if (!last) return;
  __threadfence();
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = 0; j < k; ++j) {
    const int sj = __shfl_sync(0xFFFFFFFFu, my_slot, j);
    if (sj < 0) continue;
    const float wj = d.route_w[t * k + j];
    const float4 rv = __ldcg(reinterpret_cast<const float4*>(a.out_f32 + (size_t)sj * a.H + h0));
    acc.x = fmaf(wj, rv.x, acc.x);
    acc.y = fmaf(wj, rv.y, acc.y);
    acc.z = fmaf(wj, rv.z, acc.z);
    acc.w = fmaf(wj, rv.w, acc.w);
  }
  *reinterpret_cast<float4*>(d.out + (size_t)t * a.H + h0) = acc;
  if (lane == 0) d.tok_cnt[t * d.units_m + mb] = 0;
}

// ---------------------------------------------------------------------------
// Split-K main loop.
// Shared memory: the activations (and W4A8 block scales) of the 8 routes for
// the CTA's whole column split, staged once; then one private cp.async ring
// per warp over its 16 weight rows, kDecGroup k-steps (2*kDecGroup tiles) per
// ring slot, so the main loop needs no CTA-wide barrier. A K=4 tile is 128
// bytes; the 64-byte halves of odd tiles are swapped so that the two tiles a
// warp reads in one k-step fall on different banks.
// ---------------------------------------------------------------------------
constexpr int kDecGroup = 4;   // k-steps per ring slot
constexpr int kDecRing = 4;    // ring slots per warp

struct DecSmemPlan {
  int arow, abytes, sbytes, wslot, wbytes, total;
};

__host__ __device__ inline DecSmemPlan dec_smem_plan(bool w4a8, int kmax, int kchunk) {
  DecSmemPlan p;
  // activations are held as fp16 (W4A8: E4M3 codes widened exactly); a row
  // stride of 64 mod 128 keeps the 16-byte B-fragment loads of a warp on
  // distinct banks
  const int ab = 2 * kchunk;
  const int want = 64;
  p.arow = ab + ((want - ab % 128) + 128) % 128;
  p.abytes = kDecBN * p.arow;
  p.sbytes = w4a8 ? kDecBN * (kchunk / 32) * 4 : 0;
  p.wslot = 2 * kDecGroup * 32 * kmax;
  p.wbytes = 8 * kDecRing * p.wslot;
  const int c_bytes = 2 * 128 * (kDecBN + 1) * 4;  // epilogue C (aliases the weight rings)
  p.total = p.abytes + p.sbytes + (p.wbytes > c_bytes ? p.wbytes : c_bytes) + 128;
  return p;
}

template <bool W4A8, int PROJ, int K, int KMAX>
__device__ __forceinline__ void dec_body(const DecArgs& d, int rb, int mb, int part, int sidx, int e,
                                         unsigned char* smem) {
  const FcArgs& a = d.f;
  const DecSmemPlan sp = dec_smem_plan(W4A8, KMAX, d.kchunk);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, q = lane & 3, h = q & 1, tsel = q >> 1;
  const int KDIM = (PROJ == 1) ? a.H : a.I;
  const int tiles_k = KDIM >> 4;
  const int U = (PROJ == 1) ? 2 * d.bi : kDecRows;
  unsigned char* act_s = smem;
  float* sc_s = reinterpret_cast<float*>(smem + sp.abytes);
  unsigned char* wring = smem + sp.abytes + sp.sbytes;
  int* row_src = reinterpret_cast<int*>(smem + sp.total - 128);
  int* row_slot = row_src + kDecBN;
  int* flag = row_slot + kDecBN;
  const int slot0 = rb * kDecBN;
  if (tid < kDecBN) {
    const int r = a.route_of_slot[slot0 + tid];
    row_slot[tid] = r;
    row_src[tid] = (r < 0) ? -1 : ((PROJ == 1) ? r / a.topk : slot0 + tid);
  }
  __syncthreads();
  int nvalid = 0;
#pragma unroll
  for (int n = 0; n < kDecBN; ++n) nvalid += row_slot[n] >= 0 ? 1 : 0;

  const int col0 = sidx * d.kchunk;
  const int ncols = min(d.kchunk, KDIM - col0);
  const int nsteps = ncols >> 5;
  const int ngroups = (nsteps + kDecGroup - 1) / kDecGroup;

  // ---- this warp's 16 weight rows and its ring ----
  const int lr = part * kDecRows + 16 * warp;
  const int row = (PROJ == 1) ? ((lr < d.bi) ? mb * d.bi + lr : a.I + mb * d.bi + (lr - d.bi)) : mb * kDecRows + lr;
  const unsigned char* wrow = reinterpret_cast<const unsigned char*>(a.payload) + 2 * (size_t)a.word_off[e] +
                              (size_t)(row >> 4) * tiles_k * 32 * K + (size_t)(col0 >> 4) * 32 * K;
  unsigned char* myring = wring + warp * kDecRing * sp.wslot;
  auto load_group = [&](int grp) {
    const int steps = min(kDecGroup, nsteps - grp * kDecGroup);
    const int chunks = steps * 2 * 2 * K;  // 2 tiles per k-step, 32K bytes per tile
    const unsigned char* src = wrow + (size_t)grp * kDecGroup * 2 * 32 * K;
    unsigned char* dst = myring + (grp % kDecRing) * sp.wslot;
    for (int c = lane; c < chunks; c += 32) {
      int off = c * 16;
      if (K == 4) {
        const int t = c >> 3, cc = c & 7;
        off = t * 128 + ((cc ^ ((t & 1) << 2)) << 4);
      }
      cp_async16(dst + off, src + (size_t)c * 16, 16);
    }
  };
  // the first weight groups go out before the activations are staged, so
  // their latency overlaps the staging below
#pragma unroll
  for (int gi = 0; gi < kDecRing - 1; ++gi) {
    if (gi < ngroups) load_group(gi);
    cp_async_commit();
  }
  // ---- activations and scales of the whole split (one cp.async group) ----
  {
    const unsigned char* act = reinterpret_cast<const unsigned char*>(a.act);
    if (W4A8) {
      // E4M3 codes, widened to fp16 on the way into shared memory; four
      // loads per thread are in flight before the first is used
      const int vec = ncols >> 2;  // 4 codes per step
      for (int i0 = tid; i0 < kDecBN * vec; i0 += 4 * kDecThreads) {
        uint32_t codes[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = i0 + u * kDecThreads;
          codes[u] = 0;
          if (i < kDecBN * vec) {
            const int src = row_src[i / vec];
            if (src >= 0) codes[u] = __ldg(reinterpret_cast<const uint32_t*>(act + (size_t)src * KDIM + col0) + i % vec);
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = i0 + u * kDecThreads;
          if (i < kDecBN * vec) {
            uint2 hv;
            hv.x = e4m3x2_to_f16x2(codes[u] & 0xFFFFu);
            hv.y = e4m3x2_to_f16x2(codes[u] >> 16);
            *reinterpret_cast<uint2*>(act_s + (i / vec) * sp.arow + (i % vec) * 8) = hv;
          }
        }
      }
    } else {
      const int vec = (2 * ncols) >> 4;
      for (int i = tid; i < kDecBN * vec; i += kDecThreads) {
        const int rr = i / vec, v = i % vec;
        const int src = row_src[rr];
        const unsigned char* gp = act + (size_t)(src < 0 ? 0 : src) * 2 * KDIM + (size_t)2 * col0 + v * 16;
        cp_async16(act_s + rr * sp.arow + v * 16, gp, src < 0 ? 0 : 16);
      }
    }
    if (W4A8) {
      const int nb = ncols >> 5;
      for (int i = tid; i < kDecBN * nb; i += kDecThreads) {
        const int rr = i / nb, b = i % nb;
        const int src = row_src[rr];
        sc_s[rr * nb + b] = src < 0 ? 0.0f : exp2_int((int)a.act_scale[(size_t)src * (KDIM >> 5) + (col0 >> 5) + b] - 127);
      }
    }
    cp_async_commit();
  }

  cp_async_wait<0>();   // activations (and the first weight groups) have landed
  __syncthreads();      // ... for every thread

  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  const uint32_t k16 = 0x10000u + (uint32_t)(d.T >> 30);  // 65536, opaque to the compiler
  const uint32_t nk16 = 0u - k16;
  const int swz = 64 * tsel;
  const int oc0 = (4 * (2 * g + h)) ^ swz, op0 = (4 * ((2 * g + h + 31) & 31)) ^ swz;
  const int oc1 = (4 * (2 * g + 16 + h)) ^ swz, op1 = (4 * (2 * g + 15 + h)) ^ swz;
  const unsigned char* at = act_s + g * sp.arow;
  const int nb = ncols >> 5;

  for (int grp = 0; grp < ngroups; ++grp) {
    if (grp + kDecRing - 1 < ngroups) load_group(grp + kDecRing - 1);
    cp_async_commit();
    cp_async_wait<kDecRing - 1>();
    __syncwarp();
    const unsigned char* wg = myring + (grp % kDecRing) * sp.wslot;
    const int steps = min(kDecGroup, nsteps - grp * kDecGroup);
#pragma unroll
    for (int kk = 0; kk < kDecGroup; ++kk) {
      if (kk < steps) {
        const int ks = grp * kDecGroup + kk;
        const unsigned char* tile = wg + (2 * kk + tsel) * 32 * K;
        uint32_t y0[8], y1[8];
        if (K == 4) {
          const uint32_t c0w = *reinterpret_cast<const uint32_t*>(tile + oc0);
          const uint32_t p0w = *reinterpret_cast<const uint32_t*>(tile + op0);
          const uint32_t c1w = *reinterpret_cast<const uint32_t*>(tile + oc1);
          const uint32_t p1w = *reinterpret_cast<const uint32_t*>(tile + op1);
          run_mcg_k4(p0w, c0w, k16, nk16, y0);
          run_mcg_k4(p1w, c1w, k16, nk16, y1);
        } else {
          uint32_t hi, lo, s8[8];
          int off;
          run_window_smem<K>(reinterpret_cast<const uint16_t*>(tile), 16 * g + 8 * h, hi, lo, off);
          run_states_generic<K>(hi, lo, off, s8);
#pragma unroll
          for (int i = 0; i < 8; ++i) y0[i] = mcg_raw(s8[i]);
          run_window_smem<K>(reinterpret_cast<const uint16_t*>(tile), 16 * (g + 8) + 8 * h, hi, lo, off);
          run_states_generic<K>(hi, lo, off, s8);
#pragma unroll
          for (int i = 0; i < 8; ++i) y1[i] = mcg_raw(s8[i]);
        }
        if (W4A8) {
          uint32_t wa[4], wb[4];
          raw_to_e4m3_f16(y0, wa);
          raw_to_e4m3_f16(y1, wb);
          const uint32_t a0[4] = {wa[0], wb[0], wa[1], wb[1]};
          const uint32_t a1[4] = {wa[2], wb[2], wa[3], wb[3]};
          const uint4 bv = *reinterpret_cast<const uint4*>(at + 64 * ks + 32 * tsel + 16 * h);
          float dd[4] = {0.f, 0.f, 0.f, 0.f};
          mma_f16_16816(dd, a0, bv.x, bv.y);
          mma_f16_16816(dd, a1, bv.z, bv.w);
          const float s0 = sc_s[(2 * q) * nb + ks];
          const float s1 = sc_s[(2 * q + 1) * nb + ks];
          acc[0] = fmaf(dd[0], s0, acc[0]);
          acc[1] = fmaf(dd[1], s1, acc[1]);
          acc[2] = fmaf(dd[2], s0, acc[2]);
          acc[3] = fmaf(dd[3], s1, acc[3]);
        } else {
          uint32_t wa[4], wb[4];
          raw_to_f16(y0, wa);
          raw_to_f16(y1, wb);
          const uint32_t a0[4] = {wa[0], wb[0], wa[1], wb[1]};
          const uint32_t a1[4] = {wa[2], wb[2], wa[3], wb[3]};
          const uint4 bv = *reinterpret_cast<const uint4*>(at + 64 * ks + 32 * tsel + 16 * h);
          mma_f16_16816(acc, a0, bv.x, bv.y);
          mma_f16_16816(acc, a1, bv.z, bv.w);
        }
      }
    }
    __syncwarp();
  }
  cp_async_wait<0>();
  griddep_launch();

  // ---- partial sums of this CTA (valid route columns only) ----
  const int unit = rb * d.units_m + mb;
  float* pbase = d.partial + (size_t)(unit * d.ksplit + sidx) * U * kDecBN;
  const int r0 = lr + g, c0 = 2 * q;
  if (c0 < nvalid) {
    __stcg(pbase + (size_t)r0 * kDecBN + c0, acc[0]);
    __stcg(pbase + (size_t)(r0 + 8) * kDecBN + c0, acc[2]);
  }
  if (c0 + 1 < nvalid) {
    __stcg(pbase + (size_t)r0 * kDecBN + c0 + 1, acc[1]);
    __stcg(pbase + (size_t)(r0 + 8) * kDecBN + c0 + 1, acc[3]);
  }
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const int old = atomicAdd(&d.unit_cnt[unit], 1);
    *flag = (old == d.parts * d.ksplit - 1) ? 1 : 0;
  }
  __syncthreads();
  if (!*flag) return;
  __threadfence();

  // ---- last CTA of the unit: fixed-order reduction, then the epilogue ----
  float* C = reinterpret_cast<float*>(wring);
  constexpr int CS = kDecBN + 1;
  const float* ubase = d.partial + (size_t)unit * d.ksplit * U * kDecBN;
  // (U * kDecBN / kDecThreads <= 8 values per thread; each split's loads
  // are all in flight before they are added, in split order)
  {
    constexpr int kPer = 2 * 128 * kDecBN / kDecThreads;
    float v[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) v[j] = 0.0f;
    for (int s2 = 0; s2 < d.ksplit; ++s2) {
      float x[kPer];
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int i = tid + j * kDecThreads;
        x[j] = (i < U * kDecBN && (i % kDecBN) < nvalid) ? __ldcg(ubase + (size_t)s2 * U * kDecBN + i) : 0.0f;
      }
#pragma unroll
      for (int j = 0; j < kPer; ++j) v[j] += x[j];
    }
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int i = tid + j * kDecThreads;
      if (i < U * kDecBN) C[(i / kDecBN) * CS + (i % kDecBN)] = v[j];
    }
  }
  __syncthreads();
  if (tid == 0) d.unit_cnt[unit] = 0;
  if (PROJ == 1) {
    if (d.bi == 128)
      dec_epilogue_fc1<4, W4A8>(a, e, mb, slot0, C, row_slot);
    else
      dec_epilogue_fc1<2, W4A8>(a, e, mb, slot0, C, row_slot);
  } else {
    dec_epilogue_fc2(d, e, mb, slot0, C, row_slot);
  }
}

template <bool W4A8, int PROJ, int KB>
__global__ void __launch_bounds__(kDecThreads) k_dec_fc(const DecArgs d) {
  extern __shared__ __align__(128) unsigned char smem[];
  griddep_wait();
  const int rb = blockIdx.x;
  if (rb >= *d.f.nblocks) return;
  const int mb = blockIdx.y / d.parts, part = blockIdx.y % d.parts, sidx = blockIdx.z;
  const int e = d.f.block_expert[rb];
  if (KB > 0) {
    dec_body<W4A8, PROJ, (KB > 0 ? KB : 4), (KB > 0 ? KB : 6)>(d, rb, mb, part, sidx, e, smem);
  } else {
    switch (d.f.bits[e]) {
      case 2: dec_body<W4A8, PROJ, 2, 6>(d, rb, mb, part, sidx, e, smem); break;
      case 3: dec_body<W4A8, PROJ, 3, 6>(d, rb, mb, part, sidx, e, smem); break;
      case 4: dec_body<W4A8, PROJ, 4, 6>(d, rb, mb, part, sidx, e, smem); break;
      case 5: dec_body<W4A8, PROJ, 5, 6>(d, rb, mb, part, sidx, e, smem); break;
      default: dec_body<W4A8, PROJ, 6, 6>(d, rb, mb, part, sidx, e, smem); break;
    }
  }
}

int dec_ksplit(int kdim, long units) {
  const long want = (kDecTargetCtas + units - 1) / std::max<long>(units, 1);
  const int maxs = std::max(1, kdim / 128);
  const int mins = (kdim + kDecMaxChunk - 1) / kDecMaxChunk;
  return (int)std::max<long>(mins, std::max<long>(1, std::min<long>(want, maxs)));
}

template <bool W4A8, int PROJ, int KB>
static cudaError_t launch_dec_t(const DecArgs& d, int max_blocks, cudaStream_t st) {
  const int smem = dec_smem_plan(W4A8, KB > 0 ? KB : 6, d.kchunk).total;
  auto kern = k_dec_fc<W4A8, PROJ, KB>;
  // The shared-memory limit is raised once, to the most any call can use,
  // before any capture (the first forward call).
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           dec_smem_plan(W4A8, KB > 0 ? KB : 6, kDecMaxChunk).total);
    if (err != cudaSuccess) return err;
    attr_done = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(max_blocks, d.units_m * d.parts, d.ksplit);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, d);
}

cudaError_t launch_dec_fc(const DecArgs& d, int proj, bool w4a8, int uniform_k, int max_blocks, cudaStream_t st) {
  const bool k4 = uniform_k == 4;
  if (proj == 1) {
    if (w4a8) return k4 ? launch_dec_t<true, 1, 4>(d, max_blocks, st) : launch_dec_t<true, 1, 0>(d, max_blocks, st);
    return k4 ? launch_dec_t<false, 1, 4>(d, max_blocks, st) : launch_dec_t<false, 1, 0>(d, max_blocks, st);
  }
  if (w4a8) return k4 ? launch_dec_t<true, 2, 4>(d, max_blocks, st) : launch_dec_t<true, 2, 0>(d, max_blocks, st);
  return k4 ? launch_dec_t<false, 2, 4>(d, max_blocks, st) : launch_dec_t<false, 2, 0>(d, max_blocks, st);
}

}  // namespace tmoe
