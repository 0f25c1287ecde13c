// Route-major grouped GEMM over trellis-coded expert weights, with the FC1
// activation epilogue or the FC2 unrotation epilogue fused in (sm_103a).
//
// FC1 (b12x PR #129 "feat(moe): serve canonical Fruit QSRT atoms", Hot path):
// one route-major output row per route, gate and up from the same CTA so the
// epilogue H -> svh -> SiLU(gate)*up -> suh_down -> H (sparkinfer PR #90
// "moe: integrate EXL3 Trellis into the fused W4A16 API", review of kernel.py:
// _run_activation) runs on the accumulators. FC2 stays route-major; its
// epilogue scales, applies H and down_svh (b12x PR #129, review of
// trellis_w4a8.py: down_svh in the top-k sum) and either stores the per-slot
// row (deterministic combine) or adds w * row into the output with FP32
// atomics (b12x PR #433 "Share trellis preparation across native and EXL3
// containers": opt-in FP32 atomic prefill reduction, not bitwise ordered).
//
// Weights are never materialised: each thread expands the trellis states of
// the tile rows it owns directly into mma.sync A-operand registers (fp16 for
// W4A16, E4M3 for W4A8; b12x PR #129, Hot path: "expands fixed-stride trellis
// payload directly into E4M3 MMA operands").
//
// Operand mapping. The CTA's weight rows are the MMA M dimension (swap-AB),
// routes the N dimension. For one 32-wide k-step, thread (g = lane/4,
// q = lane%4) of a warp owns, in each of its 16-row m-tiles, rows g and g+8
// of trellis tile (tn, 2*kstep + q/2) and the run of 8 consecutive states
// j = 16*row + 8*(q%2) .. +7 of each: actual columns kb .. kb+7 with
// kb = 32*kstep + 16*(q/2) + 8*(q%2). The MMA's k index is a permutation of
// the actual column, and the B operand (activations) is loaded with the same
// permutation, so the contraction is unchanged:
//   f16 m16n8k16 (two per k-step, i = 0, 1): A regs {(g, 2q..2q+1),
//     (g+8, ..), (g, 2q+8..+9), (g+8, ..)} <- run positions 4i + {0,1}, 4i + {2,3};
//   e4m3 m16n8k32 (one per k-step): A regs {(g, 4q..4q+3), (g+8, ..),
//     (g, 4q+16..+19), (g+8, ..)} <- run positions 0..3 and 4..7.
// One k-step of 32 columns is exactly one MXFP8 scale block, so the W4A8
// product of each k-step is scaled by the route's 2^e before accumulation.
#pragma once

#include "launch.h"

namespace tmoe {

constexpr int kFcThreads = 256;
constexpr int kFcWarps = 8;
constexpr int kKC = 64;        // activation columns per pipeline stage
constexpr int kStages = 4;

template <bool W4A8, int BN>
struct FcSmem {
  // activation stage row stride in bytes (keeps the 8-lane LDS phases
  // conflict-free: 192 = 64 mod 128 for 16-byte loads, 96 for 8-byte loads)
  static constexpr int kRowBytes = W4A8 ? 96 : 192;
  static constexpr int kStageBytes = BN * kRowBytes;
  static constexpr int kScaleFloats = W4A8 ? BN * (kKC / 32) : 0;
};

template <int MROWS, int BN>
__host__ __device__ constexpr int fc_smem_bytes(bool w4a8) {
  return (((MROWS * (BN + 4) * 4) > (kStages * BN * (w4a8 ? 96 : 192) + kStages * BN * 2 * 4))
              ? (MROWS * (BN + 4) * 4)
              : (kStages * BN * (w4a8 ? 96 : 192) + kStages * BN * 2 * 4)) +
         BN * 4 * 2;
}

// One CTA: route block rb (BN slots of one expert) x row block mb.
template <bool W4A8, int PROJ, int KB, int MROWS, int BN>
__device__ __forceinline__ void fc_body(const FcArgs& a, int e, int rb, int mb, unsigned char* smem) {
  constexpr int MT = MROWS / 16;
  constexpr int MPW = MT / kFcWarps;
  constexpr int NT = BN / 8;
  static_assert(MPW >= 1 && MT % kFcWarps == 0, "row block must cover 8 warps");
  using S = FcSmem<W4A8, BN>;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, q = lane & 3;
  const int KDIM = (PROJ == 1) ? a.H : a.I;
  const int NROWS = (PROJ == 1) ? 2 * a.I : a.H;  // rows of the expert's matrix
  const int tiles_k = KDIM >> 4;
  const int kbits = (KB > 0) ? KB : (int)a.bits[e];
  const int tile_words = 16 * kbits;
  const uint16_t* wbase = reinterpret_cast<const uint16_t*>(a.payload) + a.word_off[e];

  unsigned char* stage_base = smem;
  float* scale_base = reinterpret_cast<float*>(smem + kStages * S::kStageBytes);
  int* row_src = reinterpret_cast<int*>(smem + fc_smem_bytes<MROWS, BN>(W4A8) - BN * 4 * 2);
  int* row_slot = row_src + BN;

  const int slot0 = rb * BN;
  if (tid < BN) {
    const int slot = slot0 + tid;
    const int r = a.route_of_slot[slot];
    row_slot[tid] = r;  // route id or -1
    if (PROJ == 1)
      row_src[tid] = (r >= 0) ? (r / a.topk) : -1;  // token row of x~
    else
      row_src[tid] = slot;  // z~ is slot-indexed (padding rows are zero)
  }
  __syncthreads();

  // ---- tile rows owned by this warp: for m-tile i, matrix row block tn_i ----
  int tn[MPW];
#pragma unroll
  for (int i = 0; i < MPW; ++i) {
    const int lr = (warp * MPW + i) * 16;  // local row of the m-tile
    int row;
    if (PROJ == 1) {
      const int BI = MROWS / 2;
      row = (lr < BI) ? (mb * BI + lr) : (a.I + mb * BI + (lr - BI));
    } else {
      row = mb * MROWS + lr;
    }
    tn[i] = row >> 4;
  }
  (void)NROWS;

  // ---- activation stage loader ----
  const int act_row_bytes = W4A8 ? KDIM : 2 * KDIM;
  const unsigned char* act = reinterpret_cast<const unsigned char*>(a.act);
  const int nchunks = KDIM / kKC;
  auto load_stage = [&](int chunk, int buf) {
    unsigned char* dst = stage_base + buf * S::kStageBytes;
    constexpr int kChunkBytes = W4A8 ? kKC : 2 * kKC;
    constexpr int kVec = kChunkBytes / 16;  // 16-byte pieces per row
    for (int i = tid; i < BN * kVec; i += kFcThreads) {
      const int rr = i / kVec, v = i % kVec;
      const int src = row_src[rr];
      const unsigned char* gp = act + (size_t)(src < 0 ? 0 : src) * act_row_bytes + (size_t)chunk * kChunkBytes + v * 16;
      cp_async16(dst + rr * S::kRowBytes + v * 16, gp, src < 0 ? 0 : 16);
    }
    if (W4A8) {
      float* sc = scale_base + buf * BN * 2;
      for (int i = tid; i < BN * 2; i += kFcThreads) {
        const int rr = i >> 1, blk = i & 1;
        const int src = row_src[rr];
        float f = 0.0f;
        if (src >= 0) f = exp2_int((int)a.act_scale[(size_t)src * (KDIM >> 5) + chunk * 2 + blk] - 127);
        sc[i] = f;
      }
    }
  };

  float acc[MPW][NT][4];
#pragma unroll
  for (int i = 0; i < MPW; ++i)
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[i][n][c] = 0.0f;

  // per-thread run coordinates inside a tile
  const int h = q & 1;
  const int ktile_off = q >> 1;

#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) {
    if (s < nchunks) load_stage(s, s);
    cp_async_commit();
  }

  for (int chunk = 0; chunk < nchunks; ++chunk) {
    {
      const int nxt = chunk + kStages - 1;
      if (nxt < nchunks) load_stage(nxt, nxt % kStages);
      cp_async_commit();
    }
    cp_async_wait<kStages - 1>();
    __syncthreads();
    const int buf = chunk % kStages;
    const unsigned char* st = stage_base + buf * S::kStageBytes;
    const float* sc = scale_base + buf * BN * 2;
#pragma unroll
    for (int ks = 0; ks < kKC / 32; ++ks) {
      const int kstep = chunk * (kKC / 32) + ks;
      const int tk = 2 * kstep + ktile_off;
      // ---- decode A operands ----
      uint32_t afr[MPW][W4A8 ? 4 : 8];
#pragma unroll
      for (int i = 0; i < MPW; ++i) {
        const uint16_t* tile = wbase + ((size_t)tn[i] * tiles_k + tk) * tile_words;
        uint32_t sA[8], sB[8];
        if (KB == 4 || (KB == 0 && kbits == 4)) {
          uint32_t p0, c0, p1, c1;
          run_load_k4(tile, g, h, p0, c0);
          run_load_k4(tile, g + 8, h, p1, c1);
          run_states_k4(p0, c0, sA);
          run_states_k4(p1, c1, sB);
        } else {
          uint32_t hi0, lo0, hi1, lo1;
          int off0, off1;
          switch (kbits) {
            case 2: run_window_generic<2>(tile, 16 * g + 8 * h, hi0, lo0, off0);
                    run_window_generic<2>(tile, 16 * (g + 8) + 8 * h, hi1, lo1, off1);
                    run_states_generic<2>(hi0, lo0, off0, sA); run_states_generic<2>(hi1, lo1, off1, sB); break;
            case 3: run_window_generic<3>(tile, 16 * g + 8 * h, hi0, lo0, off0);
                    run_window_generic<3>(tile, 16 * (g + 8) + 8 * h, hi1, lo1, off1);
                    run_states_generic<3>(hi0, lo0, off0, sA); run_states_generic<3>(hi1, lo1, off1, sB); break;
            case 5: run_window_generic<5>(tile, 16 * g + 8 * h, hi0, lo0, off0);
                    run_window_generic<5>(tile, 16 * (g + 8) + 8 * h, hi1, lo1, off1);
                    run_states_generic<5>(hi0, lo0, off0, sA); run_states_generic<5>(hi1, lo1, off1, sB); break;
            default: run_window_generic<6>(tile, 16 * g + 8 * h, hi0, lo0, off0);
                    run_window_generic<6>(tile, 16 * (g + 8) + 8 * h, hi1, lo1, off1);
                    run_states_generic<6>(hi0, lo0, off0, sA); run_states_generic<6>(hi1, lo1, off1, sB); break;
          }
        }
        if (W4A8) {
          uint32_t qa[2], qb[2];
          run_weights_e4m3(sA, qa);
          run_weights_e4m3(sB, qb);
          afr[i][0] = qa[0];
          afr[i][1] = qb[0];
          afr[i][2] = qa[1];
          afr[i][3] = qb[1];
        } else {
          uint32_t wa[4], wb[4];
          run_weights_f16(sA, wa);
          run_weights_f16(sB, wb);
          // MMA 0: positions 0..3; MMA 1: positions 4..7
          afr[i][0] = wa[0]; afr[i][1] = wb[0]; afr[i][2] = wa[1]; afr[i][3] = wb[1];
          afr[i][4] = wa[2]; afr[i][5] = wb[2]; afr[i][6] = wa[3]; afr[i][7] = wb[3];
        }
      }
      // ---- B operands per n-tile, MMAs ----
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        const int rr = n * 8 + g;
        if (W4A8) {
          const uint2 bv = *reinterpret_cast<const uint2*>(st + rr * S::kRowBytes + ks * 32 + 16 * ktile_off + 8 * h);
          const float s0 = sc[(n * 8 + 2 * q) * 2 + ks];
          const float s1 = sc[(n * 8 + 2 * q + 1) * 2 + ks];
#pragma unroll
          for (int i = 0; i < MPW; ++i) {
            float d[4];
            const uint32_t af[4] = {afr[i][0], afr[i][1], afr[i][2], afr[i][3]};
            mma_e4m3_16832(d, af, bv.x, bv.y);
            acc[i][n][0] = fmaf(d[0], s0, acc[i][n][0]);
            acc[i][n][1] = fmaf(d[1], s1, acc[i][n][1]);
            acc[i][n][2] = fmaf(d[2], s0, acc[i][n][2]);
            acc[i][n][3] = fmaf(d[3], s1, acc[i][n][3]);
          }
        } else {
          const uint4 bv = *reinterpret_cast<const uint4*>(st + rr * S::kRowBytes + ks * 64 + 32 * ktile_off + 16 * h);
#pragma unroll
          for (int i = 0; i < MPW; ++i) {
            const uint32_t a0[4] = {afr[i][0], afr[i][1], afr[i][2], afr[i][3]};
            const uint32_t a1[4] = {afr[i][4], afr[i][5], afr[i][6], afr[i][7]};
            mma_f16_16816(acc[i][n], a0, bv.x, bv.y);
            mma_f16_16816(acc[i][n], a1, bv.z, bv.w);
          }
        }
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();
  __syncthreads();

  // ---- accumulators -> shared C[row][col] ----
  float* C = reinterpret_cast<float*>(smem);
  constexpr int CS = BN + 4;
#pragma unroll
  for (int i = 0; i < MPW; ++i) {
    const int r0 = (warp * MPW + i) * 16 + g;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      const int c0 = n * 8 + 2 * q;
      C[r0 * CS + c0] = acc[i][n][0];
      C[r0 * CS + c0 + 1] = acc[i][n][1];
      C[(r0 + 8) * CS + c0] = acc[i][n][2];
      C[(r0 + 8) * CS + c0 + 1] = acc[i][n][3];
    }
  }
  __syncthreads();

  // ---- epilogue: one warp per route column ----
  if (PROJ == 1) {
    constexpr int BI = MROWS / 2;
    constexpr int PER = BI / 32;
    const uint16_t* s1 = a.scale + (size_t)e * 2 * a.I;
    const uint16_t* rt = a.rot_tab + (size_t)e * 3 * a.I;
    const int c0 = mb * BI + lane * PER;  // first intermediate channel of this lane
    float sg[PER], su[PER], vg[PER], vu[PER], vd[PER];
#pragma unroll
    for (int p = 0; p < PER; ++p) {
      sg[p] = __half2float(__ushort_as_half(s1[c0 + p]));
      su[p] = __half2float(__ushort_as_half(s1[a.I + c0 + p]));
      vg[p] = __half2float(__ushort_as_half(rt[c0 + p]));
      vu[p] = __half2float(__ushort_as_half(rt[a.I + c0 + p]));
      vd[p] = __half2float(__ushort_as_half(rt[2 * a.I + c0 + p]));
    }
    const float hs = hadamard_scale(a.rot_b);
    for (int col = warp; col < BN; col += kFcWarps) {
      const int slot = slot0 + col;
      const bool valid = row_slot[col] >= 0;
      float gv[PER], uv[PER];
#pragma unroll
      for (int p = 0; p < PER; ++p) {
        gv[p] = C[(lane * PER + p) * CS + col] * sg[p];
        uv[p] = C[(BI + lane * PER + p) * CS + col] * su[p];
      }
      warp_fwht<PER>(gv, a.rot_b);
      warp_fwht<PER>(uv, a.rot_b);
      float av[PER];
#pragma unroll
      for (int p = 0; p < PER; ++p) {
        const float gg = gv[p] * hs * vg[p];
        const float uu = uv[p] * hs * vu[p];
        av[p] = (gg / (1.0f + __expf(-gg))) * uu * vd[p];
      }
      warp_fwht<PER>(av, a.rot_b);
#pragma unroll
      for (int p = 0; p < PER; ++p) av[p] = valid ? av[p] * hs : 0.0f;
      if (!W4A8) {
        uint16_t* z = reinterpret_cast<uint16_t*>(a.out_act) + (size_t)slot * a.I + c0;
        if (PER == 4) {
          __half2 x0 = __floats2half2_rn(av[0], av[1]);
          __half2 x1 = __floats2half2_rn(av[PER > 2 ? 2 : 0], av[PER > 3 ? 3 : 0]);
          uint2 o;
          o.x = *reinterpret_cast<uint32_t*>(&x0);
          o.y = *reinterpret_cast<uint32_t*>(&x1);
          *reinterpret_cast<uint2*>(z) = o;
        } else {
          __half2 x0 = __floats2half2_rn(av[0], av[PER > 1 ? 1 : 0]);
          *reinterpret_cast<__half2*>(z) = x0;
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
        if (PER == 4) {
          const uint32_t qv = e4m3x2_from_float2(av[0] * inv, av[1] * inv) |
                              (e4m3x2_from_float2(av[PER > 2 ? 2 : 0] * inv, av[PER > 3 ? 3 : 0] * inv) << 16);
          *reinterpret_cast<uint32_t*>(z) = qv;
        } else {
          *reinterpret_cast<uint16_t*>(z) = (uint16_t)e4m3x2_from_float2(av[0] * inv, av[PER > 1 ? 1 : 0] * inv);
        }
        if ((lane % LPB) == 0)
          a.out_scale[(size_t)slot * (a.I >> 5) + (c0 >> 5)] = valid ? (uint8_t)(ex + 127) : (uint8_t)0;
      }
    }
  } else {
    const uint16_t* s2 = a.scale + (size_t)e * a.H;
    const uint16_t* sv = a.rot_tab + (size_t)e * a.H;  // out_svh
    const int h0 = mb * MROWS + lane * 4;
    float sc2[4], svh[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      sc2[p] = __half2float(__ushort_as_half(s2[h0 + p]));
      svh[p] = __half2float(__ushort_as_half(sv[h0 + p]));
    }
    const float hs = hadamard_scale(a.rot_b);
    for (int col = warp; col < BN; col += kFcWarps) {
      const int r = row_slot[col];
      if (r < 0) continue;  // padding slot: nothing to store
      float v[4];
#pragma unroll
      for (int p = 0; p < 4; ++p) v[p] = C[(lane * 4 + p) * CS + col] * sc2[p];
      warp_fwht<4>(v, a.rot_b);
#pragma unroll
      for (int p = 0; p < 4; ++p) v[p] = v[p] * hs * svh[p];
      if (!a.atomic) {
        float4 o = make_float4(v[0], v[1], v[2], v[3]);
        *reinterpret_cast<float4*>(a.out_f32 + (size_t)(slot0 + col) * a.H + h0) = o;
      } else {
        const int t = r / a.topk;
        const float wr = a.route_w[r];
        float* dst = a.out_f32 + (size_t)t * a.H + h0;
#pragma unroll
        for (int p = 0; p < 4; ++p) atomicAdd(dst + p, wr * v[p]);
      }
    }
  }
}

template <bool W4A8, int PROJ, int KB, int MROWS, int BN>
__global__ void __launch_bounds__(kFcThreads, 2) k_fc(const FcArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int rb = blockIdx.x;
  if (rb >= *a.nblocks) return;
  const int mb = blockIdx.y;
  const int e = a.block_expert[rb];
  fc_body<W4A8, PROJ, KB, MROWS, BN>(a, e, rb, mb, smem);
}

template <bool W4A8, int PROJ, int KB, int MROWS, int BN>
cudaError_t launch_fc_t(const FcArgs& a, int max_blocks, cudaStream_t st) {
  const int smem = fc_smem_bytes<MROWS, BN>(W4A8);
  auto kern = k_fc<W4A8, PROJ, KB, MROWS, BN>;
  // Set once per process (the first forward call, which must precede any
  // stream capture of the forward pass).
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    attr_done = true;
  }
  const int rows = (PROJ == 1) ? a.I : a.H;
  const int mblocks = (PROJ == 1) ? rows / (MROWS / 2) : rows / MROWS;
  dim3 grid(max_blocks, mblocks);
  kern<<<grid, kFcThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace tmoe
