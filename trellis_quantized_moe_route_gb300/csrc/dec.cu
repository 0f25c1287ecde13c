// Decode-rows path (sm_103a): the layer for a few tokens (T * topk <= 1024),
// where every expert is touched by a handful of routes and the layer is bound
// by streaming and decoding the touched trellis payload (b12x PR #129 "feat(moe):
// serve canonical Fruit QSRT atoms", Hot path: W4A8 only for bounded decode
// rows; the decode expands the payload directly into E4M3 MMA operands).
//
// Three kernels on one stream: this prologue (router when logits are given,
// route map in blocks of 8 slots, and the fused rotate+quantize -- W4A8 keeps
// the E4M3 codes as fp16 next to their E8M0 exponents -- plus the clearing of
// counters and output), then the persistent FC1 and FC2 kernels of decw.cu,
// launched with programmatic dependent launch so that each can be scheduled
// while its predecessor drains. No kernel spins.
#include <algorithm>

#include "rotate_dev.cuh"
#include "route_dev.cuh"

namespace tmoe {

__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

// ---------------------------------------------------------------------------
// Prologue. CTA 0: router (when logits are given) and the route map for R <=
// 1024 routes (one per thread), held in shared memory from the ranks to the
// route-block table; the other CTAs: rotate+quantize (one warp per token x
// chunk of 128 columns, 512 with 512-point rotation blocks), clearing of
// counters and output.
// ---------------------------------------------------------------------------
struct DecRouteSmem {
  int cnt[32][kMaxExperts];  // per-warp counts, then per-warp bases within the expert
  int count[kMaxExperts];
  int boff[kMaxExperts + 1];  // first route block of each expert
  long long off1[kMaxExperts], off2[kMaxExperts];
  int bits[kMaxExperts];
  int ids[1024];
};

__device__ __forceinline__ void dec_route_map(const DecPrologueArgs& a, DecRouteSmem& sm) {
  const RouteMapArgs& r = a.rm;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = r.E, R = r.R;
  // per-expert tables (their loads overlap the router's)
  for (int x = tid; x < E; x += blockDim.x) {
    sm.bits[x] = a.bits[x];
    sm.off1[x] = 2 * (long long)a.word_off1[x];
    sm.off2[x] = 2 * (long long)a.word_off2[x];
  }
  const int nw = (R + 31) / 32;  // warps holding routes
  for (int i = tid; i < nw * E; i += blockDim.x) sm.cnt[i / E][i % E] = 0;
  if (a.logits) {
    for (int t = warp; t < a.T; t += 32) route_token_redux(a.logits + (size_t)t * E, E, a.topk, t, a.ids_out, a.w_out, sm.ids);
  } else {
    for (int i = tid; i < R; i += blockDim.x) sm.ids[i] = r.ids[i];
  }
  __syncthreads();
  // stable rank within the expert: within the warp by lane, across warps by warp
  int e = -1;
  if (tid < R) {
    e = sm.ids[tid];
    if (e < 0 || e >= E) {
      atomicOr(r.err, 1u);
      e = -1;
    }
  }
  const uint32_t same = __match_any_sync(0xFFFFFFFFu, e);
  const int lane_rank = __popc(same & ((1u << lane) - 1u));
  if (e >= 0 && lane_rank == 0) sm.cnt[warp][e] = __popc(same);
  __syncthreads();
  for (int x = tid; x < E; x += blockDim.x) {
    int run = 0;
    for (int wv = 0; wv < nw; ++wv) {
      const int c = sm.cnt[wv][x];
      sm.cnt[wv][x] = run;
      run += c;
    }
    sm.count[x] = run;
  }
  __syncthreads();
  if (warp == 0) {
    // exclusive scan of the experts' block counts: each lane a contiguous run
    const int per = (E + 31) / 32;
    const int b0 = min(E, lane * per), b1 = min(E, b0 + per);
    int local = 0;
    for (int x = b0; x < b1; ++x) local += (sm.count[x] + kDecBlock - 1) / kDecBlock;
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += v;
    }
    int acc = incl - local;
    for (int x = b0; x < b1; ++x) {
      sm.boff[x] = acc;
      acc += (sm.count[x] + kDecBlock - 1) / kDecBlock;
    }
    if (lane == 31) sm.boff[E] = incl;
  }
  __syncthreads();
  const int nbl = sm.boff[E];
  if (tid == 0) *r.nblocks = nbl;
  if (tid < R) {
    int slot = -1;
    if (e >= 0) {
      slot = sm.boff[e] * kDecBlock + sm.cnt[warp][e] + lane_rank;
      r.route_of_slot[slot] = tid;
    }
    r.slot_of_route[tid] = slot;
  }
  for (int i = tid; i < E * kDecBlock; i += blockDim.x) {
    const int x = i / kDecBlock, p = i % kDecBlock;
    const int s = sm.boff[x] * kDecBlock + sm.count[x] + p;
    if (s < sm.boff[x + 1] * kDecBlock) r.route_of_slot[s] = -1;
  }
  for (int x = tid; x <= E; x += blockDim.x) {
    r.offsets[x] = sm.boff[x] * kDecBlock;
    if (x < E) r.counts[x] = sm.count[x];
  }
  // route-block table: expert, bits, valid slots (a prefix of the block), payload offsets
  for (int x = tid; x < E; x += blockDim.x) {
    for (int b = sm.boff[x]; b < sm.boff[x + 1]; ++b) {
      const int nv = min(kDecBlock, sm.count[x] - (b - sm.boff[x]) * kDecBlock);
      r.block_expert[b] = x;
      if (b < a.max_blocks) {
        a.blk_meta[b] = x | (sm.bits[x] << 16) | (nv << 24);
        a.blk_off1[b] = sm.off1[x];
        a.blk_off2[b] = sm.off2[x];
      }
    }
  }
  for (int b = nbl + tid; b < a.max_blocks; b += blockDim.x) {
    a.blk_meta[b] = 0;
    a.blk_off1[b] = 0;
    a.blk_off2[b] = 0;
  }
}

// The prologue's rotation of warp gw (PER values per lane: rot_per).
template <int PER>
__device__ __forceinline__ void dec_rotate(const DecPrologueArgs& a, int gw) {
  if (a.split_signs) {
    // one gate and one up rotation per route (their rows indexed by route);
    // with logits the warp selects its token's experts itself, as CTA 0 does
    if (a.w4a8)
      rotate_routes_warp<true, PER>(a.rr, gw);
    else
      rotate_routes_warp<false, PER>(a.rr, gw);
  } else if (a.w4a8) {
    rotate_quant_warp<true, PER>(a.x, a.suh, a.T, a.H, a.rot_b, a.xq, a.xs, gw, nullptr, 0, true, a.xq_scaled);
  } else {
    rotate_quant_warp<false, PER>(a.x, a.suh, a.T, a.H, a.rot_b, a.xq, a.xs, gw);
  }
}

template <int PER>
__global__ void __launch_bounds__(1024) k_dec_prologue(const DecPrologueArgs a) {
  const int tid = threadIdx.x, warp = tid >> 5;
  griddep_launch();  // FC1's CTAs may take free SMs now; they wait for this grid to finish
  if (blockIdx.x == 0) {
    __shared__ DecRouteSmem sm;
    if (tid == 0) *a.rm.err = 0;  // ordered before the rank's flags by the barriers
    dec_route_map(a, sm);
    return;
  }
  const int nrot = gridDim.x - 1;
  const int cta = blockIdx.x - 1;
  // a.rot_per rotation warps per CTA, so that the W4A8 rotation's fp64
  // butterflies spread over many SMs' fp64 units
  const int gw = (warp < a.rot_per) ? cta * a.rot_per + warp : 0x7FFFFFFF;
  dec_rotate<PER>(a, gw);
  const long gtid = (long)cta * blockDim.x + tid, gstride = (long)nrot * blockDim.x;
  for (long i = gtid; i < a.n_zero_i32; i += gstride) a.zero_i32[i] = 0;
  for (long i = gtid; i < a.out_n / 4; i += gstride) reinterpret_cast<float4*>(a.out)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

cudaError_t launch_dec_prologue(const DecPrologueArgs& a_in, cudaStream_t st) {
  // one rotation warp per CTA while the SMs last (T*H/128 warps), then more
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
  }
  DecPrologueArgs a = a_in;
  const long warps = (long)a.T * (a.H / (32 * rot_per(a.rot_b)));
  const long slots = std::max(1, sms - 1);
  a.rot_per = (int)std::min<long>(32, std::max<long>(1, (warps + slots - 1) / slots));
  const int nrot = (int)std::max<long>(1, (warps + a.rot_per - 1) / a.rot_per);
  // (one kernel per rotation width, so that the 512-point variant's
  // registers do not constrain the common one)
  if (a.rot_b > 128)
    k_dec_prologue<16><<<1 + nrot, 1024, 0, st>>>(a);
  else
    k_dec_prologue<4><<<1 + nrot, 1024, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace tmoe
