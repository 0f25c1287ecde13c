// Device bodies of the router and the route map, shared by the stand-alone
// kernels (route.cu) and the fused decode prologue (dec.cu).
#pragma once

#include "launch.h"

namespace tmoe {

// ---------------------------------------------------------------------------
// Router: one warp per token.
// ---------------------------------------------------------------------------
// Top-k of token t's logits (E <= 256) by the calling warp; writes ids and
// weights of row t.
static __device__ __forceinline__ void route_token_warp(const float* __restrict__ logits, int t, int E, int k,
                                                        int32_t* __restrict__ ids, float* __restrict__ w) {
  const int warp = t;
  const int lane = threadIdx.x & 31;
  const float* row = logits + (size_t)warp * E;
  float v[8];
  uint32_t taken = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane + 32 * i;
    v[i] = (e < E) ? row[e] : 0.0f;
    if (e >= E) taken |= 1u << i;
  }
  float best0 = 0.0f, wsum = 0.0f, my_w = 0.0f;
  int my_id = 0;
  for (int j = 0; j < k; ++j) {
    // lane-local best: larger value, then lower id
    float bv = -INFINITY;
    int bid = 0x7FFFFFFF;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      if (!(taken & (1u << i)) && (v[i] > bv || (v[i] == bv && e < bid) || bid == 0x7FFFFFFF)) {
        bv = v[i];
        bid = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
      const int oid = __shfl_xor_sync(0xFFFFFFFFu, bid, o);
      if (oid != 0x7FFFFFFF && (bid == 0x7FFFFFFF || ov > bv || (ov == bv && oid < bid))) {
        bv = ov;
        bid = oid;
      }
    }
    if ((bid & 31) == lane) taken |= 1u << (bid >> 5);
    if (j == 0) best0 = bv;
    const float ex = __expf(bv - best0);
    wsum += ex;
    if (lane == j) {
      my_id = bid;
      my_w = ex;
    }
  }
  if (lane < k) {
    ids[(size_t)warp * k + lane] = my_id;
    w[(size_t)warp * k + lane] = my_w / wsum;
  }
}

// ---------------------------------------------------------------------------
// Route map. A "tile" is 1024 consecutive routes, one per thread.
// Phase A (per tile): stable rank of each route among the tile's routes of the
// same expert, and the tile's per-expert counts.
// ---------------------------------------------------------------------------
constexpr int kRouteTile = 1024;

struct RankScratch {
  int cnt[32][kMaxExperts];  // per-warp counts, then per-warp exclusive prefixes
};

// Computes local ranks for the routes of tile `tile` into `rank` (-1 = dropped
// id) and the tile's per-expert totals into `tile_count[E]`.
static __device__ __forceinline__ void tile_rank(const int32_t* __restrict__ ids, int R, int E, int tile, RankScratch& sm,
                          int32_t* __restrict__ rank, int32_t* __restrict__ tile_count,
                          uint32_t* __restrict__ err) {
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  // only the warps that hold routes of this tile take part in the counts
  const int nw = min(32, (R - tile * kRouteTile + 31) / 32);
  for (int i = tid; i < nw * E; i += blockDim.x) (&sm.cnt[0][0])[(i / E) * kMaxExperts + (i % E)] = 0;
  __syncthreads();
  const int r = tile * kRouteTile + tid;
  int e = -1;
  if (r < R) {
    e = ids[r];
    if (e < 0 || e >= E) {
      atomicOr(err, 1u);
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
    tile_count[x] = run;
  }
  __syncthreads();
  if (r < R) rank[r] = (e >= 0) ? sm.cnt[warp][e] + lane_rank : -1;
}

// Phase B (one CTA): per-expert running sum over tiles -> tile bases and
// counts; padded exclusive scan over experts -> offsets; route-block table.
static __device__ __forceinline__ void scan_experts(int E, int ntiles, int block, int32_t* __restrict__ tile_counts,
                             int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                             int32_t* __restrict__ block_expert, int32_t* __restrict__ nblocks) {
  __shared__ int s_pad[kMaxExperts + 1];
  const int tid = threadIdx.x;
  for (int e = tid; e < E; e += blockDim.x) {
    int run = 0;
    for (int t = 0; t < ntiles; ++t) {
      const int c = tile_counts[(size_t)t * E + e];
      tile_counts[(size_t)t * E + e] = run;  // becomes the tile's base within the expert
      run += c;
    }
    counts[e] = run;
    s_pad[e] = (run + block - 1) / block;  // route blocks of this expert
  }
  __syncthreads();
  if (tid < 32) {
    // exclusive scan of the per-expert block counts by one warp: each lane
    // sums a contiguous run of up to 8 experts, then the lanes scan
    const int lane = tid;
    const int per = (E + 31) / 32;
    const int b0 = min(E, lane * per), b1 = min(E, b0 + per);
    int local = 0;
    for (int e = b0; e < b1; ++e) local += s_pad[e];
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += v;
    }
    int acc = incl - local;
    for (int e = b0; e < b1; ++e) {
      const int nb = s_pad[e];
      s_pad[e] = acc;
      acc += nb;
    }
    if (lane == 31) {
      s_pad[E] = incl;
      *nblocks = incl;
    }
  }
  __syncthreads();
  for (int e = tid; e <= E; e += blockDim.x) offsets[e] = s_pad[e] * block;
  for (int e = tid; e < E; e += blockDim.x) {
    for (int b = s_pad[e]; b < s_pad[e + 1]; ++b) block_expert[b] = e;
  }
}

// Phase C: scatter routes to their slots and mark padding slots -1.
static __device__ __forceinline__ void pack_routes(const int32_t* __restrict__ ids, int R, int E, int block, int gtid, int gstride,
                            const int32_t* __restrict__ rank, const int32_t* __restrict__ tile_base,
                            const int32_t* __restrict__ counts, const int32_t* __restrict__ offsets,
                            int32_t* __restrict__ route_of_slot, int32_t* __restrict__ slot_of_route) {
  for (int r = gtid; r < R; r += gstride) {
    const int rk = rank[r];
    if (rk < 0) {
      slot_of_route[r] = -1;
      continue;
    }
    const int e = ids[r];
    const int slot = offsets[e] + tile_base[(size_t)(r / kRouteTile) * E + e] + rk;
    route_of_slot[slot] = r;
    slot_of_route[r] = slot;
  }
  for (int i = gtid; i < E * block; i += gstride) {
    const int e = i / block, p = i % block;
    const int s = offsets[e] + counts[e] + p;
    if (s < offsets[e + 1]) route_of_slot[s] = -1;
  }
}

}  // namespace tmoe
