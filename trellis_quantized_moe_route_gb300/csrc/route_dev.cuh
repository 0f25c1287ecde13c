// Device bodies of the router and the route map, shared by the stand-alone
// kernels (route.cu) and the fused decode prologue (dec.cu).
#pragma once

#include "launch.h"

namespace tmoe {

// Orderable key of a finite float (larger float, larger key; -0 as +0) and back.
static __device__ __forceinline__ uint32_t route_key(float f) {
  const uint32_t b = __float_as_uint(f + 0.0f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
static __device__ __forceinline__ float route_unkey(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Top-k selection of one token's logits by one warp: k rounds of a warp-wide
// max of the remaining keys, ties to the lowest expert id. Lane j < k gets the
// j-th selected id and its unnormalised weight exp(l - l_max); *wsum the sum
// of those weights in selection order (every lane).
static __device__ __forceinline__ void route_token_select(const float* __restrict__ row, int E, int k, int& my_id,
                                                          float& my_w, float& wsum) {
  const int lane = threadIdx.x & 31;
  uint32_t key[kMaxExperts / 32];
#pragma unroll
  for (int i = 0; i < kMaxExperts / 32; ++i) {
    const int e = lane + 32 * i;
    key[i] = (e < E) ? route_key(__ldg(row + e)) : 0u;  // 0: absent or taken
  }
  float best0 = 0.0f;
  wsum = 0.0f;
  my_w = 0.0f;
  my_id = 0;
  for (int j = 0; j < k; ++j) {
    uint32_t lm = 0;
#pragma unroll
    for (int i = 0; i < kMaxExperts / 32; ++i) lm = max(lm, key[i]);
    const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, lm);
    uint32_t lid = 0xFFFFFFFFu;
#pragma unroll
    for (int i = kMaxExperts / 32 - 1; i >= 0; --i)
      if (key[i] == m) lid = lane + 32 * i;
    const uint32_t id = __reduce_min_sync(0xFFFFFFFFu, lid);
#pragma unroll
    for (int i = 0; i < kMaxExperts / 32; ++i)
      if (lane + 32 * i == (int)id) key[i] = 0u;
    const float bv = route_unkey(m);
    if (j == 0) best0 = bv;
    const float ex = __expf(bv - best0);
    wsum += ex;
    if (lane == j) {
      my_id = (int)id;
      my_w = ex;
    }
  }
}

// Top-k softmax of one token's logits by one warp (route_token_select); the
// weights are exp(l - l_max) / sum over the selected, summed in selection
// order.
static __device__ __forceinline__ void route_token_redux(const float* __restrict__ row, int E, int k, int t,
                                                int32_t* __restrict__ ids, float* __restrict__ w, int* s_ids = nullptr) {
  const int lane = threadIdx.x & 31;
  int my_id;
  float my_w, wsum;
  route_token_select(row, E, k, my_id, my_w, wsum);
  if (lane < k) {
    ids[(size_t)t * k + lane] = my_id;
    w[(size_t)t * k + lane] = my_w / wsum;
    if (s_ids) s_ids[t * k + lane] = my_id;
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
    // sixteen tiles' counts in flight at a time, then their bases written
    for (int t0 = 0; t0 < ntiles; t0 += 16) {
      int c[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) c[u] = (t0 + u < ntiles) ? tile_counts[(size_t)(t0 + u) * E + e] : 0;
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        if (t0 + u < ntiles) {
          tile_counts[(size_t)(t0 + u) * E + e] = run;  // becomes the tile's base within the expert
          run += c[u];
        }
      }
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
