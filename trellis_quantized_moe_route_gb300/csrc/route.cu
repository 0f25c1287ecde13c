// Router and route map (sm_103a).
//
// Router: top-k of the router logits with the weights renormalised over the k
// selected experts (the workloads' "softmax then top-k renormalised"; routing
// ids and route weights as the outputs of flashinfer PR #69 "b12x fused MoE:
// TrellisMX (procedural NPK) source format with an in-tree P8 runtime",
// commit list, routing ops).
//
// Route map: per-expert counts, an exclusive scan with every expert segment
// padded to the route block size, and a stable (token-major) permutation
// (sparkinfer PR #90 "moe: integrate EXL3 Trellis into the fused W4A16 API",
// review of route_pack.py: count kernel, prefix-from-counts kernel with
// BLOCK_SIZE; b12x PR #433 "Share trellis preparation across native and EXL3
// containers", review of route_pack.py: the stable order should come from
// per-tile expert prefix counts so that each route is read O(1) times).
#include "launch.h"

namespace tmoe {

// ---------------------------------------------------------------------------
// Router: one warp per token.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_route_topk(const float* __restrict__ logits, int T, int E, int k,
                                                    int32_t* __restrict__ ids, float* __restrict__ w) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= T) return;
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
__device__ void tile_rank(const int32_t* __restrict__ ids, int R, int E, int tile, RankScratch& sm,
                          int32_t* __restrict__ rank, int32_t* __restrict__ tile_count,
                          uint32_t* __restrict__ err) {
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < 32 * E; i += blockDim.x) (&sm.cnt[0][0])[(i / E) * kMaxExperts + (i % E)] = 0;
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
    for (int wv = 0; wv < 32; ++wv) {
      const int c = sm.cnt[wv][x];
      sm.cnt[wv][x] = run;
      run += c;
    }
    tile_count[x] = run;
  }
  __syncthreads();
  if (r < R) rank[r] = (e >= 0) ? sm.cnt[warp][e] + lane_rank : -1;
}

__global__ void __launch_bounds__(kRouteTile) k_route_rank(const int32_t* __restrict__ ids, int R, int E,
                                                           int32_t* __restrict__ rank,
                                                           int32_t* __restrict__ tile_counts,
                                                           uint32_t* __restrict__ err) {
  __shared__ RankScratch sm;
  tile_rank(ids, R, E, blockIdx.x, sm, rank, tile_counts + (size_t)blockIdx.x * E, err);
}

// Phase B (one CTA): per-expert running sum over tiles -> tile bases and
// counts; padded exclusive scan over experts -> offsets; route-block table.
__device__ void scan_experts(int E, int ntiles, int block, int32_t* __restrict__ tile_counts,
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
  if (tid == 0) {
    int acc = 0;
    for (int e = 0; e < E; ++e) {
      const int nb = s_pad[e];
      s_pad[e] = acc;
      acc += nb;
    }
    s_pad[E] = acc;
    *nblocks = acc;
  }
  __syncthreads();
  for (int e = tid; e <= E; e += blockDim.x) offsets[e] = s_pad[e] * block;
  for (int e = tid; e < E; e += blockDim.x) {
    for (int b = s_pad[e]; b < s_pad[e + 1]; ++b) block_expert[b] = e;
  }
}

__global__ void __launch_bounds__(kRouteTile) k_route_scan(int E, int ntiles, int block,
                                                           int32_t* __restrict__ tile_counts,
                                                           int32_t* __restrict__ counts,
                                                           int32_t* __restrict__ offsets,
                                                           int32_t* __restrict__ block_expert,
                                                           int32_t* __restrict__ nblocks) {
  scan_experts(E, ntiles, block, tile_counts, counts, offsets, block_expert, nblocks);
}

// Phase C: scatter routes to their slots and mark padding slots -1.
__device__ void pack_routes(const int32_t* __restrict__ ids, int R, int E, int block, int gtid, int gstride,
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

__global__ void __launch_bounds__(256) k_route_pack(const int32_t* __restrict__ ids, int R, int E, int block,
                                                    const int32_t* __restrict__ rank,
                                                    const int32_t* __restrict__ tile_base,
                                                    const int32_t* __restrict__ counts,
                                                    const int32_t* __restrict__ offsets,
                                                    int32_t* __restrict__ route_of_slot,
                                                    int32_t* __restrict__ slot_of_route) {
  pack_routes(ids, R, E, block, blockIdx.x * blockDim.x + threadIdx.x, gridDim.x * blockDim.x, rank,
              tile_base, counts, offsets, route_of_slot, slot_of_route);
}

// All three phases in one CTA, for R <= 1024 routes (one tile).
__global__ void __launch_bounds__(kRouteTile) k_route_map_small(
    const int32_t* __restrict__ ids, int R, int E, int block, int32_t* __restrict__ rank,
    int32_t* __restrict__ tile_counts, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
    int32_t* __restrict__ block_expert, int32_t* __restrict__ nblocks, int32_t* __restrict__ route_of_slot,
    int32_t* __restrict__ slot_of_route, uint32_t* __restrict__ err) {
  __shared__ RankScratch sm;
  tile_rank(ids, R, E, 0, sm, rank, tile_counts, err);
  __syncthreads();
  __threadfence_block();
  scan_experts(E, 1, block, tile_counts, counts, offsets, block_expert, nblocks);
  __syncthreads();
  __threadfence_block();
  pack_routes(ids, R, E, block, threadIdx.x, blockDim.x, rank, tile_counts, counts, offsets, route_of_slot,
              slot_of_route);
}

cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                              cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const int threads = 256;
  const int blocks = (T * 32 + threads - 1) / threads;
  k_route_topk<<<blocks, threads, 0, st>>>(logits, T, E, k, ids, w);
  return cudaGetLastError();
}

cudaError_t launch_route_map(const RouteMapArgs& a, cudaStream_t st) {
  if (a.R <= kRouteTile) {
    k_route_map_small<<<1, kRouteTile, 0, st>>>(a.ids, a.R, a.E, a.block, a.rank, a.tile_counts, a.counts,
                                                a.offsets, a.block_expert, a.nblocks, a.route_of_slot,
                                                a.slot_of_route, a.err);
    return cudaGetLastError();
  }
  const int ntiles = (a.R + kRouteTile - 1) / kRouteTile;
  k_route_rank<<<ntiles, kRouteTile, 0, st>>>(a.ids, a.R, a.E, a.rank, a.tile_counts, a.err);
  k_route_scan<<<1, kRouteTile, 0, st>>>(a.E, ntiles, a.block, a.tile_counts, a.counts, a.offsets,
                                         a.block_expert, a.nblocks);
  const int pack_blocks = (max(a.R, a.E * a.block) + 255) / 256;
  k_route_pack<<<pack_blocks, 256, 0, st>>>(a.ids, a.R, a.E, a.block, a.rank, a.tile_counts, a.counts,
                                            a.offsets, a.route_of_slot, a.slot_of_route);
  return cudaGetLastError();
}

int route_map_tiles(int R) { return (R + kRouteTile - 1) / kRouteTile; }

}  // namespace tmoe
