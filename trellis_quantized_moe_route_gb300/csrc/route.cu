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
#include "route_dev.cuh"

namespace tmoe {

__global__ void __launch_bounds__(256) k_route_topk(const float* __restrict__ logits, int T, int E, int k,
                                                    int32_t* __restrict__ ids, float* __restrict__ w) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (warp >= T) return;
  route_token_redux(logits + (size_t)warp * E, E, k, warp, ids, w);
}


__global__ void __launch_bounds__(kRouteTile) k_route_rank(const int32_t* __restrict__ ids, int R, int E,
                                                           int32_t* __restrict__ rank,
                                                           int32_t* __restrict__ tile_counts,
                                                           uint32_t* __restrict__ err) {
  __shared__ RankScratch sm;
  tile_rank(ids, R, E, blockIdx.x, sm, rank, tile_counts + (size_t)blockIdx.x * E, err);
}

__global__ void __launch_bounds__(kRouteTile) k_route_scan(int E, int ntiles, int block,
                                                           int32_t* __restrict__ tile_counts,
                                                           int32_t* __restrict__ counts,
                                                           int32_t* __restrict__ offsets,
                                                           int32_t* __restrict__ block_expert,
                                                           int32_t* __restrict__ nblocks) {
  scan_experts(E, ntiles, block, tile_counts, counts, offsets, block_expert, nblocks);
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
