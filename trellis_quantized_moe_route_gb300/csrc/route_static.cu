// Route map that needs no scratch from its caller.
//
// trellis_moe_route_map takes a caller-provided workspace for its scratch
// (per-route ranks, per-tile counts, the route-block table). Some callers
// cannot hand over scratch memory: hosts that own every byte of device memory
// through a fixed plan and pass the library only its inputs and outputs, and
// latency-critical loops that must never enter the allocator after start-up,
// because an allocation can synchronise the device. For them,
// trellis_moe_route_map_static keeps its scratch in one statically sized
// array in device memory that exists for as long as the library is loaded.
//
// Limits and sharing: at most kStaticMaxRoutes routes (T * topk) and
// tmoe::kMaxExperts experts per call. Every call on a device uses the same
// array, so two calls whose kernels overlap on the GPU (different streams
// without ordering between them) race and corrupt each other's result; order
// them on one stream. The array keeps the previous call's contents; the parts
// that must start from zero (the error word) are cleared by every call. The
// array's device address is looked up once per device and kept for the life
// of the process, so a device reset (cudaDeviceReset) while the library is
// loaded is not supported: the kept address would be stale afterwards.
#include <mutex>

#include "../../include/trellis_moe.h"
#include "launch.h"

namespace {

constexpr int kStaticMaxRoutes = 1024;   // T * topk per call
constexpr int kMaxDevices = 64;
// int32 words: [0] error flags, [1] route-block count, [8..) ranks,
// then per-expert tile counts, then the route-block -> expert table
// (at most R + E entries for any block size).
constexpr int kOffErr = 0;
constexpr int kOffNBlocks = 1;
constexpr int kOffRank = 8;
constexpr int kOffTileCounts = kOffRank + kStaticMaxRoutes;
constexpr int kOffBlockExpert = kOffTileCounts + tmoe::kMaxExperts;
constexpr int kStaticWords = kOffBlockExpert + kStaticMaxRoutes + tmoe::kMaxExperts + 1;

static __device__ __align__(256) int32_t g_route_scratch[kStaticWords];

std::mutex g_setup_mu;
int32_t* g_scratch_ptr[kMaxDevices] = {};

tm_status static_fail(tm_status s, const char* msg) {
  tmoe::set_last_error(msg);
  return s;
}

}  // namespace

extern "C" {

tm_status trellis_moe_route_map_static(const int32_t* topk_ids, int32_t T, int32_t E, int32_t topk, int32_t block,
                                       int32_t* counts, int32_t* offsets, int32_t* route_of_slot,
                                       int32_t* slot_of_route, void* stream) {
  tmoe::set_last_error("");
  if (T < 0) return static_fail(TM_EINVAL, "T must be >= 0");
  if (E < 1 || E > tmoe::kMaxExperts) return static_fail(TM_EUNSUPPORTED, "E must be in 1..256");
  if (topk < 1 || topk > 32 || topk > E) return static_fail(TM_EINVAL, "topk must be in 1..min(E, 32)");
  if (block < 1 || block > 256) return static_fail(TM_EINVAL, "block must be in 1..256");
  if ((long)T * topk > kStaticMaxRoutes)
    return static_fail(TM_EUNSUPPORTED,
                       "T*topk exceeds the 1024 routes the static scratch holds; "
                       "use trellis_moe_route_map with a workspace");
  if (T == 0) return TM_OK;
  if (!topk_ids || !counts || !offsets || !route_of_slot || !slot_of_route)
    return static_fail(TM_EINVAL, "route map arguments must be non-NULL");

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return static_fail(TM_ECUDA, "cudaGetDevice failed or device index too large");
  int32_t* scratch = nullptr;
  {
    // Once per device, with that device current: the device address of the
    // static array (its host-side name is not a device address).
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_scratch_ptr[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || p == nullptr)
        return static_fail(TM_ECUDA, "cudaGetSymbolAddress of the static route-map scratch failed");
      g_scratch_ptr[dev] = static_cast<int32_t*>(p);
    }
    scratch = g_scratch_ptr[dev];
  }
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemsetAsync(scratch + kOffErr, 0, sizeof(int32_t), st) != cudaSuccess)
    return static_fail(TM_ECUDA, "clearing the error word failed");

  tmoe::RouteMapArgs rm;
  rm.ids = topk_ids;
  rm.R = T * topk;
  rm.E = E;
  rm.block = block;
  rm.rank = scratch + kOffRank;
  rm.tile_counts = scratch + kOffTileCounts;
  rm.counts = counts;
  rm.offsets = offsets;
  rm.block_expert = scratch + kOffBlockExpert;
  rm.nblocks = scratch + kOffNBlocks;
  rm.route_of_slot = route_of_slot;
  rm.slot_of_route = slot_of_route;
  rm.err = reinterpret_cast<uint32_t*>(scratch + kOffErr);
  if (tmoe::launch_route_map(rm, st) != cudaSuccess) return static_fail(TM_ECUDA, "route map launch failed");
  return TM_OK;
}

}  // extern "C"
