// Internal kernel launchers of the trellis-MoE library.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

namespace tmoe {

constexpr int kMaxExperts = 256;

struct RouteMapArgs {
  const int32_t* ids;
  int R, E, block;
  int32_t* rank;          // [R]
  int32_t* tile_counts;   // [ntiles][E]
  int32_t* counts;        // [E]
  int32_t* offsets;       // [E+1]
  int32_t* block_expert;  // [max route blocks]
  int32_t* nblocks;       // [1]
  int32_t* route_of_slot; // [R + E*(block-1)]
  int32_t* slot_of_route; // [R]
  uint32_t* err;          // [1]
};

struct FcArgs {
  int E, H, I, topk;
  int rot_b;                  // Hadamard block along this projection's output channels
  const int16_t* payload;     // this projection's payload words
  const int64_t* word_off;    // [E] word offset of each expert's block
  const uint8_t* bits;        // [E]
  const uint16_t* scale;      // fp16 [E, rows]
  const uint16_t* rot_tab;    // FC1: [E, 3I]; FC2: out_svh [E, H]
  const void* act;            // FC1: x~ [T, H]; FC2: z~ [slots, I]
  const uint8_t* act_scale;   // W4A8: E8M0 [rows, K/32]
  const int32_t* route_of_slot;
  const int32_t* block_expert;
  const int32_t* nblocks;
  void* out_act;              // FC1: z~ [slots, I]
  uint8_t* out_scale;         // FC1 W4A8: E8M0 [slots, I/32]
  float* out_f32;             // FC2: per-slot rows [slots, H], or out [T, H] when atomic
  const float* route_w;       // FC2 atomic: route weights [T*topk]
  int atomic;
};

cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w, cudaStream_t st);
cudaError_t launch_route_map(const RouteMapArgs& a, cudaStream_t st);
int route_map_tiles(int R);

cudaError_t launch_rotate_quant(const uint16_t* x, const uint16_t* suh, int T, int H, int rot_b, bool w4a8,
                                void* xq, uint8_t* xs, cudaStream_t st);

// FC kernels. `bn` is the route block (8 or 64), `bi` the FC1 half-row block
// (64 or 128), `uniform_k` the trellis K of every expert or 0 when mixed.
cudaError_t launch_fc1(const FcArgs& a, bool w4a8, int bi, int bn, int uniform_k, int max_blocks, cudaStream_t st);
cudaError_t launch_fc2(const FcArgs& a, bool w4a8, int bn, int uniform_k, int max_blocks, cudaStream_t st);

cudaError_t launch_combine(const float* rows, const int32_t* slot_of_route, const float* w, int T, int H, int k,
                           float* out, cudaStream_t st);

// Sets the calling thread's message returned by trellis_moe_last_error().
void set_last_error(const char* msg);

cudaError_t launch_decode_tiles(const int16_t* tiles, int K, int ntiles, bool e4m3, void* dst, cudaStream_t st);

}  // namespace tmoe
