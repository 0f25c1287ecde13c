// Internal kernel launchers of the trellis-MoE library.
#pragma once

#include <cuda.h>
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
  int raw_rows;               // FC2 (tensor-core kernel, not atomic): rows leave the last Hadamard level and down_svh to the combine
  // TrellisMX-style weights: UE8M0 bytes of this projection, [E][wrows][wcols]
  // (one per 32 weights of a row along the contraction axis), or NULL
  const uint8_t* wscale;
  int wrows, wcols;
};

// Separate gate / up input signs (one row shared by the experts, or one row
// per expert: b12x PR #129 "feat(moe): serve canonical Fruit QSRT atoms",
// review of trellis_w4a8.py, gate_suh and up_suh of shape (1, H) or
// (num_experts, H)). The FC1 gate rows then see x~_g = H_b(gate_suh_e * x) and
// the up rows x~_u = H_b(up_suh_e * x), one pair per route.
struct RouteRotArgs {
  const uint16_t* x;             // bf16 [T, H]
  const uint16_t* gsuh;          // fp16 [sign_rows, H]
  const uint16_t* usuh;          // fp16 [sign_rows, H]
  int sign_rows;                 // 1 or E
  const int32_t* ids;            // [T * topk] expert ids, or nullptr: select them from `logits`
  const float* logits;           // [T, E] (when ids == nullptr)
  const int32_t* slot_of_route;  // row of route r = its slot (tensor-core path), or nullptr: row r (decode rows)
  int T, H, E, topk, rot_b;
  uint16_t* out_g;               // x~_g rows [.][H]: fp16 (W4A16) or E4M3 codes as fp16 (W4A8)
  uint16_t* out_u;
  uint16_t* scaled_g;            // W4A8: code * 2^e rows
  uint16_t* scaled_u;
  uint8_t* xs_g;                 // W4A8: E8M0 [.][H/32]
  uint8_t* xs_u;
};

// Decode-rows path (few tokens): one fused prologue, then FC1 and FC2 as
// persistent warp-granular kernels over items of 16 weight rows x 256
// contraction columns of one route block of 8 slots, each followed by an
// epilogue kernel (one warp per epilogue unit and slot) that sums the unit's
// partial sums in fixed order.
struct DecPrologueArgs {
  const float* logits;      // router logits [T, E], or nullptr when ids are given
  int32_t* ids_out;         // router outputs (when logits != nullptr)
  float* w_out;
  RouteMapArgs rm;          // rm.ids = given ids or ids_out
  const uint16_t* x;        // bf16 [T, H]
  const uint16_t* suh;      // fp16 [H]
  int T, H, topk, rot_b, w4a8;
  void* xq;                 // fp16 [T, H] (W4A8: the E4M3 codes, as fp16)
  uint16_t* xq_scaled;      // W4A8: fp16 [T, H] code * 2^e (exact where e in [-15, 7])
  uint8_t* xs;              // E8M0 [T, H/32]
  int32_t* zero_i32;        // counters to clear
  int n_zero_i32;
  float* out;               // [T, H], cleared here (tokens without a valid route stay 0)
  long out_n;
  // per route block b < max_blocks, written after the route map: expert |
  // bits << 16 | valid slots << 24 (0 past the last block), and the byte
  // offsets of the expert's FC1 and FC2 payload
  const int64_t* word_off1;
  const int64_t* word_off2;
  const uint8_t* bits;
  int max_blocks;
  int32_t* blk_meta;
  long long* blk_off1;
  long long* blk_off2;
  int split_signs;          // separate gate / up input signs: rotate per route with `rr` (rows = routes)
  RouteRotArgs rr;
  int rot_per;              // rotation warps per rotation CTA (set by launch_dec_prologue)
};

constexpr int kDecSeg = 256;  // contraction columns of one decode-rows item
constexpr int kDecBlock = 8;  // slots per route block
// Routes from which the K=4 decode kernels take items of 2 * kDecSeg columns:
// fewer, longer items halve the per-item bookkeeping once each warp holds
// several of them, and cost time when most warps hold at most one.
constexpr int kDecWideRoutes = 48;

struct DecArgs {
  FcArgs f;                 // act: fp16 rows (W4A8: E4M3 codes as fp16, E8M0 scales in act_scale)
  const uint16_t* act_scaled;  // W4A8: the same rows as code * 2^e (used where every e is in [-15, 7])
  uint16_t* out_act_scaled;    // FC1 W4A8: z~ as code * 2^e
  const int32_t* blk_meta;  // per route block: expert | bits << 16 | valid slots << 24
  const long long* blk_off; // per route block: byte offset of the expert's payload (this projection)
  int nseg;                 // contraction segments of kDecSeg * segs columns (one item each)
  int segs;                 // kDecSeg-column pieces per item: 1, or 2 (K=4 layers, >= kDecWideRoutes routes)
  int units_m;              // epilogue units per route block (FC1: I/BI, FC2: H/128)
  int bi;                   // FC1 half-row block (64 or 128)
  int max_blocks;           // route blocks the route map can produce
  int fc_warps;             // warps of the FC kernel's grid (dec_fc_warps)
  float* partial;           // [blocks][nseg][rows/16][8 slots][16 rows] fp32 partial sums
  const int32_t* ids;       // [T*topk] expert ids (FC2 epilogue)
  const int32_t* slot_of_route;
  const float* route_w;     // [T*topk]
  float* out;               // FC2: final output [T, H]
  int T;
  const uint16_t* lut;      // codebook table of the mode (65,536 fp16), or NULL: expand by the hash
  // FC1 with separate gate / up input signs: activation rows are routes (not
  // tokens); the gate strips read f.act / act_scaled / f.act_scale, the up
  // strips these
  int split;
  const void* act2;
  const uint16_t* act_scaled2;
  const uint8_t* act_scale2;
};

cudaError_t launch_dec_prologue(const DecPrologueArgs& a, cudaStream_t st);
// Warps of the decode-rows FC kernel's grid (all resident: CTAs per SM x SMs);
// fixed on the first call, which also sets the kernel's attributes.
cudaError_t dec_fc_warps(int proj, bool w4a8, int uniform_k, bool lut, bool mx, int segs, int* warps);
// Codebook tables for the lookup variant: decode_lut_bytes() bytes, built on `st`.
size_t decode_lut_bytes();
cudaError_t build_decode_lut(uint16_t* lut, cudaStream_t st);
cudaError_t launch_dec_fc(const DecArgs& d, int proj, bool w4a8, int uniform_k, cudaStream_t st);
cudaError_t launch_dec_epilogue(const DecArgs& d, int proj, bool w4a8, cudaStream_t st);

// FC1 / FC2 on tcgen05 outside the decode regime (W4A16): x~ [slots][H] and
// z~ [slots][I] fp16 in slot order, route blocks of tc_route_block() slots.
struct TcArgs {
  FcArgs f;
  int bi;          // FC1 half-row block (64 or 128)
  uint32_t* err;   // device error word (bit 1: a pipeline wait gave up)
  uint32_t* sched; // device unit counter, zero before the launch
  int act_rows;    // rows of the activation operand, in slot order: slots
  uint64_t wait_ns;  // limit of every pipeline wait in ns (0: the default, 2 s)
  int stall_issuer;  // test of the bounded waits: the MMA issuer first waits on a barrier nothing arrives on
  int route_block;   // slots per route block: 256, or 128 with split activations
  const void* act2;  // FC1 with separate gate / up input signs: the up rows' operand (f.act: the gate rows'), else NULL
  // FC1 and FC2 in one launch (proj 3): f holds FC1's arguments, f2 FC2's;
  // dep[rb] counts the FC1 epilogue warps that have stored their z~ rows of
  // route block rb (zero before the launch, one entry per route block)
  FcArgs f2;
  uint32_t* dep;
  CUtensorMap amap2; // filled by launch_tc_fc from act2
  CUtensorMap amap;  // filled by launch_tc_fc: the activations as [act_rows][K] fp16, box 64 x 128, 128-byte swizzle
  CUtensorMap amapz; // proj 3: filled by launch_tc_fc from f2.act (z~ [act_rows][I])
};
// proj 1 (FC1), 2 (FC2) or 3 (both in one launch: every FC1 unit is queued
// before every FC2 unit, and an FC2 unit waits until its route block's z~
// rows are complete); 3 needs N = 256 for both (bi = 128, H % 256 == 0) and
// no split operands (tc_fused_supported).
cudaError_t launch_tc_fc(const TcArgs& args, int proj, int uniform_k, int max_blocks, cudaStream_t st);
bool tc_fused_supported(int H, int bi, bool split);
// The variants of each projection (tc_fc1.cu, tc_fc2.cu, tc_fused.cu), called
// by launch_tc_fc once the tensor maps are in args.
cudaError_t launch_tc_fc1(const TcArgs& args, int uniform_k, int max_blocks, cudaStream_t st);
cudaError_t launch_tc_fc2(const TcArgs& args, int uniform_k, int max_blocks, cudaStream_t st);
cudaError_t launch_tc_fused(const TcArgs& args, int uniform_k, int max_blocks, cudaStream_t st);
int tc_route_block();
// Geometry the tcgen05 kernels handle (H, I, FC1 half-row block, rotation blocks).
bool tc_supported(int H, int I, int bi, int rot_h, int rot_i);

cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w, cudaStream_t st);
cudaError_t launch_route_map(const RouteMapArgs& a, cudaStream_t st);
int route_map_tiles(int R);

cudaError_t launch_rotate_quant(const uint16_t* x, const uint16_t* suh, int T, int H, int rot_b, bool w4a8,
                                void* xq, uint8_t* xs, cudaStream_t st, const int32_t* slot_of_route = nullptr,
                                int topk = 0);
// Separate gate / up input signs: both rotations per route (rotate_routes_warp).
cudaError_t launch_rotate_routes(const RouteRotArgs& a, bool w4a8, cudaStream_t st);

struct CombineUnrotArgs {
  const float* rows;            // [slots, H]: per 128-column block, (I_2 x H_64)(scale * FC2 accumulator)
  const int32_t* slot_of_route; // [T*k]
  const int32_t* block_expert;  // expert of each block of bn slots
  int bn;
  const float* w;               // route weights [T*k]
  const uint16_t* svh;          // fp16 down_svh [E, H]
  int rot_b, T, H, k;
  float* out;                   // [T, H]
};
cudaError_t launch_combine_unrot(const CombineUnrotArgs& a, cudaStream_t st);
cudaError_t launch_combine(const float* rows, const int32_t* slot_of_route, const float* w, int T, int H, int k,
                           float* out, cudaStream_t st);

// Sets the calling thread's message returned by trellis_moe_last_error().
void set_last_error(const char* msg);

cudaError_t launch_decode_tiles(const int16_t* tiles, int K, int ntiles, bool e4m3, void* dst, cudaStream_t st);

}  // namespace tmoe
