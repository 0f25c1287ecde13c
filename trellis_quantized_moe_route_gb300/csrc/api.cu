// C ABI of the trellis-MoE layer: host-side validation, workspace layout and
// the launch sequence of one forward pass. Declared in include/trellis_moe.h.
//
// Lifecycle after the pages' own (sparkinfer PR #90 "moe: integrate EXL3
// Trellis into the fused W4A16 API", Summary: plan -> prepare -> scratch/bind
// -> run; flashinfer PR #69 "b12x fused MoE: TrellisMX ...", Description: the
// plan declares the scratch bytes, bind carves them, no call allocates, and a
// missing, short or misaligned arena is rejected).
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "../../include/trellis_moe.h"
#include "launch.h"

struct tm_layer {
  tm_layer_desc desc;
  std::vector<uint8_t> bits;
  int uniform_k;       // trellis K of every expert, or 0 when mixed
  int bi;              // FC1 half-row block (64 or 128)
  int64_t* d_off1;     // [E] word offsets of each expert's FC1 block
  int64_t* d_off2;     // [E]
  uint8_t* d_bits;     // [E]
  uint16_t* d_lut;     // codebook tables for the decode-rows lookup variant (fp16 | E4M3 as fp16)
  int use_lut;         // decode rows expand by table lookup (1) or by the hash (0)
  int device;
  uint64_t wait_ns;    // limit of the tensor-core kernels' pipeline waits (0: their default)
  int stall_issuer;    // test of the bounded waits (trellis_moe_set_wait_test)
  cudaEvent_t stage_ev[7];  // optional stage-boundary events (NULL = off)
  // Host-buffer calls on mapped page-locked buffers replay a captured graph of
  // the layer once the same buffers come back; one entry per buffer set, least
  // recently used evicted. exec == NULL: seen once, not captured yet (or the
  // capture failed).
  struct HostGraph {
    const void* x;
    const void* logits;
    void* out;
    void* ws;
    int T;
    int mode;
    bool failed;
    uint64_t used;
    cudaGraphExec_t exec;
  };
  std::mutex graph_mu;
  std::vector<HostGraph> graphs;
  uint64_t graph_clock = 0;
  cudaStream_t capture_stream = nullptr;  // private stream the graphs are captured on
};

namespace {

thread_local char g_err[512] = "";

tm_status fail(tm_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}

tm_status cuda_fail(cudaError_t e, const char* what) {
  return fail(TM_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Records stage-boundary event i if the caller asked for it: inside a stream
// capture as an external event node (so that replays record it), else as a
// plain record (the external flag is invalid outside a capture).
cudaError_t stage_mark(const tm_layer* layer, int i, cudaStream_t st) {
  if (!layer->stage_ev[i]) return cudaSuccess;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  const cudaError_t e = cudaStreamIsCapturing(st, &cs);
  if (e != cudaSuccess) return e;
  return cs == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags(layer->stage_ev[i], st, cudaEventRecordExternal)
                                             : cudaEventRecord(layer->stage_ev[i], st);
}

// Frees the captured host-call graphs. Caller holds graph_mu.
void drop_host_graphs(tm_layer* layer) {
  for (auto& g : layer->graphs)
    if (g.exec) cudaGraphExecDestroy(g.exec);
  layer->graphs.clear();
}

constexpr size_t kAlign = 256;
constexpr int kBlockMax = 256;  // largest route block (tcgen05 path): expert segments pad to it

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

// FC1 half-row block: the epilogue needs whole rotation blocks of I.
int fc1_bi(const tm_layer_desc& d) {
  int bi = (d.rot_block_i == 128 || (d.I % 128 == 0 && d.rot_block_i != 64)) ? 128 : 64;
  if (d.I % bi != 0) bi = 64;
  return bi;
}

// Decode-rows path plan (route blocks of 8). W4A8 always runs here (the pages
// select W4A8 only for bounded decode rows; T*topk <= 1024); W4A16 does when
// T*topk <= 1024 and experts see fewer than 4 routes on average.
struct DecPlan {
  bool use;
  int max_blocks, bi, units1, units2, nseg1, nseg2;
  size_t partial_floats, cnt_ints;
};

constexpr long kDecMaxRoutes = 1024;

DecPlan dec_plan(const tm_layer_desc& d, int T, bool w4a8) {
  DecPlan p{};
  const long R = (long)T * d.topk;
  p.use = R >= 1 && R <= kDecMaxRoutes && (w4a8 || R < 4L * d.E);
  p.bi = fc1_bi(d);
  p.units1 = d.I / p.bi;
  p.units2 = d.H / (d.rot_block_h > 128 ? 512 : 128);  // FC2 epilogue: one CTA per token x rotation span
  p.max_blocks = (int)(R / tmoe::kDecBlock + std::min<long>(d.E, R) + 1);
  p.nseg1 = (d.H + tmoe::kDecSeg - 1) / tmoe::kDecSeg;
  p.nseg2 = (d.I + tmoe::kDecSeg - 1) / tmoe::kDecSeg;
  // per (block, segment, 16-row strip): 8 x 16 partial sums
  p.partial_floats = (size_t)p.max_blocks * std::max<size_t>((size_t)p.nseg1 * (2 * d.I / 16), (size_t)p.nseg2 * (d.H / 16)) * 128;
  p.cnt_ints = 0;  // (no counters: every reduction runs in a kernel of its own)
  if (!p.use) p.partial_floats = p.cnt_ints = 0;
  return p;
}

// The precision a call runs in: W4A8 when asked for, or in AUTO mode for
// T <= decode_max_rows, and only on bounded decode rows (check_rows rejects an
// explicit W4A8 call beyond them).
bool uses_w4a8(const tm_layer_desc& d, int T, int mode) {
  const long R = (long)T * d.topk;
  return mode == TM_MODE_W4A8 || (mode == TM_MODE_AUTO && T <= d.decode_max_rows && R <= kDecMaxRoutes);
}

tm_status check_rows(const tm_layer_desc& d, int T, int mode) {
  const long R = (long)T * d.topk;
  if (mode == TM_MODE_W4A8 && R > kDecMaxRoutes)
    return fail(TM_EUNSUPPORTED, "W4A8 runs on bounded decode rows: T*topk=%ld exceeds %ld", R, kDecMaxRoutes);
  return TM_OK;
}

// Regions of a workspace sized for T tokens (T*topk routes).
struct Layout {
  enum {
    ERR, XQ, XS, ZQ, ZS, ROWS, SLOT_OF_ROUTE, XQ2, XS2,
    IDS, W, RANK, TILE_COUNTS, COUNTS, OFFSETS, BLOCK_EXPERT, NBLOCKS, ROUTE_OF_SLOT,
    HOST_X, HOST_LOGITS, HOST_OUT, DEC_PARTIAL, DEC_CNT, DEC_META, COUNT
  };
  size_t off[COUNT];
  size_t bytes[COUNT];
  size_t total;
};

Layout make_layout(const tm_layer_desc& d, int T) {
  Layout L;
  const size_t R = (size_t)T * d.topk;
  const size_t slots = R + (size_t)d.E * (kBlockMax - 1);
  const size_t ntiles = (R + 1023) / 1024;
  // The decode path's scratch is not monotonic in T (larger T switches to the
  // general path), so size it for the worst T' <= T: a workspace that fits T
  // then fits every smaller call too. Its x~ region holds the codes and the
  // pre-multiplied copy (2T rows), its z~ region both for every route-block
  // slot (2 * 8 * max_blocks rows).
  size_t dec_partial = 0, dec_cnt = 0, dec_blocks = 0, dec_x_rows = 0, dec_z_rows = 0;
  for (int t = 1; t <= T && (long)t * d.topk <= kDecMaxRoutes; ++t) {
    const DecPlan dp = dec_plan(d, t, true);
    dec_partial = std::max(dec_partial, dp.partial_floats);
    dec_cnt = std::max(dec_cnt, dp.cnt_ints);
    dec_blocks = std::max(dec_blocks, (size_t)dp.max_blocks);
    dec_x_rows = std::max(dec_x_rows, (size_t)2 * t);
    dec_z_rows = std::max(dec_z_rows, (size_t)2 * tmoe::kDecBlock * dp.max_blocks);
  }
  // With separate gate / up input signs the decode rows keep x~ per route (R
  // rows of codes + R pre-multiplied rows), the up operand in XQ2 / XS2.
  const bool split = d.gate_suh != nullptr;
  if (split) dec_x_rows = std::max(dec_x_rows, 2 * std::min<size_t>(R, kDecMaxRoutes));
  L.bytes[Layout::XQ] = std::max(slots, dec_x_rows) * d.H * 2;  // fp16 in slot order (tcgen05 path), else [T][H]
  L.bytes[Layout::XS] = (split ? std::max<size_t>(T, R) : (size_t)T) * (d.H / 32);
  L.bytes[Layout::XQ2] = split ? L.bytes[Layout::XQ] : 0;
  L.bytes[Layout::XS2] = split ? L.bytes[Layout::XS] : 0;
  L.bytes[Layout::ZQ] = std::max(slots, dec_z_rows) * d.I * 2;
  L.bytes[Layout::ZS] = std::max(slots, dec_z_rows / 2) * (d.I / 32);
  L.bytes[Layout::ROWS] = slots * d.H * 4;
  L.bytes[Layout::SLOT_OF_ROUTE] = R * 4;
  // error word, the tcgen05 kernels' unit counters, then one z~ completion
  // counter per route block of the fused FC1 + FC2 launch
  L.bytes[Layout::ERR] = 16 + (R / 128 + (size_t)d.E + 2) * 4;
  L.bytes[Layout::IDS] = R * 4;
  L.bytes[Layout::W] = R * 4;
  L.bytes[Layout::RANK] = R * 4;
  L.bytes[Layout::TILE_COUNTS] = ntiles * d.E * 4;
  L.bytes[Layout::COUNTS] = (size_t)d.E * 4;
  L.bytes[Layout::OFFSETS] = ((size_t)d.E + 1) * 4;
  L.bytes[Layout::BLOCK_EXPERT] = (slots / tmoe::kDecBlock + 1) * 4;
  L.bytes[Layout::NBLOCKS] = 4;
  L.bytes[Layout::ROUTE_OF_SLOT] = slots * 4;
  L.bytes[Layout::HOST_X] = (size_t)T * d.H * 2;
  L.bytes[Layout::HOST_LOGITS] = (size_t)T * d.E * 4;
  L.bytes[Layout::HOST_OUT] = (size_t)T * d.H * 4;
  L.bytes[Layout::DEC_PARTIAL] = dec_partial * 4;
  L.bytes[Layout::DEC_CNT] = dec_cnt * 4;
  L.bytes[Layout::DEC_META] = dec_blocks * (8 + 8 + 8);  // int64 FC1 and FC2 offsets, then int32 metadata
  size_t o = 0;
  for (int i = 0; i < Layout::COUNT; ++i) {
    L.off[i] = o;
    o += align_up(std::max<size_t>(L.bytes[i], 1));
  }
  L.total = o;
  return L;
}

template <typename P>
P* at(void* ws, const Layout& L, int region) {
  return reinterpret_cast<P*>(reinterpret_cast<char*>(ws) + L.off[region]);
}

bool pow2_block_ok(int b) { return b == 1 || b == 64 || b == 128; }
// Hidden-side blocks may also be 512 wide (the coupled H512 boundary of
// TrellisMX-style layers).
bool h_block_ok(int b, int H) { return pow2_block_ok(b) || (b == 512 && H % 512 == 0); }

tm_status check_ws(const tm_layer* layer, int T, void* ws, size_t bytes, Layout* out) {
  if (T > layer->desc.max_tokens) return fail(TM_EINVAL, "T=%d exceeds prepared max_tokens=%d", T, layer->desc.max_tokens);
  const Layout L = make_layout(layer->desc, T);
  if (ws == nullptr) return fail(TM_EWORKSPACE, "workspace is NULL");
  if (((uintptr_t)ws) % kAlign != 0) return fail(TM_EWORKSPACE, "workspace must be %zu-byte aligned", kAlign);
  if (bytes < L.total) return fail(TM_EWORKSPACE, "workspace has %zu bytes, %zu needed for T=%d", bytes, L.total, T);
  *out = L;
  return TM_OK;
}

tm_status run_decode_path(tm_layer* layer, const uint16_t* x, const int32_t* ids, const float* w,
                          const float* logits, int T, bool w4a8, float* out, void* ws, const Layout& L,
                          const DecPlan& dp, cudaStream_t st);

// One forward pass. With `logits` non-NULL the router runs first (fused into
// the decode-path prologue) and writes ids and w into the workspace.
tm_status run_layer(tm_layer* layer, const uint16_t* x, const int32_t* ids, const float* w, const float* logits,
                    int T, int mode, float* out, void* ws, const Layout& L, cudaStream_t st) {
  const tm_layer_desc& d = layer->desc;
  const bool w4a8 = uses_w4a8(d, T, mode);
  const int R = T * d.topk;
  // Outside the decode regime FC1 and FC2 run on the tcgen05 kernels (W4A16,
  // route blocks of up to 256 routes).
  const bool split = d.gate_suh != nullptr;  // separate gate / up input signs
  // Route blocks of 128 routes give every unit one tensor-memory accumulator,
  // so a unit's epilogue overlaps the next unit's contraction; blocks of 256
  // expand each weight once for up to 256 routes. Measured on one GB300:
  // with 128 routes per expert on average (Zipf prefill) the 128-route blocks
  // win (step 236 -> 221 us), with 205 (the large layer) the 256-route ones
  // (FC1 1.14 vs 1.96 ms).
  const int bn = (split || R <= 128L * d.E) ? 128 : tmoe::tc_route_block();
  cudaError_t e;
  uint32_t* err = at<uint32_t>(ws, L, Layout::ERR);
  if (logits) {
    ids = at<int32_t>(ws, L, Layout::IDS);
    w = at<float>(ws, L, Layout::W);
  }
  const DecPlan dp = dec_plan(d, T, w4a8);
  // (the decode prologue clears the error word itself)
  if (dp.use) return run_decode_path(layer, x, ids, w, logits, T, w4a8, out, ws, L, dp, st);
  if ((e = cudaMemsetAsync(err, 0, L.bytes[Layout::ERR], st)) != cudaSuccess) return cuda_fail(e, "clear error word");
  if (logits) {
    e = tmoe::launch_route_topk(logits, T, d.E, d.topk, const_cast<int32_t*>(ids), const_cast<float*>(w), st);
    if (e != cudaSuccess) return cuda_fail(e, "router");
    if ((e = stage_mark(layer, 1, st)) != cudaSuccess) return cuda_fail(e, "stage event");
  }

  tmoe::RouteMapArgs rm;
  rm.ids = ids;
  rm.R = R;
  rm.E = d.E;
  rm.block = bn;
  rm.rank = at<int32_t>(ws, L, Layout::RANK);
  rm.tile_counts = at<int32_t>(ws, L, Layout::TILE_COUNTS);
  rm.counts = at<int32_t>(ws, L, Layout::COUNTS);
  rm.offsets = at<int32_t>(ws, L, Layout::OFFSETS);
  rm.block_expert = at<int32_t>(ws, L, Layout::BLOCK_EXPERT);
  rm.nblocks = at<int32_t>(ws, L, Layout::NBLOCKS);
  rm.route_of_slot = at<int32_t>(ws, L, Layout::ROUTE_OF_SLOT);
  rm.slot_of_route = at<int32_t>(ws, L, Layout::SLOT_OF_ROUTE);
  rm.err = err;
  if ((e = tmoe::launch_route_map(rm, st)) != cudaSuccess) return cuda_fail(e, "route map");
  if ((e = stage_mark(layer, 2, st)) != cudaSuccess) return cuda_fail(e, "stage event");

  void* xq = at<void>(ws, L, Layout::XQ);
  uint8_t* xs = at<uint8_t>(ws, L, Layout::XS);
  // the tcgen05 path reads x~ in slot order (one copy per route)
  if (split) {
    tmoe::RouteRotArgs rr{};
    rr.x = x;
    rr.gsuh = d.gate_suh;
    rr.usuh = d.up_suh;
    rr.sign_rows = d.input_sign_rows;
    rr.ids = ids;
    rr.slot_of_route = rm.slot_of_route;
    rr.T = T;
    rr.H = d.H;
    rr.E = d.E;
    rr.topk = d.topk;
    rr.rot_b = d.rot_block_h;
    rr.out_g = static_cast<uint16_t*>(xq);
    rr.out_u = at<uint16_t>(ws, L, Layout::XQ2);
    e = tmoe::launch_rotate_routes(rr, false, st);
  } else {
    e = tmoe::launch_rotate_quant(x, d.in_suh, T, d.H, d.rot_block_h, false, xq, xs, st, rm.slot_of_route, d.topk);
  }
  if (e != cudaSuccess) return cuda_fail(e, "rotate+quantize");
  if ((e = stage_mark(layer, 3, st)) != cudaSuccess) return cuda_fail(e, "stage event");

  const int max_blocks = R / bn + std::min(d.E, R) + 1;
  tmoe::FcArgs a1{};
  a1.E = d.E; a1.H = d.H; a1.I = d.I; a1.topk = d.topk;
  a1.rot_b = d.rot_block_i;
  a1.payload = d.fc1_payload;
  a1.word_off = layer->d_off1;
  a1.bits = layer->d_bits;
  a1.scale = d.fc1_scale;
  a1.rot_tab = d.rot_tab;
  a1.act = xq;
  a1.act_scale = xs;
  a1.route_of_slot = rm.route_of_slot;
  a1.block_expert = rm.block_expert;
  a1.nblocks = rm.nblocks;
  a1.out_act = at<void>(ws, L, Layout::ZQ);
  a1.out_scale = at<uint8_t>(ws, L, Layout::ZS);
  a1.wscale = d.fc1_wscale;
  a1.wrows = 2 * d.I;
  a1.wcols = d.H / 32;
  tmoe::TcArgs t1{};
  t1.f = a1;
  t1.bi = layer->bi;
  t1.err = err;
  t1.sched = err + 1;
  t1.act_rows = (int)(R + (size_t)d.E * (kBlockMax - 1));  // slots
  t1.wait_ns = layer->wait_ns;
  t1.stall_issuer = layer->stall_issuer;
  t1.route_block = bn;
  t1.act2 = split ? at<void>(ws, L, Layout::XQ2) : nullptr;

  tmoe::FcArgs a2 = a1;
  a2.rot_b = d.rot_block_h;
  a2.payload = d.fc2_payload;
  a2.word_off = layer->d_off2;
  a2.scale = d.fc2_scale;
  a2.rot_tab = d.out_svh;
  a2.act = a1.out_act;
  a2.act_scale = a1.out_scale;
  a2.out_act = nullptr;
  a2.out_scale = nullptr;
  a2.route_w = w;
  a2.wscale = d.fc2_wscale;
  a2.wrows = d.H;
  a2.wcols = d.I / 32;
  // (512-point output rotations always take the ordered combine)
  a2.atomic = (d.deterministic || d.rot_block_h > 128) ? 0 : 1;
  // the tensor-core FC2 leaves the route's output scale, H and down_svh to the combine
  a2.raw_rows = (!a2.atomic && d.topk <= 32) ? 1 : 0;
  if (a2.atomic) {
    if ((e = cudaMemsetAsync(out, 0, (size_t)T * d.H * 4, st)) != cudaSuccess) return cuda_fail(e, "clear output");
    a2.out_f32 = out;
  } else {
    a2.out_f32 = at<float>(ws, L, Layout::ROWS);
  }
  // FC1 and FC2 in one launch where both take 256-row units: the FC2 units
  // fill the last wave of FC1 units instead of waiting for all of them
  if (tmoe::tc_fused_supported(d.H, layer->bi, split)) {
    t1.f2 = a2;
    t1.dep = err + 4;
    if ((e = tmoe::launch_tc_fc(t1, 3, layer->uniform_k, max_blocks, st)) != cudaSuccess)
      return cuda_fail(e, "FC1+FC2");
    if ((e = stage_mark(layer, 4, st)) != cudaSuccess) return cuda_fail(e, "stage event");
  } else {
    if ((e = tmoe::launch_tc_fc(t1, 1, layer->uniform_k, max_blocks, st)) != cudaSuccess) return cuda_fail(e, "FC1");
    if ((e = stage_mark(layer, 4, st)) != cudaSuccess) return cuda_fail(e, "stage event");
    tmoe::TcArgs t2 = t1;
    t2.f = a2;
    t2.sched = err + 2;
    t2.act2 = nullptr;
    if ((e = tmoe::launch_tc_fc(t2, 2, layer->uniform_k, max_blocks, st)) != cudaSuccess) return cuda_fail(e, "FC2");
  }
  if ((e = stage_mark(layer, 5, st)) != cudaSuccess) return cuda_fail(e, "stage event");
  if (a2.raw_rows) {
    tmoe::CombineUnrotArgs c{a2.out_f32, rm.slot_of_route, rm.block_expert, bn, w, d.out_svh,
                             d.rot_block_h, T, d.H, d.topk, out};
    if ((e = tmoe::launch_combine_unrot(c, st)) != cudaSuccess) return cuda_fail(e, "combine");
  } else if (!a2.atomic) {
    if ((e = tmoe::launch_combine(a2.out_f32, rm.slot_of_route, w, T, d.H, d.topk, out, st)) != cudaSuccess)
      return cuda_fail(e, "combine");
  }
  if ((e = stage_mark(layer, 6, st)) != cudaSuccess) return cuda_fail(e, "stage event");
  return TM_OK;
}

tm_status run_decode_path(tm_layer* layer, const uint16_t* x, const int32_t* ids, const float* w,
                          const float* logits, int T, bool w4a8, float* out, void* ws, const Layout& L,
                          const DecPlan& dp, cudaStream_t st) {
  const tm_layer_desc& d = layer->desc;
  const int R = T * d.topk;
  cudaError_t e;
  tmoe::DecPrologueArgs pa{};
  pa.logits = logits;
  pa.ids_out = const_cast<int32_t*>(ids);
  pa.w_out = const_cast<float*>(w);
  pa.rm.ids = ids;
  pa.rm.R = R;
  pa.rm.E = d.E;
  pa.rm.block = tmoe::kDecBlock;
  pa.rm.rank = at<int32_t>(ws, L, Layout::RANK);
  pa.rm.tile_counts = at<int32_t>(ws, L, Layout::TILE_COUNTS);
  pa.rm.counts = at<int32_t>(ws, L, Layout::COUNTS);
  pa.rm.offsets = at<int32_t>(ws, L, Layout::OFFSETS);
  pa.rm.block_expert = at<int32_t>(ws, L, Layout::BLOCK_EXPERT);
  pa.rm.nblocks = at<int32_t>(ws, L, Layout::NBLOCKS);
  pa.rm.route_of_slot = at<int32_t>(ws, L, Layout::ROUTE_OF_SLOT);
  pa.rm.slot_of_route = at<int32_t>(ws, L, Layout::SLOT_OF_ROUTE);
  pa.rm.err = at<uint32_t>(ws, L, Layout::ERR);
  pa.x = x;
  pa.suh = d.in_suh;
  pa.T = T;
  pa.H = d.H;
  pa.topk = d.topk;
  pa.rot_b = d.rot_block_h;
  pa.w4a8 = w4a8 ? 1 : 0;
  pa.xq = at<void>(ws, L, Layout::XQ);
  // W4A8: the pre-multiplied copy of x~ after the codes (make_layout sizes the region for 2T rows)
  pa.xq_scaled = at<uint16_t>(ws, L, Layout::XQ) + (size_t)T * d.H;
  pa.xs = at<uint8_t>(ws, L, Layout::XS);
  pa.zero_i32 = at<int32_t>(ws, L, Layout::DEC_CNT);
  pa.n_zero_i32 = (int)dp.cnt_ints;
  pa.out = out;
  pa.out_n = 0;  // (the FC2 epilogue writes every output row)
  pa.word_off1 = layer->d_off1;
  pa.word_off2 = layer->d_off2;
  pa.bits = layer->d_bits;
  pa.max_blocks = dp.max_blocks;
  pa.blk_off1 = at<long long>(ws, L, Layout::DEC_META);
  pa.blk_off2 = pa.blk_off1 + dp.max_blocks;
  pa.blk_meta = reinterpret_cast<int32_t*>(pa.blk_off2 + dp.max_blocks);
  // separate gate / up input signs: x~_g and x~_u per route (rows r = t*topk+j),
  // codes then the pre-multiplied copy (R rows each) in XQ and XQ2
  const bool split = d.gate_suh != nullptr;
  pa.split_signs = split ? 1 : 0;
  if (split) {
    tmoe::RouteRotArgs& rr = pa.rr;
    rr.x = x;
    rr.gsuh = d.gate_suh;
    rr.usuh = d.up_suh;
    rr.sign_rows = d.input_sign_rows;
    rr.ids = logits ? nullptr : ids;
    rr.logits = logits;
    rr.slot_of_route = nullptr;
    rr.T = T;
    rr.H = d.H;
    rr.E = d.E;
    rr.topk = d.topk;
    rr.rot_b = d.rot_block_h;
    rr.out_g = at<uint16_t>(ws, L, Layout::XQ);
    rr.out_u = at<uint16_t>(ws, L, Layout::XQ2);
    rr.scaled_g = rr.out_g + (size_t)R * d.H;
    rr.scaled_u = rr.out_u + (size_t)R * d.H;
    rr.xs_g = at<uint8_t>(ws, L, Layout::XS);
    rr.xs_u = at<uint8_t>(ws, L, Layout::XS2);
  }
  if ((e = tmoe::launch_dec_prologue(pa, st)) != cudaSuccess) return cuda_fail(e, "decode prologue");
  for (int i = 1; i <= 3; ++i)
    if ((e = stage_mark(layer, i, st)) != cudaSuccess) return cuda_fail(e, "stage event");

  tmoe::DecArgs d1{};
  tmoe::FcArgs& a1 = d1.f;
  a1.E = d.E; a1.H = d.H; a1.I = d.I; a1.topk = d.topk;
  a1.rot_b = d.rot_block_i;
  a1.payload = d.fc1_payload;
  a1.word_off = layer->d_off1;
  a1.bits = layer->d_bits;
  a1.scale = d.fc1_scale;
  a1.rot_tab = d.rot_tab;
  a1.act = pa.xq;
  a1.act_scale = pa.xs;
  a1.route_of_slot = pa.rm.route_of_slot;
  a1.block_expert = pa.rm.block_expert;
  a1.nblocks = pa.rm.nblocks;
  a1.out_act = at<void>(ws, L, Layout::ZQ);
  a1.out_scale = at<uint8_t>(ws, L, Layout::ZS);
  a1.route_w = w;
  a1.atomic = d.deterministic ? 0 : 1;
  d1.units_m = dp.units1;
  d1.bi = dp.bi;
  d1.partial = at<float>(ws, L, Layout::DEC_PARTIAL);
  d1.ids = pa.rm.ids;
  d1.act_scaled = split ? pa.rr.scaled_g : pa.xq_scaled;
  d1.split = split ? 1 : 0;
  d1.act2 = split ? pa.rr.out_u : nullptr;
  d1.act_scaled2 = split ? pa.rr.scaled_u : nullptr;
  d1.act_scale2 = split ? pa.rr.xs_u : nullptr;
  // z~ rows are slots < max_blocks * 8; the pre-multiplied copy follows them
  // (make_layout sizes the region for 2 * max_blocks * 8 rows)
  d1.out_act_scaled = at<uint16_t>(ws, L, Layout::ZQ) + (size_t)dp.max_blocks * tmoe::kDecBlock * d.I;
  d1.blk_meta = pa.blk_meta;
  d1.blk_off = pa.blk_off1;
  d1.slot_of_route = pa.rm.slot_of_route;
  d1.route_w = w;
  d1.out = out;
  d1.T = T;
  d1.max_blocks = dp.max_blocks;
  a1.wscale = d.fc1_wscale;
  a1.wrows = 2 * d.I;
  a1.wcols = d.H / 32;
  const bool mx = d.fc1_wscale != nullptr;  // (TrellisMX-style weights expand by the hash)
  d1.lut = (layer->use_lut && !mx) ? layer->d_lut + (w4a8 ? 65536 : 0) : nullptr;
  // Items of two kDecSeg-column pieces for K=4 layers once there are enough
  // routes (measured on one GB300: T=8 step 53.5 -> 52.2 us; at T=1 and 2,
  // where most warps hold at most one item, always-wide items took 22.4 ->
  // 28.5 and 27.4 -> 29.7 us, hence the route threshold). The hash and table
  // expansions take the same items, so that they sum in the same order. The
  // partial-sum region is sized for one-piece items, the larger count.
  d1.segs = (layer->uniform_k == 4 && !mx && T * d.topk >= tmoe::kDecWideRoutes) ? 2 : 1;
  const int seg = tmoe::kDecSeg * d1.segs;
  d1.nseg = (d.H + seg - 1) / seg;
  if ((e = tmoe::dec_fc_warps(1, w4a8, layer->uniform_k, d1.lut != nullptr, mx, d1.segs, &d1.fc_warps)) != cudaSuccess)
    return cuda_fail(e, "FC1 (decode rows) setup");
  if ((e = tmoe::launch_dec_fc(d1, 1, w4a8, layer->uniform_k, st)) != cudaSuccess)
    return cuda_fail(e, "FC1 (decode rows)");
  // (stage 4 marks the FC1 GEMM kernel; its epilogue kernel counts with FC2)
  if ((e = stage_mark(layer, 4, st)) != cudaSuccess) return cuda_fail(e, "stage event");
  if ((e = tmoe::launch_dec_epilogue(d1, 1, w4a8, st)) != cudaSuccess)
    return cuda_fail(e, "FC1 epilogue (decode rows)");

  tmoe::DecArgs d2 = d1;
  d2.split = 0;
  d2.act2 = nullptr;
  d2.act_scaled2 = nullptr;
  d2.act_scale2 = nullptr;
  tmoe::FcArgs& a2 = d2.f;
  a2.rot_b = d.rot_block_h;
  a2.payload = d.fc2_payload;
  a2.word_off = layer->d_off2;
  a2.scale = d.fc2_scale;
  a2.rot_tab = d.out_svh;
  a2.act = a1.out_act;
  a2.act_scale = a1.out_scale;
  a2.out_act = nullptr;
  a2.out_scale = nullptr;
  a2.out_f32 = at<float>(ws, L, Layout::ROWS);
  a2.wscale = d.fc2_wscale;
  a2.wrows = d.H;
  a2.wcols = d.I / 32;
  d2.nseg = (d.I + seg - 1) / seg;
  d2.act_scaled = d1.out_act_scaled;
  d2.units_m = dp.units2;
  d2.blk_off = pa.blk_off2;
  if ((e = tmoe::dec_fc_warps(2, w4a8, layer->uniform_k, d2.lut != nullptr, mx, d2.segs, &d2.fc_warps)) != cudaSuccess)
    return cuda_fail(e, "FC2 (decode rows) setup");
  if ((e = tmoe::launch_dec_fc(d2, 2, w4a8, layer->uniform_k, st)) != cudaSuccess)
    return cuda_fail(e, "FC2 (decode rows)");
  if ((e = tmoe::launch_dec_epilogue(d2, 2, w4a8, st)) != cudaSuccess)
    return cuda_fail(e, "FC2 epilogue (decode rows)");
  for (int i = 5; i <= 6; ++i)
    if ((e = stage_mark(layer, i, st)) != cudaSuccess) return cuda_fail(e, "stage event");
  return TM_OK;
}

}  // namespace

namespace tmoe {
void set_last_error(const char* msg) { snprintf(g_err, sizeof(g_err), "%s", msg); }

}  // namespace tmoe

extern "C" {

const char* trellis_moe_last_error(void) { return g_err; }

tm_status trellis_moe_prepare(const tm_layer_desc* desc, tm_layer** out, size_t* workspace_bytes) {
  g_err[0] = 0;
  if (out) *out = nullptr;
  if (!desc || !out) return fail(TM_EINVAL, "desc and out must be non-NULL");
  const tm_layer_desc& d = *desc;
  if (d.E < 1 || d.E > tmoe::kMaxExperts) return fail(TM_EUNSUPPORTED, "E=%d outside 1..%d", d.E, tmoe::kMaxExperts);
  if (d.H < 128 || d.H % 128 != 0) return fail(TM_EUNSUPPORTED, "H=%d must be a positive multiple of 128", d.H);
  if (d.I < 64 || d.I % 64 != 0) return fail(TM_EUNSUPPORTED, "I=%d must be a positive multiple of 64", d.I);
  if (d.topk < 1 || d.topk > 32 || d.topk > d.E) return fail(TM_EINVAL, "topk=%d outside 1..min(E,32)", d.topk);
  if (!h_block_ok(d.rot_block_h, d.H) || d.H % d.rot_block_h != 0)
    return fail(TM_EUNSUPPORTED, "rot_block_h=%d must be 1, 64, 128 or 512 and divide H", d.rot_block_h);
  if (!pow2_block_ok(d.rot_block_i) || d.I % d.rot_block_i != 0)
    return fail(TM_EUNSUPPORTED, "rot_block_i=%d must be 1, 64 or 128 and divide I", d.rot_block_i);
  if (d.max_tokens < 1) return fail(TM_EINVAL, "max_tokens=%d must be >= 1", d.max_tokens);
  if ((long)d.max_tokens * d.topk > (1L << 24)) return fail(TM_EUNSUPPORTED, "max_tokens*topk too large");
  if (!d.bits_per_expert) return fail(TM_EINVAL, "bits_per_expert is NULL");
  const bool split = d.gate_suh != nullptr || d.up_suh != nullptr;
  if (split) {
    if (!d.gate_suh || !d.up_suh) return fail(TM_EINVAL, "gate_suh and up_suh must be given together");
    if (d.input_sign_rows != 1 && d.input_sign_rows != d.E)
      return fail(TM_EINVAL, "input_sign_rows=%d must be 1 or E=%d", d.input_sign_rows, d.E);
  }
  // (with separate gate / up signs in_suh is not read and may be NULL)
  const void* ptrs[] = {d.fc1_payload, d.fc2_payload, d.fc1_scale, d.fc2_scale, split ? d.gate_suh : d.in_suh,
                        d.rot_tab, d.out_svh, split ? d.up_suh : d.rot_tab};
  const char* names[] = {"fc1_payload", "fc2_payload", "fc1_scale", "fc2_scale", split ? "gate_suh" : "in_suh",
                         "rot_tab", "out_svh", "up_suh"};
  for (int i = 0; i < 8; ++i) {
    if (!ptrs[i]) return fail(TM_EINVAL, "%s is NULL", names[i]);
    if (((uintptr_t)ptrs[i]) % 16 != 0) return fail(TM_EINVAL, "%s must be 16-byte aligned", names[i]);
  }
  if ((d.fc1_wscale != nullptr) != (d.fc2_wscale != nullptr))
    return fail(TM_EINVAL, "fc1_wscale and fc2_wscale must be given together");
  if (d.fc1_wscale && (((uintptr_t)d.fc1_wscale) % 16 || ((uintptr_t)d.fc2_wscale) % 16))
    return fail(TM_EINVAL, "fc1_wscale and fc2_wscale must be 16-byte aligned");
  if (d.fc1_wscale) {
    // every scale exponent within [-15, 13]: E4M3(cb) * 2^k is then an exact
    // fp16 value (|E4M3(cb)| <= 4), as the tensor-core path holds it
    const size_t n1 = (size_t)d.E * 2 * d.I * (d.H / 32), n2 = (size_t)d.E * d.H * (d.I / 32);
    std::vector<uint8_t> h(std::max(n1, n2));
    const uint8_t* src[2] = {d.fc1_wscale, d.fc2_wscale};
    const size_t cnt[2] = {n1, n2};
    for (int i = 0; i < 2; ++i) {
      cudaError_t e = cudaMemcpy(h.data(), src[i], cnt[i], cudaMemcpyDeviceToHost);
      if (e != cudaSuccess) return cuda_fail(e, "read weight scales");
      for (size_t j = 0; j < cnt[i]; ++j)
        if (h[j] < 127 - 15 || h[j] > 127 + 13)
          return fail(TM_EUNSUPPORTED, "fc%d_wscale[%zu] = %u: exponent %d outside [-15, 13]", i + 1, j, h[j],
                      (int)h[j] - 127);
    }
  }
  tm_layer* L = new tm_layer();
  L->desc = d;
  for (int i = 0; i < 7; ++i) L->stage_ev[i] = nullptr;
  L->bits.assign(d.bits_per_expert, d.bits_per_expert + d.E);
  L->uniform_k = L->bits[0];
  std::vector<int64_t> off1(d.E), off2(d.E);
  int64_t o1 = 0, o2 = 0;
  for (int e = 0; e < d.E; ++e) {
    const int k = L->bits[e];
    if (k < 2 || k > 6) {
      delete L;
      return fail(TM_EUNSUPPORTED, "expert %d has K=%d bits; supported 2..6", e, k);
    }
    if (k != L->uniform_k) L->uniform_k = 0;
    off1[e] = o1;
    off2[e] = o2;
    o1 += (int64_t)(2 * d.I / 16) * (d.H / 16) * 16 * k;
    o2 += (int64_t)(d.H / 16) * (d.I / 16) * 16 * k;
  }
  L->bi = fc1_bi(d);
  if (!tmoe::tc_supported(d.H, d.I, L->bi, d.rot_block_h, d.rot_block_i)) {
    delete L;
    return fail(TM_EUNSUPPORTED, "geometry H=%d I=%d rot %d/%d not covered by the tensor-core kernels", d.H, d.I,
                d.rot_block_h, d.rot_block_i);
  }
  cudaError_t e;
  if ((e = cudaGetDevice(&L->device)) != cudaSuccess) { delete L; return cuda_fail(e, "cudaGetDevice"); }
  L->d_off1 = L->d_off2 = nullptr;
  L->d_bits = nullptr;
  L->d_lut = nullptr;
  L->use_lut = 0;
  L->wait_ns = 0;
  L->stall_issuer = 0;
  if ((e = cudaMalloc(&L->d_off1, d.E * 8)) != cudaSuccess ||
      (e = cudaMalloc(&L->d_off2, d.E * 8)) != cudaSuccess ||
      (e = cudaMalloc(&L->d_bits, d.E)) != cudaSuccess ||
      (e = cudaMalloc(&L->d_lut, tmoe::decode_lut_bytes())) != cudaSuccess ||
      (e = cudaMemcpy(L->d_off1, off1.data(), d.E * 8, cudaMemcpyHostToDevice)) != cudaSuccess ||
      (e = cudaMemcpy(L->d_off2, off2.data(), d.E * 8, cudaMemcpyHostToDevice)) != cudaSuccess ||
      (e = cudaMemcpy(L->d_bits, L->bits.data(), d.E, cudaMemcpyHostToDevice)) != cudaSuccess ||
      (e = tmoe::build_decode_lut(L->d_lut, nullptr)) != cudaSuccess ||
      (e = cudaStreamSynchronize(nullptr)) != cudaSuccess) {
    cudaFree(L->d_off1);
    cudaFree(L->d_off2);
    cudaFree(L->d_bits);
    cudaFree(L->d_lut);
    delete L;
    return cuda_fail(e, "upload descriptor tables");
  }
  *out = L;
  if (workspace_bytes) *workspace_bytes = make_layout(d, d.max_tokens).total;
  return TM_OK;
}

size_t trellis_moe_workspace_size(const tm_layer* layer, int32_t max_tokens) {
  if (!layer || max_tokens < 0) return 0;
  return make_layout(layer->desc, max_tokens).total;
}

void trellis_moe_destroy(tm_layer* layer) {
  if (!layer) return;
  {
    std::lock_guard<std::mutex> lock(layer->graph_mu);
    drop_host_graphs(layer);
  }
  if (layer->capture_stream) cudaStreamDestroy(layer->capture_stream);
  cudaFree(layer->d_off1);
  cudaFree(layer->d_off2);
  cudaFree(layer->d_bits);
  cudaFree(layer->d_lut);
  delete layer;
}

static tm_status check_mode(int32_t mode) {
  if (mode != TM_MODE_AUTO && mode != TM_MODE_W4A16 && mode != TM_MODE_W4A8)
    return fail(TM_EINVAL, "mode=%d is not a tm_mode", mode);
  return TM_OK;
}

tm_status trellis_moe_forward(tm_layer* layer, const uint16_t* x, const int32_t* topk_ids, const float* topk_w,
                              int32_t T, int32_t mode, float* out, void* workspace, size_t workspace_bytes,
                              void* stream) {
  g_err[0] = 0;
  if (!layer) return fail(TM_EINVAL, "layer is NULL");
  if (T < 0) return fail(TM_EINVAL, "T=%d < 0", T);
  if (check_mode(mode) != TM_OK) return TM_EINVAL;
  if (T == 0) return TM_OK;
  if (!x || !topk_ids || !topk_w || !out) return fail(TM_EINVAL, "x, topk_ids, topk_w and out must be non-NULL");
  if (((uintptr_t)x) % 8 || ((uintptr_t)out) % 16) return fail(TM_EINVAL, "x must be 8-byte and out 16-byte aligned");
  Layout L;
  tm_status s = check_ws(layer, T, workspace, workspace_bytes, &L);
  if (s != TM_OK) return s;
  if ((s = check_rows(layer->desc, T, mode)) != TM_OK) return s;
  cudaError_t e;
  if ((e = stage_mark(layer, 0, (cudaStream_t)stream)) != cudaSuccess) return cuda_fail(e, "stage event");
  return run_layer(layer, x, topk_ids, topk_w, nullptr, T, mode, out, workspace, L, (cudaStream_t)stream);
}

tm_status trellis_moe_forward_logits(tm_layer* layer, const uint16_t* x, const float* logits, int32_t T,
                                     int32_t mode, float* out, void* workspace, size_t workspace_bytes,
                                     void* stream) {
  g_err[0] = 0;
  if (!layer) return fail(TM_EINVAL, "layer is NULL");
  if (T < 0) return fail(TM_EINVAL, "T=%d < 0", T);
  if (check_mode(mode) != TM_OK) return TM_EINVAL;
  if (T == 0) return TM_OK;
  if (!x || !logits || !out) return fail(TM_EINVAL, "x, logits and out must be non-NULL");
  if (((uintptr_t)x) % 8 || ((uintptr_t)out) % 16) return fail(TM_EINVAL, "x must be 8-byte and out 16-byte aligned");
  Layout L;
  tm_status s = check_ws(layer, T, workspace, workspace_bytes, &L);
  if (s != TM_OK) return s;
  if ((s = check_rows(layer->desc, T, mode)) != TM_OK) return s;
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e;
  if ((e = stage_mark(layer, 0, st)) != cudaSuccess) return cuda_fail(e, "stage event");
  return run_layer(layer, x, nullptr, nullptr, logits, T, mode, out, workspace, L, st);
}

namespace {

// Copy-in, layer and copy-out of one host-buffer call, enqueued on `st`.
tm_status enqueue_host(tm_layer* layer, const uint16_t* x_host, const float* logits_host, int32_t T, int32_t mode,
                       float* out_host, void* workspace, const Layout& L, cudaStream_t st) {
  const tm_layer_desc& d = layer->desc;
  uint16_t* dx = at<uint16_t>(workspace, L, Layout::HOST_X);
  float* dl = at<float>(workspace, L, Layout::HOST_LOGITS);
  float* dout = at<float>(workspace, L, Layout::HOST_OUT);
  cudaError_t e;
  if ((e = cudaMemcpyAsync(dx, x_host, (size_t)T * d.H * 2, cudaMemcpyHostToDevice, st)) != cudaSuccess)
    return cuda_fail(e, "copy x to device");
  if ((e = cudaMemcpyAsync(dl, logits_host, (size_t)T * d.E * 4, cudaMemcpyHostToDevice, st)) != cudaSuccess)
    return cuda_fail(e, "copy logits to device");
  if ((e = stage_mark(layer, 0, st)) != cudaSuccess) return cuda_fail(e, "stage event");
  tm_status s = run_layer(layer, dx, nullptr, nullptr, dl, T, mode, dout, workspace, L, st);
  if (s != TM_OK) return s;
  if ((e = cudaMemcpyAsync(out_host, dout, (size_t)T * d.H * 4, cudaMemcpyDeviceToHost, st)) != cudaSuccess)
    return cuda_fail(e, "copy out to host");
  return TM_OK;
}

// The device address of page-locked host memory mapped into the device's
// address space (with unified addressing, the host address itself); NULL for
// pageable or unmapped memory.
const void* mapped_ptr(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

// The layer on mapped host buffers: the kernels read x and the logits and
// write the result across the host link themselves, no staging copies.
tm_status enqueue_mapped(tm_layer* layer, const uint16_t* x_dev, const float* logits_dev, int32_t T, int32_t mode,
                         float* out_dev, void* workspace, const Layout& L, cudaStream_t st) {
  cudaError_t e;
  if ((e = stage_mark(layer, 0, st)) != cudaSuccess) return cuda_fail(e, "stage event");
  return run_layer(layer, x_dev, nullptr, nullptr, logits_dev, T, mode, out_dev, workspace, L, st);
}

constexpr size_t kMaxHostGraphs = 16;

// Captures enqueue_mapped on the layer's private stream and instantiates it.
// Returns NULL if any step fails; the caller then runs the call directly, which
// reports a real argument or launch error itself.
cudaGraphExec_t capture_host(tm_layer* layer, const uint16_t* x_dev, const float* logits_dev, int32_t T,
                             int32_t mode, float* out_dev, void* workspace, const Layout& L) {
  if (!layer->capture_stream &&
      cudaStreamCreateWithFlags(&layer->capture_stream, cudaStreamNonBlocking) != cudaSuccess) {
    layer->capture_stream = nullptr;
    cudaGetLastError();
    return nullptr;
  }
  cudaStream_t cs = layer->capture_stream;
  if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  const tm_status s = enqueue_mapped(layer, x_dev, logits_dev, T, mode, out_dev, workspace, L, cs);
  cudaGraph_t graph = nullptr;
  const cudaError_t e = cudaStreamEndCapture(cs, &graph);
  cudaGraphExec_t exec = nullptr;
  if (s == TM_OK && e == cudaSuccess && graph && cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess)
    exec = nullptr;
  if (graph) cudaGraphDestroy(graph);
  cudaGetLastError();
  g_err[0] = 0;
  return exec;
}

// The graph for this buffer set, capturing it on its second use; NULL on the
// first use or after a failed capture (run directly). Caller holds graph_mu.
cudaGraphExec_t host_graph(tm_layer* layer, const uint16_t* x_dev, const float* logits_dev, int32_t T,
                           int32_t mode, float* out_dev, void* workspace, const Layout& L) {
  auto& v = layer->graphs;
  const uint64_t now = ++layer->graph_clock;
  for (auto& g : v) {
    if (g.x != x_dev || g.logits != logits_dev || g.out != out_dev || g.ws != workspace || g.T != T || g.mode != mode)
      continue;
    g.used = now;
    if (!g.exec && !g.failed) {
      g.exec = capture_host(layer, x_dev, logits_dev, T, mode, out_dev, workspace, L);
      g.failed = g.exec == nullptr;
    }
    return g.exec;
  }
  if (v.size() >= kMaxHostGraphs) {
    auto lru = std::min_element(v.begin(), v.end(),
                                [](const tm_layer::HostGraph& a, const tm_layer::HostGraph& b) { return a.used < b.used; });
    if (lru->exec) cudaGraphExecDestroy(lru->exec);
    v.erase(lru);
  }
  v.push_back({x_dev, logits_dev, out_dev, workspace, T, mode, false, now, nullptr});
  return nullptr;
}

}  // namespace

tm_status trellis_moe_forward_host(tm_layer* layer, const uint16_t* x_host, const float* logits_host, int32_t T,
                                   int32_t mode, float* out_host, void* workspace, size_t workspace_bytes,
                                   void* stream) {
  g_err[0] = 0;
  if (!layer) return fail(TM_EINVAL, "layer is NULL");
  if (T < 0) return fail(TM_EINVAL, "T=%d < 0", T);
  if (check_mode(mode) != TM_OK) return TM_EINVAL;
  if (T == 0) return TM_OK;
  if (!x_host || !logits_host || !out_host) return fail(TM_EINVAL, "x_host, logits_host and out_host must be non-NULL");
  Layout L;
  tm_status s = check_ws(layer, T, workspace, workspace_bytes, &L);
  if (s != TM_OK) return s;
  if ((s = check_rows(layer->desc, T, mode)) != TM_OK) return s;
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e;
  const auto* xd = static_cast<const uint16_t*>(mapped_ptr(x_host));
  const auto* ld = static_cast<const float*>(mapped_ptr(logits_host));
  auto* od = static_cast<float*>(const_cast<void*>(mapped_ptr(out_host)));
  // (the opt-in atomic combine clears and accumulates into the output: it
  // keeps the staged copies)
  if (layer->desc.deterministic && xd && ld && od && ((uintptr_t)xd) % 8 == 0 && ((uintptr_t)od) % 16 == 0) {
    std::lock_guard<std::mutex> lock(layer->graph_mu);
    cudaGraphExec_t exec = host_graph(layer, xd, ld, T, mode, od, workspace, L);
    if (exec) {
      if ((e = cudaGraphLaunch(exec, st)) != cudaSuccess) return cuda_fail(e, "graph launch");
    } else if ((s = enqueue_mapped(layer, xd, ld, T, mode, od, workspace, L, st)) != TM_OK) {
      return s;
    }
  } else if ((s = enqueue_host(layer, x_host, logits_host, T, mode, out_host, workspace, L, st)) != TM_OK) {
    return s;
  }
  if ((e = cudaStreamSynchronize(st)) != cudaSuccess) return cuda_fail(e, "synchronize");
  return TM_OK;
}

tm_status trellis_moe_route(const float* logits, int32_t T, int32_t E, int32_t k, int32_t* ids, float* w,
                            void* stream) {
  g_err[0] = 0;
  if (T < 0) return fail(TM_EINVAL, "T=%d < 0", T);
  if (E < 1 || E > tmoe::kMaxExperts) return fail(TM_EUNSUPPORTED, "E=%d outside 1..%d", E, tmoe::kMaxExperts);
  if (k < 1 || k > 32 || k > E) return fail(TM_EINVAL, "k=%d outside 1..min(E,32)", k);
  if (T == 0) return TM_OK;
  if (!logits || !ids || !w) return fail(TM_EINVAL, "logits, ids and w must be non-NULL");
  cudaError_t e = tmoe::launch_route_topk(logits, T, E, k, ids, w, (cudaStream_t)stream);
  return e == cudaSuccess ? TM_OK : cuda_fail(e, "router");
}

tm_status trellis_moe_route_map(tm_layer* layer, const int32_t* topk_ids, int32_t T, int32_t block, int32_t* counts,
                                int32_t* offsets, int32_t* route_of_slot, int32_t* slot_of_route, void* workspace,
                                size_t workspace_bytes, void* stream) {
  g_err[0] = 0;
  if (!layer) return fail(TM_EINVAL, "layer is NULL");
  if (T < 0) return fail(TM_EINVAL, "T=%d < 0", T);
  if (block < 1 || block > kBlockMax) return fail(TM_EINVAL, "block=%d outside 1..%d", block, kBlockMax);
  if (T == 0) return TM_OK;
  if (!topk_ids || !counts || !offsets || !route_of_slot || !slot_of_route)
    return fail(TM_EINVAL, "route map arguments must be non-NULL");
  Layout L;
  tm_status s = check_ws(layer, T, workspace, workspace_bytes, &L);
  if (s != TM_OK) return s;
  const tm_layer_desc& d = layer->desc;
  const int R = T * d.topk;
  const size_t need_blocks = ((size_t)R + (size_t)d.E * (block - 1)) / block + 1;
  if (need_blocks * 4 > L.bytes[Layout::BLOCK_EXPERT]) return fail(TM_EWORKSPACE, "workspace too small for block=%d", block);
  cudaStream_t st = (cudaStream_t)stream;
  uint32_t* err = at<uint32_t>(workspace, L, Layout::ERR);
  cudaError_t e;
  if ((e = cudaMemsetAsync(err, 0, L.bytes[Layout::ERR], st)) != cudaSuccess) return cuda_fail(e, "clear error word");
  tmoe::RouteMapArgs rm;
  rm.ids = topk_ids;
  rm.R = R;
  rm.E = d.E;
  rm.block = block;
  rm.rank = at<int32_t>(workspace, L, Layout::RANK);
  rm.tile_counts = at<int32_t>(workspace, L, Layout::TILE_COUNTS);
  rm.counts = counts;
  rm.offsets = offsets;
  rm.block_expert = at<int32_t>(workspace, L, Layout::BLOCK_EXPERT);
  rm.nblocks = at<int32_t>(workspace, L, Layout::NBLOCKS);
  rm.route_of_slot = route_of_slot;
  rm.slot_of_route = slot_of_route;
  rm.err = err;
  e = tmoe::launch_route_map(rm, st);
  return e == cudaSuccess ? TM_OK : cuda_fail(e, "route map");
}

tm_status trellis_moe_rotate_quant(tm_layer* layer, const uint16_t* x, int32_t T, int32_t mode, void* xq,
                                   uint8_t* xs, void* stream) {
  g_err[0] = 0;
  if (!layer) return fail(TM_EINVAL, "layer is NULL");
  if (T < 0) return fail(TM_EINVAL, "T=%d < 0", T);
  if (mode != TM_MODE_W4A16 && mode != TM_MODE_W4A8) return fail(TM_EINVAL, "mode must be W4A16 or W4A8");
  if (T == 0) return TM_OK;
  if (!x || !xq || (mode == TM_MODE_W4A8 && !xs)) return fail(TM_EINVAL, "x, xq (and xs for W4A8) must be non-NULL");
  if (((uintptr_t)x) % 8 || ((uintptr_t)xq) % 8) return fail(TM_EINVAL, "x and xq must be 8-byte aligned");
  const tm_layer_desc& d = layer->desc;
  if (d.gate_suh) return fail(TM_EUNSUPPORTED, "the layer has separate gate / up input signs (one rotation per route)");
  cudaError_t e = tmoe::launch_rotate_quant(x, d.in_suh, T, d.H, d.rot_block_h, mode == TM_MODE_W4A8, xq, xs,
                                          (cudaStream_t)stream);
  return e == cudaSuccess ? TM_OK : cuda_fail(e, "rotate+quantize");
}

tm_status trellis_moe_decode_tiles(tm_layer* layer, int32_t proj, int32_t expert, int32_t tile0, int32_t ntiles,
                                   int32_t mode, void* dst, void* stream) {
  g_err[0] = 0;
  if (!layer) return fail(TM_EINVAL, "layer is NULL");
  const tm_layer_desc& d = layer->desc;
  if (proj != 1 && proj != 2) return fail(TM_EINVAL, "proj=%d must be 1 or 2", proj);
  if (expert < 0 || expert >= d.E) return fail(TM_EINVAL, "expert=%d outside 0..%d", expert, d.E - 1);
  if (mode != TM_MODE_W4A16 && mode != TM_MODE_W4A8) return fail(TM_EINVAL, "mode must be W4A16 or W4A8");
  const long tiles = (long)(proj == 1 ? 2 * d.I : d.H) / 16 * ((proj == 1 ? d.H : d.I) / 16);
  if (tile0 < 0 || ntiles < 0 || tile0 + (long)ntiles > tiles)
    return fail(TM_EINVAL, "tiles %d..%d outside 0..%ld", tile0, tile0 + ntiles, tiles);
  if (ntiles == 0) return TM_OK;
  if (!dst || ((uintptr_t)dst) % 16) return fail(TM_EINVAL, "dst must be non-NULL and 16-byte aligned");
  const int K = layer->bits[expert];
  int64_t off = 0;
  for (int e = 0; e < expert; ++e)
    off += (int64_t)tiles * 16 * layer->bits[e];
  const int16_t* base = (proj == 1 ? d.fc1_payload : d.fc2_payload) + off + (int64_t)tile0 * 16 * K;
  cudaError_t e = tmoe::launch_decode_tiles(base, K, ntiles, mode == TM_MODE_W4A8, dst, (cudaStream_t)stream);
  return e == cudaSuccess ? TM_OK : cuda_fail(e, "decode tiles");
}

tm_status trellis_moe_workspace_region(const tm_layer* layer, int32_t T, int32_t which, size_t* offset,
                                       size_t* bytes) {
  g_err[0] = 0;
  if (!layer || !offset || !bytes) return fail(TM_EINVAL, "NULL argument");
  if (T < 0) return fail(TM_EINVAL, "T=%d < 0", T);
  static const int map[] = {Layout::XQ, Layout::XS, Layout::ZQ, Layout::ZS, Layout::ROWS, Layout::SLOT_OF_ROUTE, Layout::ERR};
  if (which < 0 || which >= (int)(sizeof(map) / sizeof(map[0]))) return fail(TM_EINVAL, "unknown region %d", which);
  const Layout L = make_layout(layer->desc, T);
  *offset = L.off[map[which]];
  *bytes = L.bytes[map[which]];
  return TM_OK;
}

tm_status trellis_moe_set_stage_events(tm_layer* layer, void* const* events, int32_t n) {
  g_err[0] = 0;
  if (!layer) return fail(TM_EINVAL, "layer is NULL");
  {
    // Captured host-call graphs record the old events: drop them.
    std::lock_guard<std::mutex> lock(layer->graph_mu);
    drop_host_graphs(layer);
  }
  if (events == nullptr || n == 0) {
    for (int i = 0; i < 7; ++i) layer->stage_ev[i] = nullptr;
    return TM_OK;
  }
  if (n != 7) return fail(TM_EINVAL, "n=%d: pass 7 events (NULL entries allowed) or none", n);
  for (int i = 0; i < 7; ++i) layer->stage_ev[i] = (cudaEvent_t)events[i];
  return TM_OK;
}

tm_status trellis_moe_set_decode_lut(tm_layer* layer, int32_t on) {
  g_err[0] = 0;
  if (!layer) return fail(TM_EINVAL, "layer is NULL");
  if (on != 0 && on != 1) return fail(TM_EINVAL, "on=%d must be 0 or 1", on);
  {
    // captured host-call graphs hold the other variant's kernels: drop them
    std::lock_guard<std::mutex> lock(layer->graph_mu);
    drop_host_graphs(layer);
  }
  layer->use_lut = on;
  return TM_OK;
}

tm_status trellis_moe_set_wait_test(tm_layer* layer, uint64_t wait_limit_ns, int32_t stall_issuer) {
  g_err[0] = 0;
  if (!layer) return fail(TM_EINVAL, "layer is NULL");
  if (stall_issuer != 0 && stall_issuer != 1) return fail(TM_EINVAL, "stall_issuer=%d must be 0 or 1", stall_issuer);
  {
    // captured host-call graphs hold the old settings: drop them
    std::lock_guard<std::mutex> lock(layer->graph_mu);
    drop_host_graphs(layer);
  }
  layer->wait_ns = wait_limit_ns;
  layer->stall_issuer = stall_issuer;
  return TM_OK;
}

tm_status trellis_moe_poll_error(tm_layer* layer, void* workspace, uint32_t* flags, void* stream) {
  g_err[0] = 0;
  if (!layer || !workspace || !flags) return fail(TM_EINVAL, "NULL argument");
  // The error word is the first region of every layout, at offset 0.
  cudaStream_t st = (cudaStream_t)stream;
  uint32_t h = 0;
  cudaError_t e;
  if ((e = cudaMemcpyAsync(&h, workspace, 4, cudaMemcpyDeviceToHost, st)) != cudaSuccess) return cuda_fail(e, "read error word");
  if ((e = cudaStreamSynchronize(st)) != cudaSuccess) return cuda_fail(e, "synchronize");
  if ((e = cudaMemsetAsync(workspace, 0, 4, st)) != cudaSuccess) return cuda_fail(e, "clear error word");
  *flags = h;
  if (h != 0)
    return fail(TM_EDEVICE, "device error flags 0x%x (bit 0: expert id out of range; bit 1: a pipeline wait gave up)", h);
  return TM_OK;
}

}  // extern "C"
