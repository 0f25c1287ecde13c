// Dense trellis-coded linear layer (sm_103a): the MoE layer's input rotation
// and tensor-core projection with no routing, for dense projections whose
// weights use the same bitshift-trellis code (sparkinfer PR #90 "moe:
// integrate EXL3 Trellis into the fused W4A16 API", review of kernel.py:
// run_trellis256_dense -- fp16 input conversion, rotation, fp16 GEMM, output
// rotation; review of tests/gemm/test_trellis_linear.py).
//
//   x~ = Hblk_in(suh (.) x) in fp16            k_rotate_quant (W4A16)
//   out = svh (.) Hblk_out(s (.) (W~ x~))      k_tc_fc<FC2> with one expert
//
// Token t is slot t of a single expert's segment, so the route map is the
// identity (k_linear_map) and the projection's epilogue stores each token's
// finished fp32 row; there is nothing to combine.
#include <stdarg.h>
#include <stdio.h>

#include <algorithm>

#include "../../include/trellis_moe.h"
#include "launch.h"

struct tm_linear {
  tm_linear_desc desc;
  int64_t* d_word_off;  // [1] = 0: the one expert's payload starts at word 0
  uint8_t* d_bits;      // [1]
};

namespace {

constexpr size_t kLinAlign = 256;
size_t lin_align(size_t v) { return (v + kLinAlign - 1) / kLinAlign * kLinAlign; }

tm_status lin_fail(tm_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  tmoe::set_last_error(buf);
  return s;
}

tm_status lin_cuda_fail(cudaError_t e, const char* what) {
  return lin_fail(TM_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Workspace of a call of up to T tokens: error word and unit counter | route
// of slot [blocks*256] | block expert [blocks] | block count | x~ fp16
// [blocks*256][K] (rows past T are operand padding that no epilogue stores).
struct LinLayout {
  size_t err, ros, bexp, nblk, xq, total;
  int blocks;
};

LinLayout lin_layout(const tm_linear_desc& d, int T) {
  LinLayout L{};
  const int bn = tmoe::tc_route_block();
  L.blocks = std::max(1, (T + bn - 1) / bn);
  size_t o = 0;
  L.err = o;
  o += lin_align(16);
  L.ros = o;
  o += lin_align((size_t)L.blocks * bn * 4);
  L.bexp = o;
  o += lin_align((size_t)L.blocks * 4);
  L.nblk = o;
  o += lin_align(4);
  L.xq = o;
  o += lin_align((size_t)L.blocks * bn * d.K * 2);
  L.total = o;
  return L;
}

__global__ void k_linear_map(int T, int slots, int blocks, int32_t* route_of_slot, int32_t* block_expert,
                             int32_t* nblocks) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < slots) route_of_slot[i] = (i < T) ? i : -1;
  if (i < blocks) block_expert[i] = 0;
  if (i == 0) *nblocks = blocks;
}

bool rot_ok(int b, int n) { return (b == 1 || b == 64 || b == 128) && n % b == 0; }

}  // namespace

extern "C" {

tm_status trellis_linear_prepare(const tm_linear_desc* desc, tm_linear** out, size_t* workspace_bytes) {
  tmoe::set_last_error("");
  if (out) *out = nullptr;
  if (!desc || !out) return lin_fail(TM_EINVAL, "desc and out must be non-NULL");
  const tm_linear_desc& d = *desc;
  if (d.N < 128 || d.N % 128 != 0) return lin_fail(TM_EUNSUPPORTED, "N=%d must be a positive multiple of 128", d.N);
  if (d.K < 128 || d.K % 128 != 0) return lin_fail(TM_EUNSUPPORTED, "K=%d must be a positive multiple of 128", d.K);
  if (d.bits < 2 || d.bits > 6) return lin_fail(TM_EUNSUPPORTED, "bits=%d outside 2..6", d.bits);
  if (!rot_ok(d.rot_in, d.K)) return lin_fail(TM_EUNSUPPORTED, "rot_in=%d must be 1, 64 or 128 and divide K", d.rot_in);
  if (!rot_ok(d.rot_out, d.N)) return lin_fail(TM_EUNSUPPORTED, "rot_out=%d must be 1, 64 or 128 and divide N", d.rot_out);
  if (d.max_tokens < 1) return lin_fail(TM_EINVAL, "max_tokens=%d must be >= 1", d.max_tokens);
  if ((long)d.max_tokens * d.K > (1L << 31)) return lin_fail(TM_EUNSUPPORTED, "max_tokens*K too large");
  const void* ptrs[] = {d.payload, d.scale, d.suh, d.svh};
  const char* names[] = {"payload", "scale", "suh", "svh"};
  for (int i = 0; i < 4; ++i) {
    if (!ptrs[i]) return lin_fail(TM_EINVAL, "%s is NULL", names[i]);
    if (((uintptr_t)ptrs[i]) % 16 != 0) return lin_fail(TM_EINVAL, "%s must be 16-byte aligned", names[i]);
  }
  tm_linear* L = new tm_linear();
  L->desc = d;
  L->d_word_off = nullptr;
  L->d_bits = nullptr;
  const int64_t zero = 0;
  const uint8_t bits = (uint8_t)d.bits;
  cudaError_t e;
  if ((e = cudaMalloc(&L->d_word_off, 8)) != cudaSuccess || (e = cudaMalloc(&L->d_bits, 1)) != cudaSuccess ||
      (e = cudaMemcpy(L->d_word_off, &zero, 8, cudaMemcpyHostToDevice)) != cudaSuccess ||
      (e = cudaMemcpy(L->d_bits, &bits, 1, cudaMemcpyHostToDevice)) != cudaSuccess) {
    cudaFree(L->d_word_off);
    cudaFree(L->d_bits);
    delete L;
    return lin_cuda_fail(e, "upload descriptor tables");
  }
  *out = L;
  if (workspace_bytes) *workspace_bytes = lin_layout(d, d.max_tokens).total;
  return TM_OK;
}

size_t trellis_linear_workspace_size(const tm_linear* lin, int32_t max_tokens) {
  if (!lin || max_tokens < 0) return 0;
  return lin_layout(lin->desc, max_tokens).total;
}

tm_status trellis_linear_forward(tm_linear* lin, const uint16_t* x, int32_t T, float* out, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  tmoe::set_last_error("");
  if (!lin) return lin_fail(TM_EINVAL, "linear is NULL");
  if (T < 0) return lin_fail(TM_EINVAL, "T=%d < 0", T);
  if (T == 0) return TM_OK;
  const tm_linear_desc& d = lin->desc;
  if (T > d.max_tokens) return lin_fail(TM_EINVAL, "T=%d > max_tokens=%d", T, d.max_tokens);
  if (!x || !out || !workspace) return lin_fail(TM_EINVAL, "x, out and workspace must be non-NULL");
  if (((uintptr_t)x) % 8 || ((uintptr_t)out) % 16) return lin_fail(TM_EINVAL, "x must be 8-byte and out 16-byte aligned");
  if (((uintptr_t)workspace) % kLinAlign) return lin_fail(TM_EWORKSPACE, "workspace must be 256-byte aligned");
  const LinLayout L = lin_layout(d, T);
  if (workspace_bytes < L.total)
    return lin_fail(TM_EWORKSPACE, "workspace of %zu bytes < %zu needed for T=%d", workspace_bytes, L.total, T);
  cudaStream_t st = (cudaStream_t)stream;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  uint32_t* err = reinterpret_cast<uint32_t*>(ws + L.err);
  int32_t* ros = reinterpret_cast<int32_t*>(ws + L.ros);
  int32_t* bexp = reinterpret_cast<int32_t*>(ws + L.bexp);
  int32_t* nblk = reinterpret_cast<int32_t*>(ws + L.nblk);
  void* xq = ws + L.xq;
  const int slots = L.blocks * tmoe::tc_route_block();
  cudaError_t e;
  if ((e = cudaMemsetAsync(err, 0, 16, st)) != cudaSuccess) return lin_cuda_fail(e, "clear error word");
  k_linear_map<<<(slots + 255) / 256, 256, 0, st>>>(T, slots, L.blocks, ros, bexp, nblk);
  if ((e = cudaGetLastError()) != cudaSuccess) return lin_cuda_fail(e, "route map");
  if ((e = tmoe::launch_rotate_quant(x, d.suh, T, d.K, d.rot_in, false, xq, nullptr, st, nullptr, 1)) != cudaSuccess)
    return lin_cuda_fail(e, "rotate");
  tmoe::FcArgs a{};
  a.E = 1;
  a.H = d.N;
  a.I = d.K;
  a.topk = 1;
  a.rot_b = d.rot_out;
  a.payload = d.payload;
  a.word_off = lin->d_word_off;
  a.bits = lin->d_bits;
  a.scale = d.scale;
  a.rot_tab = d.svh;
  a.act = xq;
  a.route_of_slot = ros;
  a.block_expert = bexp;
  a.nblocks = nblk;
  a.out_f32 = out;
  a.atomic = 0;
  a.raw_rows = 0;
  tmoe::TcArgs t{};
  t.f = a;
  t.bi = 128;
  t.err = err;
  t.sched = err + 1;
  t.act_rows = slots;
  t.route_block = tmoe::tc_route_block();
  if ((e = tmoe::launch_tc_fc(t, 2, d.bits, L.blocks, st)) != cudaSuccess) return lin_cuda_fail(e, "projection");
  return TM_OK;
}

tm_status trellis_linear_poll_error(tm_linear* lin, void* workspace, uint32_t* flags, void* stream) {
  tmoe::set_last_error("");
  if (!lin || !workspace || !flags) return lin_fail(TM_EINVAL, "NULL argument");
  cudaStream_t st = (cudaStream_t)stream;
  uint32_t h = 0;
  cudaError_t e;
  if ((e = cudaMemcpyAsync(&h, workspace, 4, cudaMemcpyDeviceToHost, st)) != cudaSuccess)
    return lin_cuda_fail(e, "read error word");
  if ((e = cudaStreamSynchronize(st)) != cudaSuccess) return lin_cuda_fail(e, "synchronize");
  if ((e = cudaMemsetAsync(workspace, 0, 4, st)) != cudaSuccess) return lin_cuda_fail(e, "clear error word");
  *flags = h;
  return h ? TM_EDEVICE : TM_OK;
}

void trellis_linear_destroy(tm_linear* lin) {
  if (!lin) return;
  cudaFree(lin->d_word_off);
  cudaFree(lin->d_bits);
  delete lin;
}

}  // extern "C"
