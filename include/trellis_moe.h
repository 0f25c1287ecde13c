/*
 * trellis_moe.h -- C ABI of a fused mixture-of-experts layer whose expert
 * weights are bitshift-trellis codes, for NVIDIA GB300 (sm_103a).
 *
 * What the layer computes (sources are four pull-request pages, cited by title
 * and section):
 *   1. route:    top-k expert ids and weights from router logits (optional);
 *   2. route map: per-expert counts, padded exclusive scan, stable route order
 *                (sparkinfer PR #90 "moe: integrate EXL3 Trellis into the fused
 *                W4A16 API", review of route_pack.py; b12x PR #433 "Share
 *                trellis preparation across native and EXL3 containers",
 *                review of route_pack.py);
 *   3. x~ = H_b(suh * x), one kernel that also quantises it: fp16 for W4A16,
 *      MXFP8 (E4M3 + one E8M0 exponent per 32) for W4A8 (b12x PR #129
 *      "feat(moe): serve canonical Fruit QSRT atoms", Hot path);
 *   4. FC1 gate/up grouped GEMM over route-major rows, expanding 256-weight
 *      trellis tiles (16*K int16 words, 16-bit tail-biting state, MCG codebook
 *      0xCBAC1FED / 0x8fff8fff / 0x3b603b60, per-output-channel fp16 scales)
 *      straight into MMA operands -- dense weights are never written to
 *      memory (same page, Hot path; sparkinfer PR #90, review of
 *      intrinsics.py and prepare.py);
 *   5. fused epilogue: H -> svh -> SiLU(gate)*up -> suh_down -> H (sparkinfer
 *      PR #90, review of kernel.py: _run_activation);
 *   6. FC2 route-major grouped GEMM with the same decode, then the output
 *      rotation is undone (output scale, H, down_svh; with the tensor-core
 *      FC2 these per-route steps run inside the deterministic combine);
 *   7. top-k weighted combine into an FP32 output, in fixed slot order
 *      (deterministic) or by FP32 atomics (opt-in, not bitwise reproducible:
 *      b12x PR #433, conversation: "does not guarantee bitwise summation
 *      order").
 *
 * Conventions for every entry point:
 *   - Pointers named *_host are host memory; all others are device memory of
 *     the current CUDA device, owned by the caller, never freed by the library.
 *   - "fp16" / "bf16" arrays are passed as uint16_t bit patterns.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   - Every argument is validated on the host before any launch; a call that
 *     returns an error has launched nothing and written nothing.
 *   - Errors: a negative tm_status; trellis_moe_last_error() gives a message
 *     for the calling thread.
 *   - Only trellis_moe_prepare and trellis_linear_prepare allocate device
 *     memory (small descriptor tables), and trellis_moe_forward_host builds
 *     the CUDA graphs it caches on the handle (see there).
 *     trellis_moe_forward, trellis_moe_forward_logits and
 *     trellis_linear_forward use only the caller's workspace, launch only on
 *     `stream`, and can be captured in a CUDA graph (the workspace pointer must
 *     then stay the same for every replay); trellis_moe_forward_host
 *     synchronises its stream and is not capturable.
 *
 * Also here: a dense trellis-coded linear layer on the same kernels
 * (trellis_linear_*, at the end of this file).
 */
#ifndef TRELLIS_MOE_H_
#define TRELLIS_MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct tm_layer tm_layer; /* opaque; created by prepare, freed by destroy */

typedef enum {
  TM_OK = 0,
  TM_EINVAL = -1,        /* bad argument (null pointer, shape, range, alignment) */
  TM_EUNSUPPORTED = -2,  /* well-formed but outside what this build implements */
  TM_EWORKSPACE = -3,    /* workspace missing, too small or misaligned */
  TM_ECUDA = -4,         /* a CUDA runtime call failed */
  TM_EDEVICE = -5        /* a kernel reported bad device data (see poll_error) */
} tm_status;

typedef enum {
  TM_MODE_AUTO = 0,   /* W4A8 when T <= decode_max_rows and T*topk <= 1024, else W4A16 */
  TM_MODE_W4A16 = 1,  /* fp16 activations x fp16 codebook weights, fp32 accumulate */
  TM_MODE_W4A8 = 2    /* MXFP8 activations x E4M3-rounded codebook weights; bounded
                         decode rows only (b12x PR #129, Hot path): T*topk <= 1024,
                         else the forward calls return TM_EUNSUPPORTED */
} tm_mode;

/* Layer description. Device arrays must stay valid until trellis_moe_destroy. */
typedef struct {
  int32_t E;              /* experts, 1..256 */
  int32_t H;              /* hidden size, multiple of 128 */
  int32_t I;              /* intermediate size per half, multiple of 64 */
  int32_t topk;           /* experts per token, 1..min(E, 32) */
  int32_t rot_block_h;    /* Hadamard block on H: 1 (identity), 64, 128, or 512 (H4 (x) H128 in
                             Sylvester order, the coupled H512/H128 boundary of TrellisMX-style
                             layers; H a multiple of 512; the output side then always takes the
                             ordered combine) */
  int32_t rot_block_i;    /* Hadamard block on I: 1, 64 or 128 (must divide I) */
  const uint8_t* bits_per_expert; /* HOST [E], trellis bits K_e in 2..6 */
  /* Payload words, experts concatenated in order. Expert e's FC1 block is
   * [2I/16][H/16][16*K_e] int16 (tile rows = output channels: rows 0..I-1 gate,
   * I..2I-1 up); its FC2 block is [H/16][I/16][16*K_e]. Base 16-byte aligned. */
  const int16_t* fc1_payload;
  const int16_t* fc2_payload;
  const uint16_t* fc1_scale;  /* fp16 [E, 2I] per-output-channel scale */
  const uint16_t* fc2_scale;  /* fp16 [E, H] */
  const uint16_t* in_suh;     /* fp16 [H] input signs (shared by gate and up; see gate_suh) */
  const uint16_t* rot_tab;    /* fp16 [E, 3I] = gate svh | up svh | down suh */
  const uint16_t* out_svh;    /* fp16 [E, H] output (down) svh */
  int32_t max_tokens;         /* largest T any forward call will pass, >= 1 */
  int32_t decode_max_rows;    /* AUTO picks W4A8 iff T <= this (default 8) and T*topk <= 1024 */
  int32_t deterministic;      /* 1: fixed-order FP32 combine; 0: FP32 atomics on the
                                 tensor-core path. The decode-rows path (W4A8, and W4A16
                                 at T*topk < 4E) sums every token's routes in fixed order
                                 in either setting, so there 0 gives the deterministic
                                 result. */
  /* Optional separate input signs of the FC1 gate rows and of the up rows
   * (b12x PR #129 "feat(moe): serve canonical Fruit QSRT atoms", review of
   * trellis_w4a8.py: gate_suh and up_suh of shape (1, H) or (num_experts, H)).
   * Both NULL: every route's gate and up rows see x~ = H_b(in_suh * x). Both
   * set: fp16 [input_sign_rows, H] each, input_sign_rows 1 (shared by the
   * experts) or E (row e for expert e); the gate rows of a route to expert e
   * see H_b(gate_suh[e] * x) and its up rows H_b(up_suh[e] * x), and in_suh is
   * not read (may be NULL). Tensor-core route blocks are then 128 routes. */
  const uint16_t* gate_suh;
  const uint16_t* up_suh;
  int32_t input_sign_rows;
  /* Optional TrellisMX-style weight scales (flashinfer PR #69 "b12x fused
   * MoE: TrellisMX ...", Description: trellis streams that decode to E4M3,
   * one UE8M0 scale per 32 weights). Both NULL: plain trellis weights. Both
   * set: UE8M0 bytes u, one per 32 consecutive weights of a row along the
   * contraction axis, fc1_wscale [E][2I][H/32] and fc2_wscale [E][H][I/32]
   * (16-byte aligned); every weight is then E4M3(cb(s)) * 2^(u - 127) in both
   * modes. prepare reads them once and requires u - 127 in [-15, 13], the
   * range in which the tensor-core path's fp16 operands hold the weights
   * exactly (TM_EUNSUPPORTED otherwise). Such layers expand by the codebook
   * hash (set_decode_lut has no effect on them). */
  const uint8_t* fc1_wscale;
  const uint8_t* fc2_wscale;
} tm_layer_desc;

/* Validate `desc`, upload the per-expert offset tables and return a handle and
 * the workspace size (bytes) a forward call of up to desc->max_tokens tokens
 * needs. Allocates only the small descriptor tables; call before any stream
 * capture. Errors: TM_EINVAL / TM_EUNSUPPORTED / TM_ECUDA; *out is then NULL. */
tm_status trellis_moe_prepare(const tm_layer_desc* desc, tm_layer** out, size_t* workspace_bytes);

/* Workspace bytes for forward calls of up to `max_tokens` tokens (<= the
 * prepared max_tokens). */
size_t trellis_moe_workspace_size(const tm_layer* layer, int32_t max_tokens);

/* Full layer from given routes.
 *   x        bf16 [T, H] activations (8-byte aligned)
 *   topk_ids int32 [T, topk] expert ids; out-of-range ids are dropped from the
 *            sum and flagged in the device error word (trellis_moe_poll_error)
 *   topk_w   fp32 [T, topk] route weights
 *   mode     tm_mode
 *   out      fp32 [T, H] result (overwritten; 16-byte aligned)
 *   workspace >= trellis_moe_workspace_size(layer, T) bytes, 256-byte aligned;
 *            contents on entry are ignored (any bytes give the same result).
 * T = 0 is a no-op. Errors: TM_EINVAL, TM_EWORKSPACE, TM_ECUDA, and
 * TM_EUNSUPPORTED for mode W4A8 with T*topk > 1024. */
tm_status trellis_moe_forward(tm_layer* layer, const uint16_t* x, const int32_t* topk_ids,
                              const float* topk_w, int32_t T, int32_t mode, float* out,
                              void* workspace, size_t workspace_bytes, void* stream);

/* Router + full layer: logits fp32 [T, E] are routed on the device (top-k,
 * softmax over the selected logits) into the workspace, then as forward. */
tm_status trellis_moe_forward_logits(tm_layer* layer, const uint16_t* x, const float* logits,
                                     int32_t T, int32_t mode, float* out,
                                     void* workspace, size_t workspace_bytes, void* stream);

/* As forward_logits, but x_host, logits_host and out_host are HOST buffers
 * (pinned memory recommended). Copies the inputs into the workspace, runs the
 * layer and copies the result back, all on `stream`, then synchronises the
 * stream. Workspace: trellis_moe_workspace_size(layer, T) bytes.
 * When all three buffers are page-locked and mapped into the device's address
 * space (pinned memory under unified addressing; x_host 8-byte and out_host
 * 16-byte aligned) and the layer is deterministic, no staging copies are made:
 * the kernels read x and the logits and write the result over the host link
 * (NVLink-C2C on Grace systems) themselves, the same bytes in each direction.
 * The handle then also remembers the buffer set (x_host, logits_host,
 * out_host, workspace, T, mode): its second call captures the layer as a CUDA
 * graph on a private stream and later calls launch that graph on `stream`.
 * Each call reads the buffers' contents at that call. Up to 16 sets are kept,
 * least recently used evicted; set_stage_events and destroy free them; the
 * cache is guarded by a mutex. Otherwise the inputs are copied into the
 * workspace and the result out of it on `stream`. */
tm_status trellis_moe_forward_host(tm_layer* layer, const uint16_t* x_host,
                                   const float* logits_host, int32_t T, int32_t mode,
                                   float* out_host, void* workspace, size_t workspace_bytes,
                                   void* stream);

/* Top-k softmax router. logits fp32 [T, E] -> ids int32 [T, k] (descending
 * logit, ties to the lower id) and w fp32 [T, k] = softmax over the k selected
 * logits. E <= 256, 1 <= k <= min(E, 32). No workspace. */
tm_status trellis_moe_route(const float* logits, int32_t T, int32_t E, int32_t k,
                            int32_t* ids, float* w, void* stream);

/* Route map of topk_ids int32 [T, topk] with expert segments padded to `block`
 * (1..256): counts int32 [E], offsets int32 [E+1] (padded exclusive scan),
 * route_of_slot int32 [offsets[E]] (route r = t*topk + j, -1 for padding;
 * within an expert in ascending r), slot_of_route int32 [T*topk] (-1 for a
 * dropped id). The caller sizes route_of_slot for the worst case
 * T*topk + E*(block-1). Uses the workspace for scratch. */
tm_status trellis_moe_route_map(tm_layer* layer, const int32_t* topk_ids, int32_t T, int32_t block,
                                int32_t* counts, int32_t* offsets, int32_t* route_of_slot,
                                int32_t* slot_of_route, void* workspace, size_t workspace_bytes,
                                void* stream);

/* Step 3 alone: x bf16 [T, H] -> W4A16: fp16 [T, H] into xq; W4A8: E4M3 bytes
 * [T, H] into xq and E8M0 bytes [T, H/32] into xs (xs unused for W4A16), with
 * the layer's shared in_suh (TM_EUNSUPPORTED for a layer with separate gate /
 * up signs). W4A8 rotates in fp64 and rounds each value once to fp32 before
 * quantising. */
tm_status trellis_moe_rotate_quant(tm_layer* layer, const uint16_t* x, int32_t T, int32_t mode,
                                   void* xq, uint8_t* xs, void* stream);

/* Decode `ntiles` tiles of expert `expert`'s projection `proj` (1 = FC1,
 * 2 = FC2) starting at tile index `tile0` (row-tile major order) into dst:
 * W4A16 -> fp16 bits [ntiles][256], W4A8 -> E4M3 bytes [ntiles][256], in
 * in-tile weight order j (row j/16, column j%16). For parity tests. */
tm_status trellis_moe_decode_tiles(tm_layer* layer, int32_t proj, int32_t expert, int32_t tile0,
                                   int32_t ntiles, int32_t mode, void* dst, void* stream);

/* Where a forward call of `T` tokens keeps its intermediates inside the
 * workspace (for tests): which = 0 x~, 1 x~ E8M0 exponents, 2 FC1 epilogue
 * output z~, 3 z~ E8M0 exponents (x~ and z~: fp16 for W4A16, in slot order on
 * the tensor-core path; for W4A8, which runs on the decode rows, the E4M3
 * codes held as fp16), 4 per-slot
 * FC2 output (fp32 [slots, H]: the unrotated route output, or, for the
 * tensor-core FC2 with the deterministic combine, the scaled FC2 accumulator
 * after the Hadamard levels within each 64-column half; not written by the
 * decode-rows path, whose combine is part of the FC2 epilogue), 5
 * slot_of_route (int32 [T*topk]),
 * 6 device error word (uint32). Returns TM_EINVAL for an unknown `which`. */
tm_status trellis_moe_workspace_region(const tm_layer* layer, int32_t T, int32_t which,
                                       size_t* offset, size_t* bytes);

/* Stage timing for benchmarks and profilers. With `events` non-NULL (n = 7
 * cudaEvent_t handles created by the caller, NULL entries skipped), every later
 * forward call on this handle records events[i] on its stream (inside a stream
 * capture with cudaEventRecordExternal, so that the records become nodes of the
 * captured CUDA graph; otherwise as a plain record), at these boundaries: 0 start, 1 after the router (forward_logits
 * and forward_host only), 2 after the route map, 3 after rotate+quantize,
 * 4 after FC1, 5 after FC2, 6 after the combine. In the decode-rows path the
 * router, route map and rotation are one kernel (1..3 follow it together),
 * 4 follows the FC1 GEMM kernel (FC1's epilogue kernel counts with FC2) and
 * the combine is part of the FC2 epilogue (5 and 6 follow it together).
 * events = NULL or n = 0 turns recording off. The handles are copied; the
 * caller keeps ownership. */
tm_status trellis_moe_set_stage_events(tm_layer* layer, void* const* events, int32_t n);

/* How the decode-rows path (T*topk <= 1024: every W4A8 call, and W4A16 calls
 * with fewer than 4E routes) expands trellis
 * states into weights. on = 0 (the default): by the codebook hash in
 * registers (several CTAs per SM); on = 1: by lookup in a table of the
 * codebook value of every 16-bit state (65,536 fp16 entries; in W4A8 mode the
 * value of its E4M3 rounding), built on the device when the layer is prepared
 * and copied into each FC CTA's shared memory (one CTA per SM). On sm_103 the
 * lookups' random bank conflicts make the table the slower variant; it is
 * kept as the measured alternative. Both give the same
 * weights bit for bit: the table is the full-codeword shared lookup table
 * that b12x PR #129 "feat(moe): serve canonical Fruit QSRT atoms" (its commit
 * notes) splits out of that change for separate review, here filled from the
 * same expansion functions as the hash path. Drops the handle's captured
 * host-call graphs. Errors: TM_EINVAL. */
tm_status trellis_moe_set_decode_lut(tm_layer* layer, int32_t on);

/* Test hook for the tensor-core kernels' bounded waits (the failure detection
 * of a stalled pipeline). Every mbarrier wait of those kernels gives up after
 * wait_limit_ns of wall time (0 restores the default of 2 s); the CTA then
 * sets bit 1 of the error word, lets the copies it has in flight land, frees
 * its tensor memory and returns, leaving the call's output incomplete. With
 * stall_issuer = 1 the MMA issuer first waits on a barrier that nothing
 * arrives on, before it issues any MMA, so that wait runs out on every CTA:
 * a test then sees the error bit from trellis_moe_poll_error and checks that
 * the next call with stall_issuer = 0 is correct. Applies to later forward
 * calls on tensor-core shapes (the decode-rows kernels do not wait on one
 * another). Drops the handle's captured host-call graphs. Errors: TM_EINVAL. */
tm_status trellis_moe_set_wait_test(tm_layer* layer, uint64_t wait_limit_ns, int32_t stall_issuer);

/* Read and clear the device error word of `workspace` (synchronises `stream`).
 * *flags: bit 0 = an expert id was out of range; bit 1 = a tensor-core
 * kernel's pipeline wait gave up (the kernel stopped, released its tensor
 * memory and left its outputs incomplete). Returns TM_EDEVICE if any flag was
 * set, else TM_OK. */
tm_status trellis_moe_poll_error(tm_layer* layer, void* workspace, uint32_t* flags, void* stream);

/* Route map with no scratch from the caller and no allocation. No counterpart
 * on the source pages: it exists for callers that cannot allocate or lend
 * device memory -- hosts that own all device memory through a fixed plan and
 * pass only inputs and outputs, and latency-critical loops that must not
 * enter the allocator after start-up because allocation can synchronise the
 * device. Same arguments and results as trellis_moe_route_map, with the
 * layer's E and topk passed directly. Its scratch is one static device array
 * of about 10 KB per GPU, held while the library is loaded; limits:
 * T*topk <= 1024 routes, E <= 256 (TM_EUNSUPPORTED beyond, with a message).
 * The first call on a device looks up that array's device address, so make it
 * before any stream capture; the address is kept for the process's lifetime,
 * so a device reset (cudaDeviceReset) while the library is loaded is not
 * supported. All calls on a device share the array: calls whose kernels
 * overlap on the GPU race, so order them on one stream. Every call clears what
 * must start at zero. Dropped (out-of-range) ids get slot_of_route -1 as in
 * trellis_moe_route_map; no error word is kept. */
tm_status trellis_moe_route_map_static(const int32_t* topk_ids, int32_t T, int32_t E, int32_t topk,
                                       int32_t block, int32_t* counts, int32_t* offsets,
                                       int32_t* route_of_slot, int32_t* slot_of_route, void* stream);

/* Message of the last failed call on this thread ("" if none). */
const char* trellis_moe_last_error(void);

/* Free the handle and its descriptor tables (not the caller's arrays). */
void trellis_moe_destroy(tm_layer* layer);

/* ------------------------------------------------------------------------
 * Dense trellis-coded linear layer (no routing): one matrix W~ [N, K] with
 * the layer's weight code, output scales and Hadamard-and-sign rotations, for
 * dense projections (sparkinfer PR #90 "moe: integrate EXL3 Trellis into the
 * fused W4A16 API", review of kernel.py: run_trellis256_dense and of
 * tests/gemm/test_trellis_linear.py). For bf16 x [T, K]:
 *   x~  = Hblk_in(suh (.) x) rounded to fp16,
 *   out = svh (.) Hblk_out(s (.) (W~ x~))          fp32 [T, N]
 * with an FP16 x FP16 -> FP32 tensor-core contraction (W4A16). */
typedef struct tm_linear tm_linear;

typedef struct {
  int32_t N, K;             /* output / input channels: multiples of 128 */
  int32_t bits;             /* trellis K of every weight, 2..6 */
  int32_t rot_in, rot_out;  /* Hadamard blocks along K and N: 1, 64 or 128, dividing them */
  int32_t max_tokens;       /* workspace_bytes from prepare covers T <= max_tokens */
  /* DEVICE pointers, caller-owned, 16-byte aligned, outliving the handle: */
  const int16_t* payload;   /* [N/16][K/16][16*bits] words, tile (tn, tk) weight j at
                               row 16 tn + j/16, column 16 tk + j%16 (as the layer's) */
  const uint16_t* scale;    /* fp16 [N] */
  const uint16_t* suh;      /* fp16 [K] input signs */
  const uint16_t* svh;      /* fp16 [N] output signs */
} tm_linear_desc;

/* Validates desc and uploads two small tables; *workspace_bytes = the
 * workspace a call of max_tokens tokens needs. Errors: TM_EINVAL,
 * TM_EUNSUPPORTED, TM_ECUDA. */
tm_status trellis_linear_prepare(const tm_linear_desc* desc, tm_linear** out, size_t* workspace_bytes);

/* Workspace bytes for a call of max_tokens tokens (0 for a NULL handle). */
size_t trellis_linear_workspace_size(const tm_linear* lin, int32_t max_tokens);

/* x bf16 [T, K] (8-byte aligned), out fp32 [T, N] (16-byte aligned, written),
 * workspace >= trellis_linear_workspace_size(lin, T) bytes, 256-byte aligned
 * (contents on entry ignored), T <= max_tokens. Enqueued on `stream`; no
 * allocation, graph-capturable. T = 0 is a no-op. The first 4 bytes of the
 * workspace are the device error word (bit 1: a pipeline wait gave up).
 * Errors: TM_EINVAL, TM_EWORKSPACE, TM_ECUDA. */
tm_status trellis_linear_forward(tm_linear* lin, const uint16_t* x, int32_t T, float* out, void* workspace,
                                 size_t workspace_bytes, void* stream);

/* Read and clear the device error word of `workspace` (synchronises
 * `stream`). Returns TM_EDEVICE if any flag was set, else TM_OK. */
tm_status trellis_linear_poll_error(tm_linear* lin, void* workspace, uint32_t* flags, void* stream);

void trellis_linear_destroy(tm_linear* lin);

#ifdef __cplusplus
}
#endif

#endif /* TRELLIS_MOE_H_ */
