/*
 * klt.h -- C ABI of the GB300 latent-MoE layer tail library (libklt.so).
 *
 * The tail (Kimi K3 latent MoE, as described in the vLLM pull request "Fuse BF16 shared
 * experts into latent MegaMoE tail", Summary, and DeepGEMM PR 416 "Fuse and publish Kimi
 * K3's BF16 shared expert", Summary) computes, for every token t:
 *
 *   ids, w   = top-k of logits[t] and the softmax of the selected logits   (routing)
 *   zq, zs   = e4m3 quantisation of z[t] per 128 columns, fp32 scale amax/448
 *   r[t]     = sum_j w_j * SwiGLU-expert_{ids_j}(zq)       (routed experts, latent width L)
 *   n[t]     = RMSNorm(r[t]) * gamma                       (fp32 statistics)
 *   out[t]   = bf16( n[t] W_up^T + SwiGLU-shared(x[t]) )   (3584 -> 7168 up-projection
 *                                                           plus the BF16 shared expert,
 *                                                           summed in fp32, rounded once)
 *
 * Routed expert e: h = zq W13_e^T with gate = rows [0, I), up = rows [I, 2I);
 * a = silu(gate) * up quantised per 128 like z; y = aq W2_e^T.  Shared expert:
 * hs = x Ws13^T (gate rows [0, Is), up rows [Is, 2 Is)); s = (silu(g) * u) Ws2^T.
 *
 * Conventions for every entry point:
 *  - every function returns a klt status code (KLT_OK == 0);
 *  - pointers named "device" must be CUDA device pointers on the current device and
 *    16-byte aligned; the library never frees caller memory;
 *  - arguments are checked on the host before anything is launched; a failed check
 *    launches nothing and changes no state;
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).
 */
#ifndef KLT_H_
#define KLT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------------ status codes */
enum klt_status_code {
  KLT_OK = 0,
  KLT_ERR_INVALID_ARG = 1,     /* null pointer, M < 0, M > max_tokens, bad eps, ...     */
  KLT_ERR_UNSUPPORTED = 2,     /* a width not a multiple of 128, topk > E, E > 256,
                                  routed format unknown, device is not sm_103          */
  KLT_ERR_ALIGN = 3,           /* a pointer is not 16-byte aligned                     */
  KLT_ERR_CUDA = 4,            /* a CUDA runtime call or launch failed                 */
  KLT_ERR_DEVICE_TIMEOUT = 5,  /* a bounded on-device wait ran out (sticky)            */
  KLT_ERR_OOM = 6,             /* device allocation failed in klt_create               */
  KLT_ERR_TOO_LARGE = 7        /* request exceeds the fixed scratch of klt_route_noalloc */
};

/* Routed expert weight formats. */
enum klt_routed_format {
  KLT_FMT_FP8_B128 = 0,  /* e4m3 codes, one fp32 scale per 128 x 128 block            */
  KLT_FMT_NVFP4 = 1,     /* e2m1 codes (two per byte, even K in the low nibble), one
                            e4m3 scale per 16 K-elements, one fp32 scale per matrix    */
  KLT_FMT_MXFP8 = 2,     /* e4m3 codes, one power-of-two scale per 32 K-elements of a row
                            (an UE8M0 byte b: scale 2^(b-127)); the routed activations are
                            quantised the same way (scale 2^(floor(log2 amax) - 8)) and the
                            tensor core applies the scales (block-scaled MMA, no epilogue
                            promotion).  Needs H and L multiples of 256; always runs the
                            token-major engine.                                         */
  KLT_FMT_NVFP4_W4A4 = 3 /* NVFP4 weights as in KLT_FMT_NVFP4, kept packed in device
                            memory (0.5625 bytes per weight), and NVFP4 routed
                            activations: per 16 elements an e4m3 scale s = e4m3(amax / 6)
                            and e2m1 codes of v / s (nearest even, saturating, no tensor
                            scale).  The tensor core applies both operands' e4m3 scales
                            (block-scaled FP4 MMA, scale vector of 4 per 64 K) and the
                            epilogue the weights' fp32 per-matrix scale.  Needs H, L and I
                            multiples of 256; always runs the token-major engine.      */
};

/* klt_create flags. */
enum klt_flags {
  KLT_FLAG_NO_PDL = 1u << 0,  /* launch the kernels with plain stream ordering instead of
                                 programmatic dependent launch                          */
  KLT_FLAG_PHASED = 1u << 1,  /* run the GEMM stages as three launches plus a norm launch
                                 instead of one persistent launch with device-side
                                 dependencies (same results; for comparison)            */
  KLT_FLAG_DETERMINISTIC = 1u << 2 /* combine the routed experts' outputs in a fixed order:
                                 each (token, choice) slot's weighted output is stored and
                                 the norm sums a token's topk slots in choice order, so the
                                 output is bitwise reproducible run to run (by default the
                                 routed L2 units add into an fp32 row as they finish).
                                 Costs max_tokens * topk * L * 4 bytes of workspace and
                                 that traffic per forward.  Not combinable with
                                 KLT_FLAG_PHASED (klt_create: KLT_ERR_UNSUPPORTED).       */
};

/* Layer shape.  H, L, I, Is must be multiples of 128; 1 <= topk <= min(E, 32);
 * 1 <= E <= 256; 1 <= max_tokens and max_tokens * topk <= 2^20; eps > 0. */
typedef struct klt_dims {
  int32_t H;           /* hidden width (7168): shared-expert input and tail output   */
  int32_t L;           /* latent width (3584): routed-expert input and output         */
  int32_t E;           /* routed experts                                              */
  int32_t topk;        /* experts per token                                           */
  int32_t I;           /* routed expert intermediate width                            */
  int32_t Is;          /* shared expert intermediate width                            */
  int32_t routed_fmt;  /* enum klt_routed_format                                      */
  float eps;           /* RMSNorm epsilon                                             */
  int32_t max_tokens;  /* largest M klt_forward accepts; sizes the workspace          */
} klt_dims;

/* Layer weights, all device pointers, row-major.  klt_create copies them into memory the
 * handle owns (re-laid out for the kernels); the caller's buffers are not referenced after
 * klt_create returns.
 *   FP8 routed:   w13 e4m3 [E, 2I, L]; w13_scale f32 [E, 2I/128, L/128];
 *                 w2  e4m3 [E, L, I];  w2_scale  f32 [E, L/128, I/128];
 *                 w13_global, w2_global unused (may be NULL).
 *   NVFP4 routed (KLT_FMT_NVFP4 and KLT_FMT_NVFP4_W4A4):
 *                 w13 packed e2m1 [E, 2I, L/2]; w13_scale e4m3 [E, 2I, L/16];
 *                 w13_global f32 [E]; w2 packed [E, L, I/2]; w2_scale e4m3 [E, L, I/16];
 *                 w2_global f32 [E].
 *   MXFP8 routed: w13 e4m3 [E, 2I, L]; w13_scale uint8 UE8M0 [E, 2I, L/32];
 *                 w2 e4m3 [E, L, I];  w2_scale uint8 UE8M0 [E, L, I/32];
 *                 w13_global, w2_global unused (may be NULL).
 *   Shared/dense: ws13 bf16 [2 Is, H] (gate rows first); ws2 bf16 [H, Is];
 *                 w_up bf16 [H, L]; gamma bf16 [L]. */
typedef struct klt_weights {
  const void* w13;
  const void* w13_scale;
  const float* w13_global;
  const void* w2;
  const void* w2_scale;
  const float* w2_global;
  const void* ws13;
  const void* ws2;
  const void* w_up;
  const void* gamma;
  /* Optional: the step before the tail (both or neither; NULL = klt_forward_hidden is not
   * available on the handle).  w_lat bf16 [L, H] maps the hidden state to the latent
   * input; w_gate bf16 [E, H] gives the router logits. */
  const void* w_lat;
  const void* w_gate;
} klt_weights;

/* Optional routing outputs of klt_forward (every pointer may be NULL; device memory,
 * caller owned).  Pair i = t * topk + j.  Pairs are grouped by expert, pairs of one expert
 * in ascending i; p indexes that order.
 *   ids int32 [M, topk] (descending logit, ties to the lower expert index);
 *   weights f32 [M, topk] (softmax over the selected logits);
 *   cnt int32 [E]; off int32 [E + 1] (exclusive prefix of cnt);
 *   gidx int32 [M * topk] (token of pair p); slot int32 [M * topk] (i of pair p);
 *   pos int32 [M, topk] (p of pair (t, j)). */
typedef struct klt_routing {
  int32_t* ids;
  float* weights;
  int32_t* cnt;
  int32_t* off;
  int32_t* gidx;
  int32_t* slot;
  int32_t* pos;
} klt_routing;

/* Optional stage outputs for testing and profiling (every pointer may be NULL; device
 * memory, caller owned; copied on `stream` after the stage that writes them).
 *   zq e4m3 [M, L], zs f32 [M, L/128]: quantised latent input (MXFP8 layers: zsx below;
 *     NVFP4_W4A4 layers: zq packed e2m1 [M, L/2], even column in the low nibble, and zsx);
 *   aq e4m3 [M * topk, I], as f32 [M * topk, I/128]: quantised routed SwiGLU output,
 *     rows in pair order p (MXFP8 layers: aq only; NVFP4_W4A4 layers: aq packed e2m1
 *     [M * topk, I/2] only);
 *   r f32 [M, L]: routed combine (not formed with KLT_FLAG_DETERMINISTIC, whose norm sums
 *     the per-pair outputs directly; the norm normally zeroes it for the next forward, so
 *     asking for it makes the next forward clear the buffer first); n bf16 [M, L]:
 *     RMSNorm output (gamma applied);
 *   a_s bf16 [M, Is]: shared-expert SwiGLU output;
 *   events: up to 8 cudaEvent_t handles, events[i] recorded after launch i (NULL skips);
 *   stall_after_kblocks: test hook, 0 = off; when > 0 the tile producer of the first
 *     GEMM stops feeding data after that many k-blocks, so its consumers' bounded waits
 *     run out and klt_status reports KLT_ERR_DEVICE_TIMEOUT;
 *   timeout_ms: bound of every on-device wait for this call (0 = the default, 1000 ms);
 *   trace: optional device int64 buffer of 3 * trace_entries * 4 * (SM count) entries; when
 *     set, each GEMM launch g (0..2) records globaltimer stamps (ns) per CTA c and role r
 *     (0 = weight tile copy issued, 1 = work unit published to the MMA issuer and epilogue,
 *     2 = epilogue step done, 3 = task index + 1 of that unit, not a time) at
 *     trace[((g * SMs + c) * 4 + r) * trace_entries + i], first trace_entries
 *     events each; unused entries are left untouched;
 *   force_bn: GEMM engine and token-tile width for this call, for tuning sweeps:
 *     16, 32, 64 or 128 = feature-major engine (128 weight rows x force_bn tokens per
 *     MMA); 256 = token-major engine (128 tokens x 256 features per MMA; needs H and L
 *     multiples of 256 and the fused schedule, else KLT_ERR_UNSUPPORTED); 0 = chosen
 *     from M (feature-major with 16-token tiles up to 16 tokens, token-major above when
 *     available). */
typedef struct klt_debug {
  uint8_t* zq;
  float* zs;
  uint8_t* aq;
  float* as;
  float* r;
  void* n;
  void* a_s;
  void* events[8];
  int32_t stall_after_kblocks;
  int32_t timeout_ms;
  int64_t* trace;
  int32_t trace_entries;
  int32_t force_bn;
  /* klt_forward_hidden only: the latent input bf16 [M, L] and router logits f32 [M, E]
   * it computed from the hidden state */
  void* z;
  float* logits;
  /* MXFP8 layers: the latent input's UE8M0 scale bytes uint8 [M, L/32]; NVFP4_W4A4
   * layers: its e4m3 scale bytes uint8 [M, L/16] (zs is not formed in either) */
  uint8_t* zsx;
} klt_debug;

typedef struct klt_handle klt_handle;

/* Create a tail for one layer on the current device.
 * Defined by: DeepGEMM PR 416 "Fuse and publish Kimi K3's BF16 shared expert", Summary
 * (routed FP8/FP4 experts scheduled with a BF16 shared expert's L1/L2), and the vLLM pull
 * request "Fuse BF16 shared experts into latent MegaMoE tail", Summary (the routed result's
 * RMSNorm and 3584 -> 7168 up-projection before the two branches are added); the weight
 * formats are the readings of those pages' "FP8/FP4" listed with klt_weights.
 * Synchronous.  Copies and re-lays out
 * the weights, allocates the workspace for `d->max_tokens` tokens and encodes the TMA
 * descriptors.  Errors: KLT_ERR_INVALID_ARG (null d/w/out or a null weight pointer),
 * KLT_ERR_UNSUPPORTED (shape rules above; device is not compute capability 10.3),
 * KLT_ERR_ALIGN, KLT_ERR_OOM, KLT_ERR_CUDA.  On error *out is left NULL. */
int klt_create(const klt_dims* d, const klt_weights* w, uint32_t flags, klt_handle** out);

/* Run the tail for M tokens, asynchronously on `stream`.
 * Defined by: the vLLM pull request "Fuse BF16 shared experts into latent MegaMoE tail",
 * Summary (route, routed experts in the 3584-wide latent space, routed RMSNorm, 3584 -> 7168
 * up-projection, shared-expert output added in FP32, BF16 result) and tokenspeed PR 1062
 * "MNNVL CuTe-DSL finalize tail", commit notes (top-k weighted combine as the finalize step;
 * fp32-internal norm, one rounding).
 *   x      device bf16 [M, H]  hidden state (shared-expert input);
 *   z      device bf16 [M, L]  latent state (routed-expert input);
 *   logits device f32  [M, E]  router logits (finite values);
 *   out    device bf16 [M, H]  result.
 * M == 0 launches nothing and returns KLT_OK.  The handle's workspace is reused by every
 * call, so calls on one handle must be ordered on one stream (or synchronised).
 * Errors: KLT_ERR_INVALID_ARG (null handle or pointer, M < 0, M > max_tokens),
 * KLT_ERR_ALIGN, KLT_ERR_CUDA (a launch failed).  Device-side faults of bounded waits are
 * reported later by klt_status. */
int klt_forward(klt_handle* h, const void* x, const void* z, const float* logits, int32_t M,
                void* out, klt_routing* routing_out, klt_debug* dbg, void* stream);

/* Run the step before the tail and then the tail for M tokens, from the hidden state alone,
 * asynchronously on `stream`.
 * Defined by: tokenspeed PR 1062 "MNNVL CuTe-DSL finalize tail", commit notes (the model's
 * latent input projections feeding the latent MoE).  Computes, on the GPU,
 *   z      = bf16( x W_lat^T )     bf16 [M, L]  (fp32 accumulation, one rounding)
 *   logits = x W_gate^T            f32  [M, E]
 * into the handle's workspace and then runs exactly what klt_forward runs on them.
 *   x   device bf16 [M, H];  out device bf16 [M, H].
 * Launches one kernel more than klt_forward (the projection, first).  The handle must have
 * been created with w_lat and w_gate.  Errors: as klt_forward, and KLT_ERR_UNSUPPORTED
 * when the handle has no projection weights. */
int klt_forward_hidden(klt_handle* h, const void* x, int32_t M, void* out,
                       klt_routing* routing_out, klt_debug* dbg, void* stream);

/* Sticky device status of the handle: KLT_OK or KLT_ERR_DEVICE_TIMEOUT.  Reads device
 * memory synchronously, so call it after the forward's stream has been synchronised.  A
 * handle that reported a device error must be destroyed. */
int klt_status(klt_handle* h);

/* Free everything the handle owns (synchronises the device first).  NULL is a no-op. */
int klt_destroy(klt_handle* h);

/* Static description of a status code. */
const char* klt_strerror(int code);

/* Number of kernels one klt_forward launches for the given M and handle at the automatic
 * GEMM configuration (0 for M == 0): the routing launches (one for a feature-major batch of
 * at most 256 (token, choice) pairs with e4m3 activations; otherwise routing, an expert
 * histogram above 1024 pairs, scatter and gather) and then the GEMM launches (one; two for
 * the block-scaled formats; four with KLT_FLAG_PHASED). */
int klt_launch_count(const klt_handle* h, int32_t M);

/* GEMM configuration klt_forward uses for M tokens when klt_debug.force_bn = force_bn
 * (0 = automatic): 16, 32, 64 or 128 = the feature-major engine with that token tile,
 * 256 = the token-major engine (128-token x 256-feature units).  A negative value is the
 * negated status klt_forward would return: -KLT_ERR_UNSUPPORTED when force_bn = 256 is not
 * available for this handle, -KLT_ERR_INVALID_ARG for a NULL handle. */
int klt_gemm_tile(const klt_handle* h, int32_t M, int32_t force_bn);

/* Largest M * topk klt_route_noalloc accepts (its fixed scratch size, about 320 KB). */
#define KLT_NOALLOC_MAX_PAIRS 65536

/* Routing and expert permutation without a handle and without any device allocation.
 * The pages describe no such entry point; it exists for callers that cannot allocate
 * device memory where they route (inside another framework's memory pool, serving loops
 * that fix every allocation at start-up, runtimes without allocator access).
 * Computes the same ids, weights, cnt, off, gidx, slot and pos as klt_forward's routing
 * outputs (same layouts as klt_routing) for `logits` f32 [M, E], all pointers device
 * memory, caller owned, 16-byte aligned, none NULL.  Internal buffers live in one
 * fixed-size device array (KLT_NOALLOC_MAX_PAIRS pairs) that every GPU loading the library
 * holds until exit; calls share it, so calls whose kernels overlap on the GPU race; order
 * them on one stream.  The first call on a device resolves the array's device address
 * and caches it for the life of the process; make that first call before any stream
 * capture.  A device reset (cudaDeviceReset) after that first call is not supported: the
 * library may then load the array at another address while the cache keeps the old one.
 * Asynchronous on `stream`.
 * Errors: KLT_ERR_INVALID_ARG (M < 0, E or topk < 1, NULL pointer), KLT_ERR_UNSUPPORTED
 * (E > 256, topk > E, topk > 32), KLT_ERR_TOO_LARGE (M * topk > KLT_NOALLOC_MAX_PAIRS),
 * KLT_ERR_ALIGN, KLT_ERR_CUDA.  M == 0 launches nothing. */
int klt_route_noalloc(const float* logits, int32_t M, int32_t E, int32_t topk, int32_t* ids,
                      float* weights, int32_t* cnt, int32_t* off, int32_t* gidx,
                      int32_t* slot, int32_t* pos, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KLT_H_ */
