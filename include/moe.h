/* moe.h -- C ABI of libmoe.so, the GB300 (sm_103a) MoE expert layer.
 *
 * The layer (source: "Perplexity open-sources Lily, a Rust + Metal inference
 * engine for Qwen3.6-35B-A3B on Apple Silicon"):
 *   - "three workload shapes": a router scores 256 experts per token and picks
 *     8; a shared expert processes every token;
 *   - "Prefill": weights are groupwise-affine 4-bit, 64 weights sharing one
 *     bf16 scale and one bf16 bias; they are rebuilt to bf16 tile by tile
 *     inside the grouped GEMM with FP32 accumulation, so no unpacked weight
 *     array reaches memory; routing (histogram, prefix scan, scatter, block
 *     map) stays on the GPU with no CPU sync inside the layer;
 *   - "Decode": one token at a time reuses next to none of the weights it
 *     reads, so HBM bandwidth sets the limit; only the selected experts'
 *     bytes are streamed.
 *
 * Arithmetic (where the pages are silent, the plainest reading):
 *   w      = bf16_rne(scale * q + bias), q = (word[k/8] >> 4*(k%8)) & 15
 *   key    = fp32(x . router_row) (+ logit_bias[e] in fp32)
 *   top-k  = k largest keys, ties to the lower expert index, NaN lowest;
 *            weights = softmax over the k picked keys (slot order = rank)
 *   h      = bf16(silu(x.Wg^T) * (x.Wu^T)),  y = bf16(h.Wd^T)   (fp32 sums)
 *   out    = bf16(residual + y_shared + sum_j w_j * y_j)         (fp32 sum)
 *
 * Conventions for every entry point:
 *   - Pointers named *_d are DEVICE pointers; every other pointer is host.
 *   - bf16 tensors are passed as raw 16-bit patterns (uint16_t / void*).
 *   - Every device pointer must be 16-byte aligned (MOE_ERR_MISALIGNED).
 *   - Argument checks run on the host before anything is enqueued; on any
 *     error nothing is enqueued.  Launch failures return MOE_ERR_CUDA.
 *   - No entry point allocates device memory, synchronises, or reads device
 *     memory on the host, except moe_device_status (documented below).  The
 *     caller owns every device buffer, including the workspace.
 *   - A workspace may serve one call at a time; concurrent calls on different
 *     streams need different workspaces.  A plan is immutable after creation
 *     and may be shared across threads and streams.
 */
#ifndef MOE_H
#define MOE_H
#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARGUMENT = 1,   /* null pointer, bad size, bad flag        */
  MOE_ERR_UNSUPPORTED = 2,        /* dims outside the supported set          */
  MOE_ERR_MISALIGNED = 3,         /* a device pointer not 16-byte aligned    */
  MOE_ERR_WORKSPACE_TOO_SMALL = 4,
  MOE_ERR_TOO_MANY_TOKENS = 5,    /* T > max_tokens: the caller chunks       */
  MOE_ERR_CUDA = 6,               /* a CUDA call or launch failed            */
  MOE_ERR_DEVICE_TIMEOUT = 7,     /* device status: a bounded wait gave up   */
  MOE_ERR_NONFINITE = 8,          /* device status: NaN/Inf router key       */
  MOE_ERR_DEVICE_BOUNDS = 9       /* device status: debug bounds check hit   */
} moe_status;

/* Layer dimensions.  Supported: hidden % 128 == 0, inter % 64 == 0,
 * group_size == 64, 1 <= top_k <= min(16, n_experts), n_experts <= 1024,
 * n_shared in {0, 1}.  The pages' model: {2048, 256, 8, 512, 1, 64}. */
typedef struct {
  int32_t hidden;      /* H */
  int32_t n_experts;   /* E routed experts */
  int32_t top_k;       /* k */
  int32_t inter;       /* I, expert intermediate size */
  int32_t n_shared;    /* S, 0 or 1; the shared expert is stored at index E */
  int32_t group_size;  /* G = 64 */
} moe_config;

/* Packed expert weights, device pointers, experts stacked 0..E+S-1:
 *   gate_q, up_q   uint32 [E+S][I][H/8]   8 codes per word, code k at bits 4*(k%8)
 *   gate_s, gate_b, up_s, up_b  bf16 [E+S][I][H/G]  scale and bias per group
 *   down_q         uint32 [E+S][H][I/8]
 *   down_s, down_b bf16   [E+S][H][I/G]
 *   router         fp32   [E][H]
 *   shared_gate    fp32   [H], or NULL
 * Rows are output features; groups run along the input (K) dimension.  The
 * library only reads these buffers.
 * shared_gate (optional, a variant the pages do not print): the shared
 * expert's output is scaled by g = sigmoid(x . shared_gate) per token, x the
 * layer's expert input (after the pre-norm of stacked layers), the dot
 * product in fp32: out = bf16(res + g * y_shared + sum_j w_j y_j).  NULL: g = 1.
 * router_split_d (optional): the router as three bf16 parts, [3][E][H]
 * (hi, mid, lo; moe_router_split writes them once per set of weights).  The
 * tensor-core router (T >= 32) reads them instead of splitting router_d on
 * every call; the keys are the same bit for bit.  NULL: split per call. */
typedef struct {
  const float *router_d;
  const uint32_t *gate_q_d, *up_q_d;
  const uint16_t *gate_s_d, *gate_b_d, *up_s_d, *up_b_d;
  const uint32_t *down_q_d;
  const uint16_t *down_s_d, *down_b_d;
  const float *shared_gate_d;
  const uint16_t *router_split_d;
} moe_weights;

/* Device pointers into a workspace, for tests and tools (moe_route_view). */
typedef struct {
  float *keys_d;       /* [T][E] fp32 selection keys (logits + bias)         */
  int32_t *topk_id_d;  /* [T][k] picked experts in slot (rank) order          */
  float *topk_w_d;     /* [T][k] softmax weights over the picked keys         */
  int32_t *counts_d;   /* [E] pairs per expert (histogram)                    */
  int32_t *offsets_d;  /* [E+1] exclusive scan of counts, offsets[E] = k*T    */
  int32_t *perm_d;     /* [k*T] pair id t*k+j, experts in index order, tokens ascending */
  int32_t *inv_d;      /* [k*T] position of pair t*k+j in perm                */
  int32_t *blockmap_d; /* [max_tiles][4] (expert, first row, rows, 0)         */
  int32_t *n_tiles_d;  /* [1] entries in use                                 */
  uint16_t *h_d;       /* [(k+S)*T][I] bf16 SwiGLU rows (routed in perm order, then shared);
                          tensor-core plans store each run of 8 columns as 0,4,1,5,2,6,3,7 */
  uint16_t *y_d;       /* [(k+S)*T][H] bf16 expert outputs, same row order    */
  int32_t *status_d;   /* [1] sticky device status (moe_status values)        */
  uint64_t *trace_d;   /* [MOE_TRACE_CTAS][MOE_TRACE_SLOTS] phase timestamps (ns), MOE_FLAG_TRACE */
  int32_t max_tiles;   /* capacity of blockmap_d                             */
  int32_t block_rows;  /* rows per block-map tile for this plan              */
  int32_t *blockmap2_d; /* [max_tiles2][4] the same map with tiles of block_rows2 rows
                           (tensor-core plans: the down GEMM's tiles); unused otherwise */
  int32_t *n_tiles2_d;  /* [1] entries in use in blockmap2_d                 */
  int32_t max_tiles2;   /* capacity of blockmap2_d (0: no second map)         */
  int32_t block_rows2;  /* rows per tile of blockmap2_d                       */
} moe_route_ptrs;

/* Plan flags. */
#define MOE_FLAG_DEBUG_CHECKS   0x1u  /* device bounds checks -> MOE_ERR_DEVICE_BOUNDS in the status */
#define MOE_FLAG_FORCE_GROUPED  0x2u  /* T == 1 runs the grouped path instead of the decode path */
#define MOE_FLAG_SIMT_EXPERTS   0x4u  /* CUDA-core grouped GEMMs instead of the tensor-core ones */
#define MOE_FLAG_TILE_ROWS_64   0x8u  /* tensor-core path: 64-token tiles instead of 128 */
#define MOE_FLAG_TRACE          0x20u /* tracing aid, into moe_route_ptrs.trace_d, per CTA:
                                         decode kernel: %globaltimer at each phase of the last layer
                                         of a launch; grouped tensor-core GEMMs: clock64 cycles each
                                         role spent waiting on its barriers and in total (gate/up in
                                         slots 0-12, down in slots 16-28) */
#define MOE_TRACE_CTAS 256             /* CTAs with a row in the trace buffer */
#define MOE_TRACE_SLOTS 32             /* timestamps in a row */
#define MOE_FLAG_PRENORM        0x10u /* pre-norm block: x_d is the residual stream r, the layer
                                         computes x = RMSNorm(r) (unit gain, eps 1e-6) and
                                         out = r + MoE(x); residual_d must be NULL and out_d
                                         may alias x_d (in-place residual update) */
#define MOE_FLAG_TEST_WITHHOLD  0x40u /* test aid for the failure path of the T == 1 decode kernel:
                                         the CTA that computes expert 0's router key never
                                         publishes it, and every wait of the decode kernel gives
                                         up after 1 ms instead of 1 s, so the other CTAs' bounded
                                         waits run out, MOE_ERR_DEVICE_TIMEOUT lands in the status
                                         word and the kernel returns (its copies drained).  The
                                         workspace then needs moe_workspace_init.  Other paths
                                         are unaffected. */

typedef struct moe_plan moe_plan_t;

/* Validate dims and build a host-only plan for up to max_tokens tokens per
 * call (1 <= max_tokens <= 65536).  *out owns host memory only; free it with
 * moe_plan_destroy.  Errors: MOE_ERR_INVALID_ARGUMENT (null pointers, bad
 * max_tokens or unknown flags), MOE_ERR_UNSUPPORTED (dims), MOE_ERR_CUDA (no
 * device or not sm_103). */
moe_status moe_plan(const moe_config *cfg, int32_t max_tokens, uint32_t flags, moe_plan_t **out);
void moe_plan_destroy(moe_plan_t *plan);

/* Bytes of device workspace a call of this plan needs (0 for a null plan). */
size_t moe_workspace_bytes(const moe_plan_t *plan);

/* Zero the workspace's status word, counters and the decode kernel's tagged
 * exchange words (enqueued on stream).  Call once after allocating a
 * workspace, and again after a call has left an error in the device status
 * (a decode launch cut short by a timeout can leave words that a later launch
 * would take for its own).  A workspace serves one stream at a time. */
moe_status moe_workspace_init(const moe_plan_t *plan, void *ws_d, size_t ws_bytes, void *stream);

/* Routing only ("Prefill": histogram, prefix scan, scatter, block map, all on
 * the GPU).  x_d: bf16 [T][H]; router_d: fp32 [E][H]; logit_bias_d: fp32 [E]
 * or NULL.  Writes keys, top-k ids and weights, counts, offsets, perm, inv
 * and the block map into ws (see moe_route_view).  1 <= T <= max_tokens. */
moe_status moe_route(const moe_plan_t *plan, const void *x_d, int32_t T, const float *router_d,
                     const float *logit_bias_d, void *ws_d, size_t ws_bytes, void *stream);

/* Routing from given selection keys (test hook: lets the oracle and the GPU
 * select from identical fp32 keys).  keys_d: fp32 [T][E]; it is copied into
 * the workspace's key buffer first. */
moe_status moe_route_from_logits(const moe_plan_t *plan, const float *keys_d, int32_t T, void *ws_d,
                                 size_t ws_bytes, void *stream);

/* Routing from given expert choices (test hook and teacher-forced routing):
 * ids_d int32 [T][k] (distinct experts per token, in slot order) and w_d fp32
 * [T][k] are copied into the workspace's top-k buffers, then the histogram,
 * scan, scatter and block maps run as in moe_route (the key buffer is left
 * as it was).  An id outside [0, E) is not counted and sets
 * MOE_ERR_DEVICE_BOUNDS in the device status; with MOE_FLAG_DEBUG_CHECKS a
 * token that names one expert twice does too (the scatter then finds fewer
 * pairs than the histogram counted).  After such a status the routing
 * buffers hold no valid routing. */
moe_status moe_route_from_ids(const moe_plan_t *plan, const int32_t *ids_d, const float *w_d, int32_t T, void *ws_d,
                              size_t ws_bytes, void *stream);

/* The whole layer: routing, shared + routed SwiGLU experts over the packed
 * weights, and the weighted combine with the residual.
 *   x_d        bf16 [T][H] layer input (read only), or with MOE_FLAG_PRENORM
 *              the residual stream r (the layer normalises it itself)
 *   residual_d bf16 [T][H] or NULL (NULL: the residual is x); NULL with PRENORM
 *   out_d      bf16 [T][H]; may alias residual_d; may alias x_d only with PRENORM
 * T == 1 takes the bandwidth-bound decode path (one cooperative launch per
 * layer, "Decode" section) unless the plan has MOE_FLAG_FORCE_GROUPED.  Never
 * allocates or synchronises, so the call can be captured into a CUDA graph. */
moe_status moe_forward(const moe_plan_t *plan, const void *x_d, const void *residual_d, int32_t T,
                       const moe_weights *w, const float *logit_bias_d, void *out_d, void *ws_d,
                       size_t ws_bytes, void *stream);

/* Single-token decode through a stack of n_layers pre-norm MoE layers (the
 * pages' model stacks 40 of them; "Decode" section: at batch 1 bandwidth
 * bounds the step):  for l = 0 .. n_layers-1,  r = r + MoE_l(RMSNorm(r)),
 * each layer routed on its own fp32 keys, RMSNorm as in moe_rmsnorm.  The same
 * arithmetic as n_layers moe_forward calls of a MOE_FLAG_PRENORM plan at
 * T == 1, run as ceil(n_layers / 7) cooperative launches that fetch each
 * layer's router and shared-expert weights during the previous layer.
 *   r_d           bf16 [H] residual stream, updated in place (device)
 *   w             host array of n_layers moe_weights (device pointers)
 *   logit_bias_d  host array of n_layers device pointers (entries may be
 *                 NULL), or NULL
 * The workspace keeps the last layer's keys and top-k.  Errors: as
 * moe_forward; MOE_ERR_UNSUPPORTED when the plan's shape has no decode path. */
moe_status moe_decode_stack(const moe_plan_t *plan, void *r_d, int32_t n_layers, const moe_weights *w,
                            const float *const *logit_bias_d, void *ws_d, size_t ws_bytes, void *stream);

/* A long prompt through a stack of n_layers pre-norm MoE layers in bounded
 * chunks ("Prefill" section: long prompts are processed in chunks of bounded
 * size, so temporary activations stay small next to the resident weights):
 *   for c0 = 0, m, 2m, ... (m = the plan's max_tokens):
 *     rows c0 .. c0 + n - 1 of r (n = min(m, T - c0)), for l = 0 .. n_layers-1:
 *       r_c = r_c + MoE_l(RMSNorm(r_c))
 * chunk-major (each chunk passes through every layer before the next chunk
 * starts), every call on the one workspace.  The same results, bit for bit,
 * as the moe_forward calls of that loop (a one-token tail chunk takes the
 * decode path); on the grouped path each layer's combine also writes the
 * next layer's RMSNorm, with the norm step's arithmetic, so that step is not
 * launched again.  The plan must have MOE_FLAG_PRENORM.
 *   r_d           bf16 [T][H] residual stream, updated in place (device)
 *   T             1 <= T (no upper bound beyond the caller's buffer)
 *   w             host array of n_layers moe_weights (device pointers)
 *   logit_bias_d  host array of n_layers device pointers (entries may be
 *                 NULL), or NULL
 * Errors: as moe_forward (nothing is enqueued when an argument check fails;
 * a launch failure part-way returns MOE_ERR_CUDA with the earlier calls
 * enqueued). */
moe_status moe_prefill_stack(const moe_plan_t *plan, void *r_d, int32_t T, int32_t n_layers, const moe_weights *w,
                             const float *const *logit_bias_d, void *ws_d, size_t ws_bytes, void *stream);

/* The router's three bf16 parts, for moe_weights.router_split_d (the
 * tensor-core router's operand): split_d[p][e][h], p = 0, 1, 2, with
 * hi = bf16(w), mid = bf16(w - hi), lo = bf16(w - hi - mid) (round to
 * nearest even, each difference exact in fp32).  router_d fp32 [E][H];
 * split_d bf16 [3][E][H] (moe_router_split_bytes(E, H) bytes, caller-owned).
 * Enqueued on stream; run it once per set of router weights and pass split_d
 * as moe_weights.router_split_d.  E * H must be a multiple of 4. */
size_t moe_router_split_bytes(int32_t E, int32_t H);
moe_status moe_router_split(const float *router_d, int32_t E, int32_t H, void *split_d, size_t split_bytes,
                            void *stream);

/* Device pointers of the workspace's routing buffers for T tokens (host-side
 * arithmetic only; nothing is read or enqueued). */
moe_status moe_route_view(const moe_plan_t *plan, void *ws_d, int32_t T, moe_route_ptrs *out);

/* Unit-gain RMSNorm used between stacked layers (the pages' model is a stack
 * of 40 such layers; the norm is not printed there):
 *   x = bf16(r / sqrt(mean(r^2) + eps)), fp32 arithmetic.
 * r_d, x_d: bf16 [T][H]; H % 8 == 0; r_d may not alias x_d. */
moe_status moe_rmsnorm(const void *r_d, int32_t T, int32_t H, float eps, void *x_d, void *stream);

/* Dequantise one packed matrix to bf16 (test hook for the rebuild step of
 * "Prefill"):  w_d[n][k] = bf16_rne(s[n][k/G] * q + b[n][k/G]).
 * q_d: uint32 [rows][K/8]; s_d, b_d: bf16 [rows][K/G]; w_d: bf16 [rows][K]. */
moe_status moe_dequant(const uint32_t *q_d, const uint16_t *s_d, const uint16_t *b_d, int32_t rows,
                       int32_t K, int32_t G, void *w_d, void *stream);

/* Synchronises the stream, reads the workspace's sticky status word into
 * *host_status, and (if reset != 0) zeroes it.  The only entry point that
 * synchronises. */
moe_status moe_device_status(const moe_plan_t *plan, void *ws_d, void *stream, int32_t *host_status,
                             int32_t reset);

/* Number of kernel launches the last moe_forward/moe_route call on this
 * thread enqueued (for launch accounting in benchmarks). */
int32_t moe_last_launch_count(void);

/* Kernels of the library, for moe_profile_events. */
typedef enum {
  MOE_KERNEL_ROUTER = 1,         /* router keys, T > 1                        */
  MOE_KERNEL_TOPK = 2,           /* top-k + histogram                          */
  MOE_KERNEL_SCATTER = 3,        /* scan + stable scatter + block map          */
  MOE_KERNEL_GATEUP = 4,         /* grouped gate/up dequant-GEMM + SwiGLU      */
  MOE_KERNEL_DOWN = 5,           /* grouped down dequant-GEMM                  */
  MOE_KERNEL_COMBINE = 6,        /* weighted gather-combine + residual         */
  MOE_KERNEL_DECODE_LAYER = 7,   /* T == 1: the whole layer in one launch      */
  MOE_KERNEL_RMSNORM = 10,
  MOE_KERNEL_GATHER = 11,        /* routed x rows copied into perm order (tensor-core path) */
  MOE_KERNEL_GDN_SCAN = 12,      /* Gated DeltaNet scan (gdn.h)                */
  MOE_KERNEL_ATTN_DECODE = 13    /* decode attention, per-block pass (attn.h)  */
} moe_kernel;

/* Profiling hook (one per kernel).  From now on, on the calling thread, the
 * i-th launch of `kernel` is bracketed by cudaEventRecord(start_events[i % n]) and
 * cudaEventRecord(stop_events[i % n]) on that launch's stream (also inside a
 * stream capture, where the records become graph nodes).  start_events and
 * stop_events are host arrays of n cudaEvent_t handles, copied by the call;
 * the caller owns the events.  n == 0 (arrays may be NULL) turns the hook off.
 * Errors: MOE_ERR_INVALID_ARGUMENT for an unknown kernel, n < 0, n > 4096,
 * null arrays with n > 0, or a null event handle. */
moe_status moe_profile_events(int32_t kernel, void *const *start_events, void *const *stop_events, int32_t n);

/* Thin the hook of `kernel` out (after moe_profile_events turned it on):
 * only launches 0, stride, 2*stride, ... of the kernel, counted from this
 * call, are bracketed (the j-th of them by event j % n).  Errors:
 * MOE_ERR_INVALID_ARGUMENT for an unknown kernel, stride < 1 or a kernel
 * whose hook is off. */
moe_status moe_profile_stride(int32_t kernel, int32_t stride);

/* Allocation-free single-token layer.  The paper has no counterpart to this
 * entry point: it serves callers that cannot call cudaMalloc -- code running
 * inside another runtime that owns all of the device's memory (a serving
 * engine or framework whose allocator has reserved it, or a process held to
 * a fixed memory cap), and code that must not risk the implicit device-wide
 * synchronisation an allocation can bring.  It computes what moe_forward
 * computes for T == 1 on its decode path (one cooperative launch), with the
 * scratch that path keeps in the workspace -- router keys, top-k ids and
 * weights, the decode epoch counter, the tagged words the kernel's CTAs
 * exchange (keys, h, residual) and the status word -- held instead in one
 * static device array of
 * MOE_DECODE_STATIC_SCRATCH_BYTES that every device loading the library keeps
 * until the process exits.  It needs no plan and calls no cudaMalloc,
 * cudaFree or allocating library routine.
 *   cfg          the layer's dimensions (checked as moe_plan checks them)
 *   x_d          bf16 [H] input token, or with MOE_FLAG_PRENORM the residual
 *                stream r (the call normalises it itself)
 *   residual_d   bf16 [H] or NULL (NULL: the residual is x); NULL with PRENORM
 *   w            packed weights, as for moe_forward; logit_bias_d fp32 [E] or NULL
 *   out_d        bf16 [H]; may alias residual_d; may alias x_d only with PRENORM
 *   status_d     device int32 or NULL: zeroed, then set to a moe_status code if
 *                the kernel meets a device-side error (NULL: not reported)
 *   flags        0 or MOE_FLAG_PRENORM
 * The first call on a device (with that device current) resolves the array's
 * address with cudaGetSymbolAddress and raises the decode kernel's
 * shared-memory limit; make that first call before any stream capture.
 * Every call clears the status word on the stream before its launch, and
 * the tagged words too when the dimensions differ from the previous call's;
 * the epoch counter carries over, and keys and top-k are rewritten, so the
 * array otherwise keeps the previous call's contents.  All calls on a device
 * share the one array: calls that can overlap on the GPU (other streams,
 * other threads) race and must be serialised by the caller.
 * Errors: MOE_ERR_WORKSPACE_TOO_SMALL when the layer's scratch exceeds the
 * array.  The scratch is 256 bytes of status and counter, then
 * 8 * (2 W + (k + n_shared) I + H) bytes of tagged words with
 * W = round_up(E + 1, 16), then 4E bytes of keys, 4k of top-k ids and 4k of
 * weights, each part starting on a 256-byte boundary: 59,168 bytes for
 * H=2048, E=256, k=8, n_shared=1, I=512 (6,368 bytes below the limit);
 * MOE_ERR_UNSUPPORTED for dimensions the decode path does not take
 * (H and I powers of two, the kernel's shared memory within the device's
 * limit); MOE_ERR_INVALID_ARGUMENT / MOE_ERR_MISALIGNED as for moe_forward;
 * MOE_ERR_CUDA when a CUDA call fails (moe_last_cuda_error). */
#define MOE_DECODE_STATIC_SCRATCH_BYTES 65536
moe_status moe_decode_static(const moe_config *cfg, const void *x_d, const void *residual_d,
                             const moe_weights *w, const float *logit_bias_d, void *out_d, int32_t *status_d,
                             uint32_t flags, void *stream);

const char *moe_status_str(moe_status s);

/* Text of the CUDA error behind the last MOE_ERR_CUDA returned on the
 * calling thread ("no error" if there was none). */
const char *moe_last_cuda_error(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H */
