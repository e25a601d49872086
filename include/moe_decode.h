/*
 * moe_decode.h — C ABI of the GB300 (sm_103a) MoE decode-layer library.
 *
 * The library computes the memory-bound decode step of a large MoE
 * transformer at batch M = 1..64 on one GPU: weight-streaming projections
 * chosen by batch size, the out-projection fused with its residual, sigmoid
 * router scoring with top-k, and the routed and shared SwiGLU experts.
 * Sources (the vLLM "Kimi K3" decode article and its summaries):
 *   [K3 P1§1] Part 1 §1 "Ajustar las formas": small-matrix kernels at batch
 *             1-2, split-K kernels at larger batch, for the projections.
 *   [K3 P1§2] Part 1 §2 "Superposición de computación y comunicación": the
 *             attention out-projection fused with the residual after it.
 *   [K3 P1§3] Part 1 §3 "Mejorar la programación de MoE": router scores,
 *             routed experts, the shared expert on a separate stream.
 *   [K3 P1§4] Part 1 §4 "Prefetching": small-batch decode is bound by weight
 *             reads; a side-stream kernel warms the cache with the next
 *             operator's weights during phases that leave bandwidth idle.
 *   [hu-sum]  aihirek.info summary, "Kevesebb kernel, összehangoltabb
 *             végrehajtás": the same kernel choice by batch size.
 *
 * Conventions (all entry points):
 *  - Tensors are caller-owned DEVICE memory, row-major. Weights use the
 *    nn.Linear layout W[N][K] (K contiguous), so y = x W^T. bf16 values are
 *    passed as their 16-bit patterns (dec_bf16). Every pointer must be
 *    16-byte aligned and every K (inner extent) a multiple of 8.
 *  - Calls are asynchronous on the given stream and never allocate device
 *    memory. Scratch space is the caller's workspace `ws` of `ws_bytes`
 *    bytes, sized by the matching *_workspace_size() query. A workspace must
 *    be zeroed (dec_workspace_init) before its first use and before it is
 *    reused by a call of another entry point or another shape; calls of the
 *    same entry point and shape leave it ready for the next one. One
 *    workspace must not be used by two calls that can run at the same time.
 *  - Arguments are checked on the host before anything is launched; a bad
 *    argument returns DEC_ERR_INVALID_ARG or DEC_ERR_UNSUPPORTED and launches
 *    nothing. A failed launch returns DEC_ERR_CUDA. No call aborts, exits or
 *    traps. Device waits are bounded: a wait that runs past the handle's
 *    limit makes its kernel stop early and sets the handle's device error
 *    word, which dec_check_device_error() reports as DEC_ERR_TIMEOUT.
 *  - Accumulation is fp32 everywhere; each bf16 output is rounded once.
 *  - A handle serves one thread at a time (it holds the side streams,
 *    events and the last-variant record).
 */
#ifndef MOE_DECODE_H
#define MOE_DECODE_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t dec_bf16; /* bit pattern of a bfloat16 value */

typedef enum dec_status {
  DEC_OK = 0,
  DEC_ERR_INVALID_ARG = 1, /* null or misaligned pointer, size out of range, workspace too small */
  DEC_ERR_UNSUPPORTED = 2, /* well-formed request outside the implemented shapes */
  DEC_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed */
  DEC_ERR_TIMEOUT = 4      /* a device wait ran past its limit (see dec_check_device_error) */
} dec_status;

/* Kernel families of the projections [K3 P1§1]. */
typedef enum dec_variant {
  DEC_VARIANT_AUTO = 0,    /* choose by batch and size (measured on GB300): SMALL_M for M <= 2, and for
                              M <= 4 when the weight matrix is at most 48 MB; SPLIT_K otherwise */
  DEC_VARIANT_SMALL_M = 1, /* CUDA-core small-matrix kernel: each CTA streams whole weight rows */
  DEC_VARIANT_SPLIT_K = 2  /* tcgen05 kernel; the weight k-blocks are split evenly over all SMs */
} dec_variant;

typedef struct dec_handle dec_handle;

/* ------------------------------------------------------------------ handle */

/* Create a handle on CUDA device `device`. The handle owns two side streams
 * (shared expert, L2 prefetch), their fork/join events and a 4-byte device
 * error word; nothing else. Returns DEC_ERR_CUDA if the device is absent. */
dec_status dec_create(dec_handle** out, int device);

/* Destroy a handle (synchronises its side streams first). NULL is allowed. */
dec_status dec_destroy(dec_handle* h);

/* Static description of a status code. Never NULL. */
const char* dec_status_string(dec_status s);

/* Zero a workspace before its first use (cudaMemsetAsync on `stream`). */
dec_status dec_workspace_init(dec_handle* h, void* ws, size_t ws_bytes, cudaStream_t stream);

/* Limit, in nanoseconds, of every device-side wait (default 500 ms). */
dec_status dec_set_wait_limit_ns(dec_handle* h, uint64_t ns);

/* Enable (1, default) or disable (0) programmatic dependent launch: kernels
 * start while their predecessor drains and stream static weights before
 * waiting for it [K3 Part 2, "Validar la corrección": activation reads stay
 * behind the dependency wait, weight reads may go before it]. */
dec_status dec_set_pdl(dec_handle* h, int enable);

/* How the shared expert and the routed experts share the SMs [K3 P1§3: the
 * schedule sets how many GPU resources each operation uses]. The shared
 * expert is always launched first, beside the router / top-k phase.
 *  0 (default): it keeps its share of the expected weight bytes (rounded
 *     up), except from four tokens on with a shared expert of at least 48 MB,
 *     where it acts as -1 (measured on GB300: as fast with independent
 *     tokens, up to 17% faster when tokens share experts, as the drafts of a
 *     speculative-verify batch do; with a small shared expert the byte share
 *     is faster);
 * -1: it starts on every SM and the routed experts take SMs as it finishes;
 *  n > 0: it keeps n SMs. */
dec_status dec_set_shared_sms(dec_handle* h, int sms);

/* The small-matrix kernels (batch 1) keep about `bytes` of each CTA's
 * upcoming weight rows requested into L2 (bulk L2 prefetches, issued from
 * before the dependency wait on), beyond the rows their registers hold, so
 * that far more of the weight stream is in flight than registers allow.
 * 0 disables it; bytes in [0, 16 MiB]; default 49152 (measured on GB300:
 * 32-64 KB per CTA take the batch-1 layer step from 193 to 172 us; above
 * 128 KB the requested lines start to crowd L2). No counterpart on the pages:
 * a GB300 tuning of the small-matrix kernels [K3 P1§1]. */
dec_status dec_set_l2_ahead(dec_handle* h, int bytes);

/* Force a projection kernel family (DEC_VARIANT_AUTO restores the choice by
 * batch) so that tests can run both families at the same batch. */
dec_status dec_set_force_variant(dec_handle* h, int variant);

/* Variant used by the most recent dec_linear / dec_linear_residual call on
 * this handle (a dec_variant value; 0 before any call). */
int dec_last_variant(const dec_handle* h);

/* Kernel family of the most recent expert launches (moe_experts,
 * decode_layer): DEC_VARIANT_SMALL_M (batch 1: one token per expert) or
 * DEC_VARIANT_SPLIT_K; 0 before any call. dec_set_force_variant(SPLIT_K)
 * also forces the split-K family for the experts. */
int dec_last_expert_variant(const dec_handle* h);

/* Synchronise the device and read the device error word: DEC_OK if clear,
 * DEC_ERR_TIMEOUT if a kernel gave up a wait since the last check (the word
 * is cleared), DEC_ERR_CUDA if the device reports an error. */
dec_status dec_check_device_error(dec_handle* h);

/* ------------------------------------------------------------------ projections */

/* Workspace bytes that dec_linear / dec_linear_residual need for (M, N, K). */
dec_status dec_linear_workspace_size(const dec_handle* h, int M, int N, int K, size_t* bytes);

/* y[M][N] = x[M][K] W[N][K]^T  (bf16 in, fp32 accumulate, bf16 out).
 * [K3 P1§1], [hu-sum]: the small-matrix kernel at M <= 2 (and up to M = 4
 * for matrices of at most 48 MB, where the split-K kernel's fixed cost per
 * launch dominates), the split-K tcgen05 kernel above (or as forced with
 * dec_set_force_variant). x has row stride ldx >= K elements (ldx = K
 * for a dense matrix; a larger stride reads the leading K columns of a wider
 * activation). 1 <= M <= 64, N >= 1, 8 <= K, K % 8 == 0, ldx % 8 == 0.
 * y must not overlap x or W. */
dec_status dec_linear(dec_handle* h, const dec_bf16* x, int ldx, const dec_bf16* W, dec_bf16* y, int M, int N,
                      int K, void* ws, size_t ws_bytes, cudaStream_t stream);

/* out[M][N] = r[M][N] + x[M][K] W[N][K]^T, the out-projection fused with the
 * residual add [K3 P1§2] (the all-reduce between them has no counterpart on
 * one GPU). fp32 sum, one bf16 rounding. out may alias r exactly. Same shape
 * rules as dec_linear. */
dec_status dec_linear_residual(dec_handle* h, const dec_bf16* x, int ldx, const dec_bf16* W, const dec_bf16* r,
                               dec_bf16* out, int M, int N, int K, void* ws, size_t ws_bytes,
                               cudaStream_t stream);

/* out[M][N] = [r[M][N] +] x[M][K] W[N][K]^T with no workspace argument and
 * no device allocation, for callers that cannot provide scratch memory: for
 * example a plugin running inside a serving runtime whose memory pool owns
 * all device memory and gives plugins no allocator, or a latency-critical
 * caller that must not call cudaMalloc (which can block and synchronise the
 * device). The paper has no counterpart; this is an interface convenience.
 * It runs the split-K tcgen05 kernel of dec_linear with its scratch (10 MiB
 * of split-K partial sums and 4 KiB of tile counters) in one static device
 * array that every GPU loading the library holds until the process exits.
 * - The first call on a device looks up that array's address
 *   (cudaGetSymbolAddress, with the handle's device made current, then the
 *   caller's device restored) and keeps it for the process; make that first
 *   call before any stream capture. A device reset (cudaDeviceReset) after
 *   that first call is not supported: the kept address may no longer be the
 *   array's. A call that fails with DEC_ERR_CUDA drops the kept address, so
 *   the next call looks it up again.
 * - Every call shares the array and it keeps the last call's contents: each
 *   call clears the counters it uses, and calls that overlap on the GPU (for
 *   instance on two streams at once) race on it.
 * - Sizes: the shape rules of dec_linear apply (M outside 1..64, K or ldx
 *   not a multiple of 8 and the like return DEC_ERR_INVALID_ARG); N above
 *   131072, the array's limit, returns DEC_ERR_UNSUPPORTED. r may be NULL;
 *   out may alias r exactly.
 * - Calls no cudaMalloc, cudaFree or other allocating routine. */
dec_status dec_linear_noalloc(dec_handle* h, const dec_bf16* x, int ldx, const dec_bf16* W, const dec_bf16* r,
                              dec_bf16* out, int M, int N, int K, cudaStream_t stream);

/* y[M][H] = x / sqrt(mean(x^2) + eps) * gamma per row (fp32 math, bf16 out).
 * The RMSNorm of the pre-norm decode layer; not named on the pages. y may
 * alias x. 1 <= M <= 64, 8 <= H <= 65536, H % 8 == 0. */
dec_status dec_rmsnorm(dec_handle* h, const dec_bf16* x, const dec_bf16* gamma, dec_bf16* y, int M, int H,
                       float eps, cudaStream_t stream);

/* ------------------------------------------------------------------ router */

dec_status moe_route_topk_workspace_size(const dec_handle* h, int M, int H, int E, size_t* bytes);

/* Router scoring and top-k [K3 P1§3]: logits = x W_r^T (x bf16 [M][H], W_r
 * fp32 [E][H], fp32 math), scores s = sigmoid(logits); per token the k
 * largest scores in descending order, ties to the lower expert id, and
 * weights w_j = s_j / sum of the k selected scores.
 * Outputs: idx int32 [M][k], w fp32 [M][k], scores fp32 [M][E] (scores may be
 * NULL). 1 <= M <= 64, 1 <= k <= 16, k <= E <= 1024, H % 8 == 0. */
dec_status moe_route_topk(dec_handle* h, const dec_bf16* x, const float* Wr, int M, int H, int E, int k,
                          int32_t* idx, float* w, float* scores, void* ws, size_t ws_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------ experts */

dec_status moe_experts_workspace_size(const dec_handle* h, int M, int k, int E, int H, int I, size_t* bytes);

/* MoE layer body [K3 P1§3]:
 *   out_t = [residual_t +] sum_j w_tj E_{idx_tj}(x_t) [+ S(x_t)]
 * with SwiGLU experts E_e(x) = Wd_e (silu(Wg_e x) * (Wu_e x)).
 * x bf16 [M][H] (the normed hidden state); idx int32 [M][k] in [0, E);
 * w fp32 [M][k]; expert banks Wg, Wu bf16 [E][I][H] and Wd bf16 [E][H][I];
 * shared expert Wg_s, Wu_s bf16 [I][H], Wd_s bf16 [H][I] (all three NULL for
 * none); residual bf16 [M][H] or NULL; out bf16 [M][H] (may alias residual,
 * not x). Each selected expert's weights are read once for all its tokens
 * (at M = 1 each entry is its own problem, so an expert listed twice is read
 * twice). For M >= 2 the shared expert runs on the handle's side stream,
 * overlapped with the routing table and the routed experts, and joins
 * `stream` before return; at M = 1 it is one more problem of the routed
 * launches.
 * The SwiGLU output h is rounded to bf16; everything else stays fp32 until
 * the single bf16 rounding of out.
 * 1 <= M <= 64, 1 <= k <= 16, H and I multiples of 128. */
dec_status moe_experts(dec_handle* h, const dec_bf16* x, const int32_t* idx, const float* w, int M, int k,
                       const dec_bf16* Wg, const dec_bf16* Wu, const dec_bf16* Wd, int E, int H, int I,
                       const dec_bf16* Wg_s, const dec_bf16* Wu_s, const dec_bf16* Wd_s, const dec_bf16* residual,
                       dec_bf16* out, void* ws, size_t ws_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------ MoE layer */

/* Weights and shape of one MoE layer. */
typedef struct dec_moe_weights {
  int H;                /* hidden size */
  int E;                /* routed experts */
  int k;                /* experts per token */
  int I;                /* expert intermediate size */
  float eps;            /* RMSNorm epsilon (used with gamma) */
  const dec_bf16* gamma;  /* [H] RMSNorm gains applied to the input first, or NULL for none */
  const float* W_r;     /* [E][H] fp32 router */
  const dec_bf16* Wg;   /* [E][I][H] */
  const dec_bf16* Wu;   /* [E][I][H] */
  const dec_bf16* Wd;   /* [E][H][I] */
  const dec_bf16* Wg_s; /* [I][H] or NULL (no shared expert) */
  const dec_bf16* Wu_s; /* [I][H] */
  const dec_bf16* Wd_s; /* [H][I] */
} dec_moe_weights;

dec_status moe_layer_workspace_size(const dec_handle* h, const dec_moe_weights* Wt, int M, size_t* bytes);

/* The MoE layer of a decode step in one call [K3 P1§3, §4]: routing and the
 * experts with the schedule of decode_layer's MoE block:
 *   b       = gamma ? RMSNorm(x; gamma, eps) : x
 *   idx, w  = top-k(sigmoid(b W_r^T)), renormalised
 *   out     = [residual +] sum_j w_j E_idx_j(b) [+ S(b)]
 * x bf16 [M][H]; residual bf16 [M][H] or NULL; out bf16 [M][H] (may alias
 * residual, not x); idx int32 [M][k], w fp32 [M][k] and scores fp32 [M][E]
 * receive the routing when given (each may be NULL). At one token (and two,
 * with a shared expert) the routing, the shared expert's gate/up and the
 * selected experts' gate/up are one launch whose CTAs wait, with the handle's
 * limit, for the routing that one of them publishes; the down projection
 * follows with the combine and the residual. Above, the split-K family runs
 * the shared expert on the handle's side stream. Same shape rules as
 * moe_experts (1 <= M <= 64, 1 <= k <= 16, k <= E <= 1024, H and I multiples
 * of 128). */
dec_status moe_layer(dec_handle* h, const dec_moe_weights* Wt, const dec_bf16* x, const dec_bf16* residual,
                     dec_bf16* out, int M, int32_t* idx, float* w, float* scores, void* ws, size_t ws_bytes,
                     cudaStream_t stream);

/* ------------------------------------------------------------------ decode layer */

/* Weights and shape of one decode layer. */
typedef struct dec_layer_weights {
  int H;     /* hidden size */
  int N_in;  /* width of the attention input projection */
  int K_out; /* input width of the out-projection, K_out <= N_in */
  int E;     /* routed experts */
  int k;     /* experts per token */
  int I;     /* expert intermediate size */
  float eps; /* RMSNorm epsilon */
  const dec_bf16* gamma1; /* [H] */
  const dec_bf16* W_in;   /* [N_in][H] */
  const dec_bf16* W_o;    /* [H][K_out] */
  const dec_bf16* gamma2; /* [H] */
  const float* W_r;       /* [E][H] fp32 */
  const dec_bf16* Wg;     /* [E][I][H] */
  const dec_bf16* Wu;     /* [E][I][H] */
  const dec_bf16* Wd;     /* [E][H][I] */
  const dec_bf16* Wg_s;   /* [I][H] or NULL (no shared expert) */
  const dec_bf16* Wu_s;   /* [I][H] */
  const dec_bf16* Wd_s;   /* [H][I] */
  const void* prefetch_next;   /* optional: weights of the next operator to warm in L2 */
  size_t prefetch_bytes;       /* (multiple of 16; 0 for none) */
} dec_layer_weights;

/* Optional device buffers that receive intermediates of decode_layer (any
 * member may be NULL): h1 bf16 [M][H], idx int32 [M][k], w fp32 [M][k],
 * scores fp32 [M][E]. */
typedef struct dec_layer_trace {
  dec_bf16* h1;
  int32_t* idx;
  float* w;
  float* scores;
} dec_layer_trace;

dec_status decode_layer_workspace_size(const dec_handle* h, const dec_layer_weights* Wt, int M, size_t* bytes);

/* One decode layer in place on h bf16 [M][H]:
 *   a  = RMSNorm(h; gamma1)
 *   y  = a W_in^T                        (small-matrix / split-K by M) [K3 P1§1]
 *   h1 = h + y[:, :K_out] W_o^T           (out-projection + residual)   [K3 P1§2]
 *   b  = RMSNorm(h1; gamma2)
 *   idx, w = top-k(sigmoid(b W_r^T))                                    [K3 P1§3]
 *   h  = h1 + sum_j w_j E_idx_j(b) + S(b)
 * The attention core, which the pages do not define, is read as the identity
 * on the first K_out columns of y. At M = 1 the layer is four launches on
 * `stream`: in-projection with the first RMSNorm, out-projection with the
 * residual, the MoE front (second RMSNorm, router, top-k, routing table, the
 * shared expert's gate/up streamed meanwhile, then the selected experts'
 * gate/up), and the down projection (selected and shared experts) fused with
 * the combine and the residual; M = 2 is the same with two rows. For M >= 3
 * the split-K family runs the shared expert on the handle's side stream
 * [K3 P1§3]. While the router and top-k run, the `prefetch_next` region (if
 * any) is pulled into L2 [K3 P1§4]: by the MoE front's CTAs while they wait
 * for the routing, else by a kernel on a second side stream. trace may be
 * NULL. */
dec_status decode_layer(dec_handle* h, const dec_layer_weights* Wt, dec_bf16* hidden, int M,
                        const dec_layer_trace* trace, void* ws, size_t ws_bytes, cudaStream_t stream);

/* Pull [ptr, ptr + bytes) into L2 on `stream` with an evict-last policy
 * [K3 P1§4]. ptr and bytes multiples of 16. */
dec_status dec_prefetch_l2(dec_handle* h, const void* ptr, size_t bytes, cudaStream_t stream);

/* ------------------------------------------------------------------ measurement */

/* Per-kernel timing record returned by dec_profile_read. */
typedef struct dec_kernel_time {
  char name[32];   /* kernel tag, e.g. "in_proj", "gate_up", "shared_down" */
  int launches;    /* launches since the last read */
  double total_ms; /* summed device time of those launches */
} dec_kernel_time;

/* Enable (1) or disable (0) per-kernel timing: every kernel launch is then
 * bracketed by CUDA events on the stream it is launched on. The events
 * separate kernels, so programmatic dependent launch overlap is lost while
 * profiling is on; use it for per-kernel durations, not for step times. */
dec_status dec_set_profiling(dec_handle* h, int enable);

/* Synchronise, then aggregate the timing records by kernel tag into
 * out[0 .. capacity) (*count receives the number of tags) and clear them. */
dec_status dec_profile_read(dec_handle* h, dec_kernel_time* out, int capacity, int* count);

/* Number of kernels this handle has launched since it was created. */
uint64_t dec_launch_count(const dec_handle* h);

/* ------------------------------------------------------------------ test hooks */

/* Launch a kernel whose mbarrier wait can never complete; it must give up
 * after the handle's wait limit and set the device error word. Used to test
 * that timeouts surface as DEC_ERR_TIMEOUT with the context still usable. */
dec_status dec_test_wait_timeout(dec_handle* h, cudaStream_t stream);

/* Run the MoE front launch (tokens: 1, or 2 for the few-token kernel) on a
 * small zeroed problem whose routing hand-off can never complete (its arrival
 * counter starts past the grid size), so the routing flag is never set: every
 * CTA's wait for it must give up after the handle's wait limit and set the
 * device error word. Allocates and frees its own buffers and synchronises
 * `stream`. Used to test that the routing wait surfaces as DEC_ERR_TIMEOUT
 * with the context still usable. tokens outside {1, 2}: DEC_ERR_INVALID_ARG. */
dec_status dec_test_routing_wait_timeout(dec_handle* h, int tokens, cudaStream_t stream);

/* 1 (default): decode_layer and moe_layer use the MoE front launches at one
 * and two tokens when there is a shared expert (routing, the shared expert's
 * gate/up and the selected experts' gate/up in one launch). 0: they use the
 * launches taken where a front does not apply (no shared expert, or shapes
 * outside its limits): the routing launch, then the grouped gate/up with the
 * shared expert as one more problem, then the down projection. Both compute
 * the same layer; the hook lets tests run the second path with a shared
 * expert. */
dec_status dec_test_set_moe_front(dec_handle* h, int enable);

/* How the split-K kernel finishes a tile split between CTAs (a tile's partial
 * sums from several CTAs' ranges of k). 0 (default): the CTA holding the
 * first piece waits a bounded time for the others, then adds all pieces in k
 * order from shared memory; past the bound it publishes its piece, and the
 * CTA that completes the count finishes the tile. 1: every CTA publishes its
 * piece at once, so the tile is always finished by the CTA that completes the
 * count (from shared memory when that CTA is at the end of its range). 2: as
 * 1, and the finishing CTA always reads the pieces with batched loads from
 * L2. All three add the same fp32 partials in the same k order, so they give
 * the same bits; the hook lets tests check that. Other values:
 * DEC_ERR_INVALID_ARG. */
dec_status dec_test_set_engine_finish(dec_handle* h, int mode);

/* Hold `ctas` SMs (1 <= ctas <= the device's SM count) for hold_ns
 * nanoseconds (at most 2 s) with a kernel on `stream`: one CTA per SM that
 * takes the whole per-block shared memory, so nothing else fits beside it,
 * and sleeps on the global timer. It writes nothing. Used to test that the
 * MoE fronts complete when another stream's kernel holds part of the SMs, so
 * that not all of their CTAs can be resident at once. */
dec_status dec_test_occupy_sms(dec_handle* h, int ctas, uint64_t hold_ns, cudaStream_t stream);

/* Copy `bytes` from src to dst on `stream` after spinning for delay_ns
 * (bounded by the clock): a slow producer for ordering tests of the
 * programmatic-dependent-launch path. */
dec_status dec_test_delayed_copy(dec_handle* h, void* dst, const void* src, size_t bytes, uint64_t delay_ns,
                                 cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_DECODE_H */
