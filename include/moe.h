/*
 * moe.h -- C ABI of the GB300 (sm_103a) routed-expert SwiGLU MoE layer.
 *
 * The layer (one per call of moe_forward), for every token row x_t of x[T, d]:
 *   1. router logits  l[t, e] = sum_i x[t, i] * router_w[e, i] (+ router_b[e]),
 *      computed to fp32 accuracy;
 *   2. the top_k experts with the largest logits, listed in ascending expert id;
 *   3. their weights: softmax over all E logits, renormalised over the chosen k;
 *   4. tokens grouped by expert: per-expert counts, exclusive-prefix offsets, and
 *      a permutation listing each expert's tokens in ascending token order;
 *   5. each chosen expert's SwiGLU FFN  o = W_down (silu(W_gate x) * (W_up x)),
 *      bf16 weights, fp32 accumulation;
 *   6. y_t = sum_j w[t, j] * o_{e_j}(x_t) + o_shared(x_t), summed in fp32 and
 *      stored in x's dtype.
 * Source: "Optimizing on-device inference for Apple Silicon" (Perplexity), section
 * "Qwen creates three different workload shapes" (a router scores 256 experts,
 * picks eight, plus one shared expert that processes every token), section
 * "Keeping expert routing on the GPU" (histogram, prefix pass to start offsets,
 * scatter into expert groups, block map, all without a CPU round trip), section
 * "Dequantizing weights during matrix multiplication" (fp32 accumulation, bf16
 * output) and section "Reducing intermediate and state traffic" (the two expert
 * input projections fused with the gated activation; the output projection fused
 * with the routing score and the shared expert's result).
 *
 * Conventions shared by every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library
 *    never frees them.  Row-major, densely packed, 16-byte aligned
 *    (MOE_ERR_ALIGN otherwise).  bf16 = 16-bit bfloat16 bit patterns.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *    stream).  They never synchronise, never copy to the host and never
 *    allocate: all scratch memory is owned by the context, sized at moe_init
 *    for cfg->max_tokens.  Two calls on one context must not overlap in time
 *    (they share that scratch memory); use one context per concurrent stream.
 *  - Return codes are the MOE_* values below.  Argument errors are detected on
 *    the host before anything is launched.  Errors detected by a kernel
 *    (MOE_ERR_TIMEOUT, MOE_ERR_BOUNDS) are latched in a device status word and
 *    reported by moe_status().
 *  - T == 0 is a valid call that launches nothing and returns MOE_OK.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* return codes */
#define MOE_OK 0
#define MOE_ERR_ARG 1          /* null pointer, bad shape, top_k not in [1, min(E, 32)], T > max_tokens */
#define MOE_ERR_ALIGN 2        /* a tensor pointer is not 16-byte aligned */
#define MOE_ERR_UNSUPPORTED 3  /* a shape outside what the kernels handle (see moe_init) */
#define MOE_ERR_CUDA 4         /* a CUDA runtime/driver call failed (launch, allocation, tensor map) */
#define MOE_ERR_TIMEOUT 5      /* device side: a bounded wait inside a kernel ran out; work abandoned */
#define MOE_ERR_BOUNDS 6       /* device side: an index read from scratch memory was out of range */
#define MOE_ERR_NOMEM 7        /* moe_init could not allocate its scratch memory */

/* dtype of x (and of y, which has the same dtype) */
#define MOE_F32 0
#define MOE_BF16 1

/* storage format of the expert weights (moe_config.weight_format) */
#define MOE_W_BF16 0           /* bf16 matrices, as described at moe_forward */
#define MOE_W_Q4G64 1          /* 4-bit group-affine ("Optimizing on-device inference for Apple Silicon",
                                  section "Dequantizing weights during matrix multiplication": 4-bit
                                  codes expanded inside the multiplication).  Along every weight row
                                  [K input columns], each group of 64 consecutive columns has one bf16
                                  scale s and one bf16 bias b, and w = s * q + b for the column's 4-bit
                                  code q in 0..15.  Each row of K weights is stored as 9 K / 16 bytes:
                                  its codes (K / 8 uint32 words, eight codes per word, the lowest
                                  nibble is the lowest column), then its K / 64 bf16 scales, then its
                                  K / 64 bf16 biases.  Matrices are these rows back to back, in the
                                  bf16 layouts' row order: experts_gate_up [E, 2I] rows of d weights,
                                  experts_down [E, d] rows of I weights, shared_w the shared gate_up
                                  [2I] rows of d weights followed by its down [d] rows of I weights.
                                  Needs inter % 256 == 0 (and, on the grouped-GEMM path, d and inter
                                  each 256 or a multiple of 512). */

/* execution path for the expert FFNs (moe_set_path) */
#define MOE_PATH_AUTO 0        /* T <= 4: GEMV over the selected experts; otherwise grouped GEMM */
#define MOE_PATH_GEMV 1        /* bandwidth-bound GEMV over the selected experts (small T only, else
                                  MOE_ERR_UNSUPPORTED); for T <= 16 when shapes allow, the whole layer
                                  runs as one cooperative kernel whose blocks wait on each other's
                                  published logits and activations (epoch-tagged words) */
#define MOE_PATH_GEMM 2        /* tcgen05/TMEM grouped GEMM */

/* router logit kernel (moe_set_router) */
#define MOE_ROUTER_AUTO 0      /* tensor-core router for bf16 x, E == 256 and T > 64; else fp32 FMA */
#define MOE_ROUTER_SIMT 1      /* fp32 FMA on the CUDA cores */
#define MOE_ROUTER_TENSOR 2    /* tcgen05: bf16 x times router_w split into bf16 hi + mid + lo terms,
                                  fp32 accumulation (needs bf16 x and E == 256; else fp32 FMA) */

typedef struct moe_config {
  int d;               /* model width; multiple of 256 */
  int n_experts;       /* routed experts E, 1..256 */
  int inter;           /* routed expert inner size I; multiple of 128 */
  int shared_inter;    /* shared expert inner size; must equal inter when has_shared */
  int top_k;           /* largest top_k a call will use, 1..min(E, 32) */
  int max_tokens;      /* largest T a call will use (scratch memory is sized for it) */
  int x_dtype;         /* MOE_F32 or MOE_BF16 */
  int has_router_bias; /* 1: calls pass router_b */
  int has_shared;      /* 1: calls pass shared_w */
  int bias_select_only; /* 1 (with has_router_bias): router_b takes part in picking the top_k experts
                           but not in their weights, which are the softmax of the unbiased logits over
                           the picks (a bias used only to balance expert load); 0: the bias enters both */
  int shared_gate;     /* 1 (with has_shared): sigmoid-gated shared expert -- router_w holds E + 1 rows,
                          row E being a gate vector g of d fp32 values, and the shared expert's output
                          for token t is scaled by sigmoid(x_t . g) (no bias); 0: weight one */
  int weight_format;   /* MOE_W_BF16 or MOE_W_Q4G64: how experts_gate_up, experts_down and shared_w
                          are stored */
} moe_config;

typedef struct moe_ctx moe_ctx;

/* Validate `cfg`, select the current CUDA device, allocate the context and its
 * device scratch memory for cfg->max_tokens tokens.  On success *out owns them
 * until moe_destroy.  Errors: MOE_ERR_ARG (null pointers, non-positive sizes),
 * MOE_ERR_UNSUPPORTED (d % 256, inter % 128, E > 256, shared_inter != inter,
 * device is not sm_103), MOE_ERR_NOMEM, MOE_ERR_CUDA.  Synchronous.
 * The GEMV path additionally needs d % 256 == 0, inter % 256 == 0 and a T small
 * enough for x and the activations to fit in shared memory. */
int moe_init(const moe_config* cfg, moe_ctx** out);

/* Steps 1-4 only, for inspection.  Inputs: x [T, d] (cfg->x_dtype), router_w
 * [E, d] fp32 (a shared-gate row E, if present, is not read), router_b [E]
 * fp32 (NULL unless cfg->has_router_bias).  Outputs
 * (caller-owned device buffers): idx [T, top_k] int32 (ascending expert id per
 * row), w [T, top_k] fp32, counts [E] int32, offsets [E + 1] int32 (exclusive
 * prefix of counts; offsets[E] = T * top_k), perm [T * top_k] int32 (token ids
 * grouped by expert, ascending within a group).  Any output may be NULL to skip
 * it.  Asynchronous on `stream`. */
int moe_route(moe_ctx* ctx, const void* x, int T, const float* router_w, const float* router_b,
              int top_k, int32_t* idx, float* w, int32_t* counts, int32_t* offsets, int32_t* perm,
              void* stream);

/* The whole layer: y [T, d] (cfg->x_dtype) from x [T, d] (cfg->x_dtype),
 * router_w [E, d] fp32 ([E + 1, d] with cfg->shared_gate), router_b [E] fp32 or NULL, experts_gate_up [E, 2I, d]
 * bf16 (per expert: rows 0..I-1 gate projection, rows I..2I-1 up projection),
 * experts_down [E, d, I] bf16, shared_w (NULL unless cfg->has_shared): one bf16
 * buffer holding the shared expert's gate_up [2I, d] followed by its down
 * [d, I].  y must not alias any input.  Asynchronous on `stream`; captures into
 * a CUDA graph (no host synchronisation, no allocation). */
int moe_forward(moe_ctx* ctx, const void* x, int T, const float* router_w, const float* router_b,
                const void* experts_gate_up, const void* experts_down, const void* shared_w,
                int top_k, void* y, void* stream);

/* Choose the expert-FFN path for later calls (MOE_PATH_*).  Used for paired
 * A/B measurements of the two paths on the same inputs.  MOE_ERR_ARG on an
 * unknown value. */
int moe_set_path(moe_ctx* ctx, int path);

/* Choose the router logit kernel for later calls (MOE_ROUTER_*).  Both give
 * fp32-accurate logits; used for paired A/B measurements.  MOE_ERR_ARG on an
 * unknown value. */
int moe_set_router(moe_ctx* ctx, int router);

/* Prefetch hint for stacked layers: the next moe_forward call on `ctx` that
 * takes the small-T path pulls `next_router_w` ([E, d] fp32) and
 * `next_shared_w` (shared gate_up + down, bf16) -- the weights the following
 * layer reads first -- into L2 while its own last phase is bound by latency,
 * so that the following layer starts from L2.  Either may be NULL.  The hint
 * serves one call, then clears.  It only moves data into the cache; results
 * do not depend on it.  MOE_ERR_ALIGN if a pointer is not 16-byte aligned. */
int moe_set_prefetch(moe_ctx* ctx, const float* next_router_w, const void* next_shared_w);

/* Launch overlap for back-to-back layers (no counterpart in the source pages;
 * a CUDA launch option).  With on = 1, later moe_forward calls that take the
 * fused small-T kernel launch it with programmatic stream serialization: its
 * blocks may start while the preceding kernel on the stream is finishing, and
 * read only the weights (router_w, shared_w) before they wait for that kernel
 * to complete; x, y and all scratch are touched after the wait.  The caller
 * promises that the work preceding each such call on its stream does not
 * write those weight arrays.  on = 0 (the default) launches normally.
 * MOE_ERR_ARG on other values. */
int moe_set_overlap(moe_ctx* ctx, int on);

/* Chunked prefill with bounded workspace ("Optimizing on-device inference for
 * Apple Silicon", section on bounding temporary memory by splitting the prompt
 * into chunks: a long prompt runs as a sequence of bounded chunks whose
 * temporary buffers are reused, so working memory does not grow with it).
 * With chunk > 0, moe_forward accepts any T >= 0 (not only T <= max_tokens)
 * and runs the layer on consecutive slices of at most `chunk` tokens through
 * the context's workspace, which stays sized for max_tokens.  The result is
 * the layer over all T tokens (tokens are independent; each slice may take
 * its own path by size); the selected experts' weights are read once per
 * slice.  chunk = 0 (the default) turns it off.  MOE_ERR_ARG if chunk < 0 or
 * chunk > max_tokens.  moe_route keeps the T <= max_tokens limit. */
int moe_set_chunk_tokens(moe_ctx* ctx, int chunk);

/* Synchronise the device, then read and clear the context's device status
 * word: MOE_OK, or the first MOE_ERR_TIMEOUT / MOE_ERR_BOUNDS latched by a
 * kernel since the last call; MOE_ERR_CUDA if the synchronisation itself
 * reported an error. */
int moe_status(moe_ctx* ctx);

/* Bounded waits: how long (nanoseconds, measured in SM clock cycles at 2 per
 * ns) a kernel polls a barrier or a published value before giving up with MOE_ERR_TIMEOUT.  A wait
 * always polls at least 256 times before it looks at the clock.  0 restores
 * the default (1 s).  MOE_ERR_ARG if negative. */
int moe_set_spin_limit(moe_ctx* ctx, long long limit);

/* Kernel ids for moe_time_kernel. */
#define MOE_K_ROUTER 0         /* router logits (fp32 FMA or tensor-core) */
#define MOE_K_SELECT 1         /* top-k selection and weights */
#define MOE_K_GROUP 2          /* prefix over chunks/experts and the stable scatter (on the grouped-GEMM
                                  path the scatter also writes the token rows in grouped order) */
#define MOE_K_GEMV_GATE_UP 3   /* GEMV path: gate/up projections + SwiGLU */
#define MOE_K_GEMV_DOWN 4      /* GEMV path: down projection + weighted combine + shared */
#define MOE_K_GEMM_GATE_UP 5   /* grouped GEMM: gate/up projections + SwiGLU */
#define MOE_K_GEMM_DOWN 6      /* grouped GEMM: down projection */
#define MOE_K_COMBINE 7        /* grouped-GEMM path: weighted combine + shared */
#define MOE_K_DECODE_FUSED 8   /* small-T path: the whole layer in one cooperative kernel */

/* Profiling hook: the next moe_forward/moe_route call on `ctx` records the
 * CUDA events `ev_start` / `ev_stop` (cudaEvent_t, created by the caller with
 * timing enabled) on its stream immediately before and after launching kernel
 * `kernel_id` (MOE_K_*), then disarms.  Works under stream capture (the
 * records become graph nodes).  If that call does not launch the kernel the
 * events are not recorded.  MOE_ERR_ARG on a bad id or null event. */
int moe_time_kernel(moe_ctx* ctx, int kernel_id, void* ev_start, void* ev_stop);

/* Record the CUDA event `event` (a cudaEvent_t created with timing) on
 * `stream`; under stream capture the record becomes a timeable event node of
 * the graph (plain cudaEventRecord there only orders streams).  Profiling
 * helper for timing a run of launches.  MOE_ERR_ARG on a null event. */
int moe_record_event(void* event, void* stream);

/* Number of kernels this context has launched (or captured) so far. */
long long moe_launch_count(moe_ctx* ctx);

/* Test hook for failure detection without a GPU fault: with on = 1, later
 * calls make the grouped GEMM's MMA thread, and every block of the fused
 * decode kernel where it waits for the router logits, wait once for an event that never
 * happens.  The bounded wait runs out after the spin limit, the kernel records
 * MOE_ERR_TIMEOUT, drains its in-flight copies, frees its tensor memory and
 * returns; moe_status then reports the timeout.  on = 0 turns it off.
 * MOE_ERR_ARG on other values. */
int moe_inject_stall(moe_ctx* ctx, int on);

/* Allocation-free decode layer (no counterpart in the source pages; added for
 * callers that cannot allocate device memory).  A plugin running inside a host
 * application whose device memory belongs to the host's own allocator (every
 * buffer comes from the host's pool; allocating outside it is forbidden), or a
 * serving loop with a fixed latency budget (an allocation may synchronise the
 * device and stall every stream), cannot call cudaMalloc, and so cannot create
 * a context with moe_init.  This entry point runs the same fused decode kernel
 * as moe_forward's small-T path, but its scratch memory is a fixed device array
 * inside the library (1,312,256 bytes, about 1.3 MB, held on every GPU that
 * loads the library until the process exits).  It calls no cudaMalloc, cudaFree
 * or allocating library routine.
 *
 * Inputs and outputs are as for moe_forward, with the shapes passed directly:
 * x [T, d] (x_dtype), router_w [E, d] fp32, router_b [E] fp32 or NULL,
 * experts_gate_up [E, 2*inter, d] bf16, experts_down [E, d, inter] bf16,
 * shared_w (shared gate_up [2*inter, d] then down [d, inter], bf16) or NULL,
 * y [T, d] (x_dtype).  The two moe_config variants are fixed: a router bias, if
 * given, enters both the selection and the weights (bias_select_only = 0), and
 * the shared expert, if given, has weight one (shared_gate = 0).
 * status: optional device word (NULL = none) into which a
 * kernel ORs a failure it detects (1 = a bounded wait ran out, 2 = an index was
 * out of range); it is not cleared by the call.
 * Limits of the fixed scratch: T <= 16, top_k <= 8, inter <= 1024, E <= 256,
 * plus the fused kernel's own (d in {512, 1024, 2048}, inter a multiple of 256,
 * its shared-memory staging); larger shapes return MOE_ERR_UNSUPPORTED before
 * anything is launched.  The first call on each device looks up the array's
 * device address (cudaGetSymbolAddress) and sets kernel attributes, with that
 * device current: make that first call before any stream capture.  Every call
 * shares the one array, which keeps the previous call's contents (its zero
 * start and every later state are valid starts), so calls that overlap on the
 * GPU -- on different streams, or from different threads -- race and must not
 * be issued.  Asynchronous on `stream`; one kernel launch per call. */
int moe_decode_noalloc(const void* x, int T, int x_dtype, int d, int n_experts, int inter, int top_k,
                       const float* router_w, const float* router_b, const void* experts_gate_up,
                       const void* experts_down, const void* shared_w, void* y, unsigned* status, void* stream);

/* Test and inspection hook: copy the routing tables that the last moe_forward
 * call on `ctx` computed and used itself (for a chunked call: its last slice),
 * device to device, asynchronously on `stream`.  T and top_k are that call's.
 * Outputs (caller-owned device buffers, any may be NULL to skip it): idx
 * [T, top_k] int32 (ascending expert id per row), w [T, top_k] fp32, counts [E]
 * int32, offsets [E + 1] int32, perm [T * top_k] int32 (token ids grouped by
 * expert, ascending within a group), slot [T, top_k] int32 (the position in
 * perm of each (token, pick)).  Every path writes all six: the grouped GEMMs and
 * the GEMV kernels through the grouping kernels, the fused small-T kernel from
 * its first block's in-kernel grouping.  *T_out / *k_out (host pointers, may be
 * NULL) receive that call's T and top_k.  MOE_ERR_ARG if ctx is NULL or no
 * moe_forward call has run on it yet; MOE_ERR_ALIGN for unaligned outputs. */
int moe_last_routing(moe_ctx* ctx, int32_t* idx, float* w, int32_t* counts, int32_t* offsets, int32_t* perm,
                     int32_t* slot, int* T_out, int* k_out, void* stream);

/* Static description of a return code. */
const char* moe_strerror(int code);

/* Free the context and its scratch memory (synchronises the device first).
 * NULL is a no-op. */
void moe_destroy(moe_ctx* ctx);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
