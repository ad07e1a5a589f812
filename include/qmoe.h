/*
 * qmoe.h -- C ABI of the GB300 (sm_103a) weight-only block-quantised
 * Mixture-of-Experts layer forward (QMoE).
 *
 * The layer computes, for T tokens x[T,H] and router logits[T,E]:
 *
 *   1. routing: per token, the top_k experts by fp32 logit under a total
 *      order (-0.0 < +0.0), ties to the lower expert index, in rank order;
 *      weights exp(l - max_all) / (sum over all E, or over the k chosen when
 *      renormalising).  [onnx-runtime-ep-cuda src/kernels/qmoe.rs, CUDA_SRC:
 *      total_order_key, route_value_is_better, qmoe_route]
 *   2. grouping: per-expert counts, exclusive offsets and a stable route
 *      permutation, then a tile work-list (experts ascending).  [qmoe.rs
 *      launch_grouping; metrale gemm_quant_moe.rs moe_build_tile_worklist]
 *   3. fc1: a[r,n] = sum_d x[t,d] * W1[e,n,d] with W = R_D((q - zp) * s) per
 *      block of B along d.  [qmoe.rs decode_affine_weight; onnxruntime PR
 *      "fused int2 mixed-input GEMM + GeGLU + fractional zero-point"
 *      (zero_point_offset); PR "fast INT3 QMoE kernels" review item "Round
 *      dequantized weights before accumulation"]
 *   4. gated activation h = act(gate) * up, gate = a[:, :I], up = a[:, I:],
 *      act = SiLU (SwiGLU) or tanh-GELU (GeGLU).  [qmoe.rs qmoe_activate,
 *      swiglu_value; PR "fused int2 ..." GeGLU]
 *   5. fc2: y[r,m] = sum_n h[r,n] * W2[e,m,n].
 *   6. combine: out[t,m] = R_D(sum_j w[t,j] * y[t*k+j, m]) in slot order j.
 *      [qmoe.rs qmoe_combine_impl]
 *
 * Canonical (input) tensor layouts, all contiguous row-major:
 *   x        [T, H]   dtype D (QMOE_F32 / QMOE_F16 / QMOE_BF16)
 *   logits   [T, E]   float32
 *   out      [T, H]   dtype D
 *   codes    uint8 [E, N, K*bits/8]: each row an LSB-first bit stream of K
 *            codes (code d occupies bits [d*bits, d*bits+bits) of the row).
 *            fc1: N = 2*inter rows [gate | up], K = hidden.
 *            fc2: N = hidden rows, K = inter.
 *   scales   dtype D [E, N, K/B]
 *   zero_points uint8 [E, N, ceil((K/B)*bits/8)]: LSB-first bit stream of the
 *            K/B per-block zero points at the weight bit width
 *            (QMOE_ZP_UINT8 only).
 *
 * Conventions.
 *   - Pointers named *_dev are device pointers; *_host are host pointers.
 *     "stream" is a cudaStream_t passed as void* (NULL = legacy default).
 *   - Ownership: the caller owns every pointer it passes.  The layer owns its
 *     prepacked weights and workspace until qmoe_destroy.  Inputs to
 *     qmoe_prepack may be freed once the stream has been synchronised.
 *   - Errors: every call returns a qmoe_status; argument and shape checks are
 *     synchronous.  qmoe_last_error() gives a message for the last failure on
 *     that layer.  Device-side conditions (bounded waits that ran out) are
 *     reported by qmoe_poll_device_status().
 *   - Concurrency: one layer serves one stream at a time.
 *   - Graph capture: qmoe_forward allocates nothing when num_tokens <= the
 *     reserved count (qmoe_reserve); it may then be captured into a CUDA
 *     graph.  Exceeding the reservation while capturing returns
 *     QMOE_ERR_STATE.
 */
#ifndef QMOE_H_
#define QMOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct qmoe_layer qmoe_layer;

typedef enum {
  QMOE_OK = 0,
  QMOE_ERR_INVALID_ARG = 1,   /* bad pointer, shape or value */
  QMOE_ERR_UNSUPPORTED = 2,   /* valid QMoE, but not a supported variant */
  QMOE_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed */
  QMOE_ERR_OOM = 4,           /* device allocation failed */
  QMOE_ERR_STATE = 5,         /* call out of order (e.g. forward before prepack) */
  QMOE_ERR_TIMEOUT = 6        /* a bounded device-side wait ran out */
} qmoe_status;

enum { QMOE_ZP_SYMMETRIC = 0, QMOE_ZP_UINT8 = 1, QMOE_ZP_OFFSET = 2 };
/* Gated activations (fc1 has 2*inter rows: gate and up) and the non-gated
 * ones of [qmoe.rs qmoe_activate] (fc1 has inter rows, h = act(fc1 output)):
 * relu max(v, 0); gelu the tanh form 0.5 v (1 + tanh(0.79788456 (v + 0.044715 v^3)));
 * silu v * sigmoid(v); identity v. */
enum {
  QMOE_ACT_SWIGLU = 0,
  QMOE_ACT_GEGLU_TANH = 1,
  QMOE_ACT_RELU = 2,
  QMOE_ACT_GELU_TANH = 3,
  QMOE_ACT_SILU = 4,
  QMOE_ACT_IDENTITY = 5
};
enum { QMOE_F32 = 0, QMOE_F16 = 1, QMOE_BF16 = 2 };

/* Stage boundaries recorded by qmoe_set_trace_events (see there). */
enum {
  QMOE_TRACE_BEGIN = 0,
  QMOE_TRACE_ROUTED = 1,     /* after routing + grouping + work-lists */
  QMOE_TRACE_FC1 = 2,        /* after fc1 (+ fused activation) */
  QMOE_TRACE_FC2 = 3,        /* after fc2 */
  QMOE_TRACE_END = 4,        /* after the combine */
  QMOE_TRACE_NUM_EVENTS = 5
};

/*
 * Create a layer description.  Host-only: allocates no device memory.
 *   hidden, inter   H and I (fc1 has 2*inter rows, gate then up)
 *   experts, top_k  E (1..1024) and k (1 <= k <= E)  [qmoe.rs requires
 *                   0 < k <= num_experts]
 *   bits_fc1/fc2    code widths, each in {1, 2, 3, 4, 8}
 *   block_size      B in {32, 64, 128}; hidden and inter must be multiples
 *                   of B  [qmoe.rs: power of two >= 16 dividing K]
 *   zp_mode         QMOE_ZP_SYMMETRIC (zp = 2^(bits-1)), QMOE_ZP_UINT8
 *                   (packed zero-point tensors), QMOE_ZP_OFFSET (one
 *                   fractional centre, set by qmoe_set_zero_point_offset)
 *   activation      QMOE_ACT_SWIGLU or QMOE_ACT_GEGLU_TANH (gated: fc1 has
 *                   2*inter rows), or QMOE_ACT_RELU / _GELU_TANH / _SILU /
 *                   _IDENTITY (non-gated: fc1 has inter rows)
 *   dtype           activation / scale / output type
 * Routing renormalisation defaults to on (qmoe_set_routing).
 * Returns INVALID_ARG for out-of-range values, UNSUPPORTED (with a
 * "requantize" hint) for widths / block sizes outside the supported set.
 */
qmoe_status qmoe_create(int hidden, int inter, int experts, int top_k, int bits_fc1,
                        int bits_fc2, int block_size, int zp_mode, int activation,
                        int dtype, qmoe_layer** out);

/* Renormalise the k routing weights (1, default) or divide by the softmax
 * sum over all E experts (0).  [qmoe.rs qmoe_route, `normalize`] */
qmoe_status qmoe_set_routing(qmoe_layer* layer, int normalize);

/* Fractional zero point for QMOE_ZP_OFFSET: w = (code - offset) * scale.
 * [PR "fused int2 ...", zero_point_offset]  Supported centres are multiples
 * of 0.5 in [0, 2^bits - 1] (e.g. 1.5 for 2-bit codes); other values return
 * UNSUPPORTED with a "requantize" hint.  Must be called before qmoe_prepack
 * in that mode. */
qmoe_status qmoe_set_zero_point_offset(qmoe_layer* layer, float offset);

/* SwiGLU attributes [qmoe.rs swiglu_value]: with g = gate, u = up,
 *   h = min(g, limit) * sigmoid(alpha * min(g, limit)) * (clamp(u, -limit, limit) + beta)
 * (a NaN in u is kept).  Defaults alpha = 1, beta = 0, limit = +inf: plain
 * silu(g) * u.  GeGLU ignores them.  alpha must be finite and nonzero, beta
 * finite, limit > 0 (+inf allowed); otherwise INVALID_ARG.  May be called at
 * any time; it applies to later forwards. */
qmoe_status qmoe_set_swiglu_params(qmoe_layer* layer, float alpha, float beta, float limit);

/* Row order of fc1's canonical codes / scales / zero points / bias
 * [qmoe.rs qmoe_activate, swiglu_fusion]: QMOE_FC1_CONCAT = concatenated
 * [gate (I rows) | up (I rows)] (default, swiglu_fusion 2),
 * QMOE_FC1_INTERLEAVED = interleaved (row 2f = gate f, row 2f+1 = up f;
 * swiglu_fusion 1), QMOE_FC1_SEPARATE_FC3 = fc1 holds the I gate rows and a
 * third projection fc3 the I up rows (qmoe_activate with fc3: gate = fc1,
 * linear = fc3), each [E, I, ...] and prepacked / biased with fc = 1 and
 * fc = 3.  Other values: INVALID_ARG.  Must precede qmoe_prepack(fc = 1 or 3)
 * and qmoe_set_bias(fc = 1 or 3); STATE otherwise.  With a non-gated
 * activation only QMOE_FC1_CONCAT applies (INVALID_ARG otherwise), except
 * QMOE_ACT_SILU with QMOE_FC1_SEPARATE_FC3, which is the gated form (gate =
 * fc1, up = fc3 through the SwiGLU of qmoe_set_swiglu_params) [qmoe.rs
 * uses_separate_gate]: the layer then behaves as QMOE_ACT_SWIGLU. */
enum { QMOE_FC1_CONCAT = 0, QMOE_FC1_INTERLEAVED = 1, QMOE_FC1_SEPARATE_FC3 = 2 };
qmoe_status qmoe_set_fc1_layout(qmoe_layer* layer, int layout);

/* Projection biases [qmoe.rs qmoe_linear_impl: output = sum + bias[e*N + n]]:
 * bias_dev is a float32 device array [E, N] (fc1: N = 2*inter in the fc1 row
 * order, or inter with QMOE_FC1_SEPARATE_FC3 or a non-gated activation;
 * fc2: N = hidden; fc3: N = inter,
 * only with QMOE_FC1_SEPARATE_FC3), added to the projection output (fc1 and
 * fc3 before the gated activation, fc2 before the weighted combine).  The
 * layer keeps its own copy (the caller may free bias_dev once `stream` has
 * been synchronised).  NULL removes the bias (synchronises `stream` first;
 * for fc1 / fc3 with separate projections it zeroes that half). */
qmoe_status qmoe_set_bias(qmoe_layer* layer, int fc, const float* bias_dev, void* stream);

/* Experts with more than `min_rows` routed rows take the tensor-core grouped
 * GEMM; the others the mma.sync weight-streaming decode kernel.  Any value
 * gives the same result within tolerance.  Default 0: every expert takes the
 * tensor-core path (the faster one at every measured shape, decode included);
 * fp32 activations always take the SIMT kernel.  [qmoe.rs prefill_min_tokens;
 * PR "fast INT3" kMaxProfiledExpandedRows] */
qmoe_status qmoe_set_gemm_min_rows(qmoe_layer* layer, int min_rows);

/* Which launch sequence qmoe_forward uses for small token counts:
 * QMOE_FUSED_OFF (0) the separate kernels; QMOE_FUSED_ON (1) the single
 * launch whenever it applies; QMOE_FUSED_AUTO (2, default) the single launch
 * when it applies and T * k <= 64 (where it measured faster).  It applies to
 * 16-bit activations, at most 64 tokens, E <= 256 with E a multiple of 4,
 * k <= 32, T * k <= 512 and fc1 / fc2 code widths in {2, 3, 4}: then routing,
 * grouping, fc1 with its activation, fc2 and the slot-ordered combine run in
 * one persistent (cooperative) kernel launch.  Otherwise the separate kernels
 * run (qmoe_set_gemm_min_rows picks between their projection paths).  Either
 * gives the same result within tolerance; the single launch is bitwise
 * deterministic.  Other values: INVALID_ARG.  [The pages motivate the fusion:
 * PR "fast INT3 QMoE kernels", single-CTA FusedSoftmaxTopKMapsKernel for up
 * to 8 rows and the fused finalize of moe_gemv; ferrum moe.rs
 * SingleTokenDirectMarlin.] */
enum { QMOE_FUSED_OFF = 0, QMOE_FUSED_ON = 1, QMOE_FUSED_AUTO = 2 };
qmoe_status qmoe_set_fused_decode(qmoe_layer* layer, int mode);

/* The combine of the tensor-core grouped GEMM path.  QMOE_COMBINE_REDUCE (0)
 * adds each route's w * y into an fp32 [T, H] accumulator with fp32
 * reductions in the fc2 epilogue (the order of the k additions may vary run
 * to run: a last-bit difference at most after rounding to D);
 * QMOE_COMBINE_ORDERED (1) writes the y rows and adds the k slots in
 * ascending order in a separate pass, bitwise deterministic at the cost of
 * writing and reading T * k * H fp32 values; QMOE_COMBINE_AUTO (2, the
 * default) takes the ordered combine for forwards of at most 64 tokens and
 * the reductions above.  The single launch and the decode kernels always
 * add the slots in order.  Other values: INVALID_ARG.  [qmoe.rs
 * qmoe_combine_impl: slots summed in order] */
enum { QMOE_COMBINE_REDUCE = 0, QMOE_COMBINE_ORDERED = 1, QMOE_COMBINE_AUTO = 2 };
qmoe_status qmoe_set_deterministic(qmoe_layer* layer, int mode);

/* Which launch sequence the last qmoe_forward / qmoe_forward_host used:
 * QMOE_PATH_NONE (no forward with tokens yet), QMOE_PATH_SEPARATE (routing,
 * projection and combine kernels) or QMOE_PATH_FUSED (the single launch).
 * For tests and benchmarks that must know what they measured. */
enum { QMOE_PATH_NONE = 0, QMOE_PATH_SEPARATE = 1, QMOE_PATH_FUSED = 2 };
int qmoe_last_forward_path(const qmoe_layer* layer);

/* Size the device workspace for up to max_tokens tokens.  Required before
 * capturing qmoe_forward into a CUDA graph.  Allocates device memory.
 * [qmoe.rs QMoEKernel scratch pool (`slots`): a warmed eager pass sizes the
 * pooled scratch, `capture_support` refuses capture until then, and a slot
 * that would have to grow during capture is an error] */
qmoe_status qmoe_reserve(qmoe_layer* layer, int64_t max_tokens);

/*
 * Copy one projection's weights (fc = 1, 2, or 3 with QMOE_FC1_SEPARATE_FC3)
 * from the canonical layout into the layer's own GB300 layouts, on `stream`.
 * [onnxruntime PR "fused int2 mixed-input GEMM + GeGLU + fractional
 * zero-point": PrePack wiring for fc1/fc2 (weights re-laid once, at load);
 * PR "fast INT3 QMoE kernels": PrePack releases the canonical scales once
 * they are re-laid]
 *   codes_dev        uint8 [E, N, K*bits/8]
 *   scales_dev       D     [E, N, K/B]
 *   zero_points_dev  uint8 [E, N, ceil((K/B)*bits/8)], non-NULL iff
 *                    zp_mode == QMOE_ZP_UINT8 (else must be NULL)
 * with N = 2*inter (fc1, gated activation), inter (fc1, non-gated; fc1 and
 * fc3 with separate projections; fc3 uses fc1's code width) or hidden (fc2).  With separate projections the
 * fc1 layouts are built once both fc = 1 and fc = 3 have been given.  May be
 * called again to replace the weights.  Allocates device memory.
 */
qmoe_status qmoe_prepack(qmoe_layer* layer, int fc, const uint8_t* codes_dev,
                         const void* scales_dev, const uint8_t* zero_points_dev,
                         void* stream);

/*
 * The layer forward on device buffers, asynchronous on `stream`.
 * [qmoe.rs QMoEKernel::execute: validate the inputs, route, group by expert,
 * run fc1 + activation, fc2 and the weighted combine on the stream; no host
 * synchronisation while capturing]
 *   x_dev       D [num_tokens, H]
 *   logits_dev  float32 [num_tokens, E]
 *   out_dev     D [num_tokens, H] (written)
 * x_dev and out_dev must be 16-byte aligned (INVALID_ARG otherwise).
 * num_tokens == 0 returns QMOE_OK without launching anything.  Both fcs
 * must have been prepacked.  No host synchronisation.
 */
qmoe_status qmoe_forward(qmoe_layer* layer, const void* x_dev, const float* logits_dev,
                         void* out_dev, int64_t num_tokens, void* stream);

/*
 * The same forward on HOST buffers: copies x and logits to the device,
 * runs qmoe_forward, copies out back and synchronises `stream`.  Pinned host
 * memory makes the copies asynchronous DMA; pageable memory also works.
 *   x_host D [num_tokens, H], logits_host float32 [num_tokens, E],
 *   out_host D [num_tokens, H].
 */
qmoe_status qmoe_forward_host(qmoe_layer* layer, const void* x_host, const float* logits_host,
                              void* out_host, int64_t num_tokens, void* stream);

/*
 * Routing of the last forward (device pointers, any may be NULL), enqueued
 * on `stream`.  [qmoe.rs launch_route (route indices and weights) and
 * launch_grouping (per-expert counts, offsets, grouped routes)]
 *   ids_dev     int32 [T*k]  selected experts, slot order (rank)
 *   weights_dev float32 [T*k]
 *   perm_dev    int32 [T*k]  routes grouped by expert, ascending r inside
 *   offsets_dev int32 [E+1]  exclusive offsets into perm
 */
qmoe_status qmoe_get_routing(qmoe_layer* layer, int32_t* ids_dev, float* weights_dev,
                             int32_t* perm_dev, int32_t* offsets_dev, void* stream);

/*
 * Tile work-list of the last forward for one kernel class (which = 0: the
 * decode kernel, 1: the tensor-core grouped GEMM), enqueued on `stream`.
 *   items_dev  int32 [capacity][4]: (expert, row_start, rows, 0), experts
 *              ascending, then row_start; row_start indexes the grouped
 *              (permuted) route order.  Each item covers at most
 *              *m_tile_host rows.
 *   count_dev  int32 [1]: the number of items.
 *   m_tile_host (host, may be NULL): rows per item of that class.
 * Returns INVALID_ARG if capacity is below the worst-case item count
 * (qmoe_worklist_capacity).
 */
qmoe_status qmoe_get_worklist(qmoe_layer* layer, int which, int32_t* items_dev,
                              int32_t* count_dev, int64_t capacity, int* m_tile_host,
                              void* stream);

/* Worst-case item count of work-list `which` for num_tokens tokens. */
int64_t qmoe_worklist_capacity(const qmoe_layer* layer, int which, int64_t num_tokens);

/*
 * Record cudaEvent_t events[QMOE_TRACE_NUM_EVENTS] (passed as void*) on the
 * forward's stream at the stage boundaries QMOE_TRACE_*.  NULL disables.
 * The events are owned by the caller and must outlive their use.
 */
qmoe_status qmoe_set_trace_events(qmoe_layer* layer, void* const* events, int n);

/* Read (and clear) the device status words: QMOE_OK, or QMOE_ERR_TIMEOUT if
 * a bounded wait inside a kernel ran out -- in this layer's forwards, or in
 * any qmoe_forward_noalloc call of this context since the last poll (that
 * entry point's word is shared by all layers).  Synchronises the device.
 * [qmoe.rs QMoEKernel::execute reports device-side failures when the eager
 * pass synchronises its stream; the pages have no device status word, so
 * this word, set by the bounded waits of these kernels, is the library's own
 * counterpart of that report] */
qmoe_status qmoe_poll_device_status(qmoe_layer* layer);

/* The iteration limit of bounded device-side waits (0 = the default, about
 * 2^24 polls).  Tests lower it so an injected stall ends quickly. */
qmoe_status qmoe_set_wait_limit(qmoe_layer* layer, int64_t iterations);

/*
 * Size of the library's static scratch array used by qmoe_forward_noalloc.
 */
#define QMOE_NOALLOC_SCRATCH_BYTES (4u << 20)

/*
 * qmoe_forward without any allocation.  (No counterpart in the pages: this
 * is a convenience of this library.)
 *
 * Who needs it: callers that may not call cudaMalloc at the moment they run
 * the layer -- runtimes whose caching allocator owns all device memory (a
 * cudaMalloc from a library beside it can fail or fragment that pool),
 * embedded or safety-certified deployments with a fixed memory plan decided
 * before start-up, and code that runs where an allocation would stall other
 * work.  qmoe_forward would allocate its workspace on first use (or when
 * num_tokens outgrows qmoe_reserve); this entry point instead uses one
 * file-scope device array of QMOE_NOALLOC_SCRATCH_BYTES that every GPU
 * loading the library holds until the process exits.  It never calls
 * cudaMalloc, cudaFree or any allocating library routine.
 *
 * Arguments and layouts are those of qmoe_forward (x_dev, logits_dev,
 * out_dev are device pointers owned by the caller; x and out 16-byte
 * aligned).  The layer must already be prepacked.  Only the weight-streaming
 * decode kernels run (no grouped GEMM); the output matches qmoe_forward's
 * within the output tolerance (not necessarily bit for bit).  Returns
 * UNSUPPORTED (with the byte count in qmoe_last_error) when num_tokens needs
 * more scratch than the array holds; use qmoe_forward for such sizes.
 *
 * Set-up: the first call on a device (per CUDA context), with that device
 * current, looks up the array's device address (cudaGetSymbolAddress) and
 * caches it; a call in a new context (e.g. after cudaDeviceReset) looks it up
 * again.  All calls share the one array and it keeps the last call's
 * contents: calls that overlap on the GPU (other streams, other layers) race
 * and must be serialised by the caller.
 *
 * Failures: a bounded device-side wait that runs out in this entry point sets
 * a status word at the start of the array (shared by every layer); it stays
 * set until qmoe_poll_device_status of any layer reads and clears it, which
 * then returns QMOE_ERR_TIMEOUT.  Routing of such a call is not kept for
 * qmoe_get_routing.
 */
qmoe_status qmoe_forward_noalloc(qmoe_layer* layer, const void* x_dev, const float* logits_dev,
                                 void* out_dev, int64_t num_tokens, void* stream);

/* Test hook for failure detection without a GPU fault: while enabled, the
 * projection kernels arm their first copy-stage barrier but never issue that
 * copy (every warp of the decode kernel; the producer of every grouped-GEMM
 * CTA), so the bounded waits on it run out; the kernel records
 * QMOE_ERR_TIMEOUT (see qmoe_poll_device_status), waits for its other copies
 * (and MMAs), frees its tensor memory and returns.  Results of such forwards
 * are meaningless.  0 disables. */
qmoe_status qmoe_debug_inject_stall(qmoe_layer* layer, int enable);

/* Message of the last failed call on `layer` ("" if none); static strings
 * for NULL layers. */
const char* qmoe_last_error(const qmoe_layer* layer);

/* Human-readable name of a status code. */
const char* qmoe_status_string(qmoe_status status);

/* Free every device buffer of the layer (synchronises the device).
 * [qmoe.rs `impl Drop for QMoEKernel`: frees every scratch slot] */
void qmoe_destroy(qmoe_layer* layer);

#ifdef __cplusplus
}
#endif
#endif /* QMOE_H_ */
