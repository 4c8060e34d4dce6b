/*
 * lora_layer.h -- C ABI of the mixed-adapter LoRA linear layer on GB300 (sm_103a).
 *
 * The layer computes, for every token row i of a batch,
 *
 *     y[i,:] = x[i,:] W  +  [slot_i != -1] * (alpha_s / r_s) * (x[i,:] A_s) B_s,   s = slot_i
 *
 * where W [K,N] is the shared base weight, A_s [K,r_s] and B_s [r_s,N] are the adapter
 * held in slot s, and slot_i = -1 means "base only".
 *   - "Serving multiple LoRAs: segmented matrix multiplies and adapter scheduling",
 *     section "Not merging the weights, computing in batches": y = xW + s(xA)B with
 *     A in R^{d x r}, B in R^{r x d'}; the base product is one multiply for the whole
 *     batch; BGMV gathers each token's A and B (decode), SGMV groups same-adapter tokens
 *     into segments (prefill); real kernels shrink to rank r, then expand and add.
 *   - "LoRAX, in depth", section "Computing a batch that mixes adapters": s = alpha / r;
 *     segment boundaries of length n_segments + 1 with an owner per segment; an owner of
 *     "None" means base only.
 *   - "Serving LoRA adapters: from the model name to the wrapped layer" (vLLM), Step 3
 *     (activation copies A and B into a fixed number of stacked slot buffers sized for
 *     the maximum rank; more adapters than slots or a rank above the maximum is an
 *     error) and Step 5 (a token without an adapter gets slot -1).
 *
 * Conventions for every call:
 *   - All matrices are dense and row-major (C order).  Element type is the layer's
 *     dtype: LORA_BF16 (bfloat16, computed with fp32 accumulation; y is rounded to
 *     bf16 once, round-to-nearest-even) or LORA_F32 (fp32 throughout).
 *   - "stream" arguments are cudaStream_t values passed as void* (NULL = legacy
 *     default stream).  Calls enqueue work and return without synchronising, except
 *     where a call says it synchronises.
 *   - Return value: LORA_OK or a negative lora_status.  Host-detectable errors are
 *     returned at once and enqueue nothing.  Device-detectable errors (a token id outside
 *     [-1, num_slots), a token naming a slot that holds no adapter) never trap: the
 *     row is treated as base only and a device flag is set; lora_get_status reports it.
 *   - A layer object is not thread-safe: calls on one layer come from one host thread.
 */
#ifndef LORA_LAYER_H
#define LORA_LAYER_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct lora_layer lora_layer_t; /* opaque */

enum lora_dtype { LORA_F32 = 0, LORA_BF16 = 1 };

enum lora_status {
    LORA_OK = 0,
    LORA_EINVAL = -1,   /* bad argument: null pointer, size, dtype, T above max_tokens ... */
    LORA_ESLOT = -2,    /* slot index outside [0, num_slots) */
    LORA_ERANK = -3,    /* adapter rank outside [1, max_rank] */
    LORA_EID = -4,      /* (device) a token id outside [-1, num_slots) or naming an empty slot */
    LORA_ECUDA = -5,    /* a CUDA runtime call failed; lora_last_error has the message */
    LORA_ENOMEM = -6,   /* device or host allocation failed */
    LORA_ESTATE = -7,   /* call out of order: lora_forward without matching set_batch_segments */
    LORA_ETIMEOUT = -8, /* (device) a pipeline wait inside a kernel gave up; results invalid */
    LORA_ENOENT = -9,   /* (adapter cache) adapter id not held in the host tier */
    LORA_ECAPACITY = -10, /* (adapter cache) more distinct adapters than GPU slots */
    LORA_EBOUNDS = -11  /* (device, debug flavour only) a kernel index fell outside its
                           buffer; the access was skipped and the results are invalid */
};

/*
 * Create a layer for a K -> N projection with a table of num_slots adapter slots, each
 * max_rank wide, for batches of at most max_tokens rows.
 *   W_dev      [K,N] base weight in device memory, read during this call only: the layer
 *              keeps its own packed copy (bf16: transposed to [N,K] for the tensor-core
 *              operand layout; f32: [K,N]).
 *   stream     stream on which the packing copy runs; the call synchronises it.
 * Limits: K, N >= 1; for LORA_BF16, K and N are multiples of 8 (16-byte rows for TMA).
 * 1 <= num_slots <= 4096; 1 <= max_rank <= 128; 1 <= max_tokens <= 1<<20.
 * All slots start empty.  The layer owns every buffer it allocates (slot table, batch
 * scratch, staging for host-buffer calls) and frees them in lora_layer_destroy.
 * Errors: LORA_EINVAL, LORA_ENOMEM, LORA_ECUDA (then *out is NULL).
 */
int lora_layer_create(lora_layer_t** out, int K, int N, int num_slots, int max_rank,
                      int max_tokens, int dtype, const void* W_dev, void* stream);

/*
 * As lora_layer_create for bf16 activations and adapters, with the base product in e4m3
 * ("Multi-LoRA Serving 与 Adapter 隔离", section on quantisation: an FP8 base with an FP16
 * LoRA is the usual mixed precision; the quantised product and the LoRA term meet in the
 * kernel's accumulator and epilogue, and the float delta is never added to the packed
 * quantised weights).  For every row i and column n:
 *     y[i,n] = bf16( sx[i] sw[n] sum_k xq[i,k] wq[k,n]  +  low-rank term of x[i] )
 *   - W_dev [K,N] bf16 is quantised once here, per column: sw[n] = max_k |W[k,n]| / 448
 *     (1 for a zero column), wq = e4m3(W / sw), round to nearest even, saturating;
 *   - each forward quantises x per row the same way (sx[i] = max_k |x[i,k]| / 448) in a
 *     kernel of its own before the low-rank kernel; scales and divisions are fp32;
 *   - the low-rank term is computed from the bf16 x as in a plain layer;
 *   - the base runs as e4m3 x e4m3 tcgen05 MMAs (kind::f8f6f4) with fp32 accumulation;
 *     in batches of more than 512 rows the low-rank expand's bf16 MMAs add to the base's
 *     accumulator after the base product is scaled there.
 * Limits: K a multiple of 16.  The packed weight takes K x N bytes.
 * Errors: as lora_layer_create.
 */
int lora_layer_create_fp8(lora_layer_t** out, int K, int N, int num_slots, int max_rank,
                          int max_tokens, const void* W_dev, void* stream);

/*
 * As lora_layer_create, with adapters stored at their true rank in a row pool instead of
 * one max_rank-wide block per slot ("Multi-LoRA Serving: Architecture for Thousands of
 * Adapters", sections on heterogeneous ranks and S-LoRA's kernels: a rank-8 and a rank-64
 * adapter in one batch without padding every adapter to the maximum rank; the adapters are
 * kept in a non-contiguous, ragged layout the kernels index per request).
 *   pool_rows  rank rows of the pool, rounded up to 8: at least max_rank rounded up to 8, at
 *              most num_slots times that.  The A pool takes pool_rows x K and the B pool
 *              pool_rows x N elements (a plain layer: num_slots x max_rank rounded to 8).
 * A load takes the adapter's rank rounded up to 8 consecutive rows, first fit, after
 * returning the rows its slot held; an unload returns them.  A load that finds no such run
 * of free rows fails with LORA_ENOMEM and leaves the slot as it was.  Every kernel reads a
 * slot from its first row, so results equal those of a plain layer.  Adapter caches do
 * not manage pooled layers.
 * Errors: as lora_layer_create; LORA_EINVAL for pool_rows out of range.
 */
int lora_layer_create_pooled(lora_layer_t** out, int K, int N, int num_slots, int max_rank,
                             int max_tokens, int dtype, const void* W_dev, void* stream,
                             int pool_rows);

/*
 * The layer's pool rows in use (held by loaded slots; a plain layer: all of them) and in
 * total.  Host bookkeeping only, no synchronisation.  Errors: LORA_EINVAL (null).
 */
int lora_get_pool_usage(const lora_layer_t* layer, int* used_rows, int* pool_rows);

/*
 * Copy one adapter into slot `slot` ("activation" in vLLM's Step 3).
 *   A_src      [K,r] row-major, B_src [r,N] row-major, the layer's dtype.  Host (pinned
 *              for a truly asynchronous copy) or device memory; it must stay valid and
 *              unchanged until side_stream has executed the copy.
 *   r          the adapter's true rank, 1 <= r <= max_rank; the slot is zero-padded to
 *              max_rank and kernels read only its first r rank columns.
 *   alpha      LoRA alpha; the slot's scale is alpha / r, computed in fp32 and applied in
 *              fp32 to the rank-r intermediate (it is not folded into B).
 * (The same as load_adapter_slot_composed with one member of weight 1.)
 * Ordering: the copy waits for the most recent lora_forward of this layer, so an adapter
 * is never overwritten under a kernel still reading the slot; the next lora_forward waits
 * for the copy.  Loading into an occupied slot replaces its adapter.
 * Errors: LORA_ESLOT, LORA_ERANK, LORA_EINVAL (null), LORA_ECUDA.
 */
int load_adapter_slot(lora_layer_t* layer, int slot, const void* A_src, const void* B_src,
                      int r, float alpha, void* side_stream);

/*
 * Copy a composition of n adapters into slot `slot`: rows of this slot add
 *     sum_i weight[i] * (alpha[i] / r[i]) * (x A_i) B_i
 * to the base product.  "Multi-LoRA Serving 与 Adapter 隔离", section on adapter ownership
 * in a continuous batch: a request may compose several LoRAs, which are added, and its
 * identity is the ordered composition with its weights.
 *   A_src[i]   [K, r[i]] row-major, B_src[i] [r[i], N] row-major, the layer's dtype, host or
 *              device memory (as load_adapter_slot).
 *   r[i] >= 1, sum_i r[i] <= max_rank.  alpha[i], weight[i]: any fp32 values.
 * The members are stacked along the rank axis of the slot (member i takes the r[i] rank
 * columns after those of members 0 .. i-1), each column with its own fp32 scale
 * weight[i] * alpha[i] / r[i], applied to the rank-wide intermediate in fp32 (B is not
 * rescaled, so the stored weights are not re-rounded).  Every kernel then serves the slot like one adapter of rank
 * sum_i r[i].  load_adapter_slot is the case n = 1, weight 1.
 * Ordering: as load_adapter_slot.  A layer whose slots all hold plain adapters runs a
 * decode kernel that reads one scale per slot; the first composition with unequal column
 * scales switches the layer's later forwards to the per-column variant, so a forward
 * captured in a CUDA graph before that must be captured again.
 * Errors: LORA_ESLOT, LORA_ERANK (a member's rank, or the sum, out of range), LORA_EINVAL
 * (n < 1, null arrays or pointers), LORA_ECUDA.
 */
int load_adapter_slot_composed(lora_layer_t* layer, int slot, int n, const void* const* A_src,
                               const void* const* B_src, const int* r, const float* alpha,
                               const float* weight, void* side_stream);

/*
 * Mark slot `slot` empty (rows naming it are then flagged and computed base only).
 * Ordered after the most recent lora_forward, like a load.  Errors: LORA_ESLOT, LORA_ECUDA.
 */
int unload_adapter_slot(lora_layer_t* layer, int slot, void* side_stream);

/*
 * Set the batch: each row's slot, and its segment layout on the device.
 *   token_slot_dev  [T] int32 in device memory: each row's slot, -1 = base only.
 *   T               0 <= T <= max_tokens (T = 0 is an empty batch).
 * The layout stably sorts the adapted rows by slot (ascending slot, original row order
 * within a slot; base-only rows excluded; slots with no rows get no segment) into a row
 * permutation, segment offsets (n_seg + 1) and each segment's slot, in layer-owned device
 * memory, built by one kernel on `stream`.  bf16 batches of more than 512 rows (and every
 * fp32 batch) need it and get it here; bf16 batches of at most 512 rows are computed from
 * the ids alone, so their layout is built only when lora_get_segments asks for it.
 * The next lora_forward on the same stream uses this batch.  token_slot_dev is borrowed:
 * it must stay valid until that forward has run, and, for batches of at most 512 bf16
 * rows, until the next set_batch_segments (lora_get_segments may read it).
 * Errors: LORA_EINVAL, LORA_ECUDA.
 */
int set_batch_segments(lora_layer_t* layer, const int32_t* token_slot_dev, int T, void* stream);

/*
 * y = x W + per-row LoRA delta, for the batch described by the last set_batch_segments.
 *   x_dev   [T,K] device, y_dev [T,N] device (overwritten; must not overlap x_dev).
 *   T       must equal the T of the last set_batch_segments (else LORA_ESTATE).
 * Enqueues the low-rank kernel and the base GEMM (bf16: tensor cores), which adds the
 * low-rank term to its fp32 accumulator and writes y once:
 *   bf16, T <= 512 (decode)  BGMV: per slot, v = (alpha/r) x A_slot and delta = v B_slot in
 *                            fp32 for the slot's rows; the GEMM epilogue adds delta.  Rows
 *                            whose id is outside [-1, S) or names an empty slot are
 *                            computed base only and flagged (lora_get_status).
 *   bf16, T > 512 (prefill)  SGMV shrink on the tensor cores per window of the segment
 *                            layout, v in fp32; the GEMM multiplies v (split into two bf16
 *                            parts) by B_slot as extra K blocks of its own accumulation.
 *   fp32                     SGMV shrink per segment tile, v in fp32; the GEMM epilogue
 *                            expands it.
 * No host synchronisation; no allocation; safe to capture in a CUDA graph.
 * Errors: LORA_EINVAL, LORA_ESTATE, LORA_ECUDA.
 */
int lora_forward(lora_layer_t* layer, const void* x_dev, void* y_dev, int T, void* stream);

/*
 * The whole layer for callers holding host buffers: copies x_host [T,K] and
 * token_slot_host [T] to layer-owned device staging, runs set_batch_segments and
 * lora_forward, and copies y back to y_host [T,N].  All on `stream`, asynchronously:
 * host buffers (pinned for overlap) must stay valid until the stream has completed.
 * Errors: as set_batch_segments and lora_forward.
 */
int lora_forward_host(lora_layer_t* layer, const void* x_host, const int32_t* token_slot_host,
                      void* y_host, int T, void* stream);

/*
 * Synchronise `stream`, read and clear the layer's device error flags.
 * Returns LORA_OK, LORA_EID (bad or empty-slot token ids since the last call) or
 * LORA_ETIMEOUT (a kernel pipeline wait gave up), or LORA_ECUDA.
 */
int lora_get_status(lora_layer_t* layer, void* stream);

/*
 * Copy the current segment layout to host memory (synchronises `stream`; first builds the
 * layout on `stream` if the batch's set_batch_segments did not).
 *   perm [max_tokens], seg_offsets [num_slots + 1], seg_slot [num_slots]: caller-owned
 *   host arrays; *n_seg and *n_adapted receive the segment count and the number of
 *   adapted rows (perm[0..n_adapted) and seg_offsets[0..n_seg] are meaningful).
 * Errors: LORA_EINVAL, LORA_ESTATE (no batch set), LORA_ECUDA.
 */
int lora_get_segments(lora_layer_t* layer, int32_t* perm, int32_t* seg_offsets,
                      int32_t* seg_slot, int32_t* n_seg, int32_t* n_adapted, void* stream);

/*
 * Optional tracing of the layer's kernel launches (for timing on the launch stream).
 *   events   NULL to stop tracing, or an array of 6 cudaEvent_t (as void*) owned by the
 *            caller; afterwards every set_batch_segments records events[0] before and
 *            events[1] after the segment-builder launch (back to back when the batch
 *            needs no builder), and every lora_forward records
 *            events[2] / events[3] around the low-rank kernel launch and events[4] /
 *            events[5] around the base-GEMM launch, each on the call's stream.
 * Tracing adds event records only; it changes no result (the records between kernels
 * make each kernel wait for the previous one to finish, so traced kernels do not
 * overlap).  Errors: LORA_EINVAL.
 */
int lora_set_trace_events(lora_layer_t* layer, void* const* events);

/*
 * Tuning and testing hook: fix the tiling of the bf16 base GEMM (y = x W plus the low-rank
 * term) for the layer's later forwards, instead of the automatic plan.  It changes no
 * result beyond fp32 summation order; the automatic plan is the fast choice.
 *   block_n    N tile of a CTA: 64, 128 or 256; 0 restores the automatic plan.
 *   k_split    K ranges per output tile: 1, 2 or 4, with block_n / k_split >= 32; used for
 *              batches of at most 512 rows (larger ones never split K).
 *   cta_pair   1: pairs of CTAs share 256-row tiles (tcgen05 cta_group::2); needs
 *              block_n >= 128.
 * A forward fails with LORA_ECUDA when the fixed plan cannot run its batch (a K range that
 * would be empty).  Growing the split-K scratch for the new plan synchronises the device.
 * Errors: LORA_EINVAL (other values), LORA_ENOMEM, LORA_ECUDA.
 */
int lora_set_gemm_plan(lora_layer_t* layer, int block_n, int k_split, int cta_pair);

/*
 * The segment builder of set_batch_segments for callers that cannot allocate device memory
 * (a framework or engine that owns all device memory through its own pool and forbids
 * allocations behind its back, or a latency-critical path that cannot afford cudaMalloc's
 * implicit synchronisation).  The pages have no counterpart to this entry point: it is a
 * deployment aid of this library.
 *   token_slot_dev   [T] int32 device ids, -1 = base only; 0 <= T <= 16384.
 *   num_slots        1 <= num_slots <= 1024.
 *   slot_loaded_dev  [num_slots] int32 device flags (0 = slot empty) or NULL (every slot in
 *                    range holds an adapter).
 *   perm_dev [T], seg_offsets_dev [num_slots + 1], seg_slot_dev [num_slots],
 *   counts_dev [3]   caller-owned device outputs: the same permutation, offsets and
 *                    per-segment slots as set_batch_segments computes, and counts_dev =
 *                    {n_seg, n_adapted, error flags} (flags nonzero when an id is outside
 *                    [-1, num_slots) or names an empty slot; such rows count as base only).
 * Allocates nothing: the builder's scratch is one static device array (96 KB on every GPU
 * that loads the library, held until exit).  The first call on a device looks up that
 * array's address with the device current; make it before any stream capture.  Calls
 * share the array and it keeps the last call's contents; calls that overlap on the GPU
 * race on it.  Enqueued on `stream`, no synchronisation.
 * Errors: LORA_EINVAL (sizes above the limits, null pointers), LORA_ECUDA.
 */
int lora_build_segments_static(const int32_t* token_slot_dev, int T, int num_slots,
                               const int32_t* slot_loaded_dev, int32_t* perm_dev,
                               int32_t* seg_offsets_dev, int32_t* seg_slot_dev,
                               int32_t* counts_dev, void* stream);

/*
 * Self-test of the bounded waits that every pipeline kernel of this library uses (the pages
 * have no counterpart).  Runs one kernel on `stream` whose wait nothing will complete --
 * which = 0: a flag in global memory (as the stream-K hand-over), 1: an mbarrier phase (as
 * the TMA / MMA / epilogue pipelines) -- and synchronises `stream`.  The wait gives up
 * after its bound (2 s of global time), raises the timeout flag and returns, so the call
 * takes ~2 s and returns LORA_ETIMEOUT, the expected result; the context stays usable.
 * LORA_OK would mean the wait completed.  Allocates 8 bytes of device memory for the call.
 * Errors: LORA_EINVAL (which), LORA_ENOMEM, LORA_ECUDA.
 */
int lora_wait_selftest(int which, void* stream);

/* Text of the last error raised on this layer ("" if none).  Owned by the layer. */
const char* lora_last_error(const lora_layer_t* layer);

/*
 * Kernels this layer has launched since its last set_batch_segments (that call's segment
 * builder, if it ran, then every lora_forward and lora_get_segments on the batch), e.g.
 * 2 for a bf16 decode forward (BGMV, base GEMM), 3 when the GEMM runs as two launches or
 * the base is e4m3 (its row quantiser).  -1 for NULL.
 */
int lora_get_launch_count(const lora_layer_t* layer);

/* Synchronise the layer's device, then free everything the layer owns.  NULL is a no-op. */
void lora_layer_destroy(lora_layer_t* layer);

#ifdef __cplusplus
}
#endif

#endif /* LORA_LAYER_H */
