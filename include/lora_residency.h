/*
 * lora_residency.h -- C ABI of the adapter cache: two residency tiers (pinned host memory,
 * GPU slots) over the slot tables of one or more lora_layer objects.
 *
 * A model applies one adapter to many projections, so an adapter here is one (A, B) pair
 * per layer of a set of layers that share their slot numbering: adapter `id` sits in the
 * same slot s of every layer, and a batch's rows name adapters by id; the cache turns those
 * ids into the slot ids that set_batch_segments takes.
 *
 * Where the pages define the behaviour:
 *   - "Serving LoRA adapters: from the model name to the wrapped layer" (vLLM), Step 3:
 *     a batch naming more adapters than GPU slots is an error; an adapter missing from
 *     the CPU cache is loaded there first, and is validated (rank against the maximum)
 *     before anything is evicted; a full CPU cache drops its oldest adapter; activation
 *     copies an adapter into the first free slot, and when every slot is taken the least
 *     recently used active adapter is deactivated first; a cache hit only refreshes the
 *     adapter's recency.
 *   - "Multi-LoRA Serving: Architecture for Thousands of Adapters", sections "Unified
 *     paging of adapters and KV cache" and "Trade-offs, Gotchas, and What Goes Wrong":
 *     every adapter lives in host DRAM, the ones in use are fetched into HBM and cold ones
 *     evicted; a DRAM-to-HBM promotion is a bus copy of a millisecond or so, hidden when
 *     the fetch runs while the previous batch computes.
 *   - "LoRAX, in depth", section "Adapter exchange scheduling": adapters with queued work
 *     are prefetched asynchronously.
 *   - "Multi-LoRA Serving 与 Adapter 隔离", section on failure modes: an adapter must not
 *     be evicted while a kernel still reads its storage.
 *
 * Readings where the pages leave a step open:
 *   - The adapters of one batch are made resident in the order of their first row.
 *     Recency is one counter over both tiers: a batch (or prefetch) touches its adapters
 *     in that order, so the first-named is the least recent of them afterwards.
 *   - The host tier holds every adapter that may be GPU-resident; dropping an adapter from
 *     it (oldest first, whether or not it is resident) also empties its GPU slot.
 *   - An adapter added again under the same id replaces the old weights (vLLM's in-place
 *     load); if it was resident its slot is emptied and the next batch swaps the new
 *     weights in.
 *
 * Swap-in (DRAM -> HBM): an adapter's weights are packed at lora_cache_add time into the
 * slot layout of every layer (A transposed and zero-padded to the slot width, B padded), in
 * one pinned host block.  A swap-in is one host-to-device copy of that block into a device
 * staging buffer and one kernel that scatters it into the slot of every layer and sets the
 * slots' column scales (alpha / r), rank and loaded flag, both on the cache's own stream,
 * created at the lowest priority.
 *
 * Ordering is per slot, so that a swap-in runs beside the batch in flight unless it
 * replaces one of that batch's adapters:
 *   - lora_cache_map_batch(..., stream) first records a point on `stream`.  Everything the
 *     caller enqueued there before the call -- the previous batch's forwards, on `stream`
 *     or on streams joined into it -- ends the previous batch's use of its slots.  A
 *     swap-in into a slot waits for the point that ended the slot's last use.
 *   - Then `stream` waits for the swap-ins into the batch's own slots (and no others):
 *     enqueue the batch's set_batch_segments / lora_forward calls on `stream` (or on
 *     streams that wait for it) after the call.
 *   - Until the next lora_cache_map_batch the batch's slots count as in flight: a prefetch
 *     never takes them, and an adapter removed from one (lora_cache_remove, replaced, or
 *     dropped from the host tier) leaves the slot blocked -- still holding the old weights
 *     -- until the next batch point, which empties it.
 * Consecutive batches of a cache use one stream (or the caller joins the earlier batches'
 * streams into the later one).  Forwards replayed from a CUDA graph count like any other
 * work on the stream they are replayed on.
 *
 * Conventions: as lora_layer.h (status codes, no thread safety: one host thread per cache
 * and its layers).  While a cache manages a set of layers, their slots [0, num_slots) must
 * be loaded only through the cache.
 */
#ifndef LORA_RESIDENCY_H
#define LORA_RESIDENCY_H

#include <stdint.h>

#include "lora_layer.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct lora_adapter_cache lora_adapter_cache_t; /* opaque */

typedef struct lora_cache_stats {
    int64_t hits;           /* batch adapters found resident by lora_cache_map_batch */
    int64_t misses;         /* batch adapters swapped in by lora_cache_map_batch */
    int64_t prefetches;     /* adapters swapped in by lora_cache_prefetch */
    int64_t gpu_evictions;  /* resident adapters whose slot was given to another adapter */
    int64_t host_evictions; /* adapters dropped from the host tier to make room */
    int64_t bytes_swapped;  /* host-to-device bytes of all swap-ins */
    int32_t resident;       /* adapters in GPU slots now */
    int32_t registered;     /* adapters in the host tier now */
} lora_cache_stats_t;

/*
 * Create a cache over `n_layers` layers (borrowed: they must outlive the cache) that share
 * the slot numbering [0, num_slots).
 *   layers         n_layers layer handles, all on the current device; n_layers = 0 gives a
 *                  cache that only keeps the books (slot assignment, recency, statistics)
 *                  and touches no device: it needs no GPU.  Pooled layers
 *                  (lora_layer_create_pooled: adapters at their true rank) are served: a
 *                  swap-in gives back the rows its slot held and takes the adapter's rank
 *                  rounded up to 8 consecutive rows, first fit, from each pooled layer's
 *                  row pool.  All pooled layers of a cache must have the same pool_rows and
 *                  hold no adapter when the cache is created, and from then on their slots
 *                  change only through the cache (the cache moves their allocators in
 *                  step).  A swap-in that finds no run of free rows fails with LORA_ENOMEM
 *                  and leaves its slot empty (size the pool for the slots' ranks with room
 *                  for fragmentation).
 *   num_slots      1 <= num_slots <= every layer's num_slots (vLLM's max_loras).
 *   host_capacity  adapters the host tier holds (vLLM's max_cpu_loras), >= num_slots.
 * Allocates host_capacity pinned host blocks of the adapter image size (the sum over the
 * layers of R * (K + N) elements of the layer's dtype, R the layer's slot width), one
 * device staging block of that size, a small device table, and its own stream.
 * Errors: LORA_EINVAL (sizes, null or mixed-device layers), LORA_ENOMEM, LORA_ECUDA.
 */
int lora_cache_create(lora_adapter_cache_t** out, lora_layer_t* const* layers, int n_layers,
                      int num_slots, int host_capacity);

/*
 * Put adapter `id` (>= 0) into the host tier: A_host[l] [K_l, r] and B_host[l] [r, N_l],
 * row-major in layer l's dtype, in host memory (read during this call only; device memory
 * is rejected).  r is the adapter's rank (1 <= r <= every layer's max_rank); its scale is
 * alpha / r.  With n_layers = 0 the pointer arrays may be NULL.
 * The arguments are checked before anything is evicted; then, if the tier is full, its
 * least recently used adapter is dropped (and its GPU slot emptied).  An id already held
 * is replaced in place.  Synchronises with any swap-in still reading the reused block.
 * Errors: LORA_EINVAL, LORA_ERANK, LORA_ECUDA.
 */
int lora_cache_add(lora_adapter_cache_t* cache, int64_t id, int r, float alpha,
                   const void* const* A_host, const void* const* B_host);

/*
 * Put a composition of adapters already in the host tier into it under its own id
 * ("Multi-LoRA Serving 与 Adapter 隔离", adapter ownership: a request may compose several
 * LoRAs, which are added; its identity is the ordered members with their weights, so a
 * composition is an adapter of its own here).  Rows naming `id` then add
 *     sum_m weights[m] * (its own scaled delta of member_ids[m])
 * -- the members stacked along the rank axis as load_adapter_slot_composed does, each
 * column keeping its member's scale times the weight.  The image is packed from the
 * members' host blocks at this call (later changes to a member do not reach it).
 *   member_ids[0..n): ids in the host tier (not `id` itself); their ranks sum to at most
 *   every layer's max_rank.
 * Room is made as lora_cache_add does, never by dropping a member.
 * Errors: LORA_EINVAL, LORA_ENOENT (a member), LORA_ERANK (the summed rank),
 * LORA_ECAPACITY (the tier holds only members), LORA_ECUDA.
 */
int lora_cache_add_composed(lora_adapter_cache_t* cache, int64_t id, int n,
                            const int64_t* member_ids, const float* weights);

/*
 * Drop adapter `id` from both tiers.  Its GPU slot, if any, is emptied at once, or, if the
 * last mapped batch uses it, blocked until the next batch point (see "Ordering").
 * Errors: LORA_ENOENT, LORA_ECUDA.
 */
int lora_cache_remove(lora_adapter_cache_t* cache, int64_t id);

/*
 * Make every adapter of a batch GPU-resident and translate the batch's rows to slots.
 *   token_adapter  [T] int64 host: each row's adapter id, -1 = base only.
 *   token_slot     [T] int32 host output: each row's slot, -1 for base-only rows; pass it
 *                  (copied to the device) to set_batch_segments of every layer.
 *   stream         the stream of the batches' forwards (a cudaStream_t; see "Ordering").
 * Checked first, with nothing changed on failure: an id below -1 (LORA_EINVAL), an id not
 * in the host tier (LORA_ENOENT), more distinct adapters than slots (LORA_ECAPACITY).
 * Then the previous batch's point is recorded on `stream`, and, adapter by adapter in the
 * order of their first row: a resident one is a hit; any other takes the lowest free slot,
 * or else the slot of the least recently used resident adapter that this batch does not
 * name, and is swapped in (enqueued, not waited for).  Finally `stream` waits for the
 * batch's swap-ins.  The returned slots stay valid until the next lora_cache_map_batch,
 * lora_cache_add or lora_cache_remove.
 * Errors: as above, LORA_ENOMEM (a pooled layer has no run of free rows for an adapter:
 * that adapter's slot is left empty and the batch is not mapped), LORA_ECUDA.
 */
int lora_cache_map_batch(lora_adapter_cache_t* cache, const int64_t* token_adapter, int T,
                         int32_t* token_slot, void* stream);

/*
 * Swap adapters in ahead of the batches that will need them, e.g. while the current batch
 * computes ("LoRAX, in depth": adapters with queued work are prefetched).  ids[0..n) are
 * made resident in order, taking free slots or those of the least recently used adapters
 * that neither the list nor the last mapped batch names; the swap-ins overlap that batch.
 * Errors (nothing changes): LORA_EINVAL (an id < 0), LORA_ENOENT, LORA_ECAPACITY (more
 * adapters to swap in than slots free or held by other adapters); LORA_ECUDA.
 */
int lora_cache_prefetch(lora_adapter_cache_t* cache, const int64_t* ids, int n);

/* The slot holding adapter `id`, or -1 if it is not GPU-resident (or unknown). */
int lora_cache_slot_of(const lora_adapter_cache_t* cache, int64_t id);

/* Counters since creation and the current occupancy.  Errors: LORA_EINVAL (null). */
int lora_cache_get_stats(const lora_adapter_cache_t* cache, lora_cache_stats_t* out);

/*
 * The cache's stream (a cudaStream_t), on which every swap-in runs; NULL for a cache
 * without layers.  Callers may record events on it to time swap-ins.
 */
void* lora_cache_stream(const lora_adapter_cache_t* cache);

/* Block the host until every swap-in enqueued so far has completed.  Errors: LORA_ECUDA. */
int lora_cache_sync(lora_adapter_cache_t* cache);

/* Text of the last error raised on this cache ("" if none).  Owned by the cache. */
const char* lora_cache_last_error(const lora_adapter_cache_t* cache);

/* Synchronise the cache's stream, then free everything it owns (not the layers).  NULL is
 * a no-op. */
void lora_cache_destroy(lora_adapter_cache_t* cache);

#ifdef __cplusplus
}
#endif

#endif /* LORA_RESIDENCY_H */
