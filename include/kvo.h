/*
 * kvo.h - sparse KV residency for long-context MLA decode on GB300 (sm_103a).
 *
 * One context holds, per layer, the full MLA history in pinned host memory
 * and a fixed-size hot cache in HBM, plus the position->slot tables that
 * connect them.  Per decode step and layer the caller selects the top-K
 * history positions from indexer scores (kvo_select_topk) and resolves them
 * (kvo_resolve_gather): hits are read from the hot cache, misses from host
 * memory, least-recently-used unpinned slots receive the misses, and the K
 * rows are written contiguously in selection order.
 *
 * Sources (page title, section):
 *   [KVO]  "From 1M Total to 15+ x 1M Contexts: GLM-5.3 KV Cache Offloading"
 *   [CORR] "Making KV offload correct" (Running large language models on
 *          dual GH200, post 4)
 *
 * Conventions for every call:
 *   - Device pointers are CUDA device (or managed) memory of the current
 *     device; "host" pointers are ordinary process memory.  `stream` is a
 *     cudaStream_t passed as void* (NULL = the legacy default stream).
 *   - Calls are asynchronous and stream-ordered unless stated otherwise.
 *     Argument errors are detected synchronously, return KVO_EINVAL and
 *     change no state.  Errors found by kernels (for example a selected
 *     position outside the history) are latched in a device status word and
 *     returned by the next kvo_sync.
 *   - The caller owns every buffer it passes (scores, idx, outputs, rows)
 *     and the streams; the context owns the histories, hot caches, tables
 *     and statistics.  A context is not thread-safe; calls on one context
 *     must come from one host thread at a time.
 *   - A Q8G64 MLA row is 656 bytes ([KVO] "Separate historical capacity
 *     from the current working set"): bytes [0,512) int8 latent, [512,528)
 *     eight little-endian fp16 scales (scale g covers latent bytes
 *     [64g, 64g+64)), [528,656) 64 little-endian bf16 RoPE values.
 */
#ifndef KVO_H
#define KVO_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVO_ROW_BYTES 656
#define KVO_LATENT_BYTES 512
#define KVO_DEQUANT_VALUES 576      /* bf16 values per dequantised row */
#define KVO_MAX_K 4096              /* largest selection size per call */
#define KVO_MAX_ROUND 8192          /* most entries in one multi-query round */
#define KVO_COPYBACK_BATCH 64       /* rows per recent-ring copyback */
#define KVO_MAX_HOT_ROWS 131072     /* largest hot cache per layer */

typedef enum kvo_status {
  KVO_OK = 0,
  KVO_EINVAL = -1,     /* bad argument; nothing was changed or enqueued */
  KVO_ENOMEM = -2,     /* a device or pinned-host allocation failed */
  KVO_ECUDA = -3,      /* a CUDA runtime call failed */
  KVO_ERANGE = -4,     /* a kernel saw a selected position outside [0, length) */
  KVO_EBUSY = -5,      /* resource still referenced by in-flight work */
  KVO_ETIMEDOUT = -6,  /* a bounded device-side wait gave up (reported by kvo_sync).  The waiting
                        * CTA waits once more, again bounded; if that wait gives up too, a bulk
                        * copy into its shared memory may still land after it exits, and the
                        * context refuses every later launch (KVO_ECUDA): destroy it and create
                        * a new one. */
  KVO_ECAPACITY = -7   /* not enough blocks; allocation rolled back */
} kvo_status;

typedef struct kvo_ctx kvo_ctx;

/* Per-layer counters, accumulated on the device by every resolve call. */
typedef struct kvo_stats {
  uint64_t steps;          /* resolve calls on the layer */
  uint64_t hits;           /* selected entries found in the hot cache */
  uint64_t misses;         /* selected entries read from host memory (every occurrence) */
  uint64_t unique_misses;  /* distinct missing positions (= hot-cache fills) */
  uint64_t evictions;      /* fills that replaced a mapped position */
  uint64_t invalid;        /* selected entries outside [0, length) */
  uint64_t host_bytes;     /* bytes read from host memory by gathers */
  uint64_t rows_out;       /* rows emitted */
} kvo_stats;

/* Human-readable name of a status code (static string). */
const char* kvo_status_string(kvo_status s);

/*
 * kvo_create - allocate a context on the current device.
 *   layers       >= 1 independent layers (each with its own history and hot
 *                cache: [KVO] "Separate historical capacity ...": layers
 *                that reuse a selection keep their own KV contents).
 *   history_cap  rows of host history per layer, 1 .. 2^31-1 (pinned,
 *                device-mapped host memory, history_cap*656 bytes per layer).
 *   hot_rows     HBM hot-cache rows per layer, 1 .. KVO_MAX_HOT_ROWS
 *                (hot_rows*656 bytes per layer, exact-size allocation).
 *   row_bytes    must be KVO_ROW_BYTES.
 *   out          receives the context; untouched on error.
 * Every hot slot starts empty, every history length at 0.  Synchronous.
 * Errors: KVO_EINVAL, KVO_ENOMEM (everything allocated so far is freed).
 */
kvo_status kvo_create(int32_t layers, int64_t history_cap, int32_t hot_rows,
                      int32_t row_bytes, kvo_ctx** out);

/* kvo_destroy - wait for all work on the device, then free the context. */
kvo_status kvo_destroy(kvo_ctx* ctx);

/*
 * kvo_append_rows - append r rows to a layer's host history at positions
 * [length, length + r), then length += r ([KVO] "Decision three": new KV goes
 * to the RAM history; an appended position is a miss the first time it is
 * selected).
 *   rows   r*656 bytes, 16-byte aligned; device memory (copied by a kernel
 *          in stream order) or host memory (copied before the call returns;
 *          the new length takes effect in stream order).
 * Errors: KVO_EINVAL if layer is out of range, r < 0, length + r exceeds
 * history_cap or rows is NULL with r > 0.
 */
kvo_status kvo_append_rows(kvo_ctx* ctx, int32_t layer, const void* rows, int64_t r,
                           void* stream);

/*
 * Recent ring ([KVO] pipeline "New KV -> GPU recent ring -> batched
 * copyback -> RAM history"; "GPU cache management has hazards too": the ring
 * protects new tokens that have not yet reached RAM).
 * kvo_set_recent_ring(ctx, rows) with rows a power of two in [128, 65536]
 * gives every layer a ring of `rows` HBM rows; 0 removes it (the default:
 * device rows go straight to the host history).  Accepted only before the
 * first append to any layer (else KVO_EBUSY); KVO_ENOMEM if the rings cannot
 * be allocated.  With a ring:
 *   - rows appended from device memory (kvo_append_rows, kvo_decode_step)
 *     wait in the ring, position p in row p mod rows; as soon as
 *     KVO_COPYBACK_BATCH or more are pending, whole batches of them move to
 *     the host history with one or two asynchronous copies on the call's
 *     stream.  At most rows - KVO_COPYBACK_BATCH rows per call.
 *   - rows appended from host memory first move every pending ring row to
 *     the host history, then go there themselves.
 *   - a selected position that misses the hot cache and is not yet in the
 *     host history is read from the ring; kvo_stats.host_bytes counts only
 *     the reads from the host history.
 *   - kvo_decode_step reads the rows it appends from its own input rows and
 *     moves full batches to the host history after its resolve.
 * kvo_flush_ring moves every pending row to the host history (stream-
 * ordered): the point up to which an export of the host history is
 * complete.  kvo_ram_length gives the number of positions the host history
 * holds once the work enqueued so far has run (host only).
 */
kvo_status kvo_set_recent_ring(kvo_ctx* ctx, int32_t rows);
kvo_status kvo_flush_ring(kvo_ctx* ctx, int32_t layer, void* stream);
kvo_status kvo_ram_length(kvo_ctx* ctx, int32_t layer, int64_t* out);

/* Test hook: copies positions [start, start + count) of the layer's host
 * history (RAM) to host memory `out` (synchronises the device first). */
kvo_status kvo_debug_read_history(kvo_ctx* ctx, int32_t layer, int64_t start, int64_t count, void* out);

/*
 * Gather modes: how the selected rows reach the output (and the fills their
 * slots).  KVO_GATHER_LOADS: 16-byte loads into registers (zero-copy loads
 * for rows in host memory).  KVO_GATHER_STAGED: every row of a CTA's share
 * is pulled into shared memory by a TMA bulk copy (all in flight at once,
 * host rows included) and the share written back with one bulk store; used
 * where a CTA's share fits its shared memory, else loads.  KVO_GATHER_AUTO:
 * staged for a CTA whose misses are at least auto_miss_pct percent of its
 * entries, loads otherwise (decided per CTA and call, after classification).
 * Outputs are identical in every mode.  Default: KVO_GATHER_AUTO with 5 %
 * (per 2,048-row call on a full cache the staged gather is as fast below
 * 5 % misses and 0.4-1.4 us faster from 5 % up).  Host only; takes effect
 * from the next call.
 */
#define KVO_GATHER_LOADS 0
#define KVO_GATHER_STAGED 1
#define KVO_GATHER_AUTO 2
kvo_status kvo_set_gather_mode(kvo_ctx* ctx, int32_t mode, int32_t auto_miss_pct);

/*
 * kvo_set_miss_fetch - how kvo_decode_layers fetches the misses whose rows
 * are in the host history ([KVO] "Decision two": per-row transfers cost more
 * than their bytes, batching them paid; "Decision three": misses read the
 * registered host memory directly).
 *   KVO_MISS_ZEROCOPY  the gathers read the rows over the host link with
 *                      16-byte loads, in the same launch (default);
 *   KVO_MISS_BATCHED   the resolves list the missing positions; the call
 *                      waits for the list on the host, copies every run of
 *                      consecutive positions with one cudaMemcpyAsync into
 *                      device staging, and a placement launch writes the rows
 *                      out and fills their victim slots (the call returns
 *                      only after the resolves ran);
 *   KVO_MISS_AUTO      batched while the last measured miss share of the
 *                      calls is at least auto_miss_pct percent, else
 *                      zero-copy (the share comes from statistics copied back
 *                      asynchronously after each call; it lags by a call or
 *                      two).
 * Results are identical in every mode.  KVO_EINVAL for another mode or a
 * percentage outside 0..100.  Other entry points always use zero-copy loads.
 */
#define KVO_MISS_ZEROCOPY 0
#define KVO_MISS_BATCHED 1
#define KVO_MISS_AUTO 2
kvo_status kvo_set_miss_fetch(kvo_ctx* ctx, int32_t mode, int32_t auto_miss_pct);

/*
 * Replacement policies ([KVO] "GPU cache management has hazards too").  In
 * both, the slots used by a round (its hits, and the slots it fills) are
 * pinned, and the round's distinct missing positions, in first-occurrence
 * order, take the victims in the policy's order:
 *   KVO_POLICY_LRU       the unpinned slots by (last_use, slot) ascending
 *                        (the default);
 *   KVO_POLICY_CIRCULAR  the unpinned slots in circular slot order starting
 *                        at the layer's hand; the hand then moves past the
 *                        last victim (the pages' final rule).
 * kvo_set_policy applies to every layer of the context and is accepted only
 * before the context's first resolve (else KVO_EBUSY); KVO_EINVAL for an
 * unknown policy.  Host only.
 */
#define KVO_POLICY_LRU 0
#define KVO_POLICY_CIRCULAR 1
kvo_status kvo_set_policy(kvo_ctx* ctx, int32_t policy);

/*
 * kvo_select_topk - the k highest of n fp32 scores ([KVO] "Separate
 * historical capacity ...": the indexer selects the top 2,048 positions).
 *   scores  device fp32[n].
 *   idx     device int32[k]; receives the chosen positions in ascending
 *           order.
 * Order: higher score first, equal scores -> lower position first; -0.0
 * equals +0.0; NaN ranks below every other value (NaNs tie by position).
 * Errors: KVO_EINVAL unless 0 < k <= n, k <= KVO_MAX_K and n < 2^31, or if
 * scores or idx is not 4-byte aligned.
 */
kvo_status kvo_select_topk(kvo_ctx* ctx, const float* scores, int64_t n, int32_t k,
                           int32_t* idx, void* stream);

/*
 * kvo_select_topk_batch - kvo_select_topk for nq rows of scores in one
 * launch (one thread-block cluster per row): the rows of a multi-query
 * round ([KVO] "GPU cache management has hazards too": MTP verification
 * selects for several query rows).
 *   scores  device fp32; row q starts at scores + q*ld (ld >= n).
 *   idx     device int32[nq*k]; row q's positions, ascending, at idx + q*k.
 * Errors: KVO_EINVAL unless nq >= 1, ld >= n and kvo_select_topk's limits
 * hold (4-byte aligned scores and idx included).
 */
kvo_status kvo_select_topk_batch(kvo_ctx* ctx, const float* scores, int64_t n, int64_t ld, int32_t nq, int32_t k,
                                 int32_t* idx, void* stream);

/*
 * kvo_resolve_gather - resolve k selected positions of one layer against its
 * hot cache and emit their rows ([KVO] "Decision three: let the GPU manage
 * the hot cache directly" and "GPU cache management has hazards too").
 *   idx       device int32[k], any order, duplicates allowed.
 *   out_rows  device uint8[k*656] (16-byte aligned) or NULL: row j = the
 *             656-byte row of position idx[j].
 *   out_bf16  device uint16[k*576] (16-byte aligned) or NULL: row j =
 *             bf16 round-to-nearest-even of float(q)*float(scale[g]) for
 *             the 512 latent bytes, then the 64 RoPE bf16 values copied.
 * Per call the layer's step counter t advances by one.  Hits (positions with
 * a hot slot) read HBM and stamp last_use = t (pinning the slot for this
 * step).  Misses read host memory, every occurrence.  The distinct missing
 * positions, in first-occurrence order, take the slots with the smallest
 * (last_use, slot) among slots with last_use < t, in that order; the map is
 * updated and each such slot receives its new row, so it becomes a hit
 * source from the next call on.
 * An entry outside [0, length) gets a zero row, changes no state and latches
 * KVO_ERANGE for kvo_sync.
 * Errors: KVO_EINVAL if layer is out of range, k < 1, k > KVO_MAX_K,
 * k > hot_rows, both outputs are NULL, an output is not 16-byte aligned or
 * idx is not 4-byte aligned.
 */
kvo_status kvo_resolve_gather(kvo_ctx* ctx, int32_t layer, const int32_t* idx, int32_t k,
                              void* out_rows, uint16_t* out_bf16, void* stream);

/*
 * kvo_resolve_gather_multi - one round of several query rows ([KVO] "GPU
 * cache management has hazards too": verification with MTP processes
 * several rows, and several queries can select the same missing position).
 *   idx       device int32[nq*k]: row q's selection is idx[q*k .. q*k+k),
 *             rows one after another.
 *   out_rows  device uint8[nq*k*656] or NULL, out_bf16 device
 *             uint16[nq*k*576] or NULL: entry q*k+j in the same order.
 * The round is exactly kvo_resolve_gather over the nq*k entries in that
 * order: the layer's step advances once; the first occurrence of a missing
 * position takes the slot, every later occurrence (in this or another row)
 * reads host memory, and a slot filled in this round is a hit source only
 * from the next round on; every slot the round uses is pinned.
 * Requires 1 <= nq, 1 <= k <= KVO_MAX_K, nq*k <= KVO_MAX_ROUND and
 * nq*k <= hot_rows and a 4-byte aligned idx, else KVO_EINVAL (also when the
 * round does not fit the shared memory of the cluster size in use).
 */
kvo_status kvo_resolve_gather_multi(kvo_ctx* ctx, int32_t layer, const int32_t* idx, int32_t nq, int32_t k,
                                    void* out_rows, uint16_t* out_bf16, void* stream);

/*
 * kvo_decode_layers - one decode step of several layers; each task is what
 * kvo_decode_step does for its layer, except that a task without scores
 * resolves a selection it is given ([KVO] "Separate historical capacity from
 * the current working set": later layers reuse a layer's selection and keep
 * their own KV).  Three launches, each over every task of the call: the
 * top-K of the tasks with scores (after a whole-GPU histogram launch for
 * histories too long for one cluster's shared memory); then, one CTA per
 * task, the lookup, the victims, the map updates, the appends and the LRU
 * queue; then the row gather of every task on the whole GPU, which also
 * fills the victim slots.  Per task:
 *   layer     a layer of the context; at most one task per layer per call.
 *   new_rows  device rows to append first (16-byte aligned), r of them, or
 *             NULL with r = 0.
 *   scores    device fp32[n]: select the top k of them into idx; or NULL:
 *             idx is an input (any order, duplicates allowed, as in
 *             kvo_resolve_gather), and n is ignored.
 *   idx       device int32[k].
 *   out_rows / out_bf16  as in kvo_resolve_gather (at least one).
 * The selections of a call are made before any task resolves: a task
 * without scores may name the idx of a task of the same call that has
 * scores, and then resolves that task's new selection (one call per decode
 * step for a whole stack).  Two tasks with scores must not share an idx.
 * Memory: the context keeps the candidate lists of the selections, about 8
 * bytes per score of the call's tasks with scores, in device memory; a call
 * that needs more than it holds grows them (a device-wide synchronisation,
 * once), and KVO_ENOMEM if that allocation fails.
 * KVO_EINVAL on a bad task (nothing enqueued), misaligned scores or idx
 * (4 bytes) included.
 */
typedef struct kvo_layer_task {
  int32_t layer;
  int32_t reserved;
  const void* new_rows;
  int64_t r;
  const float* scores;
  int64_t n;
  int32_t* idx;
  void* out_rows;
  uint16_t* out_bf16;
} kvo_layer_task;
kvo_status kvo_decode_layers(kvo_ctx* ctx, const kvo_layer_task* tasks, int32_t ntasks, int32_t k, void* stream);

/*
 * Measurement of kvo_decode_layers by its phases.  kvo_set_phase_timing(ctx,
 * 1) makes every later kvo_decode_layers call record CUDA events on its
 * stream around its three launches (selections, resolves, gathers), and run
 * them in order on that one stream (no overlap of the call's parts, no
 * early scheduling of a launch before the previous one ends);
 * kvo_layers_phase_times waits for the recorded calls, adds up the elapsed
 * milliseconds of each phase into ms[0..2], returns the number of calls in
 * *calls and starts a new count.  Off by default; switching it resets the
 * count.  KVO_EINVAL for NULL arguments, KVO_ECUDA if an event call fails.
 */
kvo_status kvo_set_phase_timing(kvo_ctx* ctx, int32_t on);
kvo_status kvo_layers_phase_times(kvo_ctx* ctx, double* ms, int64_t* calls);
/* kvo_layers_counters - since the context was created: the number of
 * kernels kvo_decode_layers has launched, and the host time spent inside its
 * calls (seconds; argument checks, launch set-up and launches). */
kvo_status kvo_layers_counters(kvo_ctx* ctx, int64_t* launches, double* host_seconds);

/*
 * kvo_decode_step - one decode step of one layer in a single launch: the
 * same results as kvo_append_rows(layer, new_rows, r), then
 * kvo_select_topk(scores, n, k, idx), then kvo_resolve_gather(layer, idx, k,
 * out_rows, out_bf16), in that stream order ([KVO] "Decision three": the
 * GPU selects, looks up and gathers with no host round trip).
 *   new_rows  device uint8[r*656] (16-byte aligned), or NULL with r = 0.
 *             Host rows are refused: append them with kvo_append_rows.
 *   scores    device fp32[n]; idx device int32[k] receives the selection
 *             (ascending positions); outputs as for kvo_resolve_gather.
 * Errors: KVO_EINVAL for any argument the three calls would refuse, or for
 * host-memory new_rows.  Nothing is changed or enqueued on an error.
 */
kvo_status kvo_decode_step(kvo_ctx* ctx, int32_t layer, const void* new_rows, int64_t r,
                           const float* scores, int64_t n, int32_t k, int32_t* idx,
                           void* out_rows, uint16_t* out_bf16, void* stream);

/*
 * kvo_decode_step_host - kvo_decode_step with host buffers, for a caller
 * whose inputs and outputs live in host memory.  Page-locked (pinned)
 * buffers are used in place: the step reads the scores and the new rows and
 * writes idx and the outputs over the host link itself, with no copy before
 * or after.  Pageable buffers (and row buffers not 16-byte aligned) go
 * through device staging owned by the context: copied in before the step,
 * out after it.  Everything is in order on `stream`, and the call returns
 * once the work is enqueued: synchronise the stream (kvo_sync) before
 * reading the outputs or rewriting the inputs.
 *   new_rows  host uint8[r*656], or NULL with r = 0.
 *   scores    host fp32[n].
 *   idx       host int32[k] receives the selection (ascending positions).
 *   out_rows  host uint8[k*656] or NULL; out_bf16 host uint16[k*576] or
 *             NULL; at least one.
 * The staging a call needs (scores, rows, idx and outputs) is allocated on
 * first use and grows with r: KVO_ENOMEM if it cannot be.  One staging set per
 * context: calls on different streams must not overlap.  Errors as for
 * kvo_decode_step; nothing is changed or enqueued on an error.
 */
kvo_status kvo_decode_step_host(kvo_ctx* ctx, int32_t layer, const void* new_rows, int64_t r,
                                const float* scores, int64_t n, int32_t k, int32_t* idx,
                                void* out_rows, uint16_t* out_bf16, void* stream);

/*
 * kvo_sync - synchronise `stream`, then return and clear the device status
 * word: KVO_OK, or the first latched device error (KVO_ERANGE, ...).
 */
kvo_status kvo_sync(kvo_ctx* ctx, void* stream);

/* kvo_get_stats - copy a layer's counters to *out (synchronises the device). */
kvo_status kvo_get_stats(kvo_ctx* ctx, int32_t layer, kvo_stats* out);

/* kvo_history_length - a layer's length as of all calls made so far. */
kvo_status kvo_history_length(kvo_ctx* ctx, int32_t layer, int64_t* out);

/*
 * kvo_debug_dump_layer - copy a layer's state to host buffers (any may be
 * NULL): pos2slot int32[history_cap] (-1 = not resident), slot2pos
 * int32[hot_rows] (-1 = empty), last_use uint32[hot_rows] (0 = never),
 * hot uint8[hot_rows*656], step = the layer's step counter.  Synchronises
 * the device.  Meant for tests.
 */
kvo_status kvo_debug_dump_layer(kvo_ctx* ctx, int32_t layer, int32_t* pos2slot,
                                int32_t* slot2pos, uint32_t* last_use, void* hot,
                                uint32_t* step);

/*
 * kvo_debug_layer_counters - copy the layer's eight device counters to host
 * uint32[8]: step, history length, LRU-queue head, tail and buffer, the
 * circular hand, two unused (synchronises the device).
 */
kvo_status kvo_debug_layer_counters(kvo_ctx* ctx, int32_t layer, uint32_t* out);

/*
 * kvo_debug_raise_status - test hook: ORs `bits` into the device status word
 * (1 = an index out of range, 2 = an internal check, 4 = a bounded wait gave
 * up, 8 = its second wait gave up too), as a kernel would, so that the
 * handling in kvo_sync can be tested without making a wait run out.
 * Synchronous.
 */
kvo_status kvo_debug_raise_status(kvo_ctx* ctx, uint32_t bits);

/*
 * kvo_debug_record_evictions - when enabled (on != 0), every resolve call
 * records its fills as (slot, evicted position or -1, new position) triples,
 * in the order the misses took them.  kvo_debug_evictions copies the last
 * call's list for `layer` to host int32[3*max] and its length to *count
 * (synchronises the device).
 */
kvo_status kvo_debug_record_evictions(kvo_ctx* ctx, int32_t on);
kvo_status kvo_debug_evictions(kvo_ctx* ctx, int32_t layer, int32_t* triples, int32_t max,
                               int32_t* count);

/*
 * kvo_probe_host_read - read `bytes` (multiple of 16) of pinned host memory
 * `src` with 16-byte zero-copy loads from every SM and reduce them into
 * device uint4 `sink`; used to measure the host link.  Stream-ordered.
 */
kvo_status kvo_probe_host_read(const void* src, int64_t bytes, void* sink, void* stream);

/* kvo_probe_host_touch - the same with one 16-byte load every `stride`
 * bytes (a multiple of 16): touches every page of a buffer while moving few
 * bytes.  Stream-ordered. */
kvo_status kvo_probe_host_touch(const void* src, int64_t bytes, int64_t stride, void* sink, void* stream);

/*
 * kvo_touch_history - one 16-byte GPU load per 4 KiB of the layer's host
 * history (all layers for layer = -1), up to its current length.  The GPU's
 * first access to a host page costs more than later ones: a new session's
 * first decode step over a 2.5 GB history took 1.0 ms untouched and 0.66 ms
 * after this call (which takes ~1.4 ms per GB).  Stream-ordered; changes no
 * state.  KVO_EINVAL for a bad layer.
 */
kvo_status kvo_touch_history(kvo_ctx* ctx, int32_t layer, void* stream);

/* kvo_debug_history_host - the host address of the layer's pinned history
 * (history_cap * 656 bytes), for measurements of how the host memory behaves
 * (reading it, or probing it from the GPU).  The caller must not write it. */
kvo_status kvo_debug_history_host(kvo_ctx* ctx, int32_t layer, void** out);

/* ------------------------------------------------------------------------
 * Session block store/restore.
 *
 * Sources (page title, section):
 *   [TIER] "A 60k-token context comes back off disk in 17 seconds instead of
 *          65 seconds of prefill" (vllm-bounded-fs-kv-tier README): KV of a
 *          session lives in fixed-size blocks of a GPU pool; whole sessions
 *          are stored to a lower tier and restored from it; a restore is
 *          admitted only when every group's blocks can be placed; the tier
 *          holds tier_bytes / block_bytes blocks (floor); the pool's free
 *          queue hands out blocks from its front and takes freed blocks at
 *          its back.
 *   [CORR] "Making KV offload correct", section "A grouped allocation is a
 *          transaction": a multi-group allocation either gives every group
 *          its blocks or leaves the allocator exactly as it was (free-queue
 *          order, tables, counters); section "Response completion is not
 *          copy completion": blocks are released only after the copies that
 *          depend on them have finished.
 *
 * A pool holds `pool_blocks` HBM blocks and `tier_blocks` pinned host blocks,
 * each of block_tokens rows of 656 bytes (row t of a block at byte
 * t * 656).  A session owns ceil(tokens / block_tokens) blocks in every one
 * of `layers` groups; the group of layer l maps session token t to block
 * table[l][t / block_tokens], row t % block_tokens.  The allocators and the
 * session tables live on the host: block ids returned by the calls below are
 * final when the call returns, while the bytes move stream-ordered.  A pool
 * is not thread-safe.
 * ---------------------------------------------------------------------- */

typedef struct kvo_pool kvo_pool;

typedef struct kvo_pool_stats {
  uint64_t stores;            /* successful kvo_store_blocks calls */
  uint64_t restores;          /* successful kvo_restore_blocks calls */
  uint64_t rollbacks;         /* grouped allocations refused and undone */
  uint64_t bytes_stored;      /* pool -> tier bytes enqueued */
  uint64_t bytes_restored;    /* tier -> pool bytes enqueued */
  uint64_t free_blocks;       /* pool blocks in the free queue */
  uint64_t tier_free_blocks;  /* tier blocks in the free queue */
  uint64_t pending_copies;    /* store/restore calls whose copies are not known complete */
} kvo_pool_stats;

/* [TIER] tier capacity in blocks: tier_bytes / block_bytes, rounded down;
 * -1 if tier_bytes < 0 or block_bytes <= 0.  Host only. */
int64_t kvo_tier_blocks(int64_t tier_bytes, int64_t block_bytes);

/*
 * kvo_pool_create - allocate a pool on the current device (synchronous).
 *   layers >= 1, 1 <= pool_blocks <= INT32_MAX, block_tokens >= 1,
 *   row_bytes must be KVO_ROW_BYTES, 0 <= tier_blocks <= INT32_MAX.
 * The HBM pool starts zeroed; both free queues start 0, 1, 2, ...
 * Returns KVO_EINVAL on bad arguments, KVO_ENOMEM if an allocation fails
 * (nothing is leaked).
 */
kvo_status kvo_pool_create(int32_t layers, int64_t pool_blocks, int32_t block_tokens, int32_t row_bytes,
                           int64_t tier_blocks, kvo_pool** out);

/* Waits for the device, frees everything (KVO_ECUDA if the wait failed). */
kvo_status kvo_pool_destroy(kvo_pool* pool);

/*
 * kvo_pool_alloc - [CORR] transactional: give new session `session` (an id
 * not in use) ceil(tokens / block_tokens) pool blocks in each layer group,
 * taken from the front of the free queue group after group.  If any block
 * cannot be had, every block taken is put back where it was and
 * KVO_ECAPACITY is returned (stats.rollbacks counts it).  Host only.
 */
kvo_status kvo_pool_alloc(kvo_pool* pool, int32_t session, int64_t tokens);

/*
 * kvo_pool_write / kvo_pool_read - copy `ntokens` rows between a contiguous
 * row buffer (656-byte rows, 16-byte aligned, device memory or mapped pinned
 * host memory) and tokens [first_token, first_token + ntokens) of the
 * session's layer group in the pool.  The session must be resident in the
 * pool and the range inside its tokens, else KVO_EINVAL.  Stream-ordered.
 */
kvo_status kvo_pool_write(kvo_pool* pool, int32_t session, int32_t layer, int64_t first_token,
                          const void* rows, int64_t ntokens, void* stream);
kvo_status kvo_pool_read(kvo_pool* pool, int32_t session, int32_t layer, int64_t first_token,
                         int64_t ntokens, void* out, void* stream);

/* Sets every byte of the HBM pool to `byte` (stream-ordered). */
kvo_status kvo_pool_fill(kvo_pool* pool, uint8_t byte, void* stream);

/*
 * kvo_store_blocks - [TIER] store: take tier blocks for every group of the
 * session (transactional as kvo_pool_alloc, KVO_ECAPACITY on a shortfall)
 * and enqueue one copy of every pool block to its tier block.  The session
 * must be resident in the pool and not already stored.  Until the copy has
 * completed the session counts as busy: kvo_pool_release returns
 * KVO_EBUSY ([CORR] "Response completion is not copy completion").
 */
kvo_status kvo_store_blocks(kvo_pool* pool, int32_t session, void* stream);

/*
 * kvo_pool_release - give the session's pool blocks back to the end of the
 * free queue (layer group by group, block-table order).  KVO_EBUSY while a
 * store or restore of the session has not completed (nothing changes).  A
 * stored session keeps its tier blocks and can be restored; a session with
 * no stored copy is forgotten.  Host only.
 */
kvo_status kvo_pool_release(kvo_pool* pool, int32_t session);

/*
 * kvo_restore_blocks - [TIER] restore `ns` distinct stored, non-resident
 * sessions as one admission: pool blocks for every group of every listed
 * session (in list order, layer order) or none (KVO_ECAPACITY, state
 * unchanged).  Enqueues the tier -> pool copies; the sessions' tier blocks
 * return to the tier free queue once those copies have completed, and the
 * sessions are busy until then.
 */
kvo_status kvo_restore_blocks(kvo_pool* pool, const int32_t* sessions, int32_t ns, void* stream);

/* Waits for `stream`, then retires every completed copy (busy counts drop,
 * tier blocks of finished restores are freed). */
kvo_status kvo_pool_sync(kvo_pool* pool, void* stream);

/*
 * kvo_pool_block_table - copy the block ids of the session's layer group,
 * which = 0 for its pool blocks, 1 for its tier blocks, into out[0..max);
 * *count = the group's length (0 when the session has no such copy or does
 * not exist).  Host only.
 */
kvo_status kvo_pool_block_table(kvo_pool* pool, int32_t session, int32_t layer, int32_t which, int32_t* out,
                                int64_t max, int64_t* count);

kvo_status kvo_pool_get_stats(kvo_pool* pool, kvo_pool_stats* out);

/* Test hook: the n-th next single-block allocation (0 = the next one) from
 * the pool (which = 0) or tier (which = 1) queue fails; n < 0 disarms. */
kvo_status kvo_pool_debug_fail_after(kvo_pool* pool, int32_t which, int64_t n);

/* Copies the pool (which = 0) or tier (which = 1) free queue, front first,
 * into out[0..max); *count = its length.  Host only. */
kvo_status kvo_pool_debug_free_queue(kvo_pool* pool, int32_t which, int32_t* out, int64_t max, int64_t* count);

/*
 * kvo_copy_blocks_noalloc - copy n whole blocks of block_bytes bytes:
 * block pairs[2i] of `src` to block pairs[2i+1] of `dst`, for i < n, with
 * the block-copy kernel of kvo_store_blocks / kvo_restore_blocks.
 *
 * The sources above have no counterpart to this call.  It is for callers
 * that keep their own block arrays (their own pool, their own pinned tier)
 * and must not allocate while it runs: an engine whose allocator already
 * owns the device memory budget, or a path where the device-wide
 * synchronisation of cudaMalloc/cudaFree is not allowed.  It needs no
 * kvo_pool and allocates nothing: the pair list is staged in a fixed static
 * device array of KVO_NOALLOC_MAX_PAIRS pairs (512 KiB) inside the library.
 *
 *   src, dst     device memory or mapped pinned host memory, 16-byte
 *                aligned, holding at least (largest id + 1) blocks each;
 *                owned by the caller.  Source and destination blocks must
 *                not overlap.
 *   block_bytes  > 0, a multiple of 16, at most 16 * (2^32 - 1).
 *   pairs        host array of 2n non-negative block ids.  The library
 *                cannot see the buffers' sizes: ids past their ends are
 *                the caller's error (the Python binding checks them).  It is copied with
 *                cudaMemcpyAsync on `stream`: pageable memory may be reused
 *                when the call returns, pinned memory only once the stream
 *                has passed the call.
 *   n            0 <= n <= KVO_NOALLOC_MAX_PAIRS; a larger n is refused with
 *                KVO_EINVAL before anything is enqueued (split the list).
 * Returns KVO_EINVAL on bad arguments, KVO_ECUDA if a CUDA call fails.
 * Stream-ordered.
 *
 * The first call on each device looks up the scratch array's address
 * (cudaGetSymbolAddress, with that device current) and keeps it; n = 0 does
 * only this.  Make that first call before any stream capture begins.
 * Every call on a device shares the one scratch array: calls whose copies
 * may overlap in time (different streams, or host threads, without an
 * ordering between them) race on it and may copy the wrong blocks.  Issue
 * them on one stream, or order them explicitly.
 */
#define KVO_NOALLOC_MAX_PAIRS 65536
kvo_status kvo_copy_blocks_noalloc(const void* src, void* dst, int64_t block_bytes, const int32_t* pairs,
                                   int64_t n, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KVO_H */
