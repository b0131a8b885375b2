// One decode step of many layers (kvo_decode_layers) in three launches, each
// over every layer of the call at once:
//   A select:  the top-K of every layer that brings scores (one cluster per
//              selecting layer, the body of kvo_select_topk; histories too
//              long for a cluster's shared memory take their first key digit
//              from a whole-GPU histogram launch before it);
//   B resolve: one CTA per layer: look every selected position up (hit:
//              stamp its slot; miss: first-occurrence claim), rank the
//              unique misses, walk the LRU queue (or the circular hand) for
//              their victims, update the maps, append the new rows to the
//              host history or the recent ring, append the used slots to the
//              LRU queue, and leave one code per entry for C;
//   C gather:  every selected entry of every layer on the whole GPU: the row
//              to the output with the bf16 dequant, hits from the HBM slot,
//              misses from host memory (or the recent ring, or this call's
//              new rows) and, for a position's first occurrence, into its
//              victim slot from the same registers; the step runs at the rate
//              of HBM and of the host link rather than at the latency of one
//              cluster per layer.
//
// "From 1M Total to 15+ x 1M Contexts: GLM-5.3 KV Cache Offloading":
//   "Decision three: let the GPU manage the hot cache directly" - hits read
//   the HBM slot, misses read the registered host copy, the gather emits a
//   compact selection, and the CPU stays out of the per-selection loop;
//   "GPU cache management has hazards too" - the victims are slots the step
//   does not use (B stamps every hit slot before it picks them), so no row C
//   writes into the cache is one C reads in the same step; duplicate misses
//   read host memory;
//   "Separate historical capacity from the current working set" - later
//   layers reuse a selection: a layer without scores resolves its idx as it
//   stands after A, so it may name the idx of a selecting layer of the same
//   call.
//
// Results equal those of the single-layer calls in the order append, select,
// resolve (the same LRU queue, the same first-occurrence dedupe, the same
// (last_use, slot) victim order).  Nothing but the layers' own tables, the
// entry codes and the caller's outputs carries state from one launch to the
// next.
#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "kvo_internal.h"
#include "kvo_resolve_body.cuh"
#include "kvo_topk_body.cuh"

namespace kvo {

namespace {

using resolve_detail::dequant_row;
using resolve_detail::kRowVec;

// One layer of the call: what changes from call to call.
struct LayerCall {
  const float* scores;          // NULL: idx is resolved as it stands after A
  int32_t* idx;
  uint8_t* out_rows;
  uint16_t* out_bf16;
  const uint8_t* fresh;         // this call's new rows (device), or NULL
  uint32_t layer;
  uint32_t n;                   // scores
  uint32_t ram_len;             // rows in the host history after this call's append and copyback
  uint32_t len;                 // history length after this call's append
  uint32_t fresh_from;          // position of the first new row (the old length)
  uint32_t r;                   // new rows
  uint32_t to_ram;              // the first to_ram new rows go to the host history, the rest to the ring
  uint32_t* first_hist;         // filtered selections: the histogram of the scores' top key bits (then the
                                //   arrival count and the cut), or NULL
  uint32_t* cand_count;         // filtered selections: per slice of the scores, its candidates' count, key
  uint32_t* cand_key;           //   and position (the histogram launch's lists), or NULL
  uint32_t* cand_pos;
  uint32_t* ent;                // [k] entry codes, written by B and read by C
};

constexpr uint32_t kBatchTasks = 128;                    // layers per launch (9 KB of parameters)
// shared memory of a selecting CTA for resident keys: 50,279 of them fit one CTA
constexpr uint32_t kSelectMaxSmem = 220u * 1024u;
struct LayerBatch {
  const LayerStatic* statics;   // device array, one entry per layer of the context
  uint32_t k;
  uint32_t chunks;              // B: CTAs per layer
  uint32_t cand_bytes;          // A (filtered route): shared memory for candidates
  uint32_t ntasks;
  // Misses fetched by batched copies (deferred is non-zero): the gathers
  // leave out the rows of the host history and list them instead, (entry,
  // position) at dlist[layer * KVO_MAX_K + i], counted in dcount[layer]; the
  // host copies the rows into staging (layer * k rows per layer) and lists
  // (entry, staging row) at plist, counted in pcount, for the placement.
  uint32_t deferred;
  int2* dlist;                  // device address of mapped host memory
  uint32_t* dcount;             // device memory, zero between calls
  const int2* plist;            // device address of mapped host memory
  const uint32_t* pcount;       // device address of mapped host memory
  const uint8_t* staging;       // device memory
  LayerCall t[kBatchTasks];
};

// Programmatic dependent launch: a launch that waits for the previous one on
// the stream may be scheduled before it ends, and waits here (in hardware)
// until the previous grid has completed and its memory is visible; the
// previous grid lets it be scheduled once every CTA has signalled.
__device__ __forceinline__ void wait_previous_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_next_grid() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------- A0: histogram
// For selections on the filtered route (histories whose keys do not fit the
// cluster's shared memory): the histogram of the top kFirstBits key bits of
// every score, built by the whole GPU (each CTA a slice of one layer's
// scores) rather than by the selecting cluster alone.  The selection finds
// its bucket from it, and its CTA 0 zeroes it for the next call.
//
// In the same pass each CTA lists its slice's candidates for the layer's
// selection: every key in or above the bucket one below the bucket the
// layer's previous selection cut in (kept in the histogram buffer), with
// its position, in position order.  The selection uses the lists when its
// own bucket is at or above that one (then the lists hold every key it
// needs) and they fit its shared memory; otherwise it filters the scores
// itself.  The lists cost one compare and a block scan per slice, and save
// the selection its own pass over the scores.
constexpr uint32_t kHistThreads = 256;
constexpr uint32_t kHistSlice = 16 * kHistThreads;      // scores per CTA (4,096): four float4 per thread
constexpr uint32_t kHistCopies = 4;                      // shared histograms, one per warp mod 4
static_assert(kHistSlice == topk_detail::kSliceScores, "the lists' slices are the histogram's");
// Word of the histogram buffer (after the bins) holding the bucket from
// which the next call lists candidates (0: list none).
constexpr uint32_t kHistSpec = topk_detail::kFirstBins;

__global__ void __launch_bounds__(kHistThreads) layers_hist_kernel(const __grid_constant__ LayerBatch b) {
  __shared__ uint32_t h[kHistCopies][topk_detail::kFirstBins];
  __shared__ unsigned long long wsum[kHistThreads / 32];
  const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const LayerCall& T = b.t[blockIdx.x / b.chunks];
  const uint32_t slice = blockIdx.x % b.chunks;
  const uint32_t lo = slice * kHistSlice;
  const uint32_t hi = min(T.n, lo + kHistSlice);
  const uint32_t spec = T.cand_count ? __ldcg(&T.first_hist[kHistSpec]) : 0u;
  for (uint32_t i = tid; i < kHistCopies * topk_detail::kFirstBins; i += kHistThreads) (&h[0][0])[i] = 0;
  // group q of this thread: scores lo + 4 (q kHistThreads + tid) .. + 3
  // (coalesced), every load in flight at once
  const bool vec = (reinterpret_cast<uintptr_t>(T.scores + lo) & 15u) == 0;
  float f[4][4];
#pragma unroll
  for (uint32_t q = 0; q < 4; ++q) {
    const uint32_t i0 = lo + 4 * (q * kHistThreads + tid);
    if (vec && i0 + 3 < hi) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(T.scores + i0));
      f[q][0] = v.x, f[q][1] = v.y, f[q][2] = v.z, f[q][3] = v.w;
    } else {
      for (uint32_t e = 0; e < 4; ++e) f[q][e] = i0 + e < hi ? __ldg(T.scores + i0 + e) : 0.f;
    }
  }
  __syncthreads();                                       // the shared histograms are zero
  uint32_t* mine = h[warp % kHistCopies];
#pragma unroll
  for (uint32_t q = 0; q < 4; ++q) {
    const uint32_t i0 = lo + 4 * (q * kHistThreads + tid);
#pragma unroll
    for (uint32_t e = 0; e < 4; ++e)
      if (i0 + e < hi) atomicAdd(&mine[score_key(f[q][e]) >> topk_detail::kLowBits], 1u);
  }
  if (spec && lo < hi) {                                 // uniform over the CTA
    // the slice's candidates in position order (group row q, then thread,
    // then element): one float compare each, as in the selection's own
    // filtering pass, and one block scan of the four rows' counts packed
    // in 16-bit fields (at most 1,024 per row)
    const float t = topk_detail::key_floor_float(spec << topk_detail::kLowBits);
    uint32_t keep[4];
    unsigned long long c = 0;
#pragma unroll
    for (uint32_t q = 0; q < 4; ++q) {
      const uint32_t i0 = lo + 4 * (q * kHistThreads + tid);
      keep[q] = 0;
#pragma unroll
      for (uint32_t e = 0; e < 4; ++e) keep[q] |= (uint32_t)(i0 + e < hi && f[q][e] >= t) << e;
      c |= (unsigned long long)__popc(keep[q]) << (16 * q);
    }
    unsigned long long incl = c;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const unsigned long long o = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= (uint32_t)d) incl += o;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    unsigned long long before = 0, all_c = 0;
#pragma unroll
    for (uint32_t w = 0; w < kHistThreads / 32; ++w) {
      before += w < warp ? wsum[w] : 0ull;
      all_c += wsum[w];
    }
    const unsigned long long mine_off = before + incl - c;   // per row: entries before this thread's
    const size_t base = (size_t)slice * kHistSlice;
    uint32_t row_base = 0;                               // entries of the rows before q
#pragma unroll
    for (uint32_t q = 0; q < 4; ++q) {
      uint32_t o = row_base + (uint32_t)((mine_off >> (16 * q)) & 0xffffu);
      const uint32_t i0 = lo + 4 * (q * kHistThreads + tid);
#pragma unroll
      for (uint32_t e = 0; e < 4; ++e)
        if ((keep[q] >> e) & 1u) {
          T.cand_key[base + o] = score_key(f[q][e]);
          T.cand_pos[base + o] = i0 + e;
          ++o;
        }
      row_base += (uint32_t)((all_c >> (16 * q)) & 0xffffu);
    }
    if (tid == 0) T.cand_count[slice] = row_base;
  }
  __syncthreads();
  for (uint32_t bin = tid; bin < topk_detail::kFirstBins; bin += kHistThreads) {
    uint32_t v = 0;
#pragma unroll
    for (uint32_t c = 0; c < kHistCopies; ++c) v += h[c][bin];
    if (v) atomicAdd(&T.first_hist[bin], v);
  }
  allow_next_grid();                                     // the selections may be scheduled; they wait for this grid
}

// ------------------------------------------------------------ A: select
template <bool kResident>
__global__ void __launch_bounds__(kThreads, 1) layers_select_kernel(const __grid_constant__ LayerBatch b) {
  extern __shared__ __align__(16) uint8_t dyn_smem[];
  __shared__ RadixSmem rsm;
  const LayerCall& T = b.t[blockIdx.x / cluster_size()];
  wait_previous_grid();                                  // the histograms and the lists are complete
  allow_next_grid();                                     // the gathers may be scheduled; they wait for this grid
  int32_t* idx = T.idx;
  const int32_t* pos2slot = b.statics[T.layer].pos2slot;
  __shared__ uint32_t next_spec;
  const uint32_t spec = T.first_hist && T.cand_count ? __ldcg(&T.first_hist[kHistSpec]) : 0u;
  const topk_detail::FilterPre pre{spec, T.cand_count, T.cand_key, T.cand_pos};
  topk_detail::topk_body<kResident>(
      T.scores, T.n, b.k, dyn_smem, b.cand_bytes, &rsm,
      [&](uint32_t pos, uint32_t out) {
        idx[out] = (int32_t)pos;
        prefetch_l2(&pos2slot[pos]);                     // B looks it up next
      },
      T.first_hist, T.cand_count ? &pre : nullptr, &next_spec);
  // every CTA of the cluster has read the histogram and the listing bucket
  // (cluster barriers came after its reads): zero the histogram for the
  // next call, and set the bucket it lists from
  if (T.first_hist && cluster_rank() == 0) {
    for (uint32_t bin = threadIdx.x; bin < topk_detail::kFirstBins; bin += kThreads) T.first_hist[bin] = 0;
    if (threadIdx.x == 0) T.first_hist[kHistSpec] = T.cand_count ? next_spec : 0u;
  }
}

// ------------------------------------------------------------ B: resolve
// Entry codes: B writes one per selected entry of a layer (ent[j]), C reads
// them.  A hit holds its slot; a miss is flagged, and when it is the first
// occurrence of its position it also holds the victim slot its row goes to.
constexpr uint32_t kEntInvalid = 0xffffffffu;            // position out of range: a zero row
constexpr uint32_t kEntMiss = 1u << 31;                  // the row comes from its source
constexpr uint32_t kEntFill = 1u << 30;                  // ... and is written to the slot in the low bits too
constexpr uint32_t kEntLater = 1u << 29;                 // ... by a batched copy (placed after the copies)
constexpr uint32_t kEntSlot = (1u << 24) - 1u;
static_assert(KVO_MAX_HOT_ROWS <= kEntSlot, "a slot fits the entry code");

constexpr uint32_t kFinishPer = 4;                        // queue entries a thread examines per round
constexpr uint32_t kFinishEntries = KVO_MAX_K / kThreads;  // selection entries per thread
constexpr uint32_t kCompactPer = 16;                      // queue entries a thread keeps in flight when compacting
constexpr uint32_t kNoEntry = 0xffffffffu;

// The row of a missing position: this call's new rows from their device
// copy; rows still waiting in the recent ring from the ring; else the host
// history.  *host: the row crosses the host link.
__device__ __forceinline__ const uint4* miss_source(const LayerStatic& S, const LayerCall& T, uint32_t p,
                                                   bool* host) {
  *host = false;
  if (T.fresh && p >= T.fresh_from) return reinterpret_cast<const uint4*>(T.fresh) + (size_t)(p - T.fresh_from) * kRowVec;
  if (S.ring_rows && p >= T.ram_len)
    return reinterpret_cast<const uint4*>(S.recent) + (size_t)(p & (S.ring_rows - 1u)) * kRowVec;
  *host = true;
  return reinterpret_cast<const uint4*>(S.hist) + (size_t)p * kRowVec;
}

// Copies the current entries of [head, tail) of queue buffer `buf`, in
// order, to the front of the other buffer; returns how many (the number of
// slots).  One CTA.
__device__ uint32_t compact_queue_cta(const LayerStatic& T, uint32_t head, uint32_t tail, uint32_t buf,
                                      uint32_t* scratch) {
  const uint32_t Q = T.ring_cap, qmask = Q - 1u;
  const uint64_t* in = T.ring + (size_t)buf * Q;
  uint64_t* out = T.ring + (size_t)(buf ^ 1u) * Q;
  const uint32_t span = tail - head;
  uint32_t kept = 0;
  for (uint32_t base = 0; base < span; base += kCompactPer * kThreads) {
    uint64_t e[kCompactPer];
    uint32_t lu[kCompactPer];
#pragma unroll
    for (uint32_t q = 0; q < kCompactPer; ++q) {
      const uint32_t o = base + kCompactPer * threadIdx.x + q;
      e[q] = o < span ? __ldcg(&in[(head + o) & qmask]) : ~0ull;
    }
#pragma unroll
    for (uint32_t q = 0; q < kCompactPer; ++q) {
      const uint32_t sl = (uint32_t)e[q];
      lu[q] = e[q] != ~0ull && sl < T.hot_rows ? __ldcg(&T.last_use[sl]) : 0u;
    }
    uint32_t mine = 0, keep = 0;
#pragma unroll
    for (uint32_t q = 0; q < kCompactPer; ++q) {
      const bool cur = e[q] != ~0ull && (uint32_t)e[q] < T.hot_rows && lu[q] == (uint32_t)(e[q] >> 32);
      keep |= (uint32_t)cur << q;
      mine += cur;
    }
    uint32_t tot;
    uint32_t pos = kept + block_excl_sum(mine, scratch, &tot);
#pragma unroll
    for (uint32_t q = 0; q < kCompactPer; ++q)
      if ((keep >> q) & 1u) {
        if (pos < Q) out[pos] = e[q];
        ++pos;
      }
    kept += tot;
  }
  return kept;
}

// Shared memory of the resolve launch (4-byte words): per unique miss u its
// entry, victim slot and position; every entry's code; then the bitmap of
// the slots used in the step (hits, then victims).
__host__ __device__ inline size_t resolve_smem_bytes(uint32_t k, uint32_t H) {
  return (4u * (size_t)k + (H + 31u) / 32u) * 4u;
}

// One CTA per layer.  The loads that do not depend on one another are
// issued together (the positions and the first queue window, then the
// positions' slots and the window's stamps), so that the chain of dependent
// global accesses stays short after an L2 flush.
template <bool kLru>
__global__ void __launch_bounds__(kThreads, 1) layers_resolve_kernel(const __grid_constant__ LayerBatch b,
                                                                     uint32_t* status) {
  extern __shared__ __align__(16) uint32_t fsm[];
  __shared__ uint32_t scratch[2 * kWarps + 2];
  __shared__ uint32_t head_hit, last_vic, nevict, cnt[4];
  const uint32_t tid = threadIdx.x, lane = tid & 31;
  const LayerCall& T = b.t[blockIdx.x];
  const LayerStatic S = b.statics[T.layer];
  const uint32_t k = b.k, H = S.hot_rows;
  uint32_t* mlist = fsm;                                 // [k]: entry of unique miss u
  uint32_t* vslot = fsm + k;                             // [k]: victim slot of unique miss u
  int32_t* mpos = reinterpret_cast<int32_t*>(fsm + 2 * k);   // [k]: position of unique miss u
  uint32_t* code = fsm + 3 * k;                          // [k]: entry codes
  uint32_t* used = fsm + 4 * k;                          // [ceil(H/32)]: slots used in this step
  const uint32_t hwords = (H + 31u) / 32u;
  // Before the selections end: the layer's counters, the queue (compacted
  // if need be) and its first window with the window's stamps, none of
  // which this call's earlier launches touch.  (This launch is scheduled
  // once every CTA of the previous one runs, which is after the previous
  // call has ended.)
  const uint32_t t = __ldcg(&S.counters[0]) + 1u;
  uint32_t head = __ldcg(&S.counters[2]), tail = __ldcg(&S.counters[3]), buf = __ldcg(&S.counters[4]) & 1u;
  const uint32_t hand = __ldcg(&S.counters[5]);
  const uint32_t Q = S.ring_cap, qmask = Q - 1u;
  if (tid == 0) {
    head_hit = kNoEntry;
    nevict = 0;
  }
  if (tid < 4) cnt[tid] = 0;
  // The queue gets at most k entries in this call: make room first.
  if (kLru && tail - head > Q - k) {
    tail = compact_queue_cta(S, head, tail, buf, scratch);
    if (tid == 0 && tail != H) atomicOr(status, kFlagInternal);
    head = 0;
    buf ^= 1u;
    __syncthreads();
  }
  const uint64_t* ring_in = S.ring + (size_t)buf * Q;
  uint64_t* ring_out = S.ring + (size_t)buf * Q;
  const uint32_t span = tail - head;
  const uint32_t limit = kLru ? span : H;

  // 1. the first queue window and its slots' stamps (read before this
  //    step's hits are stamped: a window entry whose slot is hit is left out
  //    by the used bitmap below, as the stamp would leave it out)
  for (uint32_t w = tid; w < hwords; w += kThreads) used[w] = 0;
  uint64_t e[kFinishPer];
#pragma unroll
  for (uint32_t q = 0; q < kFinishPer; ++q) {
    const uint32_t o = kFinishPer * tid + q;
    if (kLru) e[q] = o < span ? __ldcg(&ring_in[(head + o) & qmask]) : ~0ull;
    else e[q] = o < H ? (uint64_t)(hand + o < H ? hand + o : hand + o - H) : ~0ull;
  }
  uint32_t lu[kFinishPer];
#pragma unroll
  for (uint32_t q = 0; q < kFinishPer; ++q) {
    const uint32_t s = (uint32_t)e[q];
    lu[q] = kLru && e[q] != ~0ull && s < H ? __ldcg(&S.last_use[s]) : 0u;
  }
  wait_previous_grid();                                  // the selections are complete
  allow_next_grid();                                     // the gathers may be scheduled; they wait for this grid

  // 2. positions of this thread's entries (and whether the whole selection
  //    increases: then every position is distinct and no claims are
  //    needed), then their slots
  int32_t pj[kFinishEntries];
  bool inc = true;
#pragma unroll
  for (uint32_t q = 0; q < kFinishEntries; ++q) {
    const uint32_t j = q * kThreads + tid;
    pj[q] = j < k ? __ldcg(&T.idx[j]) : -1;
    if (j + 1 < k) inc = inc && pj[q] < __ldcg(&T.idx[j + 1]);
  }
  int32_t sl[kFinishEntries];
#pragma unroll
  for (uint32_t q = 0; q < kFinishEntries; ++q)
    sl[q] = pj[q] >= 0 && (uint32_t)pj[q] < T.len ? __ldcg(&S.pos2slot[pj[q]]) : -1;
  const bool increasing = __syncthreads_and(inc);       // and the used bitmap is zero

  // 3. classify: a hit stamps its slot with the step and joins the used
  //    slots; a miss claims its position (the smallest entry wins: the
  //    first occurrence fills the slot, later ones read the source too)
  uint32_t nhit = 0, nmiss = 0, nram = 0, ninv = 0;
#pragma unroll
  for (uint32_t q = 0; q < kFinishEntries; ++q) {
    const uint32_t j = q * kThreads + tid;
    if (j >= k) continue;
    const int32_t p = pj[q];
    if (p < 0 || (uint32_t)p >= T.len) {
      code[j] = kEntInvalid;
      ++ninv;
      continue;
    }
    int32_t s = sl[q];
    if (s >= (int32_t)H) {
      atomicOr(status, kFlagInternal);                   // cannot happen; keep every index in bounds
      s = -1;
      sl[q] = -1;
    }
    if (s >= 0) {
      S.last_use[s] = t;                                 // pinned for this step
      atomicOr(&used[(uint32_t)s >> 5], 1u << (s & 31));
      code[j] = (uint32_t)s;
      ++nhit;
    } else {
      if (!increasing) atomicMin(&S.pos2slot[p], (int32_t)j - (int32_t)k - 1);
      bool host;
      (void)miss_source(S, T, (uint32_t)p, &host);
      code[j] = kEntMiss | (host && b.deferred ? kEntLater : 0u);
      ++nmiss;
      // a RAM read as append-then-resolve defines it: below the RAM length
      // (this call's own rows there are served from their device copy,
      // which holds the same bytes)
      nram += !(S.ring_rows && (uint32_t)p >= T.ram_len);
    }
  }
  {
    const uint32_t h = __reduce_add_sync(0xffffffffu, nhit), m = __reduce_add_sync(0xffffffffu, nmiss);
    const uint32_t rr = __reduce_add_sync(0xffffffffu, nram), iv = __reduce_add_sync(0xffffffffu, ninv);
    if (lane == 0) {
      if (h) atomicAdd(&cnt[0], h);
      if (m) atomicAdd(&cnt[1], m);
      if (rr) atomicAdd(&cnt[2], rr);
      if (iv) atomicAdd(&cnt[3], iv);
    }
  }
  __syncthreads();                                       // the claims are in place; used holds every hit

  // 4. unique misses: the entries whose claim won (every miss of an
  //    increasing selection), in entry order
  int32_t claim[kFinishEntries];
#pragma unroll
  for (uint32_t q = 0; q < kFinishEntries; ++q) {
    const uint32_t j = q * kThreads + tid;
    claim[q] = !increasing && j < k && pj[q] >= 0 && (uint32_t)pj[q] < T.len && sl[q] < 0
                   ? __ldcg(&S.pos2slot[pj[q]])
                   : (int32_t)j - (int32_t)k - 1;
  }
  uint32_t M = 0;
#pragma unroll
  for (uint32_t q = 0; q < kFinishEntries; ++q) {
    if (q * kThreads >= k) break;                        // uniform over the CTA
    const uint32_t j = q * kThreads + tid;
    const bool fl = j < k && pj[q] >= 0 && (uint32_t)pj[q] < T.len && sl[q] < 0 &&
                    claim[q] == (int32_t)j - (int32_t)k - 1;
    uint32_t tile;
    const uint32_t rank = block_flag_scan(fl, scratch, &tile);
    if (fl) {
      mlist[M + rank] = j;
      mpos[M + rank] = pj[q];
    }
    M += tile;
  }

  // 5. victims: the first M current entries of the queue from its head
  //    whose slot this step does not use, or the first M such slots from
  //    the circular hand
  uint32_t found = 0, off = 0;
  for (bool first_round = true; found < M && off < limit; first_round = false) {   // uniform over the CTA
    if (!first_round) {
#pragma unroll
      for (uint32_t q = 0; q < kFinishPer; ++q) {
        const uint32_t o = off + kFinishPer * tid + q;
        if (kLru) e[q] = o < span ? __ldcg(&ring_in[(head + o) & qmask]) : ~0ull;
        else e[q] = o < H ? (uint64_t)(hand + o < H ? hand + o : hand + o - H) : ~0ull;
      }
#pragma unroll
      for (uint32_t q = 0; q < kFinishPer; ++q) {
        const uint32_t s = (uint32_t)e[q];
        lu[q] = kLru && e[q] != ~0ull && s < H ? __ldcg(&S.last_use[s]) : 0u;
      }
    }
    uint32_t ncur = 0;
#pragma unroll
    for (uint32_t q = 0; q < kFinishPer; ++q) {
      const uint32_t s = (uint32_t)e[q];
      const bool cur = e[q] != ~0ull && s < H && (!kLru || lu[q] == (uint32_t)(e[q] >> 32)) &&
                       !((used[s >> 5] >> (s & 31)) & 1u);
      if (cur) ++ncur;
      else e[q] = ~0ull;
    }
    uint32_t tot;
    uint32_t u = found + block_excl_sum(ncur, scratch, &tot);
#pragma unroll
    for (uint32_t q = 0; q < kFinishPer; ++q) {
      if (e[q] == ~0ull) continue;
      if (u < M) {
        vslot[u] = (uint32_t)e[q];
        if (u == M - 1) last_vic = (uint32_t)e[q];
      } else if (u == M) {
        head_hit = off + kFinishPer * tid + q;           // the first current entry that stays
      }
      ++u;
    }
    found += tot;
    off += kFinishPer * kThreads;
  }
  __syncthreads();
  if (found < M && tid == 0) atomicOr(status, kFlagInternal);   // cannot happen: M <= unpinned slots
  const uint32_t nvic = found < M ? found : M;

  // 6. map updates, one thread per unique miss; the victims join the used
  //    slots, and the miss's entry code names its slot
  for (uint32_t u = tid; u < nvic; u += kThreads) {
    const uint32_t v = vslot[u];
    const int32_t p = mpos[u];
    if (v >= H || p < 0 || (uint32_t)p >= S.history_cap) {
      atomicOr(status, kFlagInternal);                   // cannot happen; never write out of bounds
      continue;
    }
    const int32_t old = __ldcg(&S.slot2pos[v]);
    if (old >= 0) {
      S.pos2slot[old] = -1;
      atomicAdd(&nevict, 1u);
    }
    S.pos2slot[p] = (int32_t)v;
    S.slot2pos[v] = p;
    S.last_use[v] = t;
    atomicOr(&used[v >> 5], 1u << (v & 31));
    code[mlist[u]] |= kEntFill | v;
    if (S.evlog) {
      S.evlog[1 + 3 * u] = (int32_t)v;
      S.evlog[2 + 3 * u] = old;
      S.evlog[3 + 3 * u] = p;
    }
  }

  // 7. the new rows, to the host history below the RAM length, else to the
  //    recent ring
  const uint32_t warp = tid >> 5;
  for (uint32_t i = warp; i < T.r; i += kWarps) {
    uint4* dst = i >= T.to_ram ? reinterpret_cast<uint4*>(S.recent) +
                                     (size_t)((T.fresh_from + i) & (S.ring_rows - 1u)) * kRowVec
                               : reinterpret_cast<uint4*>(const_cast<uint8_t*>(S.hist)) +
                                     (size_t)(T.fresh_from + i) * kRowVec;
    const uint4* src = reinterpret_cast<const uint4*>(T.fresh) + (size_t)i * kRowVec;
    dst[lane] = src[lane];
    if (lane < kRowVec - 32) dst[32 + lane] = src[32 + lane];
  }
  __syncthreads();                                       // the used bitmap and the codes are complete

  // 8. the codes for the gathers, and (batched copies) the list of the
  //    entries whose rows the host copies, in entry order
  for (uint32_t j = tid; j < k; j += kThreads) T.ent[j] = code[j];
  if (b.deferred) {
    uint32_t nl = 0;
    for (uint32_t j0 = 0; j0 < k; j0 += kThreads) {      // uniform over the CTA
      const uint32_t j = j0 + tid;
      const bool fl = j < k && code[j] != kEntInvalid && (code[j] & kEntLater);
      uint32_t tile;
      const uint32_t rank = block_flag_scan(fl, scratch, &tile);
      if (fl) b.dlist[(size_t)T.layer * KVO_MAX_K + nl + rank] = make_int2((int32_t)j, __ldcg(&T.idx[j]));
      nl += tile;
    }
    if (tid == 0) b.dcount[T.layer] = nl;
  }

  // 9. LRU queue: every slot used in this step, in slot order, stamped t,
  //    at the tail
  uint32_t appended = 0;
  if (kLru) {
    const uint64_t stamp = (uint64_t)t << 32;
    for (uint32_t w0 = 0; w0 < hwords; w0 += kThreads) {
      const uint32_t w = w0 + tid;
      uint32_t bits = w < hwords ? used[w] : 0u;
      uint32_t tot;
      uint32_t pos = tail + appended + block_excl_sum(__popc(bits), scratch, &tot);
      while (bits) {
        const uint32_t bit = __ffs(bits) - 1;
        bits &= bits - 1;
        ring_out[pos & qmask] = stamp | (uint64_t)(32 * w + bit);
        ++pos;
      }
      appended += tot;
    }
  }

  // 10. counters and stats
  if (tid == 0) {
    S.counters[0] = t;
    S.counters[1] = T.len;
    if (kLru) {
      S.counters[2] = nvic > 0 ? head + (head_hit != kNoEntry ? head_hit : min(off, span)) : head;
      S.counters[3] = tail + appended;
      S.counters[4] = buf;
    } else if (nvic > 0) {
      S.counters[5] = last_vic + 1u == H ? 0u : last_vic + 1u;
    }
    unsigned long long* st = S.stats;
    atomicAdd(st + 0, 1ull);
    if (cnt[0]) atomicAdd(st + 1, (unsigned long long)cnt[0]);
    if (cnt[1]) atomicAdd(st + 2, (unsigned long long)cnt[1]);
    if (M) atomicAdd(st + 3, (unsigned long long)M);
    if (nevict) atomicAdd(st + 4, (unsigned long long)nevict);
    if (cnt[3]) {
      atomicAdd(st + 5, (unsigned long long)cnt[3]);
      atomicOr(status, kFlagRange);
    }
    if (cnt[2]) atomicAdd(st + 6, (unsigned long long)cnt[2] * KVO_ROW_BYTES);
    atomicAdd(st + 7, (unsigned long long)k);
    if (S.evlog) S.evlog[0] = (int32_t)nvic;
  }
}

// ------------------------------------------------------------ C: gather
constexpr uint32_t kGatherThreads = 256;
constexpr uint32_t kGatherWarps = kGatherThreads / 32;
constexpr uint32_t kGatherEntries = 64;                  // entries per CTA
constexpr uint32_t kGatherInFlight = 4;                  // rows a warp loads before it stores
static_assert(kGatherEntries <= kGatherThreads, "one thread per entry reads its code");

// The row of entry j by its code: a hit's slot, a miss's source, or NULL
// (a zero row).  *fill: the slot a first-occurrence miss also fills, or
// NULL.  Codes and positions are checked again (never an access out of
// bounds, whatever the tables hold).
__device__ __forceinline__ const uint4* entry_source(const LayerStatic& S, const LayerCall& T, uint32_t c, int32_t p,
                                                     uint4** fill, uint32_t* status) {
  *fill = nullptr;
  if (c == kEntInvalid) return nullptr;
  const uint32_t s = c & kEntSlot;
  if (!(c & kEntMiss)) {
    if (s >= S.hot_rows) {
      atomicOr(status, kFlagInternal);
      return nullptr;
    }
    return reinterpret_cast<const uint4*>(S.hot) + (size_t)s * kRowVec;
  }
  if (p < 0 || (uint32_t)p >= T.len) {
    atomicOr(status, kFlagInternal);
    return nullptr;
  }
  if (c & kEntFill) {
    if (s < S.hot_rows) *fill = reinterpret_cast<uint4*>(S.hot) + (size_t)s * kRowVec;
    else atomicOr(status, kFlagInternal);
  }
  bool host;
  return miss_source(S, T, (uint32_t)p, &host);
}

// Every selected entry of every layer: the row to the output (and its bf16
// dequant), hits from the HBM slot, misses from their source and, for the
// first occurrence of a position, into the victim slot B chose as well.  No
// slot this launch writes is read by it: victims are slots the step does
// not use.
__global__ void __launch_bounds__(kGatherThreads) layers_gather_kernel(const __grid_constant__ LayerBatch b,
                                                                       uint32_t* status) {
  __shared__ const uint4* src[kGatherEntries];           // NULL: a zero row
  __shared__ uint4* fill[kGatherEntries];                // the victim slot's row, or NULL
  __shared__ uint8_t later[kGatherEntries];              // the row comes by a batched copy (placed later)
  const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const LayerCall& T = b.t[blockIdx.x / b.chunks];
  const LayerStatic S = b.statics[T.layer];
  const uint32_t k = b.k;
  const uint32_t j0 = (blockIdx.x % b.chunks) * kGatherEntries;
  const uint32_t nj = j0 < k ? min(kGatherEntries, k - j0) : 0u;
  wait_previous_grid();                                  // the resolves are complete

  if (tid < nj) {
    const uint32_t j = j0 + tid;
    const uint32_t c = __ldcg(&T.ent[j]);
    const int32_t p = __ldcg(&T.idx[j]);
    uint4* f;
    const uint4* s = entry_source(S, T, c, p, &f, status);
    const bool l = c != kEntInvalid && (c & kEntLater);
    src[tid] = l ? nullptr : s;
    fill[tid] = l ? nullptr : f;
    later[tid] = l;
  }
  __syncthreads();

  // rows: each warp keeps kGatherInFlight rows in flight in registers.
  // (Staging every piece in shared memory with 16-byte asynchronous copies,
  // all in flight at once, was slower: 90 vs 70 us for the 78-layer stack's
  // gathers, 106 vs 65 us at 1M.)
  for (uint32_t e0 = warp; e0 < nj; e0 += kGatherWarps * kGatherInFlight) {
    uint4 va[kGatherInFlight], vb[kGatherInFlight];
#pragma unroll
    for (uint32_t u = 0; u < kGatherInFlight; ++u) {
      const uint32_t e = e0 + u * kGatherWarps;
      va[u] = make_uint4(0, 0, 0, 0);
      vb[u] = make_uint4(0, 0, 0, 0);
      const uint4* s = e < nj ? src[e] : nullptr;
      if (s) {
        va[u] = s[lane];
        if (lane < kRowVec - 32) vb[u] = s[32 + lane];
      }
    }
#pragma unroll
    for (uint32_t u = 0; u < kGatherInFlight; ++u) {
      const uint32_t e = e0 + u * kGatherWarps;
      if (e >= nj) break;
      if (later[e]) continue;
      const uint32_t j = j0 + e;
      if (T.out_rows) {
        uint4* d = reinterpret_cast<uint4*>(T.out_rows) + (size_t)j * kRowVec;
        d[lane] = va[u];
        if (lane < kRowVec - 32) d[32 + lane] = vb[u];
      }
      if (uint4* f = fill[e]) {
        f[lane] = va[u];
        if (lane < kRowVec - 32) f[32 + lane] = vb[u];
      }
      if (T.out_bf16) dequant_row(va[u], vb[u], lane, reinterpret_cast<uint4*>(T.out_bf16 + (size_t)j * KVO_DEQUANT_VALUES));
    }
  }
  allow_next_grid();
}

// --------------------------------------------------- C2: batched placement
// The rows the host copied into staging, to their entries of the output
// (and their bf16 rows) and, for first occurrences, to their victim slots:
// one warp per row, kGatherInFlight rows in flight.
__global__ void __launch_bounds__(kGatherThreads) layers_place_kernel(const __grid_constant__ LayerBatch b,
                                                                      uint32_t* status) {
  const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const LayerCall& T = b.t[blockIdx.x / b.chunks];
  const uint32_t H = b.statics[T.layer].hot_rows;
  uint8_t* hot = b.statics[T.layer].hot;
  wait_previous_grid();
  const uint32_t m = b.pcount[T.layer];
  const uint32_t e0 = (blockIdx.x % b.chunks) * kGatherEntries;
  const int2* pl = b.plist + (size_t)T.layer * KVO_MAX_K;
  const uint4* stage = reinterpret_cast<const uint4*>(b.staging) + (size_t)T.layer * b.k * kRowVec;
  for (uint32_t i0 = e0 + warp; i0 < min(m, e0 + kGatherEntries); i0 += kGatherWarps * kGatherInFlight) {
    uint4 va[kGatherInFlight], vb[kGatherInFlight];
    int2 pe[kGatherInFlight];
#pragma unroll
    for (uint32_t u = 0; u < kGatherInFlight; ++u) {
      const uint32_t i = i0 + u * kGatherWarps;
      pe[u] = i < min(m, e0 + kGatherEntries) ? pl[i] : make_int2(-1, -1);
      va[u] = make_uint4(0, 0, 0, 0);
      vb[u] = make_uint4(0, 0, 0, 0);
      if (pe[u].x >= 0 && (uint32_t)pe[u].x < b.k && (uint32_t)pe[u].y < b.k) {
        const uint4* s = stage + (size_t)pe[u].y * kRowVec;
        va[u] = s[lane];
        if (lane < kRowVec - 32) vb[u] = s[32 + lane];
      }
    }
#pragma unroll
    for (uint32_t u = 0; u < kGatherInFlight; ++u) {
      if (pe[u].x < 0 || (uint32_t)pe[u].x >= b.k || (uint32_t)pe[u].y >= b.k) continue;
      const uint32_t j = (uint32_t)pe[u].x;
      if (T.out_rows) {
        uint4* d = reinterpret_cast<uint4*>(T.out_rows) + (size_t)j * kRowVec;
        d[lane] = va[u];
        if (lane < kRowVec - 32) d[32 + lane] = vb[u];
      }
      const uint32_t c = __ldcg(&T.ent[j]);
      if (c != kEntInvalid && (c & kEntMiss) && (c & kEntFill)) {
        if ((c & kEntSlot) < H) {
          uint4* f = reinterpret_cast<uint4*>(hot) + (size_t)(c & kEntSlot) * kRowVec;
          f[lane] = va[u];
          if (lane < kRowVec - 32) f[32 + lane] = vb[u];
        } else if (lane == 0) {
          atomicOr(status, kFlagInternal);
        }
      }
      if (T.out_bf16) dequant_row(va[u], vb[u], lane, reinterpret_cast<uint4*>(T.out_bf16 + (size_t)j * KVO_DEQUANT_VALUES));
    }
  }
  allow_next_grid();
}

// ------------------------------------------------------------ launch
struct LayersConfig {
  bool init = false;
  int active[5] = {0, 0, 0, 0, 0};     // select clusters of 1, 2, 4, 8, 16 CTAs that fit at once (resident)
  int active_stream[5] = {0, 0, 0, 0, 0};
  int force_select = 0;
};
LayersConfig g_layers[64];

int active_clusters(const void* kern, int C, size_t smem) {
  cudaLaunchConfig_t lc = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  lc.gridDim = dim3(C, 1, 1);
  lc.blockDim = dim3(kThreads, 1, 1);
  lc.dynamicSmemBytes = smem;
  lc.attrs = attr;
  lc.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &lc) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t layers_init(LayersConfig** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  LayersConfig& cfg = g_layers[dev & 63];
  if (!cfg.init) {
    const void* sel[2] = {(const void*)layers_select_kernel<true>, (const void*)layers_select_kernel<false>};
    // resident keys take up to kSelectMaxSmem; the filtered route's
    // candidates kTopkMaxDynSmem (its static shared memory is larger)
    const int sel_smem[2] = {(int)kSelectMaxSmem, (int)topk_detail::kTopkMaxDynSmem};
    for (int i = 0; i < 2; ++i) {
      e = cudaFuncSetAttribute(sel[i], cudaFuncAttributeMaxDynamicSharedMemorySize, sel_smem[i]);
      if (e != cudaSuccess) return e;
      if (cudaFuncSetAttribute(sel[i], cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
        cudaGetLastError();
    }
    for (const void* kern : {(const void*)layers_resolve_kernel<true>, (const void*)layers_resolve_kernel<false>}) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)resolve_smem_bytes(KVO_MAX_K, KVO_MAX_HOT_ROWS));
      if (e != cudaSuccess) return e;
    }
    for (int i = 0; i < 5; ++i) {
      cfg.active[i] = active_clusters(sel[0], 1 << i, kSelectMaxSmem);
      cfg.active_stream[i] = i ? active_clusters(sel[1], 1 << i, topk_detail::kTopkMaxDynSmem) : 0;
    }
    // KVO_SELECT_CLUSTER (1, 2, 4, 8 or 16): a tuning knob that fixes the
    // selection's cluster size where it fits
    if (const char* env = std::getenv("KVO_SELECT_CLUSTER")) {
      const int m = std::atoi(env);
      if (m == 1 || m == 2 || m == 4 || m == 8 || m == 16) cfg.force_select = m;
    }
    cfg.init = true;
  }
  *out = &cfg;
  return cudaSuccess;
}

// CTAs per selecting cluster, at least min_cluster: the size with the fewest
// waves of clusters, ties to the larger clusters (so the largest size whose
// clusters all run in one wave, when there is one).
uint32_t select_cluster(const int* active, uint32_t nsel, int max_cluster, int min_cluster = 1) {
  int best = 0;
  uint32_t best_waves = 0xffffffffu;
  for (int i = 4; i >= 0; --i) {
    const int C = 1 << i;
    if (C > max_cluster || C < min_cluster || active[i] <= 0) continue;
    const uint32_t waves = (nsel + (uint32_t)active[i] - 1) / (uint32_t)active[i];
    if (waves < best_waves) {
      best_waves = waves;
      best = C;
    }
  }
  return (uint32_t)best;
}

LayerCall make_call(const StepTask& s, uint32_t layer) {
  LayerCall t;
  std::memset(static_cast<void*>(&t), 0, sizeof t);
  const LayerView& L = s.L;
  t.scores = s.scores;
  t.idx = s.idx;
  t.out_rows = s.out_rows;
  t.out_bf16 = s.out_bf16;
  t.fresh = s.r ? static_cast<const uint8_t*>(s.new_rows) : nullptr;
  t.layer = layer;
  t.n = s.n;
  t.ram_len = L.ram_len;
  t.len = s.old_len + s.r;
  t.fresh_from = s.old_len;
  t.r = s.r;
  t.to_ram = !L.ring_rows ? s.r : L.ram_len <= s.old_len ? 0u : (L.ram_len - s.old_len < s.r ? L.ram_len - s.old_len : s.r);
  return t;
}

cudaError_t launch_config(const void* kern, dim3 grid, uint32_t threads, size_t smem, cudaStream_t stream,
                          uint32_t cluster, bool after_previous, cudaLaunchConfig_t* lc, cudaLaunchAttribute* attr) {
  (void)kern;
  *lc = cudaLaunchConfig_t{};
  lc->gridDim = grid;
  lc->blockDim = dim3(threads, 1, 1);
  lc->dynamicSmemBytes = smem;
  lc->stream = stream;
  uint32_t na = 0;
  if (cluster > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = cluster;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (after_previous) {                                  // scheduled early, waits in griddepcontrol.wait
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  lc->attrs = attr;
  lc->numAttrs = na;
  return cudaSuccess;
}

}  // namespace

namespace {

// Launch parameters, reused from call to call: clear() keeps the storage, so
// a call does not zero 10 KB per batch; push() hands out the next one.
struct BatchList {
  std::vector<LayerBatch> store;
  size_t n = 0;
  void clear() { n = 0; }
  bool empty() const { return n == 0; }
  size_t size() const { return n; }
  LayerBatch& back() { return store[n - 1]; }
  LayerBatch& operator[](size_t i) { return store[i]; }
  LayerBatch& push() {
    if (n == store.size()) store.emplace_back();
    LayerBatch& b = store[n++];
    b.ntasks = 0;
    b.deferred = 0;
    return b;
  }
  LayerBatch* begin() { return store.data(); }
  LayerBatch* end() { return store.data() + n; }
};

// Launch parameters of one part of a call, built before its first launch.
struct PartBuffers {
  BatchList sel, res;
  std::vector<uint32_t> sel_c;
  std::vector<uint8_t> sel_resident;
};

// One part of a call on one stream: the selections of its selecting layers,
// then the resolves, then the gathers of all its layers.  which[0..n): the
// part's tasks.  after_select: recorded once the selections are enqueued
// (NULL: none).  ev: the phase events (NULL: none).
cudaError_t enqueue_part(LayersConfig* cfg, const StepTask* tasks, const uint32_t* layers, const uint32_t* which,
                         uint32_t n, uint32_t k, const LayerStatic* statics, uint32_t* status, int max_cluster,
                         cudaStream_t stream, cudaEvent_t* ev, cudaEvent_t after_select, PartBuffers& pb,
                         uint32_t* hist, const LayersFilter* filt, uint32_t* ent, const LayersDefer* defer,
                         uint32_t* launched) {
  cudaError_t e;
  pb.sel.clear();
  pb.res.clear();
  pb.sel_c.clear();
  pb.sel_resident.clear();
  for (uint32_t w = 0; w < n; ++w) {
    const uint32_t i = which[w];
    if (!tasks[i].scores) continue;
    if (pb.sel.empty() || pb.sel.back().ntasks == kBatchTasks) pb.sel.push();
    LayerBatch& sb = pb.sel.back();
    sb.t[sb.ntasks++] = make_call(tasks[i], layers[i]);
  }
  size_t slices = 0;                                     // filter slices handed out so far
  for (LayerBatch& sb : pb.sel) {
    uint32_t nmax = 0;
    for (uint32_t i = 0; i < sb.ntasks; ++i) nmax = sb.t[i].n > nmax ? sb.t[i].n : nmax;
    // resident keys when every selecting layer's slice fits the CTA's
    // shared memory (the smallest such cluster and up), else the filtered
    // route
    // With the whole-GPU histogram every selection takes the filtered route
    // (the keys in and above the cut bucket, a few thousand, rather than all
    // of them: 50K positions, 4-CTA clusters: ~19 us per selection on the
    // resident route); without it, resident keys where they fit.
    int cmin = 1;
    while (cmin <= 16 && (uint64_t)topk_detail::topk_chunk(nmax, (uint32_t)cmin) * 4u > kSelectMaxSmem) cmin <<= 1;
    if (cfg->force_select && cfg->force_select >= cmin) cmin = cfg->force_select;
    uint32_t C = !hist && cmin <= 16
                     ? select_cluster(cfg->active, sb.ntasks, cfg->force_select ? cmin : max_cluster, cmin)
                     : 0u;
    const bool resident = C != 0;
    if (!resident)
      C = select_cluster(cfg->active_stream, sb.ntasks, cfg->force_select ? cfg->force_select : max_cluster,
                         cfg->force_select ? cfg->force_select : 2);
    if (!C) return cudaErrorInvalidConfiguration;
    sb.statics = statics;
    sb.k = k;
    sb.cand_bytes = resident ? (uint32_t)topk_detail::topk_chunk(nmax, C) * 4u : topk_detail::kTopkMaxDynSmem;
    // the filtered route takes its first histogram, and the candidate
    // lists, from the whole-GPU histogram launch
    for (uint32_t i = 0; i < sb.ntasks; ++i) {
      LayerCall& c = sb.t[i];
      c.first_hist = !resident && hist ? hist + (size_t)c.layer * kLayersHistWords : nullptr;
      const size_t ns = (c.n + kHistSlice - 1) / kHistSlice;
      if (c.first_hist && filt && slices + ns <= filt->slices) {
        c.cand_count = filt->count + slices;
        c.cand_key = filt->key + slices * kHistSlice;
        c.cand_pos = filt->pos + slices * kHistSlice;
        slices += ns;
      }
    }
    sb.chunks = (nmax + kHistSlice - 1) / kHistSlice;
    pb.sel_c.push_back(C);
    pb.sel_resident.push_back(resident ? 1 : 0);
  }
  for (uint32_t first = 0; first < n; first += kBatchTasks) {
    LayerBatch& rb = pb.res.push();
    rb.ntasks = n - first < kBatchTasks ? n - first : kBatchTasks;
    for (uint32_t i = 0; i < rb.ntasks; ++i) {
      rb.t[i] = make_call(tasks[which[first + i]], layers[which[first + i]]);
      rb.t[i].ent = ent + (size_t)rb.t[i].layer * KVO_MAX_K;
    }
    rb.statics = statics;
    rb.k = k;
    rb.chunks = (k + kGatherEntries - 1) / kGatherEntries;
    rb.deferred = defer ? 1u : 0u;
    if (defer) {
      rb.dlist = defer->dlist_dev;
      rb.dcount = defer->dcount_dev;
      rb.plist = defer->plist_dev;
      rb.pcount = defer->pcount_dev;
      rb.staging = defer->staging;
    }
  }

  cudaLaunchConfig_t lc;
  cudaLaunchAttribute attr[2];
  bool after = false;                                    // a launch of this part precedes on the stream
  if (ev && (e = cudaEventRecord(ev[0], stream)) != cudaSuccess) return e;
  for (size_t i = 0; i < pb.sel.size(); ++i) {
    const bool resident = pb.sel_resident[i] != 0;
    bool hist_before = false;
    if (!resident && hist) {
      layers_hist_kernel<<<pb.sel[i].ntasks * pb.sel[i].chunks, kHistThreads, 0, stream>>>(pb.sel[i]);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
      ++*launched;
      hist_before = true;
    }
    launch_config(nullptr, dim3(pb.sel_c[i] * pb.sel[i].ntasks, 1, 1), kThreads,
                  resident ? pb.sel[i].cand_bytes : topk_detail::kTopkMaxDynSmem, stream, pb.sel_c[i],
                  hist_before && !ev, &lc, attr);
    e = resident ? cudaLaunchKernelEx(&lc, layers_select_kernel<true>, pb.sel[i])
                 : cudaLaunchKernelEx(&lc, layers_select_kernel<false>, pb.sel[i]);
    if (e != cudaSuccess) return e;
    after = true;
    ++*launched;
  }
  if (after_select && (e = cudaEventRecord(after_select, stream)) != cudaSuccess) return e;
  if (ev && (e = cudaEventRecord(ev[1], stream)) != cudaSuccess) return e;
  // (an event between two launches ends the early scheduling of the second)
  const bool pdl = !ev && !after_select;
  const size_t rsmem = resolve_smem_bytes(k, tasks[which[0]].L.hot_rows);
  for (const LayerBatch& rb : pb.res) {
    launch_config(nullptr, dim3(rb.ntasks, 1, 1), kThreads, rsmem, stream, 1, pdl && after, &lc, attr);
    e = tasks[which[0]].L.policy == KVO_POLICY_LRU
            ? cudaLaunchKernelEx(&lc, layers_resolve_kernel<true>, rb, status)
            : cudaLaunchKernelEx(&lc, layers_resolve_kernel<false>, rb, status);
    if (e != cudaSuccess) return e;
    after = true;
    ++*launched;
  }
  if (ev && (e = cudaEventRecord(ev[2], stream)) != cudaSuccess) return e;
  uint32_t nl = 0;                                       // the batched-copy counters up to the part's highest layer
  if (defer) {
    for (uint32_t w = 0; w < n; ++w) nl = layers[which[w]] + 1 > nl ? layers[which[w]] + 1 : nl;
    if ((e = cudaMemcpyAsync(defer->dcount_host, defer->dcount_dev, sizeof(uint32_t) * nl, cudaMemcpyDeviceToHost,
                             stream)) != cudaSuccess)
      return e;
    if ((e = cudaEventRecord(defer->listed, stream)) != cudaSuccess) return e;
  }
  for (const LayerBatch& rb : pb.res) {
    launch_config(nullptr, dim3(rb.ntasks * rb.chunks, 1, 1), kGatherThreads, 0, stream, 1, pdl && !defer, &lc,
                  attr);
    if ((e = cudaLaunchKernelEx(&lc, layers_gather_kernel, rb, status)) != cudaSuccess) return e;
    ++*launched;
  }
  if (defer) {
    // The batched-copy fetch: wait for the lists (the gathers of the other
    // rows run meanwhile), copy every run of consecutive missing positions
    // with one cudaMemcpyAsync into staging (rows in position order), then
    // place the rows.
    if ((e = cudaEventSynchronize(defer->listed)) != cudaSuccess) return e;
    static thread_local std::vector<int2> ent;
    static thread_local std::vector<int32_t> uniq;
    for (uint32_t w = 0; w < n; ++w) {
      const uint32_t l = layers[which[w]];
      const uint32_t m = defer->dcount_host[l] < k ? defer->dcount_host[l] : k;
      const int2* dl = defer->dlist_host + (size_t)l * KVO_MAX_K;
      ent.assign(dl, dl + m);
      uniq.resize(m);
      for (uint32_t i = 0; i < m; ++i) uniq[i] = ent[i].y;
      std::sort(uniq.begin(), uniq.end());
      uniq.erase(std::unique(uniq.begin(), uniq.end()), uniq.end());
      uint8_t* stage = defer->staging + (size_t)l * k * KVO_ROW_BYTES;
      const uint8_t* hist_h = defer->hist_host[l];
      for (size_t a = 0; a < uniq.size();) {              // one copy per run of consecutive positions
        size_t z = a + 1;
        while (z < uniq.size() && uniq[z] == uniq[z - 1] + 1) ++z;
        if ((e = cudaMemcpyAsync(stage + a * KVO_ROW_BYTES, hist_h + (size_t)uniq[a] * KVO_ROW_BYTES,
                                 (z - a) * KVO_ROW_BYTES, cudaMemcpyHostToDevice, stream)) != cudaSuccess)
          return e;
        a = z;
      }
      int2* pl = defer->plist_host + (size_t)l * KVO_MAX_K;
      for (uint32_t i = 0; i < m; ++i) {
        const int32_t srow = (int32_t)(std::lower_bound(uniq.begin(), uniq.end(), ent[i].y) - uniq.begin());
        pl[i] = make_int2(ent[i].x, srow);
      }
      defer->pcount_host[l] = m;
    }
    for (const LayerBatch& rb : pb.res) {
      launch_config(nullptr, dim3(rb.ntasks * rb.chunks, 1, 1), kGatherThreads, 0, stream, 1, false, &lc, attr);
      if ((e = cudaLaunchKernelEx(&lc, layers_place_kernel, rb, status)) != cudaSuccess) return e;
      ++*launched;
    }
  }
  if (ev && (e = cudaEventRecord(ev[3], stream)) != cudaSuccess) return e;
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_layers(const StepTask* tasks, const uint32_t* layers, uint32_t ntasks, uint32_t k,
                          const LayerStatic* statics, uint32_t* status, int max_cluster, cudaStream_t stream,
                          cudaEvent_t* ev, uint32_t* hist, const LayersFilter* filt, uint32_t* ent,
                          const LayersDefer* defer, uint32_t* launched) {
  LayersConfig* cfg = nullptr;
  cudaError_t e = layers_init(&cfg);
  if (e != cudaSuccess) return e;
  static thread_local PartBuffers pb;
  static thread_local std::vector<uint32_t> all;
  all.resize(ntasks);
  for (uint32_t i = 0; i < ntasks; ++i) all[i] = i;
  return enqueue_part(cfg, tasks, layers, all.data(), ntasks, k, statics, status, max_cluster, stream, ev, nullptr,
                      pb, hist, filt, ent, defer, launched);
}

}  // namespace kvo
