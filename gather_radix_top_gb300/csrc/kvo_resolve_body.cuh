// Device body of the resolve + gather call, shared by the standalone kernel
// and the fused decode-step kernel.
//
// "From 1M Total to 15+ x 1M Contexts: GLM-5.3 KV Cache Offloading":
//   section "Decision three: let the GPU manage the hot cache directly" -
//     selection stays on the GPU, which checks hot slots directly; hits read
//     the HBM slot, misses read the registered host copy of the history, and
//     the gather emits a compact selection for attention;
//   section "GPU cache management has hazards too" - a slot filled in this
//     round is a hit source only from the next round on, duplicate misses
//     read host memory directly, and slots used by this round are pinned.
// Victims are the least recently used unpinned slots, keyed (last_use, slot).
//
// One thread-block cluster runs the whole call.  CTA 0 keeps the LRU order;
// every other CTA owns a contiguous range of selection entries j; every CTA
// owns a contiguous range of hot slots.  The LRU order
// is a per-layer queue of (stamp, slot) entries in HBM: every call appends
// one entry, stamped with its step, for every slot it used (hits and fills),
// in slot order, so the queue runs in (last_use, slot) order; an entry is
// current while last_use[slot] still equals its stamp, and older entries of
// a slot are stale and skipped.
//   P1 classify: hit = pos2slot[p] >= 0 (stamp last_use = t, set the slot's
//      bit in its owner's used-slot bitmap over DSMEM and count it for the
//      owner's range); a miss does an atomicMin of a negative
//      first-occurrence code into pos2slot[p], so the smallest j of each
//      missing position wins (dedupe without a table).  Then, while the
//      cluster barrier completes, every row is gathered: hits from the hot
//      slot (HBM), misses from host memory (zero-copy), 16-byte pieces, one
//      warp per 656-byte row, plus the bf16 dequant.  A CTA whose misses are
//      a large enough share of its entries stages instead: its device-memory
//      rows arrive by TMA bulk copies and its host rows by the same 16-byte
//      loads, into shared memory, and its output slice leaves in one bulk
//      store.
//   P2 unique misses are ranked in j order.  When idx is strictly increasing
//      (always true for kvo_select_topk output) every miss is unique and the
//      counts published at the first barrier give every rank; otherwise the
//      claims are re-read and the counts published once more.
//   P3 victims: CTA 0 copies the head of the queue (TMA bulk copy) and reads
//      its entries' last_use while the other CTAs classify and gather; after
//      the barrier it only has to drop the slots pinned in this call.  It
//      walks the queue from its head.  The current entries,
//      in order, are the unpinned slots by (last_use, slot) (a slot used in
//      this call was stamped with t, so its entry is stale); the i-th one
//      is the victim of the i-th unique miss and goes to the CTA holding
//      that miss.  CTA 0 also hands every CTA the queue position of its
//      range's used slots.
//   P4 the CTA holding a miss unmaps the evicted position, maps the new one,
//      stamps last_use = t and copies the row (its staged copy, the output
//      just written, or its source) into the victim slot.
//   P5 every CTA appends its range's used slots, in slot order, stamped t.
// When the queue nears its capacity, its current entries are first copied,
// in order, to the other of its two buffers (a compaction, once every many
// calls).
// With the circular policy there is no queue: CTA 0 walks the slots from the
// layer's hand instead, skipping the pinned ones, and P5 has nothing to do.
#pragma once

#include <cstdint>

#include <cuda_fp16.h>

#include "kvo_device.cuh"
#include "kvo_internal.h"

namespace kvo {

namespace resolve_detail {

constexpr int32_t kSlotMiss = -1;
constexpr int32_t kSlotInvalid = -2;
constexpr uint32_t kRowVec = KVO_ROW_BYTES / 16;   // 41 16-byte pieces per row
constexpr uint32_t kRowsInFlight = 4;               // rows a warp loads before it stores
constexpr uint32_t kNoRank = 0xffffffffu;
constexpr uint32_t kWindow = 4 * kThreads;          // LRU queue entries CTA 0 examines per round
constexpr uint32_t kWindowPolls = 1u << 18;         // bound on the wait for the window copy (~20 ms)
constexpr uint32_t kStageMax = 160;                 // rows one CTA stages at most (105 KB of shared memory)

struct ResolveArgs {
  LayerView L;
  const int32_t* idx;
  uint8_t* out_rows;
  uint16_t* out_bf16;
  uint32_t* status;
  uint32_t k;
  uint32_t kchunk;        // selection entries per CTA (CTAs 1..C-1; CTA 0 has none)
  uint32_t hchunk;        // hot slots per CTA, a multiple of 128
  // Staged gather (rows pulled into shared memory by TMA bulk copies, the
  // CTA's output slice written back with one bulk store) when the CTA's
  // entries fit `stage_rows` rows and its share of misses is at least
  // stage_min_miss_pct percent; else rows pass through registers.
  uint32_t stage_rows;
  uint32_t stage_min_miss_pct;
  // decode-step launches: the history length is `len`, and positions >=
  // fresh_from were appended by this very launch and are read from `fresh`
  // (device memory) rather than from host memory
  uint32_t fused;
  // the selection was handed over in shared memory (`sel`, ascending) by the
  // top-K phase of the same launch, rather than read from `idx`
  uint32_t sel_in_smem;
  uint32_t len;
  const uint8_t* fresh;
  uint32_t fresh_from;
  // out_rows is (mapped) host memory: written with plain stores only, and
  // never read back (the fills take their rows from the rows' sources)
  uint32_t out_host;
};

// The row of a missing position: for rows appended in the same fused launch
// their device copy; for rows still waiting in the recent ring (at or above
// the host history's length) the ring; else the host history.
__device__ __forceinline__ const uint4* miss_row(const ResolveArgs& a, const uint4* hist4, int32_t p) {
  if (a.fresh && (uint32_t)p >= a.fresh_from)
    return reinterpret_cast<const uint4*>(a.fresh) + (size_t)((uint32_t)p - a.fresh_from) * kRowVec;
  if (a.L.ring_rows && (uint32_t)p >= a.L.ram_len)
    return reinterpret_cast<const uint4*>(a.L.recent) + (size_t)((uint32_t)p & (a.L.ring_rows - 1u)) * kRowVec;
  return hist4 + (size_t)p * kRowVec;
}

// Whether a missing position is read from the host history.
__device__ __forceinline__ bool miss_from_host(const ResolveArgs& a, int32_t p) {
  if (a.fresh && (uint32_t)p >= a.fresh_from) return false;
  return !(a.L.ring_rows && (uint32_t)p >= a.L.ram_len);
}

// A row appended by this launch whose position the host history (RAM)
// already holds at this step: without a recent ring every appended row, with
// one the rows whose copyback batch completes in this step.  Such a miss is
// counted as a RAM read, as the append-then-resolve order defines it; the
// launch serves it from the row's device copy, which holds the same bytes.
__device__ __forceinline__ bool fresh_in_ram(const ResolveArgs& a, int32_t p) {
  return a.fresh && (uint32_t)p >= a.fresh_from && !(a.L.ring_rows && (uint32_t)p >= a.L.ram_len);
}

struct SmemLayout {
  uint32_t pinbits, meta_slot, meta_pos, uniq, sel, vslot, mlist, window, fullpin, total;
};

__host__ __device__ inline uint32_t round16(uint32_t x) { return (x + 15u) & ~15u; }

// hchunk: slots per CTA, a multiple of 128 (whole 16-byte pieces of bitmap).
__host__ __device__ inline SmemLayout smem_layout(uint32_t k, uint32_t kchunk, uint32_t hchunk, uint32_t hot_rows,
                                                  uint32_t stage_rows = 0) {
  (void)k;
  SmemLayout s;
  uint32_t o = 0;
  s.pinbits = o;   o += round16(hchunk / 8u);   // this CTA's slots used in this call
  s.meta_slot = o; o += kchunk * 4u;            // per entry: hot slot, or miss / invalid
  s.meta_pos = o;  o += kchunk * 4u;            // per entry: position
  s.uniq = o;      o += kchunk * 4u;            // per entry: rank among this CTA's unique misses, or kNoRank
  s.sel = o;       o += kchunk * 4u;            // fused step: this CTA's selected positions
  s.vslot = o;     o += kchunk * 4u;            // per unique miss (local rank): its victim slot
  s.mlist = o;     o += kchunk * 4u;            // per unique miss (local rank): its entry
  o = round16(o);
  s.window = o;                                 // CTA 0: the first queue entries, copied early;
  o += kWindow * 8u > stage_rows * (uint32_t)KVO_ROW_BYTES     // other CTAs: their staged rows
           ? kWindow * 8u
           : stage_rows * (uint32_t)KVO_ROW_BYTES;
  s.fullpin = o;   o += round16((hot_rows + 31u) / 32u * 4u);   // CTA 0: every slot hit in this call
  s.total = round16(o);
  return s;
}

// Round-to-nearest-even of a float32 to bf16, from the IEEE-754 definition:
// keep the upper 16 bits and round on the lower 16 (above half up, below
// half down, exactly half to the even result).  NaN stays a quiet NaN.
__device__ __forceinline__ uint32_t bf16_rne(float x) {
  const uint32_t u = __float_as_uint(x);
  const uint32_t upper = u >> 16, lower = u & 0xffffu;
  if ((u & 0x7fffffffu) > 0x7f800000u) return upper | 0x40u;
  const uint32_t up = (lower > 0x8000u) || (lower == 0x8000u && (upper & 1u));
  return (upper + up) & 0xffffu;
}

__device__ __forceinline__ uint32_t pack2(float a, float b) { return bf16_rne(a) | (bf16_rne(b) << 16); }

__device__ __forceinline__ void dequant4(uint32_t w, float s, float* o) {
  o[0] = (float)(int8_t)(w & 0xffu) * s;
  o[1] = (float)(int8_t)((w >> 8) & 0xffu) * s;
  o[2] = (float)(int8_t)((w >> 16) & 0xffu) * s;
  o[3] = (float)(int8_t)(w >> 24) * s;
}

// Dequantises the row held by a warp (va = piece `lane`, vb = piece 32+lane)
// into 576 bf16: latent piece `lane` lies in scale group lane / 4; lane 0's
// second piece holds the 8 fp16 scales; lanes 1..8 hold the RoPE pieces.
__device__ __forceinline__ void dequant_row(const uint4& va, const uint4& vb, uint32_t lane, uint4* d) {
  const uint32_t s01 = __shfl_sync(0xffffffffu, vb.x, 0);
  const uint32_t s23 = __shfl_sync(0xffffffffu, vb.y, 0);
  const uint32_t s45 = __shfl_sync(0xffffffffu, vb.z, 0);
  const uint32_t s67 = __shfl_sync(0xffffffffu, vb.w, 0);
  const uint32_t g = lane >> 2;
  const uint32_t w = g < 2 ? s01 : g < 4 ? s23 : g < 6 ? s45 : s67;
  const float s = __half2float(__ushort_as_half((uint16_t)((g & 1) ? (w >> 16) : (w & 0xffffu))));
  float f[16];
  dequant4(va.x, s, f);
  dequant4(va.y, s, f + 4);
  dequant4(va.z, s, f + 8);
  dequant4(va.w, s, f + 12);
  d[2 * lane] = make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]), pack2(f[6], f[7]));
  d[2 * lane + 1] = make_uint4(pack2(f[8], f[9]), pack2(f[10], f[11]), pack2(f[12], f[13]), pack2(f[14], f[15]));
  if (lane >= 1 && lane < kRowVec - 32) d[64 + (lane - 1)] = vb;   // RoPE, copied
}

// One map update: slot v receives position p, evicting `old` (or -1).
// Returns 1 when a mapped position was evicted.
__device__ __forceinline__ uint32_t map_update(const ResolveArgs& a, uint32_t v, int32_t old, int32_t p,
                                               uint32_t t, uint32_t e) {
  const LayerView& L = a.L;
  if (v >= L.hot_rows || p < 0 || (uint32_t)p >= L.history_cap) {
    atomicOr(a.status, kFlagInternal);              // cannot happen; never write out of bounds
    return 0;
  }
  if (old >= 0) L.pos2slot[old] = -1;
  L.pos2slot[p] = (int32_t)v;
  L.slot2pos[v] = p;
  L.last_use[v] = t;
  if (L.evlog) {
    L.evlog[1 + 3 * e] = (int32_t)v;
    L.evlog[2 + 3 * e] = old;
    L.evlog[3 + 3 * e] = p;
  }
  return old >= 0 ? 1u : 0u;
}

// A queue entry: stamp in the upper 32 bits, slot in the lower.
__device__ __forceinline__ bool entry_current(const LayerView& L, uint64_t e) {
  const uint32_t sl = (uint32_t)e;
  return sl < L.hot_rows && __ldcg(&L.last_use[sl]) == (uint32_t)(e >> 32);
}

// Copies the current entries of [head, tail) of ring buffer `buf`, in order,
// to the front of the other buffer.  Every CTA of the cluster calls it; it
// returns the number of entries kept (the number of slots).
static __device__ __noinline__ uint32_t compact_queue(const LayerView& L, uint32_t head, uint32_t tail, uint32_t buf,
                                  uint32_t (*scratch)[2 * kWarps + 2], uint32_t (*table)[4]) {
  const uint32_t tid = threadIdx.x, r = cluster_rank(), C = cluster_size();
  const uint32_t Q = L.ring_cap, qmask = Q - 1u;
  const uint64_t* src = L.ring + (size_t)buf * Q;
  uint64_t* dst = L.ring + (size_t)(buf ^ 1u) * Q;
  const uint32_t span = tail - head;
  const uint32_t chunk = (span + C - 1u) / C;
  const uint32_t lo = min(span, r * chunk), hi = min(span, lo + chunk);
  cluster_sync();                                   // every CTA is running before the publish below
  uint32_t c = 0;
  for (uint32_t i = lo + tid; i < hi; i += kThreads) c += entry_current(L, src[(head + i) & qmask]);
  const uint32_t mine[1] = {block_sum(c, scratch[1])};
  cluster_publish(mine, 1, table, r, C);
  uint32_t before = 0, total = 0;
  for (uint32_t q = 0; q < C; ++q) {
    before += q < r ? table[q][0] : 0u;
    total += table[q][0];
  }
  uint32_t run = 0;
  for (uint32_t base = lo; base < hi; base += kThreads) {
    const uint32_t i = base + tid;
    uint64_t e = 0;
    bool keep = false;
    if (i < hi) {
      e = src[(head + i) & qmask];
      keep = entry_current(L, e);
    }
    uint32_t tile;
    const uint32_t rank = block_flag_scan(keep, scratch[0], &tile);
    if (keep && before + run + rank < Q) dst[before + run + rank] = e;
    run += tile;
  }
  return total;
}

// No work for the CTAs that wait while CTA 0 picks the victims.
struct NoIdleWork {
  __device__ void operator()(uint32_t, uint32_t) const {}
};

// kLru: the layer's policy (KVO_POLICY_LRU, else KVO_POLICY_CIRCULAR); each
// policy gets its own kernel so that neither carries the other's code.
// idle(w, nw): called by every CTA but CTA 0 while CTA 0 picks the victims
// (w = this CTA's first warp among nw warps of those CTAs, all of them
// calling with the same nw); it must not touch the resolve's state.
template <bool kLru, typename IdleWork = NoIdleWork>
__device__ __forceinline__ void resolve_body(const ResolveArgs& a, uint8_t* dyn_smem, IdleWork idle = IdleWork()) {
  __shared__ uint32_t scratch[2][2 * kWarps + 2];
  __shared__ uint32_t table[kMaxCluster][4];       // per CTA: (idx not increasing, misses)
  __shared__ uint32_t table2[kMaxCluster][4];      // idx not increasing: (unique misses, used hit slots)
  __shared__ uint32_t hitcnt[kMaxCluster];         // CTA 0: hit slots per owner range
  __shared__ uint32_t fillcnt[kMaxCluster];        // CTA 0: victims per owner range
  __shared__ uint32_t own_hits[kMaxCluster];       // this CTA's hits per owner range
  __shared__ uint32_t mbefore[kMaxCluster + 1];    // CTA 0: unique misses of lower CTAs
  __shared__ uint32_t ring_off;                    // queue position of this range's used slots
  __shared__ uint32_t head_hit;                    // CTA 0: offset of the first current entry left
  __shared__ uint32_t last_vic;                    // CTA 0: the last victim (circular policy)
  __shared__ uint32_t nevict_cta;
  __shared__ uint32_t cta_hits, cta_inv, cta_host;
  __shared__ uint32_t cta_fresh_ram;               // misses on this launch's rows that RAM already holds
  __shared__ __align__(8) uint64_t wbar;           // CTA 0: completion of the window copy
  __shared__ __align__(8) uint64_t gbar;           // other CTAs: completion of the staged rows

  const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t r = cluster_rank(), C = cluster_size();
  const LayerView& L = a.L;
  const uint32_t k = a.k;
  const uint32_t H = L.hot_rows;

  const SmemLayout lay = smem_layout(k, a.kchunk, a.hchunk, H, a.stage_rows);
  uint32_t* pinbits = reinterpret_cast<uint32_t*>(dyn_smem + lay.pinbits);
  int32_t* meta_slot = reinterpret_cast<int32_t*>(dyn_smem + lay.meta_slot);
  int32_t* meta_pos = reinterpret_cast<int32_t*>(dyn_smem + lay.meta_pos);
  uint32_t* uniq = reinterpret_cast<uint32_t*>(dyn_smem + lay.uniq);
  const int32_t* sel = reinterpret_cast<const int32_t*>(dyn_smem + lay.sel);
  uint32_t* vslot = reinterpret_cast<uint32_t*>(dyn_smem + lay.vslot);
  uint32_t* mlist = reinterpret_cast<uint32_t*>(dyn_smem + lay.mlist);
  uint64_t* window = reinterpret_cast<uint64_t*>(dyn_smem + lay.window);
  uint32_t* fullpin = reinterpret_cast<uint32_t*>(dyn_smem + lay.fullpin);

  const uint32_t t = L.counters[0] + 1u;        // this call's step
  const uint32_t len = a.fused ? a.len : L.counters[1];
  uint32_t head = L.counters[2], tail = L.counters[3], buf = L.counters[4] & 1u;
  const uint32_t hand = L.counters[5];
  constexpr bool lru = kLru;
  const uint32_t Q = L.ring_cap, qmask = Q - 1u;
  const uint32_t jlo = r == 0 ? 0u : min(k, (r - 1u) * a.kchunk);
  const uint32_t jcnt = r == 0 ? 0u : min(k, jlo + a.kchunk) - jlo;
  const uint32_t slo = min(H, r * a.hchunk), shi = min(H, slo + a.hchunk), hcnt = shi - slo;
  const uint32_t words = a.hchunk / 32u;         // used-slot bitmap words per CTA

  // ------------------------------------------------- queue compaction
  // This call appends at most k entries; make room first when needed (every
  // CTA read the same counters, so every CTA takes the same branch).
  if (lru && tail - head > Q - k) {
    tail = compact_queue(L, head, tail, buf, scratch, table2);
    head = 0;
    buf ^= 1u;
    if (r == 0 && tid == 0 && tail != H) atomicOr(a.status, kFlagInternal);
    cluster_sync();                                 // the compacted queue is complete before CTA 0 reads it
  }
  const uint64_t* ring_in = L.ring + (size_t)buf * Q;
  uint64_t* ring_out = L.ring + (size_t)buf * Q;

  // ---------------------------------------------------------------- P0
  for (uint32_t i = tid; i < words; i += kThreads) pinbits[i] = 0;
  for (uint32_t i = tid; i < jcnt; i += kThreads) vslot[i] = kNoRank;
  if (r == 0)
    for (uint32_t i = tid; i < (H + 31u) / 32u; i += kThreads) fullpin[i] = 0;
  if (tid < kMaxCluster) {
    hitcnt[tid] = 0;
    fillcnt[tid] = 0;
    own_hits[tid] = 0;
  }
  if (tid == 0) {
    nevict_cta = 0;
    ring_off = 0;
    head_hit = kNoRank;
    cta_fresh_ram = 0;
  }
  // CTA 0 copies the head of the queue now (one or two bulk copies from a
  // 16-byte boundary: window[sh + o] is the entry o places after the head);
  // the victims come from it later.
  const uint32_t span = tail - head;
  const uint32_t sh = head & 1u;
  const uint32_t wcopy = (min(span + sh, kWindow) + 1u) & ~1u;   // entries copied, even
  uint32_t wlen = !lru ? 0u : wcopy - sh < span ? wcopy - sh : span;   // entries usable from the window
  if (lru && r == 0 && tid == 0) {
    asm volatile("fence.proxy.async.global;" ::: "memory");   // a compaction above wrote the queue
    mbar_init(&wbar, 1);
    const uint32_t a0 = (head - sh) & qmask;
    const uint32_t first = min(wcopy, Q - a0);
    mbar_arrive_expect_tx(&wbar, wcopy * 8u);
    bulk_copy_g2s(window, ring_in + a0, first * 8u, &wbar);
    if (wcopy > first) bulk_copy_g2s(window + first, ring_in, (wcopy - first) * 8u, &wbar);
  }
  __syncthreads();                                  // the counters above are zero before P1 adds into them
  // B0: every CTA of the cluster is running (and has zeroed what others add
  // into) before any DSMEM access; classification overlaps the barrier.
  cluster_arrive();

  // ---------------------------------------------------------------- P1
  uint32_t nhit = 0, nmiss = 0, nhost = 0, ninv = 0, unordered = 0;   // per thread
  for (uint32_t jj = tid; jj < jcnt; jj += kThreads) {
    const uint32_t j = jlo + jj;
    // a selection made in the same launch comes from shared memory, ascending
    const int32_t p = a.sel_in_smem ? sel[jj] : a.idx[j];
    if (!a.sel_in_smem && j > 0 && a.idx[j - 1] >= p) ++unordered;
    int32_t slot;
    if (p < 0 || (uint32_t)p >= len) {
      slot = kSlotInvalid;
      ++ninv;
    } else {
      int32_t s = L.pos2slot[p];
      if (s >= (int32_t)H) {
        atomicOr(a.status, kFlagInternal);          // cannot happen; keep every index in bounds
        s = -1;
      }
      if (s >= 0) {
        slot = s;
        L.last_use[s] = t;
        atomicAdd(&own_hits[(uint32_t)s / a.hchunk], 1u);
        ++nhit;
      } else {
        slot = kSlotMiss;
        atomicMin(&L.pos2slot[p], (int32_t)j - (int32_t)k - 1);
        ++nmiss;
        nhost += miss_from_host(a, p);
        if (fresh_in_ram(a, p)) atomicAdd(&cta_fresh_ram, 1u);
      }
    }
    meta_slot[jj] = slot;
    meta_pos[jj] = p;
  }
  // local rank of each miss in j order (the global rank once the counts of
  // lower CTAs are known); every miss is unique when idx is increasing
  uint32_t cta_miss = 0;
  for (uint32_t base = 0; base < jcnt; base += kThreads) {
    const uint32_t jj = base + tid;
    const bool f = jj < jcnt && meta_slot[jj] == kSlotMiss;
    uint32_t tile;
    const uint32_t rank = block_flag_scan(f, scratch[0], &tile);
    if (jj < jcnt) uniq[jj] = f ? cta_miss + rank : kNoRank;
    if (f) mlist[cta_miss + rank] = jj;
    cta_miss += tile;
  }
  uint32_t cta_hit_inv;
  // per-thread counts are at most the CTA's entries (< 2^16): two per word
  uint32_t cta_unord_host;
  block_sum2(unordered | (nhost << 16), nhit | (ninv << 16), scratch[1], &cta_unord_host, &cta_hit_inv);
  const uint32_t cta_unordered = cta_unord_host & 0xffffu;
  if (tid == 0) {
    cta_hits = cta_hit_inv & 0xffffu;
    cta_host = cta_unord_host >> 16;
    cta_inv = cta_hit_inv >> 16;
  }
  cluster_wait();                                   // B0
  if (tid < 2 * C) dsmem_st_u32(dsmem_addr(&table[r][tid & 1], tid >> 1), (tid & 1) ? cta_miss : cta_unordered);
  // pin: every hit slot's bit goes to the CTA that owns the slot
  for (uint32_t jj = tid; jj < jcnt; jj += kThreads) {
    const int32_t sl = meta_slot[jj];
    if (sl >= 0) {
      const uint32_t owner = (uint32_t)sl / a.hchunk, b = (uint32_t)sl - owner * a.hchunk;
      dsmem_red_or_u32(dsmem_addr(&pinbits[b >> 5], owner), 1u << (b & 31));
      dsmem_red_or_u32(dsmem_addr(&fullpin[(uint32_t)sl >> 5], 0), 1u << ((uint32_t)sl & 31));
    }
  }
  // hit counts per owner range (exact when idx does not repeat a position)
  if (tid < C && own_hits[tid]) dsmem_red_add_u32(dsmem_addr(&hitcnt[tid], 0), own_hits[tid]);
  cluster_arrive();                                 // B1: stamps, claims, counts, pins

  const uint4* hot4 = reinterpret_cast<const uint4*>(L.hot);
  const uint4* hist4 = reinterpret_cast<const uint4*>(L.hist);
  uint4* stage4 = reinterpret_cast<uint4*>(dyn_smem + lay.window);
  const bool staged = a.stage_rows && jcnt && jcnt <= a.stage_rows &&
                      cta_miss * 100u >= a.stage_min_miss_pct * jcnt;   // uniform over the CTA
  bool gather_ok = true;
  if (staged) {
    // One bulk copy per row in device memory (hot slots, this launch's new
    // rows, the recent ring) into shared memory, all in flight at once.
    // Rows of the host history come in through plain 16-byte loads, one warp
    // per row: a bulk copy's first touch of a host page can take longer than
    // the bounded wait (one took over 20 ms on a 50K-token layer), loads do
    // not.  Invalid entries get a zero row.
    const uint32_t host_rows = cta_unord_host >> 16;   // this CTA's entries served from the host history
    if (tid == 0) {
      mbar_init(&gbar, 1);
      mbar_arrive_expect_tx(&gbar, (jcnt - cta_inv - host_rows) * (uint32_t)KVO_ROW_BYTES);
    }
    __syncthreads();
    for (uint32_t jj = tid; jj < jcnt; jj += kThreads) {
      const int32_t slot = meta_slot[jj];
      const bool from_host = slot == kSlotMiss && miss_from_host(a, meta_pos[jj]);
      const uint4* src = slot >= 0 ? hot4 + (size_t)slot * kRowVec
                         : slot == kSlotMiss && !from_host ? miss_row(a, hist4, meta_pos[jj])
                                                           : nullptr;
      if (src) {
        bulk_copy_g2s(stage4 + (size_t)jj * kRowVec, src, KVO_ROW_BYTES, &gbar);
      } else if (!from_host) {
        for (uint32_t v = 0; v < kRowVec; ++v) stage4[(size_t)jj * kRowVec + v] = make_uint4(0, 0, 0, 0);
      }
    }
    if (host_rows) {                                // up to kRowsInFlight host rows per warp in flight
      for (uint32_t jj0 = warp; jj0 < jcnt; jj0 += kWarps * kRowsInFlight) {
        uint4 va[kRowsInFlight], vb[kRowsInFlight];
        uint32_t hm = 0;                            // bit u: entry jj0 + u * kWarps is a host row (warp-uniform)
#pragma unroll
        for (uint32_t u = 0; u < kRowsInFlight; ++u) {
          const uint32_t jj = jj0 + u * kWarps;
          va[u] = make_uint4(0, 0, 0, 0);
          vb[u] = make_uint4(0, 0, 0, 0);
          if (jj < jcnt && meta_slot[jj] == kSlotMiss && miss_from_host(a, meta_pos[jj])) {
            const uint4* src = miss_row(a, hist4, meta_pos[jj]);
            va[u] = src[lane];
            if (lane < kRowVec - 32) vb[u] = src[32 + lane];
            hm |= 1u << u;
          }
        }
#pragma unroll
        for (uint32_t u = 0; u < kRowsInFlight; ++u) {
          if (!((hm >> u) & 1u)) continue;
          uint4* dst = stage4 + (size_t)(jj0 + u * kWarps) * kRowVec;
          dst[lane] = va[u];
          if (lane < kRowVec - 32) dst[32 + lane] = vb[u];
        }
      }
    }
    fence_proxy_async_smem();                       // the zero and host rows, before the bulk store reads them
    gather_ok = __syncthreads_and(mbar_wait_bounded(&gbar, 0, kWindowPolls));
    if (!gather_ok) {
      if (tid == 0) atomicOr(a.status, kFlagTimeout);
    } else {
      if (a.out_rows && a.out_host) {              // host memory: plain 16-byte stores
        uint4* o4 = reinterpret_cast<uint4*>(a.out_rows) + (size_t)jlo * kRowVec;
        for (uint32_t i = tid; i < jcnt * kRowVec; i += kThreads) o4[i] = stage4[i];
      } else if (a.out_rows && tid == 0) {         // this CTA's slice of the output is contiguous
        bulk_copy_s2g(a.out_rows + (size_t)jlo * KVO_ROW_BYTES, stage4, jcnt * (uint32_t)KVO_ROW_BYTES);
        bulk_commit();
      }
      if (a.out_bf16)
        for (uint32_t jj = warp; jj < jcnt; jj += kWarps) {
          const uint4 va = stage4[(size_t)jj * kRowVec + lane];
          const uint4 vb = lane < kRowVec - 32 ? stage4[(size_t)jj * kRowVec + 32 + lane] : make_uint4(0, 0, 0, 0);
          dequant_row(va, vb, lane, reinterpret_cast<uint4*>(a.out_bf16 + (size_t)(jlo + jj) * KVO_DEQUANT_VALUES));
        }
    }
  } else {
    // Each warp loads up to kRowsInFlight rows before storing any, so that
    // all of this CTA's rows are in flight at once.
    for (uint32_t jj0 = warp; jj0 < jcnt; jj0 += kWarps * kRowsInFlight) {
      uint4 va[kRowsInFlight], vb[kRowsInFlight];
#pragma unroll
      for (uint32_t u = 0; u < kRowsInFlight; ++u) {
        const uint32_t jj = jj0 + u * kWarps;
        va[u] = make_uint4(0, 0, 0, 0);
        vb[u] = make_uint4(0, 0, 0, 0);
        if (jj < jcnt) {
          const int32_t slot = meta_slot[jj];
          const uint4* src = nullptr;
          if (slot >= 0) src = hot4 + (size_t)slot * kRowVec;
          else if (slot == kSlotMiss) src = miss_row(a, hist4, meta_pos[jj]);
          if (src) {
            va[u] = src[lane];
            if (lane < kRowVec - 32) vb[u] = src[32 + lane];
          }
        }
      }
#pragma unroll
      for (uint32_t u = 0; u < kRowsInFlight; ++u) {
        const uint32_t jj = jj0 + u * kWarps;
        if (jj >= jcnt) break;
        const uint32_t j = jlo + jj;
        if (a.out_rows) {
          uint4* d = reinterpret_cast<uint4*>(a.out_rows) + (size_t)j * kRowVec;
          d[lane] = va[u];
          if (lane < kRowVec - 32) d[32 + lane] = vb[u];
        }
        if (a.out_bf16)
          dequant_row(va[u], vb[u], lane, reinterpret_cast<uint4*>(a.out_bf16 + (size_t)j * KVO_DEQUANT_VALUES));
      }
    }
  }
  // CTA 0 (no entries to gather): wait for the window and read its slots'
  // last_use now.  A stamp of this call may or may not be seen yet; either
  // way the entry's slot is pinned, and the pin bitmap drops it after B1.
  bool win_ok = true;
  uint32_t pre4 = 0;                                // bit q: entry 4 * tid + q of the window was current
  if (lru && r == 0) {
    win_ok = __syncthreads_and(mbar_wait_bounded(&wbar, 0, kWindowPolls));
    if (!win_ok) {
      wlen = 0;                                     // read the queue from global memory instead
      if (tid == 0) atomicOr(a.status, kFlagTimeout);
    }
    uint64_t e[4];
    uint32_t lu[4];
#pragma unroll
    for (uint32_t q = 0; q < 4; ++q) e[q] = 4 * tid + q < wlen ? window[sh + 4 * tid + q] : ~0ull;
#pragma unroll
    for (uint32_t q = 0; q < 4; ++q) {
      const uint32_t sl = (uint32_t)e[q];
      lu[q] = __ldcg(&L.last_use[sl < H ? sl : 0u]);
      prefetch_l2(&L.slot2pos[sl < H ? sl : 0u]);
    }
#pragma unroll
    for (uint32_t q = 0; q < 4; ++q)
      if (e[q] != ~0ull && (uint32_t)e[q] < H && lu[q] == (uint32_t)(e[q] >> 32)) pre4 |= 1u << q;
  }
  cluster_wait();                                   // B1

  // ---------------------------------------------------------------- P2
  // per-CTA counts, one CTA per lane (every warp computes the same sums)
  const uint32_t t0 = lane < C ? table[lane][0] : 0u, t1 = lane < C ? table[lane][1] : 0u;
  const bool any_unordered = __any_sync(0xffffffffu, t0 != 0);
  uint32_t M = __reduce_add_sync(0xffffffffu, t1);
  uint32_t uniq_before = __reduce_add_sync(0xffffffffu, lane < r ? t1 : 0u);
  uint32_t nuniq_cta = cta_miss;                   // unique misses held by this CTA
  uint32_t mcount = t1;                            // lane q: unique misses of CTA q
  if (any_unordered) {
    // The smallest claiming j owns each missing position (claims came from
    // other CTAs: read them from L2); unique hit slots are counted from the
    // owners' bitmaps, so that a repeated position counts once.
    uint32_t nuniq = 0;
    for (uint32_t base = 0; base < jcnt; base += kThreads) {
      const uint32_t jj = base + tid;
      const bool f = jj < jcnt && meta_slot[jj] == kSlotMiss &&
                     __ldcg(&L.pos2slot[meta_pos[jj]]) == (int32_t)(jlo + jj) - (int32_t)k - 1;
      uint32_t tile;
      const uint32_t rank = block_flag_scan(f, scratch[0], &tile);
      if (jj < jcnt) uniq[jj] = f ? nuniq + rank : kNoRank;
      if (f) mlist[nuniq + rank] = jj;
      nuniq += tile;
    }
    uint32_t used = 0;
    for (uint32_t w = tid; w < words; w += kThreads) used += __popc(pinbits[w]);
    const uint32_t mine2[2] = {nuniq, block_sum(used, scratch[1])};
    cluster_publish(mine2, 2, table2, r, C);       // B2 (only for an idx that is not increasing)
    mcount = lane < C ? table2[lane][0] : 0u;
    M = __reduce_add_sync(0xffffffffu, mcount);
    uniq_before = __reduce_add_sync(0xffffffffu, lane < r ? mcount : 0u);
    nuniq_cta = nuniq;
  }
  if (r == 0 && tid == 0) L.counters[0] = t;       // every CTA read the old step before B1

  // ---------------------------------------------------------------- P3
  // CTA 0 walks the queue from its head: the current entries are the
  // unpinned slots in (last_use, slot) order; the u-th is the victim of
  // unique miss u, sent to the CTA holding that miss.
  if (r == 0) {
    if (warp == 0) {                               // mbefore[q]: unique misses of CTAs below q
      uint32_t incl = mcount;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const uint32_t o = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= (uint32_t)d) incl += o;
      }
      if (lane <= C) mbefore[lane] = incl - mcount;
    }
    __syncthreads();                               // mbefore, and the window copied by other threads
    // LRU: the queue from its head.  Circular: the slots from the hand.
    const uint32_t limit = lru ? span : H;
    uint32_t found = 0, off = 0;
    while (found < M && off < limit) {             // uniform over the CTA
      uint64_t e[4];                               // ~0 marks an entry that is not current
      uint32_t lu[4], ncur = 0;
#pragma unroll
      for (uint32_t q = 0; q < 4; ++q) {
        const uint32_t o = off + 4 * tid + q;
        if (!lru) {
          const uint32_t sl = hand + o < H ? hand + o : hand + o - H;
          e[q] = o < H && !((fullpin[sl >> 5] >> (sl & 31)) & 1u) ? (uint64_t)sl : ~0ull;
        } else {
          e[q] = o >= span ? ~0ull : o < wlen ? window[sh + o] : __ldcg(&ring_in[(head + o) & qmask]);
        }
      }
#pragma unroll
      for (uint32_t q = 0; q < 4; ++q) {           // four independent loads in flight
        const uint32_t o = off + 4 * tid + q, sl = (uint32_t)e[q];
        lu[q] = !lru || o < wlen ? 0u : __ldcg(&L.last_use[sl < H ? sl : 0u]);
      }
#pragma unroll
      for (uint32_t q = 0; q < 4; ++q) {
        const uint32_t o = off + 4 * tid + q, sl = (uint32_t)e[q];
        // in the window: current before this call and not pinned by it
        const bool cur = e[q] != ~0ull && sl < H &&
                         (!lru || (o < wlen ? ((pre4 >> q) & 1u) && !((fullpin[sl >> 5] >> (sl & 31)) & 1u)
                                            : lu[q] == (uint32_t)(e[q] >> 32)));
        if (cur) ++ncur;
        else e[q] = ~0ull;
      }
      uint32_t tot;
      uint32_t u = found + block_excl_sum(ncur, scratch[0], &tot);
      // the CTA holding unique miss u (this thread's victims are consecutive)
      uint32_t h = 0;
      if (ncur && u < M) {
        uint32_t hi = C;
        while (hi - h > 1) {
          const uint32_t mid = (h + hi) >> 1;
          if (mbefore[mid] <= u) h = mid;
          else hi = mid;
        }
      }
#pragma unroll
      for (uint32_t q = 0; q < 4; ++q) {
        if (e[q] == ~0ull) continue;
        const uint32_t sl = (uint32_t)e[q];
        if (u < M) {
          while (h + 1 < C && mbefore[h + 1] <= u) ++h;
          dsmem_st_u32(dsmem_addr(&vslot[u - mbefore[h]], h), sl);
          const uint32_t owner = sl / a.hchunk, b = sl - owner * a.hchunk;
          dsmem_red_or_u32(dsmem_addr(&pinbits[b >> 5], owner), 1u << (b & 31));   // used in this call
          atomicAdd(&fillcnt[owner], 1u);
          if (u == M - 1) last_vic = sl;
        } else if (u == M) {
          head_hit = off + 4 * tid + q;            // the first current entry that stays
        }
        ++u;
      }
      found += tot;
      off += 4 * kThreads;
    }
    __syncthreads();
    if (warp == 0) {
      // every range's used slots go to the tail, ranges in slot order
      const uint32_t used = lane < C ? (any_unordered ? table2[lane][1] : hitcnt[lane]) + fillcnt[lane] : 0u;
      uint32_t incl = used;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const uint32_t o = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= (uint32_t)d) incl += o;
      }
      if (lru && lane < C) dsmem_st_u32(dsmem_addr(&ring_off, lane), tail + incl - used);
      if (!lru && lane == 31) L.counters[5] = M > 0 ? (last_vic + 1u == H ? 0u : last_vic + 1u) : hand;
      if (lru && lane == 31) {
        L.counters[2] = M > 0 ? head + (head_hit != kNoRank ? head_hit : min(off, span)) : head;
        L.counters[3] = tail + incl;
        L.counters[4] = buf;
      }
    }
  }
  if (r != 0) idle((r - 1u) * kWarps + warp, (C - 1u) * kWarps);
  cluster_sync();                                   // B3: victims, bits and queue positions delivered

  // ---------------------------------------------------------------- P4
  // One warp per unique miss: the row is read first (the output row this
  // CTA wrote in P1, else the host row), then the maps are updated and the
  // row lands in the victim slot.
  for (uint32_t lr = warp; lr < nuniq_cta; lr += kWarps) {
    const uint32_t jj = mlist[lr];
    const uint32_t v = vslot[lr];
    const int32_t p = meta_pos[jj];
    if (v >= H || p < 0 || (uint32_t)p >= L.history_cap) {
      if (lane == 0) atomicOr(a.status, kFlagInternal);   // cannot happen; never write out of bounds
      continue;
    }
    uint4* dst = reinterpret_cast<uint4*>(L.hot) + (size_t)v * kRowVec;
    if (staged && gather_ok) {
      // the row is still in shared memory: one bulk store into the slot
      if (lane == 0) {
        if (map_update(a, v, __ldcg(&L.slot2pos[v]), p, t, uniq_before + lr)) atomicAdd(&nevict_cta, 1u);
        bulk_copy_s2g(dst, stage4 + (size_t)jj * kRowVec, KVO_ROW_BYTES);
        bulk_commit();
      }
      continue;
    }
    const uint4* src = a.out_rows && !a.out_host
                           ? reinterpret_cast<const uint4*>(a.out_rows) + (size_t)(jlo + jj) * kRowVec
                           : miss_row(a, hist4, p);
    const uint4 x = __ldcg(src + lane);
    uint4 y = make_uint4(0, 0, 0, 0);
    if (lane < kRowVec - 32) y = __ldcg(src + 32 + lane);
    if (lane == 0 && map_update(a, v, __ldcg(&L.slot2pos[v]), p, t, uniq_before + lr)) atomicAdd(&nevict_cta, 1u);
    dst[lane] = x;
    if (lane < kRowVec - 32) dst[32 + lane] = y;
  }
  if (staged) bulk_wait_all();                      // the output slice and the fills have left shared memory
  // A copy that outlasted the wait is waited for once more (bounded); if it
  // still has not landed, the status says so and the context refuses further
  // launches: the copy's bytes could land in shared memory that another CTA
  // owns after this one exits.
  if (staged && !gather_ok && tid == 0 && !mbar_wait_bounded(&gbar, 0, kWindowPolls)) atomicOr(a.status, kFlagInflight);

  // ---------------------------------------------------------------- P5
  // The used slots of this CTA's range, in slot order, stamped t, at the
  // queue position CTA 0 assigned: one 32-bit bitmap word per thread.
  if (lru) {
    const uint32_t hwords = (hcnt + 31u) / 32u;
    const uint64_t stamp = (uint64_t)t << 32;
    uint32_t run = 0;
    for (uint32_t w0 = 0; w0 < hwords; w0 += kThreads) {
      const uint32_t w = w0 + tid;
      uint32_t bits = w < hwords ? pinbits[w] : 0u;
      uint32_t tot;
      uint32_t pos = ring_off + run + block_excl_sum(__popc(bits), scratch[0], &tot);
      while (bits) {
        const uint32_t b = __ffs(bits) - 1;
        bits &= bits - 1;
        const uint32_t i = 32 * w + b;
        if (i < hcnt) ring_out[pos & qmask] = stamp | (uint64_t)(slo + i);
        ++pos;
      }
      run += tot;
    }
  }
  if (L.evlog && r == 0 && tid == 0) L.evlog[0] = (int32_t)M;
  // a window copy that outlasted the wait: the same second, bounded wait
  if (r == 0 && !win_ok && tid == 0 && !mbar_wait_bounded(&wbar, 0, kWindowPolls)) atomicOr(a.status, kFlagInflight);

  // ------------------------------------------------------------- stats
  __syncthreads();
  if (tid == 0) {
    unsigned long long* st = L.stats;
    if (cta_hits) atomicAdd(st + 1, (unsigned long long)cta_hits);
    if (cta_miss) {
      atomicAdd(st + 2, (unsigned long long)cta_miss);
      if (cta_host + cta_fresh_ram)
        atomicAdd(st + 6, (unsigned long long)(cta_host + cta_fresh_ram) * KVO_ROW_BYTES);
    }
    if (nevict_cta) atomicAdd(st + 4, (unsigned long long)nevict_cta);
    if (cta_inv) {
      atomicAdd(st + 5, (unsigned long long)cta_inv);
      atomicOr(a.status, kFlagRange);
    }
    if (r == 0) {
      atomicAdd(st + 0, 1ull);
      atomicAdd(st + 3, (unsigned long long)M);
      atomicAdd(st + 7, (unsigned long long)k);
    }
  }
}

}  // namespace resolve_detail
}  // namespace kvo
