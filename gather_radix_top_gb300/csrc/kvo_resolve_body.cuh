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
// One thread-block cluster runs the whole call; CTA r owns a contiguous range
// of selection entries j, a contiguous range of hot slots and the same range
// of positions of the layer's LRU order (slots sorted by (last_use, slot)).
//   P0 the CTA's range of the LRU order starts copying to shared memory
//      (cp.async) while the rest of the call proceeds.
//   P1 classify: hit = pos2slot[p] >= 0 (stamp last_use = t and set the
//      slot's bit in its owner's pin bitmap over DSMEM); a miss does an
//      atomicMin of a negative first-occurrence code into pos2slot[p], so the
//      smallest j of each missing position wins (dedupe without a table).
//      Then, while the cluster barrier completes, every row is gathered:
//      hits from the hot slot (HBM), misses from host memory (zero-copy),
//      16-byte pieces, one warp per 656-byte row, plus the bf16 dequant.
//   P2 compact: unique misses are ranked in j order and listed in CTA 0's
//      shared memory.  When idx is strictly increasing (always true for
//      kvo_select_topk output) every miss is unique: the counts published at
//      the first barrier already give every rank.
//   P3 victims: the i-th unpinned entry of the LRU order, for i < M, is the
//      victim of the i-th unique miss: one ordered count over the order (each
//      CTA pulls the whole pin bitmap, counts its unpinned entries and
//      publishes the count), no selection and no sort.
//   P4 the CTA holding a victim unmaps the evicted position, maps the new
//      one, stamps last_use = t and copies the row (from the output just
//      written) into the victim slot.
//   P5 the next LRU order: unpinned non-victim entries keep their order
//      (they shift down by M), then every slot used in this call (hits and
//      fills, all now last used at t) in slot order.
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
constexpr uint32_t kTiles = 2;                      // order range per CTA <= kTiles * 4 * kThreads

struct ResolveArgs {
  LayerView L;
  const int32_t* idx;
  uint8_t* out_rows;
  uint16_t* out_bf16;
  uint32_t* status;
  uint32_t k;
  uint32_t kchunk;        // selection entries per CTA
  uint32_t hchunk;        // hot slots (and LRU order positions) per CTA, a multiple of 128
  // fused decode step only: the selection is in shared memory, the history
  // length is `len`, and positions >= fresh_from were appended by this very
  // launch and are read from `fresh` (device memory) rather than host memory
  uint32_t fused;
  uint32_t len;
  const uint8_t* fresh;
  uint32_t fresh_from;
};

// The row of a missing position: host history, or, for rows appended in the
// same fused launch, their device copy (same bytes, no host round trip).
__device__ __forceinline__ const uint4* miss_row(const ResolveArgs& a, const uint4* hist4, int32_t p) {
  if (a.fresh && (uint32_t)p >= a.fresh_from)
    return reinterpret_cast<const uint4*>(a.fresh) + (size_t)((uint32_t)p - a.fresh_from) * kRowVec;
  return hist4 + (size_t)p * kRowVec;
}

struct SmemLayout {
  uint32_t miss_pos, miss_j, ord, pinbits, fullbits, meta_slot, meta_pos, uniq, sel, vic_rank, vic_slot, rec,
      total;
};

__host__ __device__ inline uint32_t round16(uint32_t x) { return (x + 15u) & ~15u; }

// hchunk: slots (and order positions) per CTA, a multiple of 128 so that the
// pin bitmap of a CTA is whole 16-byte pieces of the layer's bitmap.
__host__ __device__ inline SmemLayout smem_layout(uint32_t k, uint32_t kchunk, uint32_t hchunk, uint32_t hot_rows) {
  SmemLayout s;
  const uint32_t vcap = k < hchunk ? k : hchunk;   // victims one CTA can hold
  uint32_t o = 0;
  s.miss_pos = o;  o += k * 4u;                 // CTA 0: unique misses in j order
  s.miss_j = o;    o += k * 4u;
  o = round16(o);
  s.ord = o;       o += hchunk * 4u;            // this CTA's range of the LRU order
  s.pinbits = o;   o += round16(hchunk / 8u);   // this CTA's slots used in this call
  s.fullbits = o;  o += round16((hot_rows + 31u) / 32u * 4u);   // every slot pinned in this call
  s.meta_slot = o; o += kchunk * 4u;            // per entry: hot slot, or miss / invalid
  s.meta_pos = o;  o += kchunk * 4u;            // per entry: position
  s.uniq = o;      o += kchunk * 4u;            // per entry: 1 = unique miss
  s.sel = o;       o += kchunk * 4u;            // fused step: this CTA's selected positions
  s.vic_rank = o;  o += vcap * 4u;              // victims found in this CTA's order range
  s.vic_slot = o;  o += vcap * 4u;
  o = round16(o);
  s.rec = o;       o += kchunk * 16u;           // victims this CTA maps and fills: (slot, pos, j, rank)
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

// Copies one 656-byte row with a warp (L2 reads: the source may have been
// written by another CTA of this launch).
__device__ __forceinline__ void copy_row(const uint4* src, uint4* dst, uint32_t lane) {
  const uint4 x = __ldcg(src + lane);
  uint4 y = make_uint4(0, 0, 0, 0);
  if (lane < kRowVec - 32) y = __ldcg(src + 32 + lane);
  dst[lane] = x;
  if (lane < kRowVec - 32) dst[32 + lane] = y;
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

__device__ __forceinline__ void resolve_body(const ResolveArgs& a, uint8_t* dyn_smem) {
  __shared__ uint32_t scratch[2][2 * kWarps + 2];
  __shared__ uint32_t table[kMaxCluster][4];
  __shared__ uint32_t table2[kMaxCluster][4];
  __shared__ uint32_t table3[kMaxCluster][4];
  __shared__ uint32_t tcount[kMaxCluster];         // victims per slot-owner CTA, over the cluster
  __shared__ uint32_t ocount[kMaxCluster];         // victims per slot-owner CTA found here
  __shared__ uint32_t nvic;
  __shared__ uint32_t nevict_cta;
  __shared__ uint32_t cta_hits, cta_inv;

  const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t r = cluster_rank(), C = cluster_size();
  const LayerView& L = a.L;
  const uint32_t k = a.k;
  const uint32_t H = L.hot_rows;

  const SmemLayout lay = smem_layout(k, a.kchunk, a.hchunk, H);
  int32_t* miss_pos = reinterpret_cast<int32_t*>(dyn_smem + lay.miss_pos);
  int32_t* miss_j = reinterpret_cast<int32_t*>(dyn_smem + lay.miss_j);
  int32_t* ord = reinterpret_cast<int32_t*>(dyn_smem + lay.ord);
  uint32_t* pinbits = reinterpret_cast<uint32_t*>(dyn_smem + lay.pinbits);
  uint32_t* fullbits = reinterpret_cast<uint32_t*>(dyn_smem + lay.fullbits);
  int32_t* meta_slot = reinterpret_cast<int32_t*>(dyn_smem + lay.meta_slot);
  int32_t* meta_pos = reinterpret_cast<int32_t*>(dyn_smem + lay.meta_pos);
  uint32_t* uniq = reinterpret_cast<uint32_t*>(dyn_smem + lay.uniq);
  const int32_t* sel = reinterpret_cast<const int32_t*>(dyn_smem + lay.sel);
  uint32_t* vic_rank = reinterpret_cast<uint32_t*>(dyn_smem + lay.vic_rank);
  uint32_t* vic_slot = reinterpret_cast<uint32_t*>(dyn_smem + lay.vic_slot);
  uint4* rec = reinterpret_cast<uint4*>(dyn_smem + lay.rec);

  const uint32_t t = L.counters[0] + 1u;        // this call's step
  const uint32_t len = a.fused ? a.len : L.counters[1];
  const uint32_t jlo = min(k, r * a.kchunk), jhi = min(k, jlo + a.kchunk), jcnt = jhi - jlo;
  const uint32_t slo = min(H, r * a.hchunk), shi = min(H, slo + a.hchunk), hcnt = shi - slo;
  const uint32_t words = a.hchunk / 32u;         // pin-bitmap words per CTA
  const uint32_t Hp = (H + 3u) & ~3u;            // order buffers are padded to whole 16-byte pieces
  const int32_t* ord_in = L.order + (size_t)((t + 1u) & 1u) * Hp;   // written by the previous call
  int32_t* ord_out = L.order + (size_t)(t & 1u) * Hp;

  // ---------------------------------------------------------------- P0
  for (uint32_t i = tid; i < words; i += kThreads) pinbits[i] = 0;
  for (uint32_t i = tid; i < (H + 31u) / 32u; i += kThreads) fullbits[i] = 0;
  for (uint32_t i = tid; i < (hcnt + 3) / 4; i += kThreads) cp_async16(ord + 4 * i, ord_in + slo + 4 * i);
  if (tid < kMaxCluster) {
    tcount[tid] = 0;
    ocount[tid] = 0;
  }
  if (tid == 0) {
    nvic = 0;
    nevict_cta = 0;
  }
  // B0: every CTA of the cluster is running (and has zeroed what others add
  // into) before any DSMEM access; classification overlaps the barrier.
  cluster_arrive();

  // ---------------------------------------------------------------- P1
  uint32_t nhit = 0, nmiss = 0, ninv = 0, unordered = 0;   // per thread
  for (uint32_t jj = tid; jj < jcnt; jj += kThreads) {
    const uint32_t j = jlo + jj;
    // fused calls take the selection from shared memory, already ascending
    const int32_t p = a.fused ? sel[jj] : a.idx[j];
    if (!a.fused && j > 0 && a.idx[j - 1] >= p) ++unordered;
    int32_t slot;
    if (p < 0 || (uint32_t)p >= len) {
      slot = kSlotInvalid;
      ++ninv;
    } else {
      const int32_t s = L.pos2slot[p];
      if (s >= 0) {
        slot = s;
        L.last_use[s] = t;
        ++nhit;
      } else {
        slot = kSlotMiss;
        atomicMin(&L.pos2slot[p], (int32_t)j - (int32_t)k - 1);
        ++nmiss;
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
    if (f) uniq[jj] = cta_miss + rank;
    cta_miss += tile;
  }
  uint32_t cta_unordered, cta_hit_inv;
  block_sum2(unordered, nhit | (ninv << 16), scratch[1], &cta_unordered, &cta_hit_inv);
  if (tid == 0) {
    cta_hits = cta_hit_inv & 0xffffu;
    cta_inv = cta_hit_inv >> 16;
  }
  cluster_wait();                                   // B0
  if (tid < 2 * C) dsmem_st_u32(dsmem_addr(&table[r][tid & 1], tid >> 1), (tid & 1) ? cta_miss : cta_unordered);
  // pin: every CTA gets every hit slot's bit
  for (uint32_t i = tid; i < jcnt * C; i += kThreads) {
    const uint32_t jj = i / C, q = i - jj * C;
    const int32_t sl = meta_slot[jj];
    if (sl >= 0) dsmem_red_or_u32(dsmem_addr(&fullbits[(uint32_t)sl >> 5], q), 1u << ((uint32_t)sl & 31));
  }
  cluster_arrive();                                 // B1: stamps, claims, counts, pins

  // Each warp loads up to kRowsInFlight rows before storing any, so that all
  // of this CTA's rows are in flight at once.
  const uint4* hot4 = reinterpret_cast<const uint4*>(L.hot);
  const uint4* hist4 = reinterpret_cast<const uint4*>(L.hist);
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
  cp_async_wait_all();
  cluster_wait();                                   // B1

  // ---------------------------------------------------------------- P2
  bool any_unordered = false;
  uint32_t uniq_before = 0, M = 0;
  for (uint32_t q = 0; q < C; ++q) {
    any_unordered |= table[q][0] != 0;
    uniq_before += q < r ? table[q][1] : 0u;
    M += table[q][1];
  }
  if (!any_unordered) {
    // strictly increasing idx: every miss is a distinct position, ranked in P1
    if (M > 0) {
      const uint32_t mp0 = dsmem_addr(miss_pos, 0), mj0 = dsmem_addr(miss_j, 0);
      for (uint32_t jj = tid; jj < jcnt; jj += kThreads) {
        const uint32_t i = uniq_before + uniq[jj];
        if (meta_slot[jj] == kSlotMiss && i < k) {
          dsmem_st_u32(mp0 + 4u * i, (uint32_t)meta_pos[jj]);
          dsmem_st_u32(mj0 + 4u * i, jlo + jj);
        }
      }
    }
  } else {
    // The smallest claiming j owns each missing position; the claims came
    // from other CTAs, so read them from L2.
    uint32_t nuniq = 0;
    for (uint32_t jj = tid; jj < jcnt; jj += kThreads) {
      const bool u = meta_slot[jj] == kSlotMiss &&
                     __ldcg(&L.pos2slot[meta_pos[jj]]) == (int32_t)(jlo + jj) - (int32_t)k - 1;
      uniq[jj] = u;
      nuniq += u;
    }
    nuniq = block_sum(nuniq, scratch[1]);
    const uint32_t mine1[1] = {nuniq};
    cluster_publish(mine1, 1, table2, r, C);       // B2 (only for an unordered idx)
    uniq_before = 0;
    M = 0;
    for (uint32_t q = 0; q < C; ++q) {
      uniq_before += q < r ? table2[q][0] : 0u;
      M += table2[q][0];
    }
  }
  if (r == 0 && tid == 0) L.counters[0] = t;       // every CTA read the old step before B1
  if (M > 0 && any_unordered) {
    const uint32_t mp0 = dsmem_addr(miss_pos, 0), mj0 = dsmem_addr(miss_j, 0);
    uint32_t run = 0;
    for (uint32_t base = 0; base < jcnt; base += kThreads) {
      const uint32_t jj = base + tid;
      const bool f = jj < jcnt && uniq[jj];
      uint32_t tile;
      const uint32_t rank = block_flag_scan(f, scratch[0], &tile);
      const uint32_t i = uniq_before + run + rank;
      if (f && i < k) {
        dsmem_st_u32(mp0 + 4u * i, (uint32_t)meta_pos[jj]);
        dsmem_st_u32(mj0 + 4u * i, jlo + jj);
      }
      run += tile;
    }
  }

  // ---------------------------------------------------------------- P3
  // the layer's pin bitmap arrived before B1; this CTA's own slots are
  // words [slo / 32, slo / 32 + words) of it
  const uint32_t hwords = (hcnt + 31u) / 32u;     // words of this CTA's own slots (none if it has none)
  uint32_t mypins = 0;
  for (uint32_t w = tid; w < hwords; w += kThreads) mypins += __popc(fullbits[slo / 32u + w]);
  // Ordered pass over this CTA's order range, four entries per thread: the
  // unpinned entry of rank u is the victim of unique miss u when u < M, else
  // it survives at position u - M of the next order.
  uint32_t cnt4[kTiles], total4[kTiles], unpinned = 0;
#pragma unroll
  for (uint32_t tile = 0; tile < kTiles; ++tile) {
    const uint32_t i0 = 4 * (tile * kThreads + tid);
    uint32_t c = 0;
#pragma unroll
    for (uint32_t e = 0; e < 4; ++e) {
      if (i0 + e < hcnt) {
        const uint32_t sl = (uint32_t)ord[i0 + e];
        c += ((fullbits[sl >> 5] >> (sl & 31)) & 1u) ^ 1u;
      }
    }
    cnt4[tile] = c;
    unpinned += c;
  }
  uint32_t cta_unpinned, cta_pins;
  block_sum2(unpinned, mypins, scratch[1], &cta_unpinned, &cta_pins);
  const uint32_t mine3[2] = {cta_unpinned, cta_pins};
  cluster_publish(mine3, 2, table3, r, C);         // B3: also fences the pin-bitmap pulls
  uint32_t u_run = 0;
  for (uint32_t q = 0; q < r; ++q) u_run += table3[q][0];
#pragma unroll
  for (uint32_t tile = 0; tile < kTiles; ++tile) {
    if (tile * 4u * kThreads >= hcnt) break;       // uniform over the CTA
    const uint32_t i0 = 4 * (tile * kThreads + tid);
    uint32_t u = u_run + block_excl_sum(cnt4[tile], scratch[tile & 1], &total4[tile]);
#pragma unroll
    for (uint32_t e = 0; e < 4; ++e) {
      if (i0 + e < hcnt) {
        const uint32_t sl = (uint32_t)ord[i0 + e];
        if (!((fullbits[sl >> 5] >> (sl & 31)) & 1u)) {
          if (u < M) {
            const uint32_t c = atomicAdd(&nvic, 1u);
            vic_rank[c] = u;
            vic_slot[c] = sl;
          } else if (u - M < H) {
            ord_out[u - M] = (int32_t)sl;
          }
          ++u;
        }
      }
    }
    u_run += total4[tile];
  }
  __syncthreads();

  // ---------------------------------------------------------------- P4
  // The CTA holding a victim marks it used (its owner's bit), counts it for
  // its owner and sends (slot, position, entry, rank) to the handler CTA
  // rank % C, which then maps it and copies its row.
  const uint32_t nv = nvic;
  if (M > 0) {
    for (uint32_t c = tid; c < nv; c += kThreads) {
      const uint32_t u = vic_rank[c] < M ? vic_rank[c] : 0u, v = vic_slot[c];
      const uint32_t p = dsmem_ld_u32(dsmem_addr(&miss_pos[u], 0));
      const uint32_t j = dsmem_ld_u32(dsmem_addr(&miss_j[u], 0));
      const uint32_t h = u % C;
      dsmem_st_v4(dsmem_addr(&rec[u / C], h), make_uint4(v, p, j, u));
      const uint32_t owner = v / a.hchunk, b = v - owner * a.hchunk;
      dsmem_red_or_u32(dsmem_addr(&pinbits[b >> 5], owner), 1u << (b & 31));   // used in this call
      atomicAdd(&ocount[owner], 1u);
    }
    __syncthreads();
    // every CTA learns how many fills landed in each owner's slot range
    for (uint32_t i = tid; i < C * C; i += kThreads) {
      const uint32_t o = i / C, q = i - o * C;
      const uint32_t n = ocount[o];
      if (n) dsmem_red_add_u32(dsmem_addr(&tcount[o], q), n);
    }
    cluster_sync();                                 // B4: records, bits and counts delivered
    const uint32_t nrec = r < M ? (M - r + C - 1) / C : 0u;
    for (uint32_t c = tid; c < nrec; c += kThreads) {
      const uint4 rc = rec[c];
      if (map_update(a, rc.x, L.slot2pos[rc.x], (int32_t)rc.y, t, rc.w)) atomicAdd(&nevict_cta, 1u);
    }
    for (uint32_t c = warp; c < nrec; c += kWarps) {
      const uint4 rc = rec[c];
      const uint32_t v = rc.x, j = rc.z;
      const int32_t p = (int32_t)rc.y;
      if (v >= H || j >= k || p < 0 || (uint32_t)p >= L.history_cap) continue;
      // the output row written in P1 (by any CTA), else the host row
      const uint4* src = a.out_rows ? reinterpret_cast<const uint4*>(a.out_rows) + (size_t)j * kRowVec
                                    : miss_row(a, hist4, p);
      copy_row(src, reinterpret_cast<uint4*>(L.hot) + (size_t)v * kRowVec, lane);
    }
  }

  // ---------------------------------------------------------------- P5
  // The used slots, in slot order, fill the end of the next order: one
  // 32-bit word of this CTA's used-slot bitmap per thread.
  {
    uint32_t used_before = 0, used = 0;
    for (uint32_t q = 0; q < C; ++q) {
      const uint32_t n_q = table3[q][1] + tcount[q];
      used_before += q < r ? n_q : 0u;
      used += n_q;
    }
    const uint32_t tail0 = H - used + used_before;
    uint32_t run = 0;
    for (uint32_t w0 = 0; w0 < hwords; w0 += kThreads) {
      const uint32_t w = w0 + tid;
      uint32_t bits = w < hwords ? pinbits[w] | fullbits[slo / 32u + w] : 0u;
      uint32_t tot;
      uint32_t pos = tail0 + run + block_excl_sum(__popc(bits), scratch[0], &tot);
      while (bits) {
        const uint32_t b = __ffs(bits) - 1;
        bits &= bits - 1;
        const uint32_t i = 32 * w + b;
        if (i < hcnt && pos < H) ord_out[pos] = (int32_t)(slo + i);
        ++pos;
      }
      run += tot;
    }
  }
  if (L.evlog && r == 0 && tid == 0) L.evlog[0] = (int32_t)M;

  // ------------------------------------------------------------- stats
  __syncthreads();
  if (tid == 0) {
    unsigned long long* st = L.stats;
    if (cta_hits) atomicAdd(st + 1, (unsigned long long)cta_hits);
    if (cta_miss) {
      atomicAdd(st + 2, (unsigned long long)cta_miss);
      atomicAdd(st + 6, (unsigned long long)cta_miss * KVO_ROW_BYTES);
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
