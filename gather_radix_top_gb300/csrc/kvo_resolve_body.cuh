// Device body of the resolve + gather call, shared by the standalone kernel
// and the fused decode-step kernel.
//
// Resolve + gather of one layer's selection against its HBM hot cache.
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
// of selection entries j and a contiguous range of hot slots.
//   P1 classify: hit = pos2slot[p] >= 0 (stamp last_use = t); a miss does an
//      atomicMin of a negative first-occurrence code into pos2slot[p], so the
//      smallest j of each missing position wins (dedupe without a table).
//      Then, while the cluster barrier completes, every row is gathered:
//      hits from the hot slot (HBM), misses from host memory (zero-copy),
//      16-byte pieces, one warp per 656-byte row, plus the bf16 dequant.
//   P2 compact: unique misses are ranked in j order and listed in CTA 0's
//      shared memory.  When idx is strictly increasing (always true for
//      kvo_select_topk output) every miss is unique: the counts published at
//      the first barrier already give every rank.
//   P3 victims: a cluster radix select of the M oldest unpinned slots on the
//      key t - last_use (0 for pinned slots; only its significant digits are
//      examined), ties to the lower slot.  Winners go to CTA 0 as 64-bit
//      (last_use, slot) keys together with the position each slot holds.
//   P4 rank (CTA 0): the i-th oldest winner is the victim of the i-th
//      unique miss.
//   P5 fill + map update, spread over the cluster: unmap the evicted
//      position, map the new one, stamp last_use = t, copy the row (from the
//      output just written) into the victim slot.
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
constexpr uint32_t kRankMax = 512;                  // rank winners by counting up to here, else sort
constexpr uint32_t kRowsInFlight = 4;               // rows a warp loads before it stores

struct ResolveArgs {
  LayerView L;
  const int32_t* idx;
  uint8_t* out_rows;
  uint16_t* out_bf16;
  uint32_t* status;
  uint32_t k;
  uint32_t kchunk;        // selection entries per CTA
  uint32_t hchunk;        // hot slots per CTA (multiple of 4)
  uint32_t sort_len;      // power of two >= k
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
    return reinterpret_cast<const uint4*>(a.fresh) + (size_t)((uint32_t)p - a.fresh_from) * (KVO_ROW_BYTES / 16);
  return hist4 + (size_t)p * (KVO_ROW_BYTES / 16);
}

struct SmemLayout {
  uint32_t sortkeys, lukeys, meta_slot, meta_pos, uniq, miss_pos, miss_j, win_old, vic_slot, vic_old, share, sel,
      total;
};

__host__ __device__ inline SmemLayout smem_layout(uint32_t k, uint32_t kchunk, uint32_t hchunk,
                                                  uint32_t sort_len) {
  SmemLayout s;
  uint32_t o = 0;
  s.sortkeys = o;  o += sort_len * 8u;          // CTA 0: winners' (last_use, slot)
  s.lukeys = o;    o += hchunk * 4u;            // this CTA's LRU keys
  s.meta_slot = o; o += kchunk * 4u;            // per entry: hot slot, or miss / invalid
  s.meta_pos = o;  o += kchunk * 4u;            // per entry: position
  s.uniq = o;      o += kchunk * 4u;            // per entry: 1 = unique miss
  s.miss_pos = o;  o += k * 4u;                 // CTA 0: unique misses in j order
  s.miss_j = o;    o += k * 4u;
  s.win_old = o;   o += k * 4u;                 // CTA 0: position each winner holds (winner order)
  s.vic_slot = o;  o += k * 4u;                 // CTA 0: victims in rank order, and what they held
  s.vic_old = o;   o += k * 4u;
  s.share = o;     o += 4u * kchunk * 4u;       // this CTA's share of the fills (slot, old, pos, j)
  s.sel = o;       o += kchunk * 4u;            // fused step: this CTA's selected positions
  s.total = (o + 15u) & ~15u;
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

__device__ __forceinline__ void resolve_body(const ResolveArgs& a, uint8_t* dyn_smem) {
  __shared__ RadixSmem rsm;
  __shared__ uint32_t scratch[2][2 * kWarps + 2];
  __shared__ uint32_t table[kMaxCluster][4];
  __shared__ uint32_t table2[kMaxCluster][4];

  const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t r = cluster_rank(), C = cluster_size();
  const LayerView& L = a.L;
  const uint32_t k = a.k;

  const SmemLayout lay = smem_layout(k, a.kchunk, a.hchunk, a.sort_len);
  uint64_t* sortkeys = reinterpret_cast<uint64_t*>(dyn_smem + lay.sortkeys);
  uint32_t* lukeys = reinterpret_cast<uint32_t*>(dyn_smem + lay.lukeys);
  int32_t* meta_slot = reinterpret_cast<int32_t*>(dyn_smem + lay.meta_slot);
  int32_t* meta_pos = reinterpret_cast<int32_t*>(dyn_smem + lay.meta_pos);
  uint32_t* uniq = reinterpret_cast<uint32_t*>(dyn_smem + lay.uniq);
  int32_t* miss_pos = reinterpret_cast<int32_t*>(dyn_smem + lay.miss_pos);
  int32_t* miss_j = reinterpret_cast<int32_t*>(dyn_smem + lay.miss_j);
  int32_t* win_old = reinterpret_cast<int32_t*>(dyn_smem + lay.win_old);
  int32_t* vic_slot = reinterpret_cast<int32_t*>(dyn_smem + lay.vic_slot);
  int32_t* vic_old = reinterpret_cast<int32_t*>(dyn_smem + lay.vic_old);
  int32_t* share = reinterpret_cast<int32_t*>(dyn_smem + lay.share);
  const int32_t* sel = reinterpret_cast<const int32_t*>(dyn_smem + lay.sel);

  const uint32_t t = L.counters[0] + 1u;        // this call's step
  const uint32_t len = a.fused ? a.len : L.counters[1];
  const uint32_t jlo = min(k, r * a.kchunk), jhi = min(k, jlo + a.kchunk), jcnt = jhi - jlo;
  radix_smem_init(&rsm);
  // B0: every CTA of the cluster is running before any DSMEM access (its
  // wait is just before the first remote store, so classification overlaps).
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
  uint32_t cta_unordered, cta_miss;
  block_sum2(unordered, nmiss, scratch[0], &cta_unordered, &cta_miss);
  cluster_wait();                                   // B0
  if (tid < 2 * C) dsmem_st_u32(dsmem_addr(&table[r][tid & 1], tid >> 1), (tid & 1) ? cta_miss : cta_unordered);
  cluster_arrive();                                 // B1: stamps, claims, counts

  const uint4* hot4 = reinterpret_cast<const uint4*>(L.hot);
  const uint4* hist4 = reinterpret_cast<const uint4*>(L.hist);
  // Each warp loads up to kRowsInFlight rows before storing any, so that all
  // of this CTA's rows are in flight at once.
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
    // strictly increasing idx: every miss is a distinct position
    for (uint32_t jj = tid; jj < jcnt; jj += kThreads) uniq[jj] = meta_slot[jj] == kSlotMiss;
    __syncthreads();
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

  uint32_t nevict = 0;
  if (M > 0) {
    {
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
    // -------------------------------------------------------------- P3
    const uint32_t H = L.hot_rows;
    const uint32_t slo = min(H, r * a.hchunk), shi = min(H, slo + a.hchunk), hcnt = shi - slo;
    for (uint32_t i = tid; i < hcnt; i += kThreads) {
      const uint32_t lu = __ldcg(&L.last_use[slo + i]);   // stamps came from other CTAs
      lukeys[i] = lu < t ? t - lu : 0u;                   // larger = older; pinned slots 0
    }
    __syncthreads();
    const uint32_t key_bits = ((32u - (uint32_t)__clz((int)t)) + 7u) & ~7u;
    auto key4 = [&](uint32_t g) -> uint4 { return reinterpret_cast<const uint4*>(lukeys)[g]; };
    const RadixCut cut = cluster_radix_select(key4, hcnt, M, key_bits, &rsm, C);
    const uint32_t mine2[2] = {cut.above, cut.at};
    cluster_publish(mine2, 2, table, r, C);        // B3
    uint32_t sel_before, at_before;
    cut_offsets(table, 0, r, cut.need, &sel_before, &at_before);
    const uint32_t sk0 = dsmem_addr(sortkeys, 0), old0 = dsmem_addr(win_old, 0);
    cluster_compact(key4, hcnt, cut, sel_before, at_before, scratch, [&](uint32_t i, uint32_t out) {
      if (out < M) {
        const uint32_t slot = slo + i;
        const uint64_t lu = (uint64_t)(t - lukeys[i]);
        dsmem_st_u64(sk0 + 8u * out, (lu << 32) | slot);
        dsmem_st_u32(old0 + 4u * out, (uint32_t)L.slot2pos[slot]);
      }
    });
    cluster_sync();                                 // B4: miss list and winners in CTA 0

    // -------------------------------------------------------------- P4
    if (r == 0) {
      if (M <= kRankMax) {
        // rank of winner c among all winners (the keys are distinct); S
        // threads share each winner's count
        uint32_t S = 32;
        while (S > 1 && S * M > kThreads) S >>= 1;
        const uint32_t c = tid / S, part = tid % S;
        uint32_t rank = 0;
        uint64_t key = 0;
        if (c < M) {
          key = sortkeys[c];
          for (uint32_t o = part; o < M; o += S) rank += sortkeys[o] < key;
        }
        for (uint32_t d = 1; d < S; d <<= 1) rank += __shfl_xor_sync(0xffffffffu, rank, d);
        if (c < M && part == 0) {
          vic_slot[rank] = (int32_t)(key & 0xffffffffu);
          vic_old[rank] = win_old[c];
        }
      } else {
        // bitonic sort of (last_use:32, slot:18, winner index:13) keys
        const uint32_t P = a.sort_len;
        for (uint32_t i = tid; i < P; i += kThreads) {
          uint64_t v = ~0ull;
          if (i < M) {
            const uint64_t key = sortkeys[i];
            v = ((key >> 32) << 31) | ((key & 0x3ffffu) << 13) | i;
          }
          sortkeys[i] = v;
        }
        __syncthreads();
        uint32_t Pn = 1;
        while (Pn < M && Pn < P) Pn <<= 1;
        for (uint32_t size = 2; size <= Pn; size <<= 1) {
          for (uint32_t stride = size >> 1; stride > 0; stride >>= 1) {
            for (uint32_t i = tid; i < Pn / 2; i += kThreads) {
              const uint32_t lo = 2 * i - (i & (stride - 1)), hi = lo + stride;
              const bool ascending = (lo & size) == 0;
              const uint64_t x = sortkeys[lo], y = sortkeys[hi];
              if ((x > y) == ascending) {
                sortkeys[lo] = y;
                sortkeys[hi] = x;
              }
            }
            __syncthreads();
          }
        }
        for (uint32_t i = tid; i < M; i += kThreads) {
          const uint64_t v = sortkeys[i];
          vic_slot[i] = (int32_t)((v >> 13) & 0x3ffffu);
          vic_old[i] = win_old[v & 0x1fffu];
        }
      }
    }
    cluster_sync();                                 // B5: victims ranked

    // -------------------------------------------------------------- P5
    // This CTA's share of the fills: entries [f0, f1) of the rank order.
    const uint32_t per = (M + C - 1) / C;
    const uint32_t f0 = min(M, r * per), f1 = min(M, f0 + per), fn = f1 - f0;
    int32_t* sh_slot = share;
    int32_t* sh_old = share + a.kchunk;
    int32_t* sh_pos = share + 2 * a.kchunk;
    int32_t* sh_j = share + 3 * a.kchunk;
    for (uint32_t i = tid; i < fn; i += kThreads) {
      sh_slot[i] = (int32_t)dsmem_ld_u32(dsmem_addr(&vic_slot[f0 + i], 0));
      sh_old[i] = (int32_t)dsmem_ld_u32(dsmem_addr(&vic_old[f0 + i], 0));
      sh_pos[i] = (int32_t)dsmem_ld_u32(dsmem_addr(&miss_pos[f0 + i], 0));
      sh_j[i] = (int32_t)dsmem_ld_u32(dsmem_addr(&miss_j[f0 + i], 0));
    }
    __syncthreads();
    cluster_arrive();                               // B6: this CTA is done reading CTA 0
    for (uint32_t i = tid; i < fn; i += kThreads) {
      const uint32_t v = (uint32_t)sh_slot[i];
      const int32_t old = sh_old[i], p = sh_pos[i];
      if (v >= L.hot_rows || p < 0 || (uint32_t)p >= L.history_cap) {
        atomicOr(a.status, kFlagInternal);          // cannot happen; never write out of bounds
        continue;
      }
      if (old >= 0) {
        L.pos2slot[old] = -1;
        ++nevict;
      }
      L.pos2slot[p] = (int32_t)v;
      L.slot2pos[v] = p;
      L.last_use[v] = t;
      if (L.evlog) {
        const uint32_t e = f0 + i;
        L.evlog[1 + 3 * e] = (int32_t)v;
        L.evlog[2 + 3 * e] = old;
        L.evlog[3 + 3 * e] = p;
      }
    }
    for (uint32_t i = warp; i < fn; i += kWarps) {
      const uint32_t v = (uint32_t)sh_slot[i];
      const int32_t p = sh_pos[i];
      const uint32_t j = (uint32_t)sh_j[i];
      if (v >= L.hot_rows || p < 0 || (uint32_t)p >= L.history_cap || j >= k) continue;
      // the output row written in P1 (by any CTA), else the host row
      const uint4* src = a.out_rows ? reinterpret_cast<const uint4*>(a.out_rows) + (size_t)j * kRowVec
                                    : miss_row(a, hist4, p);
      uint4* d = reinterpret_cast<uint4*>(L.hot) + (size_t)v * kRowVec;
      const uint4 x = __ldcg(src + lane);
      uint4 y = make_uint4(0, 0, 0, 0);
      if (lane < kRowVec - 32) y = __ldcg(src + 32 + lane);
      d[lane] = x;
      if (lane < kRowVec - 32) d[32 + lane] = y;
    }
    cluster_wait();                                 // B6
  }
  if (L.evlog && r == 0 && tid == 0) L.evlog[0] = (int32_t)M;

  // ------------------------------------------------------------- stats
  uint32_t s_hit, s_miss, s_inv, s_evict;
  block_sum2(nhit, nmiss, scratch[0], &s_hit, &s_miss);
  block_sum2(ninv, nevict, scratch[1], &s_inv, &s_evict);
  if (tid == 0) {
    unsigned long long* st = L.stats;
    if (s_hit) atomicAdd(st + 1, (unsigned long long)s_hit);
    if (s_miss) {
      atomicAdd(st + 2, (unsigned long long)s_miss);
      atomicAdd(st + 6, (unsigned long long)s_miss * KVO_ROW_BYTES);
    }
    if (s_evict) atomicAdd(st + 4, (unsigned long long)s_evict);
    if (s_inv) {
      atomicAdd(st + 5, (unsigned long long)s_inv);
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
