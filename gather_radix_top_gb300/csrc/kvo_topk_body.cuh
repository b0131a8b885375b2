// Device body of the top-K selection of history positions from indexer
// scores, shared by the standalone kernel and the fused decode-step kernel.
//
// "From 1M Total to 15+ x 1M Contexts: GLM-5.3 KV Cache Offloading", section
// "Separate historical capacity from the current working set": the DSA
// indexer selects the top 2,048 historical positions.  Selection stays on
// the GPU ("Decision one").
//
// One thread-block cluster does the whole selection in a single launch.  Each
// CTA owns a contiguous range of positions.
//
// Resident route (a CTA's keys fit in shared memory):
//   1. the keys are loaded into shared memory once;
//   2. an MSB-first 8-bit radix select finds the cut; each pass builds a
//      per-CTA histogram in shared memory, adds each nonzero bin into the
//      one CTA that owns that bin over distributed shared memory, and after
//      one cluster barrier every CTA reads all bins back from their owners
//      and scans them, so that every CTA finds the same bucket;
//   3. an ordered compaction writes the chosen positions in ascending order:
//      per-CTA counts (taken from the radix histograms) are published over
//      DSMEM, then each CTA walks its range four keys per thread, one block
//      barrier per 4,096 keys.
//
// Filtered route (long histories, whose keys do not fit):
//   a. one streaming pass over the scores builds the cluster-wide histogram
//      of the top 11 key bits and finds the bucket that holds the k-th
//      largest key;
//   b. a second pass (the scores are now in L2) keeps every key in or above
//      that bucket, with its position, in shared memory, in position order;
//   c. steps 2 and 3 run on those candidates only, on the key bits below
//      the bucket's.
// When the candidates would not fit (a crowded bucket: many equal or nearly
// equal scores), step c streams the scores for every pass instead.  In the
// batched decode step, step a's histogram is built on the whole GPU before
// the selection, and the same launch lists, per 4,096-score slice in
// position order, the keys in or above a bucket chosen from the layer's
// previous selection; when this selection's bucket is at or above that one,
// the cluster reads its slices' lists instead of step b's pass over the
// scores.
//
// Ties at the cut go to the lowest positions because the compaction takes
// equal keys in position order, and (b) keeps position order.
#pragma once

#include <cstdint>

#include "kvo_device.cuh"

namespace kvo {

namespace topk_detail {

constexpr uint32_t kTopkStaticSmem = 40 * 1024;            // headroom for static smem (radix histograms)
constexpr uint32_t kTopkMaxDynSmem = 227 * 1024 - kTopkStaticSmem;

constexpr uint32_t kFirstBits = 11;                        // digit of the filtering pass
constexpr uint32_t kFirstBins = 1u << kFirstBits;
constexpr uint32_t kLowBits = 32 - kFirstBits;             // key bits below that digit
constexpr uint32_t kLowMask = (1u << kLowBits) - 1u;
constexpr uint32_t kHistCopies = 4;                        // filtering histogram copies (warp mod 4)
constexpr uint32_t kFilterMinBytes = (kHistCopies + 1) * kFirstBins * 4;   // the copies and the totals
constexpr int kUnroll = 4;                                 // 4-key groups in flight per thread
static_assert(kFirstBins % kThreads == 0, "whole bins per thread in the cut scan");

// Scores per slice of the whole-GPU histogram and filter launches.
constexpr uint32_t kSliceScores = 4096;

// Candidate lists made before the selection (the batched step's histogram
// launch): every key in or above bucket `spec` (0: none listed), per slice
// of kSliceScores scores its count and the keys and positions at
// slice * kSliceScores + i, in position order.
struct FilterPre {
  uint32_t spec;
  const uint32_t* count;
  const uint32_t* key;
  const uint32_t* pos;
};

__host__ __device__ __forceinline__ uint32_t topk_chunk(uint32_t n, uint32_t C) {
  return ((n + C - 1) / C + 3u) & ~3u;   // multiples of 4 positions: 16-byte aligned slices
}

// Candidates that a filtered selection can keep per CTA in `bytes` of shared
// memory (a key and a position each; 0 when the histograms do not fit).
__host__ __device__ __forceinline__ uint32_t topk_candidates(uint32_t bytes) {
  return bytes >= kFilterMinBytes ? (bytes / 8u) & ~3u : 0u;
}

// Calls f(g, keys of group g) for g = tid, tid + kThreads, ... up to the
// CTA's groups rounded up to kUnroll * kThreads (every thread of the CTA calls
// f equally often; f must ignore g >= ngroups, whose keys are zero).  The
// loads of kUnroll groups are issued before any of them is used.
template <typename Load4, typename F>
__device__ __forceinline__ void for_groups(Load4 load4, uint32_t ngroups, F f) {
  for (uint32_t g0 = 0; g0 < ngroups; g0 += kUnroll * kThreads) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t g = g0 + u * kThreads + threadIdx.x;
      v[u] = g < ngroups ? load4(g) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) f(g0 + u * kThreads + threadIdx.x, v[u]);
  }
}

// Over kPer * kThreads bins in increasing key order, finds the bin holding
// the want-th largest key: out[0] = the bin, out[1] = keys in higher bins,
// out[2] = the bin's count.  want must be in 1..(sum of the bins).  Ends with
// a block barrier, after which out[] is visible to the whole CTA.
template <uint32_t kPer>
__device__ __forceinline__ void find_cut(const uint32_t* tot, uint32_t want, uint32_t* warp_sum, uint32_t* out) {
  constexpr uint32_t nb = kPer * kThreads;
  const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t c[kPer], sum = 0;
#pragma unroll
  for (uint32_t e = 0; e < kPer; ++e) {
    c[e] = tot[nb - 1 - kPer * tid - e];
    sum += c[e];
  }
  uint32_t incl = sum;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t o = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= (uint32_t)d) incl += o;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  uint32_t before = lane < warp ? warp_sum[lane] : 0u;
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) before += __shfl_xor_sync(0xffffffffu, before, d);
  const uint32_t excl = before + incl - sum;
  if (excl < want && want <= excl + sum) {
    uint32_t above = excl;
#pragma unroll
    for (uint32_t e = 0; e < kPer; ++e) {
      if (above + c[e] >= want) {
        out[0] = nb - 1 - kPer * tid - e;
        out[1] = above;
        out[2] = c[e];
        break;
      }
      above += c[e];
    }
  }
  __syncthreads();
}

// The key seen by the selection after the filtering pass found `bucket`:
// keys below the bucket become 0, keys in it their low bits + 1, keys above
// it 2^kLowBits + 1.  Monotone, and one-to-one inside the bucket, so the k
// largest (ties to the lower position) are the same keys as before whenever
// fewer than k keys lie above the bucket and at least k in or above it.
__device__ __forceinline__ uint32_t narrow_key(uint32_t x, uint32_t bucket) {
  const uint32_t top = x >> kLowBits;
  return top > bucket ? kLowMask + 2u : (top == bucket ? (x & kLowMask) + 1u : 0u);
}
constexpr uint32_t kNarrowBits = kLowBits + 1;           // narrowed keys are below 2^kNarrowBits

__device__ __forceinline__ uint4 narrow4(uint4 v, uint32_t bucket) {
  return make_uint4(narrow_key(v.x, bucket), narrow_key(v.y, bucket), narrow_key(v.z, bucket),
                    narrow_key(v.w, bucket));
}

// Radix select over key4 (keys below 2^key_bits), then the ordered
// compaction: emit_local(i, out) for each of the k chosen keys, i its index
// in this CTA's key order and out its rank in the cluster-wide selection.
template <typename Key4, typename EmitLocal>
__device__ __forceinline__ void select_and_emit(Key4 key4, uint32_t count, uint32_t k, uint32_t key_bits,
                                                RadixSmem* rsm, uint32_t (*scratch)[2 * kWarps + 2],
                                                uint32_t (*table)[4], EmitLocal emit_local) {
  const uint32_t r = cluster_rank(), C = cluster_size();
  const RadixCut cut = cluster_radix_select(key4, count, k, key_bits, rsm, C);
  uint32_t above, at;
  cut_counts(key4, count, cut, scratch[1], &above, &at);
  const uint32_t mine[2] = {above, at};
  cluster_publish(mine, 2, table, r, C);
  uint32_t sel_before, at_before;
  cut_offsets(table, 0, r, cut.need, &sel_before, &at_before);
  cluster_compact(key4, count, cut, sel_before, at_before, scratch, [&](uint32_t i, uint32_t out) {
    if (out < k) emit_local(i, out);
  });
}

// Filtering pass (a): h = kHistCopies kFirstBins-word histograms, tot one
// more, in shared memory, zeroed before a cluster barrier that precedes this
// call.  Each warp adds into copy (warp mod kHistCopies), so that the few
// bins that most keys fall into are not all contended by every warp; the
// copies are summed, added into every CTA's tot, and the cut bucket of the
// `want` largest keys found (out[0..2] as in find_cut).
template <typename Load4>
__device__ __forceinline__ void first_digit_cut(Load4 load4, uint32_t count, uint32_t want, uint32_t* h,
                                                uint32_t* tot, uint32_t* warp_sum, uint32_t* out) {
  const uint32_t C = cluster_size();
  const uint32_t ngroups = (count + 3) / 4;
  for_groups(load4, ngroups, [&](uint32_t g, uint4 kk) {
    const uint32_t bins[4] = {kk.x >> kLowBits, kk.y >> kLowBits, kk.z >> kLowBits, kk.w >> kLowBits};
    uint32_t vm = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) vm |= (uint32_t)(g < ngroups && 4 * g + e < count) << e;
    hist_add_warp4(h + ((threadIdx.x >> 5) % kHistCopies) * kFirstBins, bins, vm);
  });
  __syncthreads();
  for (uint32_t b = threadIdx.x; b < kFirstBins; b += kThreads) {
    uint32_t v = h[b];
#pragma unroll
    for (uint32_t c = 1; c < kHistCopies; ++c) v += h[c * kFirstBins + b];
    h[b] = v;
  }
  __syncthreads();
  for (uint32_t i = threadIdx.x; i < kFirstBins * C; i += kThreads) {
    const uint32_t v = h[i & (kFirstBins - 1u)];
    if (v) dsmem_red_add_u32(dsmem_addr(&tot[i & (kFirstBins - 1u)], i >> kFirstBits), v);
  }
  cluster_sync();
  find_cut<kFirstBins / kThreads>(tot, want, warp_sum, out);
}

// The lowest float whose key is at least T: for T > 0 the keys at or above T
// are exactly the non-NaN floats at or above it (-0 compares equal to +0, as
// its key does).  Above the key of +inf it is a NaN, which admits nothing.
__device__ __forceinline__ float key_floor_float(uint32_t T) {
  if (T >= 0x80000000u) return __uint_as_float(T & 0x7fffffffu);   // +0 .. +inf
  if (T <= 0x007fffffu) return __uint_as_float(0xff800000u);       // at or below the key of -inf
  return __uint_as_float(~T);                                      // a negative float
}

// Filtering pass (b): stores, in index order, every key of this CTA whose top
// bits are at least `bucket` (ckey) with its index (cpos).  Returns how many;
// the caller guarantees that they fit.  A score is tested with one float
// compare against the bucket's lowest float.  Rounds of 16 keys per thread:
// warp w takes the 128 consecutive groups of 4 keys at round base + 128 w,
// lane l of them groups l, l + 32, l + 64, l + 96 (coalesced), so that the
// order is (warp, group row, lane); one packed warp scan (a byte per group
// row) and one block barrier per round (scratch buffers alternate as in
// cluster_compact).
template <typename LoadF4>
__device__ __forceinline__ uint32_t filter_keys(LoadF4 loadf4, uint32_t count, uint32_t bucket, uint32_t* ckey,
                                                uint32_t* cpos, uint32_t (*scratch)[2 * kWarps + 2]) {
  const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t ngroups = (count + 3) / 4;
  const float t = key_floor_float(bucket << kLowBits);
  const bool all = bucket == 0;                  // every key, NaN included
  uint32_t base = 0, parity = 0;
  for (uint32_t r0 = 0; r0 < ngroups; r0 += 4 * kThreads, parity ^= 1u) {
    const uint32_t g0 = r0 + warp * 128u + lane;
    float4 v[4];
#pragma unroll
    for (uint32_t u = 0; u < 4; ++u) {
      const uint32_t g = g0 + 32u * u;
      v[u] = g < ngroups ? loadf4(g) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    uint32_t m[4], packed = 0;
#pragma unroll
    for (uint32_t u = 0; u < 4; ++u) {
      const uint32_t g = g0 + 32u * u;
      const float f[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
      m[u] = 0;
#pragma unroll
      for (uint32_t e = 0; e < 4; ++e)
        m[u] |= (uint32_t)(g < ngroups && 4 * g + e < count && (all || f[e] >= t)) << e;
      packed |= (uint32_t)__popc(m[u]) << (8u * u);
    }
    uint32_t incl = packed;                      // bytes stay below 129: no carries
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint32_t o = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= (uint32_t)d) incl += o;
    }
    const uint32_t excl = incl - packed;
    const uint32_t tot = __shfl_sync(0xffffffffu, incl, 31);
    uint32_t* sc = scratch[parity];
    if (lane == 31) sc[warp] = (tot & 0xffu) + ((tot >> 8) & 0xffu) + ((tot >> 16) & 0xffu) + (tot >> 24);
    __syncthreads();
    const uint32_t w_l = lane < (uint32_t)kWarps ? sc[lane] : 0u;
    uint32_t w_incl = w_l;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint32_t o = __shfl_up_sync(0xffffffffu, w_incl, d);
      if (lane >= (uint32_t)d) w_incl += o;
    }
    const uint32_t woff = __shfl_sync(0xffffffffu, w_incl - w_l, warp);
    const uint32_t round = __shfl_sync(0xffffffffu, w_incl, 31);
    uint32_t row = base + woff;
#pragma unroll
    for (uint32_t u = 0; u < 4; ++u) {
      if (m[u]) {
        const uint32_t g = g0 + 32u * u;
        const float f[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
        uint32_t o = row + ((excl >> (8u * u)) & 0xffu);
#pragma unroll
        for (uint32_t e = 0; e < 4; ++e) {
          if ((m[u] >> e) & 1u) {
            ckey[o] = score_key(f[e]);
            cpos[o] = 4 * g + e;
            ++o;
          }
        }
      }
      row += (tot >> (8u * u)) & 0xffu;
    }
    base += round;
  }
  return base;
}

// The listed candidates of this CTA's slices (CTA r of C takes
// a contiguous run of slices, so that the cluster's order is position
// order) into ckey / cpos; returns how many.  One block scan of the slice
// counts per kThreads slices, then every thread copies entries, finding
// each one's slice by binary search over the scanned counts.
__device__ __forceinline__ uint32_t load_candidates(const FilterPre* pre, uint32_t n, uint32_t r, uint32_t C,
                                                    uint32_t cap, uint32_t* ckey, uint32_t* cpos,
                                                    uint32_t* scratch) {
  __shared__ uint32_t off[kThreads];
  const uint32_t tid = threadIdx.x;
  const uint32_t S = (n + kSliceScores - 1) / kSliceScores;
  const uint32_t per = (S + C - 1) / C;
  const uint32_t s0 = min(S, r * per), s1 = min(S, s0 + per);
  uint32_t m = 0;
  for (uint32_t base = s0; base < s1; base += kThreads) {   // uniform over the CTA
    const uint32_t sl = base + tid;
    const uint32_t c = sl < s1 ? min(__ldcg(&pre->count[sl]), kSliceScores) : 0u;
    uint32_t tot;
    off[tid] = block_excl_sum(c, scratch, &tot);
    __syncthreads();
    const uint32_t nsl = min((uint32_t)kThreads, s1 - base);
    for (uint32_t i = tid; i < tot; i += kThreads) {
      uint32_t lo = 0, hi = nsl;                         // the last slice whose offset is at most i
      while (hi - lo > 1) {
        const uint32_t mid = (lo + hi) >> 1;
        if (off[mid] <= i) lo = mid;
        else hi = mid;
      }
      const size_t at = (size_t)(base + lo) * kSliceScores + (i - off[lo]);
      if (m + i < cap) {                                 // always: the cut's count bounds the lists
        ckey[m + i] = __ldcg(&pre->key[at]);
        cpos[m + i] = __ldcg(&pre->pos[at]);
      }
    }
    m += tot;
    __syncthreads();                                     // off is rewritten next round
  }
  return min(m, cap);
}

// Selects the k largest of n scores with the whole cluster.  first_hist:
// NULL, or (filtered route) the counts of the top kFirstBits key bits of all
// n scores, made beforehand.  dyn_smem holds
// topk_chunk(n, C) keys when kResident, else `cand_bytes` of room for the
// filtered route's candidates (0: stream every pass).  emit(pos, out) is
// called once for every chosen position with its rank `out` in ascending
// position order (0 <= out < k).  Every remote access ends at a cluster
// barrier inside; emit may itself write to other CTAs, which the caller must
// then fence with a cluster barrier.
template <bool kResident, typename Emit>
__device__ __forceinline__ void topk_body(const float* __restrict__ scores, uint32_t n, uint32_t k,
                                          uint8_t* dyn_smem, uint32_t cand_bytes, RadixSmem* rsm, Emit emit,
                                          const uint32_t* first_hist = nullptr, const FilterPre* pre = nullptr,
                                          uint32_t* cut_out = nullptr) {
  __shared__ uint32_t scratch[2][2 * kWarps + 2];
  __shared__ uint32_t table[kMaxCluster][4];
  __shared__ uint32_t cutw[4];

  const uint32_t tid = threadIdx.x;
  const uint32_t r = cluster_rank(), C = cluster_size();
  const uint32_t chunk = topk_chunk(n, C);
  const uint64_t lo64 = (uint64_t)chunk * r;
  const uint32_t lo = lo64 < n ? (uint32_t)lo64 : n;
  const uint32_t hi = (lo64 + chunk) < n ? (uint32_t)(lo64 + chunk) : n;
  const uint32_t cnt = hi - lo;
  uint32_t* keys = reinterpret_cast<uint32_t*>(dyn_smem);
  const float* src = scores + lo;
  const bool vec = ((reinterpret_cast<uintptr_t>(src) & 15u) == 0);

  // keys 4g..4g+3 of this CTA's slice, straight from the scores
  auto load4 = [&](uint32_t g) -> uint4 {
    const uint32_t i = 4 * g;
    if (vec && i + 3 < cnt) {
      const float4 f = __ldg(reinterpret_cast<const float4*>(src) + g);
      return make_uint4(score_key(f.x), score_key(f.y), score_key(f.z), score_key(f.w));
    }
    uint32_t v[4] = {0, 0, 0, 0};
    for (uint32_t e = 0; e < 4; ++e)
      if (i + e < cnt) v[e] = score_key(__ldg(src + i + e));
    return make_uint4(v[0], v[1], v[2], v[3]);
  };
  // the same four scores, raw
  auto loadf4 = [&](uint32_t g) -> float4 {
    const uint32_t i = 4 * g;
    if (vec && i + 3 < cnt) return __ldg(reinterpret_cast<const float4*>(src) + g);
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    for (uint32_t e = 0; e < 4; ++e)
      if (i + e < cnt) v[e] = __ldg(src + i + e);
    return make_float4(v[0], v[1], v[2], v[3]);
  };
  auto emit_at = [&](uint32_t i, uint32_t out) { emit(lo + i, out); };

  radix_smem_init(rsm);
  const uint32_t cap = kResident ? 0u : topk_candidates(cand_bytes);
  if (kResident) {
    for (uint32_t g = tid; g < (cnt + 3) / 4; g += kThreads) reinterpret_cast<uint4*>(keys)[g] = load4(g);
  } else if (cap && !pre) {
    for (uint32_t b = tid; b < (kHistCopies + 1) * kFirstBins; b += kThreads) keys[b] = 0;   // the filtering histograms
  }
  cluster_sync();                                  // histograms zeroed everywhere, keys in place

  if (kResident) {
    select_and_emit([&](uint32_t g) { return reinterpret_cast<const uint4*>(keys)[g]; }, cnt, k, 32, rsm, scratch,
                    table, emit_at);
    return;
  }
  if (!cap) {
    select_and_emit(load4, cnt, k, 32, rsm, scratch, table, emit_at);
    return;
  }
  if (first_hist) {
    // the filtering pass's histogram was built beforehand over the whole
    // history (device memory, kFirstBins counts): only the cut is found here
    uint32_t* tot = keys + kHistCopies * kFirstBins;
    for (uint32_t b = tid; b < kFirstBins; b += kThreads) tot[b] = __ldcg(&first_hist[b]);
    __syncthreads();
    find_cut<kFirstBins / kThreads>(tot, k, &scratch[0][0], cutw);
    const uint32_t bucket = cutw[0];
    // keys from the bucket below the cut: the next call lists from there
    // while that leaves half the room free (a margin for the cut moving
    // down), else from the cut's own bucket
    const uint32_t below = bucket > 0 ? tot[bucket - 1] : 0u;
    uint32_t mine = 0;
    if (pre && pre->spec)
      for (uint32_t b = tid; b < kFirstBins; b += kThreads) mine += b >= pre->spec ? tot[b] : 0u;
    uint32_t listed;
    block_excl_sum(mine, &scratch[1][0], &listed);       // after it no thread reads tot
    if (cut_out && tid == 0)
      *cut_out = bucket > 1 && cutw[1] + cutw[2] + below <= cap / 2 ? bucket - 1 : bucket;
    if (pre && pre->spec) {
      // the lists hold every key in or above bucket spec: enough when the
      // cut is at or above it, and usable when they fit
      if (bucket >= pre->spec && listed <= cap) {        // uniform over the cluster
        uint32_t* ckey = keys;
        uint32_t* cpos = keys + cap;
        const uint32_t m = load_candidates(pre, n, r, C, cap, ckey, cpos, &scratch[0][0]);
        select_and_emit([&](uint32_t g) { return narrow4(reinterpret_cast<const uint4*>(ckey)[g], bucket); }, m,
                        k, kNarrowBits, rsm, scratch, table, [&](uint32_t i, uint32_t out) { emit(cpos[i], out); });
        return;
      }
    }
  } else {
    first_digit_cut(load4, cnt, k, keys, keys + kHistCopies * kFirstBins, &scratch[0][0], cutw);
  }
  const uint32_t bucket = cutw[0];
  const uint32_t total = cutw[1] + cutw[2];        // keys in or above the bucket, cluster-wide
  if (total <= cap) {
    uint32_t* ckey = keys;
    uint32_t* cpos = keys + cap;
    const uint32_t m = filter_keys(loadf4, cnt, bucket, ckey, cpos, scratch);
    select_and_emit([&](uint32_t g) { return narrow4(reinterpret_cast<const uint4*>(ckey)[g], bucket); }, m, k,
                    kNarrowBits, rsm, scratch, table, [&](uint32_t i, uint32_t out) { emit(lo + cpos[i], out); });
  } else {
    select_and_emit([&](uint32_t g) { return narrow4(load4(g), bucket); }, cnt, k, kNarrowBits, rsm, scratch,
                    table, emit_at);
  }
}

}  // namespace topk_detail
}  // namespace kvo
