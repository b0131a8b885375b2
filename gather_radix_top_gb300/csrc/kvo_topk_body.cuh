// Device body of the top-K selection of history positions from indexer
// scores, shared by the standalone kernel and the fused decode-step kernel.
//
// "From 1M Total to 15+ x 1M Contexts: GLM-5.3 KV Cache Offloading", section
// "Separate historical capacity from the current working set": the DSA
// indexer selects the top 2,048 historical positions.  Selection stays on
// the GPU ("Decision one").
//
// One thread-block cluster does the whole selection in a single launch:
//   1. each CTA owns a contiguous range of positions and keeps its keys in
//      shared memory when they fit (else re-reads the scores each pass);
//   2. an MSB-first 8-bit radix select finds the cut; each pass builds a
//      warp-aggregated per-CTA histogram and adds its nonzero bins into every
//      CTA's cluster-wide histogram over distributed shared memory (one
//      cluster barrier per pass);
//   3. an ordered compaction writes the chosen positions in ascending order:
//      per-CTA counts (taken from the radix histograms) are published over
//      DSMEM, then each CTA walks its range four keys per thread, one block
//      barrier per 4,096 keys.
// Ties at the cut go to the lowest positions because the compaction takes
// equal keys in position order.
#pragma once

#include <cstdint>

#include "kvo_device.cuh"

namespace kvo {

namespace topk_detail {

constexpr uint32_t kTopkStaticSmem = 40 * 1024;            // headroom for static smem (radix histograms)
constexpr uint32_t kTopkMaxDynSmem = 227 * 1024 - kTopkStaticSmem;

__host__ __device__ __forceinline__ uint32_t topk_chunk(uint32_t n, uint32_t C) {
  return ((n + C - 1) / C + 3u) & ~3u;   // multiples of 4 positions: 16-byte aligned slices
}

// Selects the k largest of n scores with the whole cluster.  Keys live in
// dyn_smem (topk_chunk(n, C) words) when kResident.  emit(pos, out) is called
// once for every chosen position with its rank `out` in ascending position
// order (0 <= out < k).  Every remote access ends at a cluster barrier inside;
// emit may itself write to other CTAs, which the caller must then fence with
// a cluster barrier.
template <bool kResident, typename Emit>
__device__ __forceinline__ void topk_body(const float* __restrict__ scores, uint32_t n, uint32_t k,
                                          uint8_t* dyn_smem, RadixSmem* rsm, Emit emit) {
  __shared__ uint32_t scratch[2][2 * kWarps + 2];
  __shared__ uint32_t table[kMaxCluster][4];

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

  radix_smem_init(rsm);
  if (kResident) {
    for (uint32_t g = tid; g < (cnt + 3) / 4; g += kThreads) reinterpret_cast<uint4*>(keys)[g] = load4(g);
  }
  cluster_sync();                                  // histograms zeroed everywhere, keys in place
  auto key4 = [&](uint32_t g) -> uint4 {
    if (kResident) return reinterpret_cast<const uint4*>(keys)[g];
    return load4(g);
  };

  const RadixCut cut = cluster_radix_select(key4, cnt, k, 32, rsm, C);
  uint32_t above, at;
  cut_counts(key4, cnt, cut, scratch[1], &above, &at);
  const uint32_t mine[2] = {above, at};
  cluster_publish(mine, 2, table, r, C);
  uint32_t sel_before, at_before;
  cut_offsets(table, 0, r, cut.need, &sel_before, &at_before);
  cluster_compact(key4, cnt, cut, sel_before, at_before, scratch, [&](uint32_t i, uint32_t out) {
    if (out < k) emit(lo + i, out);
  });
}

}  // namespace topk_detail
}  // namespace kvo
