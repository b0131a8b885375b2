// Top-K selection of history positions from indexer scores.
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
#include <cstdint>

#include "kvo_device.cuh"
#include "kvo_internal.h"

namespace kvo {

namespace {

constexpr uint32_t kTopkStaticSmem = 6144;                 // headroom for static smem
constexpr uint32_t kTopkMaxDynSmem = 227 * 1024 - kTopkStaticSmem;

__host__ __device__ __forceinline__ uint32_t topk_chunk(uint32_t n, uint32_t C) {
  return ((n + C - 1) / C + 3u) & ~3u;   // multiples of 4 positions: 16-byte aligned slices
}

template <bool kResident>
__global__ void __launch_bounds__(kThreads, 1)
    topk_kernel(const float* __restrict__ scores, uint32_t n, uint32_t k, int32_t* __restrict__ idx) {
  extern __shared__ __align__(16) uint8_t dyn_smem[];
  __shared__ RadixSmem rsm;
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

  radix_smem_init(&rsm);
  if (kResident) {
    for (uint32_t g = tid; g < (cnt + 3) / 4; g += kThreads) reinterpret_cast<uint4*>(keys)[g] = load4(g);
  }
  cluster_sync();                                  // histograms zeroed everywhere, keys in place
  auto key4 = [&](uint32_t g) -> uint4 {
    if (kResident) return reinterpret_cast<const uint4*>(keys)[g];
    return load4(g);
  };

  const RadixCut cut = cluster_radix_select(key4, cnt, k, 32, &rsm, C);
  const uint32_t mine[2] = {cut.above, cut.at};
  cluster_publish(mine, 2, table, r, C);
  uint32_t sel_before, at_before;
  cut_offsets(table, 0, r, cut.need, &sel_before, &at_before);
  cluster_compact(key4, cnt, cut, sel_before, at_before, scratch, [&](uint32_t i, uint32_t out) {
    if (out < k) idx[out] = (int32_t)(lo + i);
  });
  // Every remote access happened before the publish barrier: CTAs may exit.
}

struct TopkConfig {
  bool init = false;
  int cluster_res = 0, cluster_stream = 0;
};
TopkConfig g_topk[64];

}  // namespace

cudaError_t launch_topk(const float* scores, uint32_t n, uint32_t k, int32_t* idx,
                        int max_cluster, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  TopkConfig& cfg = g_topk[dev & 63];
  if (!cfg.init) {
    e = cudaFuncSetAttribute(topk_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kTopkMaxDynSmem);
    if (e != cudaSuccess) return e;
    cfg.cluster_res = best_cluster((const void*)topk_kernel<true>, kTopkMaxDynSmem, (int)kMaxCluster);
    cfg.cluster_stream = best_cluster((const void*)topk_kernel<false>, 0, (int)kMaxCluster);
    if (cfg.cluster_res == 0 || cfg.cluster_stream == 0) return cudaErrorInvalidConfiguration;
    cfg.init = true;
  }
  // Resident when one CTA's share of the keys fits in shared memory.
  int C = cfg.cluster_res < max_cluster ? cfg.cluster_res : max_cluster;
  uint32_t chunk = topk_chunk(n, (uint32_t)C);
  const bool resident = (uint64_t)chunk * 4u <= kTopkMaxDynSmem;
  if (!resident) {
    C = cfg.cluster_stream < max_cluster ? cfg.cluster_stream : max_cluster;
    chunk = topk_chunk(n, (uint32_t)C);
  }

  cudaLaunchConfig_t lc = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  lc.gridDim = dim3(C, 1, 1);
  lc.blockDim = dim3(kThreads, 1, 1);
  lc.dynamicSmemBytes = resident ? (size_t)chunk * 4u : 0;
  lc.stream = stream;
  lc.attrs = attr;
  lc.numAttrs = 1;
  if (resident) return cudaLaunchKernelEx(&lc, topk_kernel<true>, scores, n, k, idx);
  return cudaLaunchKernelEx(&lc, topk_kernel<false>, scores, n, k, idx);
}

int best_cluster(const void* kernel, size_t smem, int want) {
  if (want >= 16) {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
      cudaGetLastError();
      want = 8;
    }
  }
  for (int c = want; c >= 2; c >>= 1) {
    cudaLaunchConfig_t lc = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = c;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    lc.gridDim = dim3(c, 1, 1);
    lc.blockDim = dim3(kThreads, 1, 1);
    lc.dynamicSmemBytes = smem;
    lc.attrs = attr;
    lc.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, kernel, &lc) == cudaSuccess && clusters > 0) return c;
    cudaGetLastError();
  }
  return 0;
}

}  // namespace kvo
