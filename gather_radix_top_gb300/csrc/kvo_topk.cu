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
//   2. an MSB-first 8-bit radix select finds the cut; each pass builds
//      per-CTA histograms, and every CTA sums all of them over distributed
//      shared memory (one cluster barrier per pass);
//   3. an ordered compaction writes the chosen positions in ascending order:
//      per-CTA counts are exchanged over DSMEM, then each CTA scans its range
//      tile by tile with warp ballots.
// Ties at the cut go to the lowest positions because the compaction takes
// equal keys in position order.
#include <cstdint>

#include "kvo_device.cuh"
#include "kvo_internal.h"

namespace kvo {

namespace {

constexpr uint32_t kTopkStaticSmem = 4096;                 // headroom for static smem
constexpr uint32_t kTopkMaxDynSmem = 227 * 1024 - kTopkStaticSmem;

__device__ __forceinline__ void range_of(uint32_t n, uint32_t r, uint32_t C, uint32_t* lo,
                                         uint32_t* hi) {
  // chunk boundaries on multiples of 4 positions (16-byte aligned scores)
  const uint32_t chunk = ((n + C - 1) / C + 3u) & ~3u;
  const uint64_t a = (uint64_t)chunk * r;
  *lo = a < n ? (uint32_t)a : n;
  *hi = (a + chunk) < n ? (uint32_t)(a + chunk) : n;
}

template <bool kResident>
__global__ void __launch_bounds__(kThreads, 1)
    topk_kernel(const float* __restrict__ scores, uint32_t n, uint32_t k, int32_t* __restrict__ idx) {
  extern __shared__ __align__(16) uint8_t dyn_smem[];
  __shared__ RadixSmem rsm;
  __shared__ uint32_t scratch[kWarps + 1];
  __shared__ uint32_t counts[2];          // this CTA's (above-cut, at-cut) counts, read remotely
  __shared__ uint32_t offsets[2];         // (selected before this CTA, at-cut before this CTA)

  const uint32_t tid = threadIdx.x;
  const uint32_t r = cluster_rank(), C = cluster_size();
  uint32_t lo, hi;
  range_of(n, r, C, &lo, &hi);
  const uint32_t cnt = hi - lo;
  uint32_t* keys = reinterpret_cast<uint32_t*>(dyn_smem);
  const float* src = scores + lo;

  if (kResident) {
    const bool vec = ((reinterpret_cast<uintptr_t>(src) & 15u) == 0);
    const uint32_t nvec = vec ? cnt / 4 : 0;
    const float4* src4 = reinterpret_cast<const float4*>(src);
    for (uint32_t i = tid; i < nvec; i += kThreads) {
      const float4 f = __ldg(src4 + i);
      reinterpret_cast<uint4*>(keys)[i] =
          make_uint4(score_key(f.x), score_key(f.y), score_key(f.z), score_key(f.w));
    }
    for (uint32_t i = nvec * 4 + tid; i < cnt; i += kThreads) keys[i] = score_key(__ldg(src + i));
    __syncthreads();
  }
  auto key_at = [&](uint32_t i) -> uint32_t {
    if (kResident) return keys[i];
    return score_key(__ldg(src + i));
  };

  const RadixCut cut = cluster_radix_select(key_at, cnt, k, &rsm, C);
  const uint32_t shift = cut.shift, top = cut.prefix >> shift, need = cut.need;

  uint32_t above = 0, at = 0;
  for (uint32_t i = tid; i < cnt; i += kThreads) {
    const uint32_t t = key_at(i) >> shift;
    above += t > top;
    at += t == top;
  }
  above = block_sum(above, scratch);
  at = block_sum(at, scratch);
  if (tid == 0) {
    counts[0] = above;
    counts[1] = at;
  }
  cluster_sync();
  if (tid == 0) {
    uint32_t sel_before = 0, at_before = 0;
    for (uint32_t q = 0; q < r; ++q) {
      const uint32_t a = dsmem_ld_u32(dsmem_addr(&counts[0], q));
      const uint32_t e = dsmem_ld_u32(dsmem_addr(&counts[1], q));
      const uint32_t left = need > at_before ? need - at_before : 0u;
      sel_before += a + (e < left ? e : left);
      at_before += e;
    }
    offsets[0] = sel_before;
    offsets[1] = at_before;
  }
  __syncthreads();
  const uint32_t sel_before = offsets[0], at_before = offsets[1];

  uint32_t run_sel = 0, run_at = 0;
  for (uint32_t base = 0; base < cnt; base += kThreads) {
    const uint32_t i = base + tid;
    const bool valid = i < cnt;
    const uint32_t t = valid ? key_at(i) >> shift : 0u;
    const bool is_at = valid && t == top;
    const bool is_above = valid && t > top;
    uint32_t tile_at, tile_sel;
    const uint32_t at_rank = block_flag_scan(is_at, scratch, &tile_at);
    const bool sel = is_above || (is_at && at_before + run_at + at_rank < need);
    const uint32_t sel_rank = block_flag_scan(sel, scratch, &tile_sel);
    const uint32_t out = sel_before + run_sel + sel_rank;
    if (sel && out < k) idx[out] = (int32_t)(lo + i);
    run_at += tile_at;
    run_sel += tile_sel;
  }
  // Keep this CTA's shared memory alive until every remote read is done.
  cluster_sync();
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
    cfg.cluster_res = best_cluster((const void*)topk_kernel<true>, kTopkMaxDynSmem, 16);
    cfg.cluster_stream = best_cluster((const void*)topk_kernel<false>, 0, 16);
    if (cfg.cluster_res == 0 || cfg.cluster_stream == 0) return cudaErrorInvalidConfiguration;
    cfg.init = true;
  }
  // Resident when one CTA's share of the keys fits in shared memory.
  int C = cfg.cluster_res < max_cluster ? cfg.cluster_res : max_cluster;
  uint32_t chunk = ((n + C - 1) / C + 3u) & ~3u;
  bool resident = (uint64_t)chunk * 4u <= kTopkMaxDynSmem;
  if (!resident) C = cfg.cluster_stream < max_cluster ? cfg.cluster_stream : max_cluster;

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
