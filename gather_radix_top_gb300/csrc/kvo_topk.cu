// Standalone top-K launch (kvo_select_topk); the device body is in
// kvo_topk_body.cuh.
#include <cstdint>

#include "kvo_internal.h"
#include "kvo_topk_body.cuh"

namespace kvo {

namespace {

using namespace topk_detail;

// One cluster per row of scores: cluster blockIdx.x / clusterDim.x selects
// from row scores + row * ld into idx + row * k.
template <bool kResident>
__global__ void __launch_bounds__(kThreads, 1)
    topk_kernel(const float* __restrict__ scores, uint32_t n, uint64_t ld, uint32_t k, int32_t* __restrict__ idx) {
  extern __shared__ __align__(16) uint8_t dyn_smem[];
  __shared__ RadixSmem rsm;
  const uint32_t row = blockIdx.x / cluster_size();
  const float* s = scores + row * ld;
  int32_t* out_idx = idx + (size_t)row * k;
  topk_body<kResident>(s, n, k, dyn_smem, kTopkMaxDynSmem, &rsm,
                       [&](uint32_t pos, uint32_t out) { out_idx[out] = (int32_t)pos; });
}

struct TopkConfig {
  bool init = false;
  int cluster_res = 0, cluster_stream = 0;
};
TopkConfig g_topk[64];

}  // namespace

cudaError_t launch_topk(const float* scores, uint32_t n, uint32_t k, int32_t* idx,
                        int max_cluster, cudaStream_t stream, uint32_t nq, uint64_t ld) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  TopkConfig& cfg = g_topk[dev & 63];
  if (!cfg.init) {
    for (const void* kern : {(const void*)topk_kernel<true>, (const void*)topk_kernel<false>}) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTopkMaxDynSmem);
      if (e != cudaSuccess) return e;
    }
    cfg.cluster_res = best_cluster((const void*)topk_kernel<true>, kTopkMaxDynSmem, (int)kMaxCluster);
    cfg.cluster_stream = best_cluster((const void*)topk_kernel<false>, kTopkMaxDynSmem, (int)kMaxCluster);
    if (cfg.cluster_res == 0 || cfg.cluster_stream == 0) return cudaErrorInvalidConfiguration;
    cfg.init = true;
  }
  // Resident when one CTA's share of the keys fits in shared memory, else
  // the filtered route with all of it for candidates.
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
  lc.gridDim = dim3((unsigned)C * nq, 1, 1);
  lc.blockDim = dim3(kThreads, 1, 1);
  lc.dynamicSmemBytes = resident ? (size_t)chunk * 4u : kTopkMaxDynSmem;   // streamed: room for candidates
  lc.stream = stream;
  lc.attrs = attr;
  lc.numAttrs = 1;
  if (resident) return cudaLaunchKernelEx(&lc, topk_kernel<true>, scores, n, ld, k, idx);
  return cudaLaunchKernelEx(&lc, topk_kernel<false>, scores, n, ld, k, idx);
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
