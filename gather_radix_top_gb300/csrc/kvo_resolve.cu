// Standalone resolve + gather launch (kvo_resolve_gather); the device body
// is in kvo_resolve_body.cuh.
#include <cstdint>

#include "kvo_resolve_body.cuh"

namespace kvo {

namespace {

using namespace resolve_detail;

template <bool kLru>
__global__ void __launch_bounds__(kThreads, 1) resolve_gather_kernel(const ResolveArgs a) {
  extern __shared__ __align__(16) uint8_t dyn_smem[];
  resolve_body<kLru>(a, dyn_smem);
}

struct ResolveConfig {
  bool init = false;
  int cluster = 0;
};
ResolveConfig g_resolve[64];

constexpr size_t kResolveMaxDynSmem = 220 * 1024;

}  // namespace

cudaError_t launch_resolve(const LayerView& L, const int32_t* idx, uint32_t k, uint8_t* out_rows,
                           uint16_t* out_bf16, uint32_t* status, int max_cluster,
                           cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  ResolveConfig& cfg = g_resolve[dev & 63];
  if (!cfg.init) {
    e = cudaFuncSetAttribute(resolve_gather_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kResolveMaxDynSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(resolve_gather_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kResolveMaxDynSmem);
    if (e != cudaSuccess) return e;
    const int c1 = best_cluster((const void*)resolve_gather_kernel<true>, kResolveMaxDynSmem, (int)kMaxCluster);
    const int c2 = best_cluster((const void*)resolve_gather_kernel<false>, kResolveMaxDynSmem, (int)kMaxCluster);
    cfg.cluster = c1 < c2 ? c1 : c2;
    if (cfg.cluster == 0) return cudaErrorInvalidConfiguration;
    cfg.init = true;
  }
  const uint32_t C = (uint32_t)(cfg.cluster < max_cluster ? cfg.cluster : max_cluster);
  ResolveArgs a;
  a.L = L;
  a.idx = idx;
  a.out_rows = out_rows;
  a.out_bf16 = out_bf16;
  a.status = status;
  a.k = k;
  a.kchunk = (k + C - 2) / (C - 1);                 // CTA 0 keeps the LRU order, CTAs 1..C-1 the entries
  a.hchunk = ((L.hot_rows + C - 1) / C + 127u) & ~127u;
  a.fused = 0;
  a.sel_in_smem = 0;
  a.len = 0;
  a.fresh = nullptr;
  a.fresh_from = 0;
  a.stage_rows = L.gather_mode != KVO_GATHER_LOADS ? (a.kchunk < kStageMax ? a.kchunk : kStageMax) : 0u;
  a.stage_min_miss_pct = L.gather_mode == KVO_GATHER_STAGED ? 0u : L.auto_miss_pct;
  SmemLayout lay = smem_layout(k, a.kchunk, a.hchunk, L.hot_rows, a.stage_rows);
  if (a.stage_rows && lay.total > kResolveMaxDynSmem) {
    a.stage_rows = 0;
    lay = smem_layout(k, a.kchunk, a.hchunk, L.hot_rows, 0);
  }
  if (lay.total > kResolveMaxDynSmem) return cudaErrorInvalidValue;

  cudaLaunchConfig_t lc = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  lc.gridDim = dim3(C, 1, 1);
  lc.blockDim = dim3(kThreads, 1, 1);
  lc.dynamicSmemBytes = lay.total;
  lc.stream = stream;
  lc.attrs = attr;
  lc.numAttrs = 1;
  if (L.policy == KVO_POLICY_LRU) return cudaLaunchKernelEx(&lc, resolve_gather_kernel<true>, a);
  return cudaLaunchKernelEx(&lc, resolve_gather_kernel<false>, a);
}

}  // namespace kvo
