// Fused decode step of one layer (kvo_decode_step): append the new rows,
// select the top-K positions and resolve + gather them, in one cluster
// launch.  (Many layers at once go through kvo_layers.cu.)
//
// "From 1M Total to 15+ x 1M Contexts: GLM-5.3 KV Cache Offloading",
// "Decision three: let the GPU manage the hot cache directly": the CPU stays
// out of the per-selection loop; selection, lookup and gather run on the GPU
// back to back.  Fusing them also removes two kernel launches and the trip of
// the selection through global memory: the top-K compaction hands each
// selected position straight to the CTA that resolves it, over distributed
// shared memory.
//
// The step's results are those of append, then select, then resolve: the
// selection sees the new rows, and the resolve reads them from their device
// copy; their copy in the host history (or the recent ring) is written while
// the resolve waits for CTA 0's victims.
#include <cstdint>
#include <cstring>

#include "kvo_internal.h"
#include "kvo_resolve_body.cuh"
#include "kvo_topk_body.cuh"

namespace kvo {

namespace {

using namespace resolve_detail;
using namespace topk_detail;

struct StepArgs {
  ResolveArgs R;              // fused = 1; R.len = history length after the append
  const float* scores;        // NULL: resolve the selection in R.idx as given
  uint32_t n;
  int32_t* idx;               // the selection, also returned to the caller
  const uint4* new_rows;      // r rows appended in this step (device memory)
  uint4* hist_dst;            // device address of history row `old length`
  uint32_t old_len;
  uint32_t r;
  uint32_t to_ram;            // the first to_ram new rows go to the host history, the rest to the recent ring
  uint32_t topk_bytes;        // dynamic shared memory of the top-K phase (resident keys or candidates)
};

// One layer's step, run by one cluster: select (with scores), resolve, append.
template <bool kResident, bool kLru>
__device__ __forceinline__ void decode_body(const StepArgs& s, uint8_t* dyn_smem, RadixSmem* rsm) {
  const uint32_t tid = threadIdx.x, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  constexpr uint32_t kVec = KVO_ROW_BYTES / 16;

  uint8_t* rdyn = dyn_smem + s.topk_bytes;
  if (s.scores) {
    const SmemLayout lay = smem_layout(s.R.k, s.R.kchunk, s.R.hchunk, s.R.L.hot_rows, s.R.stage_rows);
    int32_t* sel = reinterpret_cast<int32_t*>(rdyn + lay.sel);
    const uint32_t kchunk = s.R.kchunk;
    topk_body<kResident>(s.scores, s.n, s.R.k, dyn_smem, s.topk_bytes, rsm, [&](uint32_t pos, uint32_t out) {
      s.idx[out] = (int32_t)pos;
      prefetch_l2(&s.R.L.pos2slot[pos]);           // the resolve looks it up next
      const uint32_t q = out / kchunk;               // CTA q + 1 resolves entries [q * kchunk, ...)
      dsmem_st_u32(dsmem_addr(&sel[out - q * kchunk], q + 1), pos);
    });
    cluster_sync();                                // every selected position delivered
  }
  // The append: one warp per new row, to the host history when the row is
  // below the step's RAM length (always without a recent ring; with one,
  // the rows whose batch of the copyback completes in this step), else to
  // the ring.  This call reads these rows from their device copy (the
  // resolve's fresh rows), so they are written while CTAs 1..C-1 wait for
  // CTA 0's victims rather than by CTA 0 ahead of the top-K.
  const LayerView& L = s.R.L;
  resolve_body<kLru>(s.R, rdyn, [&](uint32_t w, uint32_t nw) {
    for (uint32_t i = w; i < s.r; i += nw) {
      uint4* dst = i >= s.to_ram ? reinterpret_cast<uint4*>(L.recent) + (size_t)((s.old_len + i) & (L.ring_rows - 1u)) * kVec
                                 : s.hist_dst + (size_t)i * kVec;
      dst[lane] = s.new_rows[(size_t)i * kVec + lane];
      if (lane < kVec - 32) dst[32 + lane] = s.new_rows[(size_t)i * kVec + 32 + lane];
    }
  });
  if (rank == 0 && tid == 0) s.R.L.counters[1] = s.R.len;
}

template <bool kResident, bool kLru>
__global__ void __launch_bounds__(kThreads, 1) decode_step_kernel(const StepArgs s) {
  extern __shared__ __align__(16) uint8_t dyn_smem[];
  __shared__ RadixSmem rsm;                        // the top-K phase's radix histograms
  decode_body<kResident, kLru>(s, dyn_smem, &rsm);
}

struct StepConfig {
  bool init = false;
  int cluster = 0;
};
StepConfig g_step[64];

constexpr size_t kStepMaxDynSmem = 187 * 1024;     // 227 KB less the static radix histograms

cudaError_t step_init(int* cluster) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  StepConfig& cfg = g_step[dev & 63];
  if (!cfg.init) {
    const void* kernels[4] = {(const void*)decode_step_kernel<true, true>, (const void*)decode_step_kernel<false, true>,
                              (const void*)decode_step_kernel<true, false>, (const void*)decode_step_kernel<false, false>};
    int c1 = (int)kMaxCluster;
    for (const void* kern : kernels) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kStepMaxDynSmem);
      if (e != cudaSuccess) return e;
      const int c = best_cluster(kern, kStepMaxDynSmem, (int)kMaxCluster);
      c1 = c < c1 ? c : c1;
    }
    cfg.cluster = c1;
    if (cfg.cluster == 0) return cudaErrorInvalidConfiguration;
    cfg.init = true;
  }
  *cluster = cfg.cluster;
  return cudaSuccess;
}

// Fills one layer's StepArgs for a cluster of C CTAs.  *need_res / *need_stream:
// dynamic shared memory with the keys resident / streamed (0 when it does not
// fit); *stream_topk: the top-K phase's share when streamed (what the resolve
// phase leaves, for the filtered route's candidates).
void build_step(const StepTask& t, uint32_t k, uint32_t* status, uint32_t C, StepArgs* s, size_t* need_res,
                size_t* need_stream, uint32_t* stream_topk) {
  const LayerView& L = t.L;
  ResolveArgs& a = s->R;
  std::memset(static_cast<void*>(s), 0, sizeof *s);
  a.L = L;
  a.idx = t.idx;
  a.out_rows = t.out_rows;
  a.out_bf16 = t.out_bf16;
  a.out_host = t.out_host;
  a.status = status;
  a.k = k;
  a.kchunk = (k + C - 2) / (C - 1);                 // CTA 0 keeps the LRU order, CTAs 1..C-1 the entries
  a.hchunk = ((L.hot_rows + C - 1) / C + 127u) & ~127u;
  a.fused = 1;
  a.sel_in_smem = t.scores ? 1u : 0u;
  a.len = t.old_len + t.r;
  a.fresh = t.r ? static_cast<const uint8_t*>(t.new_rows) : nullptr;
  a.fresh_from = t.old_len;
  s->scores = t.scores;
  s->n = t.n;
  s->idx = t.idx;
  s->new_rows = static_cast<const uint4*>(t.new_rows);
  s->hist_dst = reinterpret_cast<uint4*>(const_cast<uint8_t*>(L.hist) + (size_t)t.old_len * KVO_ROW_BYTES);
  s->old_len = t.old_len;
  s->r = t.r;
  // L.ram_len is the RAM length after this step's append and copyback
  s->to_ram = !L.ring_rows ? t.r
              : L.ram_len <= t.old_len ? 0u
              : L.ram_len - t.old_len < t.r ? L.ram_len - t.old_len : t.r;
  // staged gather when the rows fit, else rows through registers
  a.stage_rows = L.gather_mode != KVO_GATHER_LOADS ? (a.kchunk < kStageMax ? a.kchunk : kStageMax) : 0u;
  a.stage_min_miss_pct = L.gather_mode == KVO_GATHER_STAGED ? 0u : L.auto_miss_pct;
  SmemLayout lay = smem_layout(k, a.kchunk, a.hchunk, L.hot_rows, a.stage_rows);
  if (a.stage_rows && lay.total > kStepMaxDynSmem) {
    a.stage_rows = 0;
    lay = smem_layout(k, a.kchunk, a.hchunk, L.hot_rows, 0);
  }
  const size_t topk_res = t.scores ? ((size_t)topk_chunk(t.n, C) * 4u + 15u) & ~(size_t)15u : 0u;
  const size_t cand = t.scores && lay.total <= kStepMaxDynSmem ? (kStepMaxDynSmem - lay.total) & ~(size_t)15u : 0u;
  *stream_topk = (uint32_t)cand;
  *need_stream = lay.total <= kStepMaxDynSmem ? cand + lay.total : 0u;
  *need_res = topk_res + lay.total <= kStepMaxDynSmem ? topk_res + lay.total : 0u;
  s->topk_bytes = (uint32_t)topk_res;               // replaced by *stream_topk when keys are streamed
}

cudaError_t launch(uint32_t C, size_t smem, cudaStream_t stream, bool resident, bool lru, const StepArgs& one) {
  cudaLaunchConfig_t lc = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  lc.gridDim = dim3(C, 1, 1);
  lc.blockDim = dim3(kThreads, 1, 1);
  lc.dynamicSmemBytes = smem;
  lc.stream = stream;
  lc.attrs = attr;
  lc.numAttrs = 1;
  if (resident) return lru ? cudaLaunchKernelEx(&lc, decode_step_kernel<true, true>, one)
                           : cudaLaunchKernelEx(&lc, decode_step_kernel<true, false>, one);
  return lru ? cudaLaunchKernelEx(&lc, decode_step_kernel<false, true>, one)
             : cudaLaunchKernelEx(&lc, decode_step_kernel<false, false>, one);
}

}  // namespace

cudaError_t launch_decode_step(const LayerView& L, const void* new_rows, uint32_t r, uint32_t old_len,
                               const float* scores, uint32_t n, uint32_t k, int32_t* idx, uint8_t* out_rows,
                               uint16_t* out_bf16, uint32_t* status, int max_cluster, cudaStream_t stream,
                               bool out_host) {
  int cl = 0;
  cudaError_t e = step_init(&cl);
  if (e != cudaSuccess) return e;
  const uint32_t C = (uint32_t)(cl < max_cluster ? cl : max_cluster);
  const StepTask t = {L, new_rows, r, old_len, scores, n, idx, out_rows, out_bf16, out_host ? 1u : 0u};
  StepArgs s;
  size_t need_res = 0, need_stream = 0;
  uint32_t stream_topk = 0;
  build_step(t, k, status, C, &s, &need_res, &need_stream, &stream_topk);
  if (!need_stream) return cudaErrorInvalidValue;
  const bool resident = need_res != 0;
  if (!resident) s.topk_bytes = stream_topk;
  return launch(C, resident ? need_res : need_stream, stream, resident, L.policy == KVO_POLICY_LRU, s);
}

}  // namespace kvo
