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
//      smallest j of each missing position wins (dedupe, no extra table).
//   P2 compact: unique misses are ranked in j order (per-CTA counts over
//      DSMEM, then warp-ballot scans) and written to CTA 0's shared memory.
//   P3 victims: a cluster radix select of the M smallest last_use among
//      slots with last_use < t (ties -> lower slot); the winners go to CTA 0
//      as 64-bit (last_use, slot) keys and CTA 0 bitonic-sorts them.
//   P4 map update (CTA 0): unmap the evicted position, map the new one,
//      stamp last_use = t, tell the owning CTA which slot to fill.
//   P5 gather: one warp per row, 16-byte loads (41 per 656-byte row) from
//      the hot slot (HBM) or from host memory (zero-copy), stores to the
//      output rows, the victim slot and, optionally, the bf16 dequant.
#include <cstdint>

#include <cuda_fp16.h>

#include "kvo_device.cuh"
#include "kvo_internal.h"

namespace kvo {

namespace {

constexpr int32_t kSlotMiss = -1;
constexpr int32_t kSlotInvalid = -2;
constexpr int32_t kFillUnique = -3;      // unique miss whose victim is not known yet
constexpr uint32_t kRowVec = KVO_ROW_BYTES / 16;   // 41 16-byte pieces per row

struct ResolveArgs {
  LayerView L;
  const int32_t* idx;
  uint8_t* out_rows;
  uint16_t* out_bf16;
  uint32_t* status;
  uint32_t k;
  uint32_t kchunk;        // selection entries per CTA
  uint32_t hchunk;        // hot slots per CTA
  uint32_t sort_len;      // power of two >= k
};

struct SmemLayout {
  uint32_t sortkeys_off, lukeys_off, meta_slot_off, meta_fill_off, meta_pos_off, miss_pos_off,
      miss_j_off, total;
};

__host__ __device__ inline SmemLayout smem_layout(uint32_t k, uint32_t kchunk, uint32_t hchunk,
                                                  uint32_t sort_len) {
  SmemLayout s;
  uint32_t o = 0;
  s.sortkeys_off = o;  o += sort_len * 8u;
  s.lukeys_off = o;    o += hchunk * 4u;
  s.meta_slot_off = o; o += kchunk * 4u;
  s.meta_fill_off = o; o += kchunk * 4u;
  s.meta_pos_off = o;  o += kchunk * 4u;
  s.miss_pos_off = o;  o += k * 4u;
  s.miss_j_off = o;    o += k * 4u;
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

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  return bf16_rne(a) | (bf16_rne(b) << 16);
}

__device__ __forceinline__ void dequant16(uint32_t w, float s, float* o) {
  o[0] = (float)(int8_t)(w & 0xffu) * s;
  o[1] = (float)(int8_t)((w >> 8) & 0xffu) * s;
  o[2] = (float)(int8_t)((w >> 16) & 0xffu) * s;
  o[3] = (float)(int8_t)(w >> 24) * s;
}

__global__ void __launch_bounds__(kThreads, 1) resolve_gather_kernel(const ResolveArgs a) {
  extern __shared__ __align__(16) uint8_t dyn_smem[];
  __shared__ RadixSmem rsm;
  __shared__ uint32_t scratch[kWarps + 1];
  __shared__ uint32_t xch[4];          // per-CTA values read by other CTAs
  __shared__ uint32_t bcast[4];

  const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t r = cluster_rank(), C = cluster_size();
  const LayerView& L = a.L;
  const uint32_t k = a.k;

  const SmemLayout lay = smem_layout(k, a.kchunk, a.hchunk, a.sort_len);
  uint64_t* sortkeys = reinterpret_cast<uint64_t*>(dyn_smem + lay.sortkeys_off);
  uint32_t* lukeys = reinterpret_cast<uint32_t*>(dyn_smem + lay.lukeys_off);
  int32_t* meta_slot = reinterpret_cast<int32_t*>(dyn_smem + lay.meta_slot_off);
  int32_t* meta_fill = reinterpret_cast<int32_t*>(dyn_smem + lay.meta_fill_off);
  int32_t* meta_pos = reinterpret_cast<int32_t*>(dyn_smem + lay.meta_pos_off);
  int32_t* miss_pos = reinterpret_cast<int32_t*>(dyn_smem + lay.miss_pos_off);
  int32_t* miss_j = reinterpret_cast<int32_t*>(dyn_smem + lay.miss_j_off);

  const uint32_t t = L.counters[0] + 1u;        // this call's step
  const uint32_t len = L.counters[1];
  const uint32_t jlo = min(k, r * a.kchunk), jhi = min(k, jlo + a.kchunk), jcnt = jhi - jlo;

  // ---------------------------------------------------------------- P1
  uint32_t nhit = 0, nmiss = 0, ninv = 0;
  for (uint32_t jj = tid; jj < jcnt; jj += kThreads) {
    const uint32_t j = jlo + jj;
    const int32_t p = a.idx[j];
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
    meta_fill[jj] = -1;
  }
  cluster_sync();                                   // B1: stamps and claims visible

  // ---------------------------------------------------------------- P2
  uint32_t nuniq = 0;
  for (uint32_t jj = tid; jj < jcnt; jj += kThreads) {
    // __ldcg: the claims were made by other CTAs; read them from L2.
    if (meta_slot[jj] == kSlotMiss &&
        __ldcg(&L.pos2slot[meta_pos[jj]]) == (int32_t)(jlo + jj) - (int32_t)k - 1) {
      meta_fill[jj] = kFillUnique;
      ++nuniq;
    }
  }
  nuniq = block_sum(nuniq, scratch);
  if (tid == 0) xch[0] = nuniq;
  if (r == 0 && tid == 0) L.counters[0] = t;       // every CTA read the old step before B1
  cluster_sync();                                   // B2
  if (tid < 32) {
    const uint32_t v = lane < C ? dsmem_ld_u32(dsmem_addr(&xch[0], lane)) : 0u;
    uint32_t incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint32_t o = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= (uint32_t)d) incl += o;
    }
    if (lane == r) bcast[0] = incl - v;
    if (lane == 31) bcast[1] = incl;
  }
  __syncthreads();
  const uint32_t uniq_before = bcast[0], M = bcast[1];
  __syncthreads();
  {
    const uint32_t mp0 = dsmem_addr(miss_pos, 0), mj0 = dsmem_addr(miss_j, 0);
    uint32_t run = 0;
    for (uint32_t base = 0; base < jcnt; base += kThreads) {
      const uint32_t jj = base + tid;
      const bool f = jj < jcnt && meta_fill[jj] == kFillUnique;
      uint32_t tile;
      const uint32_t rank = block_flag_scan(f, scratch, &tile);
      const uint32_t i = uniq_before + run + rank;
      if (f && i < k) {
        dsmem_st_u32(mp0 + 4u * i, (uint32_t)meta_pos[jj]);
        dsmem_st_u32(mj0 + 4u * i, jlo + jj);
      }
      run += tile;
    }
  }

  uint32_t nevict = 0;
  if (M > 0) {
    // -------------------------------------------------------------- P3
    const uint32_t H = L.hot_rows;
    const uint32_t slo = min(H, r * a.hchunk), shi = min(H, slo + a.hchunk), hcnt = shi - slo;
    for (uint32_t i = tid; i < hcnt; i += kThreads) {
      const uint32_t lu = __ldcg(&L.last_use[slo + i]);   // stamps came from other CTAs
      lukeys[i] = lu < t ? ~lu : 0u;               // larger key = older; pinned slots excluded
    }
    __syncthreads();
    auto key_at = [&](uint32_t i) -> uint32_t { return lukeys[i]; };
    const RadixCut cut = cluster_radix_select(key_at, hcnt, M, &rsm, C);
    const uint32_t shift = cut.shift, top = cut.prefix >> shift, need = cut.need;
    uint32_t above = 0, at = 0;
    for (uint32_t i = tid; i < hcnt; i += kThreads) {
      const uint32_t v = lukeys[i] >> shift;
      above += v > top;
      at += v == top;
    }
    above = block_sum(above, scratch);
    at = block_sum(at, scratch);
    if (tid == 0) {
      xch[1] = above;
      xch[2] = at;
    }
    cluster_sync();                                 // B3
    if (tid == 0) {
      uint32_t sel_before = 0, at_before = 0;
      for (uint32_t q = 0; q < r; ++q) {
        const uint32_t av = dsmem_ld_u32(dsmem_addr(&xch[1], q));
        const uint32_t e = dsmem_ld_u32(dsmem_addr(&xch[2], q));
        const uint32_t left = need > at_before ? need - at_before : 0u;
        sel_before += av + (e < left ? e : left);
        at_before += e;
      }
      bcast[2] = sel_before;
      bcast[3] = at_before;
    }
    __syncthreads();
    const uint32_t sel_before = bcast[2], at_before = bcast[3];
    const uint32_t sk0 = dsmem_addr(sortkeys, 0);
    uint32_t run_sel = 0, run_at = 0;
    for (uint32_t base = 0; base < hcnt; base += kThreads) {
      const uint32_t i = base + tid;
      const bool valid = i < hcnt;
      const uint32_t key = valid ? lukeys[i] : 0u;
      const uint32_t v = key >> shift;
      const bool is_at = valid && v == top;
      const bool is_above = valid && v > top;
      uint32_t tile_at, tile_sel;
      const uint32_t at_rank = block_flag_scan(is_at, scratch, &tile_at);
      const bool sel = is_above || (is_at && at_before + run_at + at_rank < need);
      const uint32_t sel_rank = block_flag_scan(sel, scratch, &tile_sel);
      const uint32_t out = sel_before + run_sel + sel_rank;
      if (sel && out < M) {
        const uint64_t lu = (uint64_t)(~key);
        dsmem_st_u64(sk0 + 8u * out, (lu << 32) | (slo + i));
      }
      run_at += tile_at;
      run_sel += tile_sel;
    }
    cluster_sync();                                 // B4: sort keys and miss list complete

    // -------------------------------------------------------------- P4
    if (r == 0) {
      const uint32_t P = a.sort_len;
      for (uint32_t i = M + tid; i < P; i += kThreads) sortkeys[i] = ~0ull;
      __syncthreads();
      uint32_t Pn = 1;
      while (Pn < M && Pn < P) Pn <<= 1;            // sort only the used power of two
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
        const uint32_t v = (uint32_t)(sortkeys[i] & 0xffffffffu);
        const int32_t p = miss_pos[i];
        const uint32_t j = (uint32_t)miss_j[i];
        if (v >= L.hot_rows || j >= k || p < 0 || (uint32_t)p >= L.history_cap) {
          atomicOr(a.status, kFlagInternal);         // cannot happen; never write out of bounds
          continue;
        }
        const int32_t old = L.slot2pos[v];
        if (old >= 0) {
          L.pos2slot[old] = -1;
          ++nevict;
        }
        L.pos2slot[p] = (int32_t)v;
        L.slot2pos[v] = p;
        L.last_use[v] = t;
        const uint32_t owner = j / a.kchunk;
        dsmem_st_u32(dsmem_addr(&meta_fill[j - owner * a.kchunk], owner), v);
        if (L.evlog) {
          L.evlog[1 + 3 * i] = (int32_t)v;
          L.evlog[2 + 3 * i] = old;
          L.evlog[3 + 3 * i] = p;
        }
      }
      if (L.evlog && tid == 0) L.evlog[0] = (int32_t)M;
    }
    cluster_sync();                                 // B5: fills known to their owners
  } else if (L.evlog && r == 0 && tid == 0) {
    L.evlog[0] = 0;
  }

  // ---------------------------------------------------------------- P5
  const uint4* hot4 = reinterpret_cast<const uint4*>(L.hot);
  const uint4* hist4 = reinterpret_cast<const uint4*>(L.hist);
  for (uint32_t jj = warp; jj < jcnt; jj += kWarps) {
    const uint32_t j = jlo + jj;
    const int32_t slot = meta_slot[jj];
    const int32_t fill = meta_fill[jj];
    const uint4* src = nullptr;
    if (slot >= 0) src = hot4 + (size_t)slot * kRowVec;
    else if (slot == kSlotMiss) src = hist4 + (size_t)meta_pos[jj] * kRowVec;
    uint4 va = make_uint4(0, 0, 0, 0), vb = make_uint4(0, 0, 0, 0);
    if (src) {
      va = src[lane];
      if (lane < kRowVec - 32) vb = src[32 + lane];
    }
    if (a.out_rows) {
      uint4* d = reinterpret_cast<uint4*>(a.out_rows) + (size_t)j * kRowVec;
      d[lane] = va;
      if (lane < kRowVec - 32) d[32 + lane] = vb;
    }
    if (fill >= 0) {
      uint4* d = reinterpret_cast<uint4*>(L.hot) + (size_t)fill * kRowVec;
      d[lane] = va;
      if (lane < kRowVec - 32) d[32 + lane] = vb;
    }
    if (a.out_bf16) {
      // lane 0's second piece holds the 8 fp16 scales; latent piece `lane`
      // (16 bytes) lies in group lane / 4.
      const uint32_t s01 = __shfl_sync(0xffffffffu, vb.x, 0);
      const uint32_t s23 = __shfl_sync(0xffffffffu, vb.y, 0);
      const uint32_t s45 = __shfl_sync(0xffffffffu, vb.z, 0);
      const uint32_t s67 = __shfl_sync(0xffffffffu, vb.w, 0);
      const uint32_t g = lane >> 2;
      const uint32_t w = g < 2 ? s01 : g < 4 ? s23 : g < 6 ? s45 : s67;
      const uint16_t hb = (uint16_t)((g & 1) ? (w >> 16) : (w & 0xffffu));
      const float s = __half2float(__ushort_as_half(hb));
      float f[16];
      dequant16(va.x, s, f);
      dequant16(va.y, s, f + 4);
      dequant16(va.z, s, f + 8);
      dequant16(va.w, s, f + 12);
      uint4* d = reinterpret_cast<uint4*>(a.out_bf16 + (size_t)j * KVO_DEQUANT_VALUES);
      d[2 * lane] = make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]), pack2(f[6], f[7]));
      d[2 * lane + 1] =
          make_uint4(pack2(f[8], f[9]), pack2(f[10], f[11]), pack2(f[12], f[13]), pack2(f[14], f[15]));
      if (lane >= 1 && lane < kRowVec - 32) d[64 + (lane - 1)] = vb;   // RoPE, copied
    }
  }

  // ------------------------------------------------------------- stats
  nhit = block_sum(nhit, scratch);
  nmiss = block_sum(nmiss, scratch);
  ninv = block_sum(ninv, scratch);
  if (r == 0) nevict = block_sum(nevict, scratch);
  if (tid == 0) {
    unsigned long long* st = L.stats;
    if (nhit) atomicAdd(st + 1, (unsigned long long)nhit);
    if (nmiss) {
      atomicAdd(st + 2, (unsigned long long)nmiss);
      atomicAdd(st + 6, (unsigned long long)nmiss * KVO_ROW_BYTES);
    }
    if (ninv) {
      atomicAdd(st + 5, (unsigned long long)ninv);
      atomicOr(a.status, kFlagRange);
    }
    if (r == 0) {
      atomicAdd(st + 0, 1ull);
      atomicAdd(st + 3, (unsigned long long)M);
      atomicAdd(st + 4, (unsigned long long)nevict);
      atomicAdd(st + 7, (unsigned long long)k);
    }
  }
}

struct ResolveConfig {
  bool init = false;
  int cluster = 0;
};
ResolveConfig g_resolve[64];

constexpr size_t kResolveMaxDynSmem = 200 * 1024;

}  // namespace

cudaError_t launch_resolve(const LayerView& L, const int32_t* idx, uint32_t k, uint8_t* out_rows,
                           uint16_t* out_bf16, uint32_t* status, int max_cluster,
                           cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  ResolveConfig& cfg = g_resolve[dev & 63];
  if (!cfg.init) {
    e = cudaFuncSetAttribute(resolve_gather_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kResolveMaxDynSmem);
    if (e != cudaSuccess) return e;
    cfg.cluster = best_cluster((const void*)resolve_gather_kernel, kResolveMaxDynSmem, 16);
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
  a.kchunk = (k + C - 1) / C;
  a.hchunk = ((L.hot_rows + C - 1) / C + 3u) & ~3u;
  a.sort_len = 1;
  while (a.sort_len < k) a.sort_len <<= 1;
  const SmemLayout lay = smem_layout(k, a.kchunk, a.hchunk, a.sort_len);
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
  return cudaLaunchKernelEx(&lc, resolve_gather_kernel, a);
}

}  // namespace kvo
