// Device-side building blocks shared by the kvo kernels: thread-block-cluster
// barriers and distributed shared memory (inline PTX), block-wide scans, and
// the cluster-wide radix select used by both the top-K selection and the LRU
// victim choice.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace kvo {

constexpr int kThreads = 1024;          // threads per CTA of the cluster kernels
constexpr int kWarps = kThreads / 32;
constexpr int kRadixBins = 256;         // 8-bit digits, most significant first

// Device status word bits (returned by kvo_sync).
constexpr uint32_t kFlagRange = 1u;
constexpr uint32_t kFlagInternal = 2u;      // an internal consistency check failed

// ---------------------------------------------------------------- cluster
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

// Full cluster barrier with release/acquire semantics at cluster scope: every
// shared, distributed-shared and global write made by any thread of the
// cluster before it is visible to every thread of the cluster after it.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// Address of the same shared variable in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t dsmem_addr(const void* local, uint32_t rank) {
  uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local));
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}

__device__ __forceinline__ uint32_t dsmem_ld_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ void dsmem_st_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void dsmem_st_u64(uint32_t addr, uint64_t v) {
  asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}

// ------------------------------------------------------------------ scans
// Exclusive prefix count of a per-thread flag over the CTA in thread order.
// `scratch` holds kWarps + 1 words.  Returns the thread's prefix; *total gets
// the CTA's count.  Contains two __syncthreads and leaves scratch reusable.
__device__ __forceinline__ uint32_t block_flag_scan(bool flag, uint32_t* scratch, uint32_t* total) {
  const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t ballot = __ballot_sync(0xffffffffu, flag);
  const uint32_t before = __popc(ballot & ((1u << lane) - 1u));
  if (lane == 0) scratch[warp] = __popc(ballot);
  __syncthreads();
  if (warp == 0) {
    uint32_t v = lane < kWarps ? scratch[lane] : 0u;
    uint32_t incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      uint32_t o = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= (uint32_t)d) incl += o;
    }
    if (lane < kWarps) scratch[lane] = incl - v;
    if (lane == 31) scratch[kWarps] = incl;
  }
  __syncthreads();
  const uint32_t r = scratch[warp] + before;
  *total = scratch[kWarps];
  __syncthreads();
  return r;
}

// Sum of a per-thread value over the CTA (result valid in every thread).
__device__ __forceinline__ uint32_t block_sum(uint32_t v, uint32_t* scratch) {
  const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = lane < kWarps ? scratch[lane] : 0u;
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) w += __shfl_xor_sync(0xffffffffu, w, d);
    if (lane == 0) scratch[kWarps] = w;
  }
  __syncthreads();
  const uint32_t r = scratch[kWarps];
  __syncthreads();
  return r;
}

// ----------------------------------------------------- cluster radix select
// Outcome of selecting the `want` largest 32-bit keys over the cluster: the
// selected keys are those whose top (32 - shift) bits exceed those of
// `prefix`, plus the first `need` keys (in index order) whose top bits equal
// them.  When the last examined bucket is taken whole, `need` equals its
// count.
struct RadixCut {
  uint32_t prefix;
  uint32_t shift;
  uint32_t need;
};

struct RadixSmem {
  uint32_t hist[2][kRadixBins];   // this CTA's histograms (double-buffered)
  uint32_t total[kRadixBins];     // cluster-wide histogram of the current pass
  uint32_t cut[4];                // bucket, count above it, bucket count
};

// Finds the cut.  `key_at(i)` returns this CTA's i-th key for i < count.
// Every CTA of the cluster must call it with the same `want`, and `want` must
// not exceed the cluster's key count.  One cluster barrier per digit pass.
template <typename KeyAt>
__device__ RadixCut cluster_radix_select(KeyAt key_at, uint32_t count, uint32_t want,
                                         RadixSmem* sm, uint32_t nrank) {
  uint32_t prefix = 0, mask = 0, remaining = want;
  uint32_t shift = 32;
  const uint32_t tid = threadIdx.x, lane = tid & 31;
  for (int pass = 0; pass < 4; ++pass) {
    shift -= 8;
    uint32_t* h = sm->hist[pass & 1];
    for (uint32_t b = tid; b < kRadixBins; b += kThreads) h[b] = 0;
    __syncthreads();
    for (uint32_t i = tid; i < count; i += kThreads) {
      const uint32_t key = key_at(i);
      if ((key & mask) == prefix) atomicAdd(&h[(key >> shift) & 0xffu], 1u);
    }
    cluster_sync();
    if (tid < kRadixBins) {
      uint32_t s = 0;
      for (uint32_t r = 0; r < nrank; ++r) s += dsmem_ld_u32(dsmem_addr(&h[tid], r));
      sm->total[tid] = s;
    }
    __syncthreads();
    if (tid < 32) {
      // lane l covers bins 255-8l down to 248-8l (largest digits first)
      uint32_t c[8], sum = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        c[e] = sm->total[255 - 8 * lane - e];
        sum += c[e];
      }
      uint32_t incl = sum;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        uint32_t o = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= (uint32_t)d) incl += o;
      }
      const uint32_t excl = incl - sum;
      if (excl < remaining && remaining <= incl) {
        uint32_t above = excl;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          if (above + c[e] >= remaining) {
            sm->cut[0] = 255 - 8 * lane - e;
            sm->cut[1] = above;
            sm->cut[2] = c[e];
            break;
          }
          above += c[e];
        }
      }
    }
    __syncthreads();
    const uint32_t bucket = sm->cut[0], above = sm->cut[1], inbucket = sm->cut[2];
    __syncthreads();
    remaining -= above;
    prefix |= bucket << shift;
    mask |= 0xffu << shift;
    if (remaining == inbucket) break;   // the whole bucket is selected
  }
  return RadixCut{prefix, shift, remaining};
}

// ------------------------------------------------------------------ keys
// Order-preserving map of an fp32 score to a uint32 (larger score -> larger
// key).  -0.0 maps like +0.0; every NaN maps to 0, below -inf.
__device__ __forceinline__ uint32_t score_key(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0u;
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

}  // namespace kvo
