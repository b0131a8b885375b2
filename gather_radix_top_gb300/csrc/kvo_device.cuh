// Device-side building blocks shared by the kvo kernels: thread-block-cluster
// barriers and distributed shared memory (inline PTX), block-wide scans, and
// the cluster-wide radix select + ordered compaction used by both the top-K
// selection and the LRU victim choice.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace kvo {

constexpr int kThreads = 1024;          // threads per CTA of the cluster kernels
constexpr int kWarps = kThreads / 32;
constexpr uint32_t kMaxCluster = 16;

// Device status word bits (returned by kvo_sync).
constexpr uint32_t kFlagRange = 1u;
constexpr uint32_t kFlagInternal = 2u;  // an internal consistency check failed
constexpr uint32_t kFlagTimeout = 4u;   // a bounded device-side wait gave up
constexpr uint32_t kFlagInflight = 8u;  // and its second wait too: a bulk copy may still be in flight into the
                                        // shared memory of a CTA that has exited

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

// The two halves of cluster_sync, so that a thread can work between its
// arrival and its wait (each arrive must be followed by a wait before the
// next arrive).
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
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

__device__ __forceinline__ uint4 dsmem_ld_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ void dsmem_st_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void dsmem_st_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void dsmem_st_u64(uint32_t addr, uint64_t v) {
  asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}

__device__ __forceinline__ void dsmem_red_add_u32(uint32_t addr, uint32_t v) {
  asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void dsmem_red_or_u32(uint32_t addr, uint32_t v) {
  asm volatile("red.shared::cluster.or.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// ------------------------------------------------- bulk copies (TMA engine)
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Arrives on `bar` and tells it to expect `bytes` more from bulk copies.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned)
// from global to this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits for phase `parity` of `bar` to complete; gives up after `max_polls`
// polls (about 64 ns apart) and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint32_t max_polls) {
  for (uint32_t i = 0; i < max_polls; ++i) {
    if (mbar_test(bar, parity)) return true;
    __nanosleep(64);
  }
  return false;
}

// Bulk copy of `bytes` (a multiple of 16; 16-byte aligned) from this CTA's
// shared memory to global memory, in the calling thread's bulk async-group.
__device__ __forceinline__ void bulk_copy_s2g(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until the calling thread's bulk stores have completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Orders this thread's earlier generic shared-memory writes before later
// bulk copies that read them.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Brings the line holding `p` into L2 without waiting for it.
__device__ __forceinline__ void prefetch_l2(const void* p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }


// Each CTA publishes `nval` (<= 4) values; afterwards every CTA reads every
// CTA's values from its own shared memory (table[rank][i]).  Contains one
// cluster barrier; `table` must not be written again before the next one.
__device__ __forceinline__ void cluster_publish(const uint32_t* vals, uint32_t nval, uint32_t (*table)[4],
                                                uint32_t rank, uint32_t nrank) {
  const uint32_t tid = threadIdx.x;
  if (tid < nrank * nval) {
    const uint32_t dst = tid / nval, i = tid % nval;
    dsmem_st_u32(dsmem_addr(&table[rank][i], dst), vals[i]);
  }
  cluster_sync();
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

// Exclusive prefix sum of a per-thread value over the CTA in thread order;
// *total gets the CTA's sum.  `scratch` holds kWarps + 1 words.  Two
// __syncthreads; scratch is reusable afterwards.
__device__ __forceinline__ uint32_t block_excl_sum(uint32_t v, uint32_t* scratch, uint32_t* total) {
  const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t o = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= (uint32_t)d) incl += o;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  uint32_t before = lane < warp ? scratch[lane] : 0u;
  uint32_t all = lane < (uint32_t)kWarps ? scratch[lane] : 0u;
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) {
    before += __shfl_xor_sync(0xffffffffu, before, d);
    all += __shfl_xor_sync(0xffffffffu, all, d);
  }
  __syncthreads();
  *total = all;
  return before + incl - v;
}

// Sum of a per-thread value over the CTA (result valid in every thread).
// `scratch` holds kWarps + 1 words.
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

// Sums of two per-thread values over the CTA, returned in every thread.
// `scratch` holds 2 * kWarps words.
__device__ __forceinline__ void block_sum2(uint32_t a, uint32_t b, uint32_t* scratch, uint32_t* sa,
                                           uint32_t* sb) {
  static_assert(kWarps <= 32, "one lane per warp of the CTA");
  const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, d);
    b += __shfl_xor_sync(0xffffffffu, b, d);
  }
  if (lane == 0) {
    scratch[2 * warp] = a;
    scratch[2 * warp + 1] = b;
  }
  __syncthreads();
  a = lane < (uint32_t)kWarps ? scratch[2 * lane] : 0u;
  b = lane < (uint32_t)kWarps ? scratch[2 * lane + 1] : 0u;
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, d);
    b += __shfl_xor_sync(0xffffffffu, b, d);
  }
  __syncthreads();
  *sa = a;
  *sb = b;
}

// ----------------------------------------------------- cluster radix select
// Outcome of selecting the `want` largest keys over the cluster: the selected
// keys are those whose bits above `shift` exceed those of `prefix`, plus the
// first `need` keys (in index order) whose bits above `shift` equal them.
// When the last examined bucket is taken whole, `need` equals its count.
struct RadixCut {
  uint32_t prefix;
  uint32_t shift;
  uint32_t need;
};

constexpr int kDigitBits = 8;                    // 256-bin digits (wider ones cost more in DSMEM traffic)
constexpr uint32_t kBins = 1u << kDigitBits;
constexpr uint32_t kBinsPerThread = kBins >= (uint32_t)kThreads ? kBins / kThreads : 1u;
constexpr uint32_t kScanThreads = kBins / kBinsPerThread;   // threads taking part in the bin scan
static_assert(kScanThreads % 32 == 0 && kScanThreads <= (uint32_t)kThreads, "whole warps scan the bins");

struct __align__(16) RadixSmem {
  uint32_t hist[kBins];             // this CTA's histogram of the current pass
  uint32_t total[3][kBins];         // cluster-wide counts of the bins this CTA owns (pass mod 3)
  uint32_t gath[kBins];             // every bin's cluster-wide count, read back from the owners
  uint32_t warp_sum[kWarps];        // block scan of the cluster-wide histogram
  uint32_t cut[4];                  // bucket, count above it, bucket count
};

// Zeroes the cluster-wide histograms.  A cluster barrier must separate this
// from the first cluster_radix_select of any CTA.
__device__ __forceinline__ void radix_smem_init(RadixSmem* sm) {
  for (uint32_t b = threadIdx.x; b < 3 * kBins; b += kThreads) (&sm->total[0][0])[b] = 0;
}

// Adds one to bin[e] for each of this lane's four keys whose bit e of vmask
// is set.  A warp whose valid keys all share one bin (equal or nearly equal
// keys) adds their count once; otherwise every key adds on its own: the
// shared-memory atomics resolve the few colliding lanes faster than a match
// over the warp would (3.4x on a 1M-key histogram pass).  Every lane of the
// warp must call it.
__device__ __forceinline__ void hist_add_warp4(uint32_t* h, const uint32_t (&bin)[4], uint32_t vmask) {
  const uint32_t b0 = __shfl_sync(0xffffffffu, bin[0], 0);
  bool same = true;
#pragma unroll
  for (int e = 0; e < 4; ++e) same &= !((vmask >> e) & 1u) || bin[e] == b0;
  if (__all_sync(0xffffffffu, same)) {
    const uint32_t c = __reduce_add_sync(0xffffffffu, (uint32_t)__popc(vmask));
    if ((threadIdx.x & 31) == 0 && c) atomicAdd(&h[b0], c);
  } else {
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if ((vmask >> e) & 1u) atomicAdd(&h[bin[e]], 1u);
  }
}

// A CTA's keys are read four at a time: key4(g) returns keys 4g..4g+3.
// Entries at or beyond `count` are ignored, but key4 must be safe to call for
// every g < ceil(count / 4).
//
// cluster_radix_select finds the cut.  Keys are below 2^key_bits (1..32), so
// only significant digits are examined: digits of up to 11 bits, most
// significant first.  Every CTA of the cluster must call it with the same
// `want` and `key_bits`, and `want` must not exceed the cluster's key count.
// Each pass: a shared-memory histogram; every nonzero bin added into the
// one CTA that owns it (CTA b / (kBins / nrank) for bin b); one cluster
// barrier; every CTA reads all bins back from their owners (one remote load
// per bin) and scans them from the largest digit down, so that every CTA
// finds the same bucket.  Sending each bin to its owner only, rather than
// into every CTA, cuts a spread-out pass's remote adds from 16 x 256 to 256
// per CTA (second pass of a 50K selection: 1.9 -> 0.3 us, for 0.37 us of
// read-back in every pass).  The owners' counts rotate
// over three buffers: a buffer is zeroed two passes after it was read, with
// a cluster barrier in between.
template <typename Key4>
__device__ RadixCut cluster_radix_select(Key4 key4, uint32_t count, uint32_t want, uint32_t key_bits,
                                         RadixSmem* sm, uint32_t nrank) {
  uint32_t prefix = 0, mask = 0, remaining = want;
  uint32_t shift = key_bits;
  const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t ngroups = (count + 3) / 4;
  for (int pass = 0;; ++pass) {
    const uint32_t d = shift < (uint32_t)kDigitBits ? shift : (uint32_t)kDigitBits;
    shift -= d;
    const uint32_t dmask = (1u << d) - 1u;
    uint32_t* tot = sm->total[pass % 3];
    for (uint32_t b = tid; b < kBins; b += kThreads) {
      sm->hist[b] = 0;
      sm->total[(pass + 1) % 3][b] = 0;     // added into by the next pass, after the barrier below
    }
    __syncthreads();
    for (uint32_t g0 = 0; g0 < ngroups; g0 += kThreads) {
      const uint32_t g = g0 + tid;
      const uint4 kk = g < ngroups ? key4(g) : make_uint4(0, 0, 0, 0);
      const uint32_t kv[4] = {kk.x, kk.y, kk.z, kk.w};
      uint32_t bins[4], vm = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        bins[e] = (kv[e] >> shift) & dmask;
        vm |= (uint32_t)(g < ngroups && 4 * g + e < count && (kv[e] & mask) == prefix) << e;
      }
      hist_add_warp4(sm->hist, bins, vm);
    }
    __syncthreads();
    const uint32_t per_owner = (kBins + nrank - 1) / nrank;   // bins per owning CTA (the last may own fewer)
    for (uint32_t b = tid; b <= dmask; b += kThreads) {
      const uint32_t v = sm->hist[b];
      if (v) dsmem_red_add_u32(dsmem_addr(&tot[b], b / per_owner), v);
    }
    cluster_sync();
    for (uint32_t b = tid; b < kBins; b += kThreads)
      sm->gath[b] = b <= dmask ? dsmem_ld_u32(dsmem_addr(&tot[b], b / per_owner)) : 0u;
    __syncthreads();
    // block scan from the largest digit down: thread t holds bins
    // kBins-1-2t and kBins-2-2t (bins above dmask are zero)
    const bool scans = tid < kScanThreads;
    uint32_t c[kBinsPerThread], sum = 0;
#pragma unroll
    for (uint32_t e = 0; e < kBinsPerThread; ++e) {
      c[e] = scans ? sm->gath[kBins - 1 - kBinsPerThread * tid - e] : 0u;
      sum += c[e];
    }
    uint32_t incl = sum;
#pragma unroll
    for (int dd = 1; dd < 32; dd <<= 1) {
      const uint32_t o = __shfl_up_sync(0xffffffffu, incl, dd);
      if (lane >= (uint32_t)dd) incl += o;
    }
    if (lane == 31) sm->warp_sum[warp] = incl;
    __syncthreads();
    uint32_t before = lane < warp ? sm->warp_sum[lane] : 0u;
#pragma unroll
    for (int dd = 16; dd > 0; dd >>= 1) before += __shfl_xor_sync(0xffffffffu, before, dd);
    const uint32_t excl = before + incl - sum;
    if (scans && excl < remaining && remaining <= excl + sum) {
      uint32_t above = excl;
#pragma unroll
      for (uint32_t e = 0; e < kBinsPerThread; ++e) {
        if (above + c[e] >= remaining) {
          sm->cut[0] = kBins - 1 - kBinsPerThread * tid - e;
          sm->cut[1] = above;
          sm->cut[2] = c[e];
          break;
        }
        above += c[e];
      }
    }
    __syncthreads();
    const uint32_t bucket = sm->cut[0], above = sm->cut[1], inbucket = sm->cut[2];
    remaining -= above;
    prefix |= bucket << shift;
    mask |= dmask << shift;
    if (remaining == inbucket || shift == 0) break;   // the whole bucket is selected, or keys are exhausted
  }
  return RadixCut{prefix, shift, remaining};
}

// This CTA's keys above and at the cut (one pass over the keys).
template <typename Key4>
__device__ void cut_counts(Key4 key4, uint32_t count, const RadixCut& cut, uint32_t* scratch, uint32_t* above,
                           uint32_t* at) {
  const uint32_t top = cut.prefix >> cut.shift;
  uint32_t a = 0, e = 0;
  for (uint32_t g = threadIdx.x; g < (count + 3) / 4; g += kThreads) {
    const uint4 kk = key4(g);
    const uint32_t kv[4] = {kk.x, kk.y, kk.z, kk.w};
#pragma unroll
    for (uint32_t q = 0; q < 4; ++q) {
      if (4 * g + q < count) {
        const uint32_t v = kv[q] >> cut.shift;
        a += v > top;
        e += v == top;
      }
    }
  }
  block_sum2(a, e, scratch, above, at);
}

// Selected-before and at-cut-before counts of CTA `rank`, from every CTA's
// published (above, at) counts in columns col, col+1 and the cut's `need`.
__device__ __forceinline__ void cut_offsets(const uint32_t (*table)[4], uint32_t col, uint32_t rank,
                                            uint32_t need, uint32_t* sel_before, uint32_t* at_before) {
  uint32_t s = 0, e = 0;
  for (uint32_t q = 0; q < rank; ++q) {
    const uint32_t a = table[q][col], c = table[q][col + 1];
    const uint32_t left = need > e ? need - e : 0u;
    s += a + (c < left ? c : left);
    e += c;
  }
  *sel_before = s;
  *at_before = e;
}

// Ordered compaction after a cut: visits this CTA's keys in index order and
// calls emit(i, out) for each selected key i, with `out` its index in the
// cluster-wide selection.  sel_before / at_before: selected and at-cut keys
// of lower-ranked CTAs.  Four keys per thread per tile; one block barrier per
// tile (the two scratch buffers alternate).
template <typename Key4, typename Emit>
__device__ void cluster_compact(Key4 key4, uint32_t count, const RadixCut& cut, uint32_t sel_before,
                                uint32_t at_before, uint32_t (*scratch)[2 * kWarps + 2], Emit emit) {
  static_assert(kWarps <= 32, "one lane per warp of the CTA");
  const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t ngroups = (count + 3) / 4;
  const uint32_t shift = cut.shift, top = cut.prefix >> shift, need = cut.need;
  uint32_t run_sel = 0, run_at = 0, parity = 0;
  for (uint32_t g0 = 0; g0 < ngroups; g0 += kThreads, parity ^= 1u) {
    const uint32_t g = g0 + tid;
    const uint4 kk = g < ngroups ? key4(g) : make_uint4(0, 0, 0, 0);
    const uint32_t kv[4] = {kk.x, kk.y, kk.z, kk.w};
    uint32_t amask = 0, emask = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (g < ngroups && 4 * g + e < count) {
        const uint32_t v = kv[e] >> shift;
        amask |= (uint32_t)(v > top) << e;
        emask |= (uint32_t)(v == top) << e;
      }
    }
    const uint32_t a = __popc(amask), e_ = __popc(emask);
    uint32_t a_incl = a, e_incl = e_;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint32_t oa = __shfl_up_sync(0xffffffffu, a_incl, d);
      const uint32_t oe = __shfl_up_sync(0xffffffffu, e_incl, d);
      if (lane >= (uint32_t)d) {
        a_incl += oa;
        e_incl += oe;
      }
    }
    uint32_t* sc = scratch[parity];
    if (lane == 31) {
      sc[2 * warp] = a_incl;
      sc[2 * warp + 1] = e_incl;
    }
    __syncthreads();
    const uint32_t used = at_before + run_at;
    const uint32_t left = need > used ? need - used : 0u;   // at-cut keys still to take
    // lane l works on warp l's totals
    const uint32_t A_l = lane < (uint32_t)kWarps ? sc[2 * lane] : 0u;
    const uint32_t E_l = lane < (uint32_t)kWarps ? sc[2 * lane + 1] : 0u;
    uint32_t E_incl = E_l;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint32_t o = __shfl_up_sync(0xffffffffu, E_incl, d);
      if (lane >= (uint32_t)d) E_incl += o;
    }
    const uint32_t E_excl = E_incl - E_l;
    const uint32_t left_l = left > E_excl ? left - E_excl : 0u;
    const uint32_t S_l = A_l + (E_l < left_l ? E_l : left_l);
    uint32_t S_incl = S_l;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint32_t o = __shfl_up_sync(0xffffffffu, S_incl, d);
      if (lane >= (uint32_t)d) S_incl += o;
    }
    const uint32_t Eoff = __shfl_sync(0xffffffffu, E_excl, warp);
    const uint32_t Soff = __shfl_sync(0xffffffffu, S_incl - S_l, warp);
    const uint32_t tile_at = __shfl_sync(0xffffffffu, E_incl, 31);
    const uint32_t tile_sel = __shfl_sync(0xffffffffu, S_incl, 31);
    const uint32_t e_before = Eoff + e_incl - e_;
    uint32_t take_at = left > e_before ? left - e_before : 0u;
    take_at = take_at < e_ ? take_at : e_;
    const uint32_t s = a + take_at;
    uint32_t s_incl = s;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint32_t o = __shfl_up_sync(0xffffffffu, s_incl, d);
      if (lane >= (uint32_t)d) s_incl += o;
    }
    uint32_t out = sel_before + run_sel + Soff + s_incl - s;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if ((amask >> e) & 1u) {
        emit(4 * g + e, out++);
      } else if (((emask >> e) & 1u) && take_at) {
        emit(4 * g + e, out++);
        --take_at;
      }
    }
    run_sel += tile_sel;
    run_at += tile_at;
  }
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
