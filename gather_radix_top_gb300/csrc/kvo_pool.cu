// Session block store/restore between an HBM block pool and a pinned host
// tier.
//
// "A 60k-token context comes back off disk in 17 seconds instead of 65
// seconds of prefill" (vllm-bounded-fs-kv-tier README): KV lives in
// fixed-size blocks of a GPU pool, whole sessions are stored to a tier and
// restored, a restore is admitted only when every group can be placed, the
// tier holds bytes // block_bytes blocks, and the pool's free queue hands out
// blocks from its front and takes freed blocks at its back.
// "Making KV offload correct": a grouped allocation is a transaction (reserve
// every group, then commit; a failure undoes every earlier mutation), and a
// block is released only after the copies that depend on it have finished.
//
// The allocators and session tables live on the host; the bytes move in one
// kernel launch per call (a plan of (source block, destination block) pairs,
// each block copied with 16-byte loads and stores by one CTA; tier blocks are
// reached through the device mapping of the pinned host memory).
#include <cstdint>
#include <cstring>
#include <deque>
#include <map>
#include <new>
#include <vector>

#include "kvo.h"
#include "kvo_internal.h"

namespace {

struct Session {
  int64_t tokens = 0;
  std::vector<std::vector<int32_t>> pool;   // per layer, when resident in the pool
  std::vector<std::vector<int32_t>> tier;   // per layer, when stored in the tier
  int busy = 0;                             // copies in flight that touch its blocks
};

struct Pending {
  cudaEvent_t done = nullptr;
  std::vector<int32_t> sessions;
  std::vector<int32_t> tier_free;           // tier blocks to give back once done
};

struct Allocator {
  std::deque<int32_t> free;
  int64_t fail_after = -1;                  // the n-th allocation from arming fails

  explicit Allocator(int64_t n = 0) {
    for (int64_t i = 0; i < n; ++i) free.push_back((int32_t)i);
  }

  void give_front(const std::vector<int32_t>& b) {
    for (auto it = b.rbegin(); it != b.rend(); ++it) free.push_front(*it);
  }
  void give_back(const std::vector<int32_t>& b) { free.insert(free.end(), b.begin(), b.end()); }

  bool take(size_t n, std::vector<int32_t>* out) {
    out->clear();
    for (size_t i = 0; i < n; ++i) {
      if (fail_after == 0 || free.empty()) {
        if (fail_after == 0) fail_after = -1;
        give_front(*out);
        out->clear();
        return false;
      }
      if (fail_after > 0) --fail_after;
      out->push_back(free.front());
      free.pop_front();
    }
    return true;
  }

  // every group's blocks, or none: earlier groups go back front first
  bool take_groups(const std::vector<size_t>& sizes, std::vector<std::vector<int32_t>>* out) {
    out->clear();
    for (size_t n : sizes) {
      std::vector<int32_t> g;
      if (!take(n, &g)) {
        for (auto it = out->rbegin(); it != out->rend(); ++it) give_front(*it);
        out->clear();
        return false;
      }
      out->push_back(std::move(g));
    }
    return true;
  }
};

// One CTA per (source block, destination block) pair at a time; each thread
// keeps four 16-byte loads in flight before it stores them.
__global__ void block_copy_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                  const int2* __restrict__ plan, int64_t n, uint32_t block_vec) {
  for (int64_t i = blockIdx.x; i < n; i += gridDim.x) {
    const int2 pr = plan[i];
    const uint4* s = src + (size_t)pr.x * block_vec;
    uint4* d = dst + (size_t)pr.y * block_vec;
    for (uint32_t v0 = threadIdx.x; v0 < block_vec; v0 += 4 * blockDim.x) {
      uint4 r[4];
#pragma unroll
      for (uint32_t u = 0; u < 4; ++u) {
        const uint32_t v = v0 + u * blockDim.x;
        if (v < block_vec) r[u] = s[v];
      }
#pragma unroll
      for (uint32_t u = 0; u < 4; ++u) {
        const uint32_t v = v0 + u * blockDim.x;
        if (v < block_vec) d[v] = r[u];
      }
    }
  }
}

// rows[t - first] <-> block tbl[t / bt] row t % bt, for t in [first, first+n);
// one warp per row; to_pool selects the direction.
__global__ void rows_kernel(uint4* __restrict__ pool, uint4* __restrict__ rows, const int32_t* __restrict__ tbl,
                            int64_t first, int64_t n, int32_t bt, bool to_pool) {
  constexpr uint32_t kVec = KVO_ROW_BYTES / 16;
  const uint32_t lane = threadIdx.x & 31;
  const int64_t w0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t i = w0; i < n; i += nw) {
    const int64_t t = first + i;
    uint4* p = pool + ((size_t)tbl[t / bt] * bt + (size_t)(t % bt)) * kVec;
    uint4* r = rows + (size_t)i * kVec;
    for (uint32_t v = lane; v < kVec; v += 32) {
      if (to_pool) p[v] = r[v];
      else r[v] = p[v];
    }
  }
}

__global__ void fill_kernel(uint4* __restrict__ p, size_t nvec, uint32_t word) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += stride)
    p[i] = make_uint4(word, word, word, word);
}

bool ok(cudaError_t e) { return e == cudaSuccess; }

// Device memory, or pinned host memory mapped into the device's address space.
bool device_accessible(const void* ptr) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, ptr) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) return true;
  return at.type == cudaMemoryTypeHost && at.devicePointer == ptr;
}

int sm_count() {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms > 0 ? sms : 1;
}

}  // namespace

struct kvo_pool {
  int32_t layers = 0, block_tokens = 0;
  int64_t pool_blocks = 0, tier_blocks = 0;
  size_t block_bytes = 0;
  uint8_t* pool = nullptr;        // device
  uint8_t* tier_host = nullptr;   // pinned, mapped
  uint8_t* tier_dev = nullptr;    // device address of tier_host
  Allocator pool_alloc, tier_alloc;
  std::map<int32_t, Session> sessions;
  std::vector<Pending> pending;
  int2* plan_host = nullptr;      // pinned staging for copy plans
  int2* plan_dev = nullptr;
  size_t plan_cap = 0;            // int2 entries
  cudaEvent_t plan_uploaded = nullptr;   // the last plan has left plan_host
  cudaEvent_t plan_consumed = nullptr;   // the last kernel that read plan_dev is done
  kvo_pool_stats stats = {};
};

namespace {

// Completed copies: sessions are no longer busy, tier blocks go back.
void reap(kvo_pool* p, bool wait) {
  std::vector<Pending> keep;
  for (Pending& q : p->pending) {
    if (wait) cudaEventSynchronize(q.done);
    if (cudaEventQuery(q.done) == cudaSuccess) {
      for (int32_t sid : q.sessions) {
        auto it = p->sessions.find(sid);
        if (it != p->sessions.end() && it->second.busy > 0) --it->second.busy;
      }
      p->tier_alloc.give_back(q.tier_free);
      cudaEventDestroy(q.done);
    } else {
      cudaGetLastError();
      keep.push_back(std::move(q));
    }
  }
  p->pending.swap(keep);
}

// Uploads `plan` (n entries of plan_host) to plan_dev in stream order.
cudaError_t upload_plan(kvo_pool* p, size_t n, cudaStream_t s) {
  cudaError_t e = cudaStreamWaitEvent(s, p->plan_consumed, 0);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyAsync(p->plan_dev, p->plan_host, n * sizeof(int2), cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return e;
  return cudaEventRecord(p->plan_uploaded, s);
}

// Host may write plan_host again once the previous upload has left it.
cudaError_t plan_host_ready(kvo_pool* p) { return cudaEventSynchronize(p->plan_uploaded); }

cudaError_t launch_copy(kvo_pool* p, const uint8_t* src, uint8_t* dst, size_t n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  cudaError_t e = upload_plan(p, n, s);
  if (e != cudaSuccess) return e;
  const int64_t grid = (int64_t)n < (int64_t)sm_count() * 8 ? (int64_t)n : (int64_t)sm_count() * 8;
  block_copy_kernel<<<(unsigned)grid, 256, 0, s>>>(reinterpret_cast<const uint4*>(src), reinterpret_cast<uint4*>(dst),
                                                  p->plan_dev, (int64_t)n, (uint32_t)(p->block_bytes / 16));
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return cudaEventRecord(p->plan_consumed, s);
}

kvo_status track(kvo_pool* p, std::vector<int32_t> sids, std::vector<int32_t> tier_free, cudaStream_t s) {
  Pending q;
  if (!ok(cudaEventCreateWithFlags(&q.done, cudaEventDisableTiming))) return KVO_ECUDA;
  if (!ok(cudaEventRecord(q.done, s))) return KVO_ECUDA;
  for (int32_t sid : sids) ++p->sessions[sid].busy;
  q.sessions = std::move(sids);
  q.tier_free = std::move(tier_free);
  p->pending.push_back(std::move(q));
  return KVO_OK;
}

size_t blocks_per_layer(const kvo_pool* p, int64_t tokens) {
  return (size_t)((tokens + p->block_tokens - 1) / p->block_tokens);
}

void free_pool(kvo_pool* p) {
  if (!p) return;
  reap(p, true);
  cudaFree(p->pool);
  cudaFreeHost(p->tier_host);
  cudaFreeHost(p->plan_host);
  cudaFree(p->plan_dev);
  if (p->plan_uploaded) cudaEventDestroy(p->plan_uploaded);
  if (p->plan_consumed) cudaEventDestroy(p->plan_consumed);
  delete p;
}

}  // namespace

extern "C" {

int64_t kvo_tier_blocks(int64_t tier_bytes, int64_t block_bytes) {
  if (tier_bytes < 0 || block_bytes <= 0) return -1;
  return tier_bytes / block_bytes;
}

kvo_status kvo_pool_create(int32_t layers, int64_t pool_blocks, int32_t block_tokens, int32_t row_bytes,
                           int64_t tier_blocks, kvo_pool** out) {
  if (!out || layers < 1 || pool_blocks < 1 || pool_blocks > INT32_MAX || block_tokens < 1 ||
      row_bytes != KVO_ROW_BYTES || tier_blocks < 0 || tier_blocks > INT32_MAX)
    return KVO_EINVAL;
  kvo_pool* p = new (std::nothrow) kvo_pool;
  if (!p) return KVO_ENOMEM;
  p->layers = layers;
  p->block_tokens = block_tokens;
  p->pool_blocks = pool_blocks;
  p->tier_blocks = tier_blocks;
  p->block_bytes = (size_t)block_tokens * KVO_ROW_BYTES;
  p->pool_alloc = Allocator(pool_blocks);
  p->tier_alloc = Allocator(tier_blocks);
  p->plan_cap = (size_t)(pool_blocks > tier_blocks ? pool_blocks : tier_blocks);
  bool good = ok(cudaMalloc(&p->pool, p->block_bytes * (size_t)pool_blocks)) &&
              ok(cudaMemset(p->pool, 0, p->block_bytes * (size_t)pool_blocks)) &&
              ok(cudaMalloc(&p->plan_dev, sizeof(int2) * p->plan_cap)) &&
              ok(cudaHostAlloc((void**)&p->plan_host, sizeof(int2) * p->plan_cap, cudaHostAllocDefault)) &&
              ok(cudaEventCreateWithFlags(&p->plan_uploaded, cudaEventDisableTiming)) &&
              ok(cudaEventCreateWithFlags(&p->plan_consumed, cudaEventDisableTiming)) &&
              ok(cudaEventRecord(p->plan_uploaded, 0)) && ok(cudaEventRecord(p->plan_consumed, 0));
  if (good && tier_blocks > 0) {
    good = ok(cudaHostAlloc((void**)&p->tier_host, p->block_bytes * (size_t)tier_blocks,
                            cudaHostAllocMapped | cudaHostAllocPortable));
    void* d = nullptr;
    good = good && ok(cudaHostGetDevicePointer(&d, p->tier_host, 0));
    p->tier_dev = static_cast<uint8_t*>(d);
  }
  if (good) good = ok(cudaDeviceSynchronize());
  if (!good) {
    cudaGetLastError();
    free_pool(p);
    return KVO_ENOMEM;
  }
  p->stats.free_blocks = (uint64_t)pool_blocks;
  p->stats.tier_free_blocks = (uint64_t)tier_blocks;
  *out = p;
  return KVO_OK;
}

kvo_status kvo_pool_destroy(kvo_pool* p) {
  if (!p) return KVO_EINVAL;
  const bool synced = ok(cudaDeviceSynchronize());
  free_pool(p);
  return synced ? KVO_OK : KVO_ECUDA;
}

kvo_status kvo_pool_alloc(kvo_pool* p, int32_t session, int64_t tokens) {
  if (!p || tokens < 1 || p->sessions.count(session)) return KVO_EINVAL;
  reap(p, false);
  std::vector<std::vector<int32_t>> got;
  if (!p->pool_alloc.take_groups(std::vector<size_t>(p->layers, blocks_per_layer(p, tokens)), &got)) {
    ++p->stats.rollbacks;
    return KVO_ECAPACITY;
  }
  Session& s = p->sessions[session];
  s.tokens = tokens;
  s.pool = std::move(got);
  return KVO_OK;
}

static kvo_status rows_call(kvo_pool* p, int32_t session, int32_t layer, int64_t first, const void* rows,
                            int64_t n, void* stream, bool to_pool) {
  if (!p || !rows || n < 0 || first < 0 || layer < 0 || layer >= p->layers ||
      (reinterpret_cast<uintptr_t>(rows) & 15u) || !device_accessible(rows))
    return KVO_EINVAL;
  auto it = p->sessions.find(session);
  if (it == p->sessions.end() || it->second.pool.empty() || first + n > it->second.tokens) return KVO_EINVAL;
  if (n == 0) return KVO_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const std::vector<int32_t>& tbl = it->second.pool[layer];
  if (!ok(plan_host_ready(p))) return KVO_ECUDA;
  std::memcpy(p->plan_host, tbl.data(), tbl.size() * sizeof(int32_t));   // the block table, as int32
  if (!ok(upload_plan(p, (tbl.size() + 1) / 2, s))) return KVO_ECUDA;
  int64_t blocks = (n * 32 + 255) / 256;
  const int64_t cap = (int64_t)sm_count() * 8;
  if (blocks > cap) blocks = cap;
  rows_kernel<<<(unsigned)blocks, 256, 0, s>>>(reinterpret_cast<uint4*>(p->pool),
                                                reinterpret_cast<uint4*>(const_cast<void*>(rows)),
                                                reinterpret_cast<const int32_t*>(p->plan_dev), first, n,
                                                p->block_tokens, to_pool);
  if (!ok(cudaGetLastError()) || !ok(cudaEventRecord(p->plan_consumed, s))) return KVO_ECUDA;
  return KVO_OK;
}

kvo_status kvo_pool_write(kvo_pool* p, int32_t session, int32_t layer, int64_t first_token, const void* rows,
                          int64_t ntokens, void* stream) {
  return rows_call(p, session, layer, first_token, rows, ntokens, stream, true);
}

kvo_status kvo_pool_read(kvo_pool* p, int32_t session, int32_t layer, int64_t first_token, int64_t ntokens,
                         void* out, void* stream) {
  return rows_call(p, session, layer, first_token, out, ntokens, stream, false);
}

kvo_status kvo_pool_fill(kvo_pool* p, uint8_t byte, void* stream) {
  if (!p) return KVO_EINVAL;
  const uint32_t word = 0x01010101u * byte;
  fill_kernel<<<sm_count() * 4, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<uint4*>(p->pool), p->block_bytes * (size_t)p->pool_blocks / 16, word);
  return ok(cudaGetLastError()) ? KVO_OK : KVO_ECUDA;
}

kvo_status kvo_pool_block_table(kvo_pool* p, int32_t session, int32_t layer, int32_t which, int32_t* out,
                                int64_t max, int64_t* count) {
  if (!p || !count || layer < 0 || layer >= p->layers || (which != 0 && which != 1) || max < 0 ||
      (max > 0 && !out))
    return KVO_EINVAL;
  *count = 0;
  auto it = p->sessions.find(session);
  if (it == p->sessions.end()) return KVO_OK;
  const std::vector<std::vector<int32_t>>& groups = which == 0 ? it->second.pool : it->second.tier;
  if (groups.empty()) return KVO_OK;
  const std::vector<int32_t>& tbl = groups[layer];
  *count = (int64_t)tbl.size();
  const size_t m = tbl.size() < (size_t)max ? tbl.size() : (size_t)max;
  if (m) std::memcpy(out, tbl.data(), m * sizeof(int32_t));
  return KVO_OK;
}

kvo_status kvo_store_blocks(kvo_pool* p, int32_t session, void* stream) {
  if (!p) return KVO_EINVAL;
  auto it = p->sessions.find(session);
  if (it == p->sessions.end() || it->second.pool.empty() || !it->second.tier.empty()) return KVO_EINVAL;
  reap(p, false);
  Session& s = it->second;
  std::vector<size_t> sizes;
  for (auto& g : s.pool) sizes.push_back(g.size());
  std::vector<std::vector<int32_t>> got;
  if (!p->tier_alloc.take_groups(sizes, &got)) {
    ++p->stats.rollbacks;
    return KVO_ECAPACITY;
  }
  if (!ok(plan_host_ready(p))) return KVO_ECUDA;
  size_t n = 0;
  for (int32_t l = 0; l < p->layers; ++l)
    for (size_t b = 0; b < s.pool[l].size(); ++b) p->plan_host[n++] = make_int2(s.pool[l][b], got[l][b]);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (!ok(launch_copy(p, p->pool, p->tier_dev, n, st))) return KVO_ECUDA;
  s.tier = std::move(got);
  ++p->stats.stores;
  p->stats.bytes_stored += (uint64_t)n * p->block_bytes;
  return track(p, {session}, {}, st);
}

kvo_status kvo_pool_release(kvo_pool* p, int32_t session) {
  if (!p) return KVO_EINVAL;
  auto it = p->sessions.find(session);
  if (it == p->sessions.end() || it->second.pool.empty()) return KVO_EINVAL;
  reap(p, false);
  if (it->second.busy) return KVO_EBUSY;
  for (auto& g : it->second.pool) p->pool_alloc.give_back(g);
  it->second.pool.clear();
  if (it->second.tier.empty()) p->sessions.erase(it);
  return KVO_OK;
}

kvo_status kvo_restore_blocks(kvo_pool* p, const int32_t* sessions, int32_t ns, void* stream) {
  if (!p || !sessions || ns < 1) return KVO_EINVAL;
  std::vector<Session*> ss;
  for (int32_t i = 0; i < ns; ++i) {
    for (int32_t j = 0; j < i; ++j)
      if (sessions[j] == sessions[i]) return KVO_EINVAL;
    auto it = p->sessions.find(sessions[i]);
    if (it == p->sessions.end() || it->second.tier.empty() || !it->second.pool.empty()) return KVO_EINVAL;
    ss.push_back(&it->second);
  }
  reap(p, false);
  std::vector<size_t> sizes;
  for (Session* s : ss)
    for (auto& g : s->tier) sizes.push_back(g.size());
  std::vector<std::vector<int32_t>> got;
  if (!p->pool_alloc.take_groups(sizes, &got)) {
    ++p->stats.rollbacks;
    return KVO_ECAPACITY;
  }
  if (!ok(plan_host_ready(p))) return KVO_ECUDA;
  size_t n = 0, gi = 0;
  std::vector<int32_t> tier_free;
  for (Session* s : ss) {
    for (int32_t l = 0; l < p->layers; ++l, ++gi)
      for (size_t b = 0; b < s->tier[l].size(); ++b) p->plan_host[n++] = make_int2(s->tier[l][b], got[gi][b]);
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (!ok(launch_copy(p, p->tier_dev, p->pool, n, st))) return KVO_ECUDA;
  gi = 0;
  for (Session* s : ss) {
    s->pool.assign(got.begin() + gi, got.begin() + gi + p->layers);
    gi += p->layers;
    for (auto& g : s->tier) tier_free.insert(tier_free.end(), g.begin(), g.end());
    s->tier.clear();
  }
  ++p->stats.restores;
  p->stats.bytes_restored += (uint64_t)n * p->block_bytes;
  return track(p, std::vector<int32_t>(sessions, sessions + ns), std::move(tier_free), st);
}

kvo_status kvo_pool_sync(kvo_pool* p, void* stream) {
  if (!p) return KVO_EINVAL;
  if (!ok(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)))) return KVO_ECUDA;
  reap(p, true);
  return KVO_OK;
}

kvo_status kvo_pool_get_stats(kvo_pool* p, kvo_pool_stats* out) {
  if (!p || !out) return KVO_EINVAL;
  reap(p, false);
  p->stats.free_blocks = p->pool_alloc.free.size();
  p->stats.tier_free_blocks = p->tier_alloc.free.size();
  p->stats.pending_copies = p->pending.size();
  *out = p->stats;
  return KVO_OK;
}

kvo_status kvo_pool_debug_fail_after(kvo_pool* p, int32_t which, int64_t n) {
  if (!p || (which != 0 && which != 1)) return KVO_EINVAL;
  (which == 0 ? p->pool_alloc : p->tier_alloc).fail_after = n < 0 ? -1 : n;
  return KVO_OK;
}

kvo_status kvo_pool_debug_free_queue(kvo_pool* p, int32_t which, int32_t* out, int64_t max, int64_t* count) {
  if (!p || !count || (which != 0 && which != 1) || max < 0 || (max > 0 && !out)) return KVO_EINVAL;
  const std::deque<int32_t>& q = (which == 0 ? p->pool_alloc : p->tier_alloc).free;
  *count = (int64_t)q.size();
  int64_t i = 0;
  for (auto it = q.begin(); it != q.end() && i < max; ++it) out[i++] = *it;
  return KVO_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// kvo_copy_blocks_noalloc: the block-copy kernel above, driven from a fixed
// static device array instead of a pool's plan buffer, for callers that own
// their block arrays and may not allocate (see include/kvo.h).
namespace {

// Scratch for the (source, destination) pairs of one call.  Nothing in it has
// to start at zero: every call writes entries [0, n) before its kernel reads
// them and no entry at or past n is ever read.
static __device__ __align__(256) int2 g_noalloc_pairs[KVO_NOALLOC_MAX_PAIRS];

int2* g_noalloc_addr[64] = {};   // per device, looked up by the first call on it

}  // namespace

extern "C" kvo_status kvo_copy_blocks_noalloc(const void* src, void* dst, int64_t block_bytes,
                                              const int32_t* pairs, int64_t n, void* stream) {
  if (n < 0 || n > KVO_NOALLOC_MAX_PAIRS || block_bytes <= 0 || (block_bytes & 15) ||
      block_bytes / 16 > (int64_t)UINT32_MAX ||   // the kernel counts a block's 16-byte pieces in 32 bits
      (n > 0 && (!src || !dst || !pairs || (reinterpret_cast<uintptr_t>(src) & 15u) ||
                 (reinterpret_cast<uintptr_t>(dst) & 15u))))
    return KVO_EINVAL;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KVO_ECUDA;
  if (!g_noalloc_addr[dev]) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_noalloc_pairs) != cudaSuccess) {
      cudaGetLastError();
      return KVO_ECUDA;
    }
    g_noalloc_addr[dev] = static_cast<int2*>(a);
  }
  if (n == 0) return KVO_OK;
  if (!device_accessible(src) || !device_accessible(dst)) return KVO_EINVAL;
  for (int64_t i = 0; i < 2 * n; ++i)
    if (pairs[i] < 0) return KVO_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(g_noalloc_addr[dev], pairs, (size_t)n * sizeof(int2), cudaMemcpyHostToDevice, s) !=
      cudaSuccess)
    return KVO_ECUDA;
  const int64_t cap = (int64_t)sm_count() * 8;
  block_copy_kernel<<<(unsigned)(n < cap ? n : cap), 256, 0, s>>>(
      static_cast<const uint4*>(src), static_cast<uint4*>(dst), g_noalloc_addr[dev], n,
      (uint32_t)(block_bytes / 16));
  return cudaGetLastError() == cudaSuccess ? KVO_OK : KVO_ECUDA;
}
