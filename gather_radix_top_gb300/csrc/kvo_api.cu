// The kvo C ABI: context lifetime, argument checks and launches.
//
// Host memory layout: each layer's history is one pinned, device-mapped host
// allocation of history_cap * 656 bytes ("From 1M Total to 15+ x 1M
// Contexts: GLM-5.3 KV Cache Offloading", "Decision three": misses read the
// registered host copy).  Device memory: per layer an exact-size hot cache
// and tables ("Ten sessions exposed a physical-allocation problem": long-lived
// caches get exact-capacity allocations, never pooled blocks).
#include <cstdint>
#include <cstdlib>
#include <algorithm>
#include <chrono>
#include <cstring>
#include <new>
#include <vector>

#include "kvo.h"
#include "kvo_device.cuh"
#include "kvo_internal.h"

struct kvo_ctx {
  int device = 0;
  int32_t layers = 0;
  int64_t history_cap = 0;
  int32_t hot_rows = 0;
  int max_cluster = 16;
  std::vector<uint8_t*> hist_host;       // pinned host history per layer
  std::vector<kvo::LayerView> views;     // device pointers per layer
  std::vector<int64_t> length;           // host copy of each history length
  uint32_t* counters = nullptr;          // device [layers][8]: step, length, queue head, tail, buffer, hand
  unsigned long long* stats = nullptr;   // device [layers][8]
  int32_t* evlog = nullptr;              // device [layers][1 + 3*KVO_MAX_ROUND] when recording
  uint32_t* status = nullptr;            // device status word
  bool resolved = false;                 // a resolve has been enqueued (the policy is fixed from then on)
  bool unusable = false;                 // a bulk copy may still land in freed shared memory: no more launches
  uint32_t ring_rows = 0;                // recent ring rows per layer (0: appends go straight to RAM)
  std::vector<int64_t> ram_len;          // per layer: rows the host history (RAM) holds
  struct {                               // kvo_decode_step_host's device staging
    float* scores = nullptr;             // history_cap fp32
    int32_t* idx = nullptr;              // KVO_MAX_K
    uint8_t* out = nullptr;              // KVO_MAX_K rows
    uint16_t* bf16 = nullptr;            // KVO_MAX_K dequantised rows (allocated on first use)
    uint8_t* rows = nullptr;             // rows_cap new rows (grows)
    int64_t rows_cap = 0;
  } stage;
  kvo::LayerStatic* statics = nullptr;   // device [layers]: what the batched decode step reads per layer
  uint32_t* first_hist = nullptr;        // device [layers][2048]: the batched step's filtering histograms (zero
                                         // between calls: each selection zeroes its own after use)
  uint32_t* ent = nullptr;               // device [layers][KVO_MAX_K]: the batched step's entry codes
  kvo::LayersFilter filt{};              // the batched step's filter lists (one allocation, grown on demand)
  bool statics_dirty = true;             // the views changed since the last upload
  int64_t launches = 0;                  // kernels kvo_decode_layers has launched
  double host_seconds = 0.0;             // host time spent inside kvo_decode_layers
  void* touch_sink = nullptr;            // kvo_touch_history's 16-byte sink
  // kvo_set_miss_fetch: how kvo_decode_layers fetches the misses of the host
  // history (zero-copy loads, batched copies, or chosen by the miss rate)
  int32_t miss_mode = KVO_MISS_ZEROCOPY;
  int32_t miss_auto_pct = 100;
  kvo::LayersDefer defer = {};           // the batched-copy buffers (made on first use)
  int32_t defer_k = 0;                   // staging rows per layer
  std::vector<const uint8_t*> hist_ptrs; // host address of each layer's history
  unsigned long long* stats_snap = nullptr;   // pinned [layers][8]: the last stats snapshot (AUTO)
  cudaEvent_t snap_ev = nullptr;         // the snapshot has landed
  bool snap_pending = false;
  double snap_hits = -1.0, snap_misses = 0.0;  // totals of the last snapshot read
  double miss_rate = 0.0;                // the last measured miss share of kvo_decode_layers
  bool phase_timing = false;             // kvo_decode_layers records events around its launches
  std::vector<cudaEvent_t> phase_ev;     // 4 per recorded call, reused
  size_t phase_calls = 0;                // calls recorded since the last kvo_layers_phase_times
};

namespace {

constexpr size_t kEvlogStride = 1 + 3 * (size_t)KVO_MAX_ROUND;

bool ok(cudaError_t e) { return e == cudaSuccess; }

void free_ctx(kvo_ctx* c) {
  if (!c) return;
  for (auto& v : c->views) {
    cudaFree(v.pos2slot);
    cudaFree(v.slot2pos);
    cudaFree(v.last_use);
    cudaFree(v.hot);
    cudaFree(v.ring);
    cudaFree(v.recent);
  }
  for (uint8_t* h : c->hist_host) cudaFreeHost(h);
  cudaFree(c->counters);
  cudaFree(c->stats);
  cudaFree(c->stage.scores);
  cudaFree(c->stage.idx);
  cudaFree(c->stage.out);
  cudaFree(c->stage.bf16);
  cudaFree(c->stage.rows);
  cudaFree(c->evlog);
  cudaFree(c->status);
  cudaFree(c->statics);
  cudaFree(c->first_hist);
  cudaFree(c->ent);
  cudaFree(c->filt.count);
  cudaFree(c->touch_sink);
  cudaFreeHost(const_cast<int2*>(c->defer.dlist_host));
  cudaFree(c->defer.dcount_dev);
  cudaFreeHost(c->defer.dcount_host);
  cudaFreeHost(c->defer.plist_host);
  cudaFreeHost(c->defer.pcount_host);
  cudaFree(c->defer.staging);
  if (c->defer.listed) cudaEventDestroy(c->defer.listed);
  cudaFreeHost(c->stats_snap);
  if (c->snap_ev) cudaEventDestroy(c->snap_ev);
  for (cudaEvent_t e : c->phase_ev) cudaEventDestroy(e);
  delete c;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// fp32 scores and int32 positions are read and written as whole words
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

bool is_device_pointer(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

// The driver's cuMemGetAddressRange (base and size of the allocation that
// holds a device address), reached through the runtime.
using GetRangeFn = int (*)(unsigned long long*, size_t*, unsigned long long);
GetRangeFn address_range_fn() {
  static const GetRangeFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      return static_cast<GetRangeFn>(nullptr);
    }
    return reinterpret_cast<GetRangeFn>(f);
  }();
  return fn;
}

// The device allocations that one call's argument checks have found: a
// buffer inside one of them needs no further driver query (the layers of a
// batched call usually take their rows from one tensor).
struct DeviceRanges {
  std::vector<std::pair<uintptr_t, uintptr_t>> r;   // [lo, hi)
  // Whether [p, p + bytes) is device memory.
  bool check(const void* p, size_t bytes) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    for (const auto& x : r)
      if (a >= x.first && a + bytes <= x.second) return true;
    if (!is_device_pointer(p)) return false;
    unsigned long long base = 0;
    size_t size = 0;
    const GetRangeFn fn = address_range_fn();
    if (fn && fn(&base, &size, (unsigned long long)a) == 0) {
      if (a + bytes > base + size) return false;     // the buffer runs past its allocation
      r.emplace_back((uintptr_t)base, (uintptr_t)(base + size));
    }
    return true;
  }
};

// Room for the filter lists of `slices` slices of 4,096 scores (grown by a
// quarter beyond the need; the old lists are freed once the device is idle).
cudaError_t ensure_filter(kvo_ctx* c, size_t slices) {
  kvo::LayersFilter& f = c->filt;
  if (slices <= f.slices) return cudaSuccess;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return e;
  cudaFree(f.count);
  f = kvo::LayersFilter{};
  const size_t want = slices + slices / 4;
  void* p = nullptr;
  if ((e = cudaMalloc(&p, want * (sizeof(uint32_t) + 2 * sizeof(uint32_t) * 4096))) != cudaSuccess) return e;
  f.count = static_cast<uint32_t*>(p);
  f.key = f.count + want;
  f.pos = f.key + want * 4096;
  f.slices = want;
  return cudaSuccess;
}

// The batched-copy buffers, made on first use (staging grows with k).
cudaError_t ensure_defer(kvo_ctx* c, int32_t k) {
  kvo::LayersDefer& d = c->defer;
  cudaError_t e = cudaSuccess;
  const size_t L = (size_t)c->layers;
  if (!d.dlist_host) {
    void* p = nullptr;
    if ((e = cudaHostAlloc(&p, L * KVO_MAX_K * sizeof(int2), cudaHostAllocMapped)) != cudaSuccess) return e;
    d.dlist_host = static_cast<const int2*>(p);
    if ((e = cudaHostGetDevicePointer(reinterpret_cast<void**>(&d.dlist_dev), p, 0)) != cudaSuccess) return e;
    if ((e = cudaMalloc(&d.dcount_dev, L * sizeof(uint32_t))) != cudaSuccess) return e;
    if ((e = cudaMemset(d.dcount_dev, 0, L * sizeof(uint32_t))) != cudaSuccess) return e;
    if ((e = cudaHostAlloc(reinterpret_cast<void**>(&d.dcount_host), L * sizeof(uint32_t), 0)) != cudaSuccess)
      return e;
    if ((e = cudaHostAlloc(reinterpret_cast<void**>(&d.plist_host), L * KVO_MAX_K * sizeof(int2),
                           cudaHostAllocMapped)) != cudaSuccess)
      return e;
    if ((e = cudaHostGetDevicePointer(const_cast<void**>(reinterpret_cast<const void**>(&d.plist_dev)), d.plist_host,
                                      0)) != cudaSuccess)
      return e;
    if ((e = cudaHostAlloc(reinterpret_cast<void**>(&d.pcount_host), L * sizeof(uint32_t), cudaHostAllocMapped)) !=
        cudaSuccess)
      return e;
    if ((e = cudaHostGetDevicePointer(const_cast<void**>(reinterpret_cast<const void**>(&d.pcount_dev)),
                                      d.pcount_host, 0)) != cudaSuccess)
      return e;
    if ((e = cudaEventCreateWithFlags(&d.listed, cudaEventDisableTiming)) != cudaSuccess) return e;
    c->hist_ptrs.assign(c->hist_host.begin(), c->hist_host.end());
    d.hist_host = c->hist_ptrs.data();
  }
  if (c->defer_k < k) {
    cudaFree(d.staging);
    d.staging = nullptr;
    c->defer_k = 0;
    if ((e = cudaMalloc(&d.staging, L * (size_t)k * KVO_ROW_BYTES)) != cudaSuccess) return e;
    c->defer_k = k;
  }
  return cudaSuccess;
}

// AUTO: the miss share of the recent kvo_decode_layers calls, from stats
// snapshots copied asynchronously after a call and read at a later call once
// they have landed (no wait).
cudaError_t measure_miss_rate(kvo_ctx* c, cudaStream_t s) {
  cudaError_t e;
  if (!c->stats_snap) {
    if ((e = cudaHostAlloc(reinterpret_cast<void**>(&c->stats_snap), sizeof(unsigned long long) * 8 * c->layers, 0)) !=
        cudaSuccess)
      return e;
    if ((e = cudaEventCreateWithFlags(&c->snap_ev, cudaEventDisableTiming)) != cudaSuccess) return e;
  }
  if (c->snap_pending && cudaEventQuery(c->snap_ev) == cudaSuccess) {
    double hits = 0, misses = 0;
    for (int32_t l = 0; l < c->layers; ++l) {
      hits += (double)c->stats_snap[8 * l + 1];
      misses += (double)c->stats_snap[8 * l + 2];
    }
    if (c->snap_hits >= 0.0 && hits + misses > c->snap_hits + c->snap_misses)
      c->miss_rate = (misses - c->snap_misses) / (hits + misses - c->snap_hits - c->snap_misses);
    c->snap_hits = hits;
    c->snap_misses = misses;
    c->snap_pending = false;
  }
  cudaGetLastError();                                    // a query that is not ready is not an error
  if (!c->snap_pending) {
    if ((e = cudaMemcpyAsync(c->stats_snap, c->stats, sizeof(unsigned long long) * 8 * c->layers,
                             cudaMemcpyDeviceToHost, s)) != cudaSuccess)
      return e;
    if ((e = cudaEventRecord(c->snap_ev, s)) != cudaSuccess) return e;
    c->snap_pending = true;
  }
  return cudaSuccess;
}

// Uploads the per-layer table the batched decode step reads, when the views
// changed (the work in flight that reads the old table is waited for first).
cudaError_t upload_statics(kvo_ctx* c) {
  if (!c->statics_dirty) return cudaSuccess;
  std::vector<kvo::LayerStatic> h(c->layers);
  for (int32_t l = 0; l < c->layers; ++l) {
    const kvo::LayerView& v = c->views[l];
    h[l] = kvo::LayerStatic{v.pos2slot, v.slot2pos, v.last_use, v.hot, v.hist, v.counters, v.stats,
                            c->evlog ? c->evlog + kEvlogStride * l : nullptr, v.ring, v.recent,
                            v.hot_rows, v.history_cap, v.ring_cap, v.ring_rows};
  }
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(c->statics, h.data(), h.size() * sizeof(h[0]), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) c->statics_dirty = false;
  return e;
}

// Copies device rows into the mapped host history and publishes the new
// length (block 0) in stream order.
__global__ void append_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, uint64_t nvec,
                              uint32_t* counters, uint32_t new_len) {
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += stride) dst[i] = src[i];
  if (blockIdx.x == 0 && threadIdx.x == 0) counters[1] = new_len;
}

// Copies device rows into the recent ring (row i to slot (start + i) mod
// ring rows) and publishes the new length (block 0) in stream order.
__global__ void ring_append_kernel(const uint4* __restrict__ src, uint4* __restrict__ ring, uint32_t r,
                                   uint32_t start, uint32_t ring_mask, uint32_t* counters, uint32_t new_len) {
  constexpr uint32_t kVec = KVO_ROW_BYTES / 16;
  const uint64_t total = (uint64_t)r * kVec;
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    const uint32_t row = (uint32_t)(i / kVec), v = (uint32_t)(i - (uint64_t)row * kVec);
    ring[(size_t)((start + row) & ring_mask) * kVec + v] = src[i];
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) counters[1] = new_len;
}

// Reads pinned host memory with 16-byte zero-copy loads, one piece every
// `step` pieces; XOR-folds into sink.
__global__ void probe_kernel(const uint4* __restrict__ src, uint64_t nvec, uint64_t step, uint4* sink) {
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  uint4 acc = make_uint4(0, 0, 0, 0);
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i * step < nvec; i += stride) {
    const uint4 v = src[i * step];
    acc.x ^= v.x;
    acc.y ^= v.y;
    acc.z ^= v.z;
    acc.w ^= v.w;
  }
  if ((acc.x | acc.y | acc.z | acc.w) == 0xdeadbeefu) sink[0] = acc;   // keeps the loads live
}

}  // namespace

namespace kvo {

cudaError_t launch_append(const void* src_dev, uint8_t* hist_dev_dst, uint64_t bytes,
                          uint32_t* counters, uint32_t new_len, cudaStream_t stream) {
  const uint64_t nvec = bytes / 16;
  int sms = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  uint64_t blocks = (nvec + 255) / 256;
  const uint64_t cap = (uint64_t)(sms > 0 ? sms : 1) * 4;
  if (blocks > cap) blocks = cap;
  if (blocks == 0) blocks = 1;
  append_kernel<<<(unsigned)blocks, 256, 0, stream>>>(static_cast<const uint4*>(src_dev),
                                                     reinterpret_cast<uint4*>(hist_dev_dst), nvec,
                                                     counters, new_len);
  return cudaGetLastError();
}

cudaError_t launch_ring_append(const void* src_dev, uint8_t* ring, uint32_t r, uint32_t start, uint32_t ring_mask,
                               uint32_t* counters, uint32_t new_len, cudaStream_t stream) {
  const uint64_t nvec = (uint64_t)r * (KVO_ROW_BYTES / 16);
  uint64_t blocks = (nvec + 255) / 256;
  if (blocks > 1024) blocks = 1024;
  if (blocks == 0) blocks = 1;
  ring_append_kernel<<<(unsigned)blocks, 256, 0, stream>>>(static_cast<const uint4*>(src_dev),
                                                          reinterpret_cast<uint4*>(ring), r, start, ring_mask,
                                                          counters, new_len);
  return cudaGetLastError();
}

cudaError_t launch_probe(const void* src, uint64_t bytes, void* sink, cudaStream_t stream, uint64_t stride) {
  int sms = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  probe_kernel<<<sms * 4, 512, 0, stream>>>(static_cast<const uint4*>(src), bytes / 16, stride / 16,
                                            static_cast<uint4*>(sink));
  return cudaGetLastError();
}

}  // namespace kvo

namespace {

// Moves the layer's ring rows [ram_len, upto) to the host history (one or
// two copies; the ring wraps) and advances ram_len, in stream order.
cudaError_t ring_copyback(kvo_ctx* ctx, int32_t layer, int64_t upto, cudaStream_t s) {
  const int64_t from = ctx->ram_len[layer];
  if (!ctx->ring_rows || upto <= from) return cudaSuccess;
  const kvo::LayerView& v = ctx->views[layer];
  const int64_t R = ctx->ring_rows;
  int64_t pos = from;
  while (pos < upto) {
    const int64_t slot = pos & (R - 1);
    const int64_t n = std::min(upto - pos, R - slot);
    const cudaError_t e = cudaMemcpyAsync(ctx->hist_host[layer] + (size_t)pos * KVO_ROW_BYTES,
                                          v.recent + (size_t)slot * KVO_ROW_BYTES, (size_t)n * KVO_ROW_BYTES,
                                          cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return e;
    pos += n;
  }
  ctx->ram_len[layer] = upto;
  return cudaSuccess;
}

// After device rows were appended: whole batches of KVO_COPYBACK_BATCH rows
// move to RAM.
cudaError_t ring_after_append(kvo_ctx* ctx, int32_t layer, cudaStream_t s) {
  if (!ctx->ring_rows) return cudaSuccess;
  const int64_t pending = ctx->length[layer] - ctx->ram_len[layer];
  return ring_copyback(ctx, layer, ctx->ram_len[layer] + pending / KVO_COPYBACK_BATCH * KVO_COPYBACK_BATCH, s);
}

// The rows RAM holds once r device rows are appended to the layer: every
// appended row without the ring; with it, the rows before the ring's pending
// ones plus every whole batch of KVO_COPYBACK_BATCH pending rows (a batch is
// copied back as soon as it is complete).
int64_t ram_after_append(const kvo_ctx* ctx, int32_t layer, int64_t r) {
  const int64_t len = ctx->length[layer] + r;
  if (!ctx->ring_rows) return len;
  const int64_t ram = ctx->ram_len[layer];
  return ram + (len - ram) / KVO_COPYBACK_BATCH * KVO_COPYBACK_BATCH;
}

// A launch that appends r device rows and resolves in the same step sees the
// append's copyback already done: the ring rows it moves to RAM that were
// appended by earlier calls are copied here, before the launch; the launch
// itself writes its own rows below the new RAM length to the host history
// rather than to the ring.  Returns the new RAM length (the launch's
// ram_len); the caller stores it once the launch is enqueued.
cudaError_t copyback_before_step(kvo_ctx* ctx, int32_t layer, int64_t r, cudaStream_t s, int64_t* ram) {
  *ram = ram_after_append(ctx, layer, r);
  if (!ctx->ring_rows) return cudaSuccess;
  return ring_copyback(ctx, layer, std::min(*ram, ctx->length[layer]), s);
}

}  // namespace

extern "C" {

const char* kvo_status_string(kvo_status s) {
  switch (s) {
    case KVO_OK: return "ok";
    case KVO_EINVAL: return "invalid argument";
    case KVO_ENOMEM: return "out of memory";
    case KVO_ECUDA: return "CUDA error";
    case KVO_ERANGE: return "selected position outside the history";
    case KVO_EBUSY: return "busy";
    case KVO_ETIMEDOUT: return "device wait timed out";
    case KVO_ECAPACITY: return "not enough blocks";
  }
  return "unknown status";
}

kvo_status kvo_create(int32_t layers, int64_t history_cap, int32_t hot_rows, int32_t row_bytes,
                      kvo_ctx** out) {
  if (!out || layers < 1 || history_cap < 1 || history_cap > INT32_MAX || hot_rows < 1 ||
      hot_rows > KVO_MAX_HOT_ROWS || row_bytes != KVO_ROW_BYTES)
    return KVO_EINVAL;
  kvo_ctx* c = new (std::nothrow) kvo_ctx;
  if (!c) return KVO_ENOMEM;
  if (!ok(cudaGetDevice(&c->device))) {
    delete c;
    return KVO_ECUDA;
  }
  // KVO_MAX_CLUSTER (2, 4, 8 or 16) caps the CTAs per cluster: a tuning knob
  if (const char* env = std::getenv("KVO_MAX_CLUSTER")) {
    const int m = std::atoi(env);
    if (m == 2 || m == 4 || m == 8 || m == 16) c->max_cluster = m;
  }
  c->layers = layers;
  c->history_cap = history_cap;
  c->hot_rows = hot_rows;
  c->length.assign(layers, 0);
  c->ram_len.assign(layers, 0);
  bool good = ok(cudaMalloc(&c->counters, sizeof(uint32_t) * 8 * layers)) &&
              ok(cudaMalloc(&c->stats, sizeof(unsigned long long) * 8 * layers)) &&
              ok(cudaMalloc(&c->status, sizeof(uint32_t))) &&
              ok(cudaMalloc(&c->statics, sizeof(kvo::LayerStatic) * layers)) &&
              ok(cudaMalloc(&c->first_hist, sizeof(uint32_t) * kvo::kLayersHistWords * layers)) &&
              ok(cudaMemset(c->first_hist, 0, sizeof(uint32_t) * kvo::kLayersHistWords * layers)) &&
              ok(cudaMalloc(&c->ent, sizeof(uint32_t) * KVO_MAX_K * layers)) &&
              ok(cudaMemset(c->counters, 0, sizeof(uint32_t) * 8 * layers)) &&
              ok(cudaMemset(c->stats, 0, sizeof(unsigned long long) * 8 * layers)) &&
              ok(cudaMemset(c->status, 0, sizeof(uint32_t)));
  // slot tables padded to whole 16-byte pieces: kernels copy them in 16-byte units
  const size_t padded_rows = ((size_t)hot_rows + 3) & ~(size_t)3;
  // every slot starts empty (last_use 0): the LRU queue starts as one entry
  // per slot, stamped 0, in slot order; head 0, tail hot_rows
  uint32_t ring_cap = 1;
  while (ring_cap < 8u * (uint32_t)hot_rows) ring_cap <<= 1;
  std::vector<uint64_t> first(hot_rows);
  for (int32_t i = 0; i < hot_rows; ++i) first[i] = (uint64_t)(uint32_t)i;
  const uint32_t init_counters[8] = {0, 0, 0, (uint32_t)hot_rows, 0, 0, 0, 0};
  for (int32_t l = 0; good && l < layers; ++l) {
    kvo::LayerView v = {};
    v.hot_rows = (uint32_t)hot_rows;
    v.history_cap = (uint32_t)history_cap;
    v.counters = c->counters + 8 * l;
    v.ring_cap = ring_cap;
    v.gather_mode = KVO_GATHER_AUTO;              // staged from 5 % misses on: the measured crossover
    v.auto_miss_pct = 5;
    v.stats = c->stats + 8 * l;
    uint8_t* h = nullptr;
    good = ok(cudaHostAlloc((void**)&h, (size_t)history_cap * KVO_ROW_BYTES,
                            cudaHostAllocMapped | cudaHostAllocPortable));
    if (!good) break;
    c->hist_host.push_back(h);
    void* hd = nullptr;
    good = ok(cudaHostGetDevicePointer(&hd, h, 0));
    v.hist = static_cast<const uint8_t*>(hd);
    good = good && ok(cudaMalloc(&v.pos2slot, sizeof(int32_t) * (size_t)history_cap)) &&
           ok(cudaMalloc(&v.slot2pos, sizeof(int32_t) * padded_rows)) &&
           ok(cudaMalloc(&v.last_use, sizeof(uint32_t) * padded_rows)) &&
           ok(cudaMalloc(&v.hot, (size_t)hot_rows * KVO_ROW_BYTES)) &&
           ok(cudaMalloc(&v.ring, sizeof(uint64_t) * 2 * (size_t)ring_cap));
    c->views.push_back(v);
    good = good && ok(cudaMemset(v.pos2slot, 0xff, sizeof(int32_t) * (size_t)history_cap)) &&
           ok(cudaMemset(v.slot2pos, 0xff, sizeof(int32_t) * padded_rows)) &&
           ok(cudaMemset(v.last_use, 0, sizeof(uint32_t) * padded_rows)) &&
           ok(cudaMemset(v.hot, 0, (size_t)hot_rows * KVO_ROW_BYTES)) &&
           ok(cudaMemcpy(v.ring, first.data(), sizeof(uint64_t) * (size_t)hot_rows, cudaMemcpyHostToDevice)) &&
           ok(cudaMemcpy(v.counters, init_counters, sizeof(init_counters), cudaMemcpyHostToDevice));
  }
  if (good) good = ok(cudaDeviceSynchronize());
  if (!good) {
    cudaGetLastError();
    free_ctx(c);
    return KVO_ENOMEM;
  }
  *out = c;
  return KVO_OK;
}

kvo_status kvo_destroy(kvo_ctx* ctx) {
  if (!ctx) return KVO_EINVAL;
  const bool synced = ok(cudaDeviceSynchronize());
  free_ctx(ctx);
  return synced ? KVO_OK : KVO_ECUDA;
}

kvo_status kvo_append_rows(kvo_ctx* ctx, int32_t layer, const void* rows, int64_t r, void* stream) {
  if (ctx && ctx->unusable) return KVO_ECUDA;
  if (!ctx || layer < 0 || layer >= ctx->layers || r < 0) return KVO_EINVAL;
  if (r == 0) return KVO_OK;
  if (!rows || !aligned16(rows) || ctx->length[layer] + r > ctx->history_cap) return KVO_EINVAL;
  const bool dev_rows = is_device_pointer(rows);
  if (dev_rows && ctx->ring_rows && r > (int64_t)ctx->ring_rows - KVO_COPYBACK_BATCH) return KVO_EINVAL;
  const int64_t start = ctx->length[layer];
  const uint64_t bytes = (uint64_t)r * KVO_ROW_BYTES;
  kvo::LayerView& v = ctx->views[layer];
  uint8_t* dst_dev = const_cast<uint8_t*>(v.hist) + (size_t)start * KVO_ROW_BYTES;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (dev_rows && ctx->ring_rows) {
    e = kvo::launch_ring_append(rows, v.recent, (uint32_t)r, (uint32_t)start, ctx->ring_rows - 1, v.counters,
                                (uint32_t)(start + r), s);
    if (!ok(e)) return KVO_ECUDA;
    ctx->length[layer] = start + r;
    return ok(ring_after_append(ctx, layer, s)) ? KVO_OK : KVO_ECUDA;
  }
  if (dev_rows) {
    e = kvo::launch_append(rows, dst_dev, bytes, v.counters, (uint32_t)(start + r), s);
  } else {
    // Host rows: the ring's pending rows go first (they precede these
    // positions), then the rows are copied now (the positions are beyond
    // every enqueued read) and the length is published in stream order.
    if (!ok(ring_copyback(ctx, layer, start, s))) return KVO_ECUDA;
    std::memcpy(ctx->hist_host[layer] + (size_t)start * KVO_ROW_BYTES, rows, bytes);
    e = kvo::launch_append(nullptr, dst_dev, 0, v.counters, (uint32_t)(start + r), s);
  }
  if (!ok(e)) return KVO_ECUDA;
  ctx->length[layer] = start + r;
  ctx->ram_len[layer] = start + r;
  return KVO_OK;
}

kvo_status kvo_select_topk(kvo_ctx* ctx, const float* scores, int64_t n, int32_t k, int32_t* idx,
                           void* stream) {
  if (ctx && ctx->unusable) return KVO_ECUDA;
  if (!ctx || !scores || !idx || k < 1 || k > KVO_MAX_K || n < k || n > INT32_MAX) return KVO_EINVAL;
  if (!aligned4(scores) || !aligned4(idx)) return KVO_EINVAL;
  const cudaError_t e = kvo::launch_topk(scores, (uint32_t)n, (uint32_t)k, idx, ctx->max_cluster,
                                         static_cast<cudaStream_t>(stream));
  return ok(e) ? KVO_OK : KVO_ECUDA;
}

kvo_status kvo_set_recent_ring(kvo_ctx* ctx, int32_t rows) {
  if (!ctx || rows < 0 || (rows && (rows < 128 || rows > 65536 || (rows & (rows - 1))))) return KVO_EINVAL;
  for (int64_t n : ctx->length)
    if (n) return KVO_EBUSY;
  if (!ok(cudaDeviceSynchronize())) return KVO_ECUDA;
  for (kvo::LayerView& v : ctx->views) {
    cudaFree(v.recent);
    v.recent = nullptr;
    v.ring_rows = 0;
  }
  ctx->ring_rows = 0;
  ctx->statics_dirty = true;
  if (!rows) return KVO_OK;
  for (kvo::LayerView& v : ctx->views) {
    if (!ok(cudaMalloc(&v.recent, (size_t)rows * KVO_ROW_BYTES))) {
      cudaGetLastError();
      for (kvo::LayerView& w : ctx->views) {
        cudaFree(w.recent);
        w.recent = nullptr;
        w.ring_rows = 0;
      }
      return KVO_ENOMEM;
    }
    v.ring_rows = (uint32_t)rows;
  }
  ctx->ring_rows = (uint32_t)rows;
  return KVO_OK;
}

kvo_status kvo_flush_ring(kvo_ctx* ctx, int32_t layer, void* stream) {
  if (ctx && ctx->unusable) return KVO_ECUDA;
  if (!ctx || layer < 0 || layer >= ctx->layers) return KVO_EINVAL;
  return ok(ring_copyback(ctx, layer, ctx->length[layer], static_cast<cudaStream_t>(stream))) ? KVO_OK
                                                                                                : KVO_ECUDA;
}

kvo_status kvo_set_phase_timing(kvo_ctx* ctx, int32_t on) {
  if (!ctx) return KVO_EINVAL;
  ctx->phase_timing = on != 0;
  ctx->phase_calls = 0;
  return KVO_OK;
}

kvo_status kvo_layers_counters(kvo_ctx* ctx, int64_t* launches, double* host_seconds) {
  if (!ctx || !launches || !host_seconds) return KVO_EINVAL;
  *launches = ctx->launches;
  *host_seconds = ctx->host_seconds;
  return KVO_OK;
}

kvo_status kvo_layers_phase_times(kvo_ctx* ctx, double* ms, int64_t* calls) {
  if (!ctx || !ms || !calls) return KVO_EINVAL;
  ms[0] = ms[1] = ms[2] = 0.0;
  for (size_t c = 0; c < ctx->phase_calls; ++c) {
    cudaEvent_t* ev = ctx->phase_ev.data() + 4 * c;
    if (!ok(cudaEventSynchronize(ev[3]))) return KVO_ECUDA;
    for (int i = 0; i < 3; ++i) {
      float t = 0.f;
      if (!ok(cudaEventElapsedTime(&t, ev[i], ev[i + 1]))) return KVO_ECUDA;
      ms[i] += t;
    }
  }
  *calls = (int64_t)ctx->phase_calls;
  ctx->phase_calls = 0;
  return KVO_OK;
}

kvo_status kvo_ram_length(kvo_ctx* ctx, int32_t layer, int64_t* out) {
  if (!ctx || !out || layer < 0 || layer >= ctx->layers) return KVO_EINVAL;
  *out = ctx->ram_len[layer];
  return KVO_OK;
}

kvo_status kvo_debug_read_history(kvo_ctx* ctx, int32_t layer, int64_t start, int64_t count, void* out) {
  if (!ctx || !out || layer < 0 || layer >= ctx->layers || start < 0 || count < 0 ||
      start + count > ctx->history_cap)
    return KVO_EINVAL;
  if (!ok(cudaDeviceSynchronize())) return KVO_ECUDA;
  std::memcpy(out, ctx->hist_host[layer] + (size_t)start * KVO_ROW_BYTES, (size_t)count * KVO_ROW_BYTES);
  return KVO_OK;
}

kvo_status kvo_set_gather_mode(kvo_ctx* ctx, int32_t mode, int32_t auto_miss_pct) {
  if (!ctx || mode < KVO_GATHER_LOADS || mode > KVO_GATHER_AUTO || auto_miss_pct < 0 || auto_miss_pct > 100)
    return KVO_EINVAL;
  for (kvo::LayerView& v : ctx->views) {
    v.gather_mode = (uint32_t)mode;
    v.auto_miss_pct = (uint32_t)auto_miss_pct;
  }
  return KVO_OK;
}

kvo_status kvo_set_miss_fetch(kvo_ctx* ctx, int32_t mode, int32_t auto_miss_pct) {
  if (!ctx || mode < KVO_MISS_ZEROCOPY || mode > KVO_MISS_AUTO || auto_miss_pct < 0 || auto_miss_pct > 100)
    return KVO_EINVAL;
  ctx->miss_mode = mode;
  ctx->miss_auto_pct = auto_miss_pct;
  return KVO_OK;
}

kvo_status kvo_set_policy(kvo_ctx* ctx, int32_t policy) {
  if (!ctx || (policy != KVO_POLICY_LRU && policy != KVO_POLICY_CIRCULAR)) return KVO_EINVAL;
  if (ctx->resolved) return KVO_EBUSY;
  for (kvo::LayerView& v : ctx->views) v.policy = (uint32_t)policy;
  return KVO_OK;
}

kvo_status kvo_debug_raise_status(kvo_ctx* ctx, uint32_t bits) {
  if (!ctx || bits > 15u) return KVO_EINVAL;
  uint32_t st = 0;
  if (!ok(cudaDeviceSynchronize()) || !ok(cudaMemcpy(&st, ctx->status, sizeof st, cudaMemcpyDeviceToHost)))
    return KVO_ECUDA;
  st |= bits;
  return ok(cudaMemcpy(ctx->status, &st, sizeof st, cudaMemcpyHostToDevice)) ? KVO_OK : KVO_ECUDA;
}

kvo_status kvo_debug_layer_counters(kvo_ctx* ctx, int32_t layer, uint32_t* out) {
  if (!ctx || !out || layer < 0 || layer >= ctx->layers) return KVO_EINVAL;
  if (!ok(cudaDeviceSynchronize())) return KVO_ECUDA;
  return ok(cudaMemcpy(out, ctx->views[layer].counters, 8 * sizeof(uint32_t), cudaMemcpyDeviceToHost)) ? KVO_OK
                                                                                                  : KVO_ECUDA;
}

kvo_status kvo_select_topk_batch(kvo_ctx* ctx, const float* scores, int64_t n, int64_t ld, int32_t nq, int32_t k,
                                 int32_t* idx, void* stream) {
  if (ctx && ctx->unusable) return KVO_ECUDA;
  if (!ctx || !scores || !idx || nq < 1 || nq > 65535 || k < 1 || k > KVO_MAX_K || n < k || n > INT32_MAX ||
      ld < n || !aligned4(scores) || !aligned4(idx))
    return KVO_EINVAL;
  const cudaError_t e = kvo::launch_topk(scores, (uint32_t)n, (uint32_t)k, idx, ctx->max_cluster,
                                         static_cast<cudaStream_t>(stream), (uint32_t)nq, (uint64_t)ld);
  return ok(e) ? KVO_OK : KVO_ECUDA;
}

kvo_status kvo_resolve_gather(kvo_ctx* ctx, int32_t layer, const int32_t* idx, int32_t k,
                              void* out_rows, uint16_t* out_bf16, void* stream) {
  if (ctx && ctx->unusable) return KVO_ECUDA;
  if (!ctx || layer < 0 || layer >= ctx->layers || !idx || !aligned4(idx) || k < 1 || k > KVO_MAX_K ||
      k > ctx->hot_rows || (!out_rows && !out_bf16))
    return KVO_EINVAL;
  if ((out_rows && !aligned16(out_rows)) || (out_bf16 && !aligned16(out_bf16))) return KVO_EINVAL;
  kvo::LayerView v = ctx->views[layer];
  v.evlog = ctx->evlog ? ctx->evlog + kEvlogStride * layer : nullptr;
  v.ram_len = (uint32_t)ctx->ram_len[layer];
  const cudaError_t e =
      kvo::launch_resolve(v, idx, (uint32_t)k, static_cast<uint8_t*>(out_rows), out_bf16, ctx->status,
                          ctx->max_cluster, static_cast<cudaStream_t>(stream));
  ctx->resolved = true;
  return ok(e) ? KVO_OK : KVO_ECUDA;
}

kvo_status kvo_resolve_gather_multi(kvo_ctx* ctx, int32_t layer, const int32_t* idx, int32_t nq, int32_t k,
                                    void* out_rows, uint16_t* out_bf16, void* stream) {
  if (ctx && ctx->unusable) return KVO_ECUDA;
  if (!ctx || layer < 0 || layer >= ctx->layers || !idx || !aligned4(idx) || nq < 1 || k < 1 || k > KVO_MAX_K ||
      (int64_t)nq * k > KVO_MAX_ROUND || (int64_t)nq * k > ctx->hot_rows || (!out_rows && !out_bf16))
    return KVO_EINVAL;
  if ((out_rows && !aligned16(out_rows)) || (out_bf16 && !aligned16(out_bf16))) return KVO_EINVAL;
  kvo::LayerView v = ctx->views[layer];
  v.evlog = ctx->evlog ? ctx->evlog + kEvlogStride * layer : nullptr;
  v.ram_len = (uint32_t)ctx->ram_len[layer];
  const cudaError_t e =
      kvo::launch_resolve(v, idx, (uint32_t)(nq * k), static_cast<uint8_t*>(out_rows), out_bf16, ctx->status,
                          ctx->max_cluster, static_cast<cudaStream_t>(stream));
  ctx->resolved = true;
  if (e == cudaErrorInvalidValue) return KVO_EINVAL;   // the round does not fit this cluster's shared memory
  return ok(e) ? KVO_OK : KVO_ECUDA;
}

static kvo_status decode_layers_impl(kvo_ctx* ctx, const kvo_layer_task* tasks, int32_t ntasks, int32_t k,
                                     void* stream);

kvo_status kvo_decode_layers(kvo_ctx* ctx, const kvo_layer_task* tasks, int32_t ntasks, int32_t k, void* stream) {
  const auto t0 = std::chrono::steady_clock::now();
  const kvo_status rc = decode_layers_impl(ctx, tasks, ntasks, k, stream);
  if (ctx) ctx->host_seconds += std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count();
  return rc;
}

static kvo_status decode_layers_impl(kvo_ctx* ctx, const kvo_layer_task* tasks, int32_t ntasks, int32_t k,
                                     void* stream) {
  if (ctx && ctx->unusable) return KVO_ECUDA;
  if (!ctx || !tasks || ntasks < 0 || ntasks > ctx->layers || k < 1 || k > KVO_MAX_K || k > ctx->hot_rows)
    return KVO_EINVAL;
  if (ntasks == 0) return KVO_OK;
  static thread_local std::vector<kvo::StepTask> st;
  static thread_local std::vector<uint32_t> lay;
  static thread_local std::vector<uint8_t> seen;
  static thread_local DeviceRanges dev;
  st.resize(ntasks);
  lay.resize(ntasks);
  seen.assign(ctx->layers, 0);
  dev.r.clear();
  for (int32_t i = 0; i < ntasks; ++i) {
    const kvo_layer_task& t = tasks[i];
    if (t.layer < 0 || t.layer >= ctx->layers || seen[t.layer] || t.r < 0 || !t.idx || !aligned4(t.idx) ||
        (t.scores && !aligned4(t.scores)) || (!t.out_rows && !t.out_bf16) || (t.out_rows && !aligned16(t.out_rows)) ||
        (t.out_bf16 && !aligned16(t.out_bf16)))
      return KVO_EINVAL;
    seen[t.layer] = 1;
    lay[i] = (uint32_t)t.layer;
    if (t.r > 0 && (!t.new_rows || !aligned16(t.new_rows) || !dev.check(t.new_rows, (size_t)t.r * KVO_ROW_BYTES)))
      return KVO_EINVAL;
    if (ctx->ring_rows && t.r > (int64_t)ctx->ring_rows - KVO_COPYBACK_BATCH) return KVO_EINVAL;
    const int64_t start = ctx->length[t.layer];
    if (start + t.r > ctx->history_cap) return KVO_EINVAL;
    if (t.scores && (t.n < k || t.n > start + t.r)) return KVO_EINVAL;
    kvo::LayerView v = ctx->views[t.layer];
    v.evlog = ctx->evlog ? ctx->evlog + kEvlogStride * t.layer : nullptr;
    st[i] = kvo::StepTask{v, t.r ? t.new_rows : nullptr, (uint32_t)t.r, (uint32_t)start, t.scores,
                          (uint32_t)(t.scores ? t.n : 0), t.idx, static_cast<uint8_t*>(t.out_rows), t.out_bf16};
  }
  cudaEvent_t* ev = nullptr;
  if (ctx->phase_timing) {
    const size_t need = 4 * (ctx->phase_calls + 1);
    while (ctx->phase_ev.size() < need) {
      cudaEvent_t e = nullptr;
      if (!ok(cudaEventCreate(&e))) return KVO_ECUDA;
      ctx->phase_ev.push_back(e);
    }
    ev = ctx->phase_ev.data() + 4 * ctx->phase_calls;
  }
  if (!ok(upload_statics(ctx))) return KVO_ECUDA;
  const bool batched = ctx->miss_mode == KVO_MISS_BATCHED ||
                       (ctx->miss_mode == KVO_MISS_AUTO && 100.0 * ctx->miss_rate >= ctx->miss_auto_pct);
  if (batched && !ok(ensure_defer(ctx, k))) return KVO_ENOMEM;
  size_t slices = 0;                                     // the selections' filter lists
  for (int32_t i = 0; i < ntasks; ++i)
    if (tasks[i].scores) slices += (size_t)(tasks[i].n + 4095) / 4096;
  if (!ok(ensure_filter(ctx, slices))) return KVO_ENOMEM;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  static thread_local std::vector<int64_t> ram;
  ram.resize(ntasks);
  for (int32_t i = 0; i < ntasks; ++i) {
    if (!ok(copyback_before_step(ctx, tasks[i].layer, tasks[i].r, s, &ram[i]))) return KVO_ECUDA;
    st[i].L.ram_len = (uint32_t)ram[i];
  }
  uint32_t launched = 0;
  const cudaError_t e = kvo::launch_layers(st.data(), lay.data(), (uint32_t)ntasks, (uint32_t)k, ctx->statics,
                                           ctx->status, ctx->max_cluster, s, ev, ctx->first_hist, &ctx->filt,
                                           ctx->ent,
                                           batched ? &ctx->defer : nullptr, &launched);
  if (!ok(e)) return KVO_ECUDA;
  ctx->launches += launched;
  if (ctx->miss_mode == KVO_MISS_AUTO && !ok(measure_miss_rate(ctx, s))) return KVO_ECUDA;
  if (ev) ++ctx->phase_calls;
  ctx->resolved = true;
  for (int32_t i = 0; i < ntasks; ++i) {
    const int32_t l = tasks[i].layer;
    ctx->length[l] += tasks[i].r;
    ctx->ram_len[l] = ram[i];
  }
  return KVO_OK;
}

// Argument checks shared by kvo_decode_step and kvo_decode_step_host (the
// buffers' memory kind is each caller's own check).
static bool decode_step_args_ok(const kvo_ctx* ctx, int32_t layer, const void* new_rows, int64_t r,
                                const float* scores, int64_t n, int32_t k, const int32_t* idx, const void* out_rows,
                                const uint16_t* out_bf16) {
  if (!ctx || layer < 0 || layer >= ctx->layers || r < 0 || !scores || !idx || k < 1 || k > KVO_MAX_K ||
      n < k || n > INT32_MAX || k > ctx->hot_rows || (!out_rows && !out_bf16))
    return false;
  if (!aligned4(scores) || !aligned4(idx)) return false;
  if (r > 0 && !new_rows) return false;
  if (ctx->ring_rows && r > (int64_t)ctx->ring_rows - KVO_COPYBACK_BATCH) return false;
  return ctx->length[layer] + r <= ctx->history_cap;
}

// The step on device buffers (arguments already checked).
static kvo_status decode_step_enqueue(kvo_ctx* ctx, int32_t layer, const void* new_rows, int64_t r,
                                      const float* scores, int64_t n, int32_t k, int32_t* idx, void* out_rows,
                                      uint16_t* out_bf16, cudaStream_t stream, bool out_host = false) {
  const int64_t start = ctx->length[layer];
  kvo::LayerView v = ctx->views[layer];
  v.evlog = ctx->evlog ? ctx->evlog + kEvlogStride * layer : nullptr;
  int64_t ram = 0;
  if (!ok(copyback_before_step(ctx, layer, r, stream, &ram))) return KVO_ECUDA;
  v.ram_len = (uint32_t)ram;
  const cudaError_t e = kvo::launch_decode_step(v, r ? new_rows : nullptr, (uint32_t)r, (uint32_t)start, scores,
                                                (uint32_t)n, (uint32_t)k, idx, static_cast<uint8_t*>(out_rows),
                                                out_bf16, ctx->status, ctx->max_cluster, stream, out_host);
  if (!ok(e)) return KVO_ECUDA;
  ctx->resolved = true;
  ctx->length[layer] = start + r;
  ctx->ram_len[layer] = ram;
  return KVO_OK;
}

kvo_status kvo_decode_step(kvo_ctx* ctx, int32_t layer, const void* new_rows, int64_t r,
                           const float* scores, int64_t n, int32_t k, int32_t* idx,
                           void* out_rows, uint16_t* out_bf16, void* stream) {
  if (ctx && ctx->unusable) return KVO_ECUDA;
  if (!decode_step_args_ok(ctx, layer, new_rows, r, scores, n, k, idx, out_rows, out_bf16)) return KVO_EINVAL;
  if ((out_rows && !aligned16(out_rows)) || (out_bf16 && !aligned16(out_bf16))) return KVO_EINVAL;
  if (r > 0 && (!aligned16(new_rows) || !is_device_pointer(new_rows))) return KVO_EINVAL;
  return decode_step_enqueue(ctx, layer, new_rows, r, scores, n, k, idx, out_rows, out_bf16,
                             static_cast<cudaStream_t>(stream));
}

// The device address of page-locked host memory (the kernels read and write
// it directly over the host link), or NULL for pageable memory.
static void* mapped_host(const void* p) {
  cudaPointerAttributes at;
  if (!p || cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

kvo_status kvo_decode_step_host(kvo_ctx* ctx, int32_t layer, const void* new_rows, int64_t r,
                                const float* scores, int64_t n, int32_t k, int32_t* idx,
                                void* out_rows, uint16_t* out_bf16, void* stream) {
  if (ctx && ctx->unusable) return KVO_ECUDA;
  if (!decode_step_args_ok(ctx, layer, new_rows, r, scores, n, k, idx, out_rows, out_bf16)) return KVO_EINVAL;
  if (is_device_pointer(scores) || is_device_pointer(idx) || (r > 0 && is_device_pointer(new_rows)) ||
      (out_rows && is_device_pointer(out_rows)) || (out_bf16 && is_device_pointer(out_bf16)))
    return KVO_EINVAL;
  // Page-locked buffers are used in place: the step reads the scores and the
  // new rows and writes idx and the outputs over the host link itself, with
  // no copy before or after.  Pageable (or, for rows, unaligned) buffers go
  // through the context's device staging.
  const float* d_scores = static_cast<const float*>(mapped_host(scores));
  const void* d_rows = r > 0 ? mapped_host(new_rows) : nullptr;
  if (d_rows && !aligned16(d_rows)) d_rows = nullptr;
  int32_t* d_idx = static_cast<int32_t*>(mapped_host(idx));
  void* d_out = out_rows ? mapped_host(out_rows) : nullptr;
  if (d_out && !aligned16(d_out)) d_out = nullptr;
  uint16_t* d_bf16 = out_bf16 ? static_cast<uint16_t*>(mapped_host(out_bf16)) : nullptr;
  if (d_bf16 && !aligned16(d_bf16)) d_bf16 = nullptr;
  auto& st = ctx->stage;
  // staging first (sized for the largest call), so that a failure enqueues nothing
  bool good = true;
  if (!d_scores && !st.scores) good = ok(cudaMalloc(&st.scores, sizeof(float) * (size_t)ctx->history_cap));
  if (good && !d_idx && !st.idx) good = ok(cudaMalloc(&st.idx, sizeof(int32_t) * KVO_MAX_K));
  if (good && out_rows && !d_out && !st.out) good = ok(cudaMalloc(&st.out, (size_t)KVO_MAX_K * KVO_ROW_BYTES));
  if (good && out_bf16 && !d_bf16 && !st.bf16)
    good = ok(cudaMalloc(&st.bf16, sizeof(uint16_t) * (size_t)KVO_MAX_K * KVO_DEQUANT_VALUES));
  if (good && r > 0 && !d_rows && r > st.rows_cap) {
    const int64_t cap = r > 2 * st.rows_cap ? r : 2 * st.rows_cap;
    good = ok(cudaDeviceSynchronize());            // earlier steps may still read the old rows
    if (good) {
      cudaFree(st.rows);
      st.rows = nullptr;
      st.rows_cap = 0;
      good = ok(cudaMalloc(&st.rows, (size_t)cap * KVO_ROW_BYTES));
      if (good) st.rows_cap = cap;
    }
  }
  if (!good) {
    cudaGetLastError();
    return KVO_ENOMEM;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (!d_scores) {
    if (!ok(cudaMemcpyAsync(st.scores, scores, sizeof(float) * (size_t)n, cudaMemcpyHostToDevice, s)))
      return KVO_ECUDA;
    d_scores = st.scores;
  }
  if (r > 0 && !d_rows) {
    if (!ok(cudaMemcpyAsync(st.rows, new_rows, (size_t)r * KVO_ROW_BYTES, cudaMemcpyHostToDevice, s)))
      return KVO_ECUDA;
    d_rows = st.rows;
  }
  const bool out_mapped = d_out != nullptr;
  const kvo_status rc = decode_step_enqueue(ctx, layer, d_rows, r, d_scores, n, k, d_idx ? d_idx : st.idx,
                                            out_rows ? (out_mapped ? d_out : st.out) : nullptr,
                                            out_bf16 ? (d_bf16 ? d_bf16 : st.bf16) : nullptr, s, out_mapped);
  if (rc != KVO_OK) return rc;
  if (!d_idx && !ok(cudaMemcpyAsync(idx, st.idx, sizeof(int32_t) * (size_t)k, cudaMemcpyDeviceToHost, s)))
    return KVO_ECUDA;
  if (out_rows && !out_mapped &&
      !ok(cudaMemcpyAsync(out_rows, st.out, (size_t)k * KVO_ROW_BYTES, cudaMemcpyDeviceToHost, s)))
    return KVO_ECUDA;
  if (out_bf16 && !d_bf16 && !ok(cudaMemcpyAsync(out_bf16, st.bf16, sizeof(uint16_t) * (size_t)k * KVO_DEQUANT_VALUES,
                                                 cudaMemcpyDeviceToHost, s)))
    return KVO_ECUDA;
  return KVO_OK;
}

kvo_status kvo_sync(kvo_ctx* ctx, void* stream) {
  if (!ctx) return KVO_EINVAL;
  if (!ok(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)))) return KVO_ECUDA;
  uint32_t st = 0;
  if (!ok(cudaMemcpy(&st, ctx->status, sizeof st, cudaMemcpyDeviceToHost))) return KVO_ECUDA;
  if (st == 0) return KVO_OK;
  if (!ok(cudaMemset(ctx->status, 0, sizeof st))) return KVO_ECUDA;
  if (st & kvo::kFlagInflight) ctx->unusable = true;
  if (st & kvo::kFlagTimeout) return KVO_ETIMEDOUT;
  if (st & kvo::kFlagRange) return KVO_ERANGE;
  return KVO_ECUDA;
}

kvo_status kvo_get_stats(kvo_ctx* ctx, int32_t layer, kvo_stats* out) {
  if (!ctx || !out || layer < 0 || layer >= ctx->layers) return KVO_EINVAL;
  unsigned long long v[8];
  if (!ok(cudaDeviceSynchronize())) return KVO_ECUDA;
  if (!ok(cudaMemcpy(v, ctx->stats + 8 * layer, sizeof v, cudaMemcpyDeviceToHost))) return KVO_ECUDA;
  out->steps = v[0];
  out->hits = v[1];
  out->misses = v[2];
  out->unique_misses = v[3];
  out->evictions = v[4];
  out->invalid = v[5];
  out->host_bytes = v[6];
  out->rows_out = v[7];
  return KVO_OK;
}

kvo_status kvo_history_length(kvo_ctx* ctx, int32_t layer, int64_t* out) {
  if (!ctx || !out || layer < 0 || layer >= ctx->layers) return KVO_EINVAL;
  *out = ctx->length[layer];
  return KVO_OK;
}

kvo_status kvo_debug_dump_layer(kvo_ctx* ctx, int32_t layer, int32_t* pos2slot, int32_t* slot2pos,
                                uint32_t* last_use, void* hot, uint32_t* step) {
  if (!ctx || layer < 0 || layer >= ctx->layers) return KVO_EINVAL;
  const kvo::LayerView& v = ctx->views[layer];
  if (!ok(cudaDeviceSynchronize())) return KVO_ECUDA;
  const size_t H = (size_t)ctx->hot_rows;
  bool good = true;
  if (pos2slot)
    good = good && ok(cudaMemcpy(pos2slot, v.pos2slot, sizeof(int32_t) * (size_t)ctx->history_cap,
                                 cudaMemcpyDeviceToHost));
  if (slot2pos) good = good && ok(cudaMemcpy(slot2pos, v.slot2pos, sizeof(int32_t) * H, cudaMemcpyDeviceToHost));
  if (last_use) good = good && ok(cudaMemcpy(last_use, v.last_use, sizeof(uint32_t) * H, cudaMemcpyDeviceToHost));
  if (hot) good = good && ok(cudaMemcpy(hot, v.hot, H * KVO_ROW_BYTES, cudaMemcpyDeviceToHost));
  if (step) good = good && ok(cudaMemcpy(step, v.counters, sizeof(uint32_t), cudaMemcpyDeviceToHost));
  return good ? KVO_OK : KVO_ECUDA;
}

kvo_status kvo_debug_record_evictions(kvo_ctx* ctx, int32_t on) {
  if (!ctx) return KVO_EINVAL;
  if (!ok(cudaDeviceSynchronize())) return KVO_ECUDA;
  if (on && !ctx->evlog) {
    const size_t bytes = sizeof(int32_t) * kEvlogStride * (size_t)ctx->layers;
    if (!ok(cudaMalloc(&ctx->evlog, bytes))) {
      cudaGetLastError();
      ctx->evlog = nullptr;
      return KVO_ENOMEM;
    }
    if (!ok(cudaMemset(ctx->evlog, 0, bytes))) return KVO_ECUDA;
  } else if (!on && ctx->evlog) {
    cudaFree(ctx->evlog);
    ctx->evlog = nullptr;
  }
  ctx->statics_dirty = true;
  return KVO_OK;
}

kvo_status kvo_debug_evictions(kvo_ctx* ctx, int32_t layer, int32_t* triples, int32_t max,
                               int32_t* count) {
  if (!ctx || !count || layer < 0 || layer >= ctx->layers || max < 0 || (max > 0 && !triples))
    return KVO_EINVAL;
  if (!ctx->evlog) {
    *count = 0;
    return KVO_OK;
  }
  if (!ok(cudaDeviceSynchronize())) return KVO_ECUDA;
  const int32_t* base = ctx->evlog + kEvlogStride * layer;
  int32_t n = 0;
  if (!ok(cudaMemcpy(&n, base, sizeof n, cudaMemcpyDeviceToHost))) return KVO_ECUDA;
  *count = n;
  const int32_t m = n < max ? n : max;
  if (m > 0 && !ok(cudaMemcpy(triples, base + 1, sizeof(int32_t) * 3 * (size_t)m, cudaMemcpyDeviceToHost)))
    return KVO_ECUDA;
  return KVO_OK;
}

kvo_status kvo_probe_host_read(const void* src, int64_t bytes, void* sink, void* stream) {
  return kvo_probe_host_touch(src, bytes, 16, sink, stream);
}

kvo_status kvo_probe_host_touch(const void* src, int64_t bytes, int64_t stride, void* sink, void* stream) {
  if (!src || !sink || bytes <= 0 || (bytes & 15) || stride < 16 || (stride & 15) || !aligned16(src) ||
      !aligned16(sink))
    return KVO_EINVAL;
  void* dev = nullptr;
  if (!ok(cudaHostGetDevicePointer(&dev, const_cast<void*>(src), 0))) {
    cudaGetLastError();
    return KVO_EINVAL;
  }
  return ok(kvo::launch_probe(dev, (uint64_t)bytes, sink, static_cast<cudaStream_t>(stream), (uint64_t)stride))
             ? KVO_OK
             : KVO_ECUDA;
}

kvo_status kvo_touch_history(kvo_ctx* ctx, int32_t layer, void* stream) {
  if (!ctx || layer < -1 || layer >= ctx->layers) return KVO_EINVAL;
  if (ctx->unusable) return KVO_ECUDA;
  if (!ctx->touch_sink && !ok(cudaMalloc(&ctx->touch_sink, 16))) return KVO_ENOMEM;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (int32_t l = layer < 0 ? 0 : layer; l < (layer < 0 ? ctx->layers : layer + 1); ++l) {
    const int64_t bytes = ctx->length[l] * KVO_ROW_BYTES;
    if (bytes <= 0) continue;
    if (!ok(kvo::launch_probe(ctx->views[l].hist, (uint64_t)bytes, ctx->touch_sink, s, 4096))) return KVO_ECUDA;
  }
  return KVO_OK;
}

kvo_status kvo_debug_history_host(kvo_ctx* ctx, int32_t layer, void** out) {
  if (!ctx || !out || layer < 0 || layer >= ctx->layers) return KVO_EINVAL;
  *out = ctx->hist_host[layer];
  return KVO_OK;
}

}  // extern "C"
