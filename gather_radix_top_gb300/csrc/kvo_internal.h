// Host-side internals shared by the kvo translation units (not part of the
// public C ABI).
#pragma once

#include <cstdint>
#include <vector>

#include <cuda_runtime.h>

#include "kvo.h"

namespace kvo {

// Fixed per-layer device pointers (the tables never move after create).
struct LayerView {
  int32_t* pos2slot;              // [history_cap], -1 = not resident
  int32_t* slot2pos;              // [hot_rows],    -1 = empty
  uint32_t* last_use;             // [hot_rows],    0 = never
  uint8_t* hot;                   // [hot_rows * 656]
  const uint8_t* hist;            // device address of the mapped host history
  uint32_t* counters;             // [0] step, [1] history length, [2] queue head, [3] queue tail,
                                  // [4] queue buffer in use, [5] circular hand
  unsigned long long* stats;      // kvo_stats fields, in declaration order
  int32_t* evlog;                 // NULL, or [1 + 3 * KVO_MAX_K]: count then triples
  uint64_t* ring;                 // [2][ring_cap]: LRU queue entries (stamp << 32 | slot), two buffers
  uint32_t hot_rows;
  uint32_t history_cap;
  uint32_t ring_cap;              // entries per queue buffer, a power of two >= 8 * hot_rows
  uint32_t policy;                // KVO_POLICY_LRU or KVO_POLICY_CIRCULAR
  uint8_t* recent;                // NULL, or the recent ring: [ring_rows * 656] in HBM
  uint32_t ring_rows;             // 0, or a power of two: position p waits in slot p mod ring_rows
  uint32_t ram_len;               // per launch: positions below it are in the host history (for a
                                  // launch that appends, the length after its append's copyback)
  uint32_t gather_mode;           // KVO_GATHER_LOADS, KVO_GATHER_STAGED or KVO_GATHER_AUTO
  uint32_t auto_miss_pct;         // KVO_GATHER_AUTO: staged when a CTA's misses are at least this share
};

struct ClusterShape {
  int cluster = 0;                // CTAs per cluster
  size_t smem = 0;                // dynamic shared memory per CTA
};

// Launchers (return a CUDA error code; arguments are validated by the caller).
cudaError_t launch_topk(const float* scores, uint32_t n, uint32_t k, int32_t* idx,
                        int max_cluster, cudaStream_t stream, uint32_t nq = 1, uint64_t ld = 0);
cudaError_t launch_resolve(const LayerView& L, const int32_t* idx, uint32_t k, uint8_t* out_rows,
                           uint16_t* out_bf16, uint32_t* status, int max_cluster,
                           cudaStream_t stream);
// One layer of a batched decode step (kvo_decode_layers).
struct StepTask {
  LayerView L;
  const void* new_rows;           // device rows to append, or NULL
  uint32_t r;
  uint32_t old_len;               // the layer's history length before the append
  const float* scores;            // device scores to select from, or NULL: resolve idx as given
  uint32_t n;
  int32_t* idx;                   // device int32[k]: written with scores, read without
  uint8_t* out_rows;
  uint16_t* out_bf16;
  uint32_t out_host;              // out_rows is mapped host memory (plain stores, never read back)
};
// One layer's fixed device pointers and sizes, as the batched decode step
// reads them from device memory (one entry per layer of a context).
struct LayerStatic {
  int32_t* pos2slot;
  int32_t* slot2pos;
  uint32_t* last_use;
  uint8_t* hot;
  const uint8_t* hist;          // device address of the mapped host history
  uint32_t* counters;
  unsigned long long* stats;
  int32_t* evlog;               // NULL unless evictions are recorded
  uint64_t* ring;               // LRU queue, two buffers of ring_cap entries
  uint8_t* recent;              // recent ring rows, or NULL
  uint32_t hot_rows, history_cap, ring_cap, ring_rows;
};

// The buffers of the batched-copy miss fetch (kvo_set_miss_fetch): lists
// the GPU writes and the host reads, and the reverse, in mapped pinned host
// memory; a device counter per layer; the staging rows; the per-layer host
// history.
struct LayersDefer {
  int2* dlist_dev;              // [layers][KVO_MAX_K] (entry, position), written by the resolves
  const int2* dlist_host;
  uint32_t* dcount_dev;         // [layers], the length of each layer's list
  uint32_t* dcount_host;        // [layers], pinned, copied from dcount_dev
  int2* plist_host;             // [layers][KVO_MAX_K] (entry, staging row), written by the host
  const int2* plist_dev;
  uint32_t* pcount_host;        // [layers]
  const uint32_t* pcount_dev;
  uint8_t* staging;             // device [layers][k][656]
  cudaEvent_t listed;           // the lists are complete
  const uint8_t* const* hist_host;   // [layers]: host address of each layer's history
};

// Words per layer of the batched step's histogram buffer: 2,048 bins, then
// the arrival count and the cut of the whole-GPU histogram launch.
constexpr uint32_t kLayersHistWords = 2048 + 16;

// The whole-GPU filter's lists (device): per slice of 4,096 scores its
// candidates' count, and room for 4,096 keys and positions.
struct LayersFilter {
  uint32_t* count;              // [slices]
  uint32_t* key;                // [slices * 4096]
  uint32_t* pos;                // [slices * 4096]
  size_t slices;
};

// One decode step of many layers in three launches over all of them
// (select, resolve, gather); tasks without scores read their idx after the
// selections.  layers[i]: task i's layer (its entry of `statics`, a device
// array).  ev: NULL, or four events recorded before the selections, before
// the resolves, before the gathers and after them (without events, each
// launch may be scheduled before the previous one ends and waits for it on
// the GPU).  hist: device [layers][kLayersHistWords] words, zero between
// calls (the filtered selections' histograms), or NULL.  filt: NULL, or room
// for the filter's lists of every selecting task (ceil(n / 4096) slices
// each; without it, or without room, a filtered selection filters inside its
// cluster).  ent: device
// [layers][KVO_MAX_K] words, the entry codes the resolves hand to the
// gathers.  defer: NULL for zero-copy loads of the misses, else the
// batched-copy fetch (the host waits for the resolves' lists, then copies
// the missing rows with one cudaMemcpyAsync per run of consecutive
// positions).  *launched grows by the number of kernels launched.
cudaError_t launch_layers(const StepTask* tasks, const uint32_t* layers, uint32_t ntasks, uint32_t k,
                          const LayerStatic* statics, uint32_t* status, int max_cluster, cudaStream_t stream,
                          cudaEvent_t* ev, uint32_t* hist, const LayersFilter* filt, uint32_t* ent,
                          const LayersDefer* defer, uint32_t* launched);
cudaError_t launch_decode_step(const LayerView& L, const void* new_rows, uint32_t r, uint32_t old_len,
                               const float* scores, uint32_t n, uint32_t k, int32_t* idx, uint8_t* out_rows,
                               uint16_t* out_bf16, uint32_t* status, int max_cluster, cudaStream_t stream,
                               bool out_host = false);
cudaError_t launch_append(const void* src_dev, uint8_t* hist_dev_dst, uint64_t bytes,
                          uint32_t* counters, uint32_t new_len, cudaStream_t stream);
cudaError_t launch_ring_append(const void* src_dev, uint8_t* ring, uint32_t r, uint32_t start, uint32_t ring_mask,
                               uint32_t* counters, uint32_t new_len, cudaStream_t stream);
cudaError_t launch_probe(const void* src, uint64_t bytes, void* sink, cudaStream_t stream, uint64_t stride = 16);

// Largest cluster size (16 non-portable, else 8, 4, 2) that can run with the
// given kernel's resources; 0 if none.
int best_cluster(const void* kernel, size_t smem, int want);

}  // namespace kvo
