// residency.cu -- the adapter cache of include/lora_residency.h: a host tier of pinned
// adapter images and a GPU tier of slots shared by a set of layers.
//
// "Serving LoRA adapters: from the model name to the wrapped layer" (vLLM), Step 3: a batch
// may name at most as many adapters as there are GPU slots; an adapter is validated before
// anything is evicted to make room for it; a full CPU cache drops its oldest adapter;
// activation takes the first free slot, or first deactivates the least recently used active
// adapter; a hit only refreshes recency.  "Multi-LoRA Serving: Architecture for Thousands of
// Adapters", sections "Unified paging of adapters and KV cache" and "Trade-offs, Gotchas,
// and What Goes Wrong": all adapters in host DRAM, the active ones fetched into HBM by a
// bus copy, cold ones evicted.
//
// A swap-in moves one adapter image (every layer's slot blocks, already packed on the host
// in the slot layout) with ONE host-to-device copy into a staging buffer, then ONE kernel
// scatters it into the slot of every layer and writes the slots' metadata -- instead of
// two copies and two small kernels per layer -- on the cache's own stream (the lowest
// priority).  Measured beside a pass of the 8B stack (9.3 ms): a swap-in of 80 MiB takes
// 0.44 ms and makes that pass ~0.3 ms longer; a variant with only the copy engines (two
// copies per layer straight into the slots, no scatter kernel) took 1.4 ms, most of it
// host time for the 448 copy calls, and lengthened the pass just as much.
// Ordering is per slot, so that a swap-in overlaps the batch in flight unless it must
// replace one of that batch's adapters:
//   - lora_cache_map_batch(batch, stream) records a point on `stream`: everything enqueued
//     there before it -- the previous batch's forwards -- is the last use of the previous
//     batch's slots.  A swap-in into a slot waits for the last point that covered it.
//   - after making the batch resident, `stream` waits for the swap-ins of the batch's own
//     slots only (not for a prefetch into some other slot).
//   - until the next point, the previous batch's slots are in flight: a prefetch never
//     takes them, and an adapter removed from them leaves its slot blocked (emptied at the
//     next point) instead of rewriting it under a running kernel.
// Pooled layers (lora_layer_create_pooled: adapters at their true rank in a row pool) are
// served too.  A swap-in frees the rows its slot held and takes the adapter's rank rounded
// up to 8 rows, first fit, from each pooled layer's allocator (the cache makes the same
// moves in every pooled layer, so they all place the slot at the same row); the scatter
// copies those rows only and sets the slot's first row.  Rows freed from one slot may be
// reused by another slot while an earlier batch still reads them, so the cache remembers
// per pool row the batch point of its last user, and a swap-in into rows waits for those
// points as it waits for its slot's own.

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <unordered_map>
#include <vector>

#include "layer_state.h"
#include "lora_kernels.h"
#include "lora_layer.h"
#include "lora_residency.h"

namespace {

constexpr size_t kImageAlign = 256;  // every block of an adapter image starts 256-aligned
constexpr int kSwapThreads = 256;

size_t align_up(size_t v) { return (v + kImageAlign - 1) / kImageAlign * kImageAlign; }

// Where one layer's blocks live: in the layer's slot pools, and in an adapter image.
struct SwapDesc {
  char* A_pool;  // [S][R][K] (A transposed, zero-padded)
  char* B_pool;  // [S][R][N]
  float* scale;  // [S][R] column scales
  int32_t* rank;
  int32_t* loaded;
  int R;         // the layer's slot width
  unsigned long long a_bytes, b_bytes;  // one slot's A and B block: R*K and R*N elements
  unsigned long long off_a, off_b;      // offsets of those blocks in the adapter image
  // pooled layers: the slot's rows start at the row the swap-in took (its first row table,
  // null for a plain layer) and number rows (the rank rounded up to 8); bytes of a row
  int32_t* row_base;
  unsigned long long a_row, b_row;
};

// Slot `slot` of every layer (blockIdx.y) from the staged adapter image (copy != 0), and
// the slot's column scales (cols on the r columns of the adapter, 0 beyond), rank and
// loaded flag (copy == 0: only those, to empty the slot).  The blocks are multiples of 16
// bytes (R is a multiple of 8) and start 16-byte aligned.
// Pooled layers: rows `rows` from pool row `rb` (the same in every pooled layer); a plain
// layer ignores both.  The image's blocks hold R rows; a pooled layer takes the first rows.
__global__ void __launch_bounds__(kSwapThreads)
    swap_in_kernel(const SwapDesc* __restrict__ desc, const char* __restrict__ image, int slot,
                   int copy, lora::SlotScales cols, int r, int is_loaded, int rb, int rows) {
  const SwapDesc d = desc[blockIdx.y];
  const bool pooled = d.row_base != nullptr;
  if (copy) {
    const size_t stride = (size_t)gridDim.x * kSwapThreads;
    const size_t first = (size_t)blockIdx.x * kSwapThreads + threadIdx.x;
    const size_t a_bytes = pooled ? (size_t)rows * d.a_row : d.a_bytes;
    const size_t b_bytes = pooled ? (size_t)rows * d.b_row : d.b_bytes;
    const uint4* sa = reinterpret_cast<const uint4*>(image + d.off_a);
    uint4* da = reinterpret_cast<uint4*>(
        d.A_pool + (pooled ? (size_t)rb * d.a_row : (size_t)slot * d.a_bytes));
    for (size_t i = first; i < a_bytes / 16; i += stride) da[i] = __ldg(sa + i);
    const uint4* sb = reinterpret_cast<const uint4*>(image + d.off_b);
    uint4* db = reinterpret_cast<uint4*>(
        d.B_pool + (pooled ? (size_t)rb * d.b_row : (size_t)slot * d.b_bytes));
    for (size_t i = first; i < b_bytes / 16; i += stride) db[i] = __ldg(sb + i);
  }
  if (blockIdx.x == 0) {
    for (int j = threadIdx.x; j < d.R; j += kSwapThreads)
      d.scale[(size_t)slot * d.R + j] = j < r ? cols.v[j] : 0.f;
    if (threadIdx.x == 0) {
      d.rank[slot] = r;
      d.loaded[slot] = is_loaded;
      if (pooled) d.row_base[slot] = is_loaded ? rb : -1;
    }
  }
}

struct Entry {
  int block = -1;          // host block holding the packed image
  int r = 0;               // rank (a composition: the sum of its members' ranks)
  float alpha = 0.f;
  std::vector<float> cols;  // a composition's column scales (empty: alpha / r on all r)
  int slot = -1;           // GPU slot, -1 = not resident
  unsigned long long last_use = 0;
  unsigned long long pin = 0;  // == the cache's pin generation: named by the current request
};

constexpr long long kFree = -1;    // slot_owner: nothing in the slot
constexpr long long kBlocked = -2; // slot_owner: adapter removed while its batch may run

}  // namespace

struct lora_adapter_cache {
  std::vector<lora_layer*> layers;
  int num_slots = 0, host_capacity = 0, device = 0, num_sms = 1, max_r = 0;
  size_t image_bytes = 0;
  std::vector<SwapDesc> desc;   // host copy of the descriptor table
  SwapDesc* desc_dev = nullptr;
  char* arena = nullptr;        // pinned: host_capacity blocks of image_bytes
  char* staging = nullptr;      // device: one image
  cudaStream_t stream = nullptr;
  std::vector<cudaEvent_t> block_ev;    // recorded after the last copy out of the block
  std::vector<char> block_ev_used;
  std::vector<int> free_blocks;         // stack, lowest index on top
  std::unordered_map<long long, Entry> entries;
  std::vector<long long> slot_owner;    // adapter id per slot, or kFree / kBlocked
  // per-slot ordering
  std::vector<cudaEvent_t> ready_ev;    // recorded after the slot's last swap-in / emptying
  std::vector<char> ready_pending;      // ... not yet waited for by a batch stream
  std::vector<int> busy_point;          // batch point covering the slot's last use, -1 none
  std::vector<cudaEvent_t> point_ev;    // batch points, shared by slots (reference counted)
  std::vector<int> point_refs;
  std::vector<int> last_slots;          // slots of the last mapped batch (maybe in flight)
  std::vector<long long> last_names;    // its adapters
  // pooled layers (all with the same row pool, moved in step): per pool row, the batch point
  // of the last slot that held it and gave it back (-1: none pending); each entry holds a
  // reference on that point
  bool any_pooled = false;
  std::vector<int> row_point;
  unsigned long long clock = 0, pin_gen = 0;
  lora_cache_stats_t stats{};
  char last_error[512] = {0};
};

namespace {

using Cache = lora_adapter_cache;

int fail(Cache* c, int code, const char* fmt, ...) {
  if (c) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(c->last_error, sizeof(c->last_error), fmt, ap);
    va_end(ap);
  }
  return code;
}

#define CACHE_CUDA(C, expr)                                                          \
  do {                                                                               \
    cudaError_t e_ = (expr);                                                         \
    if (e_ != cudaSuccess)                                                           \
      return fail((C), LORA_ECUDA, "%s: %s", #expr, cudaGetErrorString(e_));         \
  } while (0)

void free_cache(Cache* c) {
  if (c->stream) cudaStreamSynchronize(c->stream);
  for (cudaEvent_t e : c->block_ev)
    if (e) cudaEventDestroy(e);
  for (cudaEvent_t e : c->ready_ev)
    if (e) cudaEventDestroy(e);
  for (cudaEvent_t e : c->point_ev)
    if (e) cudaEventDestroy(e);
  if (c->arena) cudaFreeHost(c->arena);
  if (c->staging) cudaFree(c->staging);
  if (c->desc_dev) cudaFree(c->desc_dev);
  if (c->stream) cudaStreamDestroy(c->stream);
}

// The cache's stream waits for the end of the slot's last use.
int wait_slot_idle(Cache* c, int slot) {
  if (c->busy_point[slot] >= 0)
    CACHE_CUDA(c, cudaStreamWaitEvent(c->stream, c->point_ev[c->busy_point[slot]], 0));
  return LORA_OK;
}

int swap_grid_x(const Cache* c) {
  const int n = (int)c->layers.size();
  return std::max(1, std::min(1024, (4 * c->num_sms + n - 1) / n));
}

// Pooled layers: `slot` gives back the rows it holds (in every pooled layer, where they are
// the same rows); until a swap-in takes them again they remember the slot's last use.
void give_back_rows(Cache* c, int slot) {
  if (!c->any_pooled) return;
  int first = -1, rows = 0;
  for (lora_layer* L : c->layers)
    if (L->pooled) lora::layer_release_rows(L, slot, &first, &rows);
  const int p = c->busy_point[slot];
  for (int i = 0; i < rows; ++i) {
    int& rp = c->row_point[first + i];
    if (rp >= 0) --c->point_refs[rp];
    rp = p;
    if (p >= 0) ++c->point_refs[p];
  }
}

// Pooled layers: `rows` rows for `slot` (holding none) in every pooled layer, and the
// cache's stream made to wait for the last users of those rows.  *first: the first row.
int take_rows(Cache* c, int slot, int rows, int* first) {
  *first = 0;
  if (!c->any_pooled) return LORA_OK;
  int rb = -2;
  for (lora_layer* L : c->layers) {
    if (!L->pooled) continue;
    const int got = lora::layer_take_rows(L, slot, rows);
    if (got < 0 || (rb != -2 && got != rb)) {  // no run of free rows (or pools out of step)
      for (lora_layer* M : c->layers) {
        int f = 0, n = 0;
        if (M->pooled) lora::layer_release_rows(M, slot, &f, &n);
      }
      return fail(c, LORA_ENOMEM, "the row pools have no %d free consecutive rows", rows);
    }
    rb = got;
  }
  std::vector<int> waited;
  for (int i = 0; i < rows; ++i) {
    int& rp = c->row_point[rb + i];
    if (rp < 0) continue;
    if (std::find(waited.begin(), waited.end(), rp) == waited.end()) {
      CACHE_CUDA(c, cudaStreamWaitEvent(c->stream, c->point_ev[rp], 0));
      waited.push_back(rp);
    }
    --c->point_refs[rp];
    rp = -1;
  }
  *first = rb;
  return LORA_OK;
}

// Copy adapter e's image into `slot` of every layer.  LORA_ENOMEM: a pooled layer has no
// run of rows for it; the slot is then left empty.
int swap_in(Cache* c, const Entry& e, int slot) {
  if (c->layers.empty()) return LORA_OK;
  int rc = wait_slot_idle(c, slot);
  if (rc != LORA_OK) return rc;
  // pooled layers: the rows of the slot's previous adapter go back, the new adapter's rank
  // rounded up to 8 rows are taken
  const int rows = (e.r + 7) / 8 * 8;
  int rb = 0;
  if (c->any_pooled) {
    give_back_rows(c, slot);
    rc = take_rows(c, slot, rows, &rb);
    if (rc != LORA_OK) {  // the slot holds no rows now: empty it in every layer
      lora::SlotScales none;
      for (int j = 0; j < lora::kMaxSlotRank; ++j) none.v[j] = 0.f;
      swap_in_kernel<<<dim3(1, (unsigned)c->layers.size()), kSwapThreads, 0, c->stream>>>(
          c->desc_dev, c->staging, slot, 0, none, 0, 0, 0, 0);
      for (lora_layer* L : c->layers) lora::layer_set_percol(L, slot, false);
      return rc;
    }
  }
  CACHE_CUDA(c, cudaMemcpyAsync(c->staging, c->arena + (size_t)e.block * c->image_bytes,
                                c->image_bytes, cudaMemcpyHostToDevice, c->stream));
  CACHE_CUDA(c, cudaEventRecord(c->block_ev[e.block], c->stream));
  c->block_ev_used[e.block] = 1;
  lora::SlotScales cols;
  bool varied = false;
  for (int j = 0; j < lora::kMaxSlotRank; ++j)
    cols.v[j] = j >= e.r ? 0.f : e.cols.empty() ? e.alpha / (float)e.r : e.cols[j];
  for (int j = 1; j < e.r; ++j) varied |= cols.v[j] != cols.v[0];
  dim3 grid(swap_grid_x(c), (unsigned)c->layers.size());
  swap_in_kernel<<<grid, kSwapThreads, 0, c->stream>>>(c->desc_dev, c->staging, slot, 1, cols,
                                                       e.r, 1, rb, rows);
  CACHE_CUDA(c, cudaGetLastError());
  // layers that expand v on the tensor cores keep a transposed copy of B per slot
  for (lora_layer* L : c->layers)
    if (L->Bx_pool) {
      const size_t es = L->esize;
      const size_t first_row = L->pooled ? (size_t)rb : (size_t)slot * L->R;
      CACHE_CUDA(c, lora::launch_pack_bx(
                        static_cast<char*>(L->B_pool) + first_row * L->N * es,
                        static_cast<char*>(L->Bx_pool) +
                            (size_t)slot * L->N * lora::expand_layout(L->R).wx * es,
                        L->R, L->pooled ? rows : L->R, L->N, c->stream));
    }
  CACHE_CUDA(c, cudaEventRecord(c->ready_ev[slot], c->stream));
  c->ready_pending[slot] = 1;
  for (lora_layer* L : c->layers) lora::layer_set_percol(L, slot, varied);
  c->stats.bytes_swapped += (int64_t)c->image_bytes;
  return LORA_OK;
}

// Mark `slot` empty in every layer now (rows still naming it are flagged, base only).
int empty_slot(Cache* c, int slot) {
  c->slot_owner[slot] = kFree;
  if (c->layers.empty()) return LORA_OK;
  int rc = wait_slot_idle(c, slot);
  if (rc != LORA_OK) return rc;
  lora::SlotScales none;
  for (int j = 0; j < lora::kMaxSlotRank; ++j) none.v[j] = 0.f;
  swap_in_kernel<<<dim3(1, (unsigned)c->layers.size()), kSwapThreads, 0, c->stream>>>(
      c->desc_dev, c->staging, slot, 0, none, 0, 0, 0, 0);
  CACHE_CUDA(c, cudaGetLastError());
  for (lora_layer* L : c->layers) lora::layer_set_percol(L, slot, false);
  give_back_rows(c, slot);  // pooled layers: after the slot's last use
  CACHE_CUDA(c, cudaEventRecord(c->ready_ev[slot], c->stream));
  c->ready_pending[slot] = 1;
  return LORA_OK;
}

bool in_flight(const Cache* c, int slot) {
  return std::find(c->last_slots.begin(), c->last_slots.end(), slot) != c->last_slots.end();
}

// An adapter leaves `slot`: empty it now, or at the next batch point if the last mapped
// batch (maybe still running) uses it.
int release_slot(Cache* c, int slot) {
  if (in_flight(c, slot)) {
    c->slot_owner[slot] = kBlocked;
    return LORA_OK;
  }
  return empty_slot(c, slot);
}

// A point on `stream` after the last mapped batch's forwards: the end of its slots' use.
// Blocked slots are emptied after it.
int batch_point(Cache* c, cudaStream_t stream) {
  if (!c->last_slots.empty() && !c->layers.empty()) {
    int p = -1;
    for (size_t i = 0; i < c->point_ev.size() && p < 0; ++i)
      if (c->point_refs[i] == 0) p = (int)i;
    if (p < 0) {
      cudaEvent_t ev = nullptr;
      CACHE_CUDA(c, cudaEventCreateWithFlags(&ev, cudaEventDisableTiming));
      c->point_ev.push_back(ev);
      c->point_refs.push_back(0);
      p = (int)c->point_ev.size() - 1;
    }
    CACHE_CUDA(c, cudaEventRecord(c->point_ev[p], stream));
    for (int s : c->last_slots) {
      if (c->busy_point[s] >= 0) --c->point_refs[c->busy_point[s]];
      c->busy_point[s] = p;
      ++c->point_refs[p];
    }
  }
  const std::vector<int> done = c->last_slots;
  c->last_slots.clear();
  c->last_names.clear();
  for (int s : done)
    if (c->slot_owner[s] == kBlocked) {
      const int rc = empty_slot(c, s);
      if (rc != LORA_OK) return rc;
    }
  return LORA_OK;
}

// Pin the adapters `ids` and (for a prefetch) the last batch's; slots that can take a new
// adapter: free ones, and those of unpinned resident adapters.
int mark_pins(Cache* c, const std::vector<long long>& ids, bool with_last) {
  ++c->pin_gen;
  for (long long id : ids) c->entries[id].pin = c->pin_gen;
  if (with_last)
    for (long long id : c->last_names) {
      auto it = c->entries.find(id);
      if (it != c->entries.end()) it->second.pin = c->pin_gen;
    }
  int avail = 0;
  for (long long o : c->slot_owner)
    if (o == kFree || (o >= 0 && c->entries[o].pin != c->pin_gen)) ++avail;
  return avail;
}

// Make the adapters `ids` (distinct, registered, pinned by mark_pins) resident, in order.
int make_resident(Cache* c, const std::vector<long long>& ids, bool batch) {
  for (long long id : ids) {
    Entry& e = c->entries[id];
    if (e.slot >= 0) {
      if (batch) ++c->stats.hits;
      e.last_use = ++c->clock;
      continue;
    }
    int slot = -1;
    for (int s = 0; s < c->num_slots && slot < 0; ++s)
      if (c->slot_owner[s] == kFree) slot = s;
    if (slot < 0) {  // the least recently used resident adapter the request does not pin
      Entry* victim = nullptr;
      for (int s = 0; s < c->num_slots; ++s) {
        if (c->slot_owner[s] < 0) continue;
        auto it = c->entries.find(c->slot_owner[s]);
        if (it == c->entries.end()) continue;
        Entry& o = it->second;
        if (o.pin != c->pin_gen && (!victim || o.last_use < victim->last_use)) victim = &o;
      }
      if (!victim) return fail(c, LORA_ECAPACITY, "no slot can take adapter %lld", id);
      slot = victim->slot;
      victim->slot = -1;
      ++c->stats.gpu_evictions;
    }
    c->slot_owner[slot] = id;
    e.slot = slot;
    e.last_use = ++c->clock;
    if (batch) ++c->stats.misses;
    else ++c->stats.prefetches;
    const int rc = swap_in(c, e, slot);
    if (rc != LORA_OK) {
      if (rc == LORA_ENOMEM) {  // the slot was left empty
        c->slot_owner[slot] = kFree;
        e.slot = -1;
      }
      return rc;
    }
  }
  return LORA_OK;
}

// dst[j][k] = src[k][j] for j < r, k < K, in blocks of 64 k so that the r source rows of a
// block stay in the cache while its r destination rows are written.
template <typename E>
void transpose_rows(E* dst, const E* src, size_t K, int r) {
  for (size_t k0 = 0; k0 < K; k0 += 64) {
    const size_t k1 = std::min(K, k0 + 64);
    for (int j = 0; j < r; ++j) {
      E* d = dst + (size_t)j * K;
      for (size_t k = k0; k < k1; ++k) d[k] = src[k * r + j];
    }
  }
}

// Pack adapter (A_l [K,r], B_l [r,N] per layer) into the host block: At [R][K] with rows
// >= r zero, B [R][N] with rows >= r zero, at the layer's offsets.
void pack_image(const Cache* c, char* blk, int r, const void* const* A_host,
                const void* const* B_host) {
  for (size_t l = 0; l < c->layers.size(); ++l) {
    const lora_layer* L = c->layers[l];
    const size_t es = L->esize, K = L->K, N = L->N, R = L->R;
    char* at = blk + c->desc[l].off_a;
    const char* A = static_cast<const char*>(A_host[l]);
    // At[j][k] = A[k][j]: typed element copies (a memcpy call per element would dominate)
    if (es == 2)
      transpose_rows(reinterpret_cast<uint16_t*>(at), reinterpret_cast<const uint16_t*>(A), K, r);
    else
      transpose_rows(reinterpret_cast<uint32_t*>(at), reinterpret_cast<const uint32_t*>(A), K, r);
    memset(at + (size_t)r * K * es, 0, (R - r) * K * es);
    char* b = blk + c->desc[l].off_b;
    memcpy(b, B_host[l], (size_t)r * N * es);
    memset(b + (size_t)r * N * es, 0, (R - r) * N * es);
  }
}

bool is_device_memory(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeDevice;
}

// Drop entry `id` from the host tier (and its slot).
int drop(Cache* c, long long id) {
  Entry& e = c->entries[id];
  if (e.slot >= 0) {
    const int rc = release_slot(c, e.slot);
    if (rc != LORA_OK) return rc;
  }
  c->free_blocks.push_back(e.block);
  std::sort(c->free_blocks.begin(), c->free_blocks.end(), std::greater<int>());
  c->entries.erase(id);
  return LORA_OK;
}

// Distinct ids in order of first appearance, checked: -1 skipped when allow_base, other
// negatives EINVAL, unknown ENOENT.
int distinct_ids(Cache* c, const int64_t* ids, int n, bool allow_base,
                 std::vector<long long>& out) {
  std::unordered_map<long long, int> seen;
  for (int i = 0; i < n; ++i) {
    const long long id = ids[i];
    if (id == -1 && allow_base) continue;
    if (id < 0) return fail(c, LORA_EINVAL, "entry %d: adapter id %lld", i, id);
    if (c->entries.find(id) == c->entries.end())
      return fail(c, LORA_ENOENT, "entry %d: adapter %lld is not in the cache", i, id);
    if (seen.emplace(id, 0).second) out.push_back(id);
  }
  return LORA_OK;
}

}  // namespace

extern "C" {

int lora_cache_create(lora_adapter_cache_t** out, lora_layer_t* const* layers, int n_layers,
                      int num_slots, int host_capacity) {
  if (!out) return LORA_EINVAL;
  *out = nullptr;
  if (n_layers < 0 || (n_layers > 0 && !layers) || num_slots < 1 || host_capacity < num_slots)
    return LORA_EINVAL;
  Cache* c = new (std::nothrow) Cache();
  if (!c) return LORA_ENOMEM;
  auto bail = [&](int code) {
    free_cache(c);
    delete c;
    return code;
  };
  c->num_slots = num_slots;
  c->host_capacity = host_capacity;
  c->max_r = 1 << 30;
  size_t off = 0;
  for (int l = 0; l < n_layers; ++l) {
    lora_layer* L = layers[l];
    if (!L || num_slots > L->S) return bail(LORA_EINVAL);
    if (l > 0 && L->device != c->layers[0]->device) return bail(LORA_EINVAL);
    if (L->pooled) {
      // pooled layers move in step: the same row pool, and no slot holding rows yet
      for (int q = 0; q < L->S; ++q)
        if (L->rows_h[q] > 0) return bail(LORA_EINVAL);
      if (c->any_pooled && (int)c->row_point.size() != L->P) return bail(LORA_EINVAL);
      c->any_pooled = true;
      c->row_point.assign(L->P, -1);
    }
    c->layers.push_back(L);
    c->max_r = std::min(c->max_r, L->max_rank);
    SwapDesc d;
    d.A_pool = static_cast<char*>(L->A_pool);
    d.B_pool = static_cast<char*>(L->B_pool);
    d.scale = L->scale;
    d.rank = L->rank;
    d.loaded = L->loaded;
    d.R = L->R;
    d.a_bytes = (unsigned long long)L->R * L->K * L->esize;
    d.b_bytes = (unsigned long long)L->R * L->N * L->esize;
    d.off_a = off;
    off = align_up(off + d.a_bytes);
    d.off_b = off;
    off = align_up(off + d.b_bytes);
    d.row_base = L->pooled ? L->row_base : nullptr;
    d.a_row = (unsigned long long)L->K * L->esize;
    d.b_row = (unsigned long long)L->N * L->esize;
    c->desc.push_back(d);
  }
  if (n_layers == 0) c->max_r = 1 << 30;
  c->image_bytes = off;
  c->slot_owner.assign(num_slots, -1);
  for (int b = host_capacity - 1; b >= 0; --b) c->free_blocks.push_back(b);
  c->block_ev.assign(host_capacity, nullptr);
  c->block_ev_used.assign(host_capacity, 0);
  c->ready_ev.assign(num_slots, nullptr);
  c->ready_pending.assign(num_slots, 0);
  c->busy_point.assign(num_slots, -1);
  if (n_layers > 0) {
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess || cur != c->layers[0]->device)
      return bail(LORA_EINVAL);  // the layers' device must be current
    c->device = cur;
    c->num_sms = std::max(1, c->layers[0]->num_sms);
    if (cudaHostAlloc(reinterpret_cast<void**>(&c->arena), (size_t)host_capacity * c->image_bytes,
                      cudaHostAllocPortable) != cudaSuccess ||
        cudaMalloc(reinterpret_cast<void**>(&c->staging), c->image_bytes) != cudaSuccess ||
        cudaMalloc(reinterpret_cast<void**>(&c->desc_dev), sizeof(SwapDesc) * n_layers) !=
            cudaSuccess) {
      cudaGetLastError();
      return bail(LORA_ENOMEM);
    }
    // swap-ins are background work: the lowest priority, so that the scatter's CTAs take
    // SMs only after the forwards' pending CTAs
    int least = 0, greatest = 0;
    if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess ||
        cudaStreamCreateWithPriority(&c->stream, cudaStreamNonBlocking, least) != cudaSuccess)
      return bail(LORA_ECUDA);
    for (int b = 0; b < host_capacity; ++b)
      if (cudaEventCreateWithFlags(&c->block_ev[b], cudaEventDisableTiming) != cudaSuccess)
        return bail(LORA_ECUDA);
    for (int q = 0; q < num_slots; ++q)
      if (cudaEventCreateWithFlags(&c->ready_ev[q], cudaEventDisableTiming) != cudaSuccess)
        return bail(LORA_ECUDA);
    if (cudaMemcpyAsync(c->desc_dev, c->desc.data(), sizeof(SwapDesc) * n_layers,
                        cudaMemcpyHostToDevice, c->stream) != cudaSuccess ||
        cudaStreamSynchronize(c->stream) != cudaSuccess)
      return bail(LORA_ECUDA);
  }
  *out = c;
  return LORA_OK;
}

}  // extern "C"

namespace {

// Take a host block for adapter `id` (its own block if it is held already: the adapter is
// replaced in place and its slot emptied; else a free block, dropping the least recently
// used adapter -- never one of `keep` -- if the tier is full) and wait until no swap-in
// still reads it.  The caller has checked the adapter; only now is room made.
int take_block(Cache* c, long long id, const std::vector<long long>& keep, int* block) {
  auto it = c->entries.find(id);
  if (it != c->entries.end()) {  // in-place replacement
    *block = it->second.block;
    if (it->second.slot >= 0) {
      const int rc = release_slot(c, it->second.slot);
      if (rc != LORA_OK) return rc;
      it->second.slot = -1;
    }
  } else {
    if (c->free_blocks.empty()) {
      long long oldest = -1;
      unsigned long long t = ~0ull;
      for (const auto& kv : c->entries)
        if (kv.second.last_use < t &&
            std::find(keep.begin(), keep.end(), kv.first) == keep.end()) {
          t = kv.second.last_use;
          oldest = kv.first;
        }
      if (oldest < 0) return fail(c, LORA_ECAPACITY, "no host block can be freed");
      const int rc = drop(c, oldest);
      if (rc != LORA_OK) return rc;
      ++c->stats.host_evictions;
    }
    *block = c->free_blocks.back();
    c->free_blocks.pop_back();
  }
  if (!c->layers.empty() && c->block_ev_used[*block])
    CACHE_CUDA(c, cudaEventSynchronize(c->block_ev[*block]));
  return LORA_OK;
}

}  // namespace

extern "C" {

int lora_cache_add(lora_adapter_cache_t* c, int64_t id, int r, float alpha,
                   const void* const* A_host, const void* const* B_host) {
  if (!c) return LORA_EINVAL;
  if (id < 0) return fail(c, LORA_EINVAL, "adapter id %lld < 0", (long long)id);
  if (r < 1 || r > c->max_r)
    return fail(c, LORA_ERANK, "rank %d outside [1, %d]", r, c->max_r);
  if (!c->layers.empty()) {
    if (!A_host || !B_host) return fail(c, LORA_EINVAL, "null weight arrays");
    for (size_t l = 0; l < c->layers.size(); ++l) {
      if (!A_host[l] || !B_host[l]) return fail(c, LORA_EINVAL, "null weights of layer %zu", l);
      if (is_device_memory(A_host[l]) || is_device_memory(B_host[l]))
        return fail(c, LORA_EINVAL, "layer %zu: weights must be in host memory", l);
    }
  }
  // the adapter is valid: only now make room for it
  int block = -1;
  const int rc = take_block(c, id, {}, &block);
  if (rc != LORA_OK) return rc;
  if (!c->layers.empty())
    pack_image(c, c->arena + (size_t)block * c->image_bytes, r, A_host, B_host);
  Entry& e = c->entries[id];
  e.block = block;
  e.r = r;
  e.alpha = alpha;
  e.cols.clear();
  e.slot = -1;
  e.last_use = ++c->clock;
  return LORA_OK;
}

int lora_cache_add_composed(lora_adapter_cache_t* c, int64_t id, int n,
                            const int64_t* member_ids, const float* weights) {
  if (!c) return LORA_EINVAL;
  if (id < 0) return fail(c, LORA_EINVAL, "adapter id %lld < 0", (long long)id);
  if (n < 1 || !member_ids || !weights) return fail(c, LORA_EINVAL, "bad composition");
  int r_sum = 0;
  std::vector<long long> members;
  for (int m = 0; m < n; ++m)
    if (member_ids[m] == id)
      return fail(c, LORA_EINVAL, "a composition cannot name its own id");
  for (int m = 0; m < n; ++m) {
    auto it = c->entries.find(member_ids[m]);
    if (it == c->entries.end())
      return fail(c, LORA_ENOENT, "member %lld is not in the cache", (long long)member_ids[m]);
    r_sum += it->second.r;
    members.push_back(member_ids[m]);
  }
  if (r_sum > c->max_r)
    return fail(c, LORA_ERANK, "composed rank %d above %d", r_sum, c->max_r);
  // the members' column scales, weighted, in member order
  std::vector<float> cols;
  for (int m = 0; m < n; ++m) {
    const Entry& me = c->entries[members[m]];
    for (int j = 0; j < me.r; ++j)
      cols.push_back(weights[m] * (me.cols.empty() ? me.alpha / (float)me.r : me.cols[j]));
  }
  int block = -1;
  const int rc = take_block(c, id, members, &block);  // never drops a member
  if (rc != LORA_OK) return rc;
  if (!c->layers.empty()) {
    // rank rows of member m follow those of members 0 .. m-1, in every layer's blocks
    char* dst = c->arena + (size_t)block * c->image_bytes;
    for (size_t l = 0; l < c->layers.size(); ++l) {
      const lora_layer* L = c->layers[l];
      const size_t es = L->esize, K = L->K, N = L->N, R = L->R;
      size_t o = 0;
      for (int m = 0; m < n; ++m) {
        const Entry& me = c->entries[members[m]];
        const char* src = c->arena + (size_t)me.block * c->image_bytes;
        memmove(dst + c->desc[l].off_a + o * K * es, src + c->desc[l].off_a, me.r * K * es);
        memmove(dst + c->desc[l].off_b + o * N * es, src + c->desc[l].off_b, me.r * N * es);
        o += me.r;
      }
      memset(dst + c->desc[l].off_a + o * K * es, 0, (R - o) * K * es);
      memset(dst + c->desc[l].off_b + o * N * es, 0, (R - o) * N * es);
    }
  }
  Entry& e = c->entries[id];
  e.block = block;
  e.r = r_sum;
  e.alpha = 0.f;
  e.cols = cols;
  e.slot = -1;
  e.last_use = ++c->clock;
  return LORA_OK;
}

int lora_cache_remove(lora_adapter_cache_t* c, int64_t id) {
  if (!c) return LORA_EINVAL;
  if (c->entries.find(id) == c->entries.end())
    return fail(c, LORA_ENOENT, "adapter %lld is not in the cache", (long long)id);
  return drop(c, id);
}

int lora_cache_map_batch(lora_adapter_cache_t* c, const int64_t* token_adapter, int T,
                         int32_t* token_slot, void* stream_) {
  if (!c) return LORA_EINVAL;
  if (T < 0 || (T > 0 && (!token_adapter || !token_slot)))
    return fail(c, LORA_EINVAL, "bad batch arguments");
  std::vector<long long> names;
  int rc = distinct_ids(c, token_adapter, T, true, names);
  if (rc != LORA_OK) return rc;
  if ((int)names.size() > c->num_slots)
    return fail(c, LORA_ECAPACITY, "the batch names %zu adapters; %d GPU slots", names.size(),
                c->num_slots);
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  rc = batch_point(c, stream);
  if (rc != LORA_OK) return rc;
  mark_pins(c, names, false);  // with no batch in flight every slot can serve the batch
  rc = make_resident(c, names, true);
  if (rc != LORA_OK) return rc;
  for (long long id : names) {
    const int s = c->entries[id].slot;
    if (c->ready_pending[s]) {  // the batch's forwards wait for its own slots' swap-ins
      CACHE_CUDA(c, cudaStreamWaitEvent(stream, c->ready_ev[s], 0));
      c->ready_pending[s] = 0;
    }
    c->last_slots.push_back(s);
  }
  c->last_names = names;
  for (int i = 0; i < T; ++i)
    token_slot[i] = token_adapter[i] == -1 ? -1 : c->entries[token_adapter[i]].slot;
  return LORA_OK;
}

int lora_cache_prefetch(lora_adapter_cache_t* c, const int64_t* ids, int n) {
  if (!c) return LORA_EINVAL;
  if (n < 0 || (n > 0 && !ids)) return fail(c, LORA_EINVAL, "bad prefetch arguments");
  std::vector<long long> names;
  const int rc = distinct_ids(c, ids, n, false, names);
  if (rc != LORA_OK) return rc;
  // the last batch's adapters stay put (it may still run); the rest must fit around them
  const int avail = mark_pins(c, names, true);
  int missing = 0;
  for (long long id : names) missing += c->entries[id].slot < 0;
  if (missing > avail)
    return fail(c, LORA_ECAPACITY, "%d adapters to swap in; %d slots can take one", missing,
                avail);
  return make_resident(c, names, false);
}

int lora_cache_slot_of(const lora_adapter_cache_t* c, int64_t id) {
  if (!c) return -1;
  auto it = c->entries.find(id);
  return it == c->entries.end() ? -1 : it->second.slot;
}

int lora_cache_get_stats(const lora_adapter_cache_t* c, lora_cache_stats_t* out) {
  if (!c || !out) return LORA_EINVAL;
  *out = c->stats;
  int resident = 0;
  for (long long o : c->slot_owner) resident += o >= 0;
  out->resident = resident;
  out->registered = (int32_t)c->entries.size();
  return LORA_OK;
}

void* lora_cache_stream(const lora_adapter_cache_t* c) { return c ? c->stream : nullptr; }

int lora_cache_sync(lora_adapter_cache_t* c) {
  if (!c) return LORA_EINVAL;
  if (c->stream) CACHE_CUDA(c, cudaStreamSynchronize(c->stream));
  return LORA_OK;
}

const char* lora_cache_last_error(const lora_adapter_cache_t* c) {
  return c ? c->last_error : "null cache";
}

void lora_cache_destroy(lora_adapter_cache_t* c) {
  if (!c) return;
  free_cache(c);
  delete c;
}

}  // extern "C"
