// static_scratch.cu -- the segment builder for callers that cannot allocate device memory.
//
// Some callers of this library must not call cudaMalloc: a framework or serving engine that
// owns all device memory through its own pool or memory plan and forbids allocations behind
// its back, or a latency-critical path where cudaMalloc's implicit device-wide
// synchronisation is unacceptable.  Such callers cannot create a lora_layer (it allocates
// its slot table and batch scratch), but they can still use the segment builder through
// lora_build_segments_static: they pass the ids and their own output buffers, and the
// builder's scratch -- the checked slot of every row, the work-tile lists, the counters and
// the error flags -- lives in one file-scope device array below, sized for at most
// kStaticMaxTokens rows and kStaticMaxSlots slots.
//
// Every GPU that loads this library holds that array (96 KB) until the process exits.  All
// calls on a device share it and it keeps the last call's contents; calls whose work
// overlaps on the GPU (other streams, or other host threads) race on it and must be
// serialised by the caller.
#include <cuda_runtime.h>

#include <mutex>

#include "lora_common.cuh"
#include "lora_kernels.h"
#include "lora_layer.h"

namespace {

constexpr int kStaticMaxTokens = 16384;
constexpr int kStaticMaxSlots = 1024;
constexpr int kStaticMaxTiles = kStaticMaxTokens / lora::kTileRows + kStaticMaxSlots;
// int32 layout of the scratch array
constexpr int kOffRowSlot = 0;                                   // [kStaticMaxTokens]
constexpr int kOffTileSeg = kOffRowSlot + kStaticMaxTokens;      // [kStaticMaxTiles]
constexpr int kOffTileRow0 = kOffTileSeg + kStaticMaxTiles;      // [kStaticMaxTiles]
constexpr int kOffMeta = kOffTileRow0 + kStaticMaxTiles;         // [4] n_seg, n_adapted, tiles
constexpr int kOffErr = kOffMeta + 4;                            // [4] error flags (first int)
constexpr int kOffAllLoaded = kOffErr + 4;                       // [kStaticMaxSlots] nonzero
constexpr int kScratchInts = kOffAllLoaded + kStaticMaxSlots;    // 22536 ints
constexpr int kScratchIntsAlloc = 24576;                         // 96 KB
static_assert(kScratchInts <= kScratchIntsAlloc, "scratch layout exceeds the array");

// The scratch array.  In host code this name is only a host-side stand-in for the device
// symbol; its device address comes from cudaGetSymbolAddress (scratch_address below).
static __device__ __align__(256) int32_t g_builder_scratch[kScratchIntsAlloc];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
int32_t* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device, looked up once per device
// (with that device current) on the first call made there.
cudaError_t scratch_address(int32_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_builder_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = static_cast<int32_t*>(p);
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" int lora_build_segments_static(const int32_t* token_slot_dev, int T, int num_slots,
                                          const int32_t* slot_loaded_dev, int32_t* perm_dev,
                                          int32_t* seg_offsets_dev, int32_t* seg_slot_dev,
                                          int32_t* counts_dev, void* stream_) {
  if (T < 0 || T > kStaticMaxTokens) return LORA_EINVAL;  // more rows than the array holds
  if (num_slots < 1 || num_slots > kStaticMaxSlots) return LORA_EINVAL;
  if ((T > 0 && (!token_slot_dev || !perm_dev)) || !seg_offsets_dev || !seg_slot_dev ||
      !counts_dev)
    return LORA_EINVAL;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  int32_t* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return LORA_ECUDA;

  int32_t* err = scratch + kOffErr;
  int32_t* meta = scratch + kOffMeta;
  // the error flags accumulate with atomic ORs: clear them (the array keeps the last
  // call's contents); everything else the builder writes in full on every call
  if (cudaMemsetAsync(err, 0, sizeof(int32_t), stream) != cudaSuccess) return LORA_ECUDA;
  const int32_t* loaded = slot_loaded_dev;
  if (!loaded) {  // every slot in range counts as holding an adapter
    if (cudaMemsetAsync(scratch + kOffAllLoaded, 0x01, sizeof(int32_t) * num_slots, stream) !=
        cudaSuccess)
      return LORA_ECUDA;
    loaded = scratch + kOffAllLoaded;
  }

  lora::BuilderArgs a;
  a.token_slot = token_slot_dev;
  a.T = T;
  a.S = num_slots;
  a.loaded = loaded;
  a.rows_per_tile = lora::kTileRows;
  a.window_rows = 0;
  a.window_groups = 0;
  a.row_slot = scratch + kOffRowSlot;
  a.perm = perm_dev;
  a.seg_offsets = seg_offsets_dev;
  a.seg_slot = seg_slot_dev;
  a.tile_seg = scratch + kOffTileSeg;
  a.tile_row0 = scratch + kOffTileRow0;
  a.meta = meta;
  a.err = err;
  if (lora::launch_segment_builder(a, stream) != cudaSuccess) return LORA_ECUDA;
  // counts: n_seg, n_adapted, error flags (device to device, no allocation)
  if (cudaMemcpyAsync(counts_dev, meta, 2 * sizeof(int32_t), cudaMemcpyDeviceToDevice, stream) !=
          cudaSuccess ||
      cudaMemcpyAsync(counts_dev + 2, err, sizeof(int32_t), cudaMemcpyDeviceToDevice, stream) !=
          cudaSuccess)
    return LORA_ECUDA;
  return LORA_OK;
}
