// builder.cu -- segment/offset builder: token->slot map to SGMV segments, on the device.
//
// "Serving multiple LoRAs: segmented matrix multiplies and adapter scheduling", section
// "Not merging the weights, computing in batches" (SGMV: place the tokens of one adapter
// together -- a stable argsort by adapter, then run lengths) and "LoRAX, in depth",
// section "Computing a batch that mixes adapters" (segment boundaries of length
// n_segments + 1 with one owner per segment).
//
// One CTA of 1024 threads computes, bit-exactly and deterministically:
//   row_slot[T]      each row's slot after validation (-1 = base only, also for bad ids)
//   perm[T_a]        adapted rows sorted by ascending slot, original order within a slot
//   seg_offsets[n_seg+1], seg_slot[n_seg]   one segment per slot that owns rows
//   tile_seg/tile_row0[n_tiles]             the shrink kernel's work list: each segment
//                                           cut into pieces of at most rows_per_tile rows,
//                                           or (window mode) units: a window of window_rows
//                                           consecutive perm positions (tile_row0 = its
//                                           first position) and the first of at most
//                                           window_groups of its segments (tile_seg)
//   meta = {n_seg, T_a, n_tiles}
// Method (a counting sort that needs no atomics, so the order is unique):
//   0. The slots' loaded flags are staged in shared memory.
//   1. W "walker" warps each own a contiguous range of rows and count, per slot, the rows
//      of their range (warp match_any groups equal slots within 32 rows).  A walker reads
//      the ids of up to kWalkBatch x 32 rows in one batch and keeps their checked slots in
//      registers for step 3, so its loads are not one dependent round trip per 32 rows.
//   2. Per slot, an exclusive prefix over the walkers, then one block-wide exclusive scan
//      over slots gives each slot's segment start, segment index and first tile.
//   3. Each walker re-walks its range in row order and scatters row indices to
//      segment start + rows of the slot already seen: stable by construction.
#include "lora_kernels.h"
#include "lora_common.cuh"

namespace lora {

static constexpr int kBuilderThreads = 1024;
static constexpr int kWalkBatch = 8;  // 32-row groups a walker loads (and keeps) at once
// windows per thread in window mode: 1024 * 8 windows of 128 rows cover 2^20 rows
static constexpr int kMaxWinPerThread = 8;

struct Scan3 {
  int a, b, c;
};

__device__ __forceinline__ Scan3 warp_inclusive_scan3(Scan3 v, int lane) {
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    int a = __shfl_up_sync(0xffffffffu, v.a, d);
    int b = __shfl_up_sync(0xffffffffu, v.b, d);
    int c = __shfl_up_sync(0xffffffffu, v.c, d);
    if (lane >= d) {
      v.a += a;
      v.b += b;
      v.c += c;
    }
  }
  return v;
}

__global__ void __launch_bounds__(kBuilderThreads, 1)
    segment_builder_kernel(const int32_t* __restrict__ token_slot, int T, int S,
                           const int32_t* __restrict__ loaded, int n_walk, int rows_per_tile,
                           int window_rows, int window_groups,
                           int32_t* __restrict__ row_slot, int32_t* __restrict__ perm,
                           int32_t* __restrict__ seg_offsets, int32_t* __restrict__ seg_slot,
                           int32_t* __restrict__ tile_seg, int32_t* __restrict__ tile_row0,
                           int32_t* __restrict__ meta, int32_t* __restrict__ err) {
  extern __shared__ int32_t sm[];
  int32_t* hist = sm;                      // [n_walk][S]: counts, then cursors
  int32_t* total = sm + (size_t)n_walk * S;  // [S]
  int32_t* loaded_s = total + S;             // [S]
  __shared__ Scan3 warp_tot[32];
  __shared__ Scan3 grand;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned lt_mask = (1u << lane) - 1u;
  // the tile kernel and the base GEMM may be scheduled now; both wait for this grid to
  // finish before they read what it writes
  griddep_launch_dependents();

  for (int i = tid; i < n_walk * S; i += blockDim.x) hist[i] = 0;
  for (int q = tid; q < S; q += blockDim.x) loaded_s[q] = loaded[q];

  // rows [w*chunk, min(T, (w+1)*chunk)) belong to walker w
  const int chunk = (T + n_walk - 1) / n_walk;
  const int r_begin = warp * chunk;
  const int r_end = min(T, r_begin + chunk);
  // a walker whose range fits one batch keeps its rows' checked slots for step 3
  const bool kept = r_end - r_begin <= 32 * kWalkBatch;
  int slot_kept[kWalkBatch];
  // the first batch of ids is requested before the barrier, alongside the flags
  int raw_b[kWalkBatch];
#pragma unroll
  for (int u = 0; u < kWalkBatch; ++u) {
    const int i = r_begin + u * 32 + lane;
    raw_b[u] = warp < n_walk && i < r_end ? token_slot[i] : -1;
  }
  __syncthreads();

  // ---- 1. validate ids and count per (walker, slot) ----
  if (warp < n_walk) {
    int32_t* my_hist = hist + (size_t)warp * S;
    for (int b0 = r_begin; b0 < r_end; b0 += 32 * kWalkBatch) {
      if (b0 != r_begin) {
#pragma unroll
        for (int u = 0; u < kWalkBatch; ++u) {
          const int i = b0 + u * 32 + lane;
          raw_b[u] = i < r_end ? token_slot[i] : -1;
        }
      }
#pragma unroll
      for (int u = 0; u < kWalkBatch; ++u) {
        const int i = b0 + u * 32 + lane;
        const bool valid = i < r_end;
        int s = -1;
        if (valid) {
          const int raw = raw_b[u];
          if (raw < -1 || raw >= S) {
            atomicOr(err, LORA_ERRF_BAD_ID);
          } else if (raw >= 0 && loaded_s[raw] == 0) {
            atomicOr(err, LORA_ERRF_EMPTY_SLOT);
          } else {
            s = raw;
          }
          row_slot[i] = s;
        }
        slot_kept[u] = s;
        const int key = valid ? s : -2;
        const unsigned peers = __match_any_sync(0xffffffffu, key);
        if (valid && s >= 0 && lane == __ffs(peers) - 1) my_hist[s] += __popc(peers);
        __syncwarp();
      }
    }
  }
  __syncthreads();

  // ---- 2a. per slot: exclusive prefix over walkers, total rows ----
  for (int s = tid; s < S; s += blockDim.x) {
    int run = 0;
    for (int w = 0; w < n_walk; ++w) {
      const int c = hist[(size_t)w * S + s];
      hist[(size_t)w * S + s] = run;
      run += c;
    }
    total[s] = run;
  }
  __syncthreads();

  // ---- 2b. block exclusive scan over slots of (rows, non-empty, tiles) ----
  const int ipt = (S + blockDim.x - 1) / blockDim.x;  // consecutive slots per thread
  const int s_begin = min(S, tid * ipt), s_end = min(S, s_begin + ipt);
  Scan3 mine = {0, 0, 0};
  for (int s = s_begin; s < s_end; ++s) {
    const int t = total[s];
    mine.a += t;
    mine.b += t > 0;
    if (window_rows == 0) mine.c += (t + rows_per_tile - 1) / rows_per_tile;
  }
  const Scan3 inc = warp_inclusive_scan3(mine, lane);
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    Scan3 v = lane < nw ? warp_tot[lane] : Scan3{0, 0, 0};
    const Scan3 vinc = warp_inclusive_scan3(v, lane);
    if (lane < nw) warp_tot[lane] = Scan3{vinc.a - v.a, vinc.b - v.b, vinc.c - v.c};
    if (lane == 31) grand = vinc;
  }
  __syncthreads();
  Scan3 pre = warp_tot[warp];
  pre.a += inc.a - mine.a;
  pre.b += inc.b - mine.b;
  pre.c += inc.c - mine.c;
  for (int s = s_begin; s < s_end; ++s) {
    const int t = total[s];
    if (t > 0) {
      seg_slot[pre.b] = s;
      seg_offsets[pre.b] = pre.a;
      if (window_rows == 0) {
        const int nt = (t + rows_per_tile - 1) / rows_per_tile;
        for (int q = 0; q < nt; ++q) {
          tile_seg[pre.c + q] = pre.b;
          tile_row0[pre.c + q] = pre.a + q * rows_per_tile;
        }
        pre.c += nt;
      } else {
        // per window, provisionally: tile_seg = the segment holding its first position,
        // tile_row0 = the segment holding its last position (T_a - 1 for the last window)
        const int T_a = grand.a, W = window_rows;
        const int nwin = (T_a + W - 1) / W;
        for (int q = (pre.a + W - 1) / W; q * W < pre.a + t; ++q) tile_seg[q] = pre.b;
        for (int q = pre.a / W; q < nwin && min(q * W + W - 1, T_a - 1) < pre.a + t; ++q)
          tile_row0[q] = pre.b;
      }
      for (int w = 0; w < n_walk; ++w) hist[(size_t)w * S + s] += pre.a;  // -> cursors
      pre.b += 1;
    }
    pre.a += t;
  }
  if (tid == 0) {
    seg_offsets[grand.b] = grand.a;
    meta[0] = grand.b;  // n_seg
    meta[1] = grand.a;  // T_a
    if (window_rows == 0) meta[2] = grand.c;  // n_tiles
  }
  __syncthreads();

  // ---- 2c. window mode: one work unit per window and group of <= window_groups of its
  //      segments (a window spans segments tile_seg .. tile_row0 of step 2b) ----
  if (window_rows > 0) {
    const int W = window_rows, G = window_groups;
    const int nwin = (grand.a + W - 1) / W;
    const int wpt = (nwin + (int)blockDim.x - 1) / (int)blockDim.x;  // <= kMaxWinPerThread
    int first[kMaxWinPerThread], units[kMaxWinPerThread];
    int my_units = 0;
#pragma unroll
    for (int i = 0; i < kMaxWinPerThread; ++i) {
      const int w = tid * wpt + i;
      units[i] = 0;
      first[i] = 0;
      if (i < wpt && w < nwin) {
        first[i] = tile_seg[w];
        units[i] = (tile_row0[w] - first[i] + G) / G;
        my_units += units[i];
      }
    }
    const Scan3 uinc = warp_inclusive_scan3(Scan3{my_units, 0, 0}, lane);
    __syncthreads();  // every window read; warp_tot free again
    if (lane == 31) warp_tot[warp] = uinc;
    __syncthreads();
    if (warp == 0) {
      const int nw = blockDim.x >> 5;
      Scan3 v = lane < nw ? warp_tot[lane] : Scan3{0, 0, 0};
      const Scan3 vinc = warp_inclusive_scan3(v, lane);
      if (lane < nw) warp_tot[lane] = Scan3{vinc.a - v.a, 0, 0};
      if (lane == 31) {
        meta[2] = vinc.a;  // n_units
        meta[4] = 0;       // the shrink's work and exit counters start at zero
        meta[5] = 0;
      }
    }
    __syncthreads();
    int u = warp_tot[warp].a + uinc.a - my_units;
#pragma unroll
    for (int i = 0; i < kMaxWinPerThread; ++i) {
      for (int q = 0; q < units[i]; ++q, ++u) {
        tile_seg[u] = first[i] + q * G;
        tile_row0[u] = (tid * wpt + i) * W;
      }
    }
  }

  // ---- 3. stable scatter: walkers re-walk their rows in order ----
  if (warp < n_walk) {
    int32_t* cursor = hist + (size_t)warp * S;
    auto scatter32 = [&](int i, int s) {
      const bool valid = i < r_end;
      const int key = valid ? s : -2;
      const unsigned peers = __match_any_sync(0xffffffffu, key);
      const int leader = __ffs(peers) - 1;
      const bool adapted = valid && s >= 0;
      int my_base = 0;
      if (adapted && lane == leader) my_base = cursor[s];
      const int b = __shfl_sync(0xffffffffu, my_base, leader);
      if (adapted) {
        perm[b + __popc(peers & lt_mask)] = i;
        if (lane == leader) cursor[s] = b + __popc(peers);
      }
      __syncwarp();
    };
    if (kept) {
#pragma unroll
      for (int u = 0; u < kWalkBatch; ++u)
        if (r_begin + u * 32 < r_end) scatter32(r_begin + u * 32 + lane, slot_kept[u]);
    } else {
      for (int base = r_begin; base < r_end; base += 32) {
        const int i = base + lane;
        scatter32(i, i < r_end ? row_slot[i] : -1);
      }
    }
  }
}

int builder_smem_bytes(int S, int* n_walk_out) {
  // walkers x slots counters must fit next to the per-slot totals and flags in 200 KB
  const int budget_ints = 200 * 1024 / 4 - 2 * S;
  int n_walk = budget_ints / S;
  if (n_walk > kBuilderThreads / 32) n_walk = kBuilderThreads / 32;
  if (n_walk < 1) n_walk = 1;
  *n_walk_out = n_walk;
  return (n_walk * S + 2 * S) * 4;
}

cudaError_t launch_segment_builder(const BuilderArgs& a, cudaStream_t stream) {
  if (a.window_rows > 0 &&
      (a.window_groups < 1 ||
       (a.T + a.window_rows - 1) / a.window_rows > kBuilderThreads * kMaxWinPerThread))
    return cudaErrorInvalidValue;
  int n_walk = 1;
  const int smem = builder_smem_bytes(a.S, &n_walk);
  static int limit[kAttrDevices] = {};
  static bool carveout[kAttrDevices] = {};
  cudaError_t e = ensure_smem_limit(segment_builder_kernel, smem, limit);
  if (e == cudaSuccess) e = prefer_max_smem_carveout(segment_builder_kernel, carveout);
  if (e != cudaSuccess) return e;
  segment_builder_kernel<<<1, kBuilderThreads, smem, stream>>>(
      a.token_slot, a.T, a.S, a.loaded, n_walk, a.rows_per_tile, a.window_rows,
      a.window_groups, a.row_slot, a.perm,
      a.seg_offsets, a.seg_slot, a.tile_seg, a.tile_row0, a.meta, a.err);
  return cudaGetLastError();
}

}  // namespace lora
