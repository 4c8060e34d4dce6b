// shrink.cu -- LoRA shrink v = x A_slot over SGMV segments (BGMV when segments are short).
//
// "Serving multiple LoRAs: segmented matrix multiplies and adapter scheduling", section
// "Not merging the weights, computing in batches": real kernels first shrink x -> xA (down
// to r dimensions), then expand; "Serving LoRA adapters ..." (vLLM) Step 4: the shrink
// writes an fp32 buffer of rank width.
//
// Work list: the segment builder cut every segment into tiles of <= rows_per_tile rows;
// each (tile, K-chunk) pair is one work item, taken by persistent CTAs.  Inside an item a
// warp computes, for one row and a group of JG rank columns j, the partial dot products
// sum_{k in chunk} x[row,k] * At[slot][j][k] with 16-byte vector loads of x and of the
// transposed slot matrix At (K contiguous, so both streams are coalesced), then reduces
// across the 32 lanes with shuffles.  Partial sums land in vpart[kchunk][row][j] (fp32);
// the GEMM epilogue adds the K-chunks, so the result is deterministic (no atomics).
// Only j < rank[slot] is computed: the zero padding of a slot is never read.
#include "lora_kernels.h"
#include "lora_common.cuh"

namespace lora {

static constexpr int kShrinkThreads = 256;
static constexpr int kShrinkJG = 8;

template <typename T, int VEC>
struct VecLoad;

template <>
struct VecLoad<__nv_bfloat16, 8> {
  float v[8];
  __device__ __forceinline__ void load(const __nv_bfloat16* p) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    v[0] = bf16_lo(u.x); v[1] = bf16_hi(u.x);
    v[2] = bf16_lo(u.y); v[3] = bf16_hi(u.y);
    v[4] = bf16_lo(u.z); v[5] = bf16_hi(u.z);
    v[6] = bf16_lo(u.w); v[7] = bf16_hi(u.w);
  }
};

template <>
struct VecLoad<float, 4> {
  float v[4];
  __device__ __forceinline__ void load(const float* p) {
    const float4 u = __ldg(reinterpret_cast<const float4*>(p));
    v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
  }
};

template <>
struct VecLoad<float, 1> {
  float v[1];
  __device__ __forceinline__ void load(const float* p) { v[0] = __ldg(p); }
};

template <typename T, int VEC>
__global__ void __launch_bounds__(kShrinkThreads)
    shrink_kernel(const T* __restrict__ x, int K, int R, const T* __restrict__ At_pool,
                  const int32_t* __restrict__ rank, const int32_t* __restrict__ perm,
                  const int32_t* __restrict__ seg_offsets, const int32_t* __restrict__ seg_slot,
                  const int32_t* __restrict__ tile_seg, const int32_t* __restrict__ tile_row0,
                  const int32_t* __restrict__ meta, int rows_per_tile, int ksplit, int kchunk,
                  float* __restrict__ vpart, int v_stride_rows) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = kShrinkThreads / 32;
  const int n_items = meta[2] * ksplit;

  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int t = item / ksplit, kc = item - t * ksplit;
    const int g = tile_seg[t];
    const int s = seg_slot[g];
    const int r = rank[s];
    const int p0 = tile_row0[t];
    const int p1 = min(p0 + rows_per_tile, seg_offsets[g + 1]);
    const int nr = p1 - p0;
    const int njg = (r + kShrinkJG - 1) / kShrinkJG;
    const int k0 = kc * kchunk, k1 = min(K, k0 + kchunk);
    const T* At = At_pool + (size_t)s * R * K;

    for (int task = warp; task < nr * njg; task += nwarps) {
      const int q = task / njg, jg = task - q * njg;
      const int row = perm[p0 + q];
      const int j0 = jg * kShrinkJG;
      const int jn = min(kShrinkJG, r - j0);
      const T* xr = x + (size_t)row * K;
      float acc[kShrinkJG];
#pragma unroll
      for (int jj = 0; jj < kShrinkJG; ++jj) acc[jj] = 0.f;

      for (int k = k0 + lane * VEC; k < k1; k += 32 * VEC) {
        VecLoad<T, VEC> xv;
        xv.load(xr + k);
#pragma unroll
        for (int jj = 0; jj < kShrinkJG; ++jj) {
          if (jj < jn) {
            VecLoad<T, VEC> av;
            av.load(At + (size_t)(j0 + jj) * K + k);
#pragma unroll
            for (int e = 0; e < VEC; ++e) acc[jj] = fmaf(xv.v[e], av.v[e], acc[jj]);
          }
        }
      }
#pragma unroll
      for (int jj = 0; jj < kShrinkJG; ++jj) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc[jj] += __shfl_xor_sync(0xffffffffu, acc[jj], o);
      }
      if (lane == 0) {
        float* dst = vpart + ((size_t)kc * v_stride_rows + row) * R + j0;
#pragma unroll
        for (int jj = 0; jj < kShrinkJG; ++jj)
          if (jj < jn) dst[jj] = acc[jj];
      }
    }
  }
}

cudaError_t launch_shrink(const ShrinkArgs& a, bool bf16, cudaStream_t stream) {
  int grid = a.max_items;
  const int cap = a.num_sms * 8;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  if (bf16) {
    shrink_kernel<__nv_bfloat16, 8><<<grid, kShrinkThreads, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(a.x), a.K, a.R,
        static_cast<const __nv_bfloat16*>(a.At_pool), a.rank, a.perm, a.seg_offsets,
        a.seg_slot, a.tile_seg, a.tile_row0, a.meta, a.rows_per_tile, a.ksplit, a.kchunk,
        a.vpart, a.v_stride_rows);
  } else {
    const bool vec4 = (a.K % 4 == 0) && (reinterpret_cast<uintptr_t>(a.x) % 16 == 0) &&
                      (reinterpret_cast<uintptr_t>(a.At_pool) % 16 == 0) && (a.kchunk % 4 == 0);
    if (vec4)
      shrink_kernel<float, 4><<<grid, kShrinkThreads, 0, stream>>>(
          static_cast<const float*>(a.x), a.K, a.R, static_cast<const float*>(a.At_pool),
          a.rank, a.perm, a.seg_offsets, a.seg_slot, a.tile_seg, a.tile_row0, a.meta,
          a.rows_per_tile, a.ksplit, a.kchunk, a.vpart, a.v_stride_rows);
    else
      shrink_kernel<float, 1><<<grid, kShrinkThreads, 0, stream>>>(
          static_cast<const float*>(a.x), a.K, a.R, static_cast<const float*>(a.At_pool),
          a.rank, a.perm, a.seg_offsets, a.seg_slot, a.tile_seg, a.tile_row0, a.meta,
          a.rows_per_tile, a.ksplit, a.kchunk, a.vpart, a.v_stride_rows);
  }
  return cudaGetLastError();
}

}  // namespace lora
