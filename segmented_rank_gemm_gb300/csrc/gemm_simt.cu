// gemm_simt.cu -- fp32 path of the layer on the CUDA cores: y = x W + scale * v B_slot.
//
// Used when the layer's dtype is fp32 (e.g. the six-row worked example of "Multi-LoRA
// Serving 与 Adapter 隔离", computed in float32): tf32 tensor cores round the inputs to a
// 10-bit mantissa, which cannot meet an fp32 tolerance, so this path stays on the FMA
// pipes.  64 x 64 output tile per CTA, 16-deep K slices staged in shared memory, 4 x 4
// outputs per thread; the epilogue adds the row's expand like the tensor-core kernel.
#include "lora_common.cuh"
#include "lora_kernels.h"

namespace lora {

static constexpr int kSimtTile = 64, kSimtK = 16, kSimtThreads = 256;

__global__ void __launch_bounds__(kSimtThreads)
    gemm_simt_f32_kernel(GemmArgs a) {
  extern __shared__ float vs[];  // [64][R+1] scaled shrink of the tile's rows
  __shared__ float As[kSimtK][kSimtTile + 1];
  __shared__ float Bs[kSimtK][kSimtTile];
  __shared__ int rs[kSimtTile];

  const float* __restrict__ x = static_cast<const float*>(a.x);
  const float* __restrict__ W = static_cast<const float*>(a.W);
  float* __restrict__ y = static_cast<float*>(a.y);
  const ExpandArgs& ex = a.ex;
  const int R = ex.R;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int m0 = blockIdx.x * kSimtTile, n0 = blockIdx.y * kSimtTile;

  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  for (int k0 = 0; k0 < a.K; k0 += kSimtK) {
    for (int e = tid; e < kSimtTile * kSimtK; e += kSimtThreads) {
      const int m = e / kSimtK, k = e % kSimtK;
      const int gm = m0 + m, gk = k0 + k;
      As[k][m] = (gm < a.M && gk < a.K) ? x[(size_t)gm * a.K + gk] : 0.f;
    }
    for (int e = tid; e < kSimtTile * kSimtK; e += kSimtThreads) {
      const int k = e / kSimtTile, n = e % kSimtTile;
      const int gk = k0 + k, gn = n0 + n;
      Bs[k][n] = (gk < a.K && gn < a.N) ? W[(size_t)gk * a.N + gn] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kSimtK; ++k) {
      float av[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = As[k][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) bv[j] = Bs[k][tx + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }

  // this tile's rows of v (fp32, already multiplied by alpha / r by the tile kernel)
  if (tid < kSimtTile) rs[tid] = (m0 + tid < a.M) ? ex.row_slot[m0 + tid] : -1;
  __syncthreads();
  for (int e = tid; e < kSimtTile * R; e += kSimtThreads) {
    const int m = e / R, j = e % R;
    const int s = rs[m];
    if (s >= 0 && j < ex.rank[s] && LORA_IN_BOUNDS(m0 + m < ex.v_rows, a.err))
      vs[m * (R + 1) + j] = ex.v[(size_t)(m0 + m) * R + j];
  }
  __syncthreads();

  const float* __restrict__ Bp = static_cast<const float*>(ex.B_pool);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = ty + 16 * i, gm = m0 + m;
    if (gm >= a.M) continue;
    const int s = rs[m];
    const int r = s >= 0 ? ex.rank[s] : 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int gn = n0 + tx + 16 * j;
      if (gn >= a.N) continue;
      float out = acc[i][j];
      if (s >= 0 && LORA_IN_BOUNDS(ex.row_base[s] >= 0 && ex.row_base[s] + r <= ex.pool_rows,
                                   a.err)) {
        const float* bcol = Bp + (size_t)ex.row_base[s] * a.N + gn;
        for (int jj = 0; jj < r; ++jj) out = fmaf(vs[m * (R + 1) + jj], bcol[(size_t)jj * a.N], out);
      }
      y[(size_t)gm * a.N + gn] = out;
    }
  }
}

cudaError_t launch_gemm_simt_f32(const GemmArgs& a, cudaStream_t stream) {
  const size_t smem = (size_t)kSimtTile * (a.ex.R + 1) * sizeof(float);
  static int limit[kAttrDevices] = {};
  cudaError_t e = ensure_smem_limit(gemm_simt_f32_kernel, (int)smem, limit);
  if (e != cudaSuccess) return e;
  dim3 grid((a.M + kSimtTile - 1) / kSimtTile, (a.N + kSimtTile - 1) / kSimtTile);
  gemm_simt_f32_kernel<<<grid, kSimtThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace lora
