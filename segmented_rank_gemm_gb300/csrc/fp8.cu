// fp8.cu -- the e4m3 base: quantisation of the activations (per row, every forward) and of
// the base weight (per column, once at layer creation).
//
// "Multi-LoRA Serving 与 Adapter 隔离", section on quantisation, TP and loading: an FP8 base
// with an FP16 LoRA is the usual mixed precision, the quantised product and the LoRA term
// meet in the kernel's accumulator and epilogue, and the float delta is never added to the
// packed quantised weights.  Scales are max |.| / 448 in fp32 (1 for an all-zero row or
// column); values are divided by their scale in fp32 (correctly rounded) and converted to
// e4m3 rounding to nearest even, saturating at +-448.
#include <cuda_fp8.h>

#include "lora_common.cuh"
#include "lora_kernels.h"

namespace lora {

static constexpr int kQThreads = 256;
static constexpr float kE4m3Max = 448.f;

__device__ __forceinline__ uint8_t to_e4m3(float v, float s) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(__fdiv_rn(v, s), __NV_SATFINITE, __NV_E4M3));
}

// One CTA per row; K a multiple of 16.  Each thread's 16-byte chunks of the row (at most
// kQHold of them: K <= 8 * kQThreads * kQHold = 16384) are loaded once, together, held in
// registers through the max reduction and converted from there: one round trip to memory.
// Chunks past that (longer rows) are read again for the conversion.
static constexpr int kQHold = 8;
__global__ void __launch_bounds__(kQThreads)
    quant_rows_e4m3_kernel(const __nv_bfloat16* __restrict__ x, int K, uint8_t* __restrict__ xq,
                           float* __restrict__ sx) {
  __shared__ float wmax[kQThreads / 32];
  const int row = blockIdx.x, tid = threadIdx.x;
  const int nv = K / 8;  // 16-byte chunks of the row
  const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)row * K);
  uint4 hold[kQHold];
#pragma unroll
  for (int i = 0; i < kQHold; ++i) {
    const int e = tid + i * kQThreads;
    hold[i] = e < nv ? __ldg(xr + e) : make_uint4(0u, 0u, 0u, 0u);
  }
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < kQHold; ++i) {
    const uint32_t w[4] = {hold[i].x, hold[i].y, hold[i].z, hold[i].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[j])), fabsf(bf16_hi(w[j]))));
  }
  for (int e = tid + kQHold * kQThreads; e < nv; e += kQThreads) {
    const uint4 v = __ldg(xr + e);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[j])), fabsf(bf16_hi(w[j]))));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if ((tid & 31) == 0) wmax[tid >> 5] = m;
  __syncthreads();
  float amax = 0.f;
#pragma unroll
  for (int w = 0; w < kQThreads / 32; ++w) amax = fmaxf(amax, wmax[w]);
  const float s = amax > 0.f ? __fdiv_rn(amax, kE4m3Max) : 1.f;
  if (tid == 0) sx[row] = s;
  uint2* qr = reinterpret_cast<uint2*>(xq + (size_t)row * K);
  auto convert = [&](const uint4& v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t q[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t lo = to_e4m3(bf16_lo(w[i]), s), hi = to_e4m3(bf16_hi(w[i]), s);
      q[i >> 1] |= (lo | (hi << 8)) << (16 * (i & 1));
    }
    return make_uint2(q[0], q[1]);
  };
#pragma unroll
  for (int i = 0; i < kQHold; ++i) {
    const int e = tid + i * kQThreads;
    if (e < nv) qr[e] = convert(hold[i]);
  }
  for (int e = tid + kQHold * kQThreads; e < nv; e += kQThreads) qr[e] = convert(__ldg(xr + e));
}

cudaError_t launch_quant_rows_e4m3(const void* x, int T, int K, uint8_t* xq, float* sx,
                                   cudaStream_t stream) {
  if (T < 1) return cudaSuccess;
  if (K % 16 != 0) return cudaErrorInvalidValue;
  quant_rows_e4m3_kernel<<<T, kQThreads, 0, stream>>>(static_cast<const __nv_bfloat16*>(x), K,
                                                       xq, sx);
  return cudaGetLastError();
}

// max |W[k][n]| over the rows [k0, k1) of each column, into amax[n] (float bits as int:
// non-negative floats order as their bit patterns).
__global__ void col_amax_kernel(const __nv_bfloat16* __restrict__ W, int K, int N, int rows_per,
                                int* __restrict__ amax_bits) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= N) return;
  const int k0 = blockIdx.y * rows_per, k1 = min(K, k0 + rows_per);
  float m = 0.f;
  for (int k = k0; k < k1; ++k) m = fmaxf(m, fabsf(__bfloat162float(W[(size_t)k * N + n])));
  atomicMax(amax_bits + n, __float_as_int(m));
}

__global__ void col_scale_kernel(const int* __restrict__ amax_bits, int N, float* __restrict__ sw) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= N) return;
  const float a = __int_as_float(amax_bits[n]);
  sw[n] = a > 0.f ? __fdiv_rn(a, kE4m3Max) : 1.f;
}

// Wq[n][k] = e4m3(W[k][n] / sw[n]); 32 x 32 tiles through shared memory.
__global__ void quant_transpose_kernel(const __nv_bfloat16* __restrict__ W, int K, int N,
                                       const float* __restrict__ sw, uint8_t* __restrict__ Wq) {
  __shared__ float tile[32][33];
  const int n0 = blockIdx.x * 32, k0 = blockIdx.y * 32;
  for (int dy = threadIdx.y; dy < 32; dy += blockDim.y) {
    const int k = k0 + dy, n = n0 + threadIdx.x;
    tile[dy][threadIdx.x] = (k < K && n < N) ? __bfloat162float(W[(size_t)k * N + n]) : 0.f;
  }
  __syncthreads();
  for (int dy = threadIdx.y; dy < 32; dy += blockDim.y) {
    const int n = n0 + dy, k = k0 + threadIdx.x;
    if (n < N && k < K) Wq[(size_t)n * K + k] = to_e4m3(tile[threadIdx.x][dy], sw[n]);
  }
}

cudaError_t launch_quant_cols_e4m3(const void* W_, int K, int N, uint8_t* Wq, float* sw,
                                   cudaStream_t stream) {
  const __nv_bfloat16* W = static_cast<const __nv_bfloat16*>(W_);
  int* amax = nullptr;
  cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&amax), (size_t)N * sizeof(int), stream);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(amax, 0, (size_t)N * sizeof(int), stream);
  const int rows_per = 256;
  if (e == cudaSuccess) {
    col_amax_kernel<<<dim3((N + 255) / 256, (K + rows_per - 1) / rows_per), 256, 0, stream>>>(
        W, K, N, rows_per, amax);
    col_scale_kernel<<<(N + 255) / 256, 256, 0, stream>>>(amax, N, sw);
    quant_transpose_kernel<<<dim3((N + 31) / 32, (K + 31) / 32), dim3(32, 8), 0, stream>>>(
        W, K, N, sw, Wq);
    e = cudaGetLastError();
  }
  const cudaError_t f = cudaFreeAsync(amax, stream);
  return e != cudaSuccess ? e : f;
}

}  // namespace lora
