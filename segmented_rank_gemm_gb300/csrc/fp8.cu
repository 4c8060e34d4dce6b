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

#include <algorithm>

#include "e4m3_row.cuh"
#include "lora_common.cuh"
#include "lora_kernels.h"

namespace lora {

static constexpr int kQHold = 8;  // 16-byte chunks a thread holds between the max and the conversion

// The decode step's row quantiser (see launch_quant_rows_e4m3 and quantize_rows_e4m3_cta).
// NT = 128 (4 warps of at most 112 registers) for batches of more than two rows a CTA: with
// the decode BGMV (2 warps of 120 per scheduler) and an e4m3 GEMM CTA (at most 2 warps of 80
// per scheduler), one warp of this kernel per scheduler fills an SM's 16K-register files
// exactly, so the three kernels share the SM and the GEMM's CTAs start while it runs.
// NT = 256 for at most two rows a CTA: each row then has 4 warps (a decode batch's rows are
// ready sooner), and the GEMM's CTAs start once it leaves; and ahead of the SGMV shrink
// (larger batches), where it shares its SMs with nothing.
template <int NT>
__global__ void __maxnreg__(112)
    quant_rows_e4m3_kernel(const __nv_bfloat16* __restrict__ x, int T, int K,
                           uint8_t* __restrict__ xq, float* __restrict__ sx,
                           int32_t* __restrict__ q_ready) {
  __shared__ float wmax[NT / 32];
  // the previous forward's base GEMM may still read xq, and the previous kernel may have
  // written x: wait for it; the low-rank kernel may then start at once (it relies on this
  // wait for the previous GEMM, and the base GEMM waits for the rows counted on q_ready)
  griddep_wait();
  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rows = quantize_rows_e4m3_cta<NT, kQHold>(x, T, K, xq, sx, wmax, warp, lane);
  if (q_ready) publish_rows(q_ready, rows);
}

template <int NT>
static cudaError_t launch_quant_rows_t(const void* x, int T, int K, uint8_t* xq, float* sx,
                                       int32_t* q_ready, int ctas, cudaStream_t stream) {
  // it shares SMs with the low-rank kernel and the base GEMM launched behind it: the SMs
  // must keep the shared-memory split a GEMM CTA needs, or that CTA waits for them to drain
  static bool carveout[kAttrDevices] = {};
  cudaError_t e = prefer_max_smem_carveout(quant_rows_e4m3_kernel<NT>, carveout);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(std::max(1, std::min(T, ctas)));
  cfg.blockDim = dim3(NT);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, quant_rows_e4m3_kernel<NT>, static_cast<const __nv_bfloat16*>(x),
                            T, K, xq, sx, q_ready);
}

cudaError_t launch_quant_rows_e4m3(const void* x, int T, int K, uint8_t* xq, float* sx,
                                   int32_t* q_ready, int num_sms, bool beside_bgmv,
                                   cudaStream_t stream) {
  if (T < 1) return cudaSuccess;
  if (K % 16 != 0) return cudaErrorInvalidValue;
  const int sms = std::max(1, num_sms);
  // ahead of the SGMV shrink, which waits for it: two CTAs of 8 warps per SM
  if (!beside_bgmv) return launch_quant_rows_t<256>(x, T, K, xq, sx, q_ready, 2 * sms, stream);
  return T <= 2 * sms ? launch_quant_rows_t<256>(x, T, K, xq, sx, q_ready, sms, stream)
                      : launch_quant_rows_t<128>(x, T, K, xq, sx, q_ready, sms, stream);
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
