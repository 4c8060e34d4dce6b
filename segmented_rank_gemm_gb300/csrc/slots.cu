// slots.cu -- slot table maintenance: the "activation" copy of an adapter into a slot and
// the one-time packing of the base weight.
//
// "Serving LoRA adapters: from the model name to the wrapped layer" (vLLM), Step 3: the
// activation copies each module's A and B into stacked buffers at the slot index; buffers
// are sized for the maximum rank.  Here A [K,r] is stored transposed as rank rows of At
// (K contiguous: the shrink streams it with coalesced vector loads) and B [r,N] as rank
// rows of B, both from the slot's first pool row; rows past r that the slot owns are zero.
#include "lora_common.cuh"
#include "lora_kernels.h"

namespace lora {

template <typename T>
__global__ void transpose_pad_kernel(const T* __restrict__ A, T* __restrict__ At, int K, int r,
                                     int R) {
  // At[j][k] = A[k][j] for j < r, 0 for r <= j < R.  32x32 tiles through shared memory.
  __shared__ T tile[32][33];
  const int k0 = blockIdx.x * 32, j0 = blockIdx.y * 32;
  for (int dy = threadIdx.y; dy < 32; dy += blockDim.y) {
    const int k = k0 + dy, j = j0 + threadIdx.x;
    tile[dy][threadIdx.x] = (k < K && j < r) ? A[(size_t)k * r + j] : T(0.f);
  }
  __syncthreads();
  for (int dy = threadIdx.y; dy < 32; dy += blockDim.y) {
    const int j = j0 + dy, k = k0 + threadIdx.x;
    if (j < R && k < K) At[(size_t)j * K + k] = tile[threadIdx.x][dy];
  }
}

cudaError_t launch_transpose_pad(const void* A_kr, void* At_rk, int K, int r, int R, bool bf16,
                                 cudaStream_t stream) {
  dim3 block(32, 8), grid((K + 31) / 32, (R + 31) / 32);
  if (bf16)
    transpose_pad_kernel<__nv_bfloat16><<<grid, block, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(A_kr), static_cast<__nv_bfloat16*>(At_rk), K, r, R);
  else
    transpose_pad_kernel<float><<<grid, block, 0, stream>>>(
        static_cast<const float*>(A_kr), static_cast<float*>(At_rk), K, r, R);
  return cudaGetLastError();
}

__global__ void pack_w_kernel(const __nv_bfloat16* __restrict__ W, __nv_bfloat16* __restrict__ Wt,
                              int K, int N) {
  // Wt[n][k] = W[k][n], 32x32 tiles.
  __shared__ __nv_bfloat16 tile[32][33];
  const int n0 = blockIdx.x * 32, k0 = blockIdx.y * 32;
  for (int dy = threadIdx.y; dy < 32; dy += blockDim.y) {
    const int k = k0 + dy, n = n0 + threadIdx.x;
    if (k < K && n < N) tile[dy][threadIdx.x] = W[(size_t)k * N + n];
  }
  __syncthreads();
  for (int dy = threadIdx.y; dy < 32; dy += blockDim.y) {
    const int n = n0 + dy, k = k0 + threadIdx.x;
    if (n < N && k < K) Wt[(size_t)n * K + k] = tile[threadIdx.x][dy];
  }
}

cudaError_t launch_pack_w_bf16(const void* W_kn, void* W_nk, int K, int N, cudaStream_t stream) {
  dim3 block(32, 8), grid((N + 31) / 32, (K + 31) / 32);
  pack_w_kernel<<<grid, block, 0, stream>>>(static_cast<const __nv_bfloat16*>(W_kn),
                                            static_cast<__nv_bfloat16*>(W_nk), K, N);
  return cudaGetLastError();
}

__global__ void pack_bx_kernel(const __nv_bfloat16* __restrict__ B, __nv_bfloat16* __restrict__ Bx,
                               int R, int N, int wx, int half) {
  // Bx[n][j] = B[j mod half][n] for j < wx (half = wx / 2 when both halves repeat B^T,
  // else half = wx), 0 where that rank index is >= R (here: the rows the slot owns).
  // 32x32 tiles through shared memory.
  __shared__ __nv_bfloat16 tile[32][33];
  const int n0 = blockIdx.x * 32, j0 = blockIdx.y * 32;
  for (int dy = threadIdx.y; dy < 32; dy += blockDim.y) {
    const int j = j0 + dy, n = n0 + threadIdx.x;
    const int jj = j % half;
    tile[dy][threadIdx.x] =
        (j < wx && jj < R && n < N) ? B[(size_t)jj * N + n] : __float2bfloat16(0.f);
  }
  __syncthreads();
  for (int dy = threadIdx.y; dy < 32; dy += blockDim.y) {
    const int n = n0 + dy, j = j0 + threadIdx.x;
    if (n < N && j < wx) Bx[(size_t)n * wx + j] = tile[threadIdx.x][dy];
  }
}

cudaError_t launch_pack_bx(const void* B_rn, void* Bx_nw, int R, int rows, int N,
                           cudaStream_t stream) {
  const ExpandLayout L = expand_layout(R);
  dim3 block(32, 8), grid((N + 31) / 32, (L.wx + 31) / 32);
  pack_bx_kernel<<<grid, block, 0, stream>>>(static_cast<const __nv_bfloat16*>(B_rn),
                                             static_cast<__nv_bfloat16*>(Bx_nw), min(R, rows), N,
                                             L.wx, L.nbs == 1 ? L.wx / 2 : L.wx);
  return cudaGetLastError();
}

__global__ void slot_meta_kernel(float* scale, int R, int32_t* rank, int32_t* loaded, int slot,
                                 SlotScales cols, int r, int is_loaded, int32_t* row_base,
                                 int rb) {
  for (int j = threadIdx.x; j < R; j += blockDim.x) scale[(size_t)slot * R + j] = cols.v[j];
  if (threadIdx.x == 0) {
    rank[slot] = r;
    loaded[slot] = is_loaded;
    if (row_base) row_base[slot] = rb;
  }
}

cudaError_t launch_slot_meta(float* scale, int R, int32_t* rank, int32_t* loaded, int slot,
                             const SlotScales& cols, int r, int is_loaded, int32_t* row_base,
                             int rb, cudaStream_t stream) {
  slot_meta_kernel<<<1, kMaxSlotRank, 0, stream>>>(scale, R, rank, loaded, slot, cols, r,
                                                   is_loaded, row_base, rb);
  return cudaGetLastError();
}

}  // namespace lora
