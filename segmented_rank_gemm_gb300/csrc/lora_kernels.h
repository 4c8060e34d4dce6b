// lora_kernels.h -- internal (host-side) launchers of the layer's kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace lora {

// ---- segment builder (builder.cu) ----
struct BuilderArgs {
  const int32_t* token_slot;  // [T]
  int T, S;
  const int32_t* loaded;  // [S]
  int rows_per_tile;
  int32_t* row_slot;     // [T]
  int32_t* perm;         // [T]
  int32_t* seg_offsets;  // [S+1]
  int32_t* seg_slot;     // [S]
  int32_t* tile_seg;     // [T/rows_per_tile + S]
  int32_t* tile_row0;    // [T/rows_per_tile + S]
  int32_t* meta;         // [4] n_seg, T_a, n_tiles
  int32_t* err;
};
cudaError_t launch_segment_builder(const BuilderArgs& a, cudaStream_t stream);

// ---- shrink v = x A_slot (shrink.cu) ----
struct ShrinkArgs {
  const void* x;  // [T,K] bf16 or f32
  int T, K, R;
  const void* At_pool;  // [S][R][K] (transposed slot A, K contiguous)
  const int32_t* rank;  // [S]
  const int32_t* perm, *seg_offsets, *seg_slot, *tile_seg, *tile_row0, *meta;
  int rows_per_tile;
  int ksplit, kchunk;   // K cut into ksplit chunks of kchunk elements
  float* vpart;         // [ksplit][v_stride_rows][R]
  int v_stride_rows;    // rows per k-split plane (max_tokens)
  int max_items;        // upper bound of tiles * ksplit (grid sizing)
  int num_sms;
};
cudaError_t launch_shrink(const ShrinkArgs& a, bool bf16, cudaStream_t stream);

// ---- base GEMM with the expand fused into its epilogue ----
struct ExpandArgs {
  const int32_t* row_slot;  // [T], -1 = base only
  const float* vpart;       // [ksplit][v_stride_rows][R]
  int ksplit, v_stride_rows, R;
  const void* B_pool;   // [S][R][N]
  const float* scale;   // [S]
  const int32_t* rank;  // [S]
};
struct GemmArgs {
  int M, N, K;
  const void* x;  // [M,K]
  const void* W;  // bf16: packed [N,K]; f32: [K,N]
  void* y;        // [M,N]
  ExpandArgs ex;
  int32_t* err;
  int num_sms;
};
// tcgen05 / TMEM / TMA kernel (gemm_tc.cu).  tmap_w3 holds the layer's cached maps of the
// packed weight for N tiles of 256, 128 and 64 rows (in that order).
cudaError_t launch_gemm_tc(const GemmArgs& a, const CUtensorMap* tmap_w3, cudaStream_t stream);
constexpr int kTcTileN[3] = {256, 128, 64};
// Encode a 2-D bf16 tensor map for a K-major [rows, K] matrix with a (64 x box_rows) box.
cudaError_t encode_tmap_bf16(CUtensorMap* map, const void* base, int rows, int K, int box_rows);
int gemm_tc_block_n(int M, int N, int num_sms);

// fp32 SIMT path (gemm_simt.cu)
cudaError_t launch_gemm_simt_f32(const GemmArgs& a, cudaStream_t stream);

// ---- slot table maintenance (slots.cu) ----
// At[j][k] = j < r ? A[k][j] : 0, for j < R, k < K.
cudaError_t launch_transpose_pad(const void* A_kr, void* At_rk, int K, int r, int R, bool bf16,
                                 cudaStream_t stream);
// Wp[n][k] = W[k][n] (bf16 base weight packing).
cudaError_t launch_pack_w_bf16(const void* W_kn, void* W_nk, int K, int N, cudaStream_t stream);
cudaError_t launch_slot_meta(float* scale, int32_t* rank, int32_t* loaded, int slot, float s,
                             int r, int is_loaded, cudaStream_t stream);

}  // namespace lora
