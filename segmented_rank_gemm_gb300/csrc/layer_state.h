// layer_state.h -- the private state of a lora_layer object, shared by the files that
// implement its C ABI (lora_layer.cu: the layer calls; residency.cu: the adapter cache that
// swaps adapters into the layers' slots).  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <map>
#include <vector>

#include "lora_kernels.h"

struct lora_layer {
  int K = 0, N = 0, S = 0, T_max = 0, dtype = 0, device = 0, num_sms = 0;
  int max_rank = 0;  // largest adapter rank a slot accepts
  int R = 0;         // slot rank width: max_rank rounded up to a multiple of 8 (zero padded)
  size_t esize = 0;
  void* Wp = nullptr;      // packed base weight: bf16 [N][K], f32 [K][N], e4m3 [N][K]
  bool fp8 = false;        // e4m3 base (x quantised per row each forward, W per column)
  uint8_t* xq = nullptr;   // fp8: [T_max][K] quantised x
  float* sx = nullptr;     // fp8: [T_max] row scales
  float* sw = nullptr;     // fp8: [N rounded up to 256] column scales, zero past N
  CUtensorMap tmap_xq;     // fp8: xq with (128 x 128) boxes
  int32_t* q_ready = nullptr;  // fp8: {rows of xq written, GEMM CTAs that saw them} (zeroed)
  bool q_dirty = false;    // fp8: a forward stopped between the BGMV and the GEMM launches
  int launches = 0;        // kernels of the last set_batch_segments + lora_forward
  void* A_pool = nullptr;  // [P][K] rank rows: slot s from row row_base[s]
  void* B_pool = nullptr;  // [P][N] rank rows
  int P = 0;               // pool rows: S * R, or the row budget of a pooled layer
  bool pooled = false;     // slots placed by the row allocator (their true rank, rounded to 8)
  int32_t* row_base = nullptr;      // [S] device: first pool row of each slot (-1: none)
  std::vector<int> rb_h, rows_h;    // host: each slot's first row and row count
  std::map<int, int> free_rows;     // pooled: free row ranges (first row -> count)
  void* Bx_pool = nullptr; // [S][N][wx] bf16, the B expand pool of the tensor-core expand
  void* A_stage = nullptr; // [K][R] staging for the transposition of a loaded A
  float* scale = nullptr;  // [S][R] column scales (+ 32 padding entries)
  int32_t* rank = nullptr;    // [S]
  int32_t* loaded = nullptr;  // [S]
  std::vector<char> percol;   // [S] host: the slot's columns carry different scales
  int percol_slots = 0;       // slots with percol set
  // batch layout (segment builder outputs)
  int32_t* row_slot = nullptr;   // [T_max]
  int32_t* perm = nullptr;       // [T_max]
  int32_t* seg_offsets = nullptr;// [S+1]
  int32_t* seg_slot = nullptr;   // [S]
  int32_t* tile_seg = nullptr;   // [max_tiles]
  int32_t* tile_row0 = nullptr;  // [max_tiles]
  int32_t* meta = nullptr;       // [8]: builder counts, shrink work counters
  int32_t* err = nullptr;        // [1]
  float* v = nullptr;            // [v_planes][T_max][R] fp32, scaled by alpha / r (v mode)
  int v_planes = 1;              // K-split partial planes of v (bf16: tensor-core shrink)
  float* delta = nullptr;        // [min(T_max, kDeltaMaxT)][N] fp32 (delta mode, bf16)
  CUtensorMap tmap_delta;        // delta with (32 x 128) boxes (valid when delta is set)
  float* xk = nullptr;           // split-K exchange scratch of the base GEMM (delta mode)
  float* sk_part = nullptr;      // stream-K partials of the base GEMM (v mode)
  int32_t* sk_sync = nullptr;    // stream-K epoch, exit count and flags (zeroed)
  size_t xk_floats = 0;
  lora::GemmPlan gemm_plan{0, 0, 0};   // fixed by lora_set_gemm_plan (block_n 0: automatic)
  int max_tiles = 0;
  int T_batch = -1;              // T of the last set_batch_segments, -1 = none
  bool segments_pending = false;  // that batch's builder has not run yet (decode batches)
  const int32_t* token_slot = nullptr;  // the caller's ids of that batch
  // staging for lora_forward_host
  void* x_stage = nullptr;
  int32_t* ids_stage = nullptr;
  void* y_stage = nullptr;
  // ordering
  cudaEvent_t stage_free = nullptr;    // recorded after a load's transposition
  cudaEvent_t last_forward = nullptr;  // recorded after each forward (when not capturing)
  bool have_forward = false;
  std::vector<cudaEvent_t> pending;    // loads not yet waited on by a forward
  std::vector<cudaEvent_t> spare;
  CUtensorMap tmap_w[3];
  CUtensorMap tmap_a;  // A pool [S*R rows][K] with a (64 x round_up(R, 16)) box (bf16)
  CUtensorMap tmap_bx[3];  // B expand pool [S*N rows][wx], boxes of 256/128/64 rows
  cudaEvent_t trace[6] = {nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
  bool tracing = false;
  char last_error[512] = {0};
};


namespace lora {

// An event from the layer's pool (created on demand).  nullptr if creation failed.
cudaEvent_t layer_take_event(lora_layer* L);

// Record whether slot `slot` now holds columns of different scales (a composition): the
// decode BGMV kernel reads one scale per slot while no slot of the layer does.
void layer_set_percol(lora_layer* L, int slot, bool varied);

// Pooled layers: return the rows slot `slot` holds to the row pool (its first row and row
// count before, through *first / *rows; 0 rows if it held none).  Host bookkeeping only.
void layer_release_rows(lora_layer* L, int slot, int* first, int* rows);
// Pooled layers: give slot `slot` (holding no rows) `rows` consecutive rows of the pool,
// first fit; returns the first row, or -1 if no run of free rows is that long.
int layer_take_rows(lora_layer* L, int slot, int rows);

}  // namespace lora
