// lora_layer.cu -- the C ABI of include/lora_layer.h: layer state, slot loading, batch
// segmentation and the forward pass (argument checks, buffer ownership, stream ordering).
//
// Every step of the computation runs in this library's kernels:
//   set_batch_segments -> segment_builder_kernel            (builder.cu)
//   lora_forward       -> bgmv_delta_kernel (decode: BGMV shrink + expand)  (lora_tile.cu)
//                         or lora_tile_kernel (SGMV shrink per segment tile)
//                      -> gemm_tc_kernel (bf16, tcgen05)                    (gemm_tc.cu)  or
//                         gemm_simt_f32_kernel (fp32)                       (gemm_simt.cu)
// Two regimes.  bf16 batches of at most kDeltaMaxT rows (decode) use delta mode: the BGMV
// kernel gathers each row's A and B by its slot id and writes the expanded low-rank term to
// an fp32 [T,N] buffer that the GEMM epilogue adds; it needs nothing from the segment
// builder, so builder, BGMV kernel and GEMM main loop all run at once.  Larger batches
// (prefill) and fp32 use v mode: the SGMV tile kernel (after the builder) writes v [T,r]
// and the GEMM epilogue expands it.  bf16 launches chain with programmatic dependent launch.
//   load_adapter_slot  -> copy + transpose_pad_kernel + slot_meta_kernel (slots.cu)
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include "lora_layer.h"
#include "lora_common.cuh"
#include "lora_kernels.h"
#include "layer_state.h"

using namespace lora;

namespace {

constexpr int kMaxSlots = 4096;
constexpr int kMaxRank = 128;
constexpr int kMaxTokens = 1 << 20;
constexpr int kDeltaMaxT = 512;  // largest batch computed in delta mode

}  // namespace

namespace {

int fail(lora_layer* L, int code, const char* fmt, ...) {
  if (L) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(L->last_error, sizeof(L->last_error), fmt, ap);
    va_end(ap);
  }
  return code;
}

int cuda_fail(lora_layer* L, cudaError_t e, const char* what) {
  return fail(L, LORA_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define LORA_CUDA(L, expr)                                   \
  do {                                                       \
    cudaError_t e_ = (expr);                                 \
    if (e_ != cudaSuccess) return cuda_fail((L), e_, #expr); \
  } while (0)

template <typename T>
cudaError_t dmalloc(T** p, size_t count) {
  return cudaMalloc(reinterpret_cast<void**>(p), std::max<size_t>(count, 1) * sizeof(T));
}

void free_all(lora_layer* L) {
  void* ptrs[] = {L->Wp, L->A_pool, L->B_pool, L->Bx_pool, L->A_stage, L->scale, L->rank, L->loaded,
                  L->row_slot, L->perm, L->seg_offsets, L->seg_slot, L->tile_seg,
                  L->tile_row0, L->meta, L->err, L->v, L->delta, L->xk, L->sk_part,
                  L->sk_sync, L->x_stage, L->ids_stage, L->y_stage, L->row_base,
                  L->xq, L->sx, L->sw, L->q_ready};
  for (void* p : ptrs)
    if (p) cudaFree(p);
  if (L->stage_free) cudaEventDestroy(L->stage_free);
  if (L->last_forward) cudaEventDestroy(L->last_forward);
  for (cudaEvent_t e : L->pending) cudaEventDestroy(e);
  for (cudaEvent_t e : L->spare) cudaEventDestroy(e);
}

cudaError_t trace_mark(const lora_layer* L, int idx, cudaStream_t s) {
  return L->tracing ? cudaEventRecord(L->trace[idx], s) : cudaSuccess;
}

bool is_capturing(cudaStream_t s) {
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &st) != cudaSuccess) return false;
  return st != cudaStreamCaptureStatusNone;
}

// Order `stream` after every slot load not yet waited on.  Under stream capture the loads
// are outside the graph, so the waits become external-event nodes of the graph.
cudaError_t wait_pending_loads(lora_layer* L, cudaStream_t stream) {
  const unsigned flags = is_capturing(stream) ? cudaEventWaitExternal : cudaEventWaitDefault;
  for (cudaEvent_t e : L->pending) {
    cudaError_t err = cudaStreamWaitEvent(stream, e, flags);
    if (err != cudaSuccess) return err;
  }
  L->spare.insert(L->spare.end(), L->pending.begin(), L->pending.end());
  L->pending.clear();
  return cudaSuccess;
}

}  // namespace

namespace lora {

cudaEvent_t layer_take_event(lora_layer* L) {
  if (!L->spare.empty()) {
    cudaEvent_t e = L->spare.back();
    L->spare.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return nullptr;
  return e;
}

void layer_set_percol(lora_layer* L, int slot, bool varied) {
  if ((L->percol[slot] != 0) != varied) L->percol_slots += varied ? 1 : -1;
  L->percol[slot] = varied ? 1 : 0;
}

}  // namespace lora

extern "C" {

}  // extern "C"

// pool_rows 0: slot s owns rows [s R, s R + R) of the pools; > 0: a row pool of that many
// rows (rounded up to 8) from which each load takes its rank rounded up to 8 rows.
static int create_layer(lora_layer_t** out, int K, int N, int num_slots, int max_rank,
                        int max_tokens, int dtype, const void* W_dev, void* stream_,
                        int pool_rows, bool fp8 = false) {
  if (!out) return LORA_EINVAL;
  *out = nullptr;
  if (K < 1 || N < 1 || num_slots < 1 || num_slots > kMaxSlots || max_rank < 1 ||
      max_rank > kMaxRank || max_tokens < 1 || max_tokens > kMaxTokens || !W_dev)
    return LORA_EINVAL;
  if (dtype != LORA_F32 && dtype != LORA_BF16) return LORA_EINVAL;
  if (dtype == LORA_BF16 && (K % 8 != 0 || N % 8 != 0)) return LORA_EINVAL;
  // an e4m3 base: bf16 activations, K a multiple of 16 (16-byte rows), decode batches only
  if (fp8 && (dtype != LORA_BF16 || K % 16 != 0)) return LORA_EINVAL;
  const int R8 = (max_rank + 7) / 8 * 8;
  if (pool_rows < 0 || (pool_rows > 0 && ((pool_rows + 7) / 8 * 8 < R8 ||
                                           (long long)pool_rows > (long long)num_slots * R8)))
    return LORA_EINVAL;

  lora_layer* L = new (std::nothrow) lora_layer();
  if (!L) return LORA_ENOMEM;
  L->K = K;
  L->N = N;
  L->S = num_slots;
  L->max_rank = max_rank;
  L->R = (max_rank + 7) / 8 * 8;
  L->T_max = max_tokens;
  L->dtype = dtype;
  L->esize = dtype == LORA_BF16 ? 2 : 4;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);

  auto bail = [&](int code) {
    free_all(L);
    delete L;
    return code;
  };
  cudaError_t e = cudaGetDevice(&L->device);
  if (e != cudaSuccess) return bail(LORA_ECUDA);
  e = cudaDeviceGetAttribute(&L->num_sms, cudaDevAttrMultiProcessorCount, L->device);
  if (e != cudaSuccess) return bail(LORA_ECUDA);

  const size_t es = L->esize;
  const size_t S = num_slots, R = L->R;
  L->fp8 = fp8;
  L->pooled = pool_rows > 0;
  L->P = L->pooled ? (pool_rows + 7) / 8 * 8 : (int)(S * R);
  const size_t P = L->P;
  L->max_tiles = (max_tokens + kTileRows - 1) / kTileRows + num_slots;
  L->percol.assign(S, 0);
  L->rb_h.assign(S, -1);
  L->rows_h.assign(S, 0);
  if (L->pooled) {
    L->free_rows[0] = L->P;
  } else {
    for (size_t q = 0; q < S; ++q) {
      L->rb_h[q] = (int)(q * R);
      L->rows_h[q] = (int)R;
    }
  }
  // small batches split the shrink's K range over up to 8 planes of v; large ones need none
  L->v_planes = dtype == LORA_BF16 ? std::max(1, std::min(8, 65536 / max_tokens)) : 1;
  // the base GEMM of a delta-mode batch may split K: scratch for its largest exchange
  if (dtype == LORA_BF16)
    for (int m = 1; m <= std::min(max_tokens, kDeltaMaxT); ++m)
      L->xk_floats =  // (an e4m3 row of K elements has the bytes of K / 2 bf16)
          std::max(L->xk_floats, gemm_tc_exchange_floats(m, N, fp8 ? K / 2 : K, L->num_sms));
  const size_t n256 = ((size_t)N + 255) / 256 * 256;
  bool ok = cudaMalloc(&L->Wp, (size_t)K * N * (fp8 ? 1 : es)) == cudaSuccess &&
            (!fp8 || (cudaMalloc(reinterpret_cast<void**>(&L->xq), (size_t)max_tokens * K) ==
                          cudaSuccess &&
                      dmalloc(&L->sx, max_tokens) == cudaSuccess &&
                      dmalloc(&L->sw, n256) == cudaSuccess &&
                      dmalloc(&L->q_ready, 2) == cudaSuccess)) &&
            cudaMalloc(&L->A_pool, P * K * es) == cudaSuccess &&
            cudaMalloc(&L->B_pool, P * N * es) == cudaSuccess &&
            dmalloc(&L->row_base, S) == cudaSuccess &&
            cudaMalloc(&L->A_stage, (size_t)K * R * es) == cudaSuccess &&
            // column scales [S][R], padded so that a read of 32 columns of any slot is in bounds
            dmalloc(&L->scale, S * R + 32) == cudaSuccess &&
            dmalloc(&L->rank, S) == cudaSuccess &&
            dmalloc(&L->loaded, S) == cudaSuccess &&
            dmalloc(&L->row_slot, max_tokens) == cudaSuccess &&
            dmalloc(&L->perm, max_tokens) == cudaSuccess &&
            dmalloc(&L->seg_offsets, S + 1) == cudaSuccess &&
            dmalloc(&L->seg_slot, S) == cudaSuccess &&
            dmalloc(&L->tile_seg, L->max_tiles) == cudaSuccess &&
            dmalloc(&L->tile_row0, L->max_tiles) == cudaSuccess &&
            dmalloc(&L->meta, 8) == cudaSuccess && dmalloc(&L->err, 1) == cudaSuccess &&
            dmalloc(&L->v, (size_t)L->v_planes * max_tokens * R) == cudaSuccess &&
            (dtype != LORA_BF16 ||
             dmalloc(&L->delta, (size_t)std::min(max_tokens, kDeltaMaxT) * N) == cudaSuccess) &&
            (L->xk_floats == 0 || dmalloc(&L->xk, L->xk_floats) == cudaSuccess) &&
            // v-mode batches (bf16, more than 512 rows) may cut the last tiles in two
            (dtype != LORA_BF16 || max_tokens <= kDeltaMaxT ||
             (dmalloc(&L->sk_part, (size_t)L->num_sms * 128 * 256) == cudaSuccess &&
              dmalloc(&L->sk_sync, (size_t)L->num_sms + 2) == cudaSuccess)) &&
            cudaMalloc(&L->x_stage, (size_t)max_tokens * K * es) == cudaSuccess &&
            dmalloc(&L->ids_stage, max_tokens) == cudaSuccess &&
            cudaMalloc(&L->y_stage, (size_t)max_tokens * N * es) == cudaSuccess &&
            // batches beyond kDeltaMaxT rows expand v on the tensor cores
            (dtype != LORA_BF16 || max_tokens <= kDeltaMaxT ||
             cudaMalloc(&L->Bx_pool, S * expand_layout((int)R).wx * N * es) == cudaSuccess);
  if (!ok) {
    cudaGetLastError();
    return bail(LORA_ENOMEM);
  }
  ok = cudaEventCreateWithFlags(&L->stage_free, cudaEventDisableTiming) == cudaSuccess &&
       cudaEventCreateWithFlags(&L->last_forward, cudaEventDisableTiming) == cudaSuccess;
  if (!ok) return bail(LORA_ECUDA);

  ok = cudaMemsetAsync(L->A_pool, 0, P * K * es, stream) == cudaSuccess &&
       cudaMemsetAsync(L->B_pool, 0, P * N * es, stream) == cudaSuccess &&
       cudaMemcpyAsync(L->row_base, L->rb_h.data(), S * sizeof(int32_t), cudaMemcpyHostToDevice,
                       stream) == cudaSuccess &&
       (!L->Bx_pool ||
        cudaMemsetAsync(L->Bx_pool, 0, S * expand_layout((int)R).wx * N * es, stream) ==
            cudaSuccess) &&
       cudaMemsetAsync(L->scale, 0, (S * R + 32) * 4, stream) == cudaSuccess &&
       cudaMemsetAsync(L->rank, 0, S * 4, stream) == cudaSuccess &&
       cudaMemsetAsync(L->loaded, 0, S * 4, stream) == cudaSuccess &&
       cudaMemsetAsync(L->meta, 0, 32, stream) == cudaSuccess &&
       cudaMemsetAsync(L->err, 0, 4, stream) == cudaSuccess &&
       cudaMemsetAsync(L->v, 0, (size_t)L->v_planes * max_tokens * R * 4, stream) == cudaSuccess &&
       (!L->sk_sync ||
        cudaMemsetAsync(L->sk_sync, 0, ((size_t)L->num_sms + 2) * 4, stream) == cudaSuccess);
  if (!ok) return bail(LORA_ECUDA);

  if (fp8) {  // W quantised per column into [N][K] e4m3; x's map over the layer's xq
    if (cudaMemsetAsync(L->sw, 0, n256 * sizeof(float), stream) != cudaSuccess ||
        cudaMemsetAsync(L->q_ready, 0, 2 * sizeof(int32_t), stream) != cudaSuccess ||
        launch_quant_cols_e4m3(W_dev, K, N, static_cast<uint8_t*>(L->Wp), L->sw, stream) !=
            cudaSuccess)
      return bail(LORA_ECUDA);
    for (int i = 0; i < 3; ++i)
      if (encode_tmap_u8(&L->tmap_w[i], L->Wp, N, K, kTcTileN[i]) != cudaSuccess)
        return bail(LORA_ECUDA);
    if (encode_tmap_u8(&L->tmap_xq, L->xq, max_tokens, K, kTcTileRows) != cudaSuccess)
      return bail(LORA_ECUDA);
    if (encode_tmap_bf16(&L->tmap_a, L->A_pool, (int)P, K, (L->R + 15) / 16 * 16) !=
        cudaSuccess)
      return bail(LORA_ECUDA);
    if (L->Bx_pool)  // batches beyond 512 rows: the expand blocks stay bf16
      for (int i = 0; i < 3; ++i)
        if (encode_tmap_bf16(&L->tmap_bx[i], L->Bx_pool, (int)(S * N),
                             expand_layout((int)R).wx, kTcTileN[i]) != cudaSuccess)
          return bail(LORA_ECUDA);
  } else if (dtype == LORA_BF16) {
    if (launch_pack_w_bf16(W_dev, L->Wp, K, N, stream) != cudaSuccess) return bail(LORA_ECUDA);
    for (int i = 0; i < 3; ++i)
      if (encode_tmap_bf16(&L->tmap_w[i], L->Wp, N, K, kTcTileN[i]) != cudaSuccess)
        return bail(LORA_ECUDA);
    if (encode_tmap_bf16(&L->tmap_a, L->A_pool, (int)P, K, (L->R + 15) / 16 * 16) !=
        cudaSuccess)
      return bail(LORA_ECUDA);
    if (L->Bx_pool)
      for (int i = 0; i < 3; ++i)
        if (encode_tmap_bf16(&L->tmap_bx[i], L->Bx_pool, (int)(S * N),
                             expand_layout((int)R).wx, kTcTileN[i]) != cudaSuccess)
          return bail(LORA_ECUDA);
  } else {
    if (cudaMemcpyAsync(L->Wp, W_dev, (size_t)K * N * es, cudaMemcpyDefault, stream) !=
        cudaSuccess)
      return bail(LORA_ECUDA);
  }
  // the decode GEMM's epilogue reads its delta tile through this map
  if (L->delta && encode_tmap_delta(&L->tmap_delta, L->delta, std::min(max_tokens, kDeltaMaxT),
                                    N) != cudaSuccess)
    return bail(LORA_ECUDA);
  if (cudaStreamSynchronize(stream) != cudaSuccess) return bail(LORA_ECUDA);
  *out = L;
  return LORA_OK;
}

// First fit over the free row ranges: the first row of `rows` rows, or -1.
static int pool_alloc(lora_layer* L, int rows) {
  for (auto it = L->free_rows.begin(); it != L->free_rows.end(); ++it) {
    if (it->second < rows) continue;
    const int first = it->first, left = it->second - rows;
    L->free_rows.erase(it);
    if (left > 0) L->free_rows[first + rows] = left;
    return first;
  }
  return -1;
}

// Take rows [first, first + rows), which lie inside one free range, or return -1.
static int pool_alloc_at(lora_layer* L, int first, int rows) {
  auto it = L->free_rows.upper_bound(first);
  if (it == L->free_rows.begin()) return -1;
  --it;
  const int f = it->first, n = it->second;
  if (first + rows > f + n) return -1;
  L->free_rows.erase(it);
  if (first > f) L->free_rows[f] = first - f;
  if (f + n > first + rows) L->free_rows[first + rows] = f + n - (first + rows);
  return first;
}

// Return rows [first, first + rows) to the free ranges, merging neighbours.
static void pool_free(lora_layer* L, int first, int rows) {
  auto next = L->free_rows.lower_bound(first);
  if (next != L->free_rows.end() && next->first == first + rows) {
    rows += next->second;
    next = L->free_rows.erase(next);
  }
  if (next != L->free_rows.begin()) {
    auto prev = std::prev(next);
    if (prev->first + prev->second == first) {
      prev->second += rows;
      return;
    }
  }
  L->free_rows[first] = rows;
}

namespace lora {

void layer_release_rows(lora_layer* L, int slot, int* first, int* rows) {
  *first = L->rb_h[slot];
  *rows = L->rows_h[slot];
  if (L->pooled && *rows > 0) pool_free(L, *first, *rows);
  if (L->pooled) {
    L->rb_h[slot] = -1;
    L->rows_h[slot] = 0;
  }
}

int layer_take_rows(lora_layer* L, int slot, int rows) {
  const int rb = pool_alloc(L, rows);
  if (rb >= 0) {
    L->rb_h[slot] = rb;
    L->rows_h[slot] = rows;
  }
  return rb;
}

}  // namespace lora

extern "C" {

int lora_layer_create(lora_layer_t** out, int K, int N, int num_slots, int max_rank,
                      int max_tokens, int dtype, const void* W_dev, void* stream_) {
  return create_layer(out, K, N, num_slots, max_rank, max_tokens, dtype, W_dev, stream_, 0);
}

int lora_layer_create_fp8(lora_layer_t** out, int K, int N, int num_slots, int max_rank,
                          int max_tokens, const void* W_dev, void* stream_) {
  return create_layer(out, K, N, num_slots, max_rank, max_tokens, LORA_BF16, W_dev, stream_, 0,
                      true);
}

int lora_layer_create_pooled(lora_layer_t** out, int K, int N, int num_slots, int max_rank,
                             int max_tokens, int dtype, const void* W_dev, void* stream_,
                             int pool_rows) {
  if (pool_rows < 1) return LORA_EINVAL;
  return create_layer(out, K, N, num_slots, max_rank, max_tokens, dtype, W_dev, stream_,
                      pool_rows);
}

int lora_get_pool_usage(const lora_layer_t* L, int* used_rows, int* pool_rows) {
  if (!L || !used_rows || !pool_rows) return LORA_EINVAL;
  int free_total = 0;
  for (const auto& kv : L->free_rows) free_total += kv.second;
  int used = 0;
  for (int q = 0; q < L->S; ++q) used += L->rows_h[q];
  *used_rows = L->pooled ? L->P - free_total : used;
  *pool_rows = L->P;
  return LORA_OK;
}

int load_adapter_slot_composed(lora_layer_t* L, int slot, int n, const void* const* A_src,
                               const void* const* B_src, const int* r, const float* alpha,
                               const float* weight, void* side_) {
  if (!L) return LORA_EINVAL;
  if (slot < 0 || slot >= L->S) return fail(L, LORA_ESLOT, "slot %d outside [0, %d)", slot, L->S);
  if (n < 1 || !A_src || !B_src || !r || !alpha || !weight)
    return fail(L, LORA_EINVAL, "a composition needs n >= 1 members and their arrays");
  int r_sum = 0;
  for (int i = 0; i < n; ++i) {
    if (r[i] < 1 || r[i] > L->max_rank)
      return fail(L, LORA_ERANK, "member %d: rank %d outside [1, %d]", i, r[i], L->max_rank);
    if (!A_src[i] || !B_src[i]) return fail(L, LORA_EINVAL, "member %d: null adapter pointer", i);
    r_sum += r[i];
  }
  if (r_sum > L->max_rank)
    return fail(L, LORA_ERANK, "composed rank %d above max_rank %d", r_sum, L->max_rank);
  cudaStream_t side = static_cast<cudaStream_t>(side_);
  const size_t es = L->esize;
  const size_t K = L->K, N = L->N, R = L->R;
  // the slot's pool rows: fixed [slot R, slot R + R), or (pooled) its rank rounded up to 8
  // rows from the row allocator -- the rows it held before are returned first
  const int rows = L->pooled ? (r_sum + 7) / 8 * 8 : (int)R;
  int rb = L->rb_h[slot];
  if (L->pooled) {
    const int old_rb = L->rb_h[slot], old_rows = L->rows_h[slot];
    if (old_rows > 0) pool_free(L, old_rb, old_rows);
    rb = pool_alloc(L, rows);
    if (rb < 0) {
      if (old_rows > 0) {  // the slot keeps its rows and its adapter
        const int back = pool_alloc_at(L, old_rb, old_rows);
        (void)back;
      }
      return fail(L, LORA_ENOMEM, "the row pool has no %d free consecutive rows", rows);
    }
    L->rb_h[slot] = rb;
    L->rows_h[slot] = rows;
  }

  // never overwrite a slot under a forward still in flight, nor the staging buffer under
  // the previous load's transposition
  if (L->have_forward) LORA_CUDA(L, cudaStreamWaitEvent(side, L->last_forward, 0));
  char* At = static_cast<char*>(L->A_pool) + (size_t)rb * K * es;
  char* Bs = static_cast<char*>(L->B_pool) + (size_t)rb * N * es;
  SlotScales cols;
  for (int j = 0; j < kMaxSlotRank; ++j) cols.v[j] = 0.f;
  // member i occupies rank rows [o, o + r_i) of the slot: A_i^T in At, B_i in B
  for (int i = 0, o = 0; i < n; o += r[i], ++i) {
    LORA_CUDA(L, cudaStreamWaitEvent(side, L->stage_free, 0));
    LORA_CUDA(L, cudaMemcpyAsync(L->A_stage, A_src[i], K * r[i] * es, cudaMemcpyDefault, side));
    LORA_CUDA(L, launch_transpose_pad(L->A_stage, At + (size_t)o * K * es, (int)K, r[i], r[i],
                                      L->dtype == LORA_BF16, side));
    LORA_CUDA(L, cudaEventRecord(L->stage_free, side));
    LORA_CUDA(L, cudaMemcpyAsync(Bs + (size_t)o * N * es, B_src[i], (size_t)r[i] * N * es,
                                 cudaMemcpyDefault, side));
    const float c = weight[i] * (alpha[i] / (float)r[i]);
    for (int j = o; j < o + r[i]; ++j) cols.v[j] = c;
  }
  if (r_sum < rows) {
    LORA_CUDA(L, cudaMemsetAsync(At + (size_t)r_sum * K * es, 0, (size_t)(rows - r_sum) * K * es,
                                 side));
    LORA_CUDA(L, cudaMemsetAsync(Bs + (size_t)r_sum * N * es, 0, (size_t)(rows - r_sum) * N * es,
                                 side));
  }
  if (L->Bx_pool)  // the slot's rows of the B expand pool (rank rows >= r_sum: the zeros just set)
    LORA_CUDA(L, launch_pack_bx(Bs,
                                static_cast<char*>(L->Bx_pool) +
                                    (size_t)slot * N * expand_layout((int)R).wx * es,
                                (int)R, rows, (int)N, side));
  LORA_CUDA(L, launch_slot_meta(L->scale, (int)R, L->rank, L->loaded, slot, cols, r_sum, 1,
                                L->row_base, rb, side));
  bool varied = false;
  for (int j = 1; j < r_sum; ++j) varied |= cols.v[j] != cols.v[0];
  layer_set_percol(L, slot, varied);
  cudaEvent_t ev = layer_take_event(L);
  if (!ev) return fail(L, LORA_ECUDA, "cudaEventCreate failed");
  LORA_CUDA(L, cudaEventRecord(ev, side));
  L->pending.push_back(ev);
  return LORA_OK;
}

int load_adapter_slot(lora_layer_t* L, int slot, const void* A_src, const void* B_src, int r,
                      float alpha, void* side_) {
  const float one = 1.f;
  return load_adapter_slot_composed(L, slot, 1, &A_src, &B_src, &r, &alpha, &one, side_);
}

int unload_adapter_slot(lora_layer_t* L, int slot, void* side_) {
  if (!L) return LORA_EINVAL;
  if (slot < 0 || slot >= L->S) return fail(L, LORA_ESLOT, "slot %d outside [0, %d)", slot, L->S);
  cudaStream_t side = static_cast<cudaStream_t>(side_);
  if (L->have_forward) LORA_CUDA(L, cudaStreamWaitEvent(side, L->last_forward, 0));
  SlotScales none;
  for (int j = 0; j < kMaxSlotRank; ++j) none.v[j] = 0.f;
  // a pooled slot returns its rows (a later load reusing them waits for the last forward)
  const bool had_rows = L->pooled && L->rows_h[slot] > 0;
  if (had_rows) {
    pool_free(L, L->rb_h[slot], L->rows_h[slot]);
    L->rb_h[slot] = -1;
    L->rows_h[slot] = 0;
  }
  LORA_CUDA(L, launch_slot_meta(L->scale, L->R, L->rank, L->loaded, slot, none, 0, 0,
                                L->pooled ? L->row_base : nullptr, -1, side));
  layer_set_percol(L, slot, false);
  cudaEvent_t ev = layer_take_event(L);
  if (!ev) return fail(L, LORA_ECUDA, "cudaEventCreate failed");
  LORA_CUDA(L, cudaEventRecord(ev, side));
  L->pending.push_back(ev);
  return LORA_OK;
}

static int run_builder(lora_layer_t* L, cudaStream_t stream);

int set_batch_segments(lora_layer_t* L, const int32_t* token_slot_dev, int T, void* stream_) {
  if (!L) return LORA_EINVAL;
  if (T < 0 || T > L->T_max)
    return fail(L, LORA_EINVAL, "T=%d outside [0, max_tokens=%d]", T, L->T_max);
  if (T > 0 && !token_slot_dev) return fail(L, LORA_EINVAL, "null token_slot");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  // slot loads become visible to the builder (it reads the loaded flags)
  LORA_CUDA(L, wait_pending_loads(L, stream));

  L->T_batch = T;
  L->token_slot = token_slot_dev;
  L->launches = 0;
  // A bf16 batch of at most kDeltaMaxT rows is computed without its segments (the BGMV
  // kernel and the base GEMM read the ids directly, and the GEMM reports bad ids), so the
  // builder runs only if lora_get_segments asks for them.
  L->segments_pending = L->dtype == LORA_BF16 && T <= kDeltaMaxT;
  if (L->segments_pending) {
    LORA_CUDA(L, trace_mark(L, 0, stream));
    LORA_CUDA(L, trace_mark(L, 1, stream));
    return LORA_OK;
  }
  return run_builder(L, stream);
}

static int run_builder(lora_layer_t* L, cudaStream_t stream) {
  BuilderArgs a;
  a.token_slot = L->token_slot;
  a.T = L->T_batch;
  a.S = L->S;
  a.loaded = L->loaded;
  // work list: 128-row windows of perm for the tensor-core shrink (bf16), segment tiles of
  // the CUDA-core tile kernel (fp32)
  a.rows_per_tile = kTileRows;
  a.window_rows = L->dtype == LORA_BF16 ? kTcTileRows : 0;
  a.window_groups = L->dtype == LORA_BF16 ? sgmv_shrink_tc_groups((L->R + 15) / 16 * 16) : 0;
  a.row_slot = L->row_slot;
  a.perm = L->perm;
  a.seg_offsets = L->seg_offsets;
  a.seg_slot = L->seg_slot;
  a.tile_seg = L->tile_seg;
  a.tile_row0 = L->tile_row0;
  a.meta = L->meta;
  a.err = L->err;
  LORA_CUDA(L, trace_mark(L, 0, stream));
  LORA_CUDA(L, launch_segment_builder(a, stream));
  ++L->launches;
  LORA_CUDA(L, trace_mark(L, 1, stream));
  L->segments_pending = false;
  return LORA_OK;
}

int lora_forward(lora_layer_t* L, const void* x_dev, void* y_dev, int T, void* stream_) {
  if (!L) return LORA_EINVAL;
  if (L->T_batch < 0) return fail(L, LORA_ESTATE, "lora_forward before set_batch_segments");
  if (T != L->T_batch)
    return fail(L, LORA_ESTATE, "T=%d differs from the batch's T=%d", T, L->T_batch);
  if (T == 0) return LORA_OK;
  if (!x_dev || !y_dev) return fail(L, LORA_EINVAL, "null x or y");
  const size_t es = L->esize;
  const char* xb = static_cast<const char*>(x_dev);
  const char* yb = static_cast<const char*>(y_dev);
  if (xb < yb + (size_t)T * L->N * es && yb < xb + (size_t)T * L->K * es)
    return fail(L, LORA_EINVAL, "x and y overlap");
  if (L->dtype == LORA_BF16 &&
      (reinterpret_cast<uintptr_t>(x_dev) % 16 != 0 || reinterpret_cast<uintptr_t>(y_dev) % 16 != 0))
    return fail(L, LORA_EINVAL, "bf16 x and y must be 16-byte aligned");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  LORA_CUDA(L, wait_pending_loads(L, stream));

  const bool bf16 = L->dtype == LORA_BF16;
  const bool delta_mode = bf16 && T <= kDeltaMaxT;
  // planes of v the tensor-core shrink writes (its K split); the GEMM sums them
  const int v_split = bf16 && !delta_mode
                          ? sgmv_shrink_tc_split(T, L->K, L->S, L->num_sms, L->v_planes)
                          : 1;

  LORA_CUDA(L, trace_mark(L, 2, stream));
  if (delta_mode) {
    BgmvArgs ba;
    ba.x = x_dev;
    ba.token_slot = L->token_slot;
    ba.loaded = L->loaded;
    ba.T = T;
    ba.K = L->K;
    ba.N = L->N;
    ba.R = L->R;
    ba.S = L->S;
    ba.At_pool = L->A_pool;
    ba.B_pool = L->B_pool;
    ba.row_base = L->row_base;
    ba.pool_rows = L->P;
    ba.pooled = L->pooled;
    ba.scale = L->scale;
    ba.rank = L->rank;
    ba.delta = L->delta;
    ba.delta_rows = std::min(L->T_max, kDeltaMaxT);
    ba.err = L->err;
    ba.num_sms = L->num_sms;
    ba.per_column = L->percol_slots > 0;
    if (L->fp8) {
      // e4m3 base: the row quantiser, launched ahead of the BGMV kernel, counts x's rows on
      // q_ready, which the GEMM's loads wait for and its last CTA resets.  A forward that
      // stopped between those launches left the count set: clear it first.
      if (L->q_dirty) LORA_CUDA(L, cudaMemsetAsync(L->q_ready, 0, 2 * sizeof(int32_t), stream));
      L->q_dirty = true;
      ba.xq = L->xq;
      ba.sx = L->sx;
      ba.q_ready = L->q_ready;
    }
    LORA_CUDA(L, launch_bgmv_delta(ba, stream, &L->launches));
  } else if (bf16) {
    if (L->fp8) {
      // e4m3 base: the rows quantised first (a programmatic launch; the shrink below waits
      // for it, and the GEMM's loads of xq wait for its row count)
      if (L->q_dirty) LORA_CUDA(L, cudaMemsetAsync(L->q_ready, 0, 2 * sizeof(int32_t), stream));
      L->q_dirty = true;
      LORA_CUDA(L, launch_quant_rows_e4m3(x_dev, T, L->K, L->xq, L->sx, L->q_ready, L->num_sms,
                                          false, stream));
      ++L->launches;
    }
    ShrinkTcArgs sa;
    sa.x = x_dev;
    sa.T = T;
    sa.K = L->K;
    sa.R = L->R;
    sa.Rt = (L->R + 15) / 16 * 16;
    sa.scale = L->scale;
    sa.row_base = L->row_base;
    sa.perm = L->perm;
    sa.seg_offsets = L->seg_offsets;
    sa.seg_slot = L->seg_slot;
    sa.tile_seg = L->tile_seg;
    sa.tile_row0 = L->tile_row0;
    sa.meta = L->meta;
    sa.work = L->meta + 4;
    sa.v = L->v;
    sa.plane_stride = (size_t)L->T_max * L->R;
    sa.ks = v_split;
    sa.pool_rows = L->P;
    sa.v_rows = L->T_max;
    sa.err = L->err;
    sa.num_sms = L->num_sms;
    LORA_CUDA(L, launch_sgmv_shrink_tc(sa, L->tmap_a, stream));
    ++L->launches;
  } else {
    TileArgs ta;
    ta.x = x_dev;
    ta.K = L->K;
    ta.N = L->N;
    ta.R = L->R;
    ta.At_pool = L->A_pool;
    ta.B_pool = L->B_pool;
    ta.row_base = L->row_base;
    ta.scale = L->scale;
    ta.rank = L->rank;
    ta.perm = L->perm;
    ta.seg_offsets = L->seg_offsets;
    ta.seg_slot = L->seg_slot;
    ta.tile_seg = L->tile_seg;
    ta.tile_row0 = L->tile_row0;
    ta.meta = L->meta;
    ta.out = L->v;
    ta.out_rows = L->T_max;
    ta.pool_rows = L->P;
    ta.err = L->err;
    ta.max_tiles = (T + kTileRows - 1) / kTileRows + std::min(T, L->S);
    ta.num_sms = L->num_sms;
    LORA_CUDA(L, launch_lora_tile(ta, bf16, false, stream));
    ++L->launches;
  }
  LORA_CUDA(L, trace_mark(L, 3, stream));

  GemmArgs ga;
  ga.M = T;
  ga.N = L->N;
  ga.K = L->K;
  ga.x = x_dev;
  ga.W = L->Wp;
  ga.y = y_dev;
  ga.ex.mode = delta_mode ? kExpandDelta : kExpandV;
  ga.ex.row_slot = L->row_slot;
  ga.ex.token_slot = L->token_slot;
  ga.ex.loaded = L->loaded;
  ga.ex.S = L->S;
  ga.ex.v = L->v;
  ga.ex.v_planes = v_split;
  ga.ex.v_plane_stride = (size_t)L->T_max * L->R;
  ga.ex.delta = L->delta;
  ga.ex.delta_rows = std::min(L->T_max, kDeltaMaxT);
  ga.ex.v_rows = L->T_max;
  ga.ex.pool_rows = L->P;
  ga.ex.R = L->R;
  ga.ex.B_pool = L->B_pool;
  ga.ex.row_base = L->row_base;
  ga.ex.rank = L->rank;
  ga.err = L->err;
  ga.num_sms = L->num_sms;
  ga.xk = L->xk;
  ga.xk_floats = L->xk_floats;
  ga.sk_part = L->sk_part;
  ga.sk_sync = L->sk_sync;
  ga.force_bn = L->gemm_plan.block_n;
  ga.force_cs = L->gemm_plan.ksplit;
  ga.force_pair = L->gemm_plan.pair;
  ga.fp8 = L->fp8;
  ga.tmap_xq = L->fp8 ? &L->tmap_xq : nullptr;
  ga.sx = L->sx;
  ga.sw = L->sw;
  ga.q_ready = L->fp8 ? L->q_ready : nullptr;
  ga.tmap_delta = L->delta ? &L->tmap_delta : nullptr;
  LORA_CUDA(L, trace_mark(L, 4, stream));
  if (bf16) {
    LORA_CUDA(L, launch_gemm_tc(ga, L->tmap_w, L->Bx_pool ? L->tmap_bx : nullptr, stream,
                                &L->launches));
  } else {
    LORA_CUDA(L, launch_gemm_simt_f32(ga, stream));
    ++L->launches;
  }
  L->q_dirty = false;
  LORA_CUDA(L, trace_mark(L, 5, stream));

  if (!is_capturing(stream)) {
    LORA_CUDA(L, cudaEventRecord(L->last_forward, stream));
    L->have_forward = true;
  }
  return LORA_OK;
}

int lora_forward_host(lora_layer_t* L, const void* x_host, const int32_t* token_slot_host,
                      void* y_host, int T, void* stream_) {
  if (!L) return LORA_EINVAL;
  if (T < 0 || T > L->T_max)
    return fail(L, LORA_EINVAL, "T=%d outside [0, max_tokens=%d]", T, L->T_max);
  if (T > 0 && (!x_host || !token_slot_host || !y_host))
    return fail(L, LORA_EINVAL, "null host buffer");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  const size_t es = L->esize;
  if (T > 0) {
    LORA_CUDA(L, cudaMemcpyAsync(L->x_stage, x_host, (size_t)T * L->K * es, cudaMemcpyDefault,
                                 stream));
    LORA_CUDA(L, cudaMemcpyAsync(L->ids_stage, token_slot_host, (size_t)T * 4,
                                 cudaMemcpyDefault, stream));
  }
  int rc = set_batch_segments(L, L->ids_stage, T, stream_);
  if (rc != LORA_OK) return rc;
  rc = lora_forward(L, L->x_stage, L->y_stage, T, stream_);
  if (rc != LORA_OK) return rc;
  if (T > 0)
    LORA_CUDA(L, cudaMemcpyAsync(y_host, L->y_stage, (size_t)T * L->N * es, cudaMemcpyDefault,
                                 stream));
  return LORA_OK;
}

int lora_get_status(lora_layer_t* L, void* stream_) {
  if (!L) return LORA_EINVAL;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  int32_t flags = 0;
  LORA_CUDA(L, cudaStreamSynchronize(stream));
  LORA_CUDA(L, cudaMemcpy(&flags, L->err, 4, cudaMemcpyDeviceToHost));
  LORA_CUDA(L, cudaMemset(L->err, 0, 4));
  if (flags & LORA_ERRF_BOUNDS)
    return fail(L, LORA_EBOUNDS, "a device bounds check failed (flags=%d)", flags);
  if (flags & LORA_ERRF_TIMEOUT)
    return fail(L, LORA_ETIMEOUT, "a kernel pipeline wait timed out (flags=%d)", flags);
  if (flags & (LORA_ERRF_BAD_ID | LORA_ERRF_EMPTY_SLOT))
    return fail(L, LORA_EID, "token ids out of range or naming empty slots (flags=%d)", flags);
  return LORA_OK;
}

int lora_get_segments(lora_layer_t* L, int32_t* perm, int32_t* seg_offsets, int32_t* seg_slot,
                      int32_t* n_seg, int32_t* n_adapted, void* stream_) {
  if (!L) return LORA_EINVAL;
  if (!perm || !seg_offsets || !seg_slot || !n_seg || !n_adapted)
    return fail(L, LORA_EINVAL, "null output pointer");
  if (L->T_batch < 0) return fail(L, LORA_ESTATE, "no batch set");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (L->segments_pending) {
    const int rc = run_builder(L, stream);
    if (rc != LORA_OK) return rc;
  }
  LORA_CUDA(L, cudaStreamSynchronize(stream));
  int32_t meta[4];
  LORA_CUDA(L, cudaMemcpy(meta, L->meta, sizeof(meta), cudaMemcpyDeviceToHost));
  *n_seg = meta[0];
  *n_adapted = meta[1];
  if (meta[1] > 0)
    LORA_CUDA(L, cudaMemcpy(perm, L->perm, (size_t)meta[1] * 4, cudaMemcpyDeviceToHost));
  LORA_CUDA(L, cudaMemcpy(seg_offsets, L->seg_offsets, (size_t)(meta[0] + 1) * 4,
                          cudaMemcpyDeviceToHost));
  if (meta[0] > 0)
    LORA_CUDA(L, cudaMemcpy(seg_slot, L->seg_slot, (size_t)meta[0] * 4, cudaMemcpyDeviceToHost));
  return LORA_OK;
}

int lora_set_trace_events(lora_layer_t* L, void* const* events) {
  if (!L) return LORA_EINVAL;
  if (!events) {
    L->tracing = false;
    return LORA_OK;
  }
  for (int i = 0; i < 6; ++i)
    if (!events[i]) return fail(L, LORA_EINVAL, "null trace event %d", i);
  for (int i = 0; i < 6; ++i) L->trace[i] = static_cast<cudaEvent_t>(events[i]);
  L->tracing = true;
  return LORA_OK;
}

int lora_set_gemm_plan(lora_layer_t* L, int block_n, int k_split, int cta_pair) {
  if (!L) return LORA_EINVAL;
  if (block_n == 0) {
    L->gemm_plan = GemmPlan{0, 0, 0};
    return LORA_OK;
  }
  if ((block_n != 64 && block_n != 128 && block_n != 256) ||
      (k_split != 1 && k_split != 2 && k_split != 4) || block_n / k_split < 32 ||
      (cta_pair != 0 && cta_pair != 1) || (cta_pair && block_n < 128))
    return fail(L, LORA_EINVAL, "invalid GEMM plan (block_n %d, k_split %d, cta_pair %d)",
                block_n, k_split, cta_pair);
  const GemmPlan p{block_n, k_split, cta_pair};
  // the scratch must hold the exchange of every batch that may split K with this plan
  size_t need = 0;
  if (L->dtype == LORA_BF16)
    for (int m = 1; m <= std::min(L->T_max, kDeltaMaxT); ++m)
      need = std::max(need, gemm_tc_plan_exchange_floats(p, m, L->N));
  if (need > L->xk_floats) {
    LORA_CUDA(L, cudaDeviceSynchronize());  // earlier forwards may still use the scratch
    float* grown = nullptr;
    if (dmalloc(&grown, need) != cudaSuccess) {
      cudaGetLastError();
      return fail(L, LORA_ENOMEM, "split-K scratch of %zu floats", need);
    }
    if (L->xk) cudaFree(L->xk);
    L->xk = grown;
    L->xk_floats = need;
  }
  L->gemm_plan = p;
  return LORA_OK;
}

const char* lora_last_error(const lora_layer_t* L) { return L ? L->last_error : "null layer"; }

int lora_get_launch_count(const lora_layer_t* L) { return L ? L->launches : -1; }

void lora_layer_destroy(lora_layer_t* L) {
  if (!L) return;
  const int dev = L->device;
  int cur = dev;
  if (cudaGetDevice(&cur) == cudaSuccess && cur != dev) cudaSetDevice(dev);
  cudaDeviceSynchronize();
  free_all(L);
  delete L;
  if (cur != dev) cudaSetDevice(cur);
}

}  // extern "C"
