// lora_kernels.h -- internal (host-side) launchers of the layer's kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

namespace lora {

constexpr int kTileRows = 16;     // rows per segment tile of the CUDA-core tile kernel
constexpr int kTcTileRows = 128;  // rows per segment tile of the tensor-core shrink (MMA M)

// Function attributes are set per device, so the caches below that remember which were
// already set hold one entry per device ordinal (kAttrDevices of them) and are guarded by
// one process-wide mutex (several host threads may launch at once).
constexpr int kAttrDevices = 64;
inline std::mutex& attr_mutex() {
  static std::mutex m;
  return m;
}
// The current device's ordinal, or -1 if it cannot be read or is beyond kAttrDevices (the
// attribute is then set on every call: correct, only slower).
inline int attr_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kAttrDevices) return -1;
  return d;
}

// Kernels that run beside the base GEMM prefer the largest shared-memory carveout: an SM can
// only take a GEMM CTA (~200 KB of shared memory) while it holds CTAs of other kernels if
// its L1/shared split is already the one the GEMM needs.  Set once per kernel and device,
// outside stream capture.
template <typename Kernel>
inline cudaError_t prefer_max_smem_carveout(Kernel k, bool (&done)[kAttrDevices]) {
  const int d = attr_device();
  std::lock_guard<std::mutex> lock(attr_mutex());
  if (d >= 0 && done[d]) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                                       (int)cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess && d >= 0) done[d] = true;
  return e;
}

// Raise a kernel's dynamic shared-memory limit only when a launch needs more than any
// earlier launch on this device in this process (so launches under stream capture set no
// attribute).
template <typename Kernel>
inline cudaError_t ensure_smem_limit(Kernel k, int bytes, int (&cached)[kAttrDevices]) {
  const int d = attr_device();
  std::lock_guard<std::mutex> lock(attr_mutex());
  if (d >= 0 && bytes <= cached[d]) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && d >= 0) cached[d] = bytes;
  return e;
}

// ---- segment builder (builder.cu) ----
struct BuilderArgs {
  const int32_t* token_slot;  // [T]
  int T, S;
  const int32_t* loaded;  // [S]
  int rows_per_tile;
  // 0: the work list cuts every segment into tiles of <= rows_per_tile rows.  > 0: it lists
  // units instead: a window of window_rows consecutive positions of perm (tile_row0 = its
  // first position) with the first (tile_seg) of at most window_groups segments that
  // overlap it; a window spanning more segments gives several units.
  int window_rows;
  int window_groups;
  int32_t* row_slot;     // [T]
  int32_t* perm;         // [T]
  int32_t* seg_offsets;  // [S+1]
  int32_t* seg_slot;     // [S]
  int32_t* tile_seg;     // [T/rows_per_tile + S]
  int32_t* tile_row0;    // [T/rows_per_tile + S]
  int32_t* meta;         // [4] n_seg, T_a, n_tiles (window mode: [8], [4..5] zeroed)
  int32_t* err;
};
cudaError_t launch_segment_builder(const BuilderArgs& a, cudaStream_t stream);

// ---- low-rank half per segment tile (lora_tile.cu) ----
struct TileArgs {
  const void* x;  // [T,K] bf16 or f32
  int K, N, R;
  const void* At_pool;  // [P][K] rank rows (transposed slot A, K contiguous)
  const void* B_pool;   // [P][N] rank rows
  const int32_t* row_base;  // [S] first pool row of each slot
  const float* scale;   // [S][R]: the scale of each rank column of a slot
  const int32_t* rank;  // [S]
  const int32_t* perm, *seg_offsets, *seg_slot, *tile_seg, *tile_row0, *meta;
  float* out;           // v [out_rows][R] fp32
  int out_rows;         // rows of out (T_max)
  int pool_rows;        // P: rows of the A and B pools
  int32_t* err;         // the layer's device flags (debug-flavour bounds checks)
  int max_tiles;        // upper bound of the builder's tile count (grid sizing)
  int num_sms;
};
// Launched with programmatic stream serialization (it waits for the builder itself).
cudaError_t launch_lora_tile(const TileArgs& a, bool bf16, bool delta, cudaStream_t stream);

// ---- SGMV shrink on the tensor cores (sgmv_tc.cu) ----
struct ShrinkTcArgs {
  const void* x;  // [T,K] bf16
  int T, K, R;    // R: slot rank width (multiple of 8); v has R columns
  int Rt;         // MMA N: R rounded up to 16
  const float* scale;  // [S][R]: the scale of each rank column of a slot
  const int32_t* row_base;  // [S] first row of each slot in the A pool (the TMA row)
  const int32_t* perm, *seg_offsets, *seg_slot, *tile_seg, *tile_row0, *meta;
  int32_t* work;       // [2] item and exit counters, zero between launches (builder zeroes)
  float* v;            // [max_planes][T_max][R] fp32 partial sums over K ranges, scaled
  size_t plane_stride; // floats between planes (T_max * R)
  int ks;              // K split (planes written), from sgmv_shrink_tc_split
  int pool_rows;       // P: rows of the A pool (debug-flavour bounds checks)
  int v_rows;          // rows of a plane of v (T_max)
  int32_t* err;
  int num_sms;
};
// Segments per window unit (the MMA stacks their A blocks along N) for a rank width Rt.
int sgmv_shrink_tc_groups(int Rt);
// The K split for a batch of T rows over S slots (the number of v planes the shrink writes),
// at most max_planes.
int sgmv_shrink_tc_split(int T, int K, int S, int num_sms, int max_planes);
// tmap_a: the A pool [P rows][K] bf16 with a (64 x Rt) box.  Writes planes 0 .. ks - 1 of
// v.  Launched with programmatic stream serialization (it waits for the builder itself).
cudaError_t launch_sgmv_shrink_tc(const ShrinkTcArgs& a, const CUtensorMap& tmap_a,
                                  cudaStream_t stream);

// ---- decode batches: BGMV shrink + expand into an fp32 delta (lora_tile.cu) ----
struct BgmvArgs {
  const void* x;  // [T,K] bf16
  const int32_t* token_slot;  // [T] as given by the caller
  const int32_t* loaded;      // [S]
  int T, K, N, R, S;
  const void* At_pool;  // [P][K] rank rows
  const void* B_pool;   // [P][N] rank rows
  const int32_t* row_base;  // [S] first pool row of each slot (-1: none)
  int pool_rows;        // P
  bool pooled;          // slots placed by the row allocator (else slot s at row s * R)
  const float* scale;   // [S][R]: the scale of each rank column of a slot
  const int32_t* rank;  // [S]
  float* delta;         // [delta_rows][N] fp32
  int delta_rows;       // rows of the delta buffer
  int32_t* err;         // the layer's device flags (debug-flavour bounds checks)
  int num_sms;
  bool per_column;      // some slot's columns carry different scales (a composition)
  // e4m3 base: x [T][K] is also quantised per row into xq / sx by a launch of the row
  // quantiser ahead of the BGMV kernel, which counts the rows on q_ready[0]; null: bf16
  uint8_t* xq = nullptr;
  float* sx = nullptr;
  int32_t* q_ready = nullptr;
};
// Launched with programmatic stream serialization; it does not wait for the builder.
// launches (may be null): incremented per kernel launched (the e4m3 quantiser, the BGMV).
cudaError_t launch_bgmv_delta(const BgmvArgs& a, cudaStream_t stream, int* launches = nullptr);

// ---- the tensor-core expand's layout of a slot's rank columns ----
// v of a row is split as v = hi + lo (two bf16) and multiplied by the slot's B^T on the
// tensor cores in 64-wide K blocks.  Rank width R <= 32: one block per slot, columns
// [0, 32) = hi (zero beyond R) and [32, 64) = lo, against [B^T | B^T].  R > 32: the halves
// are padded to rx = 64 or 128 and take rx / 64 blocks each (hi blocks, then lo blocks),
// all against B^T padded to rx columns.  wx = columns of a slot's row in the B expand pool.
struct ExpandLayout {
  int wx;   // B expand pool width: 64 (R <= 32) or rx
  int nbs;  // K blocks per slot
  int rx;   // padded width of each half
};
__host__ __device__ inline ExpandLayout expand_layout(int R) {
  if (R <= 32) return ExpandLayout{64, 1, 32};
  const int rx = R <= 64 ? 64 : 128;
  return ExpandLayout{rx, 2 * rx / 64, rx};
}
// The 16-column K chunks of a slot's expand block b (0 <= b < nbs) that hold rank columns
// (bit kk set); the others are padding, zero in both halves of the product.
__host__ __device__ inline unsigned expand_chunks(const ExpandLayout& xl, int R, int b) {
  if (xl.nbs == 1) return R > 16 ? 0xFu : 0x5u;  // hi in columns [0, R), lo in [32, 32 + R)
  const int sub = b % (xl.rx / 64);
  const int real = R - 64 * sub < 64 ? R - 64 * sub : 64;
  return (1u << ((real + 15) / 16)) - 1u;
}

// ---- base GEMM with the low-rank term added in its epilogue ----
// kExpandV: y += [v^hi | v^lo] [B^T ; B^T] as extra tensor-core K blocks (large batches).
// kExpandDelta: y += delta, the fp32 [T,N] low-rank term a BGMV kernel expanded.
enum ExpandMode { kExpandV = 0, kExpandDelta = 1 };
struct ExpandArgs {
  int mode;                 // kExpandV: y += v B_slot;  kExpandDelta: y += delta
  const int32_t* row_slot;  // [T] builder-checked slots, -1 = base only (v mode)
  const int32_t* token_slot;  // [T] caller's ids, checked against loaded (delta mode)
  const int32_t* loaded;      // [S]
  int S;
  const float* v;           // [planes][T_max][R] fp32, scaled by alpha / r   (v mode):
  int v_planes;             //   v of a row = the sum of its planes, in plane order
  size_t v_plane_stride;    //   floats between planes
  const float* delta;       // [delta_rows][N] fp32                          (delta mode)
  int delta_rows;           // rows of the delta buffer
  int v_rows;               // rows of a plane of v (T_max)
  int pool_rows;            // P: rows of the B pool
  int R;
  const void* B_pool;   // [P][N] rank rows
  const int32_t* row_base;  // [S] first pool row of each slot
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
  float* xk;         // split K: scratch for the exchanged fp32 partials (L2-resident)
  size_t xk_floats;  // its capacity (gemm_tc_exchange_floats of the batch)
  int force_bn, force_cs, force_pair;  // tcgen05 tiling fixed by the caller (force_bn 0: auto)
  // columns [n_begin, n_end) of y computed by this launch (0, N for the whole product; the
  // launcher sets them when it splits a batch over two launches), and whether the launch
  // lets the next kernel on its stream start at once (the second launch of such a split)
  int n_begin = 0, n_end = 0;
  bool trigger_next = false;
  // stream-K (large batches): fp32 partial per CTA [num_sms][128][256] and sync words
  // {epoch, exit count, flag per CTA} (zeroed at allocation); null: no stream-K
  float* sk_part;
  int32_t* sk_sync;
  // e4m3 base (delta mode only): x quantised per row (tmap_xq: [M rows][K] bytes, (128 x
  // 128) box), W per column (tmap_w3: [N rows][K] bytes); y = sx[row] sw[col] (xq wq) + delta
  bool fp8 = false;
  const CUtensorMap* tmap_xq = nullptr;
  const float* sx = nullptr;  // [M]
  const float* sw = nullptr;  // [N rounded up to 256], zero past N
  // xq and sx are written by the low-rank kernel running beside this one: q_ready[0] counts
  // the rows made visible, and every CTA's producer waits (bounded) for it to reach M
  // before its first load of xq.  The last launch of a batch (q_reset) also counts its CTAs
  // on q_ready[1], and the last of them sets both words back to 0 for the next batch.
  int32_t* q_ready = nullptr;
  bool q_reset = false;
  // delta mode (required there): the map of the delta buffer (encode_tmap_delta), through
  // which the epilogue's delta tile arrives by TMA
  const CUtensorMap* tmap_delta = nullptr;
};
// tcgen05 / TMEM / TMA kernel (gemm_tc.cu).  tmap_w3 holds the layer's cached maps of the
// packed weight for N tiles of 256, 128 and 64 rows (in that order); tmap_bx3 the maps of
// the B expand pool [S*N rows][wx] with (64 x 256/128/64) boxes (v mode; may be null in
// delta mode).
// launches (may be null): incremented per kernel launched (1, or 2 for a split batch).
cudaError_t launch_gemm_tc(const GemmArgs& a, const CUtensorMap* tmap_w3,
                           const CUtensorMap* tmap_bx3, cudaStream_t stream,
                           int* launches = nullptr);
constexpr int kTcTileN[3] = {256, 128, 64};

// ---- e4m3 base (fp8.cu) ----
// 2-D tensor map over [rows][K] bytes (K-major, K a multiple of 16) with a (128 x box_rows)
// box and the 128-byte swizzle.
cudaError_t encode_tmap_u8(CUtensorMap* map, const void* base, int rows, int K, int box_rows);
// x [T][K] bf16 -> xq [T][K] e4m3 and sx [T]: sx = max |x[row]| / 448 (1 for a zero row),
// xq = e4m3(x / sx), round to nearest even, saturating.  CTA b takes rows b, b + gridDim.x,
// ... (beside_bgmv: one CTA per SM, sized to share the SM with the decode BGMV and GEMM;
// else two per SM); each CTA counts its rows on q_ready once their stores are visible.
// Programmatic dependent launch: it waits for the previous kernel on the stream (which may
// read xq or write x) and then at once lets the next one launch.
cudaError_t launch_quant_rows_e4m3(const void* x, int T, int K, uint8_t* xq, float* sx,
                                   int32_t* q_ready, int num_sms, bool beside_bgmv,
                                   cudaStream_t stream);
// W [K][N] bf16 -> Wq [N][K] e4m3 (transposed, K-major) and sw [N]: per column as above.
cudaError_t launch_quant_cols_e4m3(const void* W, int K, int N, uint8_t* Wq, float* sw,
                                   cudaStream_t stream);
// Encode a 2-D bf16 tensor map for a K-major [rows, K] matrix with a (64 x box_rows) box.
cudaError_t encode_tmap_bf16(CUtensorMap* map, const void* base, int rows, int K, int box_rows);
// Encode the map of an fp32 delta buffer [rows][N] (N a multiple of 4) with (32 x 128)
// boxes and the 128-byte swizzle: a box lands as 128 rows of 128 bytes, 16-byte chunk q of
// row r at chunk q ^ (r & 7); reads past the buffer fill zeros.
cudaError_t encode_tmap_delta(CUtensorMap* map, const float* base, int rows, int N);
struct GemmPlan {
  int block_n;  // N tile: 256, 128 or 64
  int ksplit;   // K ranges per output tile, 1..4
  int pair;     // 1: CTA pairs (cta_group::2 MMAs, 256-row tiles, N tile 256 or 128)
};
// allow_pair = false keeps every tile on one CTA (the e4m3 base in v mode, where pairs
// measured slower).
GemmPlan gemm_tc_plan(int M, int N, int K, int num_sms, bool allow_split, int slots,
                      bool allow_pair = true);
// Floats of split-K exchange scratch the tcgen05 GEMM needs for an M-row batch with the
// K split allowed (0 when its plan does not split K).
size_t gemm_tc_exchange_floats(int M, int N, int K, int num_sms);
// The same for a given plan.
size_t gemm_tc_plan_exchange_floats(const GemmPlan& p, int M, int N);

// fp32 SIMT path (gemm_simt.cu)
cudaError_t launch_gemm_simt_f32(const GemmArgs& a, cudaStream_t stream);

// ---- slot table maintenance (slots.cu) ----
// At[j][k] = j < r ? A[k][j] : 0, for j < R, k < K.
cudaError_t launch_transpose_pad(const void* A_kr, void* At_rk, int K, int r, int R, bool bf16,
                                 cudaStream_t stream);
// Wp[n][k] = W[k][n] (bf16 base weight packing).
cudaError_t launch_pack_w_bf16(const void* W_kn, void* W_nk, int K, int N, cudaStream_t stream);
// B expand pool row block of one slot: Bx[n][j] from B [R][N] (see expand_layout; the
// layout is that of slot width R, rows of B at or beyond `rows` read as zero).
cudaError_t launch_pack_bx(const void* B_rn, void* Bx_nw, int R, int rows, int N,
                           cudaStream_t stream);
// A slot's metadata: the scale of each of its R rank columns (an adapter's alpha / r on its
// r columns; a composition's w_i alpha_i / r_i on the columns of member i; 0 beyond), its
// rank and its loaded flag.
constexpr int kMaxSlotRank = 128;
struct SlotScales {
  float v[kMaxSlotRank];
};
// Also sets row_base[slot] = rb when row_base is not null.
cudaError_t launch_slot_meta(float* scale, int R, int32_t* rank, int32_t* loaded, int slot,
                             const SlotScales& cols, int r, int is_loaded, int32_t* row_base,
                             int rb, cudaStream_t stream);

}  // namespace lora
