// lora_tile.cu -- the low-rank half of the layer: per segment tile, the shrink v = x A_slot
// (fp32 layers); for decode batches, BGMV shrink + expand into the fp32 delta [rows][N] =
// scale * v B_slot, rows of delta_rows.
//
// "Serving multiple LoRAs: segmented matrix multiplies and adapter scheduling", section
// "Not merging the weights, computing in batches": SGMV groups the tokens of one adapter
// and runs one small matrix multiply per segment; BGMV gathers each token's A and B; real
// kernels shrink (x -> xA, down to r) and then expand ((xA)B) and add to the base output.
// "Serving LoRA adapters ..." (vLLM) Step 4: the shrink result is an fp32 buffer of rank
// width.
//
// Work list: the segment builder cut every segment into tiles of <= 16 rows sharing one
// slot.  One CTA (8 warps) takes one tile at a time:
//   shrink   warp w owns rank columns [w*JW, w*JW + JW); its lanes split K into 16-byte
//            vectors and accumulate a block of RB rows x JW columns (RB * JW <= 16) in
//            registers, so each A vector is loaded once per RB rows and each lane keeps
//            RB + JW independent 16-byte loads in flight; a butterfly shuffle sums the
//            lanes.  v (fp32, already multiplied by alpha / r) goes to shared memory.
//   v is written to global memory [row][j]; the base GEMM's epilogue expands it.  (Decode
//   batches run the BGMV kernels further below, which expand into an fp32 delta.)
// Only the true rank r of the slot is read: the zero padding of the slot never is.
//
// Launch: programmatic dependent launch.  The kernel lets the next kernel (the base GEMM,
// whose main loop needs nothing from it) launch at once, then waits for the segment
// builder's results before reading them.
#include <algorithm>

#include "lora_common.cuh"
#include "lora_kernels.h"

namespace lora {

static constexpr int kTileThreads = 256;

template <typename T>
struct Vec16;  // 16 bytes of T widened to fp32

template <>
struct Vec16<__nv_bfloat16> {
  static constexpr int N = 8;
  uint4 raw;
  __device__ __forceinline__ void load(const __nv_bfloat16* p) {
    raw = __ldg(reinterpret_cast<const uint4*>(p));
  }
  __device__ __forceinline__ float operator[](int e) const {
    const uint32_t w = e < 2 ? raw.x : e < 4 ? raw.y : e < 6 ? raw.z : raw.w;
    return (e & 1) ? bf16_hi(w) : bf16_lo(w);
  }
};

template <>
struct Vec16<float> {  // 4 floats
  static constexpr int N = 4;
  float4 raw;
  __device__ __forceinline__ void load(const float* p) {
    raw = __ldg(reinterpret_cast<const float4*>(p));
  }
  __device__ __forceinline__ float operator[](int e) const {
    return e == 0 ? raw.x : e == 1 ? raw.y : e == 2 ? raw.z : raw.w;
  }
};

// One float: the fp32 path when K is not a multiple of 4 or x is not 16-byte aligned.
struct Scalar32 {
  static constexpr int N = 1;
  float raw;
  __device__ __forceinline__ void load(const float* p) { raw = __ldg(p); }
  __device__ __forceinline__ float operator[](int) const { return raw; }
};

// Shrink of one tile by one warp: v_s[q][j] = sc[j] * sum_k x[row_q][k] * At[j][k] for the
// warp's JW rank columns.  K is a multiple of the vector width (checked on the host).
template <typename T, typename V, int JW>
__device__ __forceinline__ void shrink_tile_warp(const T* __restrict__ x, int K,
                                                 const T* __restrict__ At, int r,
                                                 const int* rows_s, int nr,
                                                 const float* __restrict__ sc, float* v_s,
                                                 int vstride, int warp, int lane) {
  constexpr int RB = (16 / JW) < 8 ? (16 / JW) : 8;  // rows per register block
  constexpr int VEC = V::N;
  const int j0 = warp * JW;
  if (j0 >= r) return;
  const T* ar[JW];
#pragma unroll
  for (int jj = 0; jj < JW; ++jj) ar[jj] = At + (size_t)min(j0 + jj, r - 1) * K;

  for (int q0 = 0; q0 < nr; q0 += RB) {
    const T* xr[RB];
#pragma unroll
    for (int qq = 0; qq < RB; ++qq) xr[qq] = x + (size_t)rows_s[min(q0 + qq, nr - 1)] * K;
    float acc[RB][JW];
#pragma unroll
    for (int qq = 0; qq < RB; ++qq)
#pragma unroll
      for (int jj = 0; jj < JW; ++jj) acc[qq][jj] = 0.f;

    for (int k = lane * VEC; k < K; k += 32 * VEC) {
      V xv[RB], av[JW];
#pragma unroll
      for (int qq = 0; qq < RB; ++qq) xv[qq].load(xr[qq] + k);
#pragma unroll
      for (int jj = 0; jj < JW; ++jj) av[jj].load(ar[jj] + k);
#pragma unroll
      for (int e = 0; e < VEC; ++e)
#pragma unroll
        for (int qq = 0; qq < RB; ++qq)
#pragma unroll
          for (int jj = 0; jj < JW; ++jj) acc[qq][jj] = fmaf(xv[qq][e], av[jj][e], acc[qq][jj]);
    }
#pragma unroll
    for (int qq = 0; qq < RB; ++qq)
#pragma unroll
      for (int jj = 0; jj < JW; ++jj) {
        float s = acc[qq][jj];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        acc[qq][jj] = s;
      }
    if (lane == 0) {
#pragma unroll
      for (int qq = 0; qq < RB; ++qq)
#pragma unroll
        for (int jj = 0; jj < JW; ++jj)
          if (q0 + qq < nr && j0 + jj < r)
            v_s[(q0 + qq) * vstride + j0 + jj] = sc[j0 + jj] * acc[qq][jj];
    }
  }
}

// <= 128 registers a thread: two CTAs of this kernel, or one beside a base-GEMM CTA, fit
// on an SM, so the GEMM launched after it can start while it runs.
template <typename T, typename V>
__global__ void __launch_bounds__(kTileThreads, 2)
    lora_tile_kernel(const T* __restrict__ x, int K, int N, int R,
                     const T* __restrict__ At_pool, const T* __restrict__ B_pool,
                     const int32_t* __restrict__ row_base,
                     const float* __restrict__ scale, const int32_t* __restrict__ rank,
                     const int32_t* __restrict__ perm, const int32_t* __restrict__ seg_offsets,
                     const int32_t* __restrict__ seg_slot, const int32_t* __restrict__ tile_seg,
                     const int32_t* __restrict__ tile_row0, const int32_t* __restrict__ meta,
                     float* __restrict__ out /* v [out_rows][R] */, int out_rows, int pool_rows,
                     int32_t* __restrict__ err) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ int rows_s[kTileRows];
  __shared__ float v_s[kTileRows * 129];
  const int vstride = R + 1;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_tiles = meta[2];

  for (int t = blockIdx.x; t < n_tiles; t += gridDim.x) {
    const int g = tile_seg[t];
    const int s = seg_slot[g];
    const int r = rank[s];
    const float* sc = scale + (size_t)s * R;  // the slot's column scales
    const int p0 = tile_row0[t];
    const int nr = min(kTileRows, seg_offsets[g + 1] - p0);
    if (tid < nr) rows_s[tid] = perm[p0 + tid];
    __syncthreads();
    const int rb = row_base[s];  // the slot's first pool row
    if (!LORA_IN_BOUNDS(rb >= 0 && rb + r <= pool_rows, err)) {
      __syncthreads();  // rows_s is rewritten by the next tile
      continue;
    }
    const T* At = At_pool + (size_t)rb * K;
    if (r <= 8)
      shrink_tile_warp<T, V, 1>(x, K, At, r, rows_s, nr, sc, v_s, vstride, warp, lane);
    else if (r <= 16)
      shrink_tile_warp<T, V, 2>(x, K, At, r, rows_s, nr, sc, v_s, vstride, warp, lane);
    else if (r <= 32)
      shrink_tile_warp<T, V, 4>(x, K, At, r, rows_s, nr, sc, v_s, vstride, warp, lane);
    else if (r <= 64)
      shrink_tile_warp<T, V, 8>(x, K, At, r, rows_s, nr, sc, v_s, vstride, warp, lane);
    else
      shrink_tile_warp<T, V, 16>(x, K, At, r, rows_s, nr, sc, v_s, vstride, warp, lane);
    __syncthreads();
    for (int i = tid; i < nr * r; i += kTileThreads) {
      const int q = i / r, j = i - q * r;
      if (LORA_IN_BOUNDS(rows_s[q] >= 0 && rows_s[q] < out_rows, err))
        out[(size_t)rows_s[q] * R + j] = v_s[q * vstride + j];
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------------------
// Delta mode for small (decode) batches: BGMV, one row per thread-block cluster of CS CTAs.
// "Serving multiple LoRAs ...": BGMV -- each token gathers its own adapter's A and B by
// index and does a small matrix x vector.  The row's ids are checked here (slot in range
// and loaded), so the kernel needs nothing from the segment builder and runs alongside it.
// CTA c of the cluster:
//   1. partial v over K range c: warp w owns rank columns [w*JW, w*JW + JW) in groups of 4;
//      its lanes split the range into 16-byte vectors, with the K loop unrolled so a lane's
//      loads of the group's A rows and of x are in flight together;
//   2. the CS partials are summed through distributed shared memory (double-buffered, one
//      cluster barrier per row) and scaled by alpha / r;
//   3. delta[row][n] = sum_j v_j B_slot[j][n] over N range c, fp32, each thread loading up
//      to 16 rank rows of B for its 8 columns at once.
// ---------------------------------------------------------------------------------------
static constexpr int kBgmvThreads = 128;

__global__ void __launch_bounds__(kBgmvThreads, 8)  // <= 64 registers: 4 CTAs fit beside a GEMM CTA
    bgmv_delta_kernel(const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ token_slot,
                      const int32_t* __restrict__ loaded, int T, int K, int N, int R, int S,
                      const __nv_bfloat16* __restrict__ At_pool,
                      const __nv_bfloat16* __restrict__ B_pool,
                      const int32_t* __restrict__ row_base, const float* __restrict__ scale,
                      const int32_t* __restrict__ rank, float* __restrict__ delta,
                      int delta_rows, int pool_rows, int32_t* __restrict__ err, int kchunk,
                      int nchunk) {
  griddep_wait();  // the previous kernel's writes (x, the delta it read) are settled
  griddep_launch_dependents();  // the base GEMM's main loop may start now
  __shared__ float v_part[2][128];
  __shared__ float v_s[128];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t csize;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(csize));
  const uint32_t c = cluster_ctarank();
  const int n_clusters = gridDim.x / csize;
  const int k0 = c * kchunk, k1 = min(K, k0 + kchunk);
  const int nb0 = c * nchunk, nb1 = min(N, nb0 + nchunk);

  int buf = 0;
  for (int row = blockIdx.x / csize; row < T; row += n_clusters) {
    const int s = token_slot[row];
    if (s < 0 || s >= S || loaded[s] == 0) continue;  // base only (same decision in all CTAs)
    const int r = rank[s];
    const float* sc = scale + (size_t)s * R;  // the slot's column scales
    const __nv_bfloat16* xr = x + (size_t)row * K;
    const int rb = row_base[s];  // the slot's first pool row
    // (the same decision in all CTAs of the cluster: they read the same rb and r)
    if (!LORA_IN_BOUNDS(rb >= 0 && rb + r <= pool_rows && row < delta_rows, err)) continue;
    const __nv_bfloat16* At = At_pool + (size_t)rb * K;
    float* vp = v_part[buf];
    buf ^= 1;

    // ---- 1. partial v over [k0, k1) ----
    const int jw = (r + 3) / 4;  // rank columns per warp
    for (int g0 = warp * jw; g0 < min(r, warp * jw + jw); g0 += 4) {
      const __nv_bfloat16* ar[4];
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) ar[jj] = At + (size_t)min(g0 + jj, r - 1) * K;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
      for (int k = k0 + lane * 8; k < k1; k += 256) {
        Vec16<__nv_bfloat16> xv, av[4];
        xv.load(xr + k);
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) av[jj].load(ar[jj] + k);
#pragma unroll
        for (int e = 0; e < 8; ++e)
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) acc[jj] = fmaf(xv[e], av[jj][e], acc[jj]);
      }
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc[jj] += __shfl_xor_sync(0xffffffffu, acc[jj], o);
      }
      if (lane == 0) {
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
          if (g0 + jj < min(r, warp * jw + jw)) vp[g0 + jj] = acc[jj];
      }
    }
    __syncwarp();
    cluster_sync_all();  // every CTA's partial of this row is in its shared memory

    // ---- 2. sum the partials of the cluster ----
    if (tid < r) {
      const uint32_t local = smem_u32(vp + tid);
      float sum = 0.f;
      for (uint32_t d = 0; d < csize; ++d) sum += dsmem_ld(dsmem_map(local, d));
      v_s[tid] = sc[tid] * sum;
    }
    __syncthreads();

    // ---- 3. delta over [nb0, nb1) ----
    const __nv_bfloat16* Bs = B_pool + (size_t)rb * N;
    float* drow = delta + (size_t)row * N;
    for (int n = nb0 + tid * 8; n < nb1; n += kBgmvThreads * 8) {
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int j0 = 0; j0 < r; j0 += 16) {
        uint4 b[16];
#pragma unroll
        for (int jj = 0; jj < 16; ++jj)
          b[jj] = (j0 + jj < r)
                      ? __ldg(reinterpret_cast<const uint4*>(Bs + (size_t)(j0 + jj) * N + n))
                      : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
          const float vj = (j0 + jj < r) ? v_s[j0 + jj] : 0.f;
          acc[0] = fmaf(vj, bf16_lo(b[jj].x), acc[0]);
          acc[1] = fmaf(vj, bf16_hi(b[jj].x), acc[1]);
          acc[2] = fmaf(vj, bf16_lo(b[jj].y), acc[2]);
          acc[3] = fmaf(vj, bf16_hi(b[jj].y), acc[3]);
          acc[4] = fmaf(vj, bf16_lo(b[jj].z), acc[4]);
          acc[5] = fmaf(vj, bf16_hi(b[jj].z), acc[5]);
          acc[6] = fmaf(vj, bf16_lo(b[jj].w), acc[6]);
          acc[7] = fmaf(vj, bf16_hi(b[jj].w), acc[7]);
        }
      }
      float4* d = reinterpret_cast<float4*>(drow + n);
      d[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      d[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
    __syncthreads();  // v_s is rewritten by the next row
  }
  __syncwarp();
  cluster_sync_all();  // no CTA leaves while a peer may still read its partials
}

static constexpr int kSlotMaxT = 512;  // largest decode batch (the delta buffer's rows)

// ---------------------------------------------------------------------------------------
// BGMV for decode batches (rank width <= 32, T <= 512): one CTA per slot at a time (CTAs
// loop over slots), delta[row, :] = (alpha/r) (x[row] A_s) B_s for the slot's rows.
// The rows are found with one scan of the id vector.  Both halves stream the slot's
// matrices through registers, each read once per group of rows:
//   shrink  thread t takes 16-byte chunks t, t + 256, ... of K; the loads of a chunk (the
//           rows' x and a batch of 16 rank rows of A_s^T) are issued together; the block
//           sums the partials (warp shuffles, then one shared-memory pass) into v (fp32).
//   expand  thread t takes 8-column chunks t, t + 256, ... of N; a batch of 16 rank rows of
//           B_s is loaded together and applied to the group's rows; the fp32 delta rows
//           are written once.
// Few registers (see below) and ~5 KB of shared memory, so that a CTA fits on an SM beside
// a base GEMM CTA and runs while its main loop does.
// ---------------------------------------------------------------------------------------
static constexpr int kStrThreads = 256;
static constexpr int kStrRedMax = 64;  // rows x rank columns of one shrink pass

// v of NQ rows (rank columns < RMAX) into vdst[q][j]; all threads of the CTA.  Thread
// tid < NQ * RMAX finishes column j = tid % RMAX of row tid / RMAX and scales it by `sc`,
// the scale of that column (a register: a shared-memory table here costs the kernel
// registers it does not have).
template <int RMAX, int NQ>
__device__ __forceinline__ void stream_shrink(const __nv_bfloat16* __restrict__ x,
                                              const int* rows, int K, const __nv_bfloat16* At,
                                              int r, float sc, float (*red)[kStrRedMax],
                                              float (*vdst)[32]) {
  static_assert(NQ * RMAX <= kStrThreads, "one finished column per thread");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float acc[NQ][RMAX];
#pragma unroll
  for (int q = 0; q < NQ; ++q)
#pragma unroll
    for (int j = 0; j < RMAX; ++j) acc[q][j] = 0.f;
  for (int e = tid; e < K / 8; e += kStrThreads) {
    // the loads of a chunk go out together: the rows' x (through L2: after the e4m3 row
    // quantiser this kernel does not wait for the kernel that may have written x), then a
    // batch of 16 rank rows of A
    uint4 xv[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q)
      xv[q] = __ldcg(reinterpret_cast<const uint4*>(x + (size_t)rows[q] * K + e * 8));
#pragma unroll
    for (int j0 = 0; j0 < RMAX; j0 += 16) {
      if (j0 >= r) break;
      uint4 av[16];
#pragma unroll
      for (int jj = 0; jj < 16; ++jj)
        av[jj] = j0 + jj < r
                     ? __ldg(reinterpret_cast<const uint4*>(At + (size_t)(j0 + jj) * K + e * 8))
                     : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        const float xf[8] = {bf16_lo(xv[q].x), bf16_hi(xv[q].x), bf16_lo(xv[q].y),
                             bf16_hi(xv[q].y), bf16_lo(xv[q].z), bf16_hi(xv[q].z),
                             bf16_lo(xv[q].w), bf16_hi(xv[q].w)};
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
          float t = acc[q][j0 + jj];
          t = fmaf(xf[0], bf16_lo(av[jj].x), t);
          t = fmaf(xf[1], bf16_hi(av[jj].x), t);
          t = fmaf(xf[2], bf16_lo(av[jj].y), t);
          t = fmaf(xf[3], bf16_hi(av[jj].y), t);
          t = fmaf(xf[4], bf16_lo(av[jj].z), t);
          t = fmaf(xf[5], bf16_hi(av[jj].z), t);
          t = fmaf(xf[6], bf16_lo(av[jj].w), t);
          t = fmaf(xf[7], bf16_hi(av[jj].w), t);
          acc[q][j0 + jj] = t;
        }
      }
    }
  }
  // block sum: warp shuffles, then one shared-memory pass
#pragma unroll
  for (int q = 0; q < NQ; ++q)
#pragma unroll
    for (int j = 0; j < RMAX; ++j) {
      float t = acc[q][j];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
      if (lane == 0) red[warp][q * RMAX + j] = t;
    }
  __syncthreads();
  for (int i = tid; i < NQ * RMAX; i += kStrThreads) {  // one pass: i == tid
    const int q = i / RMAX, j = i - q * RMAX;
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < kStrThreads / 32; ++w) sum += red[w][i];
    vdst[q][j] = j < r ? sc * sum : 0.f;
  }
  __syncthreads();  // red is rewritten by the next pass
}

// delta rows of NG rows from v_s[0 .. NG) and the slot's B rows; all threads of the CTA.
template <int RMAX, int NG>
__device__ __forceinline__ void stream_expand(const __nv_bfloat16* __restrict__ Bs, int N, int r,
                                              const float (*v_s)[32], const int* rows,
                                              float* __restrict__ delta, int delta_rows,
                                              int32_t* __restrict__ err) {
  for (int e = threadIdx.x; e < N / 8; e += kStrThreads) {
    float o[NG][8];
#pragma unroll
    for (int q = 0; q < NG; ++q)
#pragma unroll
      for (int i = 0; i < 8; ++i) o[q][i] = 0.f;
#pragma unroll
    for (int j0 = 0; j0 < RMAX; j0 += 16) {
      if (j0 >= r) break;
      uint4 b[16];
#pragma unroll
      for (int jj = 0; jj < 16; ++jj)
        b[jj] = j0 + jj < r
                    ? __ldg(reinterpret_cast<const uint4*>(Bs + (size_t)(j0 + jj) * N + e * 8))
                    : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) {
        const float bf[8] = {bf16_lo(b[jj].x), bf16_hi(b[jj].x), bf16_lo(b[jj].y),
                             bf16_hi(b[jj].y), bf16_lo(b[jj].z), bf16_hi(b[jj].z),
                             bf16_lo(b[jj].w), bf16_hi(b[jj].w)};
#pragma unroll
        for (int q = 0; q < NG; ++q) {
          const float vj = v_s[q][j0 + jj];
#pragma unroll
          for (int i = 0; i < 8; ++i) o[q][i] = fmaf(vj, bf[i], o[q][i]);
        }
      }
    }
#pragma unroll
    for (int q = 0; q < NG; ++q) {
      if (!LORA_IN_BOUNDS(rows[q] >= 0 && rows[q] < delta_rows, err)) continue;
      float4* d = reinterpret_cast<float4*>(delta + (size_t)rows[q] * N + e * 8);
      d[0] = make_float4(o[q][0], o[q][1], o[q][2], o[q][3]);
      d[1] = make_float4(o[q][4], o[q][5], o[q][6], o[q][7]);
    }
  }
}

// Work items: (slot, group of kStrGroup of its rows, in row order), so that a slot with many
// rows is spread over several CTAs instead of making one CTA the kernel's tail.  Every CTA
// derives the same item list from the ids (a shared-memory histogram over slots and an
// exclusive scan of the groups per slot) and takes items blockIdx.x, + gridDim.x, ...
static constexpr int kStrGroup = 2;

// At most 120 registers a thread: the register file is split between the SM's four warp
// schedulers, each holding the registers of its own warps (16K), and a GEMM CTA's 6 warps
// put 2 warps of ~136 registers on two of them; 2 warps of this kernel must fit beside
// those for the two kernels to share the SM.
// PERCOL: false when every slot's columns share one scale (plain adapters: the scale of
// column 0 is the slot's), true when a slot holds a composition (one scale per column).
// POOLED: false when slot s starts at pool row s * R, true when a row allocator placed it
// (row_base[s]; the A and B rows of a slot then number its rank rounded up to 8).
template <int RMAX, int ROWS, bool PERCOL, bool POOLED>
__global__ void __maxnreg__(120)
    bgmv_stream_kernel(const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ token_slot,
                       const int32_t* __restrict__ loaded, int T, int K, int N, int R, int S,
                       const __nv_bfloat16* __restrict__ At_pool,
                       const __nv_bfloat16* __restrict__ B_pool,
                       const int32_t* __restrict__ row_base, int pool_rows,
                       const float* __restrict__ scale,
                       const int32_t* __restrict__ rank, float* __restrict__ delta,
                       int delta_rows, int32_t* __restrict__ err, int wait_prev) {
  // launched while the previous kernel (the previous forward's base GEMM) still runs: wait
  // for it before reading x or writing delta, and only then let the base GEMM start (its
  // main loop reads x, which that kernel may have written).  After the e4m3 row quantiser
  // (wait_prev 0) there is nothing to wait for: that kernel waited for the previous GEMM
  // before it let this one launch, and x is read through L2 below.
  if (wait_prev) griddep_wait();
  griddep_launch_dependents();
  extern __shared__ int grp_off[];  // [S + 1]: rows per slot, then first item of each slot
  __shared__ int rows_s[kStrGroup];
  __shared__ int warp_cnt[kStrThreads / 32];
  __shared__ float red[kStrThreads / 32][kStrRedMax];
  __shared__ float v_s[kStrGroup][32];
  __shared__ int rb_s;  // pooled: the item's slot's first pool row
  constexpr int kIds = kSlotMaxT / kStrThreads;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (S + kStrThreads - 1) / kStrThreads;  // consecutive slots per thread
  const int q_begin = min(S, tid * per), q_end = min(S, q_begin + per);
  // With at most one slot per CTA, CTA b requests slot b's A and B rows into L2 right away,
  // before the ids are read: the DRAM traffic of every slot then overlaps the item-list
  // setup below (the items' own prefetches find the lines present or in flight).  Measured:
  // requesting only the slots the batch names, once the ids are counted, costs the decode
  // step more (~1 us later) than the unused slots' reads do.
  if (S <= (int)gridDim.x && (int)blockIdx.x < S && warp == 0) {
    // (pooled: the rows from the slot's first row, as many as the pool still holds; an
    // empty slot has no first row and requests nothing)
    const int rb0 = POOLED ? row_base[blockIdx.x] : (int)blockIdx.x * R;
    const int rs = POOLED ? (rb0 < 0 ? 0 : min(min(R, RMAX), pool_rows - rb0)) : min(R, RMAX);
    const size_t a_bytes = (size_t)rs * K * 2, b_bytes = (size_t)rs * N * 2;
    const char* a0 = reinterpret_cast<const char*>(At_pool + (size_t)max(rb0, 0) * K);
    const char* b0 = reinterpret_cast<const char*>(B_pool + (size_t)max(rb0, 0) * N);
    const size_t off = (size_t)lane << 15;
    if (off < a_bytes) bulk_prefetch_l2(a0 + off, (uint32_t)min(a_bytes - off, (size_t)1 << 15));
    if (off < b_bytes) bulk_prefetch_l2(b0 + off, (uint32_t)min(b_bytes - off, (size_t)1 << 15));
  }
  // the ids and this thread's slots' loaded flags are requested together (one round trip)
  int ids[kIds];
#pragma unroll
  for (int u = 0; u < kIds; ++u) {
    const int i = tid * kIds + u;
    ids[u] = i < T ? token_slot[i] : -1;
  }
  uint32_t loaded_bits = 0;  // bit q - q_begin: slot q holds an adapter (per <= 32)
  for (int q = q_begin; q < q_end; ++q)
    loaded_bits |= (loaded[q] != 0 ? 1u : 0u) << (q - q_begin);
  // ---- the item list: rows per slot, then groups per loaded slot, exclusive scan ----
  for (int q = tid; q <= S; q += kStrThreads) grp_off[q] = 0;
  __syncthreads();
#pragma unroll
  for (int u = 0; u < kIds; ++u)
    if (ids[u] >= 0 && ids[u] < S) atomicAdd(&grp_off[ids[u]], 1);
  __syncthreads();
  int mine = 0;
  for (int q = q_begin; q < q_end; ++q) {
    const int g = (loaded_bits >> (q - q_begin)) & 1u ? (grp_off[q] + kStrGroup - 1) / kStrGroup
                                                      : 0;
    grp_off[q] = g;
    mine += g;
  }
  int inc = mine;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, inc, d);
    if (lane >= d) inc += t;
  }
  if (lane == 31) warp_cnt[warp] = inc;
  __syncthreads();
  int base = inc - mine, n_items = 0;
  for (int w = 0; w < kStrThreads / 32; ++w) {
    if (w < warp) base += warp_cnt[w];
    n_items += warp_cnt[w];
  }
  for (int q = q_begin; q < q_end; ++q) {  // groups -> first item of the slot
    const int g = grp_off[q];
    grp_off[q] = base;
    base += g;
  }
  if (tid == 0) grp_off[S] = n_items;
  __syncthreads();

  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    // the item's slot: the last s with grp_off[s] <= it
    int lo = 0, hi = S - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (grp_off[mid] <= it) lo = mid;
      else hi = mid - 1;
    }
    const int s = lo, g0 = (it - grp_off[s]) * kStrGroup;  // first row (in slot order)
    const int r = rank[s];  // requested now, needed after the row scan
    // the scale of rank column tid % RMAX, the one this thread finishes in the shrink
    // (columns >= r are zeroed there, so a lane past column R - 1 may read any value: the
    // scale table is padded by 32 entries, so the read stays inside it).  The per-column
    // read costs this register-capped kernel a few spilled registers; layers of plain
    // adapters read one scale per slot instead.
    const float sc = scale[(size_t)s * R + (PERCOL ? (lane & (RMAX - 1)) : 0)];
    // the slot's A and B rows (two contiguous ranges) requested into L2 now, in 32 KB bulk
    // prefetches from the lanes of warp 0: the DRAM round trips overlap the row scan
    // below, and the loads after it hit L2
    if (warp == 0) {
      // (pooled: warp 0 reads the slot's first row and leaves it in shared memory)
      const int rbw = POOLED ? row_base[s] : s * R;
      if (POOLED && lane == 0) rb_s = rbw;
      const int rs = min(r, min(R, RMAX));
      const size_t a_bytes = (size_t)rs * K * 2, b_bytes = (size_t)rs * N * 2;
      const char* a0 = reinterpret_cast<const char*>(At_pool + (size_t)rbw * K);
      const char* b0 = reinterpret_cast<const char*>(B_pool + (size_t)rbw * N);
      for (size_t off = (size_t)lane << 15; off < a_bytes; off += (size_t)32 << 15)
        bulk_prefetch_l2(a0 + off, (uint32_t)min(a_bytes - off, (size_t)1 << 15));
      for (size_t off = (size_t)lane << 15; off < b_bytes; off += (size_t)32 << 15)
        bulk_prefetch_l2(b0 + off, (uint32_t)min(b_bytes - off, (size_t)1 << 15));
    }
    // ---- the slot's rows g0 .. g0 + kStrGroup - 1, in row order ----
    int cnt = 0;
#pragma unroll
    for (int u = 0; u < kIds; ++u) cnt += ids[u] == s;
    int inc2 = cnt;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, inc2, d);
      if (lane >= d) inc2 += t;
    }
    if (lane == 31) warp_cnt[warp] = inc2;
    __syncthreads();
    int pos = inc2 - cnt, nrows = 0;
    for (int w = 0; w < kStrThreads / 32; ++w) {
      if (w < warp) pos += warp_cnt[w];
      nrows += warp_cnt[w];
    }
#pragma unroll
    for (int u = 0; u < kIds; ++u)
      if (ids[u] == s) {
        if (pos >= g0 && pos < g0 + kStrGroup) rows_s[pos - g0] = tid * kIds + u;
        ++pos;
      }
    __syncthreads();
    const int ng = min(kStrGroup, nrows - g0);
    const int rbi = POOLED ? rb_s : s * R;  // the slot's first pool row
    // (rbi and r are the same in every thread: the whole CTA skips the item)
    if (!LORA_IN_BOUNDS(rbi >= 0 && rbi + min(r, min(R, RMAX)) <= pool_rows, err)) {
      __syncthreads();  // rows_s and v_s are rewritten by the next item
      continue;
    }
    const __nv_bfloat16* At = At_pool + (size_t)rbi * K;
    const __nv_bfloat16* Bs = B_pool + (size_t)rbi * N;
    // shrink: v_s[0 .. ng), ROWS rows a pass (the last pass may take one)
    for (int q0 = 0; q0 < ng; q0 += ROWS) {
      if (ng - q0 >= ROWS)
        stream_shrink<RMAX, ROWS>(x, rows_s + q0, K, At, r, sc, red, v_s + q0);
      else
        stream_shrink<RMAX, 1>(x, rows_s + q0, K, At, r, sc, red, v_s + q0);
    }
    // expand: the group's delta rows
    if (ng == 1)
      stream_expand<RMAX, 1>(Bs, N, r, v_s, rows_s, delta, delta_rows, err);
    else
      stream_expand<RMAX, kStrGroup>(Bs, N, r, v_s, rows_s, delta, delta_rows, err);
    __syncthreads();  // rows_s and v_s are rewritten by the next item
  }
}

template <int RMAX, int ROWS, bool PERCOL, bool POOLED>
static cudaError_t launch_bgmv_stream_t(const BgmvArgs& a, cudaStream_t stream) {
  // the SMs it runs on must keep the shared-memory split a GEMM CTA needs, or that CTA
  // waits for them to drain
  static bool carveout[kAttrDevices] = {};
  cudaError_t e =
      prefer_max_smem_carveout(bgmv_stream_kernel<RMAX, ROWS, PERCOL, POOLED>, carveout);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  // one CTA per SM: every CTA derives the item list, so idle ones leave right after that
  cfg.gridDim = dim3(std::max(1, a.num_sms));
  cfg.blockDim = dim3(kStrThreads);
  cfg.dynamicSmemBytes = (size_t)(a.S + 1) * sizeof(int);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, bgmv_stream_kernel<RMAX, ROWS, PERCOL, POOLED>,
                            static_cast<const __nv_bfloat16*>(a.x), a.token_slot, a.loaded, a.T,
                            a.K, a.N, a.R, a.S, static_cast<const __nv_bfloat16*>(a.At_pool),
                            static_cast<const __nv_bfloat16*>(a.B_pool), a.row_base,
                            a.pool_rows, a.scale, a.rank, a.delta, a.delta_rows, a.err,
                            a.xq ? 0 : 1);
}

template <int RMAX, int ROWS>
static cudaError_t launch_bgmv_stream_r(const BgmvArgs& a, cudaStream_t stream) {
  if (a.pooled)
    return a.per_column ? launch_bgmv_stream_t<RMAX, ROWS, true, true>(a, stream)
                        : launch_bgmv_stream_t<RMAX, ROWS, false, true>(a, stream);
  return a.per_column ? launch_bgmv_stream_t<RMAX, ROWS, true, false>(a, stream)
                      : launch_bgmv_stream_t<RMAX, ROWS, false, false>(a, stream);
}

static cudaError_t launch_bgmv_stream(const BgmvArgs& a, cudaStream_t stream) {
  return a.R <= 16 ? launch_bgmv_stream_r<16, 2>(a, stream)
                   : launch_bgmv_stream_r<32, 1>(a, stream);
}

cudaError_t launch_bgmv_delta(const BgmvArgs& a, cudaStream_t stream, int* launches) {
  if (a.xq) {  // e4m3 base: the row quantiser first (it lets this kernel launch at once)
    const cudaError_t e =
        launch_quant_rows_e4m3(a.x, a.T, a.K, a.xq, a.sx, a.q_ready, a.num_sms, true, stream);
    if (e != cudaSuccess) return e;
    if (launches && a.T > 0) ++*launches;
  }
  if (launches) ++*launches;  // (counted before the launch: an error fails the forward)
  if (a.R <= 32 && a.T <= kSlotMaxT && a.K % 8 == 0 && a.N % 8 == 0)
    return launch_bgmv_stream(a, stream);  // slot-major, registers only
  // row-major: cluster of cs CTAs per row: 4 normally, fewer when K or N is small
  int cs = 4;
  while (cs > 1 && (a.K < cs * 256 || a.N < cs * 64)) cs >>= 1;
  const int kchunk = ((a.K + cs - 1) / cs + 255) / 256 * 256;
  const int nchunk = ((a.N + cs - 1) / cs + 7) / 8 * 8;
  int clusters = a.T;
  // at most 4 of these CTAs per SM, so that the base GEMM launched after this kernel still
  // finds room for its CTA on every SM and runs concurrently
  const int cap = a.num_sms * 4 / cs;
  if (clusters > cap) clusters = cap;
  if (clusters < 1) clusters = 1;
  static bool carveout[kAttrDevices] = {};
  cudaError_t e = prefer_max_smem_carveout(bgmv_delta_kernel, carveout);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cs;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.gridDim = dim3(clusters * cs);
  cfg.blockDim = dim3(kBgmvThreads);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, bgmv_delta_kernel, static_cast<const __nv_bfloat16*>(a.x),
                            a.token_slot, a.loaded, a.T, a.K, a.N, a.R, a.S,
                            static_cast<const __nv_bfloat16*>(a.At_pool),
                            static_cast<const __nv_bfloat16*>(a.B_pool), a.row_base, a.scale,
                            a.rank, a.delta, a.delta_rows, a.pool_rows, a.err, kchunk, nchunk);
}

cudaError_t launch_lora_tile(const TileArgs& a, bool bf16, bool delta, cudaStream_t stream) {
  int grid = a.max_tiles;
  if (grid > a.num_sms * 4) grid = a.num_sms * 4;
  if (grid < 1) grid = 1;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kTileThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  static bool carveout[3][kAttrDevices] = {};
  cudaError_t e = bf16 ? prefer_max_smem_carveout(lora_tile_kernel<__nv_bfloat16, Vec16<__nv_bfloat16>>, carveout[0])
                       : cudaSuccess;
  if (e == cudaSuccess && !bf16)
    e = prefer_max_smem_carveout(lora_tile_kernel<float, Vec16<float>>, carveout[1]);
  if (e == cudaSuccess && !bf16)
    e = prefer_max_smem_carveout(lora_tile_kernel<float, Scalar32>, carveout[2]);
  if (e != cudaSuccess) return e;
  if (bf16) {
    using T = __nv_bfloat16;
    using V = Vec16<T>;
    const T* x = static_cast<const T*>(a.x);
    const T* At = static_cast<const T*>(a.At_pool);
    const T* B = static_cast<const T*>(a.B_pool);
    if (delta) return cudaErrorInvalidValue;  // delta mode runs bgmv_delta_kernel
    return cudaLaunchKernelEx(&cfg, lora_tile_kernel<T, V>, x, a.K, a.N, a.R, At, B,
                              a.row_base, a.scale, a.rank, a.perm, a.seg_offsets, a.seg_slot, a.tile_seg,
                              a.tile_row0, a.meta, a.out, a.out_rows, a.pool_rows, a.err);
  }
  if (delta) return cudaErrorInvalidValue;  // delta mode is a bf16 path
  using T = float;
  const T* x = static_cast<const T*>(a.x);
  const T* At = static_cast<const T*>(a.At_pool);
  const T* B = static_cast<const T*>(a.B_pool);
  const bool vec4 = a.K % 4 == 0 && reinterpret_cast<uintptr_t>(x) % 16 == 0;
  if (vec4)
    return cudaLaunchKernelEx(&cfg, lora_tile_kernel<T, Vec16<T>>, x, a.K, a.N, a.R, At, B,
                              a.row_base, a.scale, a.rank, a.perm, a.seg_offsets, a.seg_slot, a.tile_seg,
                              a.tile_row0, a.meta, a.out, a.out_rows, a.pool_rows, a.err);
  return cudaLaunchKernelEx(&cfg, lora_tile_kernel<T, Scalar32>, x, a.K, a.N, a.R, At, B,
                            a.row_base, a.scale, a.rank, a.perm, a.seg_offsets, a.seg_slot, a.tile_seg,
                            a.tile_row0, a.meta, a.out, a.out_rows, a.pool_rows, a.err);
}

}  // namespace lora
