// gemm_tc.cu -- base GEMM y = x W on the fifth-generation tensor cores, with the layer's
// low-rank term added in the epilogue so that y is written once.
//
// "LoRAX, in depth", section "Computing a batch that mixes adapters": the base term is the
// same for every request, so it runs as one large GEMM over all tokens; only the low-rank
// term differs by adapter.  "Serving LoRA adapters ..." (vLLM) Step 4: the expand multiplies
// the fp32 rank buffer by B and adds it to the base output.
//
// A CTA computes 128 x BN blocks of y (6 warps):
//   warp 0      TMA producer: 64-wide K blocks of x [M,K] and of the packed weight W^T [N,K]
//               (both K-major, 128-byte swizzle) into a ring of shared-memory stages.
//   warp 1      allocates 2 x BN TMEM columns (two accumulators); one lane issues
//               tcgen05.mma (M=128, N=BN, K=16, bf16 x bf16 -> fp32 in TMEM) and frees each
//               stage with tcgen05.commit.
//   warps 2..5  epilogue: each thread owns one output row (one TMEM lane); it reads the
//               accumulator 32 columns at a time (tcgen05.ld) and rounds to bf16 once.
//               In delta mode it first adds the fp32 delta[row, n] the BGMV kernel
//               expanded (rows with slot -1 store the base product only).
// Large batches (v mode) run a persistent grid of at most the resident CTAs (pairs): each
// walks its tiles round-robin in bands of row tiles (a wave then shares one band of x in
// L2), the MMAs filling one accumulator while the epilogue drains the other.  When the
// last round would keep at most half of them busy, its tiles are cut in two (stream-K):
// one CTA takes the head K blocks and the tile's expand blocks and finishes the tile, the
// next the tail, handed over as an fp32 partial through L2 with a flag tagged by a
// per-launch epoch.  Small batches (delta mode) run one tile per CTA.  The mode is a
// template parameter, so the delta-mode variants carry none of the v-mode code.
// v mode (the expand on the tensor cores): while the main loop runs, the epilogue warps list
// the tile's distinct slots u (ascending) and then write extra K blocks into the same ring,
// after the base blocks: y_tile += sum_u [V_u^hi | V_u^lo] [B_u^T ; B_u^T], where V_u is v
// (fp32, already scaled by alpha / r, summed over its K-split planes) on the rows of slot u
// and zero elsewhere, V^hi = bf16(V) and V^lo = bf16(V - V^hi), and B_u^T comes from the
// transposed slot pool.  Each 64-wide block holds 8 chunks of 8 rank columns: the hi then lo
// halves of consecutive slots' R columns.  The MMA lane runs those blocks after the base
// ones, so base and low-rank products meet in the one fp32 accumulator.  Rows with slot -1
// match no slot and keep the base product only.
// Split K (small batches): the grid's z dimension cuts K into `cs` <= 4 ranges and the cs
// CTAs of one output block form a thread-block cluster (with CTA pairs, the 2 cs CTAs of a
// 256-row block).  After its main loop each CTA writes, for every other CTA d of its block,
// its fp32 partial of the columns d finishes into an L2-resident scratch block; after a
// cluster barrier (release / acquire) each CTA adds the cs - 1 blocks addressed to it and
// runs the epilogue on its BN / cs columns.  L2 carries these blocks several times faster
// than distributed shared memory.  A small batch thereby keeps W (not the re-read x)
// dominant in every stage and needs 1/cs of the K range per SM.
// CTA pairs (cta_group::2): two CTAs of a cluster share a 256 x BN tile; each loads its 128
// rows of x and half of the W tile, the even CTA issues M = 256 MMAs that read both CTAs'
// shared memory and write both CTAs' TMEM, and its commits arrive on both CTAs' barriers.
// A pair thereby moves the same operand bytes per SM as a 128 x BN/2 tile while every MMA
// instruction does the work of a 128 x BN one (the issue rate, ~124 cycles per instruction
// however narrow, bounds tiles below 256 columns).
// A whole tile starts its K range at a rotated K block (and wraps around), so the CTAs that
// share an x tile or a W tile do not all request the same lines from L2 at the same moment.
// Launch: programmatic dependent launch after the low-rank kernel: the main loop and the
// split-K exchange read only x, W and the accumulators, so they run while the low-rank
// kernel is still working; the epilogue waits (griddepcontrol.wait) only before it reads
// the low-rank results.  It lets no dependent launch early (measured: the next forward's
// low-rank kernel, resident early, slowed the step), so the next kernel on the stream sees
// y complete.  Every mbarrier wait is bounded (lora_common.cuh).
#include <cudaTypedefs.h>

#include <algorithm>

#include "lora_common.cuh"
#include "lora_kernels.h"

namespace lora {

static constexpr int kTcThreads = 192;
static constexpr int kBM = 128, kBK = 64;
static constexpr int kABytes = kBM * kBK * 2;

// Add the row's delta (delta mode, adapted rows) to 32 accumulator columns starting at
// global column n and store them as bf16.
// The 32 accumulator columns at TMEM address taddr (this thread's lane) as floats.
__device__ __forceinline__ void tmem_acc32(uint32_t taddr, float (&acc)[32]) {
  uint32_t raw[32];
  tmem_ld_32x32b_x32(taddr, raw);
  tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 32; ++i) acc[i] = __uint_as_float(raw[i]);
}

// acc += columns c .. c + 31 of a partial block ([bnc / 4][128 rows] float4; blk points at
// this thread's row of chunk 0).
__device__ __forceinline__ void add_block32(float (&acc)[32], const float4* blk, int c) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 v = blk[(size_t)((c >> 2) + i) * 128];
    acc[i * 4 + 0] += v.x;
    acc[i * 4 + 1] += v.y;
    acc[i * 4 + 2] += v.z;
    acc[i * 4 + 3] += v.w;
  }
}

// The e4m3 product back to the x and W scales: acc[i] *= sx * sw[i] (sw: 32 column scales).
__device__ __forceinline__ void scale32(float (&acc)[32], float sxr, const float* sw) {
  const float4* swp = reinterpret_cast<const float4*>(sw);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 w = swp[i];
    acc[i * 4 + 0] *= sxr * w.x;
    acc[i * 4 + 1] *= sxr * w.y;
    acc[i * 4 + 2] *= sxr * w.z;
    acc[i * 4 + 3] *= sxr * w.w;
  }
}

// Columns n .. n + 31 of row `row` of y (bf16, 16-byte stores; rows >= M and columns >= N
// are not written).
__device__ __forceinline__ void store_y32(const float (&acc)[32], const GemmArgs& a, int row,
                                          int n, __nv_bfloat16* yrow) {
  if (row < a.M) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (n + q * 8 < a.N) {
        uint4 o;
        o.x = pack_bf16x2(acc[q * 8 + 0], acc[q * 8 + 1]);
        o.y = pack_bf16x2(acc[q * 8 + 2], acc[q * 8 + 3]);
        o.z = pack_bf16x2(acc[q * 8 + 4], acc[q * 8 + 5]);
        o.w = pack_bf16x2(acc[q * 8 + 6], acc[q * 8 + 7]);
        *reinterpret_cast<uint4*>(yrow + n + q * 8) = o;
      }
    }
  }
}

// The row's v (the sum of its K-split planes) at rank columns j0 .. j0 + 7, split into bf16
// high parts (bf16 of v) and low parts (bf16 of v - high): hi + lo carries v to about 16
// significant bits through a bf16 x bf16 product.
__device__ __forceinline__ void v_hi_lo8(const ExpandArgs& ex, int row, int j0, uint4& hi,
                                         uint4& lo) {
  const float* vr = ex.v + (size_t)row * ex.R + j0;
  float4 v0 = __ldg(reinterpret_cast<const float4*>(vr));
  float4 v1 = __ldg(reinterpret_cast<const float4*>(vr + 4));
  for (int p = 1; p < ex.v_planes; ++p) {
    const float* vp = vr + (size_t)p * ex.v_plane_stride;
    const float4 a0 = __ldg(reinterpret_cast<const float4*>(vp));
    const float4 a1 = __ldg(reinterpret_cast<const float4*>(vp + 4));
    v0.x += a0.x; v0.y += a0.y; v0.z += a0.z; v0.w += a0.w;
    v1.x += a1.x; v1.y += a1.y; v1.z += a1.z; v1.w += a1.w;
  }
  const float f[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
  uint32_t h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float e0 = f[2 * i], e1 = f[2 * i + 1];
    h[i] = pack_bf16x2(e0, e1);
    l[i] = pack_bf16x2(e0 - bf16_lo(h[i]), e1 - bf16_hi(h[i]));
  }
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// Output tile (pm, nt) of work unit u: bands of group_m row tiles (pairs of them with CTA
// pairs), column tiles in turn within a band, row tiles fastest.  Consecutive units (those
// the resident CTAs run at the same time) then share one band of x, which stays in L2,
// instead of streaming all of x from DRAM again for every few column tiles.
__device__ __forceinline__ void unit_tile(int u, int mtp, int nt, int group_m, int& pm,
                                          int& ntile) {
  const int band = u / (group_m * nt);
  const int gm = min(group_m, mtp - band * group_m);  // rows of the last band may be fewer
  const int w = u - band * group_m * nt;
  pm = band * group_m + w % gm;
  ntile = w / gm;
}

// The work of CTA (pair) slot g of G: `full_rounds` whole tiles (units g, g + G, ...; fewer
// where they run past U), then -- stream-K, when the units leave a last round of at most
// half the slots busy -- those remaining tiles cut in two: slot g < sk_slots takes half
// g & 1 of tile full_rounds G + g / 2, the head (K blocks from 0, and the tile's expand
// blocks) on the even slot, which finishes the tile, the tail on the odd one, written as
// an fp32 partial.  Both are their slot's last segment.  Segment k of slot g: unit u, K
// blocks [k0, k1); false past the last one.
__device__ __forceinline__ bool seg_at(int k, int g, int G, int U, int nkb, int full_rounds,
                                       int sk_slots, int& u, int& k0, int& k1) {
  const int nfull = min(full_rounds, (U - g + G - 1) / G);  // whole units g + j G < U
  if (k < nfull) {
    u = g + k * G;
    k0 = 0;
    k1 = nkb;
    return true;
  }
  if (k > nfull || g >= sk_slots) return false;
  u = full_rounds * G + (g >> 1);
  const int half = nkb >> 1;  // the host splits only K ranges of >= 2 blocks
  k0 = (g & 1) ? half : 0;
  k1 = (g & 1) ? nkb : half;
  return true;
}

// Delta mode (decode) caps registers at 136: two warps of this kernel and two of the
// decode BGMV kernel (120 registers) share each of an SM's four 16K-register files, so the
// two kernels run side by side.  The e4m3 variants take 80, so that one warp of the row
// quantiser (112) fits beside the two as well and this kernel's CTAs start while it runs.  VMODE is a template parameter so that the delta-mode
// variants carry none of the expand-block and stream-K code; the v-mode variants share
// their SMs with no other kernel and get more registers.
// FP8: the base operands are e4m3 (x quantised per row, W per column): a 128-byte K block
// then holds 128 elements instead of 64, the MMAs are kind::f8f6f4, and the accumulator is
// scaled by sx[row] sw[col] before the low-rank term is added (delta mode: in the
// epilogue; v mode: in TMEM, between the base and the expand blocks).
template <int BN, bool PAIR, bool VMODE, bool FP8 = false>
__global__ void __maxnreg__(VMODE ? 168 : (FP8 ? 80 : 136))
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmap_x,
                   const __grid_constant__ CUtensorMap tmap_w,
                   const __grid_constant__ CUtensorMap tmap_bx,
                   const __grid_constant__ CUtensorMap tmap_delta, GemmArgs a, int stages,
                   int xscr_bytes, int group_m, int mtp, int nt, int full_rounds,
                   int sk_slots) {
  constexpr int kBRows = PAIR ? BN / 2 : BN;  // rows of the W (or B expand) tile this CTA loads
  constexpr int kBBytes = kBRows * kBK * 2;
  constexpr int kStageBytes = kABytes + kBBytes;
  constexpr int kKE = FP8 ? 2 * kBK : kBK;  // K elements per block (128 bytes of a row)

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* stage_base = smem;
  // v mode: each tile row's hi / lo v halves in the expand block layout (128 B per block)
  uint8_t* xscr = smem + (size_t)stages * kStageBytes;
  // v mode: the tile's distinct slots (a bitmap over slots, then the ascending list)
  uint32_t* slot_bits = reinterpret_cast<uint32_t*>(xscr + xscr_bytes);
  int* uslot = reinterpret_cast<int*>(slot_bits + kBM);  // [128]
  int* wsum = uslot + kBM;                               // [4] per epilogue warp
  int* x_blocks = wsum + 4;                              // expand blocks of this tile
  // e4m3: [BN] column scales, read as float4 (16-byte aligned: slot_bits is, and the four
  // words from x_blocks on round the tables to a multiple of 16 bytes)
  float* sw_tile = reinterpret_cast<float*>(x_blocks + 4);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sw_tile + (FP8 ? BN : 0));
  uint64_t* full = bars;
  uint64_t* empty = bars + stages;
  uint64_t* tmem_full = bars + 2 * stages;       // [2] accumulator buffer complete
  uint64_t* tmem_empty = bars + 2 * stages + 2;  // [2] accumulator buffer drained
  uint64_t* xinfo_bar = bars + 2 * stages + 4;   // v mode: the tile's x_blocks written
  uint64_t* xgrant = bars + 2 * stages + 5;      // [stages] v mode: stage handed to the epilogue
  uint64_t* xa_full = bars + 3 * stages + 5;     // [stages] v mode: its A half written
  uint64_t* base_full = bars + 4 * stages + 5;   // [2] e4m3 v mode: the base blocks complete
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 4 * stages + 7);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the first launch of a split batch lets the second one start while it runs (it waits for
  // this one before its epilogue reads anything this one's predecessor wrote); e4m3 base:
  // only once this CTA has seen every row of xq (below), so that the second launch, which
  // resets the row count, starts after every CTA of this one has read it
  if (a.trigger_next && !FP8) griddep_launch_dependents();
  // Work units: output tiles, one per CTA (pair) slot and round: slot g runs units
  // g, g + G, g + 2 G, ... (delta mode: G is the number of units, one each).  CTA pairs:
  // the two CTAs of a pair are neighbours in x and cover 256 consecutive rows, CTA pr of
  // the pair rows [128 pr, 128 pr + 128).
  const int pr = PAIR ? (int)(blockIdx.x & 1u) : 0;
  const int g0 = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int G = PAIR ? (int)gridDim.x / 2 : (int)gridDim.x;
  const int U = mtp * nt;
  // cluster ranks (x fastest): CTA (pr, z) is rank pr + 2 z with pairs, z without; the even
  // CTA of a pair issues its MMAs, and its barriers count both CTAs' loads
  const uint32_t lead_rank = PAIR ? 2u * blockIdx.z : 0u;
  const uint16_t pair_mask = (uint16_t)(3u << lead_rank);
  // split K: this CTA's range of K blocks (the host keeps every range non-empty)
  const int cs = gridDim.z, z = blockIdx.z;
  const int nkb_all = (a.K + kKE - 1) / kKE;
  const int per = (nkb_all + cs - 1) / cs;
  const int kb_begin = z * per;
  const int nkb = min(nkb_all, kb_begin + per) - kb_begin;
  const int bnc = BN / cs;  // columns this CTA finishes
  constexpr bool vmode = VMODE;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tmem_full[b], 1);
      mbar_init(&tmem_empty[b], PAIR ? 2 : 1);  // pairs: one arrival from each CTA's epilogue
      mbar_init(&base_full[b], 1);
    }
    mbar_init(xinfo_bar, 1);
    for (int s = 0; s < stages; ++s) {
      mbar_init(&xgrant[s], 1);
      // v-mode pairs: one arrival from each CTA's epilogue; delta mode counts one arrival
      // (the epilogue's delta-tile loads may use it)
      mbar_init(&xa_full[s], PAIR && vmode ? 2 : 1);
    }
    fence_mbar_init();
    if (FP8 && a.q_ready) {
      // the rows of xq come from the low-rank kernel running beside this one: wait until
      // all M are counted (bounded: on a timeout the error flag is set and the loads go
      // ahead), then order this thread's TMA loads after the writes seen
      wait_flag_gpu(a.q_ready, a.M, a.err);
      fence_proxy_async_global();
      if (a.q_reset &&
          atomicAdd(a.q_ready + 1, 1) == (int)(gridDim.x * gridDim.y * gridDim.z) - 1) {
        atomicExch(a.q_ready, 0);  // every CTA of the batch's launches has seen the count
        atomicExch(a.q_ready + 1, 0);
      }
    }
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmap_x);
    tma_prefetch_desc(&tmap_w);
    if (vmode) tma_prefetch_desc(&tmap_bx);
  }
  // two accumulator buffers of BN columns: the epilogue drains one while the MMAs fill the
  // other with the next tile
  if (warp == 1) {
    if (PAIR)
      tmem_alloc_pair(tmem_holder, 2 * BN);
    else
      tmem_alloc(tmem_holder, 2 * BN);
  }
  tc_fence_before();
  __syncthreads();
  if (a.trigger_next && FP8) griddep_launch_dependents();
  // pairs: the peer's barriers are initialised before this CTA's loads and MMAs signal them
  if (PAIR) cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      int hk = 0;  // head segments so far (v mode: one xinfo phase each)
      for (int k = 0; ok; ++k) {
        int u, k0, k1;
        if (!seg_at(k, g0, G, U, nkb, full_rounds, sk_slots, u, k0, k1)) break;
        int pm_i, nt_i;
        unit_tile(u, mtp, nt, group_m, pm_i, nt_i);
        const int m0 = (PAIR ? 2 * pm_i + pr : pm_i) * kBM, n0 = a.n_begin + nt_i * BN;
        // a whole tile starts its K range at a rotated block (the same for both CTAs of a
        // pair), so tiles sharing an x or W tile do not request the same lines at once;
        // stream-K pieces run in order
        const int nk = k1 - k0;
        const int rot = nk == nkb ? (int)((pm_i + nt_i) % (unsigned)nkb) : 0;
        for (int it = 0; it < nk; ++it) {
          const int kb = kb_begin + k0 + (rot + it) % nk;
          if (!mbar_wait(&empty[s], ph ^ 1u, a.err)) {
            ok = false;
            break;
          }
          uint8_t* sa = stage_base + (size_t)s * kStageBytes;
          if (PAIR) {
            // this CTA's 128 rows of x and its half of the W tile; the bytes of both CTAs
            // are counted on the even CTA's barrier, which its MMA lane waits on
            if (pr == 0) mbar_arrive_expect_tx(&full[s], 2 * kStageBytes);
            const uint32_t fb = dsmem_map(smem_u32(&full[s]), lead_rank);
            tma_load_2d_pair(sa, &tmap_x, fb, kb * kKE, m0);
            tma_load_2d_pair(sa + kABytes, &tmap_w, fb, kb * kKE, n0 + pr * kBRows);
          } else {
            mbar_arrive_expect_tx(&full[s], kStageBytes);
            tma_load_2d(sa, &tmap_x, &full[s], kb * kKE, m0);
            tma_load_2d(sa + kABytes, &tmap_w, &full[s], kb * kKE, n0);
          }
          if (++s == stages) {
            s = 0;
            ph ^= 1u;
          }
        }
        // v mode: the tile's expand blocks follow in the same ring.  The producer claims
        // each stage in order (a wait on the adjacent phase of empty, as for the base
        // blocks), loads its B half (the slot's rows of the B expand pool) with TMA and
        // hands the stage to the epilogue warps for the A half.  Their waits are on xgrant:
        // two grants of one stage are separated by their own fill, so those waits are on
        // adjacent phases too.
        if (!ok || !vmode || k0 != 0) continue;  // expand blocks go with a tile's head
        if (!mbar_wait(xinfo_bar, (uint32_t)hk & 1u, a.err)) break;
        ++hk;
        const int nx = *x_blocks;
        const ExpandLayout xl = expand_layout(a.ex.R);
        for (int e = 0; e < nx; ++e) {
          if (!mbar_wait(&empty[s], ph ^ 1u, a.err)) {
            ok = false;
            break;
          }
          const int uu = e / xl.nbs, b = e - uu * xl.nbs;
          const int col = xl.nbs == 1 ? 0 : (b % (xl.rx / 64)) * 64;
          uint8_t* sa = stage_base + (size_t)s * kStageBytes;
          // (a slot outside the table: the rows of slot 0 are loaded instead, and flagged)
          const int us = LORA_IN_BOUNDS(uslot[uu] >= 0 && uslot[uu] < a.ex.S, a.err) ? uslot[uu] : 0;
          const int brow = us * a.N + n0 + pr * kBRows;
          if (PAIR) {
            if (pr == 0) mbar_arrive_expect_tx(&full[s], 2 * kBBytes);
            tma_load_2d_pair(sa + kABytes, &tmap_bx, dsmem_map(smem_u32(&full[s]), lead_rank),
                             col, brow);
          } else {
            mbar_arrive_expect_tx(&full[s], kBBytes);
            tma_load_2d(sa + kABytes, &tmap_bx, &full[s], col, brow);
          }
          mbar_arrive(&xgrant[s]);
          if (++s == stages) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer (pairs: the even CTA's lane, for both CTAs) ----------------
    if (lane == 0 && pr == 0) {
      constexpr uint32_t idesc = FP8 ? idesc_e4m3_f32(PAIR ? 2 * kBM : kBM, BN)
                                     : idesc_bf16_f32(PAIR ? 2 * kBM : kBM, BN);
      constexpr uint32_t idesc_x = idesc_bf16_f32(PAIR ? 2 * kBM : kBM, BN);  // expand blocks
      // descriptors built once: the start-address field counts 16-byte units, so a stage
      // is + s * kStageBytes / 16 and a 16-wide K step inside the 128-byte row is + 2
      const uint64_t a_desc0 = smem_desc_sw128(smem_u32(stage_base));
      const uint64_t b_desc0 = smem_desc_sw128(smem_u32(stage_base + kABytes));
      int s = 0;
      uint32_t ph = 0, xa_par = 0;  // xa_par: bit s = parity of stage s's next xa_full phase
      bool ok = true;
      // the 16-wide K chunks of `chunks` (bit kk) of a stage; `first` starts the accumulator;
      // `expand`: a low-rank expand block (bf16 operands whatever the base's)
      auto mma4 = [&](uint32_t d_tmem, int stage, bool first, unsigned chunks, bool expand) {
        const uint64_t stage_off = (uint64_t)(stage * (kStageBytes >> 4));
        const uint64_t a_desc = a_desc0 + stage_off, b_desc = b_desc0 + stage_off;
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          if (!((chunks >> kk) & 1u)) continue;
          const uint32_t acc = (first && kk == 0) ? 0u : 1u;
          // (a 32-byte step of the row either way: 16 bf16 or 32 e4m3 elements of K)
          if (FP8 && !expand && PAIR)
            tc_mma_f8_pair(d_tmem, a_desc + (uint64_t)(kk * 2), b_desc + (uint64_t)(kk * 2),
                           idesc, acc);
          else if (FP8 && !expand)
            tc_mma_f8(d_tmem, a_desc + (uint64_t)(kk * 2), b_desc + (uint64_t)(kk * 2), idesc,
                      acc);
          else if (PAIR)
            tc_mma_bf16_pair(d_tmem, a_desc + (uint64_t)(kk * 2), b_desc + (uint64_t)(kk * 2),
                             FP8 ? idesc_x : idesc, acc);
          else
            tc_mma_bf16(d_tmem, a_desc + (uint64_t)(kk * 2), b_desc + (uint64_t)(kk * 2),
                        FP8 ? idesc_x : idesc, acc);
        }
        if (PAIR)
          tc_commit_pair_mc(&empty[stage], pair_mask);  // frees the stage in both CTAs
        else
          tc_commit(&empty[stage]);
      };
      int hk = 0;  // head segments so far (v mode: one xinfo phase each)
      for (int k = 0; ok; ++k) {
        int u, k0, k1;
        if (!seg_at(k, g0, G, U, nkb, full_rounds, sk_slots, u, k0, k1)) break;
        // buffer b of the tile; kph: the tile's use of that buffer (its barriers' phase)
        const int b = k & 1, kph = k >> 1;
        const uint32_t d_tmem = tmem_base + (uint32_t)(b * BN);
        // the epilogue has drained this buffer's previous tile (tile k - 2); pairs: both
        // CTAs' epilogues, the peer's across the cluster
        if (!(PAIR ? mbar_wait_cluster(&tmem_empty[b], ((uint32_t)kph & 1u) ^ 1u, a.err)
                   : mbar_wait(&tmem_empty[b], ((uint32_t)kph & 1u) ^ 1u, a.err)))
          break;
        tc_fence_after();
        for (int it = 0; it < k1 - k0; ++it) {
          if (!mbar_wait(&full[s], ph, a.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          mma4(d_tmem, s, it == 0, 0xFu, false);
          if (++s == stages) {
            s = 0;
            ph ^= 1u;
          }
        }
        // e4m3 base, v mode: the epilogue scales the base product in TMEM once it is
        // complete, before it releases the first expand block
        if (FP8 && VMODE && ok) {
          if (PAIR)
            tc_commit_pair_mc(&base_full[b], pair_mask);
          else
            tc_commit(&base_full[b]);
        }
        const bool head = k0 == 0;
        if (ok && vmode && head && !mbar_wait(xinfo_bar, (uint32_t)hk & 1u, a.err)) ok = false;
        if (ok && vmode && head) {
          // the low-rank expand: blocks the epilogue warps write into the same ring; only
          // the K chunks that hold rank columns are multiplied
          const int nx = *x_blocks;
          const ExpandLayout xl = expand_layout(a.ex.R);
          for (int e = 0; e < nx; ++e) {
            // B half (TMA) and A half (written by the epilogue warps; pairs: by both CTAs')
            if (!mbar_wait(&full[s], ph, a.err)) {
              ok = false;
              break;
            }
            const uint32_t xp = (xa_par >> s) & 1u;
            xa_par ^= 1u << s;
            if (!(PAIR ? mbar_wait_cluster(&xa_full[s], xp, a.err)
                       : mbar_wait(&xa_full[s], xp, a.err))) {
              ok = false;
              break;
            }
            tc_fence_after();
            mma4(d_tmem, s, false, expand_chunks(xl, a.ex.R, e % xl.nbs), true);
            if (++s == stages) {
              s = 0;
              ph ^= 1u;
            }
          }
        }
        if (vmode && head) ++hk;
        if (PAIR)
          tc_commit_pair_mc(&tmem_full[b], pair_mask);  // both CTAs' accumulators complete
        else
          tc_commit(&tmem_full[b]);
      }
    }
    __syncwarp();
  } else {
    // ---------------- epilogue warps ----------------
    const int quad = warp & 3;  // TMEM lanes [32*quad, 32*quad + 32) belong to this warp
    const int rt = quad * 32 + lane;
    const int et = threadIdx.x - 64;  // 0..127
    const ExpandLayout xl = expand_layout(a.ex.R);
    uint32_t gpar = 0;  // bit s = parity of stage s's next xgrant phase
    int ring = 0;       // ring blocks (base and expand) of this CTA's earlier tiles
    if (vmode) griddep_wait();  // v and the checked slots come from earlier kernels
    // stream-K: flags carry the launch's epoch + 1 (the epoch advances when the last CTA of a
    // launch exits, so no flag of an earlier launch matches)
    const int32_t epoch =
        VMODE && sk_slots > 0 ? *reinterpret_cast<volatile int32_t*>(a.sk_sync) : 0;
    for (int k = 0;; ++k) {
      int u, k0, k1;
      if (!seg_at(k, g0, G, U, nkb, full_rounds, sk_slots, u, k0, k1)) break;
      const bool head = k0 == 0;
      const int nk = k1 - k0;
      int pm_i, nt_i;
      unit_tile(u, mtp, nt, group_m, pm_i, nt_i);
      const int mt_i = PAIR ? 2 * pm_i + pr : pm_i;
      const int m0 = mt_i * kBM, n0 = a.n_begin + nt_i * BN;
      const int row = m0 + rt;
      const int b = k & 1, kph = k >> 1;
      const uint32_t tmem_row =
          tmem_base + (uint32_t)(b * BN) + (static_cast<uint32_t>(quad * 32) << 16);
      bool ok = true;
      int tile_nx = 0;  // v mode: the tile's expand blocks (e4m3: the accumulator is scaled
                        // in TMEM only when there are some)
      // e4m3 base, v mode: the row's scale and the tile's column scales, requested while the
      // tile's main loop runs (the previous tile's epilogue is past its last barrier)
      float sxr_v = 0.f;
      if (FP8 && VMODE) {
        sxr_v = row < a.M ? __ldcg(a.sx + row) : 0.f;
        for (int i = et; i < BN; i += 128) sw_tile[i] = __ldg(a.sw + n0 + i);
        named_barrier(1, 128);
      }
      if (vmode && head) {
        // ---- v mode: write the low-rank expand as extra K blocks of the ring ----
        // y_tile += sum over the tile's distinct slots u of [v_u^hi | v_u^lo] [B_u^T ; B_u^T],
        // where v_u holds the v rows of slot u's rows and zeros elsewhere.  A block's 8
        // chunks of 8 K-columns hold, in order, the hi then lo halves of each slot's R rank
        // columns.  The previous tile's expand blocks are all consumed (its accumulator was
        // drained), so uslot, x_blocks and the scratch are free.
        const int srow = m0 + et < a.M ? a.ex.row_slot[m0 + et] : -1;
        // pairs: both CTAs list the slots of all 256 rows, so they agree on the expand blocks
        const int pm0 = m0 + (pr == 0 ? kBM : -kBM);  // the peer's first row
        const int orow = PAIR && pm0 + et < a.M ? a.ex.row_slot[pm0 + et] : -1;
        slot_bits[et] = 0u;
        named_barrier(1, 128);
        if (srow >= 0) atomicOr(&slot_bits[srow >> 5], 1u << (srow & 31));
        if (orow >= 0) atomicOr(&slot_bits[orow >> 5], 1u << (orow & 31));
        named_barrier(1, 128);
        uint32_t word = et < (a.ex.S + 31) / 32 ? slot_bits[et] : 0u;
        const int cnt = __popc(word);
        int incl = cnt;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const int t = __shfl_up_sync(0xffffffffu, incl, d);
          if (lane >= d) incl += t;
        }
        if (lane == 31) wsum[et >> 5] = incl;
        named_barrier(1, 128);
        int pos = incl - cnt, m = 0;
        for (int i = 0; i < 4; ++i) {
          if (i < (et >> 5)) pos += wsum[i];
          m += wsum[i];
        }
        while (word) {
          const int bit = __ffs(word) - 1;
          uslot[pos++] = et * 32 + bit;
          word &= word - 1;
        }
        named_barrier(1, 128);
        const int nx = m * xl.nbs;
        tile_nx = nx;
        if (et == 0) {
          *x_blocks = nx;
          mbar_arrive(xinfo_bar);
        }
        // this row's hi and lo halves in the block layout (while the main loop runs), their
        // 16-byte chunks already XOR-swizzled by row & 7 as in the ring, so the copy below
        // moves chunk p to chunk p and neither side has bank conflicts
        uint8_t* mine = xscr + (size_t)et * xl.nbs * 128;
        const int sw = et & 7;
        if (srow >= 0 && LORA_IN_BOUNDS(m0 + et < a.ex.v_rows, a.err)) {
          for (int j0 = 0; j0 < xl.rx; j0 += 8) {
            uint4 hi = make_uint4(0u, 0u, 0u, 0u), lo = hi;
            if (j0 < a.ex.R) v_hi_lo8(a.ex, m0 + et, j0, hi, lo);
            const int hb = xl.nbs == 1 ? 0 : j0 / 64;                // block of the hi part
            const int lb = xl.nbs == 1 ? 0 : xl.rx / 64 + j0 / 64;   // block of the lo part
            const int hc = xl.nbs == 1 ? j0 / 8 : (j0 % 64) / 8;     // chunk in the block
            const int lc = hc + (xl.nbs == 1 ? 4 : 0);
            *reinterpret_cast<uint4*>(mine + hb * 128 + ((hc ^ sw) << 4)) = hi;
            *reinterpret_cast<uint4*>(mine + lb * 128 + ((lc ^ sw) << 4)) = lo;
          }
        }
        if (FP8 && nx > 0) {
          // e4m3 base: y = sx sw (xq Wq) + the expand, in one accumulator.  Once the base
          // blocks are complete their product is scaled in TMEM; the expand blocks, the
          // first released only after this, then add the low-rank term unscaled.  (base_full
          // of this buffer is at most one phase ahead: its next tile waits for this drain.)
          if (!mbar_wait(&base_full[b], (uint32_t)kph & 1u, a.err)) ok = false;
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < BN; c += 32) {  // (warp-uniform: tcgen05.ld / st are aligned)
            float acc[32];
            tmem_acc32(tmem_row + c, acc);
            scale32(acc, sxr_v, sw_tile + c);
            uint32_t raw[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) raw[i] = __float_as_uint(acc[i]);
            tmem_st_32x32b_x32(tmem_row + c, raw);
          }
          tmem_st_wait();
          tc_fence_before();  // ordered before the MMA lane's expand blocks (xa_full below)
        }
        for (int e = 0; e < nx; ++e) {
          const int st = (ring + nk + e) % stages;  // after the tile's base blocks
          const uint32_t gp = (gpar >> st) & 1u;
          gpar ^= 1u << st;
          if (!mbar_wait(&xgrant[st], gp, a.err)) {
            ok = false;
            break;
          }
          const int uu = e / xl.nbs, blk = e - uu * xl.nbs;
          const bool own = uslot[uu] == srow;  // rows of other slots contribute zeros
          uint8_t* sa = stage_base + (size_t)st * kStageBytes;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const int p = (c ^ sw) << 4;  // the 8 rows of a quarter-warp cover all banks
            const uint4 val = own ? *reinterpret_cast<const uint4*>(mine + blk * 128 + p)
                                  : make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(sa + et * 128 + p) = val;
          }
          fence_proxy_async_smem();  // generic-proxy writes -> the MMA's async-proxy reads
          named_barrier(1, 128);
          if (et == 0) {
            if (PAIR && pr != 0)
              mbar_arrive_remote(dsmem_map(smem_u32(&xa_full[st]), lead_rank));
            else
              mbar_arrive(&xa_full[st]);
          }
        }
        ring += nx;
      }
      ring += nk;
      const bool full_ok = ok && mbar_wait(&tmem_full[b], (uint32_t)kph & 1u, a.err);
      // a split K (one tile per CTA) must still meet its cluster barrier below, whatever
      // the error (the flag is set); otherwise stop here
      if (!full_ok && cs == 1) break;
      tc_fence_after();
      if (VMODE && !head) {
        // ---- stream-K tail: its fp32 partial, for the slot that finishes the tile ----
        float4* part = reinterpret_cast<float4*>(a.sk_part) + (size_t)blockIdx.x * (BN / 4) * kBM + rt;
        for (int c = 0; c < BN; c += 32) {
          uint32_t raw[32];
          tmem_ld_32x32b_x32(tmem_row + c, raw);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 8; ++i)
            __stcg(part + (size_t)((c >> 2) + i) * kBM,
                   make_float4(__uint_as_float(raw[4 * i]), __uint_as_float(raw[4 * i + 1]),
                               __uint_as_float(raw[4 * i + 2]), __uint_as_float(raw[4 * i + 3])));
        }
        __threadfence();  // the partial is visible device-wide before the flag
        tc_fence_before();
        named_barrier(1, 128);
        if (et == 0) {
          st_release_gpu(a.sk_sync + 2 + blockIdx.x, epoch + 1);
          if (PAIR && pr != 0)
            mbar_arrive_remote(dsmem_map(smem_u32(&tmem_empty[b]), lead_rank));
          else
            mbar_arrive(&tmem_empty[b]);
        }
        continue;
      }
      // stream-K head of a split tile: its tail's partial (slot g0 + 1) is added below
      const int sk_src = VMODE && nk < nkb ? (PAIR ? 2 * (g0 + 1) + pr : g0 + 1) : -1;
      if (sk_src >= 0 && et == 0 &&
          !wait_flag_gpu(a.sk_sync + 2 + sk_src, epoch + 1, a.err))
        ok = false;

      // ---------------- split K: exchange partial accumulators through L2 ----------------
      // (delta mode, one tile per CTA.)  Scratch of this output block: [d][z] blocks (CTA
      // z's partial of CTA d's columns) of [bnc / 4][128 rows] float4, rows fastest, so a
      // warp's 32 rows move 512 contiguous bytes.
      const int nq = bnc / 4;
      const float4* xk_in = nullptr;  // the cs blocks addressed to this CTA: [q][nq][128]
      if (cs > 1) {
        float4* xk_tile =
            reinterpret_cast<float4*>(a.xk) + (size_t)(mt_i * nt + nt_i) * cs * cs * nq * kBM;
        xk_in = xk_tile + (size_t)z * cs * nq * kBM;
        for (int d = 0; d < cs; ++d) {
          if (d == z) continue;
          float4* blk = xk_tile + (size_t)(d * cs + z) * nq * kBM + rt;
          for (int c = 0; c < bnc; c += 32) {
            uint32_t raw[32];
            tmem_ld_32x32b_x32(tmem_row + d * bnc + c, raw);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 8; ++i)
              __stcg(blk + (size_t)((c >> 2) + i) * kBM,
                     make_float4(__uint_as_float(raw[4 * i]), __uint_as_float(raw[4 * i + 1]),
                                 __uint_as_float(raw[4 * i + 2]),
                                 __uint_as_float(raw[4 * i + 3])));
          }
        }
        // release / acquire across the cluster: every block addressed to this CTA is
        // written (the producer and MMA warps, done with their single tile, arrive at the
        // matching barrier after their loops)
        tc_fence_before();
        cluster_arrive_release();
        cluster_wait_acquire();
        tc_fence_after();
      }

      // ---------------- the epilogue's inputs, landed in shared memory ----------------
      // (Delta mode has one tile per CTA, and a stream-K head is its slot's last segment: the
      // ring is idle once the accumulator is complete, and holds these.)
      const int n_extra = cs > 1 ? cs - 1 : (sk_src >= 0 ? 1 : 0);
      float4* xin = reinterpret_cast<float4*>(stage_base);
      __nv_bfloat16* yrow = static_cast<__nv_bfloat16*>(a.y) + (size_t)row * a.N;
      const int cbase = z * bnc;  // first accumulator column this CTA finishes
      if (!vmode) {
        // ---- delta mode ----
        // xin: the cs - 1 partial blocks addressed to this CTA ([j][bnc / 4][128 rows]
        // float4, as in the scratch), a bulk copy each; dsm: the tile's delta rows as
        // [bnc / 32][128 rows][32] fp32 (16-byte chunk q of row r at chunk q ^ (r & 7): the
        // 128-byte swizzle of a TMA box), a tensor load per 32 columns, each counted on its
        // own barrier (the v-mode stage barriers xgrant and xa_full, idle here), so that the
        // first columns are finished while the rest land.  (y leaves by 16-byte stores of
        // each thread's row: staging it for TMA stores measured no faster.)
        const uint32_t blk_bytes = (uint32_t)nq * kBM * 16;
        const int nbox = bnc / 32;
        float* dsm = reinterpret_cast<float*>(stage_base + (size_t)(cs - 1) * blk_bytes);
        uint64_t* dbar = xgrant;  // [nbox <= 2 * stages]
        if (cs > 1 && et == 0) {
          // the peers' blocks were stored by generic-proxy writes seen through the cluster
          // barrier: order the bulk copies (async proxy) after them
          fence_proxy_async_global();
          mbar_arrive_expect_tx(xinfo_bar, (uint32_t)(cs - 1) * blk_bytes);
          for (int q = 0, j = 0; q < cs; ++q) {
            if (q == z) continue;
            bulk_load_g2s(xin + (size_t)j * nq * kBM, xk_in + (size_t)q * nq * kBM, blk_bytes,
                          xinfo_bar);
            ++j;
          }
        }
        // e4m3 base: the row's scale (written by the row quantiser this kernel's producer
        // waited for: read through L2) and this CTA's column scales, staged in shared memory
        float sxr = 0.f;
        float* sw_s = sw_tile;
        if (FP8) {
          sxr = row < a.M ? __ldcg(a.sx + row) : 0.f;
          for (int i = et; i < bnc; i += 128) sw_s[i] = __ldg(a.sw + n0 + cbase + i);
        }
        // (one tile per CTA: every barrier below is in its first phase)
        if (cs > 1 && !mbar_wait(xinfo_bar, 0u, a.err)) ok = false;
        named_barrier(1, 128);  // the column scales staged
        // While the low-rank kernel may still run: this CTA's columns of the product, the
        // peers' partials added and (e4m3) scaled, back into block 0 (row rt's own entries)
        if (cs > 1) {
#pragma unroll 1
          for (int c = 0; c < bnc; c += 32) {
            float acc[32];
            tmem_acc32(tmem_row + cbase + c, acc);
            for (int j = 0; j < cs - 1; ++j) add_block32(acc, xin + (size_t)j * nq * kBM + rt, c);
            if (FP8) scale32(acc, sxr, sw_s + c);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              xin[(size_t)((c >> 2) + i) * kBM + rt] =
                  make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
          }
        }
        // only now the low-rank kernel's results are needed: the main loop, the split-K
        // exchange and the partial sums ran while it was still working
        griddep_wait();
        bool add_delta = false;  // the row adds the low-rank term of the delta buffer
        if (row < a.M) {
          const int t = a.ex.token_slot[row];
          add_delta = t >= 0 && t < a.ex.S && a.ex.loaded[t] != 0;
          // one CTA per row block reports ids outside [-1, S) or naming empty slots
          if (nt_i == 0 && z == 0) {
            if (t < -1 || t >= a.ex.S) atomicOr(a.err, LORA_ERRF_BAD_ID);
            else if (t >= 0 && !add_delta) atomicOr(a.err, LORA_ERRF_EMPTY_SLOT);
          }
        }
        if (add_delta && !LORA_IN_BOUNDS(row < a.ex.delta_rows, a.err)) add_delta = false;
        // the tile's delta rows (the buffer holds the batch's rows, at most 512; the map
        // fills zeros past its rows and past N)
        const int cfirst = n0 + cbase;  // first column this CTA finishes
        if (et == 0) {
          fence_proxy_async_global();  // written by the low-rank kernel (waited for above)
          for (int h = 0; h < nbox; ++h) {
            mbar_arrive_expect_tx(&dbar[h], (uint32_t)kBM * 32 * 4);
            tma_load_2d(dsm + (size_t)h * kBM * 32, &tmap_delta, &dbar[h], cfirst + 32 * h, m0);
          }
        }
#pragma unroll 1
        for (int c = 0; c < bnc; c += 32) {
          float acc[32];
          if (cs > 1) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float4 v = xin[(size_t)((c >> 2) + i) * kBM + rt];
              acc[4 * i] = v.x;
              acc[4 * i + 1] = v.y;
              acc[4 * i + 2] = v.z;
              acc[4 * i + 3] = v.w;
            }
          } else {
            tmem_acc32(tmem_row + cbase + c, acc);
            if (FP8) scale32(acc, sxr, sw_s + c);
          }
          if (!mbar_wait(&dbar[c >> 5], 0u, a.err)) ok = false;
          if (add_delta) {
            const float* dbox = dsm + (size_t)(c >> 5) * kBM * 32 + (size_t)rt * 32;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const float4 d = *reinterpret_cast<const float4*>(dbox + ((q ^ (rt & 7)) << 2));
              acc[4 * q] += d.x;
              acc[4 * q + 1] += d.y;
              acc[4 * q + 2] += d.z;
              acc[4 * q + 3] += d.w;
            }
          }
          store_y32(acc, a, row, cfirst + c, yrow);
        }
      } else {
        // ---- v mode: a stream-K head adds its tail's partial (one block) ----
        // (e4m3 base: the accumulator holds sx sw base + expand when the tile has expand
        // blocks, so the partial is scaled alone; else the sum is scaled here)
        if (sk_src >= 0) {
          named_barrier(1, 128);  // the flag was seen by thread 0 of the epilogue
          const float4* src = reinterpret_cast<const float4*>(a.sk_part) +
                              (size_t)sk_src * (BN / 4) * kBM + rt;
          for (int c4 = 0; c4 < nq; ++c4)
            cp_async_16(xin + (size_t)c4 * kBM + rt, src + (size_t)c4 * kBM);
          cp_async_wait_all();
          named_barrier(1, 128);
        }
#pragma unroll 1
        for (int c = 0; c < bnc; c += 32) {
          float acc[32];
          tmem_acc32(tmem_row + cbase + c, acc);
          if (FP8 && tile_nx > 0) {
            if (n_extra > 0) {
              float p[32];
#pragma unroll
              for (int i = 0; i < 32; ++i) p[i] = 0.f;
              for (int j = 0; j < n_extra; ++j) add_block32(p, xin + (size_t)j * nq * kBM + rt, c);
              scale32(p, sxr_v, sw_tile + c);
#pragma unroll
              for (int i = 0; i < 32; ++i) acc[i] += p[i];
            }
          } else {
            for (int j = 0; j < n_extra; ++j) add_block32(acc, xin + (size_t)j * nq * kBM + rt, c);
            if (FP8) scale32(acc, sxr_v, sw_tile + c);
          }
          store_y32(acc, a, row, n0 + cbase + c, yrow);
        }
      }
      // this buffer is drained: the MMAs may fill it with tile k + 2 (pairs: both CTAs'
      // epilogues arrive on the even CTA's barrier)
      tc_fence_before();
      named_barrier(1, 128);
      if (et == 0) {
        if (PAIR && pr != 0)
          mbar_arrive_remote(dsmem_map(smem_u32(&tmem_empty[b]), lead_rank));
        else
          mbar_arrive(&tmem_empty[b]);
      }
    }
  }

  // split K: the producer and MMA warps meet the epilogue warps' cluster barrier
  if (cs > 1 && warp < 2) {
    cluster_arrive_release();
    cluster_wait_acquire();
  }
  tc_fence_before();
  __syncthreads();
  // stream-K: the last CTA to leave advances the epoch (every CTA read it at its start)
  if (VMODE && sk_slots > 0 && threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(a.sk_sync + 1, 1) == (int)(gridDim.x * gridDim.z) - 1) {
      atomicExch(a.sk_sync + 1, 0);
      __threadfence();
      atomicAdd(a.sk_sync, 1);
    }
  }
  // pairs: the peer is done with this CTA's TMEM, shared memory and barriers
  if (PAIR) cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    if (PAIR)
      tmem_dealloc_pair(tmem_base, 2 * BN);
    else
      tmem_dealloc(tmem_base, 2 * BN);
  }
}

// ---------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

cudaError_t encode_tmap_bf16(CUtensorMap* map, const void* base, int rows, int K, int box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t encode_tmap_delta(CUtensorMap* map, const float* base, int rows, int N) {
  auto enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  if (N % 4 != 0 || rows < 1) return cudaErrorInvalidValue;  // rows start on 16-byte boundaries
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(N) * 4};
  const cuuint32_t box[2] = {32, static_cast<cuuint32_t>(kBM)};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t encode_tmap_u8(CUtensorMap* map, const void* base, int rows, int K, int box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  if (K % 16 != 0) return cudaErrorInvalidValue;  // rows start on 16-byte boundaries
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(2 * kBK), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Raise (never lower) one kernel variant's dynamic shared-memory limit: one cache per
// variant, shared by every caller.
template <int BN, bool PAIR, bool VMODE, bool FP8 = false>
static cudaError_t raise_smem_limit(int bytes) {
  static int limit[kAttrDevices] = {};
  return ensure_smem_limit(gemm_tc_kernel<BN, PAIR, VMODE, FP8>, bytes, limit);
}

// CTAs of this GEMM that can be resident at once in clusters of `csize` CTAs (every variant
// holds one CTA per SM; a cluster must fit in one GPC, whose sizes differ).  Queried once
// per device.
static int resident_ctas(int csize, int num_sms) {
  static int cache_all[kAttrDevices][9] = {};
  static int scratch[9] = {};
  if (csize < 1 || csize > 8) return 0;
  const int dev = attr_device();
  int* cache = dev >= 0 ? cache_all[dev] : scratch;
  {
    std::lock_guard<std::mutex> lock(attr_mutex());
    if (cache[csize] != 0) return cache[csize];
  }
  {
    const int smem = 200 * 1024;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(csize * 64);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0, v = 0;
    if (raise_smem_limit<256, false, true>(smem) == cudaSuccess &&
        cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<256, false, true>, &cfg) ==
            cudaSuccess &&
        n > 0) {
      v = std::min(num_sms, n * csize);
    } else {
      cudaGetLastError();
      v = csize == 1 ? num_sms : 8 * (num_sms / 8 / csize) * csize;
    }
    std::lock_guard<std::mutex> lock(attr_mutex());
    cache[csize] = v;
    return v;
  }
}

// Tile shape, K split and CTA pairs, by least estimated time (cycles).  Measured on this
// kernel: a 64-wide K block costs its 4 MMA instructions (~124 cycles each below N = 256,
// 128 at N = 256) plus ~50 cycles of barrier hand-off, or its operand delivery at ~75 B
// per cycle per SM when that is slower (a 128 x 256 tile's 48 KB per block; a CTA pair
// halves the W rows each CTA loads, which made 256 x 256 pair tiles ~15% faster per block
// than 128 x 256 single-CTA tiles).  Each wave adds ~3k cycles of prologue, pipeline fill
// and epilogue; a split K adds the exchange of fp32 partials through L2 (written and read
// at ~50 B per cycle per SM).  Large problems (no split allowed) weigh the same costs
// without the split; their expand blocks (one per distinct slot of a tile) are not in
// the estimate, but a pair runs the expand blocks of all its 256 rows on both CTAs, which
// doubles them where slots change every few rows: pairs are taken there only when the
// batch averages at least 128 rows per slot (`slots` = the layer's slot count, 0 = none).
// With the e4m3 base in v mode single CTAs at N = 256 measured faster than pairs on every
// shape tried but one (8-18% at K = 4096; pairs 4% ahead at K = 14336, N = 4096), so the
// caller turns pairs off there.
GemmPlan gemm_tc_plan(int M, int N, int K, int num_sms, bool allow_split, int slots,
                      bool allow_pair) {
  const int mt = (M + kBM - 1) / kBM;
  const int nkb = (K + kBK - 1) / kBK;
  // every one of the cs K ranges of ceil(nkb / cs) blocks must be non-empty
  auto ranges_ok = [nkb](int c) { return (c - 1) * ((nkb + c - 1) / c) < nkb; };
  GemmPlan p{64, 1, 0};
  double best = 1e30;
  const int cand[3] = {256, 128, 64};
  // single CTAs first: a pair is taken only where it is estimated faster
  for (int pair = 0; pair <= 1; ++pair) {
    if (pair && (mt < 2 || !allow_pair)) continue;  // (one row tile: a pair leaves a CTA idle)
    if (pair && !allow_split && slots > 0 && (long long)M < 128LL * slots) continue;
    for (int i = 0; i < 3; ++i) {
      const int bn = cand[i];
      if (pair && bn < 128) continue;
      const double bytes = kABytes + (double)(pair ? bn / 2 : bn) * kBK * 2;
      const double per_kb = std::max(bytes / 75.0, 4.0 * std::max(124.0, 0.5 * bn)) + 50.0;
      const int ctas_m = pair ? 2 * ((mt + 1) / 2) : mt;
      const int tiles = ctas_m * ((N + bn - 1) / bn);
      // each CTA finishes bn / cs >= 32 columns (its epilogue and the split-K exchange work
      // in 32-column chunks)
      for (int cs = 1; cs <= (allow_split ? 4 : 1) && bn / cs >= 32; cs *= 2) {
        if (cs > 1 && !ranges_ok(cs)) break;
        const int conc = resident_ctas((pair ? 2 : 1) * cs, num_sms);
        if (conc < 1) continue;
        const int waves = (tiles * cs + conc - 1) / conc;
        const int kb = (nkb + cs - 1) / cs;
        const double exch = cs > 1 ? 2.0 * (cs - 1) * kBM * (bn / cs) * 4.0 / 50.0 : 0.0;
        const double cost = waves * (kb * per_kb + 3000.0 + exch);
        if (cost < best * 0.999) {
          best = cost;
          p.block_n = bn;
          p.ksplit = cs;
          p.pair = pair;
        }
      }
    }
  }
  return p;
}

// Split-K scratch of a plan: per output block (one per CTA of a K range) cs x cs blocks of
// 128 rows x BN / cs columns.
static size_t exchange_floats(const GemmPlan& p, int M, int N) {
  if (p.ksplit <= 1) return 0;
  const int mt = (M + kBM - 1) / kBM;
  const size_t gx = p.pair ? 2 * ((mt + 1) / 2) : mt;
  const size_t gy = (N + p.block_n - 1) / p.block_n;
  return gx * gy * p.ksplit * p.block_n * kBM;
}

// A delta-mode batch whose no-split plan leaves a last round of tiles at most half full
// runs as two launches: the column tiles of the whole rounds without a K split, then the
// remaining column tiles with a 2-way K split (their 2 x csize-CTA clusters fit in one
// round), so the last round takes half the time.  Returns the column tiles of the first
// launch, or 0 for no split.
static int delta_split_tiles(const GemmPlan& p, int M, int N, int nkb, int num_sms) {
  if (p.ksplit != 1 || nkb < 2) return 0;
  const int csize = p.pair ? 2 : 1;
  const int mt = (M + kBM - 1) / kBM, mtp = p.pair ? (mt + 1) / 2 : mt;
  const int nt = (N + p.block_n - 1) / p.block_n, units = mtp * nt;
  const int G = resident_ctas(csize, num_sms) / csize;
  if (G < 1 || units <= G || units % G == 0 || 2 * (units % G) > G) return 0;
  const int ntA = (units / G) * G / mtp, ntB = nt - ntA;
  if (ntA < 1 || ntB < 1 || 2 * csize * mtp * ntB > resident_ctas(2 * csize, num_sms)) return 0;
  if (p.block_n / 2 < 32) return 0;
  return ntA;
}

size_t gemm_tc_exchange_floats(int M, int N, int K, int num_sms) {
  const GemmPlan p = gemm_tc_plan(M, N, K, num_sms, true, 0);
  const int ntA = delta_split_tiles(p, M, N, (K + kBK - 1) / kBK, num_sms);
  if (ntA > 0)  // the second launch: the remaining columns with a 2-way split
    return exchange_floats(GemmPlan{p.block_n, 2, p.pair}, M, N - ntA * p.block_n);
  return exchange_floats(p, M, N);
}

size_t gemm_tc_plan_exchange_floats(const GemmPlan& p, int M, int N) {
  return exchange_floats(p, M, N);
}

int gemm_tc_tile_index(int BN) { return BN == 256 ? 0 : (BN == 128 ? 1 : 2); }

static size_t tc_smem_bytes(int BN, bool pair, bool fp8, int stages, int xscr_bytes) {
  const size_t stage = (size_t)kABytes + (size_t)(pair ? BN / 2 : BN) * kBK * 2;
  return 1024 + stages * stage + xscr_bytes + (2 * kBM + 8) * 4 + (fp8 ? BN * 4 : 0) +
         (4 * stages + 8) * 8;
}

template <int BN, bool PAIR, bool VMODE, bool FP8 = false>
static cudaError_t launch_tc(const GemmArgs& a, const GemmPlan& plan, const CUtensorMap& tmap_x,
                             const CUtensorMap& tmap_w, const CUtensorMap& tmap_bx,
                             cudaStream_t stream) {
  // delta mode leaves ~8 KB of the SM's shared memory to a CTA of the BGMV kernel, which
  // then runs on the same SM while the main loop does
  const size_t budget = a.ex.mode == kExpandDelta ? 219 * 1024 : 227 * 1024;
  const int cs = plan.ksplit;
  if (cs < 1 || cs > 4 || BN / cs < 32) return cudaErrorInvalidConfiguration;
  if (a.ex.mode == kExpandV && (cs != 1 || a.ex.R % 8 != 0 || a.ex.R > 128 || a.ex.S > 32 * kBM))
    return cudaErrorInvalidValue;
  const int xscr = a.ex.mode == kExpandV ? kBM * expand_layout(a.ex.R).nbs * 128 : 0;
  if (cs > 1 && (!a.xk || a.xk_floats < exchange_floats(plan, a.M, a.n_end - a.n_begin)))
    return cudaErrorInvalidValue;
  int stages = 8;
  while (stages > 2 && tc_smem_bytes(BN, PAIR, FP8, stages, xscr) > budget) --stages;
  const size_t smem = tc_smem_bytes(BN, PAIR, FP8, stages, xscr);
  if (smem > budget) return cudaErrorInvalidConfiguration;
  // the epilogue lands its split-K partials and delta rows (128 x BN fp32) in the ring, and
  // counts each 32-column delta box on one of the 2 * stages v-mode stage barriers
  if (a.ex.mode == kExpandDelta && 2 * stages < BN / cs / 32) return cudaErrorInvalidConfiguration;
  const size_t stage = (size_t)kABytes + (size_t)(PAIR ? BN / 2 : BN) * kBK * 2;
  if ((cs > 1 || a.ex.mode == kExpandDelta || a.sk_part) &&
      (size_t)stages * stage < (size_t)kBM * BN * 4)
    return cudaErrorInvalidConfiguration;
  cudaError_t e = raise_smem_limit<BN, PAIR, VMODE, FP8>((int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = PAIR ? 2 : 1;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = cs;
  // work units: (row tile, or pair of row tiles; column tile).  v mode: a persistent grid
  // of at most the resident CTAs (pairs), each running units round-robin; delta mode (its
  // epilogue reuses the idle ring): one unit per CTA.  A pair's last CTA may lie past M: it
  // loads zeros and stores nothing.
  const int mt = (a.M + kBM - 1) / kBM;
  const int mtp = PAIR ? (mt + 1) / 2 : mt;
  const int nt = (a.n_end - a.n_begin + BN - 1) / BN;
  const int units = mtp * nt;
  const int csize = (PAIR ? 2 : 1) * cs;
  int G = units;
  if (a.ex.mode == kExpandV) G = std::max(1, std::min(units, resident_ctas(csize, a.num_sms) / csize));
  // stream-K: when the units leave a last round of at most half the slots busy, those
  // tiles are cut in two (head and tail on two slots) instead; only a K range of at least
  // two of the kernel's K blocks (128 elements each with the e4m3 base) is cut, so that
  // the head starts its accumulator with a block of its own
  constexpr int kKE = FP8 ? 2 * kBK : kBK;
  int full_rounds = (units + G - 1) / G, sk_slots = 0;
  if (a.ex.mode == kExpandV && a.sk_part && a.sk_sync && units > G && (a.K + kKE - 1) / kKE >= 2) {
    const int rem = units % G;
    if (rem > 0 && 2 * rem <= G) {
      full_rounds = units / G;
      sk_slots = 2 * rem;
    }
  }
  cfg.gridDim = dim3((PAIR ? 2 : 1) * G, 1, cs);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = (PAIR || cs > 1) ? 2 : 1;
  // row tiles (pairs) per band: x of a band at most ~32 MB
  const size_t band_rows = (size_t)kBM * (PAIR ? 2 : 1);
  const int group_m =
      std::max(1, std::min(mtp, (int)((32u << 20) / ((size_t)a.K * band_rows * 2))));
  // delta mode: the delta tile arrives through the delta buffer's map
  if (!VMODE && !a.tmap_delta) return cudaErrorInvalidValue;
  return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<BN, PAIR, VMODE, FP8>, tmap_x, tmap_w, tmap_bx,
                            VMODE ? tmap_w : *a.tmap_delta, a, stages, xscr, group_m, mtp, nt,
                            full_rounds, sk_slots);
}

static cudaError_t launch_variant_fp8(const GemmArgs& a, const GemmPlan& plan,
                                      const CUtensorMap& tmap_x, const CUtensorMap& tw,
                                      const CUtensorMap& tb, cudaStream_t stream) {
  if (a.ex.mode == kExpandV) {
    if (plan.pair) {
      if (plan.block_n == 256) return launch_tc<256, true, true, true>(a, plan, tmap_x, tw, tb, stream);
      if (plan.block_n == 128) return launch_tc<128, true, true, true>(a, plan, tmap_x, tw, tb, stream);
      return cudaErrorInvalidConfiguration;
    }
    switch (plan.block_n) {
      case 256: return launch_tc<256, false, true, true>(a, plan, tmap_x, tw, tb, stream);
      case 128: return launch_tc<128, false, true, true>(a, plan, tmap_x, tw, tb, stream);
      default: return launch_tc<64, false, true, true>(a, plan, tmap_x, tw, tb, stream);
    }
  }
  if (plan.pair) {
    if (plan.block_n == 256) return launch_tc<256, true, false, true>(a, plan, tmap_x, tw, tw, stream);
    if (plan.block_n == 128) return launch_tc<128, true, false, true>(a, plan, tmap_x, tw, tw, stream);
    return cudaErrorInvalidConfiguration;
  }
  switch (plan.block_n) {
    case 256: return launch_tc<256, false, false, true>(a, plan, tmap_x, tw, tw, stream);
    case 128: return launch_tc<128, false, false, true>(a, plan, tmap_x, tw, tw, stream);
    default: return launch_tc<64, false, false, true>(a, plan, tmap_x, tw, tw, stream);
  }
}

template <bool VMODE>
static cudaError_t launch_variant(const GemmArgs& a, const GemmPlan& plan,
                                  const CUtensorMap& tmap_x, const CUtensorMap& tw,
                                  const CUtensorMap& tb, cudaStream_t stream) {
  if (plan.pair) {
    if (plan.block_n == 256) return launch_tc<256, true, VMODE>(a, plan, tmap_x, tw, tb, stream);
    if (plan.block_n == 128) return launch_tc<128, true, VMODE>(a, plan, tmap_x, tw, tb, stream);
    return cudaErrorInvalidConfiguration;
  }
  switch (plan.block_n) {
    case 256: return launch_tc<256, false, VMODE>(a, plan, tmap_x, tw, tb, stream);
    case 128: return launch_tc<128, false, VMODE>(a, plan, tmap_x, tw, tb, stream);
    default: return launch_tc<64, false, VMODE>(a, plan, tmap_x, tw, tb, stream);
  }
}

static cudaError_t launch_one(const GemmArgs& a, const GemmPlan& plan,
                              const CUtensorMap* tmap_w3, const CUtensorMap* tmap_bx3,
                              cudaStream_t stream);

cudaError_t launch_gemm_tc(const GemmArgs& a, const CUtensorMap* tmap_w3,
                           const CUtensorMap* tmap_bx3, cudaStream_t stream, int* launches) {
  if (a.ex.mode == kExpandV && !tmap_bx3) return cudaErrorInvalidValue;
  if (a.fp8 && (!a.tmap_xq || !a.sx || !a.sw || a.K % 16 != 0)) return cudaErrorInvalidValue;
  // the plan counts K blocks of 128 bytes: an e4m3 row of K elements is K / 2 bf16 wide
  const int k_bytes2 = a.fp8 ? (a.K + 1) / 2 : a.K;
  GemmPlan plan = gemm_tc_plan(a.M, a.N, k_bytes2, a.num_sms, a.ex.mode != kExpandV,
                               a.ex.mode == kExpandV ? a.ex.S : 0,
                               !(a.fp8 && a.ex.mode == kExpandV));
  if (a.force_bn != 0) {
    // v mode never splits K: its expand blocks run after the base ones in one accumulator
    plan = GemmPlan{a.force_bn, a.ex.mode == kExpandV ? 1 : a.force_cs, a.force_pair};
    const int nkb = (k_bytes2 + kBK - 1) / kBK, c = plan.ksplit;
    if (c > 1 && (c - 1) * ((nkb + c - 1) / c) >= nkb) return cudaErrorInvalidConfiguration;
  }
  GemmArgs whole = a;
  whole.n_begin = 0;
  whole.n_end = a.N;
  whole.trigger_next = false;
  whole.q_reset = true;  // the last launch of the batch resets the e4m3 row count
  // a last round at most half full: two launches (see delta_split_tiles)
  const int ntA = a.ex.mode == kExpandDelta && a.force_bn == 0
                      ? delta_split_tiles(plan, a.M, a.N, (k_bytes2 + kBK - 1) / kBK, a.num_sms)
                      : 0;
  if (ntA > 0) {
    GemmArgs first = whole, second = whole;
    first.n_end = ntA * plan.block_n;
    first.trigger_next = true;
    first.q_reset = false;
    second.n_begin = first.n_end;
    const GemmPlan plan2{plan.block_n, 2, plan.pair};
    cudaError_t e = launch_one(first, plan, tmap_w3, tmap_bx3, stream);
    if (e != cudaSuccess) return e;
    if (launches) ++*launches;
    e = launch_one(second, plan2, tmap_w3, tmap_bx3, stream);
    if (e == cudaSuccess && launches) ++*launches;
    return e;
  }
  const cudaError_t e = launch_one(whole, plan, tmap_w3, tmap_bx3, stream);
  if (e == cudaSuccess && launches) ++*launches;
  return e;
}

// One launch of the tcgen05 GEMM with the given plan (columns a.n_begin .. a.n_end).
static cudaError_t launch_one(const GemmArgs& a, const GemmPlan& plan, const CUtensorMap* tmap_w3,
                              const CUtensorMap* tmap_bx3, cudaStream_t stream) {
  if (a.fp8) {
    const int ti = gemm_tc_tile_index(plan.pair ? plan.block_n / 2 : plan.block_n);
    return launch_variant_fp8(a, plan, *a.tmap_xq, tmap_w3[ti],
                              tmap_bx3 ? tmap_bx3[ti] : tmap_w3[ti], stream);
  }
  CUtensorMap tmap_x;
  cudaError_t e = encode_tmap_bf16(&tmap_x, a.x, a.M, a.K, kBM);
  if (e != cudaSuccess) return e;
  // a CTA of a pair loads half of the N tile's rows: the map with boxes of block_n / 2 rows
  const int ti = gemm_tc_tile_index(plan.pair ? plan.block_n / 2 : plan.block_n);
  const CUtensorMap& tw = tmap_w3[ti];
  const CUtensorMap& tb = tmap_bx3 ? tmap_bx3[ti] : tw;  // unused in delta mode
  return a.ex.mode == kExpandV ? launch_variant<true>(a, plan, tmap_x, tw, tb, stream)
                                : launch_variant<false>(a, plan, tmap_x, tw, tb, stream);
}

}  // namespace lora
