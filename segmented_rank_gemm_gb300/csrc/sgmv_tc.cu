// sgmv_tc.cu -- SGMV shrink on the fifth-generation tensor cores:
//   v[row, 0:R] = (alpha_s / r_s) * x[row, :] A_s      for every adapted row, s = its slot.
//
// "Serving multiple LoRAs: segmented matrix multiplies and adapter scheduling", section
// "Not merging the weights, computing in batches": SGMV groups the tokens of one adapter
// into a segment and runs one small matrix multiply per segment.  "Serving LoRA adapters
// ..." (vLLM) Step 4: the shrink result is an fp32 buffer of rank width, later expanded
// into the base output.
//
// Work list (from the segment builder): units.  A unit is a window of 128 consecutive
// positions of perm (the rows sorted by slot, so a window holds whole or partial segments,
// each of one slot) together with up to Gp of the segments that overlap it; a window that
// spans more segments gives several units.  A work item is one unit and one of `ks` K
// ranges; its partial product goes to plane kp of v, and the consumer of v (the base
// GEMM's epilogue) sums a row's planes in plane order, so the result does not depend on
// which CTA ran which item.  The kernel is persistent and schedules items dynamically: a
// CTA's producer takes the next item from a device counter and passes it to the CTA's MMA
// and epilogue warps through the unit description ring (items differ in cost: windows with
// one or two segments, partial windows); the last CTA to finish resets the counters.
// One MMA serves all segments of a unit: the B operand stacks their transposed A blocks
// (Rt rows each), D[128, G*Rt] = X_win[128, K] * [A_s1 .. A_sG], and each row of the unit's
// segments keeps the Rt columns of its own slot (Gp * Rt <= 128, Gp <= 8).  The stacked A
// region of a stage is sized for Gp segments only, so that most of the shared memory holds
// x stages in flight.
//   warp 0      producer.  Per item it writes the unit's description (window, segment
//               boundaries clipped to the window, slots) into a small shared-memory ring
//               read by the other warps.  Per 64-wide K block it gathers the window's 128 x
//               rows (perm[p0 + i]) with 16-byte cp.async copies into the 128-byte-swizzled
//               K-major layout the MMA reads (positions past the window end are
//               zero-filled), and lane 0 loads the G A blocks with TMA (Rt rows from
//               each slot's first pool row: rows past the slot's own rank belong to
//               other slots or lie past the pool (zero-filled); their columns carry a
//               zero scale, so only the slot's rank columns reach v).  The stage's
//               mbarrier counts the 32 lanes' cp.async completions and the TMA bytes.
//   warp 1      one lane issues tcgen05.mma (M=128, N=G*Rt, K=16; bf16 x bf16 -> fp32) and
//               frees each stage with tcgen05.commit.  Two accumulators alternate between
//               items, so an item's epilogue overlaps the next main loop.
//   warps 2..5  epilogue: each thread owns one window row (TMEM lane): if the row belongs to
//               one of the unit's segments, it multiplies that segment's Rt columns by the
//               slot's column scales (alpha / r; w_i alpha_i / r_i on the columns of member
//               i of a composition) and stores the row's R fp32 values at v[kp][perm row].
// The x bytes dominate (every adapted row is read once per K range and unit of its
// window); each A_s is read once per unit.
// Launch: programmatic dependent launch after the segment builder; the kernel lets the base
// GEMM launch at once (its main loop needs nothing from here) and waits for the builder's
// results before it reads them.  Every mbarrier wait is bounded (lora_common.cuh).
#include <cudaTypedefs.h>

#include <algorithm>

#include "lora_common.cuh"
#include "lora_kernels.h"

namespace lora {

static constexpr int kShThreads = 192;
static constexpr int kShBK = 64;                           // K elements per stage (128 bytes)
static constexpr int kShXBytes = kTcTileRows * kShBK * 2;  // 16 KB of gathered x rows
static constexpr int kShNmax = 128;                        // stacked A rows per unit, at most
static constexpr int kShMaxGroups = 8;                     // segments per unit, at most
static constexpr int kShInfo = 4;                          // unit descriptions in flight
static constexpr int kShMaxSplit = 8;

// A unit's description, written by the producer, read by the MMA and epilogue warps.
struct UnitInfo {
  int p0;                       // first perm position of the window
  int G, kp;                    // segments in the unit, K range of this item
  int off[kShMaxGroups + 1];    // segment g covers positions [off[g], off[g + 1])
  int slot[kShMaxGroups];
  int rowb[kShMaxGroups];       // the slot's first row in the A pool
};

int sgmv_shrink_tc_groups(int Rt) { return std::max(1, std::min(kShMaxGroups, kShNmax / Rt)); }

__global__ void __launch_bounds__(kShThreads, 1)
    sgmv_shrink_tc_kernel(const __grid_constant__ CUtensorMap tmap_a, ShrinkTcArgs a, int ks,
                          int kpb, int stages, int Gp) {
  const int Rt = a.Rt;
  const int Nmax = Gp * Rt;  // stacked A rows per stage
  const uint32_t stage_bytes = (uint32_t)(kShXBytes + Nmax * kShBK * 2);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  UnitInfo* info = reinterpret_cast<UnitInfo*>(smem + (size_t)stages * stage_bytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(info + kShInfo);
  uint64_t* full = bars;
  uint64_t* empty = bars + stages;
  uint64_t* acc_full = bars + 2 * stages;             // [2] accumulator ready
  uint64_t* acc_empty = acc_full + 2;                 // [2] accumulator read out
  uint64_t* info_full = acc_empty + 2;                // [kShInfo] description written
  uint64_t* info_empty = info_full + kShInfo;         // [kShInfo] description released
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(info_empty + kShInfo);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 33);  // 32 lanes' cp.async completions + lane 0's TMA arrival
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 128);
    }
    for (int i = 0; i < kShInfo; ++i) {
      mbar_init(&info_full[i], 1);
      mbar_init(&info_empty[i], 1 + 128);  // the MMA lane and the 128 epilogue threads
    }
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) tma_prefetch_desc(&tmap_a);
  if (warp == 1) tmem_alloc(tmem_holder, 2 * kShNmax);  // two accumulators of <= 128 columns
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  griddep_launch_dependents();  // the base GEMM's main loop may start now
  griddep_wait();               // the segment builder's units, perm and segments
  const int n_items = a.meta[2] * ks;
  const int n_seg = a.meta[0], T_a = a.meta[1];
  const int nkb = (a.K + kShBK - 1) / kShBK;
  const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(a.x);

  if (warp == 0) {
    // ---------------- producer ----------------
    const int c = lane & 7;      // 16-byte chunk of the 128-byte row segment
    const int rsub = lane >> 3;  // this lane copies rows rsub + 4 i, i < 32
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    int item = 0;
    for (; ok; ++item) {
      int w = 0;
      if (lane == 0) w = atomicAdd(a.work, 1);  // the next item
      w = __shfl_sync(0xffffffffu, w, 0);
      // ---- the unit's description ----
      const int ib = item % kShInfo;
      if (!mbar_wait(&info_empty[ib], ((uint32_t)(item / kShInfo) & 1u) ^ 1u, a.err)) break;
      UnitInfo& ui = info[ib];
      if (w >= n_items) {  // no items left: tell the other roles
        if (lane == 0) {
          ui.G = 0;
          mbar_arrive(&info_full[ib]);
        }
        break;
      }
      const int u = w / ks;
      const int p0 = a.tile_row0[u], p1 = min(p0 + kTcTileRows, T_a);
      const int gs = a.tile_seg[u];
      // lanes g <= Gp: start of segment gs + g (seg_offsets[n_seg] = T_a ends the list)
      const int o = lane <= Gp ? a.seg_offsets[min(gs + lane, n_seg)] : 0;
      const bool in = lane < Gp && (lane == 0 || o < p1);
      const int G = __popc(__ballot_sync(0xffffffffu, in));
      if (in) {
        ui.off[lane] = max(o, p0);
        const int sl = a.seg_slot[gs + lane];
        ui.slot[lane] = sl;
        const int rb = a.row_base[sl];
        // (a row outside the pool: its A blocks are taken from row 0, and flagged)
        ui.rowb[lane] = LORA_IN_BOUNDS(rb >= 0 && rb < a.pool_rows, a.err) ? rb : 0;
      }
      if (lane == G) ui.off[G] = min(o, p1);
      if (lane == 0) {
        ui.p0 = p0;
        ui.G = G;
        ui.kp = w - u * ks;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&info_full[ib]);
      int prow[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int r = rsub + 4 * i;
        prow[i] = p0 + r < p1 ? a.perm[p0 + r] : -1;
      }
      const int kb0 = (w - u * ks) * kpb, kb1 = min(nkb, kb0 + kpb);
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(&empty[s], ph ^ 1u, a.err)) {
          ok = false;
          break;
        }
        uint8_t* sx = smem + (size_t)s * stage_bytes;
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[s], (uint32_t)(G * Rt * 128));
          for (int g = 0; g < G; ++g)
            tma_load_2d(sx + kShXBytes + g * Rt * 128, &tmap_a, &full[s], kb * kShBK,
                        ui.rowb[g]);
        }
        const int k = kb * kShBK + c * 8;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int r = rsub + 4 * i;
          const bool v = prow[i] >= 0 && k < a.K;
          const __nv_bfloat16* src = v ? x + (size_t)prow[i] * a.K + k : x;
          cp_async_16_zfill(sx + r * 128 + ((c ^ (r & 7)) << 4), src, v ? 16u : 0u);
        }
        cp_async_mbar_arrive_noinc(&full[s]);
        if (++s == stages) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    // a stage whose consumer gave up may still be landing: let it land before exiting
    cp_async_wait_all();
    if (!ok && lane == 0) {
      const int ls = s == 0 ? stages - 1 : s - 1;
      mbar_wait(&full[ls], s == 0 ? ph ^ 1u : ph, nullptr);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint64_t x_desc0 = smem_desc_sw128(smem_u32(smem));
      const uint64_t b_desc0 = smem_desc_sw128(smem_u32(smem + kShXBytes));
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int item = 0; ok; ++item) {
        const int ib = item % kShInfo;
        if (!mbar_wait(&info_full[ib], (uint32_t)(item / kShInfo) & 1u, a.err)) break;
        const int G = info[ib].G, kp = info[ib].kp;
        mbar_arrive(&info_empty[ib]);
        if (G == 0) break;  // no items left
        const int kb0 = kp * kpb, kb1 = min(nkb, kb0 + kpb);
        const uint32_t idesc = idesc_bf16_f32(kTcTileRows, G * Rt);
        const int buf = item & 1;
        const uint32_t use = (uint32_t)(item >> 1);
        if (!mbar_wait(&acc_empty[buf], (use & 1u) ^ 1u, a.err)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(buf * kShNmax);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&full[s], ph, a.err)) {
            ok = false;
            break;
          }
          fence_proxy_async_smem();  // gathered rows were written through the generic proxy
          tc_fence_after();
          const uint64_t off = (uint64_t)(s * (stage_bytes >> 4));
#pragma unroll
          for (int kk = 0; kk < kShBK / 16; ++kk)
            tc_mma_bf16(d, x_desc0 + off + (uint64_t)(kk * 2), b_desc0 + off + (uint64_t)(kk * 2),
                        idesc, (kb > kb0 || kk > 0) ? 1u : 0u);
          tc_commit(&empty[s]);
          if (++s == stages) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (ok) tc_commit(&acc_full[buf]);
      }
    }
    __syncwarp();
  } else {
    // ---------------- epilogue: scale and store v rows of plane kp ----------------
    const int quad = warp & 3;  // TMEM lanes [32 quad, 32 quad + 32)
    const int rt = quad * 32 + lane;
    const uint32_t tmem_row = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
    for (int item = 0;; ++item) {
      const int ib = item % kShInfo;
      if (!__all_sync(0xffffffffu,
                      mbar_wait(&info_full[ib], (uint32_t)(item / kShInfo) & 1u, a.err)))
        break;
      const UnitInfo& ui = info[ib];
      const int G = ui.G, p = ui.p0 + rt, kp = ui.kp;
      if (G == 0) {  // no items left
        mbar_arrive(&info_empty[ib]);
        break;
      }
      const bool live = p >= ui.off[0] && p < ui.off[G];
      int g = 0;  // the row's segment in the unit: the last g with off[g] <= p
      for (int j = 1; j < G; ++j) g += ui.off[j] <= p ? 1 : 0;
      const int slot = ui.slot[g];
      mbar_arrive(&info_empty[ib]);
      const int grow = live ? a.perm[p] : 0;
      const float* sc = a.scale + (size_t)slot * a.R;  // the slot's column scales
      const bool vrow_ok = !live || LORA_IN_BOUNDS(grow >= 0 && grow < a.v_rows && kp < a.ks, a.err);
      float* vrow = a.v + (size_t)kp * a.plane_stride + (size_t)grow * a.R;
      const int buf = item & 1;
      const uint32_t use = (uint32_t)(item >> 1);
      if (!__all_sync(0xffffffffu, mbar_wait(&acc_full[buf], use & 1u, a.err))) break;
      tc_fence_after();
      const int col0 = g * Rt;  // the row's accumulator columns
      for (int j0 = 0; j0 < G * Rt; j0 += 16) {
        uint32_t raw[16];
        tmem_ld_32x32b_x16(tmem_row + (uint32_t)(buf * kShNmax + j0), raw);
        tmem_ld_wait();
        const int j = j0 - col0;  // rank index of raw[0]
        if (live && vrow_ok && j >= 0 && j < Rt) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (j + 4 * q < a.R) {
              // columns past the slot's rank have scale 0; select rather than multiply,
              // so that whatever the pool holds past the slot's rows cannot leak in
              const float4 c = __ldg(reinterpret_cast<const float4*>(sc + j + 4 * q));
              *reinterpret_cast<float4*>(vrow + j + 4 * q) = make_float4(
                  c.x != 0.f ? c.x * __uint_as_float(raw[4 * q]) : 0.f,
                  c.y != 0.f ? c.y * __uint_as_float(raw[4 * q + 1]) : 0.f,
                  c.z != 0.f ? c.z * __uint_as_float(raw[4 * q + 2]) : 0.f,
                  c.w != 0.f ? c.w * __uint_as_float(raw[4 * q + 3]) : 0.f);
            }
        }
      }
      tc_fence_before();
      mbar_arrive(&acc_empty[buf]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 2 * kShNmax);
  }
  // every CTA has taken its last item: the last one to get here resets the counters for
  // the next launch
  if (threadIdx.x == 0 && atomicAdd(a.work + 1, 1) == (int)gridDim.x - 1) {
    atomicExch(a.work, 0);
    atomicExch(a.work + 1, 0);
  }
}

// K split: about two items per SM when the batch has few windows, each K range at least
// 8 blocks long, at most max_planes (and kShMaxSplit) ranges.
int sgmv_shrink_tc_split(int T, int K, int S, int num_sms, int max_planes) {
  (void)S;
  const int nkb = (K + kShBK - 1) / kShBK;
  const int windows = (T + kTcTileRows - 1) / kTcTileRows;
  int ks = (2 * num_sms + windows - 1) / std::max(windows, 1);
  ks = std::min(ks, std::min(max_planes, kShMaxSplit));
  ks = std::min(ks, std::max(1, nkb / 8));
  ks = std::max(ks, 1);
  // with ceil-sized ranges every range must be non-empty
  const int kpb = (nkb + ks - 1) / ks;
  return (nkb + kpb - 1) / kpb;
}

cudaError_t launch_sgmv_shrink_tc(const ShrinkTcArgs& a, const CUtensorMap& tmap_a,
                                  cudaStream_t stream) {
  if (a.Rt < 16 || a.Rt > 128 || a.Rt % 16 != 0 || a.R % 8 != 0 || a.R > a.Rt || a.K % 8 != 0 ||
      a.T < 1)
    return cudaErrorInvalidValue;
  const int ks = a.ks;
  const int nkb = (a.K + kShBK - 1) / kShBK;
  const int kpb = (nkb + ks - 1) / ks;
  if (ks < 1 || ks > kShMaxSplit || (ks - 1) * kpb >= nkb) return cudaErrorInvalidValue;
  const int Gp = sgmv_shrink_tc_groups(a.Rt);
  const size_t stage_bytes = (size_t)kShXBytes + (size_t)Gp * a.Rt * kShBK * 2;
  const size_t fixed = 1024 + kShInfo * sizeof(UnitInfo) + 64 * 8;
  const size_t budget = 227 * 1024;
  int stages = 10;
  while (stages > 2 && fixed + (size_t)stages * stage_bytes > budget) --stages;
  const size_t smem = fixed + (size_t)stages * stage_bytes;
  static int limit[kAttrDevices] = {};
  static bool carveout[kAttrDevices] = {};
  cudaError_t e = ensure_smem_limit(sgmv_shrink_tc_kernel, (int)smem, limit);
  if (e != cudaSuccess) return e;
  e = prefer_max_smem_carveout(sgmv_shrink_tc_kernel, carveout);
  if (e != cudaSuccess) return e;
  const int units = (a.T + kTcTileRows - 1) / kTcTileRows;  // at least (one per window)
  const int grid = std::max(1, std::min(units * ks, a.num_sms));
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kShThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, sgmv_shrink_tc_kernel, tmap_a, a, ks, kpb, stages, Gp);
}

}  // namespace lora
