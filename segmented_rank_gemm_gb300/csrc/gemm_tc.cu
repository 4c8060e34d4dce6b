// gemm_tc.cu -- base GEMM y = x W on the fifth-generation tensor cores, with the LoRA expand
// y += scale_slot * v B_slot fused into the epilogue so that y is written once.
//
// "LoRAX, in depth", section "Computing a batch that mixes adapters": the base term is the
// same for every request, so it runs as one large GEMM over all tokens; only the low-rank
// term differs by adapter.  "Serving LoRA adapters ..." (vLLM) Step 4: the expand multiplies
// the fp32 rank buffer by B and adds it to the base output.
//
// Kernel structure (one 128 x BN output tile per CTA, 6 warps):
//   warp 0      TMA producer: 64-wide K blocks of x [M,K] and of the packed weight W^T [N,K]
//               (both K-major, 128-byte swizzle) into a ring of shared-memory stages.
//   warp 1      allocates BN TMEM columns; one lane issues tcgen05.mma (M=128, N=BN, K=16,
//               bf16 x bf16 -> fp32 in TMEM) and frees each stage with tcgen05.commit.
//   warps 2..5  epilogue: each thread owns one output row (one TMEM lane).  It reads the
//               accumulator 32 columns at a time (tcgen05.ld), adds the row's low-rank term
//               and rounds to bf16 once:
//                 v mode     sum_j v_j B_slot[j, n], v (fp32, scaled by alpha / r) staged in
//                            shared memory, B_slot read 4 rank rows x 32 columns at a time;
//                 delta mode the fp32 delta[row, n] the tile kernel already expanded.
//               Rows with slot -1 store the base product only.
// Each CTA starts its K loop at a different K block (and wraps around), so the CTAs that
// share an x tile (same rows) or a W tile (same columns) do not all request the same lines
// from L2 at the same moment.
// Launch: programmatic dependent launch after the tile kernel: the main loop reads only x and
// W, so it runs while the low-rank kernels finish; the epilogue waits (griddepcontrol.wait)
// before it reads their results.
// Every mbarrier wait is bounded (lora_common.cuh): a broken pipeline sets an error flag.
#include <cudaTypedefs.h>

#include "lora_common.cuh"
#include "lora_kernels.h"

namespace lora {

static constexpr int kTcThreads = 192;
static constexpr int kBM = 128, kBK = 64;
static constexpr int kABytes = kBM * kBK * 2;

template <int BN>
__global__ void __launch_bounds__(kTcThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmap_x,
                   const __grid_constant__ CUtensorMap tmap_w, GemmArgs a, int stages) {
  constexpr int kBBytes = BN * kBK * 2;
  constexpr int kStageBytes = kABytes + kBBytes;
  const int R = a.ex.R;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* stage_base = smem;
  float* vs = reinterpret_cast<float*>(smem + (size_t)stages * kStageBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(vs + kBM * (R + 1));
  uint64_t* full = bars;
  uint64_t* empty = bars + stages;
  uint64_t* tmem_full = bars + 2 * stages;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * stages + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * kBM, n0 = blockIdx.y * BN;
  const int nkb = (a.K + kBK - 1) / kBK;
  const int kb0 = (int)((blockIdx.x + blockIdx.y) % (unsigned)nkb);  // rotated K start

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tmem_full, 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmap_x);
    tma_prefetch_desc(&tmap_w);
  }
  if (warp == 1) tmem_alloc(tmem_holder, BN);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      for (int it = 0; it < nkb; ++it) {
        const int kb = (kb0 + it) % nkb;
        if (!mbar_wait(&empty[s], ph ^ 1u, a.err)) break;
        uint8_t* sa = stage_base + (size_t)s * kStageBytes;
        mbar_arrive_expect_tx(&full[s], kStageBytes);
        tma_load_2d(sa, &tmap_x, &full[s], kb * kBK, m0);
        tma_load_2d(sa + kABytes, &tmap_w, &full[s], kb * kBK, n0);
        if (++s == stages) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, BN);
      int s = 0;
      uint32_t ph = 0;
      for (int it = 0; it < nkb; ++it) {
        if (!mbar_wait(&full[s], ph, a.err)) break;
        tc_fence_after();
        const uint32_t a_addr = smem_u32(stage_base + (size_t)s * kStageBytes);
        const uint32_t b_addr = a_addr + kABytes;
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          tc_mma_bf16(tmem_base, smem_desc_sw128(a_addr + kk * 32),
                      smem_desc_sw128(b_addr + kk * 32), idesc, (it | kk) != 0 ? 1u : 0u);
        }
        tc_commit(&empty[s]);
        if (++s == stages) {
          s = 0;
          ph ^= 1u;
        }
      }
      tc_commit(tmem_full);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue: low-rank term + store ----------------
    const int quad = warp & 3;  // TMEM lanes [32*quad, 32*quad + 32) are this warp's
    const int rt = quad * 32 + lane;
    const int row = m0 + rt;
    const ExpandArgs& ex = a.ex;
    griddep_wait();  // the segment builder and the tile kernel have finished
    int s = -1, r = 0;
    float* vrow = vs + rt * (R + 1);
    if (row < a.M) s = ex.row_slot[row];
    if (s >= 0 && ex.mode == kExpandV) {
      r = ex.rank[s];
      const float* vsrc = ex.v + (size_t)row * R;
      for (int j = 0; j < r; ++j) vrow[j] = vsrc[j];
    }
    mbar_wait(tmem_full, 0, a.err);
    tc_fence_after();

    const __nv_bfloat16* Bs =
        s >= 0 ? static_cast<const __nv_bfloat16*>(ex.B_pool) + (size_t)s * R * a.N : nullptr;
    const float* drow = ex.delta + (size_t)row * a.N;
    __nv_bfloat16* yrow = static_cast<__nv_bfloat16*>(a.y) + (size_t)row * a.N;
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += 32) {
      uint32_t raw[32];
      tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + c0, raw);
      tmem_ld_wait();
      float acc[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) acc[i] = __uint_as_float(raw[i]);
      const int n = n0 + c0;
      if (s >= 0 && ex.mode == kExpandDelta) {
        float4 d[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
          d[q] = (n + q * 4 < a.N) ? *reinterpret_cast<const float4*>(drow + n + q * 4)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          acc[q * 4 + 0] += d[q].x;
          acc[q * 4 + 1] += d[q].y;
          acc[q * 4 + 2] += d[q].z;
          acc[q * 4 + 3] += d[q].w;
        }
      } else if (s >= 0) {
#pragma unroll 1
        for (int j0 = 0; j0 < r; j0 += 4) {
          uint4 b[4][4];  // 4 rank rows x 32 columns, all loads in flight together
#pragma unroll
          for (int jj = 0; jj < 4; ++jj)
#pragma unroll
            for (int q = 0; q < 4; ++q)
              b[jj][q] = (j0 + jj < r && n + q * 8 < a.N)
                             ? __ldg(reinterpret_cast<const uint4*>(Bs + (size_t)(j0 + jj) * a.N +
                                                                    n + q * 8))
                             : make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const float vj = (j0 + jj < r) ? vrow[j0 + jj] : 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              acc[q * 8 + 0] = fmaf(vj, bf16_lo(b[jj][q].x), acc[q * 8 + 0]);
              acc[q * 8 + 1] = fmaf(vj, bf16_hi(b[jj][q].x), acc[q * 8 + 1]);
              acc[q * 8 + 2] = fmaf(vj, bf16_lo(b[jj][q].y), acc[q * 8 + 2]);
              acc[q * 8 + 3] = fmaf(vj, bf16_hi(b[jj][q].y), acc[q * 8 + 3]);
              acc[q * 8 + 4] = fmaf(vj, bf16_lo(b[jj][q].z), acc[q * 8 + 4]);
              acc[q * 8 + 5] = fmaf(vj, bf16_hi(b[jj][q].z), acc[q * 8 + 5]);
              acc[q * 8 + 6] = fmaf(vj, bf16_lo(b[jj][q].w), acc[q * 8 + 6]);
              acc[q * 8 + 7] = fmaf(vj, bf16_hi(b[jj][q].w), acc[q * 8 + 7]);
            }
          }
        }
      }
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
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, BN);
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

// Widest N tile that still gives at least one tile per SM, else the narrowest.
int gemm_tc_block_n(int M, int N, int num_sms) {
  const int mt = (M + kBM - 1) / kBM;
  const int cand[3] = {256, 128, 64};
  for (int i = 0; i < 3; ++i) {
    const int tiles = mt * ((N + cand[i] - 1) / cand[i]);
    if (tiles >= num_sms) return cand[i];
  }
  return 64;
}

static size_t tc_smem_bytes(int BN, int R, int stages) {
  const size_t stage = (size_t)kABytes + (size_t)BN * kBK * 2;
  return 1024 + stages * stage + (size_t)kBM * (R + 1) * 4 + (2 * stages + 2) * 8;
}

template <int BN>
static cudaError_t launch_tc(const GemmArgs& a, const CUtensorMap& tmap_x,
                             const CUtensorMap& tmap_w, cudaStream_t stream) {
  const size_t stage = (size_t)kABytes + (size_t)BN * kBK * 2;
  const size_t budget = 227 * 1024;
  int stages = 8;
  while (stages > 2 && tc_smem_bytes(BN, a.ex.R, stages) > budget) --stages;
  const size_t smem = tc_smem_bytes(BN, a.ex.R, stages);
  if (smem > budget) return cudaErrorInvalidConfiguration;
  (void)stage;
  static int limit = 0;
  cudaError_t e = ensure_smem_limit(gemm_tc_kernel<BN>, (int)smem, &limit);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3((a.M + kBM - 1) / kBM, (a.N + BN - 1) / BN);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<BN>, tmap_x, tmap_w, a, stages);
}

int gemm_tc_tile_index(int BN) { return BN == 256 ? 0 : (BN == 128 ? 1 : 2); }

cudaError_t launch_gemm_tc(const GemmArgs& a, const CUtensorMap* tmap_w3, cudaStream_t stream) {
  const int BN = gemm_tc_block_n(a.M, a.N, a.num_sms);
  CUtensorMap tmap_x;
  cudaError_t e = encode_tmap_bf16(&tmap_x, a.x, a.M, a.K, kBM);
  if (e != cudaSuccess) return e;
  const CUtensorMap& tw = tmap_w3[gemm_tc_tile_index(BN)];
  switch (BN) {
    case 256: return launch_tc<256>(a, tmap_x, tw, stream);
    case 128: return launch_tc<128>(a, tmap_x, tw, stream);
    default: return launch_tc<64>(a, tmap_x, tw, stream);
  }
}

}  // namespace lora
