// e4m3_row.cuh -- quantisation of activation rows to e4m3 (the per-forward half of the e4m3
// base, fp8.cu) and of single values (the base weight's columns, once at creation).
//
// "Multi-LoRA Serving 与 Adapter 隔离", section on quantisation, TP and loading: an FP8 base
// with an FP16 LoRA; the quantised product and the LoRA term meet in the kernel's
// accumulator and epilogue.  The row's scale is max |x| / 448 in fp32 (1 for an all-zero
// row); each value is divided by it in fp32 (correctly rounded) and converted to e4m3,
// rounding to nearest even and saturating at +-448.
#pragma once

#include <cuda_fp8.h>

#include "lora_common.cuh"

namespace lora {

constexpr float kE4m3Max = 448.f;

__device__ __forceinline__ uint8_t to_e4m3(float v, float s) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(__fdiv_rn(v, s), __NV_SATFINITE, __NV_E4M3));
}

// Row scales whose quotients take the fast path below.
__device__ __forceinline__ bool fast_scale(float s) { return s >= 0x1p-110f && s <= 0x1p110f; }

// v / s for an element v of a row whose scale is s (|v| <= 448 s), given r = RN(1 / s).
// Fast path (fast_scale(s)): Markstein's correction (P. Markstein, "Computation of
// elementary functions on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1),
// 1990): q0 = RN(v r), the remainder v - q0 s exactly by one FMA, then q0 + rem r rounded
// once.  Over every bf16 v and every scale s = RN(a / 448) of a bf16 a >= |v| in that
// range, the e4m3 value of this quotient equals the e4m3 value of the correctly rounded
// one (checked exhaustively on the host); the quotients themselves differ only for
// subnormal v, whose quotients are far below e4m3's smallest step.  Otherwise the
// correctly rounded division.
__device__ __forceinline__ float row_quotient(float v, float s, float r, bool fast) {
  if (fast) {
    const float q0 = __fmul_rn(v, r);
    const float rem = __fmaf_rn(-q0, s, v);
    return __fmaf_rn(rem, r, q0);
  }
  return __fdiv_rn(v, s);
}

// e4m3 codes of a / s (low byte) and b / s (high byte) (row_quotient), one conversion
// instruction for the pair: round to nearest even, saturating at +-448, as to_e4m3.
__device__ __forceinline__ uint32_t to_e4m3x2(float a, float b, float s, float r, bool fast) {
  const float qa = row_quotient(a, s, r, fast), qb = row_quotient(b, s, r, fast);
  uint16_t c;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(c) : "f"(qb), "f"(qa));
  return c;
}

// The rows blockIdx.x, blockIdx.x + gridDim.x, ... (< T) quantised by the calling CTA of NT
// threads (warp, lane: the thread's warp and lane; wmax: NT / 32 floats of shared memory);
// returns the number of rows.  The CTA's warps are split between its rows, wpr warps a
// row, so that each thread's chunks of its row (chunks t, t + 32 wpr, ...) are at most
// HOLD where K allows: they are loaded together, held through the max and converted from
// registers; chunks past HOLD are read again in batches of 4.  Rows that do not fit one
// round go in further rounds.  Contains __syncthreads(): every thread of the CTA calls it.
template <int NT, int HOLD>
__device__ __forceinline__ int quantize_rows_e4m3_cta(const __nv_bfloat16* __restrict__ x, int T,
                                                      int K, uint8_t* __restrict__ xq,
                                                      float* __restrict__ sx, float* wmax,
                                                      int warp, int lane) {
  constexpr int kW = NT / 32;
  const int nr = (int)blockIdx.x < T ? (T - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  if (nr == 0) return 0;
  const int nv = K / 8;
  // warps per row: enough for HOLD chunks a thread (up to all kW), else kW / nr
  int wpr = 1;
  while (wpr < kW && (wpr * nr < kW || wpr * 32 * HOLD < nv)) wpr <<= 1;
  const int rpr = kW / wpr;  // rows a round
  const int sub = warp % wpr, t = sub * 32 + lane, ntr = wpr * 32;
  for (int q0 = 0; q0 < nr; q0 += rpr) {
    const int q = q0 + warp / wpr;
    const bool active = q < nr;
    const int row = (int)blockIdx.x + q * (int)gridDim.x;
    const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)(active ? row : 0) * K);
    uint4 hold[HOLD];
#pragma unroll
    for (int i = 0; i < HOLD; ++i) {
      const int e = t + i * ntr;
      hold[i] = active && e < nv ? __ldg(xr + e) : make_uint4(0u, 0u, 0u, 0u);
    }
    float m = 0.f;
    auto take_max = [&](const uint4& v) {
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[j])), fabsf(bf16_hi(w[j]))));
    };
#pragma unroll
    for (int i = 0; i < HOLD; ++i) take_max(hold[i]);
    for (int e0 = t + HOLD * ntr; active && e0 < nv; e0 += 4 * ntr) {
      uint4 v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int e = e0 + j * ntr;
        v[j] = e < nv ? __ldg(xr + e) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) take_max(v[j]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if (lane == 0) wmax[warp] = m;
    __syncthreads();
    float amax = 0.f;
    for (int w = warp - sub; w < warp - sub + wpr; ++w) amax = fmaxf(amax, wmax[w]);
    const float s = amax > 0.f ? __fdiv_rn(amax, kE4m3Max) : 1.f;
    const bool fast = fast_scale(s);
    const float rcp = fast ? __frcp_rn(s) : 0.f;
    if (active) {
      if (t == 0) sx[row] = s;
      uint2* qr = reinterpret_cast<uint2*>(xq + (size_t)row * K);
      auto convert = [&](const uint4& v) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t qq[2] = {0u, 0u};
#pragma unroll
        for (int i = 0; i < 4; ++i)
          qq[i >> 1] |= to_e4m3x2(bf16_lo(w[i]), bf16_hi(w[i]), s, rcp, fast) << (16 * (i & 1));
        return make_uint2(qq[0], qq[1]);
      };
#pragma unroll
      for (int i = 0; i < HOLD; ++i) {
        const int e = t + i * ntr;
        if (e < nv) qr[e] = convert(hold[i]);
      }
      for (int e0 = t + HOLD * ntr; e0 < nv; e0 += 4 * ntr) {
        uint4 v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int e = e0 + j * ntr;
          v[j] = e < nv ? __ldg(xr + e) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (e0 + j * ntr < nv) qr[e0 + j * ntr] = convert(v[j]);
      }
    }
    __syncthreads();  // wmax is rewritten by the next round
  }
  return nr;
}

// Publish `rows` rows quantised by the calling CTA: after a CTA barrier (every thread's
// stores then precede it), thread 0 adds the count to *ready with release semantics at GPU
// scope, which carries those stores to any thread that acquires the count (the GEMM
// reading xq waits for it to reach its row count).  Called by every thread of the CTA.
__device__ __forceinline__ void publish_rows(int32_t* ready, int rows) {
  __syncthreads();
  if (threadIdx.x == 0 && rows > 0)
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(ready), "r"(rows) : "memory");
}

}  // namespace lora
