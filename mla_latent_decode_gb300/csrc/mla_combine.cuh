// mla_combine.cuh -- the LSE-weighted merge of one output row ([K3-MLA],
// dcp_lse_combine), shared by the standalone combine kernel and the fused
// epilogue of the partial-decode kernels.
//
// Row `row` of `rows` over P parts (part j at O_part + j*rows*512,
// LSE_part + j*rows): M = max_j LSE_j; w_j = exp(LSE_j - M) (parts with
// LSE = -inf have weight 0 and are never read); out = sum_j w_j O_j / sum_j
// w_j in bf16 (round to nearest even); lse = M + ln sum_j w_j.  A part whose
// LSE is NaN (its range held a NaN score the row sees) makes the whole row
// NaN, out and lse, as the unsplit definition would.  One warp per
// row: lane j reads LSE_j (all weights in one round trip, reduced with
// shuffles), then each lane owns four float4 columns of every part
// (coalesced 512-byte loads), two parts' loads in flight at a time, parts
// accumulated in order; for few rows several warps share a row (below).
// kCoherent: the parts were written by other CTAs of the running kernel, so
// they are read through L2 only (no read-only or L1 copy that could be
// stale); otherwise the read-only path.
#pragma once

#include <cuda_bf16.h>

#include <cstdint>

#include "../../include/mla_decode.h"

namespace mla {

template <bool kCoherent>
__device__ __forceinline__ float load_part(const float* p) {
  return kCoherent ? __ldcg(p) : __ldg(p);
}

template <bool kCoherent>
__device__ __forceinline__ float4 load_part4(const float4* p) {
  return kCoherent ? __ldcg(p) : __ldg(p);
}

// Four consecutive values of a part row as fp32: one 16-byte load of fp32
// parts or one 8-byte load of bf16 parts (widened exactly).  `c4` counts
// groups of four values from `row`.
template <bool kCoherent>
__device__ __forceinline__ float4 load_four(const float* row, int c4) {
  return load_part4<kCoherent>(reinterpret_cast<const float4*>(row) + c4);
}
template <bool kCoherent>
__device__ __forceinline__ float4 load_four(const __nv_bfloat16* row, int c4) {
  const uint2* q = reinterpret_cast<const uint2*>(row) + c4;
  const uint2 u = kCoherent ? __ldcg(q) : __ldg(q);
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                     __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
}

// kWs warps share a row: warp `slice` of them owns value columns
// [slice * 512 / kWs, +512 / kWs), each lane kF4 = 4 / kWs float4 columns of
// every part, with kPar = 8 / kF4 parts' loads in flight at a time (eight
// float4 loads per lane whatever kWs).  Every warp of the row computes the
// weights itself; slice 0 writes lse_out.
template <bool kCoherent, int kWs = 1, typename PartT = float>
__device__ __forceinline__ void combine_row(const PartT* __restrict__ O_part,
                                            const float* __restrict__ LSE_part,
                                            int P, int64_t rows, int64_t row,
                                            __nv_bfloat16* __restrict__ out,
                                            float* __restrict__ lse_out,
                                            int lane, int slice = 0) {
  static_assert(kWs == 1 || kWs == 2 || kWs == 4, "warps per row");
  constexpr int kF4 = 4 / kWs;   // float4 columns per lane and part
  constexpr int kPar = 8 / kF4;  // parts in flight
  constexpr uint32_t kAll = 0xffffffffu;
  // M = max_j LSE_j: lane j % 32 reads LSE_j (one round trip per 32 parts)
  float M = -INFINITY;
  bool nan = false;
  for (int j0 = 0; j0 < P; j0 += 32)
    if (j0 + lane < P) {
      const float l = load_part<kCoherent>(LSE_part + (int64_t)(j0 + lane) * rows + row);
      nan |= l != l;
      M = fmaxf(M, l);
    }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kAll, M, o));
  // float4 column of this lane's k-th slot
  auto col = [&](int k) { return slice * (128 / kWs) + lane + 32 * k; };
  __nv_bfloat162* dst =
      reinterpret_cast<__nv_bfloat162*>(out + row * MLA_VALUE_DIM);
  if (__any_sync(kAll, nan)) {
    const __nv_bfloat162 qnan = __float2bfloat162_rn(__int_as_float(0x7fc00000));
#pragma unroll
    for (int k = 0; k < kF4; ++k) {
      dst[2 * col(k)] = qnan;
      dst[2 * col(k) + 1] = qnan;
    }
    if (lse_out && slice == 0 && lane == 0) lse_out[row] = __int_as_float(0x7fc00000);
    return;
  }

  float4 acc[kF4];
#pragma unroll
  for (int k = 0; k < kF4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  float W = 0.f;  // lane-partial sum of the weights, reduced below
  if (M != -INFINITY) {
    for (int j0 = 0; j0 < P; j0 += 32) {
      const int n = min(32, P - j0);
      float wl = 0.f;  // weight of part j0 + lane (0 for an empty part)
      if (lane < n) {
        const float lj = load_part<kCoherent>(LSE_part + (int64_t)(j0 + lane) * rows + row);
        wl = lj == -INFINITY ? 0.f : expf(lj - M);
      }
      W += wl;
      // parts in order, kPar at a time so their loads are in flight
      // together; an empty part (weight 0) is never read
      for (int t = 0; t < n; t += kPar) {
        float w[kPar];
        float4 x[kPar][kF4];
#pragma unroll
        for (int q = 0; q < kPar; ++q) {
          w[q] = t + q < n ? __shfl_sync(kAll, wl, t + q) : 0.f;
          const PartT* src =
              O_part + ((int64_t)(j0 + t + q) * rows + row) * MLA_VALUE_DIM;
#pragma unroll
          for (int k = 0; k < kF4; ++k)
            x[q][k] = w[q] != 0.f ? load_four<kCoherent>(src, col(k))
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int q = 0; q < kPar; ++q) {
          if (w[q] == 0.f) continue;
#pragma unroll
          for (int k = 0; k < kF4; ++k) {
            acc[k].x = fmaf(w[q], x[q][k].x, acc[k].x);
            acc[k].y = fmaf(w[q], x[q][k].y, acc[k].y);
            acc[k].z = fmaf(w[q], x[q][k].z, acc[k].z);
            acc[k].w = fmaf(w[q], x[q][k].w, acc[k].w);
          }
        }
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) W += __shfl_xor_sync(kAll, W, o);
  const float inv = W > 0.f ? 1.f / W : 0.f;
#pragma unroll
  for (int k = 0; k < kF4; ++k) {
    const int c = 2 * col(k);  // bf16x2 index of float4 column col(k)
    dst[c] = __floats2bfloat162_rn(acc[k].x * inv, acc[k].y * inv);
    dst[c + 1] = __floats2bfloat162_rn(acc[k].z * inv, acc[k].w * inv);
  }
  if (lse_out && slice == 0 && lane == 0)
    lse_out[row] = W > 0.f ? M + logf(W) : -INFINITY;
}

}  // namespace mla
