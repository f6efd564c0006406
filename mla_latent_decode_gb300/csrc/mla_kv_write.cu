// mla_kv_write.cu -- writing new tokens' latent rows into the paged KV pool
// ([VRAM-KV], [VRAM-POOL] in include/mla_decode.h: one 576-element row per
// token at its req_to_token slot), as BF16 or as the FP8 E4M3 format with one
// fp32 scale per token.
//
// HBM-bound streaming: a warp per row at a time; each lane moves 16-byte
// chunks of the bf16 row (72 chunks).  FP8: the row's largest |x| by warp reduction,
// scale = fl32(amax / 448) and codes = E4M3(fl32(x / scale)) with IEEE
// round-to-nearest divisions and the round-to-nearest-even, saturating
// E4M3 conversion; an all-zero row gets scale 0 and codes 0.  A slot outside
// the pool is skipped and reported (MLA_STATUS_BAD_SLOT).
// The 576 quotients of a row share their divisor, so each is formed from one
// correctly rounded reciprocal of the scale and one Markstein correction
// (quotient_rn below) instead of a full IEEE division: the same binary32
// values wherever they decide a code, checked exhaustively over every bf16
// element and every bf16 row maximum by mla_debug_quotients.
#include <cuda_bf16.h>

#include <algorithm>

#include "mla_internal.h"

namespace {

constexpr int kWarpsPerBlock = 8;
constexpr int kChunks = MLA_ROW_DIM * 2 / 16;  // 72 bf16 chunks of 16 bytes
constexpr uint32_t kAll = 0xffffffffu;

// The divisor range of the reciprocal path: outside it (rows whose largest
// |x| is under about 2^-81, or infinite) every element divides directly.
constexpr float kQuotMinScale = 0x1p-90f;
constexpr float kQuotMaxScale = 0x1p+120f;

__device__ __forceinline__ bool reciprocal_path(float b) {
  return b >= kQuotMinScale && b <= kQuotMaxScale;
}

// RN(a / b) for b in [2^-90, 2^120] and |a| <= 448 b a bf16 value, from
// y = RN(1 / b): q = RN(|a| y), then one Markstein correction q + RN(|a| -
// b q) y (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990), rounded once by the
// FMA; the sign goes back at the end (rounding to nearest is symmetric, and
// a = -0 gives -0).  For these operands the result equals the IEEE division
// bit for bit wherever |a / b| >= 2^-11 and gives the same E4M3 code
// everywhere: mla_debug_quotients checks every bf16 element against every
// bf16 row maximum.  (Without the correction about 6e4 of those codes
// differ.)
__device__ __forceinline__ float quotient_rn(float a, float b, float y) {
  const float m = fabsf(a);
  const float q = __fmul_rn(m, y);
  return copysignf(__fmaf_rn(__fmaf_rn(-q, b, m), y, q), a);
}

// Two binary32 values -> their E4M3 codes (round to nearest even, saturated
// to +-448), lower byte = a.
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  uint16_t h;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %2, %1;" : "=h"(h) : "f"(a), "f"(b));
  return h;
}

// One row (three 16-byte chunks per lane, loaded) to its slot as E4M3 codes
// and a scale.
__device__ __forceinline__ void write_row(const uint4 (&x)[3], int32_t slot,
                                          uint8_t* kv, float* kv_scale,
                                          int64_t num_slots, int* status,
                                          int lane) {
  if (slot < 0 || (int64_t)slot >= num_slots) {
    if (lane == 0 && status) atomicOr(status, MLA_STATUS_BAD_SLOT);
    return;
  }
  // bf16 -> binary32 is exact: element 2e of a word is its low half
  auto val = [&](int k, int i) -> float {
    const uint32_t w = i < 2 ? (i == 0 ? x[k].x : x[k].y) : (i == 2 ? x[k].z : x[k].w);
    return __uint_as_float(w << 16);
  };
  auto val_hi = [&](int k, int i) -> float {
    const uint32_t w = i < 2 ? (i == 0 ? x[k].x : x[k].y) : (i == 2 ? x[k].z : x[k].w);
    return __uint_as_float(w & 0xFFFF0000u);
  };
  float amax = 0.f;
#pragma unroll
  for (int k = 0; k < 3; ++k)
#pragma unroll
    for (int e = 0; e < 4; ++e)
      amax = fmaxf(amax, fmaxf(fabsf(val(k, e)), fabsf(val_hi(k, e))));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kAll, amax, o));
  const float scale = __fdiv_rn(amax, 448.0f);
  uint2* dst = reinterpret_cast<uint2*>(kv + (int64_t)slot * MLA_ROW_DIM);
  if (reciprocal_path(scale)) {
    const float rcp = __frcp_rn(scale);
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      const int c = lane + 32 * k;  // 8 elements -> 8 code bytes
      if (c >= kChunks) continue;
      uint32_t p[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        p[e] = e4m3x2(quotient_rn(val(k, e), scale, rcp),
                      quotient_rn(val_hi(k, e), scale, rcp));
      dst[c] = make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16));
    }
  } else {
    for (int k = 0; k < 3; ++k) {
      const int c = lane + 32 * k;
      if (c >= kChunks) continue;
      uint32_t p[4];
      for (int e = 0; e < 4; ++e)
        p[e] = scale == 0.f ? 0u
                            : e4m3x2(__fdiv_rn(val(k, e), scale),
                                     __fdiv_rn(val_hi(k, e), scale));
      dst[c] = make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16));
    }
  }
  if (lane == 0) kv_scale[slot] = scale;
}

// BF16: a plain copy of each row to its slot.  A warp takes two rows and
// loads both (and their slots) before it stores either.
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    mla_kv_copy_kernel(const uint4* __restrict__ rows, int64_t n,
                       const int32_t* __restrict__ slots, uint8_t* kv,
                       int64_t num_slots, int* status) {
  constexpr int kRows = 2;
  const int lane = threadIdx.x % 32;
  const int64_t r0 =
      ((int64_t)blockIdx.x * kWarpsPerBlock + threadIdx.x / 32) * kRows;
  if (r0 >= n) return;
  uint4 x[kRows][3];
  int32_t slot[kRows];
#pragma unroll
  for (int i = 0; i < kRows; ++i) {
    const bool live = r0 + i < n;
    slot[i] = live ? slots[r0 + i] : -1;
    const uint4* src = rows + (r0 + i) * kChunks;
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      const int c = lane + 32 * k;
      x[i][k] = live && c < kChunks ? __ldcs(src + c) : make_uint4(0, 0, 0, 0);
    }
  }
#pragma unroll
  for (int i = 0; i < kRows; ++i) {
    if (r0 + i >= n) break;
    if (slot[i] < 0 || (int64_t)slot[i] >= num_slots) {
      if (lane == 0 && status) atomicOr(status, MLA_STATUS_BAD_SLOT);
      continue;
    }
    uint4* dst = reinterpret_cast<uint4*>(kv + (int64_t)slot[i] * MLA_ROW_DIM * 2);
#pragma unroll
    for (int k = 0; k < 3; ++k)
      if (lane + 32 * k < kChunks) dst[lane + 32 * k] = x[i][k];
  }
}

// FP8: each warp takes rows r, r + W, r + 2W, ...
// (W warps in the grid) and loads the next row's chunks and slot before it
// converts and stores the current one, so the loads of one row overlap the
// arithmetic and stores of the previous.
__device__ __forceinline__ void load_row(const uint4* __restrict__ rows,
                                         const int32_t* __restrict__ slots,
                                         int64_t r, int lane, uint4 (&x)[3],
                                         int32_t& slot) {
  slot = slots[r];
  const uint4* src = rows + r * kChunks;
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    const int c = lane + 32 * k;
    x[k] = c < kChunks ? __ldcs(src + c) : make_uint4(0, 0, 0, 0);
  }
}

__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    mla_kv_write_kernel(const uint4* __restrict__ rows, int64_t n,
                        const int32_t* __restrict__ slots, uint8_t* kv,
                        float* kv_scale, int64_t num_slots, int* status) {
  const int lane = threadIdx.x % 32;
  const int64_t W = (int64_t)gridDim.x * kWarpsPerBlock;
  int64_t r = (int64_t)blockIdx.x * kWarpsPerBlock + threadIdx.x / 32;
  if (r >= n) return;
  uint4 x[3];
  int32_t slot;
  load_row(rows, slots, r, lane, x, slot);
  for (;;) {
    const int64_t rn = r + W;
    uint4 xn[3] = {};
    int32_t sn = -1;
    if (rn < n) load_row(rows, slots, rn, lane, xn, sn);
    write_row(x, slot, kv, kv_scale, num_slots, status, lane);
    if (rn >= n) break;
    r = rn;
#pragma unroll
    for (int k = 0; k < 3; ++k) x[k] = xn[k];
    slot = sn;
  }
}

// Exhaustive check of quotient_rn against the IEEE division: block k takes
// the row maximum with bf16 bits k + 1 (every positive finite bf16 value),
// its scale fl32(amax / 448) and every bf16 element a with |a| <= amax (both
// signs, zeros and subnormals).  Counted: quotients of magnitude 2^-11 or
// more whose binary32 bits differ, and E4M3 codes that differ.
__global__ void __launch_bounds__(256)
    mla_quotient_check_kernel(unsigned long long* bit_mismatches,
                              unsigned long long* code_mismatches) {
  const float amax = __uint_as_float((blockIdx.x + 1u) << 16);
  const float scale = __fdiv_rn(amax, 448.0f);
  if (!reciprocal_path(scale)) return;  // these rows divide directly
  const float rcp = __frcp_rn(scale);
  unsigned long long nb = 0, nc = 0;
  for (uint32_t bits = threadIdx.x; bits < 65536u; bits += blockDim.x) {
    const float a = __uint_as_float(bits << 16);
    if (!(fabsf(a) <= amax)) continue;  // larger, or not finite
    const float ref = __fdiv_rn(a, scale);
    const float got = quotient_rn(a, scale, rcp);
    if (fabsf(ref) >= 0x1p-11f && __float_as_uint(got) != __float_as_uint(ref)) ++nb;
    if (e4m3x2(got, 0.f) != e4m3x2(ref, 0.f)) ++nc;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    nb += __shfl_xor_sync(kAll, nb, o);
    nc += __shfl_xor_sync(kAll, nc, o);
  }
  if (threadIdx.x % 32 == 0 && (nb | nc)) {
    atomicAdd(bit_mismatches, nb);
    atomicAdd(code_mismatches, nc);
  }
}

}  // namespace

using namespace mla;

extern "C" int mla_debug_quotients(uint64_t* bit_mismatches,
                                   uint64_t* code_mismatches,
                                   mla_stream_t stream) {
  if (!bit_mismatches || !code_mismatches)
    return fail(MLA_ERR_INVALID_ARG, "both counters are required");
  if (!aligned(bit_mismatches, 8) || !aligned(code_mismatches, 8))
    return fail(MLA_ERR_MISALIGNED, "counters need 8-B alignment");
  // every positive finite bf16 value as the row maximum: bits 0x0001..0x7F7F
  mla_quotient_check_kernel<<<0x7F7F, 256, 0, (cudaStream_t)stream>>>(
      reinterpret_cast<unsigned long long*>(bit_mismatches),
      reinterpret_cast<unsigned long long*>(code_mismatches));
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch mla_quotient_check_kernel");
  return MLA_OK;
}

extern "C" int mla_kv_write(const void* rows, int64_t n, const int32_t* slots,
                            void* kv_pages, mla_kv_dtype kv_dtype,
                            float* kv_scale, int64_t num_slots, int* status,
                            mla_stream_t stream) {
  if (n < 0) return fail(MLA_ERR_INVALID_ARG, "n = %lld < 0", (long long)n);
  if (n == 0) return MLA_OK;
  if (!rows || !slots || !kv_pages)
    return fail(MLA_ERR_INVALID_ARG, "rows, slots and kv_pages are required");
  if (kv_dtype != MLA_KV_BF16 && kv_dtype != MLA_KV_FP8_E4M3)
    return fail(MLA_ERR_INVALID_ARG, "unknown kv_dtype %d", (int)kv_dtype);
  if (kv_dtype == MLA_KV_FP8_E4M3 && !kv_scale)
    return fail(MLA_ERR_INVALID_ARG, "FP8 KV needs kv_scale");
  if (num_slots < 1)
    return fail(MLA_ERR_INVALID_ARG, "num_slots %lld < 1", (long long)num_slots);
  if (!aligned(rows, 16) || !aligned(kv_pages, 16) || !aligned(slots, 4) ||
      (kv_scale && !aligned(kv_scale, 4)) || (status && !aligned(status, 4)))
    return fail(MLA_ERR_MISALIGNED, "rows and kv_pages need 16-B alignment, the "
                "other arrays 4-B");
  const uint4* src = static_cast<const uint4*>(rows);
  uint8_t* dst = static_cast<uint8_t*>(kv_pages);
  cudaError_t e = cudaSuccess;
  if (kv_dtype == MLA_KV_BF16) {
    const int64_t per_block = 2 * kWarpsPerBlock;
    const int64_t blocks = (n + per_block - 1) / per_block;
    if (blocks > 0x7fffffff) return fail(MLA_ERR_INVALID_ARG, "too many rows");
    mla_kv_copy_kernel<<<(unsigned)blocks, kWarpsPerBlock * 32, 0,
                         (cudaStream_t)stream>>>(src, n, slots, dst, num_slots,
                                                 status);
  } else {
    // A resident grid whose warps load the next row while they convert one.
    int dev = 0, sms = 0, per_sm = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
      e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          &per_sm, mla_kv_write_kernel, kWarpsPerBlock * 32, 0);
    if (e != cudaSuccess) return cuda_fail(e, "mla_kv_write: device query");
    const int64_t need = (n + kWarpsPerBlock - 1) / kWarpsPerBlock;
    const int64_t blocks =
        std::min<int64_t>(need, (int64_t)sms * std::max(per_sm, 1));
    mla_kv_write_kernel<<<(unsigned)blocks, kWarpsPerBlock * 32, 0,
                          (cudaStream_t)stream>>>(src, n, slots, dst, kv_scale,
                                                  num_slots, status);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch mla_kv_write_kernel");
  return MLA_OK;
}
