// mla_kv_write.cu -- writing new tokens' latent rows into the paged KV pool
// ([VRAM-KV], [VRAM-POOL] in include/mla_decode.h: one 576-element row per
// token at its req_to_token slot), as BF16 or as the FP8 E4M3 format with one
// fp32 scale per token.
//
// HBM-bound streaming: one warp per row; each lane moves 16-byte chunks of
// the bf16 row (72 chunks).  FP8: the row's largest |x| by warp reduction,
// scale = fl32(amax / 448) and codes = E4M3(fl32(x / scale)) with IEEE
// round-to-nearest divisions and the round-to-nearest-even, saturating
// E4M3 conversion; an all-zero row gets scale 0 and codes 0.  A slot outside
// the pool is skipped and reported (MLA_STATUS_BAD_SLOT).
#include <cuda_bf16.h>

#include "mla_internal.h"

namespace {

constexpr int kWarpsPerBlock = 8;
constexpr int kChunks = MLA_ROW_DIM * 2 / 16;  // 72 bf16 chunks of 16 bytes
constexpr uint32_t kAll = 0xffffffffu;

// Two binary32 values -> their E4M3 codes (round to nearest even, saturated
// to +-448), lower byte = a.
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  uint16_t h;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %2, %1;" : "=h"(h) : "f"(a), "f"(b));
  return h;
}

__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    mla_kv_write_kernel(const uint4* __restrict__ rows, int64_t n,
                        const int32_t* __restrict__ slots, uint8_t* kv,
                        int fp8, float* kv_scale, int64_t num_slots,
                        int* status) {
  const int lane = threadIdx.x % 32;
  const int64_t r = (int64_t)blockIdx.x * kWarpsPerBlock + threadIdx.x / 32;
  if (r >= n) return;
  const int32_t slot = slots[r];
  if (slot < 0 || (int64_t)slot >= num_slots) {
    if (lane == 0 && status) atomicOr(status, MLA_STATUS_BAD_SLOT);
    return;
  }
  const uint4* src = rows + r * kChunks;
  uint4 x[3];
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    const int c = lane + 32 * k;
    x[k] = c < kChunks ? src[c] : make_uint4(0, 0, 0, 0);
  }
  if (!fp8) {
    uint4* dst = reinterpret_cast<uint4*>(kv + (int64_t)slot * MLA_ROW_DIM * 2);
#pragma unroll
    for (int k = 0; k < 3; ++k)
      if (lane + 32 * k < kChunks) dst[lane + 32 * k] = x[k];
    return;
  }
  // bf16 pairs -> binary32 (exact)
  float v[3][8];
  float amax = 0.f;
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    const uint32_t w[4] = {x[k].x, x[k].y, x[k].z, x[k].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      v[k][2 * e] = __uint_as_float(w[e] << 16);
      v[k][2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
      amax = fmaxf(amax, fmaxf(fabsf(v[k][2 * e]), fabsf(v[k][2 * e + 1])));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kAll, amax, o));
  const float scale = __fdiv_rn(amax, 448.0f);
  uint2* dst = reinterpret_cast<uint2*>(kv + (int64_t)slot * MLA_ROW_DIM);
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    const int c = lane + 32 * k;  // 8 elements -> 8 code bytes
    if (c >= kChunks) continue;
    uint32_t p[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      p[e] = scale == 0.f ? 0u
                          : e4m3x2(__fdiv_rn(v[k][2 * e], scale),
                                   __fdiv_rn(v[k][2 * e + 1], scale));
    dst[c] = make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16));
  }
  if (lane == 0) kv_scale[slot] = scale;
}

}  // namespace

using namespace mla;

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
  const int64_t blocks = (n + kWarpsPerBlock - 1) / kWarpsPerBlock;
  if (blocks > 0x7fffffff) return fail(MLA_ERR_INVALID_ARG, "too many rows");
  mla_kv_write_kernel<<<(unsigned)blocks, kWarpsPerBlock * 32, 0,
                        (cudaStream_t)stream>>>(
      static_cast<const uint4*>(rows), n, slots, static_cast<uint8_t*>(kv_pages),
      kv_dtype == MLA_KV_FP8_E4M3, kv_scale, num_slots, status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch mla_kv_write_kernel");
  return MLA_OK;
}
