// mla_simt.cu -- partial MLA decode on plain CUDA cores.
//
// A deliberately simple GPU kernel that computes exactly what
// mla_decode_partial does (see include/mla_decode.h), used to cross-check the
// tensor-core path on the device.  One warp owns one query row; a CTA owns 8
// consecutive rows of one (virtual request, split) and streams that split's
// tokens through shared memory 32 at a time, converted to fp32.
//
// Pages ([VRAM-KV], [K3-MLA], [K3-INTRO] as defined in the public header):
// the 576-d latent row (c_kv 512 + RoPE key 64), one per token and shared by
// every head; partial (O, LSE) per split; causal visibility among the q_len
// draft tokens.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "mla_internal.h"

namespace {

constexpr int kWarps = 8;                  // query rows per CTA
constexpr int kTile = 32;                  // tokens per shared-memory tile
constexpr int kPitch = MLA_ROW_DIM + 1;    // padded row: conflict-free columns
constexpr int kSmemBytes = (kTile * kPitch + kWarps * MLA_ROW_DIM) * 4;

struct SimtParams {
  const __nv_bfloat16* q_nope;
  const __nv_bfloat16* q_rope;
  const void* kv;
  const float* kv_scale;
  int kv_fp8;
  int64_t num_slots;
  const int32_t* r2t;
  int64_t r2t_stride;
  const int32_t* seq_lens;
  const int32_t* kv_limit;
  const int32_t* split_pages;  // [V, num_splits + 1] page boundaries or NULL
  int B, q_len, H, V, num_splits, row_blocks;
  float scale_log2;  // sm_scale * log2(e): scores are kept in base 2
  float* O_part;
  float* LSE_part;
  int* status;
};

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__device__ __forceinline__ float kv_value(const SimtParams& p, int64_t slot,
                                          int d) {
  if (p.kv_fp8) {
    __nv_fp8_e4m3 f;
    f.__x = static_cast<const uint8_t*>(p.kv)[slot * MLA_ROW_DIM + d];
    return float(f) * p.kv_scale[slot];
  }
  return __bfloat162float(
      static_cast<const __nv_bfloat16*>(p.kv)[slot * MLA_ROW_DIM + d]);
}

__global__ void __launch_bounds__(kWarps * 32)
    mla_partial_simt_kernel(const SimtParams p) {
  extern __shared__ float smem[];
  float* kt = smem;                          // [kTile][kPitch]
  float* xq = smem + kTile * kPitch;         // [kWarps][576]
  __shared__ int64_t tslot[kTile];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  int bid = blockIdx.x;
  const int rb = bid % p.row_blocks;
  bid /= p.row_blocks;
  const int v = bid % p.V;
  const int split = bid / p.V;
  const int b = v % p.B, shard = v / p.B;
  const int row_in_req = rb * kWarps + warp;  // i * H + h
  const bool row_ok = row_in_req < p.q_len * p.H;
  const int i = row_ok ? row_in_req / p.H : 0;

  int64_t L = p.seq_lens[v];
  if (L > p.r2t_stride) {
    if (threadIdx.x == 0 && p.status) atomicOr(p.status, MLA_STATUS_BAD_LENGTH);
    L = p.r2t_stride;
  }
  if (L < 0) L = 0;
  int64_t n = p.kv_limit ? (int64_t)p.kv_limit[(int64_t)v * p.q_len + i]
                         : L - p.q_len + 1 + i;
  n = n > L ? L : (n < 0 ? 0 : n);

  // This split's pages (the caller's table or the uniform deal).
  const int64_t P = (L + MLA_PAGE_SIZE - 1) / MLA_PAGE_SIZE;
  int64_t pg0, pg1;
  mla::split_page_range(
      p.split_pages ? p.split_pages + (int64_t)v * (p.num_splits + 1) : nullptr,
      p.num_splits, split, P, pg0, pg1);
  const int64_t t_lo = pg0 * MLA_PAGE_SIZE;
  const int64_t t_hi = min(pg1 * MLA_PAGE_SIZE, L);

  const int64_t qrow = (int64_t)b * p.q_len * p.H + row_in_req;
  for (int d = lane; d < MLA_ROW_DIM; d += 32) {
    float x = 0.f;
    if (row_ok)
      x = d < MLA_NOPE_DIM
              ? __bfloat162float(p.q_nope[qrow * MLA_NOPE_DIM + d])
              : __bfloat162float(p.q_rope[qrow * MLA_ROPE_DIM + d - MLA_NOPE_DIM]);
    xq[warp * MLA_ROW_DIM + d] = x;
  }

  float m = -INFINITY, l = 0.f;
  float o[MLA_VALUE_DIM / 32];
#pragma unroll
  for (int j = 0; j < MLA_VALUE_DIM / 32; ++j) o[j] = 0.f;

  for (int64_t t0 = t_lo; t0 < t_hi; t0 += kTile) {
    __syncthreads();
    if (threadIdx.x < kTile) {
      const int64_t t = t0 + threadIdx.x;
      int64_t slot = -1;
      if (t < t_hi) {
        const int64_t base =
            p.r2t[(int64_t)v * p.r2t_stride + (t - t % MLA_PAGE_SIZE)];
        if (base >= 0 && base % MLA_PAGE_SIZE == 0 &&
            base + MLA_PAGE_SIZE <= p.num_slots)
          slot = base + t % MLA_PAGE_SIZE;
        else if (p.status && t % MLA_PAGE_SIZE == 0)
          atomicOr(p.status, MLA_STATUS_BAD_SLOT);
      }
      tslot[threadIdx.x] = slot;
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < kTile * MLA_ROW_DIM; idx += blockDim.x) {
      const int tt = idx / MLA_ROW_DIM, d = idx % MLA_ROW_DIM;
      const int64_t slot = tslot[tt];
      kt[tt * kPitch + d] = slot >= 0 ? kv_value(p, slot, d) : 0.f;
    }
    __syncthreads();

    // Scores, one token per lane, in base 2.
    const int64_t t = t0 + lane;
    float s = -INFINITY;
    if (row_ok && t < t_hi && t < n) {
      float acc = 0.f;
      const float* xr = xq + warp * MLA_ROW_DIM;
      const float* kr = kt + lane * kPitch;
      for (int d = 0; d < MLA_ROW_DIM; ++d) acc = fmaf(xr[d], kr[d], acc);
      s = acc * p.scale_log2;
    }
    const float tile_max = warp_max(s);
    if (tile_max == -INFINITY) continue;  // warp-uniform
    const float m_new = fmaxf(m, tile_max);
    const float alpha = exp2f(m - m_new);  // 0 when m = -inf
    const float pr = s == -INFINITY ? 0.f : exp2f(s - m_new);
    l = l * alpha + warp_sum(pr);
#pragma unroll
    for (int j = 0; j < MLA_VALUE_DIM / 32; ++j) o[j] *= alpha;
    for (int tt = 0; tt < kTile; ++tt) {
      const float pt = __shfl_sync(0xffffffffu, pr, tt);
      if (pt == 0.f) continue;  // masked tokens never touch O
#pragma unroll
      for (int j = 0; j < MLA_VALUE_DIM / 32; ++j)
        o[j] = fmaf(pt, kt[tt * kPitch + lane + 32 * j], o[j]);
    }
    m = m_new;
  }

  if (!row_ok) return;
  const int64_t rows = (int64_t)p.B * p.q_len * p.H;
  const int64_t part = (int64_t)split * (p.V / p.B) + shard;
  const int64_t orow = part * rows + qrow;
  const bool empty = !(l > 0.f);
  const float inv_l = empty ? 0.f : 1.f / l;
#pragma unroll
  for (int j = 0; j < MLA_VALUE_DIM / 32; ++j)
    p.O_part[orow * MLA_VALUE_DIM + lane + 32 * j] = empty ? 0.f : o[j] * inv_l;
  if (lane == 0)
    p.LSE_part[orow] =
        empty ? -INFINITY : (m + log2f(l)) * 0.69314718055994531f;
}

}  // namespace

namespace mla {

int launch_simt(const DecodeArgs& a) {
  SimtParams p;
  p.q_nope = static_cast<const __nv_bfloat16*>(a.q_nope);
  p.q_rope = static_cast<const __nv_bfloat16*>(a.q_rope);
  p.kv = a.kv;
  p.kv_scale = a.kv_scale;
  p.kv_fp8 = a.kv_dtype == MLA_KV_FP8_E4M3;
  p.num_slots = a.num_slots;
  p.r2t = a.req_to_token;
  p.r2t_stride = a.r2t_stride;
  p.seq_lens = a.seq_lens;
  p.kv_limit = a.kv_limit;
  p.split_pages = a.split_pages;
  p.B = a.B;
  p.q_len = a.q_len;
  p.H = a.H;
  p.V = a.B * a.num_shards;
  p.num_splits = a.num_splits;
  p.row_blocks = (a.q_len * a.H + kWarps - 1) / kWarps;
  p.scale_log2 = a.sm_scale * 1.4426950408889634f;
  p.O_part = a.O_part;
  p.LSE_part = a.LSE_part;
  p.status = a.status;
  const int64_t grid = (int64_t)p.row_blocks * p.V * p.num_splits;
  if (grid > 0x7fffffff) return fail(MLA_ERR_INVALID_ARG, "grid too large");
  cudaError_t e = cudaFuncSetAttribute(
      mla_partial_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
      kSmemBytes);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(simt)");
  mla_partial_simt_kernel<<<(unsigned)grid, kWarps * 32, kSmemBytes,
                            a.stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch mla_partial_simt_kernel");
  return MLA_OK;
}

}  // namespace mla
