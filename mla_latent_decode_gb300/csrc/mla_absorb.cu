// mla_absorb.cu -- the per-head projections on either side of the absorbed
// decode ([K3-MEM] in include/mla_decode.h: w_kc is 96 x 128 x 512 bf16 and
// the absorbed query is 512-d; kv_b_proj is absorbed into w_kc / w_vc):
//   query absorption   q_abs[m, h, :512] = q_nope[m, h, :128] . w_kc[h]
//   output projection  o_v[m, h, :128]  = o_lat[m, h, :512] . w_vc[h]
// (m = b * q_len + i).  Both are per-head batched GEMMs with few rows
// (B * q_len) and a weight slice per head, so the weights' HBM bytes bound
// them; the products run on tcgen05 tensor cores.
//
// One CTA per (head h, tile of 128 rows, chunk of NC output columns), 4
// warps: splitting N (4 chunks of 128 for the query absorption, 2 of 64 for
// the output projection) streams each head's weight slice through several
// SMs at once; these launches are latency-bound, not bandwidth-bound.  Warp 0 lane 0 loads K
// in chunks of 128 by TMA -- the activation rows of head h through a 3-D
// tensor map (64 K x 1 head x 128 rows boxes, K-major, 128-byte swizzle,
// rows past M read as zeros) and the weight slice in 64 x 64 boxes (rows =
// K, 128-byte rows of N: MN-major) -- and issues M = 128, N <= 256, K = 16
// bf16 MMAs into TMEM; the four warps then round their 32 rows to bf16.
// Launches use programmatic dependent launch: a CTA lets the stream's next
// kernel start at once and, before it waits for the kernels it depends on,
// has its whole weight slice prefetched into L2 (a prefetch reads nothing
// into the CTA, so weights written by those kernels are still read after
// they finish: L2 holds the current data).  Every wait is bounded
// (ptx_sm103.cuh); a timeout sets MLA_STATUS_WAIT_TIMEOUT.
#include <cuda_bf16.h>

#include "mla_tma.cuh"
#include "ptx_sm103.cuh"

namespace mla {
namespace {

using namespace ptx;

constexpr int kRowsPerCta = 128;
constexpr int kChunkK = 128;       // K per ring stage
constexpr int kBoxA = 128 * 128;   // 64 K x 128 rows bf16 = 16 KB
constexpr int kBoxB = 64 * 128;    // 64 K rows x 64 N bf16 = 8 KB

template <int K, int N, int NC>
struct HeadGemm {
  static constexpr int kABytes = (kChunkK / 64) * kBoxA;             // 32 KB
  static constexpr int kBBytes = (kChunkK / 64) * (NC / 64) * kBoxB;  // 64|16 KB
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kChunks = K / kChunkK;
  static constexpr int kStages = kChunks < 2 ? 1 : 2;
  static constexpr int kMmaN = NC < 256 ? NC : 256;
  static constexpr int kTmemCols = NC < 32 ? 32 : NC;
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024 + 256;
  static_assert(K % kChunkK == 0 && N % NC == 0 && NC % 64 == 0, "shape");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

template <int K, int N, int NC>
__global__ void __launch_bounds__(128, 1)
    mla_head_gemm_kernel(const __grid_constant__ CUtensorMap a_map,
                         const __grid_constant__ CUtensorMap w_map,
                         __nv_bfloat16* __restrict__ out, int M, int H,
                         int* status) {
  using G = HeadGemm<K, N, NC>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(base + G::kStages * G::kStageBytes);
  uint64_t* empty = full + G::kStages;
  uint64_t* done = empty + G::kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int h = blockIdx.y;
  const int m0 = blockIdx.x * kRowsPerCta;
  const int n_base = blockIdx.z * NC;
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < G::kStages; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), 1);
    }
    mbar_init(smem_u32(done), 1);
    fence_mbar_init();
    prefetch_tmap(&a_map);
    prefetch_tmap(&w_map);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), G::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  griddep_launch_dependents();
  bool ok = true;
  if (threadIdx.x == 0) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, G::kMmaN, false, true);
    // The weight slice into L2 while earlier kernels finish.
    for (int k0 = 0; k0 < K; k0 += 64)
      for (int nb = 0; nb < NC / 64; ++nb)
        tma_prefetch_3d(&w_map, n_base + nb * 64, k0, h);
    griddep_wait();
    for (int c = 0; c < G::kChunks && ok; ++c) {
      const int st = c % G::kStages;
      const uint32_t use = c / G::kStages;
      if (use > 0 && !mbar_wait(smem_u32(&empty[st]), (use - 1) & 1, abort_flag)) {
        ok = false;
        break;
      }
      uint8_t* sa = base + st * G::kStageBytes;
      uint8_t* sb = sa + G::kABytes;
      const uint32_t bar = smem_u32(&full[st]);
      mbar_arrive_expect_tx(bar, G::kStageBytes);
      for (int kb = 0; kb < kChunkK / 64; ++kb) {
        const int k0 = c * kChunkK + kb * 64;
        for (int nb = 0; nb < NC / 64; ++nb)
          tma_load_3d(smem_u32(sb + (kb * (NC / 64) + nb) * kBoxB), &w_map, bar,
                      n_base + nb * 64, k0, h);
        tma_load_3d(smem_u32(sa + kb * kBoxA), &a_map, bar, k0, h, m0);
      }
      if (!mbar_wait(bar, use & 1, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // A: K-major, next 16 K +32 B (2 units); B: MN-major, the next 64 N
      // one box (8 KB, LBO) on, the next 8 K rows 1 KB (SBO) on, the next 16
      // K rows 2 KB (128 units) on, the next 64 K rows N/64 boxes on.
      for (int kb = 0; kb < kChunkK / 64; ++kb) {
        const uint64_t a = sdesc_sw128(smem_u32(sa + kb * kBoxA), 16, 1024);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
          for (int n0 = 0; n0 < NC; n0 += G::kMmaN) {
            const uint64_t b = sdesc_sw128(
                smem_u32(sb + (kb * (NC / 64) + n0 / 64) * kBoxB), kBoxB, 1024);
            mma_ss(tmem + n0, a + 2 * ks, b + 128 * ks, idesc,
                   (c | kb | ks) ? 1u : 0u);
          }
        }
      }
      mma_commit(smem_u32(&empty[st]));
    }
    if (ok) mma_commit(smem_u32(done));
    if (!ok) {
      *abort_flag = 1;
      if (status) atomicOr(status, MLA_STATUS_WAIT_TIMEOUT);
      mbar_arrive(smem_u32(done));
    }
  }
  __syncwarp();
  // Epilogue: warp w's TMEM lanes are rows 32w..32w+31 of the tile.
  if (!mbar_wait(smem_u32(done), 0, abort_flag)) {
    if (lane == 0 && status) atomicOr(status, MLA_STATUS_WAIT_TIMEOUT);
  } else if (!*reinterpret_cast<volatile int*>(abort_flag)) {
    tc_fence_after();
    const int m = m0 + warp * 32 + lane;
    const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16);
#pragma unroll 1
    for (int c0 = 0; c0 < NC; c0 += 32) {
      uint32_t v[32];
      tmem_ld32(taddr + c0, v);
      tmem_wait_ld();
      if (m < M) {
        uint4* dst = reinterpret_cast<uint4*>(out + ((int64_t)m * H + h) * N +
                                              n_base + c0);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            __nv_bfloat162 b2 = __floats2bfloat162_rn(
                __uint_as_float(v[8 * q + 2 * e]), __uint_as_float(v[8 * q + 2 * e + 1]));
            w[e] = *reinterpret_cast<uint32_t*>(&b2);
          }
          dst[q] = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, G::kTmemCols);
}

template <int K, int N, int NC>
int launch_head_gemm(const void* in, const void* w, void* out, int M, int H,
                     int* status, cudaStream_t stream, const char* name) {
  using G = HeadGemm<K, N, NC>;
  if (!in || !w || !out)
    return fail(MLA_ERR_INVALID_ARG, "%s: input, weights and output are required", name);
  if (M < 1 || H < 1 || H > 65535)
    return fail(MLA_ERR_INVALID_ARG, "%s: M=%d H=%d out of range", name, M, H);
  if (!aligned(in, 16) || !aligned(w, 16) || !aligned(out, 16) ||
      (status && !aligned(status, 4)))
    return fail(MLA_ERR_MISALIGNED, "%s: arrays need 16-B alignment", name);
  CUtensorMap a_map, w_map;
  {
    const uint64_t dims[3] = {(uint64_t)K, (uint64_t)H, (uint64_t)M};
    const uint64_t strides[2] = {(uint64_t)K * 2, (uint64_t)H * K * 2};
    const uint32_t box[3] = {64, 1, kRowsPerCta};
    int rc = make_tensor_map_bf16_3d(&a_map, in, dims, strides, box);
    if (rc != MLA_OK) return rc;
  }
  {
    const uint64_t dims[3] = {(uint64_t)N, (uint64_t)K, (uint64_t)H};
    const uint64_t strides[2] = {(uint64_t)N * 2, (uint64_t)K * N * 2};
    const uint32_t box[3] = {64, 64, 1};
    int rc = make_tensor_map_bf16_3d(&w_map, w, dims, strides, box);
    if (rc != MLA_OK) return rc;
  }
  auto kernel = mla_head_gemm_kernel<K, N, NC>;
  cudaError_t e = cudaFuncSetAttribute(
      kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, G::kSmemBytes);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(head gemm)");
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((M + kRowsPerCta - 1) / kRowsPerCta),
                     (unsigned)H, (unsigned)(N / NC));
  cfg.blockDim = dim3(128, 1, 1);
  cfg.dynamicSmemBytes = G::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kernel, a_map, w_map,
                         static_cast<__nv_bfloat16*>(out), M, H, status);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch mla_head_gemm_kernel");
  return MLA_OK;
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" int mla_absorb_q(const void* q_nope, const void* w_kc,
                            void* q_absorbed, int M, int H, int* status,
                            mla_stream_t stream) {
  return launch_head_gemm<MLA_QK_NOPE_DIM, MLA_NOPE_DIM, 128>(
      q_nope, w_kc, q_absorbed, M, H, status, (cudaStream_t)stream,
      "mla_absorb_q");
}

extern "C" int mla_project_out(const void* o_latent, const void* w_vc,
                               void* o_v, int M, int H, int* status,
                               mla_stream_t stream) {
  return launch_head_gemm<MLA_VALUE_DIM, MLA_V_HEAD_DIM, 64>(
      o_latent, w_vc, o_v, M, H, status, (cudaStream_t)stream,
      "mla_project_out");
}
