// mla_absorb.cu -- the per-head projections on either side of the absorbed
// decode ([K3-MEM] in include/mla_decode.h: w_kc is 96 x 128 x 512 bf16 and
// the absorbed query is 512-d; kv_b_proj is absorbed into w_kc / w_vc):
//   query absorption   q_abs[m, h, :512] = q_nope[m, h, :128] . w_kc[h]
//   output projection  o_v[m, h, :128]  = o_lat[m, h, :512] . w_vc[h]
// (m = b * q_len + i).  Both are per-head batched GEMMs with few rows
// (B * q_len) and a weight slice per head, so the weights' HBM bytes bound
// them; the products run on tcgen05 tensor cores.
//
// A persistent grid (one CTA per SM at most) walks the output tiles (128
// rows x NC columns of one head) round-robin.  Each CTA is a small pipeline
// of three roles:
//   warp 0     streams K in steps of 64 through a ring of shared-memory
//              stages by TMA: the head's activation rows through a 3-D
//              tensor map (64 K x 1 head x 128 rows, K-major, 128-byte
//              swizzle, rows past M read as zeros) and the weight slice in
//              64 x 64 boxes (rows = K, 128-byte rows of N: MN-major);
//   warp 1     issues M = 128, N = NC, K = 16 bf16 MMAs into one of two TMEM
//              accumulators, so a tile's products overlap the previous
//              tile's epilogue;
//   warps 2-5  read the accumulator (warp w owns TMEM lanes 32 (w % 4) ..),
//              round to bf16 into a swizzled shared-memory box of their 32
//              rows and store it with one TMA store per 64 columns (rows
//              past M are clipped by the tensor map): whole 128-byte lines
//              leave the SM, where per-thread stores of 16 bytes into rows
//              H * N apart did not.
// Launches use programmatic dependent launch: a CTA lets the stream's next
// kernel start at once and, before it waits for the kernels it depends on,
// has the weight slices of all its tiles prefetched into L2 (a prefetch
// reads nothing into the CTA, so weights written by those kernels are still
// read after they finish: L2 holds the current data).  Every wait is
// bounded (ptx_sm103.cuh); a timeout sets MLA_STATUS_WAIT_TIMEOUT.
#include <cuda_bf16.h>

#include <algorithm>

#include "mla_tma.cuh"
#include "ptx_sm103.cuh"

namespace mla {
namespace {

using namespace ptx;

constexpr int kRowsPerTile = 128;
constexpr int kBoxA = 128 * 128;  // 64 K x 128 rows bf16 = 16 KB
constexpr int kBoxW = 64 * 128;   // 64 K rows x 64 N bf16 = 8 KB
constexpr int kBoxOut = 32 * 128; // 32 rows x 64 N bf16 = 4 KB
constexpr int kThreads = 192;     // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue

template <int K, int N, int NC, int STAGES>
struct HeadGemm {
  static constexpr int kStageBytes = kBoxA + (NC / 64) * kBoxW;
  static constexpr int kKSteps = K / 64;     // ring stages per tile
  static constexpr int kChunksN = N / NC;    // column chunks per head
  static constexpr int kTmemCols = 2 * NC;   // two accumulators
  static constexpr int kOutBytes = 4 * (NC / 64) * kBoxOut;  // 4 warps' boxes
  static constexpr int kSmemBytes =
      STAGES * kStageBytes + kOutBytes + 1024 + 256;
  static_assert(K % 64 == 0 && N % NC == 0 && NC % 64 == 0 && NC <= 256,
                "shape");
  static_assert((kTmemCols & (kTmemCols - 1)) == 0, "TMEM columns: power of 2");
  // One CTA per SM: it alone holds the SM's TMEM.
  static_assert(kSmemBytes <= 227 * 1024 && 2 * kSmemBytes > 228 * 1024,
                "shared memory budget");
};

struct Tile {
  int mt, h, nc;
};

__device__ __forceinline__ Tile tile_of(int t, int H, int chunks) {
  const int r = t / chunks;
  return Tile{r / H, r % H, t % chunks};
}

template <int K, int N, int NC, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
    mla_head_gemm_kernel(const __grid_constant__ CUtensorMap a_map,
                         const __grid_constant__ CUtensorMap w_map,
                         const __grid_constant__ CUtensorMap out_map, int M,
                         int H, int tiles, uint32_t stage_tx, int* status) {
  using G = HeadGemm<K, N, NC, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* obox = base + STAGES * G::kStageBytes;  // epilogue boxes
  uint64_t* full = reinterpret_cast<uint64_t*>(obox + G::kOutBytes);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;  // accumulator b holds a finished tile
  uint64_t* tempty = tfull + 2;      // accumulator b has been read out
  uint64_t* drain = tempty + 2;      // every MMA issued has completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  volatile int* abort = abort_flag;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const auto give_up = [&]() {
    *abort = 1;
    if (status) atomicOr(status, MLA_STATUS_WAIT_TIMEOUT);
  };
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&tfull[b]), 1);
      mbar_init(smem_u32(&tempty[b]), 4);
    }
    mbar_init(smem_u32(drain), 1);
    fence_mbar_init();
    prefetch_tmap(&a_map);
    prefetch_tmap(&w_map);
    prefetch_tmap(&out_map);
  }
  griddep_launch_dependents();
  if (warp == 0) {
    // The weight slices of this CTA's tiles into L2 while earlier kernels
    // finish, one box per lane in turn.
    int i = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
      const Tile tl = tile_of(t, H, G::kChunksN);
      for (int ks = 0; ks < G::kKSteps; ++ks)
        for (int nb = 0; nb < NC / 64; ++nb, ++i)
          if ((i & 31) == lane)
            tma_prefetch_3d(&w_map, tl.nc * NC + nb * 64, ks * 64, tl.h);
    }
  } else if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), G::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_wait();

  if (warp == 0) {
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
        const Tile tl = tile_of(t, H, G::kChunksN);
        for (int ks = 0; ks < G::kKSteps; ++ks, ++it) {
          const uint32_t st = it % STAGES, use = it / STAGES;
          if (use > 0 && !mbar_wait(smem_u32(&empty[st]), (use - 1) & 1, abort)) {
            ok = false;
            break;
          }
          uint8_t* sa = base + st * G::kStageBytes;
          uint8_t* sw = sa + kBoxA;
          const uint32_t bar = smem_u32(&full[st]);
          mbar_arrive_expect_tx(bar, stage_tx);
          tma_load_3d(smem_u32(sa), &a_map, bar, ks * 64, tl.h,
                      tl.mt * kRowsPerTile);
          for (int nb = 0; nb < NC / 64; ++nb)
            tma_load_3d(smem_u32(sw + nb * kBoxW), &w_map, bar,
                        tl.nc * NC + nb * 64, ks * 64, tl.h);
        }
      }
      if (!ok) give_up();
      // Every load issued has landed before the CTA may exit (bounded, and
      // regardless of the abort flag).
      int never = 0;
      for (uint32_t j = it > (uint32_t)STAGES ? it - STAGES : 0; j < it; ++j)
        mbar_wait(smem_u32(&full[j % STAGES]), (j / STAGES) & 1, &never);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kRowsPerTile, NC, false, true);
      uint32_t it = 0, tc = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++tc) {
        const uint32_t b = tc & 1, ub = tc >> 1;
        if (ub > 0 && !mbar_wait(smem_u32(&tempty[b]), (ub - 1) & 1, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + b * NC;
        for (int ks = 0; ks < G::kKSteps; ++ks, ++it) {
          const uint32_t st = it % STAGES, use = it / STAGES;
          if (!mbar_wait(smem_u32(&full[st]), use & 1, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint8_t* sa = base + st * G::kStageBytes;
          // A: K-major, the next 16 K 32 B (2 units) on.  W: MN-major, the
          // next 64 N one box (LBO) on, the next 8 K rows 1 KB (SBO) on, the
          // next 16 K rows 2 KB (128 units) on.
          const uint64_t a = sdesc_sw128(smem_u32(sa), 16, 1024);
          const uint64_t w = sdesc_sw128(smem_u32(sa + kBoxA), kBoxW, 1024);
#pragma unroll
          for (int k16 = 0; k16 < 4; ++k16)
            mma_ss(d, a + 2 * k16, w + 128 * k16, idesc, (ks | k16) ? 1u : 0u);
          mma_commit(smem_u32(&empty[st]));
        }
        if (!ok) break;
        mma_commit(smem_u32(&tfull[b]));
      }
      if (!ok) give_up();
      // No MMA may still run when the accumulators are freed.
      int never = 0;
      mma_commit(smem_u32(drain));
      mbar_wait(smem_u32(drain), 0, &never);
    }
    __syncwarp();
  } else {
    // Epilogue: warp w may read TMEM lanes 32 (w % 4) .. + 31, rows of the
    // tile; lane l writes row l of the warp's boxes (16-byte chunk j of a
    // row at chunk j ^ (l & 7): the 128-byte swizzle of the tensor map).
    const int q = warp & 3;
    uint8_t* mybox = obox + q * (NC / 64) * kBoxOut;
    uint32_t tc = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++tc) {
      const uint32_t b = tc & 1, ub = tc >> 1;
      if (!mbar_wait(smem_u32(&tfull[b]), ub & 1, abort)) {
        if (lane == 0) give_up();
        break;
      }
      tc_fence_after();
      const Tile tl = tile_of(t, H, G::kChunksN);
      const int row0 = tl.mt * kRowsPerTile + q * 32;
      const bool rows = row0 < M;
      if (rows) {
        // The boxes' previous stores have read them.
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
        const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + b * NC;
        // 64 columns (one box row) per TMEM wait.
#pragma unroll 1
        for (int c0 = 0; c0 < NC; c0 += 64) {
          uint32_t v[64];
          tmem_ld32(taddr + c0, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
          tmem_ld32(taddr + c0 + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
          tmem_wait_ld();
          uint8_t* row = mybox + (c0 / 64) * kBoxOut + lane * 128;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            uint32_t w4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              __nv_bfloat162 b2 = __floats2bfloat162_rn(
                  __uint_as_float(v[8 * j + 2 * e]),
                  __uint_as_float(v[8 * j + 2 * e + 1]));
              w4[e] = *reinterpret_cast<uint32_t*>(&b2);
            }
            *reinterpret_cast<uint4*>(row + ((j ^ (lane & 7)) << 4)) =
                make_uint4(w4[0], w4[1], w4[2], w4[3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&tempty[b]));
      if (rows) {
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          for (int bx = 0; bx < NC / 64; ++bx)
            tma_store_3d(&out_map, smem_u32(mybox + bx * kBoxOut),
                         tl.nc * NC + bx * 64, tl.h, row0);
          bulk_commit_group();
        }
      }
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, G::kTmemCols);
  }
}

template <int K, int N, int NC, int STAGES>
int launch_head_gemm(const void* in, const void* w, void* out, int M, int H,
                     int* status, cudaStream_t stream, const char* name) {
  using G = HeadGemm<K, N, NC, STAGES>;
  if (!in || !w || !out)
    return fail(MLA_ERR_INVALID_ARG, "%s: input, weights and output are required", name);
  if (M < 1 || H < 1)
    return fail(MLA_ERR_INVALID_ARG, "%s: M=%d H=%d out of range", name, M, H);
  const int64_t tiles =
      (int64_t)((M + kRowsPerTile - 1) / kRowsPerTile) * H * G::kChunksN;
  if (tiles > 0x7fffffff)
    return fail(MLA_ERR_INVALID_ARG, "%s: M=%d H=%d too large", name, M, H);
  if (!aligned(in, 16) || !aligned(w, 16) || !aligned(out, 16) ||
      (status && !aligned(status, 4)))
    return fail(MLA_ERR_MISALIGNED, "%s: arrays need 16-B alignment", name);
  CUtensorMap a_map, w_map, out_map;
  // Fewer than 128 rows: the A box holds only them (rounded up to 8, the
  // swizzle's row period) and the tile's other rows of shared memory keep
  // whatever they held; they only reach accumulator rows that are never
  // stored.
  const uint32_t a_rows =
      M >= kRowsPerTile ? kRowsPerTile : (uint32_t)((M + 7) / 8 * 8);
  const uint32_t stage_tx = a_rows * 128 + (NC / 64) * kBoxW;
  {
    const uint64_t dims[3] = {(uint64_t)K, (uint64_t)H, (uint64_t)M};
    const uint64_t strides[2] = {(uint64_t)K * 2, (uint64_t)H * K * 2};
    const uint32_t box[3] = {64, 1, a_rows};
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
  {
    const uint64_t dims[3] = {(uint64_t)N, (uint64_t)H, (uint64_t)M};
    const uint64_t strides[2] = {(uint64_t)N * 2, (uint64_t)H * N * 2};
    const uint32_t box[3] = {64, 1, 32};
    int rc = make_tensor_map_bf16_3d(&out_map, out, dims, strides, box);
    if (rc != MLA_OK) return rc;
  }
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "head gemm: device query");
  auto kernel = mla_head_gemm_kernel<K, N, NC, STAGES>;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           G::kSmemBytes);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(head gemm)");
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)std::min<int64_t>(tiles, std::max(sms, 1)), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = G::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kernel, a_map, w_map, out_map, M, H, (int)tiles,
                         stage_tx, status);
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
  return launch_head_gemm<MLA_QK_NOPE_DIM, MLA_NOPE_DIM, 256, 3>(
      q_nope, w_kc, q_absorbed, M, H, status, (cudaStream_t)stream,
      "mla_absorb_q");
}

extern "C" int mla_project_out(const void* o_latent, const void* w_vc,
                               void* o_v, int M, int H, int* status,
                               mla_stream_t stream) {
  return launch_head_gemm<MLA_VALUE_DIM, MLA_V_HEAD_DIM, 128, 5>(
      o_latent, w_vc, o_v, M, H, status, (cudaStream_t)stream,
      "mla_project_out");
}
