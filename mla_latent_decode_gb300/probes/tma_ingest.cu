// tma_ingest.cu -- how fast one SM can stream KV-shaped tiles from L2 into
// shared memory.
//
// One CTA per SM keeps a 4-stage ring of 32-KB stages full: a producer warp
// issues the copies, a consumer thread frees each stage as soon as it lands.
// The pool has the decode kernel's row shape ([rows, 576] bf16, 1152-B rows)
// and groups of 4 CTAs stream the same pages, as the row groups of one
// request do.  Variants: 2-D SW128 boxes of 32 or 64 rows (each L2 promotion
// setting), the same boxes from two issuing warps, one 3-D box per stage
// ({64 elements, 64 rows, 4 chunks}), 1-D bulk copies of 8/16/32 KB, and the
// 64-row case on fewer SMs (a per-SM limit does not move with grid size).
//
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 \
//        -o tma_ingest mla_latent_decode_gb300/probes/tma_ingest.cu && ./tma_ingest
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <cstdio>
#include <cstdint>
#include "../csrc/ptx_sm103.cuh"
using namespace mla::ptx;

constexpr int kStage = 32768;
__device__ int g_err;

__device__ __forceinline__ void tma3d(uint32_t dst, const void* map, uint32_t bar, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];"
               :: "r"(dst), "l"(map), "r"(bar), "r"(x), "r"(y), "r"(z) : "memory");
}
__device__ __forceinline__ void bulk1d(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

// mode 0: 2-D boxes of BR rows (32768 / (BR*128) boxes per stage), issued by lanes of warp 0
// mode 1: as 0 but boxes alternate between warps 0 and 2
// mode 2: one 3-D box per stage
// mode 3: 1-D bulk copies of BB bytes
__global__ void __launch_bounds__(96) ring(const __grid_constant__ CUtensorMap map, int mode, int BR, int BB,
                                           int iters, int pages_total, const uint8_t* kv, long long* cyc) {
  extern __shared__ uint8_t raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full[4], empty[4];
  __shared__ int abort_flag;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int NS = 4;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int i = 0; i < NS; ++i) { mbar_init(smem_u32(&full[i]), mode == 1 ? 2 : 1); mbar_init(smem_u32(&empty[i]), 1); }
    fence_mbar_init();
  }
  __syncthreads();
  const int group = blockIdx.x / 4;
  const long long t0 = clock64();
  const bool producer = warp == 0 || (mode == 1 && warp == 2);
  if (producer) {
    uint32_t stage = 0, phase = 0;
    const int nbox = mode == 0 || mode == 1 ? kStage / (BR * 128) : (mode == 3 ? kStage / BB : 1);
    for (int it = 0; it < iters; ++it) {
      const int c = (it % 2) * 4;  // chunk group 0..3 or 4..7
      const int pg = ((group * 97 + it * 4) % (pages_total - 8));
      bool ok = true;
      if (lane == 0) {
        ok = mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, &abort_flag);
        if (ok) mbar_arrive_expect_tx(smem_u32(&full[stage]), mode == 1 ? kStage / 2 : kStage);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) { if (lane == 0) { atomicAdd(&g_err, 1); abort_flag = 1; } break; }
      const uint32_t dst = smem_u32(ring + stage * kStage);
      if (mode == 0 || mode == 1) {
        // box b: chunk c + b % 4, rows (b / 4) * BR of page pg (BR = 64: 4 boxes; BR = 32: 8 boxes)
        for (int b = lane; b < nbox; b += 32) {
          if (mode == 1 && ((b & 1) != (warp == 2 ? 1 : 0))) continue;
          tma_load_2d(dst + b * BR * 128, &map, smem_u32(&full[stage]), (c + b % 4) * 64, pg * 64 + (b / 4) * BR);
        }
      } else if (mode == 2) {
        if (lane == 0) tma3d(dst, &map, smem_u32(&full[stage]), 0, pg * 64, c);
      } else {
        for (int b = lane; b < nbox; b += 32)
          bulk1d(dst + b * BB, kv + (int64_t)pg * 64 * 1152 + (int64_t)b * BB, BB, smem_u32(&full[stage]));
      }
      if (++stage == (uint32_t)NS) { stage = 0; phase ^= 1u; }
    }
  } else if (warp == 1 && lane == 0) {
    uint32_t stage = 0, phase = 0;
    for (int it = 0; it < iters; ++it) {
      if (!mbar_wait(smem_u32(&full[stage]), phase, &abort_flag)) { atomicAdd(&g_err, 1); abort_flag = 1; break; }
      mbar_arrive(smem_u32(&empty[stage]));
      if (++stage == (uint32_t)NS) { stage = 0; phase ^= 1u; }
    }
    cyc[blockIdx.x] = clock64() - t0;
  }
  __syncthreads();
}

int main() {
  void* p = nullptr; cudaDriverEntryPointQueryResult q;
  cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
  auto enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  const int pages_total = 2048;   // 151 MB: L2-sized working set, hot after the first pass
  const long long rows = (long long)pages_total * 64;
  uint8_t* kv; cudaMalloc(&kv, rows * 1152); cudaMemset(kv, 0, rows * 1152);
  long long* cyc; cudaMalloc(&cyc, 152 * 8);  // one slot per CTA, grid <= 152
  int nsm = 0; cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, 0);
  if (nsm > 152) nsm = 152;
  const int smem = 4 * kStage + 1024 + 64 * 1024;
  cudaFuncSetAttribute(ring, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  auto run = [&](const char* what, CUtensorMap& map, int mode, int BR, int BB, int grid = 0) {
    const int iters = 2000;
    if (grid == 0) grid = nsm;
    ring<<<grid, 96, smem>>>(map, mode, BR, BB, iters, pages_total, kv, cyc);
    ring<<<grid, 96, smem>>>(map, mode, BR, BB, iters, pages_total, kv, cyc);
    cudaError_t e = cudaDeviceSynchronize();
    long long h[152]; cudaMemcpy(h, cyc, grid * 8, cudaMemcpyDeviceToHost);
    int err = 0; cudaMemcpyFromSymbol(&err, g_err, 4);
    double avg = 0; for (int i = 0; i < grid; ++i) avg += h[i]; avg /= grid;
    printf("%-44s %3d CTAs: cycles/32KB %.0f -> %.1f B/clk/SM  %s err %d\n", what, grid, avg / iters, (double)kStage * iters / avg, cudaGetErrorString(e), err);
  };
  CUtensorMapL2promotion proms[4] = {CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_64B,
                                     CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B};
  const char* pn[4] = {"none", "64B", "128B", "256B"};
  for (int pi = 0; pi < 4; ++pi) for (int BR : {32, 64}) {
    CUtensorMap map;
    cuuint64_t dims[2] = {576, (cuuint64_t)rows};
    cuuint64_t strides[1] = {1152};
    cuuint32_t box[2] = {64, (cuuint32_t)BR}, es[2] = {1, 1};
    if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kv, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, proms[pi], CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) { printf("enc fail\n"); return 1; }
    char buf[96]; snprintf(buf, sizeof buf, "2-D box %d rows, promotion %s", BR, pn[pi]);
    run(buf, map, 0, BR, 0);
    if (BR == 64 && pi == 3) {
      run("2-D box 64 rows, two issuing warps", map, 1, 64, 0);
      run("2-D box 64 rows, promotion 256B", map, 0, 64, 0, 38);
      run("2-D box 64 rows, promotion 256B", map, 0, 64, 0, 16);
    }
  }
  {
    CUtensorMap map3;
    cuuint64_t dims[3] = {64, (cuuint64_t)rows, 9};
    cuuint64_t strides[2] = {1152, 128};
    cuuint32_t box[3] = {64, 64, 4}, es[3] = {1, 1, 1};
    CUresult r = enc(&map3, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, kv, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) printf("3-D encode failed (%d)\n", (int)r);
    else run("3-D box {64 el, 64 rows, 4 chunks}", map3, 2, 0, 0);
  }
  CUtensorMap dummy{};
  for (int BB : {8192, 16384, 32768}) { char buf[64]; snprintf(buf, sizeof buf, "1-D bulk copies of %d B", BB); run(buf, dummy, 3, 0, BB); }
  return 0;
}
