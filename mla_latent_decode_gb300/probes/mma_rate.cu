// mma_rate.cu -- issue rate of back-to-back tcgen05 kind::f16 (BF16) MMAs
// into one accumulator, by shape and operand source: the CTA-pair form
// (cta_group::2, M = 256, 128 rows per SM) and the single-CTA form (M =
// 128), N = 256 or 128, A from TMEM or from shared memory, K = 16, into one
// accumulator or alternating between two independent ones.  One thread
// issues 4096 MMAs, commits once and waits (bounded); the clock span over
// the count gives cycles per MMA, and 128 x N x 16 x 2 FLOP per SM per MMA
// gives FLOP per clock per SM.  Operand values are zero: the rate does not
// depend on them.
// Build: nvcc -gencode arch=compute_103a,code=sm_103a -O2 -std=c++17
//        -o mma_rate mma_rate.cu
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>

#include "../csrc/ptx_sm103.cuh"
using namespace mla::ptx;

constexpr int kIters = 4096;

struct __align__(1024) Sm {
  uint8_t A[16384];  // 128 rows x 64 bf16, 128-B swizzle
  uint8_t B[32768];  // up to 256 rows (single CTA, N = 256) x 64 bf16
  uint64_t bar;
  uint32_t tmem;
  int abort_flag;
};

// mode bit 0: N = 128 (else 256); bit 1: A from shared memory (else TMEM);
// bit 2: alternate between two accumulators (N = 128: columns 256 and 384;
// N = 256 with A in shared memory: columns 0 and 256)
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(128, 1)
    pair_rate(int mode, long long* cycles, int* err) {
  extern __shared__ uint8_t raw[];
  Sm& s = *reinterpret_cast<Sm*>((reinterpret_cast<uintptr_t>(raw) + 1023) &
                                 ~uintptr_t(1023));
  const uint32_t rank = cluster_ctarank();
  const int warp = threadIdx.x / 32;
  for (int i = threadIdx.x; i < (int)sizeof(s.A) / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(s.A)[i] = make_uint4(0, 0, 0, 0);
  for (int i = threadIdx.x; i < (int)sizeof(s.B) / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(s.B)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) {
    s.abort_flag = 0;
    mbar_init(smem_u32(&s.bar), 1);
    fence_mbar_init();
  }
  fence_proxy_async_smem();
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(&s.tmem), 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();
  const uint32_t tmem = s.tmem;
  if (rank == 0 && threadIdx.x == 0) {
    const int N = (mode & 1) ? 128 : 256;
    const uint32_t idesc = idesc_bf16_f32(256, N, false, false);
    const uint64_t a = sdesc_sw128(smem_u32(s.A), 16, 1024);
    const uint64_t b = sdesc_sw128(smem_u32(s.B), 16, 1024);
    const bool two = (mode & 4) != 0;
    const uint32_t d0 = two && N == 256 ? tmem : tmem + 256;
    const uint32_t d1 = two ? (N == 256 ? tmem + 256 : tmem + 384) : d0;
    const long long t0 = clock64();
    for (int it = 0; it < kIters; ++it) {
      const uint32_t acc = it > 1 ? 1u : 0u;
      const uint32_t d = (it & 1) ? d1 : d0;
      if (mode & 2)
        mma_ss_pair(d, a + 2 * (it & 3), b + 2 * (it & 3), idesc, acc);
      else
        mma_ts_pair(d, tmem + 8u * (it & 31), b + 2 * (it & 3), idesc, acc);
    }
    mma_commit_pair(smem_u32(&s.bar), 0x3);
    const bool ok = mbar_wait(smem_u32(&s.bar), 0, &s.abort_flag);
    const long long t1 = clock64();
    cycles[mode] = t1 - t0;
    if (!ok) atomicOr(err, 1);
  } else if (rank == 1 && threadIdx.x == 0) {
    if (!mbar_wait(smem_u32(&s.bar), 0, &s.abort_flag)) atomicOr(err, 2);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();
  if (warp == 1) tmem_dealloc_pair(tmem, 512);
}

__global__ void __launch_bounds__(128, 1)
    single_rate(int mode, long long* cycles, int* err) {
  extern __shared__ uint8_t raw[];
  Sm& s = *reinterpret_cast<Sm*>((reinterpret_cast<uintptr_t>(raw) + 1023) &
                                 ~uintptr_t(1023));
  const int warp = threadIdx.x / 32;
  for (int i = threadIdx.x; i < (int)sizeof(s.A) / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(s.A)[i] = make_uint4(0, 0, 0, 0);
  for (int i = threadIdx.x; i < (int)sizeof(s.B) / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(s.B)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) {
    s.abort_flag = 0;
    mbar_init(smem_u32(&s.bar), 1);
    fence_mbar_init();
  }
  fence_proxy_async_smem();
  if (warp == 1) {
    tmem_alloc(smem_u32(&s.tmem), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem;
  if (threadIdx.x == 0) {
    const int N = (mode & 1) ? 128 : 256;
    const uint32_t idesc = idesc_bf16_f32(128, N, false, false);
    const uint64_t a = sdesc_sw128(smem_u32(s.A), 16, 1024);
    const uint64_t b = sdesc_sw128(smem_u32(s.B), 16, 1024);
    const uint32_t d = tmem + 256;
    const long long t0 = clock64();
    for (int it = 0; it < kIters; ++it) {
      const uint32_t acc = it > 0 ? 1u : 0u;
      if (mode & 2)
        mma_ss(d, a + 2 * (it & 3), b + 2 * (it & 3), idesc, acc);
      else
        mma_ts(d, tmem + 8u * (it & 31), b + 2 * (it & 3), idesc, acc);
    }
    mma_commit(smem_u32(&s.bar));
    const bool ok = mbar_wait(smem_u32(&s.bar), 0, &s.abort_flag);
    const long long t1 = clock64();
    cycles[4 + mode] = t1 - t0;
    if (!ok) atomicOr(err, 4);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

int main() {
  long long* d_cycles;
  int* d_err;
  cudaMalloc(&d_cycles, 16 * sizeof(long long));
  cudaMalloc(&d_err, sizeof(int));
  cudaMemset(d_cycles, 0, 16 * sizeof(long long));
  cudaMemset(d_err, 0, sizeof(int));
  const int smem = (int)sizeof(Sm) + 1024;
  cudaFuncSetAttribute(pair_rate, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  cudaFuncSetAttribute(single_rate, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  for (int rep = 0; rep < 2; ++rep)  // the first pass warms up
    for (int mode = 0; mode < 4; ++mode) {
      pair_rate<<<2, 128, smem>>>(mode, d_cycles, d_err);
      single_rate<<<1, 128, smem>>>(mode, d_cycles, d_err);
    }
  // two accumulators: N = 128 with A in TMEM or shared memory, N = 256 with
  // A in shared memory (A in TMEM leaves room for one N = 256 accumulator)
  for (int rep = 0; rep < 2; ++rep)
    for (int mode : {5, 7, 6}) pair_rate<<<2, 128, smem>>>(mode, d_cycles + 8, d_err);
  cudaError_t e = cudaDeviceSynchronize();
  long long cyc[16];
  int err = 0;
  cudaMemcpy(cyc, d_cycles, sizeof(cyc), cudaMemcpyDeviceToHost);
  cudaMemcpy(&err, d_err, sizeof(int), cudaMemcpyDeviceToHost);
  printf("cuda: %s, wait errors: %d\n", cudaGetErrorString(e), err);
  const char* names[4] = {"N=256, A in TMEM", "N=128, A in TMEM",
                          "N=256, A in SMEM", "N=128, A in SMEM"};
  for (int k = 0; k < 8; ++k) {
    const int N = (k & 1) ? 128 : 256;
    const double per = (double)cyc[k] / kIters;
    printf("%s M=%d %-18s %7.1f cycles/MMA  %6.0f FLOP/clk/SM\n",
           k < 4 ? "pair  " : "single", k < 4 ? 256 : 128, names[k & 3], per,
           128.0 * N * 16 * 2 / per);
  }
  for (int mode : {5, 7, 6}) {
    const int N = (mode & 1) ? 128 : 256;
    const double per = (double)cyc[8 + mode] / kIters;
    printf("pair   M=256 %s, two accumulators %7.1f cycles/MMA  %6.0f FLOP/clk/SM\n",
           names[mode & 3], per, 128.0 * N * 16 * 2 / per);
  }
  return (e == cudaSuccess && err == 0) ? 0 : 1;
}
