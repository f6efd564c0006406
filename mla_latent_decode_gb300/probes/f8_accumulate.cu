// f8_accumulate.cu -- accumulation precision of one tcgen05 MMA, kind::f8f6f4
// (M = 128, N = 256, K = 32) and kind::f16 (K = 16) for comparison: one
// large product (16 x 16) per row and dot product plus many small ones of
// 2^-(r % 10) x 2^-(n % 10); the MMA's sums are compared with the exact ones.
// On GB300 both kinds keep about 21-22 bits of the sum (products below
// about 2^-16 of the largest drop out), so a two-part 8-bit operand
// (hi + lo) keeps its low part.
// Build: nvcc -gencode arch=compute_103a,code=sm_103a -O2 -std=c++17
//        -o f8_accumulate f8_accumulate.cu
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cstdio>
#include <cstdint>
#include <cstring>
#include <cmath>
#include "../csrc/ptx_sm103.cuh"
using namespace mla::ptx;

__host__ __device__ inline uint8_t e4m3_pow2(int e) {  // 2^e, e in [-9, 8]
  if (e >= -6) return (uint8_t)((e + 7) << 3);
  return (uint8_t)(1 << (e + 9));  // subnormal m * 2^-9
}
__device__ inline uint32_t sw128(int r, int c) {
  return (r >> 3) * 1024 + (r & 7) * 128 + ((((c >> 4) ^ (r & 7)) & 7) << 4) + (c & 15);
}
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
__host__ __device__ constexpr uint32_t idesc(int kind8, int M, int N) {
  // f8: formats 0 (e4m3); f16: formats 0 (f16)
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

struct __align__(1024) Sm {
  uint8_t A[16384];
  uint8_t B[32768];
  uint64_t bar;
  uint32_t tmem;
};


__global__ void __launch_bounds__(128) probe(int kind8, float* out, int* err) {
  extern __shared__ uint8_t raw[];
  Sm& s = *reinterpret_cast<Sm*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x / 32, r = threadIdx.x;
  __shared__ int abort_flag;
  const int K = kind8 ? 32 : 16;
  // A[r][k] = 16 at k = kb(r) (0 for r < 64, K-1 otherwise), else 2^-(r % 10);
  // B[n][k] = 16 at k = 0 and k = K-1, else 2^-(n % 10).
  {
    const int kb = r < 64 ? 0 : K - 1;
    for (int k = 0; k < K; ++k) {
      const int e = k == kb ? 4 : -(r % 10);
      if (kind8) s.A[sw128(r, k)] = e4m3_pow2(e);
      else { __half h = __float2half(ldexpf(1.f, e)); memcpy(s.A + sw128(r, 2 * k), &h, 2); }
    }
    for (int n2 = 0; n2 < 2; ++n2) {
      const int n = 2 * r + n2;
      for (int k = 0; k < K; ++k) {
        const int e = (k == 0 || k == K - 1) ? 4 : -(n % 10);
        if (kind8) s.B[sw128(n, k)] = e4m3_pow2(e);
        else { __half h = __float2half(ldexpf(1.f, e)); memcpy(s.B + sw128(n, 2 * k), &h, 2); }
      }
    }
  }
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&s.bar), 1);
    fence_mbar_init();
  }
  fence_proxy_async_smem();
  __syncthreads();
  if (warp == 0) { tmem_alloc(smem_u32(&s.tmem), 256); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem;
  if (threadIdx.x == 0) {
    const uint64_t a = sdesc(smem_u32(s.A), 16, 1024), b = sdesc(smem_u32(s.B), 16, 1024);
    const uint32_t id = idesc(kind8, 128, 256);
    if (kind8)
      asm volatile("tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, 0;" ::"r"(tmem), "l"(a), "l"(b), "r"(id) : "memory");
    else
      asm volatile("tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, 0;" ::"r"(tmem), "l"(a), "l"(b), "r"(id) : "memory");
    mma_commit(smem_u32(&s.bar));
    if (!mbar_wait(smem_u32(&s.bar), 0, &abort_flag)) atomicAdd(err, 1);
  }
  __syncthreads();
  tc_fence_after();
  uint32_t v[32];
  for (int c0 = 0; c0 < 256; c0 += 32) {
    tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + c0, v);
    tmem_wait_ld();
    for (int c = 0; c < 32; ++c) out[(size_t)r * 256 + c0 + c] = __uint_as_float(v[c]);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

int main() {
  float* dout; cudaMalloc(&dout, 128 * 256 * 4);
  int* derr; cudaMalloc(&derr, 4);
  const int smem = sizeof(Sm) + 1024;
  cudaFuncSetAttribute(probe, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  for (int kind8 = 1; kind8 >= 0; --kind8) {
    cudaMemset(derr, 0, 4);
    probe<<<1, 128, smem>>>(kind8, dout, derr);
    cudaError_t e = cudaDeviceSynchronize();
    static float h[128 * 256]; int er = -1;
    cudaMemcpy(h, dout, sizeof h, cudaMemcpyDeviceToHost); cudaMemcpy(&er, derr, 4, cudaMemcpyDeviceToHost);
    printf("%s: %s err %d\n", kind8 ? "kind::f8f6f4 K=32" : "kind::f16 K=16", cudaGetErrorString(e), er);
    if (e != cudaSuccess) return 2;
    const int K = kind8 ? 32 : 16;
    // exact: row r, col n: A[r][kbig_r] = 16, A[r][k] = 2^(er/2) otherwise; B[n][0] = B[n][K-1] = 16, else 2^en
    // bits of the small terms kept: log2 of (got - big) / (exact - big)
    for (int r : {0, 5, 10, 20, 70, 80, 90}) {
      printf(" row %3d (big at %s):", r, r < 64 ? "k=0" : "k=K-1");
      for (int n : {0, 3, 6, 9}) {
        const int kb = r < 64 ? 0 : K - 1;
        const int er_ = -(r % 10);
        double ex = 0;
        for (int k = 0; k < K; ++k) {
          const double a = k == kb ? 16 : ldexp(1.0, er_);
          const double b = (k == 0 || k == K - 1) ? 16 : ldexp(1.0, -(n % 10));
          ex += a * b;
        }
        const double got = h[r * 256 + n];
        printf("  n%d exact %.9g got %.9g relerr %.2e", n, ex, got, fabs(got - ex) / ex);
      }
      printf("\n");
    }
    double worst = 0;
    for (int r = 0; r < 128; ++r) for (int n = 0; n < 256; ++n) {
      const int kb = r < 64 ? 0 : K - 1;
      const int er_ = -(r % 10);
      double ex = 0;
      for (int k = 0; k < K; ++k) {
        const double a = k == kb ? 16 : ldexp(1.0, er_);
        const double b = (k == 0 || k == K - 1) ? 16 : ldexp(1.0, -(n % 10));
        ex += a * b;
      }
      const double rel = fabs(h[r * 256 + n] - ex) / ex;
      if (rel > worst) worst = rel;
    }
    printf(" worst relative error %.3e (%.1f bits)\n", worst, worst > 0 ? -log2(worst) : 99.0);
  }
  return 0;
}
