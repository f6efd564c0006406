// f8_operands.cu -- the tcgen05.mma.kind::f8f6f4 operand forms the FP8 decode
// kernel uses, checked bit-exactly on small integers (one CTA, M = 128):
//   mode 0: A (E4M3) in shared memory, K-major 128-byte swizzle; B (E4M3)
//           K-major 128-byte swizzle landed by TMA; N = 256, K = 128
//   mode 1: the same with A in TMEM (four E4M3 bytes per 32-bit column)
//   mode 2: the same with an E5M2 A operand (A format field 1)
//   mode 3: B MN-major, 128-byte swizzle: V[k tokens][n dims], the next 128
//           dims one 8-KB box on (LBO), the next 8 tokens 1 KB on (SBO)
//   mode 4: mode 3 with LBO and SBO swapped (a control: it must fail)
//   mode 5: 64-byte swizzle, K-major (the RoPE block), SBO 512
// Build: nvcc -gencode arch=compute_103a,code=sm_103a -O2 -std=c++17
//        -o f8_operands f8_operands.cu -lcuda
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <cstdio>
#include <cstdint>
#include <cstring>
#include <cmath>
#include "../csrc/ptx_sm103.cuh"
using namespace mla::ptx;

__host__ __device__ inline int aval(int r, int k) { return ((r * 3 + k) % 7) - 3; }
__host__ __device__ inline int bval(int n, int k) { return ((n * 5 + k * 3) % 5) - 2; }

// exact small-integer encodings
__host__ __device__ inline uint8_t enc_e4m3(int v) {
  const uint8_t t[5] = {0x00, 0x38, 0x40, 0x44, 0x48};  // 0,1,2,3,4
  uint8_t c = t[v < 0 ? -v : v];
  return v < 0 ? (uint8_t)(c | 0x80) : c;
}
__host__ __device__ inline uint8_t enc_e5m2(int v) {
  const uint8_t t[5] = {0x00, 0x3C, 0x40, 0x42, 0x44};  // 0,1,2,3,4
  uint8_t c = t[v < 0 ? -v : v];
  return v < 0 ? (uint8_t)(c | 0x80) : c;
}

__device__ inline uint32_t sw128(int r, int c) {  // byte c of 128-B row r
  return (r >> 3) * 1024 + (r & 7) * 128 + ((((c >> 4) ^ (r & 7)) & 7) << 4) + (c & 15);
}
__device__ inline uint32_t sw64(int r, int c) {  // byte c of 64-B row r
  return (r >> 3) * 512 + (r & 7) * 64 + ((((c >> 4) ^ ((r >> 1) & 3)) & 3) << 4) + (c & 15);
}

__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)layout << 61;
  return d;
}
__host__ __device__ constexpr uint32_t idesc_f8(int M, int N, uint32_t afmt, uint32_t bfmt, bool bmn) {
  return (1u << 4) | (afmt << 7) | (bfmt << 10) | ((bmn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void mma_ss8(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
               "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}
__device__ __forceinline__ void mma_ts8(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
               "r"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}

struct __align__(1024) Sm {
  uint8_t A[16384];
  uint8_t B[49152];
  uint64_t bar_full, bar_done;
  uint32_t tmem;
};

__global__ void __launch_bounds__(128) probe(const __grid_constant__ CUtensorMap bmap, int mode, float* out, int* err) {
  extern __shared__ uint8_t raw[];
  Sm& s = *reinterpret_cast<Sm*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x / 32;
  __shared__ int abort_flag;
  const int r = threadIdx.x;
  for (int i = r; i < 16384 / 4; i += 128) reinterpret_cast<uint32_t*>(s.A)[i] = 0;
  __syncthreads();
  if (mode <= 2) {
    for (int k = 0; k < 128; ++k) s.A[sw128(r, k)] = mode == 2 ? enc_e5m2(aval(r, k)) : enc_e4m3(aval(r, k));
  } else if (mode <= 4) {
    for (int k = 0; k < 64; ++k) s.A[sw128(r, k)] = enc_e4m3(aval(r, k));
  } else {
    for (int k = 0; k < 64; ++k) s.A[sw64(r, k)] = enc_e4m3(aval(r, k));
  }
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&s.bar_full), 1);
    mbar_init(smem_u32(&s.bar_done), 1);
    fence_mbar_init();
  }
  fence_proxy_async_smem();
  __syncthreads();
  if (warp == 0) { tmem_alloc(smem_u32(&s.tmem), 512); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem;
  if (mode == 1) {
    uint32_t v[32];
    for (int c = 0; c < 32; ++c) {
      uint32_t w = 0;
      for (int b = 0; b < 4; ++b) w |= (uint32_t)enc_e4m3(aval(r, 4 * c + b)) << (8 * b);
      v[c] = w;
    }
    tmem_st32(tmem + ((uint32_t)(warp * 32) << 16) + 256, v);
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) {
    const uint32_t full = smem_u32(&s.bar_full);
    if (mode <= 2) {
      mbar_arrive_expect_tx(full, 32768);
      for (int j = 0; j < 4; ++j) tma_load_2d(smem_u32(s.B) + 8192 * j, &bmap, full, 0, 64 * j);
    } else if (mode <= 4) {
      mbar_arrive_expect_tx(full, 16384);
      for (int j = 0; j < 2; ++j) tma_load_2d(smem_u32(s.B) + 8192 * j, &bmap, full, 128 * j, 0);
    } else {
      mbar_arrive_expect_tx(full, 16384);
      for (int j = 0; j < 4; ++j) tma_load_2d(smem_u32(s.B) + 4096 * j, &bmap, full, 0, 64 * j);
    }
    bool ok = mbar_wait(full, 0, &abort_flag);
    if (!ok) atomicAdd(err, 1);
    tc_fence_after();
    if (ok) {
      const uint32_t a0 = smem_u32(s.A), b0 = smem_u32(s.B);
      if (mode <= 2) {
        const uint32_t id = idesc_f8(128, 256, mode == 2 ? 1u : 0u, 0u, false);
        for (int k = 0; k < 4; ++k) {
          const uint64_t bd = sdesc(b0, 16, 1024, 2) + 2 * k;
          if (mode == 1) mma_ts8(tmem, tmem + 256 + 8 * k, bd, id, k > 0);
          else mma_ss8(tmem, sdesc(a0, 16, 1024, 2) + 2 * k, bd, id, k > 0);
        }
      } else if (mode <= 4) {
        const uint32_t id = idesc_f8(128, 256, 0u, 0u, true);
        const uint32_t lbo = mode == 3 ? 8192 : 1024, sbo = mode == 3 ? 1024 : 8192;
        for (int k = 0; k < 2; ++k)
          mma_ss8(tmem, sdesc(a0, 16, 1024, 2) + 2 * k, sdesc(b0 + 4096 * k, lbo, sbo, 2), id, k > 0);
      } else {
        const uint32_t id = idesc_f8(128, 256, 0u, 0u, false);
        for (int k = 0; k < 2; ++k)
          mma_ss8(tmem, sdesc(a0, 16, 512, 4) + 2 * k, sdesc(b0, 16, 512, 4) + 2 * k, id, k > 0);
      }
      mma_commit(smem_u32(&s.bar_done));
    }
    if (ok && !mbar_wait(smem_u32(&s.bar_done), 0, &abort_flag)) atomicAdd(err, 100);
  }
  __syncthreads();
  tc_fence_after();
  {
    uint32_t v[32];
    for (int c0 = 0; c0 < 256; c0 += 32) {
      tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + c0, v);
      tmem_wait_ld();
      for (int c = 0; c < 32; ++c) out[(size_t)r * 256 + c0 + c] = __uint_as_float(v[c]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

int main() {
  void* p = nullptr; cudaDriverEntryPointQueryResult q;
  cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
  auto enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  // K-major B [256 n][128 k]; MN-major V [64 k][256 n]; SW64 B [256 n][64 k]
  static uint8_t bk[256 * 128], bv[64 * 256], b64[256 * 64];
  for (int n = 0; n < 256; ++n) for (int k = 0; k < 128; ++k) bk[n * 128 + k] = enc_e4m3(bval(n, k));
  for (int k = 0; k < 64; ++k) for (int n = 0; n < 256; ++n) bv[k * 256 + n] = enc_e4m3(bval(n, k));
  for (int n = 0; n < 256; ++n) for (int k = 0; k < 64; ++k) b64[n * 64 + k] = enc_e4m3(bval(n, k));
  void *dk, *dv, *d64;
  cudaMalloc(&dk, sizeof bk); cudaMalloc(&dv, sizeof bv); cudaMalloc(&d64, sizeof b64);
  cudaMemcpy(dk, bk, sizeof bk, cudaMemcpyHostToDevice);
  cudaMemcpy(dv, bv, sizeof bv, cudaMemcpyHostToDevice);
  cudaMemcpy(d64, b64, sizeof b64, cudaMemcpyHostToDevice);
  CUtensorMap mk, mv, m64;
  cuuint32_t es[2] = {1, 1};
  {
    cuuint64_t dims[2] = {128, 256}; cuuint64_t st[1] = {128}; cuuint32_t box[2] = {128, 64};
    if (enc(&mk, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, dk, dims, st, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE)) { printf("enc k\n"); return 1; }
  }
  {
    cuuint64_t dims[2] = {256, 64}; cuuint64_t st[1] = {256}; cuuint32_t box[2] = {128, 64};
    if (enc(&mv, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, dv, dims, st, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE)) { printf("enc v\n"); return 1; }
  }
  {
    cuuint64_t dims[2] = {64, 256}; cuuint64_t st[1] = {64}; cuuint32_t box[2] = {64, 64};
    if (enc(&m64, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, d64, dims, st, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE)) { printf("enc 64\n"); return 1; }
  }
  float* dout; cudaMalloc(&dout, 128 * 256 * 4);
  int* derr; cudaMalloc(&derr, 4);
  const int smem = sizeof(Sm) + 1024;
  cudaFuncSetAttribute(probe, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  const char* names[6] = {"A smem e4m3, B K-major", "A tmem e4m3", "A smem e5m2", "B MN-major LBO 8K SBO 1K",
                          "B MN-major LBO 1K SBO 8K", "SW64 K-major"};
  for (int mode = 0; mode < 6; ++mode) {
    const CUtensorMap& m = mode <= 2 ? mk : mode <= 4 ? mv : m64;
    cudaMemset(dout, 0xff, 128 * 256 * 4); cudaMemset(derr, 0, 4);
    probe<<<1, 128, smem>>>(m, mode, dout, derr);
    cudaError_t e = cudaDeviceSynchronize();
    static float h[128 * 256]; int er = -1;
    cudaMemcpy(h, dout, sizeof h, cudaMemcpyDeviceToHost); cudaMemcpy(&er, derr, 4, cudaMemcpyDeviceToHost);
    const int K = mode <= 2 ? 128 : 64;
    int bad = 0; double maxd = 0;
    for (int mm = 0; mm < 128; ++mm) for (int n = 0; n < 256; ++n) {
      double ref = 0; for (int k = 0; k < K; ++k) ref += (double)aval(mm, k) * bval(n, k);
      double d = fabs(ref - h[mm * 256 + n]); if (!(d <= maxd)) maxd = d; if (!(d == 0)) ++bad;
    }
    printf("mode %d (%s): %s, err %d, mismatches %d, max diff %g\n", mode, names[mode], cudaGetErrorString(e), er, bad, maxd);
    if (e != cudaSuccess) return 2;
  }
  return 0;
}
