// mla_combine.cu -- LSE-weighted merge of partial (O, LSE) results.
//
// [K3-MLA] (tag defined in include/mla_decode.h): dcp_lse_combine merges the
// exchanged per-shard (O, LSE) pairs by their LSE; the same merge joins the
// KV splits of one launch.  This is pure streaming work (one read of every
// partial, one bf16 write), so the kernel is shaped for HBM bandwidth: one
// to four warps per output row (mla_combine.cuh), parts read in order, no
// shared memory.
#include <cuda_bf16.h>

#include "mla_combine.cuh"
#include "mla_internal.h"

namespace {

using namespace mla;

constexpr int kWarpsPerBlock = 8;

// kWs warps per row (column slices of 512 / kWs values): with few rows the
// merge is latency-bound, and more warps keep more loads in flight.
template <int kWs, typename PartT>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    mla_lse_combine_kernel(const PartT* __restrict__ O_part,
                           const float* __restrict__ LSE_part, int P,
                           int64_t rows, __nv_bfloat16* __restrict__ out,
                           float* __restrict__ lse_out) {
  // Launched as a programmatic dependent of the partial decode: it may be
  // scheduled before that kernel ends, and waits here until it has
  // completed and its parts are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x % 32;
  const int64_t gw = (int64_t)blockIdx.x * kWarpsPerBlock + threadIdx.x / 32;
  const int64_t row = gw / kWs;
  if (row >= rows) return;
  mla::combine_row<false, kWs, PartT>(O_part, LSE_part, P, rows, row, out,
                                      lse_out, lane, (int)(gw % kWs));
}

// Warps per row for a merge of `rows` rows: as many (up to four) as keep the
// grid within about one resident wave of warps (8192); beyond that one warp
// per row already fills the GPU and more would only repeat the weights.
int warps_per_row(int64_t rows) {
  return rows * 4 <= 8192 ? 4 : (rows * 2 <= 8192 ? 2 : 1);
}

template <typename PartT>
int launch_combine(const PartT* O_part, const float* LSE_part, int num_parts,
                   int64_t rows, void* out, float* lse_out, mla_stream_t stream) {
  if (!O_part || !LSE_part || !out)
    return fail(MLA_ERR_INVALID_ARG, "O_part, LSE_part and out are required");
  if (num_parts < 1 || rows < 1)
    return fail(MLA_ERR_INVALID_ARG, "num_parts=%d rows=%lld must be >= 1",
                num_parts, (long long)rows);
  if (!aligned(O_part, 16) || !aligned(out, 16) || !aligned(LSE_part, 4) ||
      (lse_out && !aligned(lse_out, 4)))
    return fail(MLA_ERR_MISALIGNED, "O_part/out need 16-B, LSE 4-B alignment");
  const int ws = warps_per_row(rows);
  const int64_t blocks = (rows * ws + kWarpsPerBlock - 1) / kWarpsPerBlock;
  if (blocks > 0x7fffffff) return fail(MLA_ERR_INVALID_ARG, "too many rows");
  // Programmatic dependent launch: when the stream's previous kernel is a
  // partial decode (which lets its dependents be scheduled from its start),
  // this grid's launch overlaps that kernel's tail; griddepcontrol.wait in
  // the kernel keeps the order of the data.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks, 1, 1);
  cfg.blockDim = dim3(kWarpsPerBlock * 32, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = (cudaStream_t)stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  __nv_bfloat16* const o = static_cast<__nv_bfloat16*>(out);
  cudaError_t e =
      ws == 4 ? cudaLaunchKernelEx(&cfg, mla_lse_combine_kernel<4, PartT>, O_part,
                                   LSE_part, num_parts, rows, o, lse_out)
      : ws == 2 ? cudaLaunchKernelEx(&cfg, mla_lse_combine_kernel<2, PartT>, O_part,
                                     LSE_part, num_parts, rows, o, lse_out)
                : cudaLaunchKernelEx(&cfg, mla_lse_combine_kernel<1, PartT>, O_part,
                                     LSE_part, num_parts, rows, o, lse_out);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch mla_lse_combine_kernel");
  return MLA_OK;
}

}  // namespace

using namespace mla;

extern "C" int mla_lse_combine(const float* O_part, const float* LSE_part,
                               int num_parts, int64_t rows, void* out,
                               float* lse_out, mla_stream_t stream) {
  return launch_combine(O_part, LSE_part, num_parts, rows, out, lse_out, stream);
}

extern "C" int mla_lse_combine_bf16_parts(const void* O_part,
                                          const float* LSE_part, int num_parts,
                                          int64_t rows, void* out,
                                          float* lse_out, mla_stream_t stream) {
  return launch_combine(static_cast<const __nv_bfloat16*>(O_part), LSE_part,
                        num_parts, rows, out, lse_out, stream);
}
