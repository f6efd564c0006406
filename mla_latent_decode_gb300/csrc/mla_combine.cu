// mla_combine.cu -- LSE-weighted merge of partial (O, LSE) results.
//
// [K3-MLA] (tag defined in include/mla_decode.h): dcp_lse_combine merges the
// exchanged per-shard (O, LSE) pairs by their LSE; the same merge joins the
// KV splits of one launch.  This is pure streaming work (one read of every
// partial, one bf16 write), so the kernel is shaped for HBM bandwidth: one
// warp per output row (mla_combine.cuh), parts read in order, no shared
// memory.
#include <cuda_bf16.h>

#include "mla_combine.cuh"
#include "mla_internal.h"

namespace {

constexpr int kWarpsPerBlock = 8;

__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    mla_lse_combine_kernel(const float* __restrict__ O_part,
                           const float* __restrict__ LSE_part, int P,
                           int64_t rows, __nv_bfloat16* __restrict__ out,
                           float* __restrict__ lse_out) {
  const int lane = threadIdx.x % 32;
  const int64_t row = (int64_t)blockIdx.x * kWarpsPerBlock + threadIdx.x / 32;
  if (row >= rows) return;
  mla::combine_row<false>(O_part, LSE_part, P, rows, row, out, lse_out, lane);
}

}  // namespace

using namespace mla;

extern "C" int mla_lse_combine(const float* O_part, const float* LSE_part,
                               int num_parts, int64_t rows, void* out,
                               float* lse_out, mla_stream_t stream) {
  if (!O_part || !LSE_part || !out)
    return fail(MLA_ERR_INVALID_ARG, "O_part, LSE_part and out are required");
  if (num_parts < 1 || rows < 1)
    return fail(MLA_ERR_INVALID_ARG, "num_parts=%d rows=%lld must be >= 1",
                num_parts, (long long)rows);
  if (!aligned(O_part, 16) || !aligned(out, 16) || !aligned(LSE_part, 4) ||
      (lse_out && !aligned(lse_out, 4)))
    return fail(MLA_ERR_MISALIGNED, "O_part/out need 16-B, LSE 4-B alignment");
  const int64_t blocks = (rows + kWarpsPerBlock - 1) / kWarpsPerBlock;
  if (blocks > 0x7fffffff) return fail(MLA_ERR_INVALID_ARG, "too many rows");
  mla_lse_combine_kernel<<<(unsigned)blocks, kWarpsPerBlock * 32, 0,
                           (cudaStream_t)stream>>>(
      O_part, LSE_part, num_parts, rows, static_cast<__nv_bfloat16*>(out),
      lse_out);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch mla_lse_combine_kernel");
  return MLA_OK;
}
