// mla_gather.cu -- KV tensor maps and the page-table gather through them.
//
// mla_debug_gather copies every live token row of every request into a
// dense array using exactly the decode kernel's load path: the first page
// table entry of a page gives its base slot ([VRAM-POOL] in
// include/mla_decode.h), and the page arrives as 128-byte-swizzled TMA boxes.
// The bit-exact comparison of its output with a CPU gather therefore checks
// the page addressing and the swizzle arithmetic the decode kernel uses.
#include <cudaTypedefs.h>

#include <mutex>

#include "mla_tma.cuh"
#include "ptx_sm103.cuh"

namespace mla {

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

int make_kv_tensor_map(CUtensorMap* map, const void* kv, mla_kv_dtype dtype,
                       int64_t num_slots) {
  auto fn = encode_fn();
  if (!fn) return fail(MLA_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  const bool fp8 = dtype == MLA_KV_FP8_E4M3;
  cuuint64_t dims[2] = {(cuuint64_t)MLA_ROW_DIM, (cuuint64_t)num_slots};
  cuuint64_t strides[1] = {(cuuint64_t)MLA_ROW_DIM * (fp8 ? 1 : 2)};
  cuuint32_t box[2] = {fp8 ? 128u : 64u, (cuuint32_t)kBoxRows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map,
                  fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                      : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                  2, const_cast<void*>(kv), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MLA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return MLA_OK;
}

int make_tensor_map_bf16_3d(CUtensorMap* map, const void* base,
                            const uint64_t dims[3], const uint64_t strides[2],
                            const uint32_t box[3]) {
  auto fn = encode_fn();
  if (!fn) return fail(MLA_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
  cuuint64_t st[2] = {strides[0], strides[1]};
  cuuint32_t bx[3] = {box[0], box[1], box[2]};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                  const_cast<void*>(base), d, st, bx, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MLA_ERR_CUDA, "cuTensorMapEncodeTiled (3-D bf16) failed (%d)",
                (int)r);
  return MLA_OK;
}

int make_o_part_map(CUtensorMap* map, float* O_part, int64_t total_rows) {
  auto fn = encode_fn();
  if (!fn) return fail(MLA_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  cuuint64_t dims[2] = {(cuuint64_t)MLA_VALUE_DIM, (cuuint64_t)total_rows};
  cuuint64_t strides[1] = {(cuuint64_t)MLA_VALUE_DIM * 4};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, O_part, dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MLA_ERR_CUDA, "cuTensorMapEncodeTiled (O_part) failed (%d)",
                (int)r);
  return MLA_OK;
}

int make_query_maps(CUtensorMap* nope, CUtensorMap* rope, const DecodeArgs& a,
                    int* box_rows) {
  const uint64_t rows = (uint64_t)a.B * a.q_len * a.H;
  *box_rows = (int)(rows < 128 ? rows : 128);
  const uint32_t box[3] = {64, (uint32_t)*box_rows, 1};
  const uint64_t dn[3] = {(uint64_t)MLA_NOPE_DIM, rows, 1};
  const uint64_t sn[2] = {(uint64_t)MLA_NOPE_DIM * 2, rows * MLA_NOPE_DIM * 2};
  int rc = make_tensor_map_bf16_3d(nope, a.q_nope, dn, sn, box);
  if (rc != MLA_OK) return rc;
  const uint64_t dr[3] = {(uint64_t)MLA_ROPE_DIM, rows, 1};
  const uint64_t sr[2] = {(uint64_t)MLA_ROPE_DIM * 2, rows * MLA_ROPE_DIM * 2};
  return make_tensor_map_bf16_3d(rope, a.q_rope, dr, sr, box);
}

int make_kv_tensor_map_fp8_rope(CUtensorMap* map, const void* kv,
                                int64_t num_slots) {
  auto fn = encode_fn();
  if (!fn) return fail(MLA_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  cuuint64_t dims[2] = {(cuuint64_t)MLA_ROW_DIM, (cuuint64_t)num_slots};
  cuuint64_t strides[1] = {(cuuint64_t)MLA_ROW_DIM};
  cuuint32_t box[2] = {(cuuint32_t)MLA_ROPE_DIM, (cuuint32_t)kBoxRows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(kv),
                  dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MLA_ERR_CUDA, "cuTensorMapEncodeTiled (fp8 rope) failed (%d)",
                (int)r);
  return MLA_OK;
}

namespace {

constexpr int kGatherThreads = 128;
constexpr int kGatherSmem = kBf16BoxesPerPage * kBoxBytes + 1024;

__global__ void __launch_bounds__(kGatherThreads)
    mla_gather_kernel(const __grid_constant__ CUtensorMap kv_map, int fp8,
                      int64_t num_slots, const int32_t* __restrict__ r2t,
                      int64_t stride, const int32_t* __restrict__ seq_lens,
                      const int64_t* __restrict__ row_offset,
                      int pages_per_req, uint8_t* __restrict__ out,
                      int* status) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  uint8_t* tile = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int v = blockIdx.x / pages_per_req;
  const int page = blockIdx.x % pages_per_req;
  int64_t L = seq_lens[v];
  L = L > stride ? stride : (L < 0 ? 0 : L);
  const int64_t t0 = (int64_t)page * kBoxRows;
  if (t0 >= L) return;
  const int rows = (int)((L - t0) < kBoxRows ? (L - t0) : kBoxRows);
  const int64_t base = r2t[(int64_t)v * stride + t0];
  const bool ok = base >= 0 && base % kBoxRows == 0 && base + kBoxRows <= num_slots;
  const int boxes = fp8 ? kFp8BoxesPerPage : kBf16BoxesPerPage;
  const uint32_t row_bytes = MLA_ROW_DIM * (fp8 ? 1 : 2);
  uint8_t* dst_rows = out + (row_offset[v] + t0) * row_bytes;

  if (!ok) {  // report, and write zeros so the output stays deterministic
    if (threadIdx.x == 0 && status) atomicOr(status, MLA_STATUS_BAD_SLOT);
    for (uint32_t k = threadIdx.x; k < rows * row_bytes / 16; k += blockDim.x)
      reinterpret_cast<uint4*>(dst_rows)[k] = make_uint4(0, 0, 0, 0);
    return;
  }

  const uint32_t bar_a = ptx::smem_u32(&bar);
  if (threadIdx.x == 0) {
    abort_flag = 0;
    ptx::mbar_init(bar_a, 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    ptx::mbar_arrive_expect_tx(bar_a, boxes * kBoxBytes);
    for (int c = 0; c < boxes; ++c)
      ptx::tma_load_2d(ptx::smem_u32(tile + c * kBoxBytes), &kv_map, bar_a,
                       c * (fp8 ? 128 : 64), (int32_t)base);
  }
  if (!ptx::mbar_wait(bar_a, 0, &abort_flag)) {
    if (status) atomicOr(status, MLA_STATUS_WAIT_TIMEOUT);
    abort_flag = 1;
    return;
  }
  // Un-swizzle: 16-byte chunk k of row r lives in box k/8, chunk k%8.
  const uint32_t chunks = row_bytes / 16;
  for (uint32_t idx = threadIdx.x; idx < rows * chunks; idx += blockDim.x) {
    const uint32_t r = idx / chunks, k = idx % chunks;
    const uint4 val = *reinterpret_cast<const uint4*>(
        tile + (k / 8) * kBoxBytes + box_chunk_offset(r, k % 8));
    reinterpret_cast<uint4*>(dst_rows + (size_t)r * row_bytes)[k] = val;
  }
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" int mla_debug_gather(const void* kv_pages, mla_kv_dtype kv_dtype,
                                int64_t num_slots, const int32_t* req_to_token,
                                int64_t r2t_stride, const int32_t* seq_lens,
                                const int64_t* row_offset, int V,
                                int page_size, void* dense_out,
                                mla_stream_t stream) {
  if (!kv_pages || !req_to_token || !seq_lens || !row_offset || !dense_out ||
      V < 1 || r2t_stride < 1)
    return fail(MLA_ERR_INVALID_ARG, "bad gather arguments");
  if (page_size != MLA_PAGE_SIZE)
    return fail(MLA_ERR_UNSUPPORTED, "page_size must be %d", MLA_PAGE_SIZE);
  if (kv_dtype != MLA_KV_BF16 && kv_dtype != MLA_KV_FP8_E4M3)
    return fail(MLA_ERR_INVALID_ARG, "unknown kv_dtype");
  if (num_slots < MLA_PAGE_SIZE || num_slots > ((int64_t)1 << 31) - 1)
    return fail(MLA_ERR_INVALID_ARG, "num_slots out of range");
  if (!aligned(kv_pages, 16) || !aligned(dense_out, 16))
    return fail(MLA_ERR_MISALIGNED, "kv_pages and dense_out need 16-B alignment");
  CUtensorMap map;
  int rc = make_kv_tensor_map(&map, kv_pages, kv_dtype, num_slots);
  if (rc != MLA_OK) return rc;
  const int64_t ppr = (r2t_stride + MLA_PAGE_SIZE - 1) / MLA_PAGE_SIZE;
  const int64_t grid = ppr * V;
  if (grid > 0x7fffffff) return fail(MLA_ERR_INVALID_ARG, "grid too large");
  cudaError_t e = cudaFuncSetAttribute(
      mla_gather_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
      kGatherSmem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(gather)");
  mla_gather_kernel<<<(unsigned)grid, kGatherThreads, kGatherSmem,
                      (cudaStream_t)stream>>>(
      map, kv_dtype == MLA_KV_FP8_E4M3, num_slots, req_to_token, r2t_stride,
      seq_lens, row_offset, (int)ppr, static_cast<uint8_t*>(dense_out),
      nullptr);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch mla_gather_kernel");
  return MLA_OK;
}
