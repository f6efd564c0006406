// mla_scratch.cu -- the fused decode with its workspace in the library's own
// static device memory: an entry point that allocates nothing.
//
// mla_decode needs three scratch arrays besides its inputs and outputs: the
// arrival counters of the fused combine and the per-part (O, LSE) results.
// mla_decode_scratch takes them from one static __device__ array (256-byte
// aligned, MLA_SCRATCH_BYTES), whose device address is looked up once per
// device with cudaGetSymbolAddress; no cudaMalloc or cudaFree is ever made.
// Every call clears the counters on its stream before the decode
// (cudaMemsetAsync on the array's address, no allocation): a call that left
// them non-zero (a work list naming no unit, or one unit twice) cannot
// offset a later call's counts.  The array is one per device and process:
// calls that may overlap on a device race on it (see include/mla_decode.h).
#include <mutex>

#include "mla_internal.h"

namespace mla {
namespace {

__device__ __align__(256) uint8_t g_scratch[MLA_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

int64_t round256(int64_t x) { return (x + 255) & ~(int64_t)255; }

// Device address of g_scratch on the current device, looked up on the first
// call made with that device current and kept for the life of the process
// (a cudaDeviceReset reloads the device code, after which the kept address
// is stale: such a process must not call mla_decode_scratch on that device
// again).
int scratch_base(void** base) {
  static std::mutex mu;
  static void* cache[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices)
    return fail(MLA_ERR_UNSUPPORTED, "device %d beyond the scratch table", dev);
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(scratch)");
    cache[dev] = p;
  }
  *base = cache[dev];
  return MLA_OK;
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" {

int64_t mla_scratch_bytes(int B, int q_len, int H, int num_shards,
                          int num_splits) {
  if (B < 1 || q_len < 1 || H < 1 || num_shards < 1 || num_splits < 1)
    return fail(MLA_ERR_INVALID_ARG,
                "B=%d q_len=%d H=%d num_shards=%d num_splits=%d must be >= 1",
                B, q_len, H, num_shards, num_splits);
  const int64_t rows = (int64_t)B * q_len * H;
  const int64_t parts = (int64_t)num_shards * num_splits;
  const int64_t counters = (int64_t)B * ((q_len * H + 127) / 128) * 4;
  return round256(counters) + round256(parts * rows * 4) +
         round256(parts * rows * MLA_VALUE_DIM * 4);
}

int mla_decode_scratch(const void* q_nope_absorbed, const void* q_rope,
                       const void* kv_pages, const float* kv_scale,
                       mla_kv_dtype kv_dtype, int64_t num_slots,
                       const int32_t* req_to_token, int64_t r2t_stride,
                       const int32_t* seq_lens, const int32_t* kv_limit, int B,
                       int q_len, int H, int num_shards, int page_size,
                       float sm_scale, int num_splits,
                       const int32_t* split_pages, const int32_t* work,
                       int num_work, void* out, float* lse_out, int* status,
                       mla_stream_t stream) {
  // The size limit is checked before anything else, so an oversized request
  // fails here whatever else is wrong with it.
  const int64_t need = mla_scratch_bytes(B, q_len, H, num_shards, num_splits);
  if (need < 0) return (int)need;
  if (need > (int64_t)MLA_SCRATCH_BYTES)
    return fail(MLA_ERR_SCRATCH,
                "this call needs %lld bytes of scratch (counters and %d x %lld "
                "partial rows); the library's static scratch holds %lld "
                "(MLA_SCRATCH_BYTES): use fewer splits or mla_decode with "
                "caller workspace",
                (long long)need, num_shards * num_splits,
                (long long)B * q_len * H, (long long)MLA_SCRATCH_BYTES);
  // The other arguments as mla_decode checks them (the workspace stands in
  // as an aligned placeholder), before any CUDA call.
  float* const placeholder = reinterpret_cast<float*>((uintptr_t)256);
  DecodeArgs a{q_nope_absorbed, q_rope,    kv_pages, kv_scale,  kv_dtype,
               num_slots,       req_to_token, r2t_stride, seq_lens, kv_limit,
               B,               q_len,     H,        num_shards, page_size,
               sm_scale,        num_splits, split_pages, placeholder,
               placeholder,     status,    (cudaStream_t)stream};
  a.work = work;
  a.num_work = num_work;
  int rc = check_decode_args(a);
  if (rc != MLA_OK) return rc;
  rc = check_work(a);
  if (rc != MLA_OK) return rc;
  if (!out) return fail(MLA_ERR_INVALID_ARG, "out is required");
  void* base = nullptr;
  rc = scratch_base(&base);
  if (rc != MLA_OK) return rc;
  const int64_t rows = (int64_t)B * q_len * H;
  const int64_t parts = (int64_t)num_shards * num_splits;
  uint8_t* p = static_cast<uint8_t*>(base);
  int32_t* counters = reinterpret_cast<int32_t*>(p);
  const int64_t counter_bytes = (int64_t)B * ((q_len * H + 127) / 128) * 4;
  cudaError_t e = cudaMemsetAsync(counters, 0, (size_t)counter_bytes,
                                  (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(scratch counters)");
  p += round256(counter_bytes);
  float* LSE_part = reinterpret_cast<float*>(p);
  p += round256(parts * rows * 4);
  float* O_part = reinterpret_cast<float*>(p);
  return mla_decode(q_nope_absorbed, q_rope, kv_pages, kv_scale, kv_dtype,
                    num_slots, req_to_token, r2t_stride, seq_lens, kv_limit, B,
                    q_len, H, num_shards, page_size, sm_scale, num_splits,
                    split_pages, work, num_work, O_part, LSE_part, counters, out,
                    lse_out, status, stream);
}

}  // extern "C"
