// mla_internal.h -- shared host-side helpers of the MLA decode library
// (error reporting and argument checks used by every entry point).
#pragma once

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <string>

#include <cuda_runtime.h>

#include "../../include/mla_decode.h"

namespace mla {

// Thread-local last error message, returned by mla_last_error_string().
std::string& last_error();

// Record a message and return `code` (so call sites can `return fail(...)`).
int fail(int code, const char* fmt, ...);

inline bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

inline int cuda_fail(cudaError_t e, const char* what) {
  return fail(MLA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Arguments shared by the two partial-decode entry points.
struct DecodeArgs {
  const void* q_nope;
  const void* q_rope;
  const void* kv;
  const float* kv_scale;
  mla_kv_dtype kv_dtype;
  int64_t num_slots;
  const int32_t* req_to_token;
  int64_t r2t_stride;
  const int32_t* seq_lens;
  const int32_t* kv_limit;
  int B, q_len, H, num_shards, page_size;
  float sm_scale;
  int num_splits;
  float* O_part;
  float* LSE_part;
  int* status;
  cudaStream_t stream;
};

// Host checks common to every partial-decode launch; returns MLA_OK or an
// error code with the message set.
int check_decode_args(const DecodeArgs& a);

// Launchers (defined next to their kernels).
int launch_simt(const DecodeArgs& a);
int launch_tc(const DecodeArgs& a);       // BF16 KV: 4-CTA clusters
int launch_tc_fp8(const DecodeArgs& a);   // E4M3 KV: 2-CTA clusters
int pair_slots_fp8();                     // resident 2-CTA clusters (FP8)

}  // namespace mla
