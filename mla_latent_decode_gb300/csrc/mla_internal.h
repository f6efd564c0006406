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
  const int32_t* split_pages;  // device [V, num_splits + 1] or NULL
  float* O_part;
  float* LSE_part;
  int* status;
  cudaStream_t stream;
  // Fused combine (mla_decode): the cluster that writes the last part of a
  // (request, row unit) merges the unit's rows into out (bf16 [B*q_len*H,
  // 512]) and lse_out (fp32 or NULL), counting arrivals in counters (int32
  // [B * ceil(q_len*H / 128)], zero on entry and on exit).  NULL counters:
  // partial results only.
  void* out = nullptr;
  float* lse_out = nullptr;
  int32_t* counters = nullptr;
  // Launch order of the work units (ids (s * V + v) * U + u) or NULL for
  // increasing ids; num_work = V * num_splits * U (checked by check_work).
  const int32_t* work = nullptr;
  int num_work = 0;
  // O_part holds bf16 values (same element layout) instead of fp32.
  int o_bf16 = 0;
};

// Pages [p0, p1) of split s of a request with P pages.  With a split table
// (`row` = the request's S + 1 boundaries) the boundaries are clamped to
// [0, P] and a part with p1 <= p0 is empty; without one the pages are dealt
// uniformly, floor(s P / S) .. floor((s + 1) P / S).
__host__ __device__ inline void split_page_range(const int32_t* row, int S,
                                                 int s, int64_t P, int64_t& p0,
                                                 int64_t& p1) {
  if (row) {
    int64_t a = row[s], b = row[s + 1];
    a = a < 0 ? 0 : (a > P ? P : a);
    b = b < a ? a : (b > P ? P : b);
    p0 = a;
    p1 = b;
  } else {
    p0 = (int64_t)s * P / S;
    p1 = (int64_t)(s + 1) * P / S;
  }
}

// Host checks common to every partial-decode launch; returns MLA_OK or an
// error code with the message set.
int check_decode_args(const DecodeArgs& a);

// Host checks of a work list against the tensor-core kernel that serves
// a.kv_dtype (rows per unit 256 for BF16, 128 for FP8).
int check_work(const DecodeArgs& a);

// Launchers (defined next to their kernels).
int launch_simt(const DecodeArgs& a);
int launch_tc(const DecodeArgs& a);       // BF16 KV: 4-CTA clusters
int launch_tc_fp8(const DecodeArgs& a);   // E4M3 KV: 2-CTA clusters
int pair_slots_fp8();                     // resident 2-CTA clusters (FP8)

}  // namespace mla
