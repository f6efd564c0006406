// mla_tma.cuh -- TMA tensor maps over the paged latent KV pool and the
// shared-memory geometry of one page tile.
//
// The pool is [num_slots, 576] ([VRAM-KV]/[VRAM-POOL] in include/
// mla_decode.h): a page of 64 consecutive slots is fetched as boxes of 64 rows
// x 128 bytes with the 128-byte swizzle, so one box holds 64 tokens x 64 BF16
// elements (or 128 E4M3 bytes).  A BF16 page is 9 boxes (576 = 9 x 64), an
// FP8 page 5 boxes (the fifth half out of bounds, filled with zeros by TMA).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "mla_internal.h"

namespace mla {

constexpr int kBoxRows = MLA_PAGE_SIZE;        // tokens per box (one page)
constexpr int kBoxBytes = kBoxRows * 128;      // 8 KB per box
constexpr int kBf16BoxesPerPage = MLA_ROW_DIM / 64;           // 9
constexpr int kFp8BoxesPerPage = (MLA_ROW_DIM + 127) / 128;   // 5

// Byte offset of 16-byte chunk `j` (0..7) of row `r` inside one swizzled box.
__host__ __device__ constexpr uint32_t box_chunk_offset(uint32_t r, uint32_t j) {
  return r * 128u + ((j ^ (r & 7u)) << 4);
}

// Build the tensor map of a KV pool; returns MLA_OK or an error code.
int make_kv_tensor_map(CUtensorMap* map, const void* kv, mla_kv_dtype dtype,
                       int64_t num_slots);

// Tensor map of a bf16 3-D array (dims innermost first, in elements; strides
// of dims 1 and 2 in bytes, multiples of 16) in boxes `box` with the
// 128-byte swizzle (box[0] * 2 bytes <= 128); out-of-range elements read as
// zeros.
int make_tensor_map_bf16_3d(CUtensorMap* map, const void* base,
                            const uint64_t dims[3], const uint64_t strides[2],
                            const uint32_t box[3]);

// Tensor maps of a launch's query rows, [B * q_len * H, 512] and [.., 64]
// bf16 (as 3-D arrays with one plane), in boxes of 64 values x min(128,
// rows) rows with the 128-byte swizzle; *box_rows receives the box height.
int make_query_maps(CUtensorMap* nope, CUtensorMap* rope, const DecodeArgs& a,
                    int* box_rows);

// Tensor map of the partial outputs, fp32 [total_rows, 512], in boxes of 32
// rows x 32 values (128 bytes) with the 128-byte swizzle: the O-CTAs' TMA
// stores.
int make_o_part_map(CUtensorMap* map, float* O_part, int64_t total_rows);

// Tensor map of an E4M3 pool in boxes of 64 rows x 64 bytes with the 64-byte
// swizzle (4 KB): the RoPE key columns 512..575 of one page, the K-major
// operand layout the FP8 decode kernel's tensor cores read for those dims.
int make_kv_tensor_map_fp8_rope(CUtensorMap* map, const void* kv,
                                int64_t num_slots);

}  // namespace mla
