/*
 * mla_oracle.c -- fp64 CPU oracle for weight-absorbed MLA decode over a paged
 * latent KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py may load this file's library.  The
 * product path (the CUDA library under mla_latent_decode_gb300/) never links,
 * imports or calls it, and this file shares no code, header, table or helper
 * with that path.
 *
 * It is deliberately plain and slow: every output is the textbook definition
 * written out in double precision, in the natural loop order, with one
 * OpenMP loop over independent query rows (the arithmetic of a row is never
 * split, blocked or reordered).
 *
 * Sources (pages of the method, cited by title and section):
 *   [VRAM-KV]   "Resident VRAM: weights and KV cache" (zdszero.github.io,
 *               vram_persistent), section "KV 账：每 token 字节由注意力架构决定"
 *               (the KV ledger): an MLA layer stores, per token, ONE latent
 *               row of kv_lora_rank (c_kv) + qk_rope_head_dim (RoPE key)
 *               elements, with no head dimension.
 *   [VRAM-CELL] same page, section "cell_size：每 token 字节的代码形态": the MLA
 *               pool of a layer is (size + page_size, 1, kv_cache_dim), the
 *               extra page absorbing padding writes; kv_cache_dim defaults to
 *               kv_lora_rank + qk_rope_head_dim.
 *   [VRAM-R2T]  same page, sections "不按 token 线性增长的部分" and
 *               "req_to_token 的大小从哪来": req_to_token is an int32 2-D table
 *               [requests, context] mapping a request's token index to its KV
 *               slot; row 0 is a dummy row for padding.
 *   [K3-MLA]    "Kimi K3 decode on 2x8 B200: DP16 vs DP2 x DCP8"
 *               (zdszero.github.io, kimi_k3_decode_dp16_vs_dp2), section
 *               "MLA：字节守恒，但 DP16 的 kernel 被 wave 量化拖慢": every rank
 *               computes all 96 heads with replicated Q over its share of the
 *               tokens, then exchanges (O, LSE) and merges them by LSE
 *               (dcp_exchange, dcp_lse_combine).
 *   [K3-SPLIT]  same page, section "问题：同样 16 张卡、同样的并发，按什么切":
 *               the MLA latent KV is split token-interleaved, slot p on rank
 *               p % 8.
 *   [K3-INTRO]  same page, opening paragraphs: each request verifies 5 tokens
 *               per decode step (MTP verification, q_len = 5).
 *   [K3-MEM]    same page, section "显存：固定开销决定状态池有多大": q_b_proj is
 *               96 x 192 x 1536 (96 heads, qk head dim 192 = 128 nope + 64
 *               rope) and w_kc is 96 x 128 x 512 (the absorbed query is
 *               512-d), which fixes the softmax scale 1/sqrt(192).
 *
 * Readings where the pages are silent (each one is listed with the others in
 * the design notes of the repository):
 *   - seq_lens[b] counts the q_len draft tokens already written to the cache;
 *     query i of request b sees tokens t <= seq_lens[b] - q_len + i (causal
 *     among the drafts).  A kv_limit table, when given, replaces that count.
 *   - LSE is the natural-log log-sum-exp of the scaled scores.
 *   - An empty token range gives O = 0 and LSE = -inf.
 *   - FP8 rows are OCP E4M3 bytes times one fp32 scale per token (slot).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ROW_DIM = 576, NOPE_DIM = 512, ROPE_DIM = 64, VALUE_DIM = 512 };

/* bfloat16 is, by definition, the upper half of an IEEE-754 binary32: widen it
 * by shifting the 16 bits back into place (exact). */
double oracle_bf16_to_f64(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* OCP 8-bit floating point, E4M3 ("fn" variant): 1 sign bit, 4 exponent bits
 * with bias 7, 3 mantissa bits; exponent field 0 is subnormal
 * (2^-6 * m/8); no infinities; S.1111.111 is NaN; largest finite 448. */
double oracle_e4m3_to_f64(uint8_t byte) {
  int sign = (byte >> 7) & 1;
  int e = (byte >> 3) & 0xF;
  int m = byte & 0x7;
  double mag;
  if (e == 0xF && m == 0x7) return NAN;
  if (e == 0)
    mag = ldexp((double)m / 8.0, 1 - 7);
  else
    mag = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -mag : mag;
}

/* Element d of the latent row stored in KV slot `slot`, dequantised. */
static double kv_elem(const void* kv, int kv_is_fp8, const float* kv_scale,
                      int64_t slot, int d) {
  if (kv_is_fp8)
    return oracle_e4m3_to_f64(((const uint8_t*)kv)[slot * ROW_DIM + d]) *
           (double)kv_scale[slot];
  return oracle_bf16_to_f64(((const uint16_t*)kv)[slot * ROW_DIM + d]);
}

/* Number of tokens query i of request b may attend to. */
static int64_t visible_count(const int32_t* seq_lens, const int32_t* kv_limit,
                             int q_len, int b, int i) {
  int64_t L = seq_lens[b];
  int64_t n = kv_limit ? (int64_t)kv_limit[(int64_t)b * q_len + i]
                       : L - q_len + 1 + i;
  if (n > L) n = L;
  if (n < 0) n = 0;
  return n;
}

/*
 * One query row (b, i, h) over tokens [lo, hi) intersected with its visible
 * range.  Definition ([VRAM-KV], [K3-MEM], [K3-INTRO]):
 *   x      = [q_nope_absorbed[b,i,h,0:512] ; q_rope[b,i,h,0:64]]
 *   k_t    = dequant(kv[req_to_token[b,t], 0:576])
 *   s_t    = sm_scale * <x, k_t>
 *   LSE    = log(sum_t exp(s_t))
 *   O      = sum_t exp(s_t - LSE) * k_t[0:512]     (the value is c_kv)
 */
static void oracle_row(const uint16_t* q_nope, const uint16_t* q_rope,
                       const void* kv, int kv_is_fp8, const float* kv_scale,
                       const int32_t* req_to_token, int64_t r2t_stride,
                       const int32_t* seq_lens, const int32_t* kv_limit,
                       int q_len, int H, double sm_scale, int64_t row,
                       int64_t lo, int64_t hi, double* O, double* lse) {
  int64_t bi = row / H; /* (b * q_len + i) */
  int b = (int)(bi / q_len);
  int i = (int)(bi % q_len);
  double x[ROW_DIM];
  int64_t n = visible_count(seq_lens, kv_limit, q_len, b, i);
  int64_t t0 = lo < 0 ? 0 : lo;
  int64_t t1 = hi < n ? hi : n;
  int d;

  for (d = 0; d < NOPE_DIM; ++d)
    x[d] = oracle_bf16_to_f64(q_nope[row * NOPE_DIM + d]);
  for (d = 0; d < ROPE_DIM; ++d)
    x[NOPE_DIM + d] = oracle_bf16_to_f64(q_rope[row * ROPE_DIM + d]);

  for (d = 0; d < VALUE_DIM; ++d) O[d] = 0.0;
  if (t1 <= t0) {
    *lse = -INFINITY;
    return;
  }

  int64_t cnt = t1 - t0, t;
  double* s = (double*)malloc((size_t)cnt * sizeof(double));
  int64_t* slot = (int64_t*)malloc((size_t)cnt * sizeof(int64_t));
  for (t = 0; t < cnt; ++t) {
    int64_t sl = req_to_token[(int64_t)b * r2t_stride + t0 + t];
    double acc = 0.0;
    for (d = 0; d < ROW_DIM; ++d)
      acc += x[d] * kv_elem(kv, kv_is_fp8, kv_scale, sl, d);
    s[t] = sm_scale * acc;
    slot[t] = sl;
  }

  double m = -INFINITY, sum = 0.0;
  for (t = 0; t < cnt; ++t) m = s[t] > m ? s[t] : m;
  for (t = 0; t < cnt; ++t) sum += exp(s[t] - m);
  *lse = m + log(sum);

  for (t = 0; t < cnt; ++t) {
    double w = exp(s[t] - *lse);
    for (d = 0; d < VALUE_DIM; ++d)
      O[d] += w * kv_elem(kv, kv_is_fp8, kv_scale, slot[t], d);
  }
  free(s);
  free(slot);
}

/*
 * Decode the listed query rows.  row ids are r = (b * q_len + i) * H + h,
 * i.e. the flat index of the [B, q_len, H] query layout.
 *   q_nope  bf16 bits [B, q_len, H, 512]; q_rope bf16 bits [B, q_len, H, 64]
 *   kv      bf16 bits or E4M3 bytes [num_slots, 576]; kv_scale fp32 [num_slots]
 *           (read only when kv_is_fp8)
 *   req_to_token int32 [B, r2t_stride]: entry t is the slot of token t
 *   seq_lens int32 [B]; kv_limit int32 [B, q_len] or NULL (causal MTP rule)
 *   row_lo/row_hi: optional per-listed-row token range [lo, hi) (partial mode);
 *   NULL means the whole visible range.
 *   O_out  fp64 [n_rows, 512]; lse_out fp64 [n_rows]
 */
int oracle_mla_decode_rows(const uint16_t* q_nope, const uint16_t* q_rope,
                           const void* kv, int kv_is_fp8, const float* kv_scale,
                           const int32_t* req_to_token, int64_t r2t_stride,
                           const int32_t* seq_lens, const int32_t* kv_limit,
                           int B, int q_len, int H, double sm_scale,
                           const int64_t* rows, int64_t n_rows,
                           const int64_t* row_lo, const int64_t* row_hi,
                           double* O_out, double* lse_out) {
  int64_t k;
  if (B <= 0 || q_len <= 0 || H <= 0) return -1;
  for (k = 0; k < n_rows; ++k)
    if (rows[k] < 0 || rows[k] >= (int64_t)B * q_len * H) return -2;
#pragma omp parallel for schedule(dynamic, 1)
  for (k = 0; k < n_rows; ++k) {
    int64_t lo = row_lo ? row_lo[k] : 0;
    int64_t hi = row_hi ? row_hi[k] : INT64_MAX;
    oracle_row(q_nope, q_rope, kv, kv_is_fp8, kv_scale, req_to_token,
               r2t_stride, seq_lens, kv_limit, q_len, H, sm_scale, rows[k], lo,
               hi, O_out + k * VALUE_DIM, lse_out + k);
  }
  return 0;
}

/*
 * LSE-weighted merge of P partial results ([K3-MLA]: dcp_lse_combine merges
 * the exchanged (O, LSE) pairs by their LSE):
 *   M = max_j LSE_j, w_j = exp(LSE_j - M),
 *   out = sum_j w_j O_j / sum_j w_j,  lse = M + log(sum_j w_j).
 * A part with LSE = -inf has weight 0 and is left out of both sums (its O is
 * never read); if every part is empty the output is O = 0, LSE = -inf.
 *   O_parts fp64 [P, rows, 512]; lse_parts fp64 [P, rows]
 */
void oracle_lse_combine(const double* O_parts, const double* lse_parts, int P,
                        int64_t rows, double* out, double* lse_out) {
  int64_t r;
#pragma omp parallel for schedule(static)
  for (r = 0; r < rows; ++r) {
    double M = -INFINITY, W = 0.0;
    int j, d;
    for (j = 0; j < P; ++j) {
      double l = lse_parts[(int64_t)j * rows + r];
      M = l > M ? l : M;
    }
    for (d = 0; d < VALUE_DIM; ++d) out[r * VALUE_DIM + d] = 0.0;
    if (M == -INFINITY) {
      lse_out[r] = -INFINITY;
      continue;
    }
    for (j = 0; j < P; ++j) {
      double l = lse_parts[(int64_t)j * rows + r];
      double w;
      if (l == -INFINITY) continue; /* empty part: weight 0, not added */
      w = exp(l - M);
      W += w;
      for (d = 0; d < VALUE_DIM; ++d)
        out[r * VALUE_DIM + d] +=
            w * O_parts[((int64_t)j * rows + r) * VALUE_DIM + d];
    }
    for (d = 0; d < VALUE_DIM; ++d) out[r * VALUE_DIM + d] /= W;
    lse_out[r] = M + log(W);
  }
}

/*
 * Page-table gather ([VRAM-R2T]): copy the raw bytes of token t's row,
 * kv[req_to_token[b, t]], for t < seq_lens[b], request after request, into a
 * dense [sum_b seq_lens[b], 576] array.  elem_bytes is 2 (bf16) or 1 (fp8).
 */
void oracle_gather(const uint8_t* kv, int elem_bytes,
                   const int32_t* req_to_token, int64_t r2t_stride,
                   const int32_t* seq_lens, int B, uint8_t* out) {
  int64_t row_bytes = (int64_t)ROW_DIM * elem_bytes, o = 0;
  int b;
  for (b = 0; b < B; ++b) {
    int64_t t;
    for (t = 0; t < seq_lens[b]; ++t, ++o) {
      int64_t slot = req_to_token[(int64_t)b * r2t_stride + t];
      memcpy(out + o * row_bytes, kv + slot * row_bytes, (size_t)row_bytes);
    }
  }
}

/* Nearest E4M3 code to a binary32 value v (round to nearest, ties to the
 * code with an even mantissa field, i.e. an even code), saturated to the
 * largest finite magnitude 448; the sign bit is v's (so -0.0 gives 0x80).
 * The definition written out: every finite non-negative code 0x00..0x7E is
 * tried.  v must not be NaN. */
uint8_t oracle_f32_to_e4m3(float v) {
  const double a = fabs((double)v);
  int best = 0;
  double best_d = INFINITY;
  for (int c = 0; c <= 0x7E; ++c) {
    const double d = fabs(oracle_e4m3_to_f64((uint8_t)c) - a);
    if (d < best_d || (d == best_d && (c & 1) == 0)) {
      best_d = d;
      best = c;
    }
  }
  if (a > 448.0) best = 0x7E;
  return (uint8_t)(best | (signbit(v) ? 0x80 : 0));
}

/* The FP8 cache write: quantise n latent rows (binary32 values, here the
 * bf16 rows widened exactly) to E4M3 codes with one fp32 scale per row
 * (the per-token scale of the FP8 KV format; the reading taken for its
 * quantiser is scale = amax / 448 with round-to-nearest codes):
 *   scale_r   = fl32(max_d |x_rd| / 448)     (one binary32 division)
 *   code_rd   = E4M3(fl32(x_rd / scale_r))  (one binary32 division, then the
 *               rounding above); an all-zero row gets scale 0 and codes 0.
 * Rows must be finite. */
void oracle_kv_quantize(const float* rows, int64_t n, uint8_t* codes,
                        float* scales) {
  for (int64_t r = 0; r < n; ++r) {
    const float* x = rows + r * ROW_DIM;
    float amax = 0.f;
    for (int d = 0; d < ROW_DIM; ++d)
      if (fabsf(x[d]) > amax) amax = fabsf(x[d]);
    const float scale = amax / 448.0f;
    scales[r] = scale;
    for (int d = 0; d < ROW_DIM; ++d) {
      if (scale == 0.f) {
        codes[r * ROW_DIM + d] = 0;
      } else {
        const float q = x[d] / scale;
        codes[r * ROW_DIM + d] = oracle_f32_to_e4m3(q);
      }
    }
  }
}

/* Threads the OpenMP loops above will use (reported by the CPU baseline). */
int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
