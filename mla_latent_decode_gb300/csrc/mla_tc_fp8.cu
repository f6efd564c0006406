// mla_tc_fp8.cu -- tensor-core partial MLA decode over an FP8 (E4M3) KV
// cache with one fp32 scale per token, on FP8 tensor-core MMAs.
//
// Same computation as the BF16 path (include/mla_decode.h,
// mla_decode_partial; [VRAM-KV], [K3-MLA], [K3-SPLIT], [K3-INTRO]) with
// k_t = e4m3(byte) * kv_scale[slot].
//
// Design (GB300, clusters of two CTAs, one CTA per SM):
//   The KV bytes go from TMA straight into the operand layout of
//   tcgen05.mma.kind::f8f6f4, untouched: K tiles K-major with the 128-byte
//   swizzle (dims 0..511) and the 64-byte swizzle (the 64 RoPE dims), V tiles
//   MN-major with the 128-byte swizzle.  The other operand of each product is
//   split in two 8-bit parts so that the result keeps the precision of the
//   BF16 path:
//   * Q (bf16) = 2^e (Qhi + Qlo), Qhi = e4m3(Q 2^-e), Qlo = e4m3(Q 2^-e - Qhi),
//     with a power-of-two row scale 2^e that puts the row's largest |Q| in
//     [128, 256).  A bf16 value has 8 significant bits; Qhi holds 4 and the
//     remainder is exact in Qlo for every element at least 2^-9 of the row's
//     largest; a smaller one is off by at most 2^-17 of it (E4M3's smallest
//     step, 2^-9, is the floor).  So q . k = 2^e (Qhi . k + Qlo . k): two
//     MMAs into one fp32 accumulator.  A row whose elements span more than
//     2^9 therefore carries score errors up to sm_scale * 2^-17 * max|q| *
//     sum|k| (a bound, reached only by aligned errors).
//   * The token's scale moves from V to P: P' = p * scale_t * 2^g = Phi +
//     Plo, Phi = e4m3(P'), Plo = e5m2(P' - Phi) (E5M2's wider exponent keeps
//     the small remainders), at most 2^-7 relative error per element, like a
//     bf16 P.  P' . e4m3(V) = (Phi + Plo) . e4m3(V): two MMAs.  The S-CTA
//     ships p as f16 together with the page's f16 factors scale_t * 2^g, and
//     four packer warps of the O-CTA (each owns a row) form P' and split it:
//     the per-token factors and the 8-bit conversions stay off the softmax.
//   Each product thus takes two 8-bit MMAs, as long as one 16-bit MMA, and
//   the tensor cores read the E4M3 bytes with no conversion pass.
//   * A query element far above the rest of its row (beyond 32x the row's
//     mean |q|: an outlier channel) would set the row scale and push the
//     small elements under the split's floor.  Such channels (up to 4 per
//     128-row group, shared by the group's rows) are left out of Qhi/Qlo;
//     an idle warp copies their E4M3 key bytes out of each ring stage before
//     the stage is released, and the softmax adds q_c * k8_t,c to the raw
//     score in fp32 (exact: 8 x 4 significant bits).  The split exponent
//     then comes from the remaining elements.
//   Rank 0 (S-CTA) holds Qhi/Qlo (TMEM columns [0, 256) for the 512 c_kv
//   dims, shared memory for the 64 RoPE dims), split from query rows that
//   TMA brings into the still idle ring, and one 256-column S tile; rank 1
//   (O-CTA) holds O (128 rows x 512 fp32 = all 512 TMEM columns) and writes
//   O_part through the idle ring in full 128-byte lines.
//   g is the exponent with max|scale| 2^g in [0.5, 1) over the tokens seen
//   so far (a scale warp tracks it per tile), so P' <= p <= 2^8 stays inside
//   E4M3's range whatever the scales' magnitude; O is kept in units of
//   2^(m_ref - g), l in units of 2^m_ref.  Every wait is bounded
//   (ptx_sm103.cuh).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "mla_combine.cuh"
#include "mla_tma.cuh"
#include "ptx_sm103.cuh"

namespace mla {
namespace {

using namespace ptx;

constexpr int kThreads = 640;        // 20 warps = 5 warpgroups
constexpr int kStages = 4;           // operand ring slots
constexpr int kStageBytes = 32768;   // S: 4 pages x 128 dims; O: one page of V
constexpr int kBlocksPerTile = 5;    // S tile: 4 blocks of 128 dims + RoPE
constexpr int kRopeBoxBytes = MLA_PAGE_SIZE * MLA_ROPE_DIM;  // 4 KB
constexpr int kTilePages = 4;        // pages per S tile (N <= 256)
constexpr int kNP = 4;               // P message slots (page index mod 4)
constexpr int kRows = 128;           // query rows per CTA pair
constexpr int kPage = MLA_PAGE_SIZE;      // 64 tokens
constexpr int kPBytes = kRows * 128;      // per row: 64 f16 p, then Phi | Plo
constexpr int kAlphaOff = kPBytes;        // float alpha[128]
constexpr int kFlagOff = kPBytes + kRows * 4;  // uint32 flags[4]
constexpr int kSGOff = kFlagOff + 16;          // f16 scale * 2^g of 64 tokens
constexpr int kPMsgBytes = kSGOff + 128;       // 17040 = 1065 x 16
constexpr int kPSlotStride = 17408;            // 17 KB, 1024-aligned
constexpr uint32_t kQLoCol = 128;   // Qlo columns (Qhi at 0)
constexpr uint32_t kSCol0 = 256;    // S buffer columns
constexpr float kTau = 8.f;         // lazy-rescale threshold (log2 units)
constexpr uint32_t kFull = 0xffffffffu;
constexpr int kPartials = 8;         // 32-token groups of an S tile
// Query exceptions: elements above kExcRatio x their row's mean |q| leave the
// two-part E4M3 split (whose exponent they would otherwise set) for an exact
// fp32 path; a 128-row group takes up to kExc such channels.
constexpr int kExc = 4;
constexpr float kExcRatio = 32.f;
// Register split of the S-CTA (setmaxnreg): 640 threads launch with 96
// registers each (61,440 of 65,536); the producer/MMA/scale warpgroup (warps
// 0-3) gives registers away so the four softmax warpgroups can hold their
// scores.  The split is one-way.
constexpr int kRegsLaunch = 96;
constexpr int kRegsControl = 40;
constexpr int kRegsSoftmax = 104;
static_assert(128 * kRegsControl + 512 * kRegsSoftmax <= kThreads * kRegsLaunch,
              "register split exceeds the launch allocation");

// kind::f8f6f4 instruction descriptor: fp32 accumulator, A format a_fmt
// (0 = E4M3, 1 = E5M2), B E4M3, A K-major, B K- or MN-major.
__host__ __device__ constexpr uint32_t idesc_f8(int M, int N, uint32_t a_fmt,
                                               bool b_mn) {
  return (1u << 4) | (a_fmt << 7) | ((b_mn ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__host__ __device__ constexpr uint32_t idesc_s(int pages) {
  return idesc_f8(128, 64 * pages, 0u, false);
}
constexpr uint32_t kIdescOHi = idesc_f8(128, 256, 0u, true);  // Phi: E4M3
constexpr uint32_t kIdescOLo = idesc_f8(128, 256, 1u, true);  // Plo: E5M2

struct __align__(1024) Smem {
  uint8_t ring[kStages][kStageBytes];       // 128 KB operand ring
  uint8_t qrope[2][kRows * MLA_ROPE_DIM];   // S-CTA: Qhi, Qlo RoPE (64-B swizzle)
  float tscale[4][kTilePages * kPage];      // S-CTA: token scales of tile j % 4
  uint8_t pslot[kNP][kPSlotStride];
  uint32_t tsg[4][kTilePages * kPage / 2];  // S-CTA: f16 pairs scale * 2^g
  int tg[4];                // S-CTA: scale exponent g of tile j % 4
  union {
    float fin[kRows];              // 1 / l per row (after the tile loop)
    uint16_t xe[kRows][kExc];      // S-CTA: bf16 q of the exception channels
  };
  float xch[kPartials][kRows];  // S-CTA: row values per 32-token group
  uint8_t xk[2][kExc][kTilePages * kPage];  // S-CTA: E4M3 K bytes of the
                                            // exception channels, tile j % 2
  int xtab[kExc];           // S-CTA: the group's exception channels (-1: none)
  uint64_t full[kStages];   // TMA -> MMA (bytes)
  uint64_t empty[kStages];  // MMA -> producer
  uint64_t scfull[4];       // S-CTA: scale bulk copies landed
  uint64_t scempty[4];      // S-CTA: softmax done with tscale[j % 4]
  uint64_t tsready[4];      // S-CTA: tscale, tsg, tg of tile j % 4 written
  uint64_t sfull, sempty;
  uint64_t pfull[kNP];
  uint64_t packed[kNP];     // O-CTA: P' of slot k split into Phi | Plo
  uint64_t pempty[kNP];
  uint64_t drain, corr_done, fin_full, qready, tail_go, tail_ready;
  uint64_t xkfull[2];       // S-CTA: exception K bytes of tile j % 2 copied
  uint64_t xkempty[2];      // S-CTA: the softmax warps done with them
  uint64_t qbar;            // S-CTA: the query boxes landed
  uint32_t tmem_base;
  int abort_flag;
  int ctl_slot;
  int ctl_final;
  int ctl_last;  // fused combine: this cluster wrote the unit's last part
};
constexpr int kSmemBytes = (int)sizeof(Smem) + 1024;
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
static_assert(kPMsgBytes % 16 == 0, "bulk copy size");
static_assert(kTilePages * kBoxBytes == kStageBytes, "S stage = 4 pages");
static_assert(4 * kBoxBytes == kStageBytes, "O stage = one page of V");

struct TcParams {
  const uint4* q_nope;     // bf16 [B, q_len, H, 512] as 16-B chunks
  const uint4* q_rope;     // bf16 [B, q_len, H, 64]
  const float* kv_scale;   // fp32 [num_slots]
  int64_t num_slots;
  const int32_t* r2t;
  int64_t r2t_stride;
  const int32_t* seq_lens;
  const int32_t* kv_limit;
  const int32_t* split_pages;  // [V, num_splits + 1] page boundaries or NULL
  const int32_t* work;         // unit ids in launch order or NULL
  int units;                   // V * num_splits * G
  int B, q_len, H, V, num_splits, G;
  float scale_log2;        // sm_scale * log2(e)
  float* O_part;           // fp32, or bf16 when o_bf16
  int o_bf16;
  float* LSE_part;
  int* status;
  int q_box_rows;          // rows of a query TMA box: min(128, B * q_len * H)
  __nv_bfloat16* out;      // fused combine (NULL counters: partials only)
  float* lse_out;
  int* counters;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// F with x in [2^(F-1), 2^F) for a positive finite x (a subnormal x counts
// as 2^-126).
__device__ __forceinline__ int exponent_of(float x) {
  const int f = (int)((__float_as_uint(x) >> 23) & 0xFFu);
  return (f == 0 ? 1 : f) - 126;
}

// 2^k as a float, k in [-126, 127].
__device__ __forceinline__ float exp2i(int k) {
  return __int_as_float((k + 127) << 23);
}

// Three-operand maximum (one ALU instruction on sm_100 and later).
__device__ __forceinline__ float max3(float a, float b, float c) {
  float y;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
  return y;
}

// Packed pair arithmetic: two fp32 lanes per instruction.
__device__ __forceinline__ uint64_t f2pack(float a, float b) {
  uint64_t x;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a), "f"(b));
  return x;
}
__device__ __forceinline__ void f2unpack(uint64_t x, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(x));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// |x| maximum of the 8 bf16 values of a 16-byte chunk.
__device__ __forceinline__ float absmax_bf16x8(uint4 x) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  float m = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k)
    m = max3(m, fabsf(__uint_as_float(w[k] << 16)),
             fabsf(__uint_as_float(w[k] & 0xFFFF0000u)));
  return m;
}

// Sum of |x| of the 8 bf16 values of a 16-byte chunk.
__device__ __forceinline__ float abssum_bf16x8(uint4 x) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  float m = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k)
    m += fabsf(__uint_as_float(w[k] << 16)) + fabsf(__uint_as_float(w[k] & 0xFFFF0000u));
  return m;
}

// bf16 element e (0..7) of a 16-byte chunk, as raw bits.
__device__ __forceinline__ uint32_t bf16_bits_of(uint4 x, int e) {
  const uint32_t w = (e >> 1) == 0 ? x.x : (e >> 1) == 1 ? x.y : (e >> 1) == 2 ? x.z : x.w;
  return (e & 1) ? (w >> 16) : (w & 0xFFFFu);
}

// The chunk with element e (0..7) set to zero when dim0 + e is one of the
// group's exception channels.
__device__ __forceinline__ uint4 drop_channels(uint4 x, int dim0, const int (&tab)[kExc],
                                               int ntab) {
  uint32_t w[4] = {x.x, x.y, x.z, x.w};
  for (int k = 0; k < ntab; ++k) {
    const int e = tab[k] - dim0;
    if (e >= 0 && e < 8) w[e >> 1] &= (e & 1) ? 0x0000FFFFu : 0xFFFF0000u;
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Two E4M3 bytes (lower byte first) -> two floats (exact).
__device__ __forceinline__ void e4m3x2_to_f32(uint32_t b2, float& lo, float& hi) {
  uint32_t h;
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}"
      : "=r"(h)
      : "r"(b2));
  lo = __half2float(__ushort_as_half((unsigned short)(h & 0xFFFFu)));
  hi = __half2float(__ushort_as_half((unsigned short)(h >> 16)));
}

// Q split: values a (element 2c) and b (element 2c + 1), already multiplied
// by the row's 2^-e, become hi = e4m3 pair and lo = e4m3 pair of the
// remainders (lower byte = element 2c).  The remainder a - hi(a) is exact in
// fp32, so lo rounds it once.
__device__ __forceinline__ void split_q_pair(float a, float b, uint32_t& hi,
                                             uint32_t& lo) {
  asm("{\n\t.reg .b16 h, l, h0, h1;\n\t.reg .b32 hf;\n\t.reg .f32 fa, fb;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 h, %3, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 hf, h;\n\t"
      "mov.b32 {h0, h1}, hf;\n\t"
      "cvt.f32.f16 fa, h0;\n\tcvt.f32.f16 fb, h1;\n\t"
      "sub.rn.f32 fa, %2, fa;\n\tsub.rn.f32 fb, %3, fb;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 l, fb, fa;\n\t"
      "cvt.u32.u16 %0, h;\n\tcvt.u32.u16 %1, l;\n\t}"
      : "=r"(hi), "=r"(lo)
      : "f"(a), "f"(b));
}

// 8 bf16 Q values (one 16-byte chunk) times 2^-e -> 8 Qhi bytes and 8 Qlo
// bytes, in element order.
__device__ __forceinline__ void split_q8(uint4 x, float inv, uint2& hi,
                                         uint2& lo) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  uint32_t h[4], l[4];
#pragma unroll
  for (int k = 0; k < 4; ++k)
    split_q_pair(__uint_as_float(w[k] << 16) * inv,
                 __uint_as_float(w[k] & 0xFFFF0000u) * inv, h[k], l[k]);
  hi = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
  lo = make_uint2(l[0] | (l[1] << 16), l[2] | (l[3] << 16));
}

// P split of four consecutive f16 values (two f16x2 words, P' < 256):
// hi = their 4 E4M3 bytes, lo = 4 E5M2 bytes of P' - hi (exact in f16).
__device__ __forceinline__ void split_p4(uint32_t w0, uint32_t w1, uint32_t& hi,
                                         uint32_t& lo) {
  asm("{\n\t.reg .b32 b0, b1, r0, r1;\n\t.reg .b16 h0, h1, l0, l1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f16x2 h0, %2;\n\t"
      "cvt.rn.satfinite.e4m3x2.f16x2 h1, %3;\n\t"
      "cvt.rn.f16x2.e4m3x2 b0, h0;\n\t"
      "cvt.rn.f16x2.e4m3x2 b1, h1;\n\t"
      "sub.rn.f16x2 r0, %2, b0;\n\t"
      "sub.rn.f16x2 r1, %3, b1;\n\t"
      "cvt.rn.satfinite.e5m2x2.f16x2 l0, r0;\n\t"
      "cvt.rn.satfinite.e5m2x2.f16x2 l1, r1;\n\t"
      "mov.b32 %0, {h0, h1};\n\t"
      "mov.b32 %1, {l0, l1};\n\t}"
      : "=r"(hi), "=r"(lo)
      : "r"(w0), "r"(w1));
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t y;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(y) : "r"(a), "r"(b));
  return y;
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  uint32_t y;
  asm("cvt.rn.f16x2.f32 %0, %2, %1;" : "=r"(y) : "f"(lo), "f"(hi));
  return y;
}

// Record a failed wait: device status, this CTA's and the peer's abort flag.
__device__ __forceinline__ void signal_abort(Smem& s, const TcParams& p,
                                             uint32_t rank) {
  if (p.status) atomicOr(p.status, MLA_STATUS_WAIT_TIMEOUT);
  s.abort_flag = 1;
  st_cluster_u32(mapa(smem_u32(&s.abort_flag), rank ^ 1u), 1u);
}

// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src,
                                          uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Per-pair work description, identical on both CTAs of the pair.
struct Work {
  int v, b, shard, split, r_base, nrows, npages;
  int64_t L, p0;
};

// The pair's unit id (split, virtual request v, row group g) = (split * V +
// v) * G + g: the pair's index or, with a work list, the list's entry there;
// -1 for an entry outside [0, units).
__device__ __forceinline__ int pair_unit(const TcParams& p) {
  const int k = blockIdx.x >> 1;
  if (!p.work) return k;
  const int unit = p.work[k];
  return (unsigned)unit < (unsigned)p.units ? unit : -1;
}

__device__ __forceinline__ Work pair_work(const TcParams& p, int pair) {
  Work w;
  const int g = pair % p.G;
  pair /= p.G;
  w.v = pair % p.V;
  w.split = pair / p.V;
  w.b = w.v % p.B;
  w.shard = w.v / p.B;
  const int R = p.q_len * p.H;
  w.r_base = g * kRows;
  w.nrows = min(kRows, R - w.r_base);
  int64_t L = p.seq_lens[w.v];
  if (L > p.r2t_stride) L = p.r2t_stride;
  if (L < 0) L = 0;
  w.L = L;
  const int64_t P = (L + kPage - 1) / kPage;
  int64_t p1;
  split_page_range(
      p.split_pages ? p.split_pages + (int64_t)w.v * (p.num_splits + 1) : nullptr,
      p.num_splits, w.split, P, w.p0, p1);
  w.npages = (int)(p1 - w.p0);
  return w;
}

// Tokens in [nmin, L) are visible to some query rows of the request and
// masked for others; tokens at or past L to none.  The pages of the pair's
// range from m_san on hold such tokens and are sanitised before P V reads
// them (tail_warp).  Computed only by the O-CTA roles that need it.
__device__ __forceinline__ void masked_range(const TcParams& p, const Work& w,
                                             int64_t& nmin_out, int& m_san_out) {
  int64_t nmin = w.L - p.q_len + 1;
  if (p.kv_limit) {
    nmin = w.L;
    for (int i = 0; i < p.q_len; ++i) {
      const int64_t n = p.kv_limit[(int64_t)w.v * p.q_len + i];
      nmin = n < nmin ? n : nmin;
    }
  }
  nmin_out = nmin < 0 ? 0 : (nmin > w.L ? w.L : nmin);
  const int64_t m_san = nmin_out / kPage - w.p0;
  m_san_out = (int)(m_san < 0 ? 0 : (m_san > w.npages ? w.npages : m_san));
}

// Four E4M3 bytes with every NaN code (S.1111.111; E4M3 has no infinity)
// replaced by 0.
__device__ __forceinline__ uint32_t e4m3x4_nan_to_zero(uint32_t x) {
  uint32_t keep = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k)
    if (((x >> (8 * k)) & 0x7Fu) != 0x7Fu) keep |= 0xFFu << (8 * k);
  return x & keep;
}

__device__ __forceinline__ int tile_pages(const Work& w, int j) {
  return min(kTilePages, w.npages - j * kTilePages);
}

// Base slot of page m of the pair's range, or -1 if it lies outside the pool.
__device__ __forceinline__ int32_t page_base(const TcParams& p, const Work& w,
                                             int m) {
  if (m >= w.npages) return 0;
  const int32_t base = p.r2t[(int64_t)w.v * p.r2t_stride + (w.p0 + m) * kPage];
  if (base < 0 || (base & (kPage - 1)) || (int64_t)base + kPage > p.num_slots)
    return -1;
  return base;
}

// Start the 2-D box at (x, y) of a tensor on its way into L2, and a plain
// range of `bytes` (a multiple of 16, 16-byte aligned): no shared memory is
// written and nothing waits for them.
__device__ __forceinline__ void prefetch_box_l2(const void* tmap, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(tmap),
               "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void prefetch_bytes_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes)
               : "memory");
}

// ------------------------------------------------------------ producers ---
// S-CTA: per S tile (up to 4 pages) the pages' 64 scales each into
// tscale[j % 4] by bulk copy (zeros, written here, for a page outside the
// pool), then 5 ring stages: dims 128c..128c+127 of the tile's pages
// (c = 0..3, one 8-KB box per page) and the RoPE dims (one 4-KB box per page).
// Page bases are read 32 pages ahead (one per lane).  A page outside the
// pool is loaded from row num_slots: TMA fills it with zeros.
__device__ __forceinline__ void producer_s(Smem& s, const CUtensorMap* map,
                                           const CUtensorMap* map_rope,
                                           const TcParams& p, const Work& w,
                                           uint32_t rank, int lane) {
  uint32_t stage = 0, phase = 0;
  int32_t cur = page_base(p, w, lane), nxt = page_base(p, w, 32 + lane);
  bool ok = true;
  // While the softmax warps prepare the query, the first tile's K boxes and
  // scales are pulled into L2 (lane l: page l), so their loads after qready
  // find them there.
  if (lane < min(kTilePages, w.npages) && cur >= 0) {
#pragma unroll 1
    for (int c = 0; c < kBlocksPerTile; ++c) {
      if (c == kBlocksPerTile - 1)
        prefetch_box_l2(map_rope, MLA_NOPE_DIM, cur);
      else
        prefetch_box_l2(map, 128 * c, cur);
    }
    prefetch_bytes_l2(p.kv_scale + cur, kPage * 4);
  }
  // The ring holds the query rows until every softmax warp has moved them.
  if (lane == 0 && !mbar_wait(smem_u32(&s.qready), 0, &s.abort_flag)) ok = false;
  ok = __shfl_sync(kFull, ok, 0);
  // A stage is released by the MMA's commit and by the extractor, which has
  // work only when the group has exception channels; without them this warp
  // makes that second arrival itself as soon as it takes the stage (it then
  // counts towards the stage's next release), so the release waits for the
  // MMA alone.
  const bool self_release = s.xtab[0] < 0;
  const int ntiles = (w.npages + kTilePages - 1) / kTilePages;
  for (int j = 0; j < ntiles && ok; ++j) {
    const int m0 = j * kTilePages;
    if (m0 % 32 == 0 && m0 > 0) {
      cur = nxt;
      nxt = page_base(p, w, m0 + 32 + lane);
    }
    const int np = tile_pages(w, j);
    const int32_t bq = __shfl_sync(kFull, cur, (m0 + (lane & 3)) & 31);
    const int32_t yq = bq < 0 ? (int32_t)p.num_slots : bq;
    if (lane < np && bq < 0 && p.status) atomicOr(p.status, MLA_STATUS_BAD_SLOT);
    const int ts = j & 3;
    if (lane == 0 &&
        !mbar_wait(smem_u32(&s.scempty[ts]), ((j >> 2) & 1) ^ 1u, &s.abort_flag))
      ok = false;
    ok = __shfl_sync(kFull, ok, 0);
    if (!ok) break;
    const bool bad = lane < np && bq < 0;
    if (bad) {
      for (int e = 0; e < kPage; ++e) s.tscale[ts][lane * kPage + e] = 0.f;
      fence_proxy_async_smem();
    }
    const uint32_t good = __ballot_sync(kFull, lane < np && bq >= 0);
    if (lane == 0)
      mbar_arrive_expect_tx(smem_u32(&s.scfull[ts]),
                            (uint32_t)__popc(good) * kPage * 4);
    __syncwarp();
    if (lane < np && bq >= 0)
      bulk_load(smem_u32(&s.tscale[ts][lane * kPage]), p.kv_scale + bq,
                kPage * 4, smem_u32(&s.scfull[ts]));
    for (int c = 0; c < kBlocksPerTile && ok; ++c) {
      const bool rope = c == kBlocksPerTile - 1;
      const uint32_t box = rope ? kRopeBoxBytes : kBoxBytes;
      if (lane == 0) {
        if (mbar_wait(smem_u32(&s.empty[stage]), phase ^ 1u, &s.abort_flag)) {
          if (self_release) mbar_arrive(smem_u32(&s.empty[stage]));
          mbar_arrive_expect_tx(smem_u32(&s.full[stage]), np * box);
        } else {
          ok = false;
        }
      }
      ok = __shfl_sync(kFull, ok, 0);
      if (ok && lane < np)
        tma_load_2d(smem_u32(s.ring[stage]) + lane * box, rope ? map_rope : map,
                    smem_u32(&s.full[stage]), rope ? MLA_NOPE_DIM : 128 * c, yq);
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
  if (!ok && lane == 0) signal_abort(s, p, rank);
}

// O-CTA: one ring stage per page, the 512 value dims as 4 boxes of 128.
__device__ __forceinline__ void producer_o(Smem& s, const CUtensorMap* map,
                                           const TcParams& p, const Work& w,
                                           uint32_t rank, int lane) {
  uint32_t stage = 0, phase = 0;
  int32_t cur = page_base(p, w, lane), nxt = page_base(p, w, 32 + lane);
  bool ok = true;
  for (int m = 0; m < w.npages && ok; ++m) {
    if (m % 32 == 0 && m > 0) {
      cur = nxt;
      nxt = page_base(p, w, m + 32 + lane);
    }
    const int32_t b = __shfl_sync(kFull, cur, m & 31);
    const int32_t y = b < 0 ? (int32_t)p.num_slots : b;
    if (lane == 0) {
      if (mbar_wait(smem_u32(&s.empty[stage]), phase ^ 1u, &s.abort_flag))
        mbar_arrive_expect_tx(smem_u32(&s.full[stage]), kStageBytes);
      else
        ok = false;
    }
    ok = __shfl_sync(kFull, ok, 0);
    if (ok && lane < 4)
      tma_load_2d(smem_u32(s.ring[stage]) + lane * kBoxBytes, map,
                  smem_u32(&s.full[stage]), 128 * lane, y);
    if (++stage == kStages) {
      stage = 0;
      phase ^= 1u;
    }
  }
  if (!ok && lane == 0) signal_abort(s, p, rank);
}

// S-CTA warp 2: per tile, zero the scales of tokens at or past the request's
// length (their slots are undefined; 0 keeps every product finite) and of
// pages the tile lacks; track the running max |scale| over the split and its
// exponent g (max |scale| 2^g in [0.5, 1)); publish the tile's scale * 2^g
// as f16 pairs (the factor the packers apply to p) and g.  A non-finite scale
// of a token the request holds stays in tscale, so the scores of the rows
// that see the token are NaN (as the definition gives); it counts as 0 for g
// and for the factor, so the rows that do not see it (p = 0) add exactly 0
// and keep their units.
__device__ __forceinline__ void scale_warp(Smem& s, const TcParams& p,
                                           const Work& w, uint32_t rank,
                                           int lane) {
  bool ok = true;
  float smax = 0.f;
  int g = 0;
  const int ntiles = (w.npages + kTilePages - 1) / kTilePages;
  for (int j = 0; j < ntiles; ++j) {
    const int ts = j & 3;
    if (!mbar_wait(smem_u32(&s.scfull[ts]), (j >> 2) & 1, &s.abort_flag)) {
      ok = false;
      break;
    }
    const int np = tile_pages(w, j);
    const int64_t left = w.L - (w.p0 + (int64_t)j * kTilePages) * kPage;
    const int valid = (int)(left < (int64_t)np * kPage ? left : (int64_t)np * kPage);
    float v[8];
    float mx = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {  // token pair q = lane + 32 i
      const int t = 2 * (lane + 32 * i);
      const float2 x = *reinterpret_cast<const float2*>(&s.tscale[ts][t]);
      const float x0 = t < valid ? x.x : 0.f, x1 = t + 1 < valid ? x.y : 0.f;
      *reinterpret_cast<float2*>(&s.tscale[ts][t]) = make_float2(x0, x1);
      // finite part only: NaN and +-Inf compare false
      v[2 * i] = fabsf(x0) <= 3.402823466e38f ? x0 : 0.f;
      v[2 * i + 1] = fabsf(x1) <= 3.402823466e38f ? x1 : 0.f;
      mx = max3(mx, fabsf(v[2 * i]), fabsf(v[2 * i + 1]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
    smax = fmaxf(smax, mx);
    if (smax > 0.f) g = min(126, max(-126, -exponent_of(smax)));
    const float G = exp2i(g);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      s.tsg[ts][lane + 32 * i] = pack_f16(v[2 * i] * G, v[2 * i + 1] * G);
    if (lane == 0) s.tg[ts] = g;
    fence_proxy_async_smem();  // tscale is the next bulk copy's target
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&s.tsready[ts]));
  }
  if (!ok && lane == 0) signal_abort(s, p, rank);
}

// S-CTA warp 3: the group's exception channels (xtab, final once every
// softmax warp has passed qready).  For every ring stage of every tile it
// copies those channels' E4M3 key bytes of the stage's 128-dim block (or the
// RoPE block) for the tile's tokens into xk[j % 2][k][token] and then
// releases the stage with the MMA (empty counts both).  Without exception
// channels it has nothing to do (the producer makes its arrivals).
__device__ __forceinline__ void extractor(Smem& s, const TcParams& p,
                                          const Work& w, uint32_t rank,
                                          int lane) {
  bool ok = true;
  if (!mbar_wait(smem_u32(&s.qready), 0, &s.abort_flag)) ok = false;
  int tab[kExc], ntab = 0;
#pragma unroll
  for (int k = 0; k < kExc; ++k) {
    tab[k] = s.xtab[k];
    ntab += tab[k] >= 0 ? 1 : 0;
  }
  if (ok && ntab == 0) return;
  uint32_t stage = 0, phase = 0;
  const int ntiles = (w.npages + kTilePages - 1) / kTilePages;
  for (int j = 0; j < ntiles && ok; ++j) {
    const int np = tile_pages(w, j);
    const int xb = j & 1;
    if (!mbar_wait(smem_u32(&s.xkempty[xb]), ((j >> 1) & 1) ^ 1u, &s.abort_flag)) {
      ok = false;
      break;
    }
    for (int c = 0; c < kBlocksPerTile && ok; ++c) {
      if (!mbar_wait(smem_u32(&s.full[stage]), phase, &s.abort_flag)) {
        ok = false;
        break;
      }
      for (int k = 0; k < ntab; ++k) {
        const int d = tab[k];
        if ((d < MLA_NOPE_DIM ? d >> 7 : kBlocksPerTile - 1) != c) continue;
        for (int t = lane; t < np * kPage; t += 32) {
          const int pg = t >> 6, tr = t & 63;
          uint32_t off;
          if (c < kBlocksPerTile - 1) {  // 8-KB box per page, 128-B swizzle
            const int dd = d & 127;
            off = pg * kBoxBytes + box_chunk_offset(tr, dd >> 4) + (dd & 15);
          } else {  // 4-KB RoPE box per page, 64-B swizzle
            const int dd = d - MLA_NOPE_DIM;
            off = pg * kRopeBoxBytes + (tr >> 3) * 512 + (tr & 7) * 64 +
                  ((((dd >> 4) ^ (tr >> 1)) & 3) << 4) + (dd & 15);
          }
          s.xk[xb][k][t] = s.ring[stage][off];
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&s.empty[stage]));
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (ok && lane == 0) mbar_arrive(smem_u32(&s.xkfull[xb]));
  }
  if (!ok && lane == 0) signal_abort(s, p, rank);
}

// ---------------------------------------------------------- S-CTA: MMA ----
// One issuing thread.  Per tile: for each 128-dim block 4 K steps of 32,
// each Qhi then Qlo (A from TMEM) against the same K rows; then the RoPE
// block, 2 K steps, A from shared memory.  M=128, N=64*pages, into TMEM
// columns [256, 256 + 64*pages).
__device__ __forceinline__ void mma_s(Smem& s, const TcParams& p,
                                      const Work& w, uint32_t tmem,
                                      uint32_t rank) {
  if (!mbar_wait(smem_u32(&s.qready), 0, &s.abort_flag)) {
    signal_abort(s, p, rank);
    return;
  }
  tc_fence_after();
  const uint32_t d = tmem + kSCol0;
  const uint64_t qr_hi = sdesc_sw64(smem_u32(s.qrope[0]), 16, 512);
  const uint64_t qr_lo = sdesc_sw64(smem_u32(s.qrope[1]), 16, 512);
  uint32_t stage = 0, phase = 0;
  const int ntiles = (w.npages + kTilePages - 1) / kTilePages;
  for (int j = 0; j < ntiles; ++j) {
    const uint32_t idesc = idesc_s(tile_pages(w, j));
    if (!mbar_wait(smem_u32(&s.sempty), (j & 1) ^ 1u, &s.abort_flag)) {
      signal_abort(s, p, rank);
      return;
    }
    tc_fence_after();
    for (int c = 0; c < kBlocksPerTile; ++c) {
      if (!mbar_wait(smem_u32(&s.full[stage]), phase, &s.abort_flag)) {
        signal_abort(s, p, rank);
        return;
      }
      tc_fence_after();
      if (c < kBlocksPerTile - 1) {
        const uint64_t b = sdesc_sw128(smem_u32(s.ring[stage]), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint32_t col = 32u * c + 8u * kk;
          mma_ts_f8(d, tmem + col, b + 2 * kk, idesc, (c | kk) ? 1u : 0u);
          mma_ts_f8(d, tmem + kQLoCol + col, b + 2 * kk, idesc, 1u);
        }
      } else {
        const uint64_t b = sdesc_sw64(smem_u32(s.ring[stage]), 16, 512);
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          mma_ss_f8(d, qr_hi + 2 * kk, b + 2 * kk, idesc, 1u);
          mma_ss_f8(d, qr_lo + 2 * kk, b + 2 * kk, idesc, 1u);
        }
      }
      mma_commit(smem_u32(&s.empty[stage]));
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    mma_commit(smem_u32(&s.sfull));
  }
}

// S-CTA, thread 0, at kernel entry (the boxes need only the unit id, so
// their load overlaps the rest of the set-up): initialise qbar and load the
// pair's query rows, boxes of 64 values x q_box_rows rows with the 128-byte
// swizzle, the c_kv dims into the still idle ring and the RoPE dims into P
// slot 0.
__device__ __forceinline__ void issue_query(Smem& s, const CUtensorMap* qn_map,
                                            const CUtensorMap* qr_map,
                                            const TcParams& p, int unit) {
  const int g = unit % p.G;
  const int v = (unit / p.G) % p.V;
  const int qy = (v % p.B) * p.q_len * p.H + g * kRows;
  const uint32_t qbar = smem_u32(&s.qbar);
  mbar_init(qbar, 1);
  fence_mbar_init();
  prefetch_tmap(qn_map);
  prefetch_tmap(qr_map);
  const uint32_t box = (uint32_t)p.q_box_rows * 128u;
  mbar_arrive_expect_tx(qbar, 9 * box);
  for (int k = 0; k < 8; ++k)
    tma_load_3d(smem_u32(s.ring[0]) + 16384u * k, qn_map, qbar, 64 * k, qy, 0);
  tma_load_3d(smem_u32(s.pslot[0]), qr_map, qbar, 0, qy, 0);
}

// ------------------------------------------------------ S-CTA: softmax ----
// Warps 4..19: four warpgroups; warpgroup g (warps 4g + 4 .. 4g + 7) owns
// page g of each S tile, warp quad (warp % 4) owns TMEM lanes (query rows)
// 32 quad .. 32 quad + 31.  In the tile loop each thread owns rows
// A = 32 quad + (lane % 16) and B = A + 16 over half the page (lane / 16:
// tokens 0..31 or 32..63), read with 16x32bx2 loads, so each token scale it
// loads serves two rows.  Q is prepared with thread = row r: warpgroups 0
// and 1 split the c_kv dims, warpgroup 2 takes the RoPE dims.  The query
// rows arrive by TMA (boxes of 64 values x 128 rows, 128-byte swizzle): the
// c_kv dims in the ring, idle until the producer starts the KV stream once
// every softmax warp has passed qready, the RoPE dims in P slot 0.
__device__ __forceinline__ int64_t visible_count(const TcParams& p,
                                                 const Work& w, int r) {
  // tokens query row r (of the pair's rows) may see; 0 for padding rows
  if (r >= w.nrows) return 0;
  const int i = (w.r_base + r) / p.H;
  int64_t n = p.kv_limit ? (int64_t)p.kv_limit[(int64_t)w.v * p.q_len + i]
                         : w.L - p.q_len + 1 + i;
  return n > w.L ? w.L : (n < 0 ? 0 : n);
}

// Row scale exponent e: the row's largest |q| times 2^-e lies in [128, 256).
__device__ __forceinline__ int row_exponent(float amax) {
  return amax > 0.f ? min(126, max(-126, exponent_of(amax) - 8)) : 0;
}

__device__ __forceinline__ void softmax(Smem& s, const TcParams& p,
                                        const CUtensorMap* qn_map,
                                        const CUtensorMap* qr_map,
                                        const Work& w, uint32_t tmem,
                                        uint32_t rank, int warp, int lane) {
  const int g = (warp - 4) >> 2;        // warpgroup = page of the S tile
  const int quad = warp & 3;
  const int r = quad * 32 + lane;
  const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
  const bool row_ok = r < w.nrows;
  const int hp = lane >> 4;             // half of the page: tokens 32 hp ..
  const int part = 2 * g + hp;          // 32-token group of the S tile
  const int rA = quad * 32 + (lane & 15), rB = rA + 16;
  const uint4 zero4 = make_uint4(0, 0, 0, 0);

  // The query boxes were put in flight at kernel entry (issue_query).
  const uint32_t qbar = smem_u32(&s.qbar);
  const bool qok = mbar_wait(qbar, 0, &s.abort_flag);
  // 16-byte chunk k of this row's c_kv dims (k < 64) or RoPE dims (k < 8).
  auto qchunk = [&](int k) -> uint4 {
    return row_ok && qok ? *reinterpret_cast<const uint4*>(
                               s.ring[0] + 16384 * (k >> 3) +
                               box_chunk_offset(r, k & 7))
                         : zero4;
  };
  auto qrope_chunk = [&](int k) -> uint4 {
    return row_ok && qok ? *reinterpret_cast<const uint4*>(
                               s.pslot[0] + box_chunk_offset(r, k))
                         : zero4;
  };

  // This warpgroup's dims of row r, a quarter of the 576: c_kv chunks
  // 16g .. 16g + 15 (dims 128g .. 128g + 127) and RoPE chunks 2g, 2g + 1
  // (dims 512 + 16g ..); its 16-byte chunk k (0..17) holds dims dim0(k) ..
  // dim0(k) + 7.
  constexpr int nchunks = 18;
  auto my_chunk = [&](int k) -> uint4 {
    return k < 16 ? qchunk(16 * g + k) : qrope_chunk(2 * g + k - 16);
  };
  auto dim0 = [&](int k) -> int {
    return k < 16 ? 8 * (16 * g + k) : MLA_NOPE_DIM + 8 * (2 * g + k - 16);
  };
  // Row statistics from the warpgroups' parts: largest |q| and sum of |q|.
  float amax = 0.f, asum = 0.f;
  {
    float m4[4] = {0.f, 0.f, 0.f, 0.f}, s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (int k = 0; k < nchunks; ++k) {
      const uint4 x = my_chunk(k);
      m4[k & 3] = fmaxf(m4[k & 3], absmax_bf16x8(x));
      s4[k & 3] += abssum_bf16x8(x);
    }
    amax = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
    asum = (s4[0] + s4[1]) + (s4[2] + s4[3]);
  }
  s.xch[g][r] = amax;
  s.xch[4 + g][r] = asum;
  named_bar_sync(1, 512);
  auto qmax = [&](int row) {
    return fmaxf(max3(s.xch[0][row], s.xch[1][row], s.xch[2][row]), s.xch[3][row]);
  };
  // Exception candidates: elements above kExcRatio x the row's mean |q|
  // claim a slot of the group's channel table (first come; a channel already
  // there is shared; with the table full the element stays in the split).
  {
    const float tau = kExcRatio / MLA_ROW_DIM *
                      ((s.xch[4][r] + s.xch[5][r]) + (s.xch[6][r] + s.xch[7][r]));
    if (qmax(r) > tau) {
      for (int k = 0; k < nchunks; ++k) {
        const uint4 x = my_chunk(k);
        if (absmax_bf16x8(x) <= tau) continue;
        for (int e = 0; e < 8; ++e) {
          if (fabsf(__uint_as_float(bf16_bits_of(x, e) << 16)) <= tau) continue;
          const int d = dim0(k) + e;
          for (int t = 0; t < kExc; ++t) {
            const int old = atomicCAS(&s.xtab[t], -1, d);
            if (old == -1 || old == d) break;
          }
        }
      }
    }
  }
  named_bar_sync(1, 512);
  int tab[kExc], ntab = 0;
#pragma unroll
  for (int k = 0; k < kExc; ++k) {
    tab[k] = s.xtab[k];
    ntab += tab[k] >= 0 ? 1 : 0;
  }
  if (ntab > 0) {
    // The split's row scale from the elements outside the table; the owner
    // of each table channel keeps the row's value there for the exact path.
    float m = 0.f;
    for (int k = 0; k < nchunks; ++k)
      m = fmaxf(m, absmax_bf16x8(drop_channels(my_chunk(k), dim0(k), tab, ntab)));
    for (int t = 0; t < ntab; ++t) {
      const int d = tab[t];
      const int owner = d < MLA_NOPE_DIM ? d >> 7 : (d - MLA_NOPE_DIM) >> 4;
      if (owner == g) {
        const uint4 x = d < MLA_NOPE_DIM ? qchunk(d >> 3) : qrope_chunk((d - MLA_NOPE_DIM) >> 3);
        s.xe[r][t] = (uint16_t)bf16_bits_of(x, d & 7);
      }
    }
    s.xch[g][r] = m;  // every row max was read before the barrier above
    named_bar_sync(1, 512);
  }
  const float inv = exp2i(-row_exponent(qmax(r)));
  // score factor sm_scale * log2(e) * 2^e of rows A and B
  const float crowA = p.scale_log2 * exp2i(row_exponent(qmax(rA)));
  const float crowB = p.scale_log2 * exp2i(row_exponent(qmax(rB)));
  named_bar_sync(1, 512);
  const int64_t nA = visible_count(p, w, rA), nB = visible_count(p, w, rB);

  // Qhi / Qlo: c_kv dims -> TMEM columns [0, 128) and [128, 256) (column c
  // holds elements 4c..4c+3; warpgroup g writes dims 128g .. 128g + 127,
  // 64 dims = 16 columns per step), RoPE dims -> shared memory, K-major rows
  // of 64 bytes with the 64-byte swizzle (warpgroup g: elements 16g ..
  // 16g + 15).  The four warpgroups share the work evenly.
#pragma unroll 1
  for (int c = 0; c < 2; ++c) {
    uint32_t vh[16], vl[16];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      uint2 h, l;
      uint4 x = qchunk(16 * g + 8 * c + k);
      if (ntab > 0) x = drop_channels(x, 8 * (16 * g + 8 * c + k), tab, ntab);
      split_q8(x, inv, h, l);
      vh[2 * k] = h.x;
      vh[2 * k + 1] = h.y;
      vl[2 * k] = l.x;
      vl[2 * k + 1] = l.y;
    }
    tmem_st16(tmem + lane_base + 32u * g + 16u * c, vh);
    tmem_st16(tmem + lane_base + kQLoCol + 32u * g + 16u * c, vl);
  }
  {
    const int cc = g;  // 16-byte chunk cc = elements 16cc..16cc+15
    uint2 h0, l0, h1, l1;
    uint4 x0 = qrope_chunk(2 * cc), x1 = qrope_chunk(2 * cc + 1);
    if (ntab > 0) {
      x0 = drop_channels(x0, MLA_NOPE_DIM + 16 * cc, tab, ntab);
      x1 = drop_channels(x1, MLA_NOPE_DIM + 16 * cc + 8, tab, ntab);
    }
    split_q8(x0, inv, h0, l0);
    split_q8(x1, inv, h1, l1);
    const uint32_t off = (r >> 3) * 512 + (r & 7) * 64 +
                         (((cc ^ (r >> 1)) & 3) << 4);
    *reinterpret_cast<uint4*>(s.qrope[0] + off) = make_uint4(h0.x, h0.y, h1.x, h1.y);
    *reinterpret_cast<uint4*>(s.qrope[1] + off) = make_uint4(l0.x, l0.y, l1.x, l1.y);
  }
  tmem_wait_st();
  fence_proxy_async_smem();
  if (!__all_sync(kFull, qok) && lane == 0) signal_abort(s, p, rank);
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(smem_u32(&s.qready));

  // Running state per row (A, B): m_ref (log2 units, lazy), l in units of
  // 2^m_ref over this thread's tokens; g_cur is the split's scale exponent:
  // O accumulates p * scale * 2^g_cur, so it is kept in units of
  // 2^(m_ref - g_cur).
  float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;
  int g_cur = 0;
  bool ok = true;
  const uint32_t peer_pfull0 = mapa(smem_u32(&s.pfull[0]), 1);
  const int ntiles = (w.npages + kTilePages - 1) / kTilePages;
  const uint32_t bar_wg = 2 + g;  // named barrier of this warpgroup
  const uint32_t tA = tmem + lane_base + kSCol0 + 64u * g;
  const uint32_t tB = tA + (16u << 16);
  auto all_parts_max = [&](int row) {
    return fmaxf(fmaxf(max3(s.xch[0][row], s.xch[1][row], s.xch[2][row]),
                       max3(s.xch[3][row], s.xch[4][row], s.xch[5][row])),
                 fmaxf(s.xch[6][row], s.xch[7][row]));
  };
  for (int j = 0; j < ntiles; ++j) {
    const bool has = g < tile_pages(w, j);  // this warpgroup's page exists
    uint32_t a[32], b[32];  // rows A and B, tokens 32 hp .. 32 hp + 31
    if (ok && !mbar_wait(smem_u32(&s.sfull), j & 1, &s.abort_flag)) ok = false;
    tc_fence_after();
    if (__all_sync(kFull, ok) && has) {
      tmem_ld16x2_32<32>(tA, a);
      tmem_ld16x2_32<32>(tB, b);
      tmem_wait_ld();
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&s.sempty));

    // Exception channels: raw += q_c 2^-e k8_t,c for rows A and B, exact in
    // fp32 (a bf16 value times an E4M3 byte), from the bytes warp 3 copied.
    if (s.xtab[0] >= 0) {  // the group has exception channels (uniform)
      const int xb = j & 1;
      if (ok && !mbar_wait(smem_u32(&s.xkfull[xb]), (j >> 1) & 1, &s.abort_flag))
        ok = false;
      if (ok && has) {
        // 2^-e of each row: crow / scale_log2 is a power of two
        const float invA = 1.f / (crowA / p.scale_log2);
        const float invB = 1.f / (crowB / p.scale_log2);
        for (int k = 0; k < kExc && s.xtab[k] >= 0; ++k) {
          const float xa = __uint_as_float((uint32_t)s.xe[rA][k] << 16) * invA;
          const float xb2 = __uint_as_float((uint32_t)s.xe[rB][k] << 16) * invB;
          const uint32_t* kb =
              reinterpret_cast<const uint32_t*>(&s.xk[xb][k][kPage * g + 32 * hp]);
#pragma unroll
          for (int q = 0; q < 8; ++q) {  // tokens 4q .. 4q + 3
            const uint32_t w4 = kb[q];
            float k0, k1, k2, k3;
            e4m3x2_to_f32(w4 & 0xFFFFu, k0, k1);
            e4m3x2_to_f32(w4 >> 16, k2, k3);
            a[4 * q] = __float_as_uint(fmaf(xa, k0, __uint_as_float(a[4 * q])));
            a[4 * q + 1] = __float_as_uint(fmaf(xa, k1, __uint_as_float(a[4 * q + 1])));
            a[4 * q + 2] = __float_as_uint(fmaf(xa, k2, __uint_as_float(a[4 * q + 2])));
            a[4 * q + 3] = __float_as_uint(fmaf(xa, k3, __uint_as_float(a[4 * q + 3])));
            b[4 * q] = __float_as_uint(fmaf(xb2, k0, __uint_as_float(b[4 * q])));
            b[4 * q + 1] = __float_as_uint(fmaf(xb2, k1, __uint_as_float(b[4 * q + 1])));
            b[4 * q + 2] = __float_as_uint(fmaf(xb2, k2, __uint_as_float(b[4 * q + 2])));
            b[4 * q + 3] = __float_as_uint(fmaf(xb2, k3, __uint_as_float(b[4 * q + 3])));
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&s.xkempty[xb]));
    }

    // Token scales: raw -> raw * scale_t for both rows (one broadcast load
    // of four scales serves eight scores).
    if (ok && !mbar_wait(smem_u32(&s.tsready[j & 3]), (j >> 2) & 1,
                         &s.abort_flag))
      ok = false;
    const float* tsc = &s.tscale[j & 3][kPage * g + 32 * hp];
    if (has) {
#pragma unroll
      for (int c = 0; c < 32; c += 4) {
        const float4 f = *reinterpret_cast<const float4*>(tsc + c);
        const uint64_t f01 = f2pack(f.x, f.y), f23 = f2pack(f.z, f.w);
        float v0, v1, v2, v3;
        f2unpack(fmul2(f2pack(__uint_as_float(a[c]), __uint_as_float(a[c + 1])), f01), v0, v1);
        f2unpack(fmul2(f2pack(__uint_as_float(a[c + 2]), __uint_as_float(a[c + 3])), f23), v2, v3);
        a[c] = __float_as_uint(v0);
        a[c + 1] = __float_as_uint(v1);
        a[c + 2] = __float_as_uint(v2);
        a[c + 3] = __float_as_uint(v3);
        f2unpack(fmul2(f2pack(__uint_as_float(b[c]), __uint_as_float(b[c + 1])), f01), v0, v1);
        f2unpack(fmul2(f2pack(__uint_as_float(b[c + 2]), __uint_as_float(b[c + 3])), f23), v2, v3);
        b[c] = __float_as_uint(v0);
        b[c + 1] = __float_as_uint(v1);
        b[c + 2] = __float_as_uint(v2);
        b[c + 3] = __float_as_uint(v3);
      }
    }

    // Visible tokens of rows A, B among this thread's 32 (0 for a page the
    // tile lacks); the others become -inf (a select: garbage or NaN in a
    // masked column never propagates).  Only tiles at the end of the split
    // need it.
    const int64_t t0 = (w.p0 + (int64_t)j * kTilePages + g) * kPage + 32 * hp;
    auto clampv = [&](int64_t nrow) -> int {
      const int64_t nv = nrow - t0;
      return !has || nv <= 0 ? 0 : (nv >= 32 ? 32 : (int)nv);
    };
    const int nvA = clampv(nA), nvB = clampv(nB);
    if (!__all_sync(kFull, nvA == 32 && nvB == 32)) {
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        a[c] = c < nvA ? a[c] : __float_as_uint(-INFINITY);
        b[c] = c < nvB ? b[c] : __float_as_uint(-INFINITY);
      }
    }
    // Row maxima of raw * scale over this thread's tokens, then over the
    // tile's eight 32-token groups through shared memory.  The row factor is
    // positive, so the maximum score is its multiple.
    auto max32 = [&](const uint32_t (&x)[32]) -> float {
      float m4[4];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        m4[k] = max3(max3(__uint_as_float(x[8 * k]), __uint_as_float(x[8 * k + 1]),
                          __uint_as_float(x[8 * k + 2])),
                     max3(__uint_as_float(x[8 * k + 3]), __uint_as_float(x[8 * k + 4]),
                          __uint_as_float(x[8 * k + 5])),
                     fmaxf(__uint_as_float(x[8 * k + 6]), __uint_as_float(x[8 * k + 7])));
      return fmaxf(max3(m4[0], m4[1], m4[2]), m4[3]);
    };
    s.xch[part][rA] = max32(a) * crowA;
    s.xch[part][rB] = max32(b) * crowB;
    named_bar_sync(1, 512);
    const float mtA = all_parts_max(rA), mtB = all_parts_max(rB);
    named_bar_sync(1, 512);  // all read before the next tile overwrites

    // g of this tile (from the scale warp: max |scale| so far times 2^g in
    // [0.5, 1)).  O's factor is 2^((m_ref - m_new) + (g_new - g)); l's is
    // 2^(m_ref - m_new).
    const int g_new = s.tg[j & 3];
    auto update = [&](float mt, float& m, float& lsum) -> float {
      float m_new = m;
      if (mt > -INFINITY && (m == -INFINITY || mt > m + kTau)) m_new = mt;
      float alpha = 1.f;
      if (m > -INFINITY && (m_new != m || g_new != g_cur)) {
        if (m_new != m) lsum *= ex2(m - m_new);
        alpha = ex2((m - m_new) + (float)(g_new - g_cur));
      }
      m = m_new;
      return alpha;
    };
    const float alphaA = update(mtA, mA, lA), alphaB = update(mtB, mB, lB);
    g_cur = g_new;

    // Ship page g in message slot g (four slots, four pages per tile), use
    // j.  p = 2^(raw*scale*crow - m_ref) <= 2^tau (a row with nothing visible
    // yet shifts by 0: p = ex2(-inf) = 0), l += p.  Rows A and B of p are
    // packed as f16 pairs in place of their scores (word i of a row's 16 is
    // written after the scores it replaces were read), and only then does the
    // warpgroup wait for the slot: the O pair consumes pages in order, so
    // page 3's slot frees last, and the exponentials would otherwise queue
    // behind it.  Then the rows go to the slot 16 bytes at a time (the
    // packers multiply by scale * 2^g), with the tile's rescale (page 0
    // only), the warp's flag and, from warp quad 1, the page's factors.
    const bool any = __any_sync(kFull, alphaA != 1.f || alphaB != 1.f);
    uint8_t* stg = s.pslot[g];
    auto make_row = [&](uint32_t (&x)[32], float crow, float m, float& lsum) {
      const float shift = m == -INFINITY ? 0.f : m;
      const uint64_t c2 = f2pack(crow, crow), nshift2 = f2pack(-shift, -shift);
      uint64_t acc0 = f2pack(0.f, 0.f), acc1 = acc0;
#pragma unroll
      for (int c = 0; c < 8; ++c) {  // tokens 32 hp + 4c .. + 3
        float y0, y1, y2, y3;
        f2unpack(ffma2(f2pack(__uint_as_float(x[4 * c]), __uint_as_float(x[4 * c + 1])),
                       c2, nshift2), y0, y1);
        f2unpack(ffma2(f2pack(__uint_as_float(x[4 * c + 2]), __uint_as_float(x[4 * c + 3])),
                       c2, nshift2), y2, y3);
        const float p0 = ex2(y0), p1 = ex2(y1), p2 = ex2(y2), p3 = ex2(y3);
        acc0 = fadd2(acc0, f2pack(p0, p1));
        acc1 = fadd2(acc1, f2pack(p2, p3));
        x[2 * c] = pack_f16(p0, p1);
        x[2 * c + 1] = pack_f16(p2, p3);
      }
      float u0, u1, v0, v1;
      f2unpack(acc0, u0, u1);
      f2unpack(acc1, v0, v1);
      lsum += (u0 + u1) + (v0 + v1);
    };
    // 16-B chunk 4 hp + q = tokens 32 hp + 8q .. + 7 of a row (words 4q ..
    // 4q + 3), at position chunk ^ (row % 8) of the row's 128 bytes.
    auto store_row = [&](const uint32_t (&x)[32], int row) {
      uint8_t* dst = stg + (row >> 3) * 1024;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        *reinterpret_cast<uint4*>(dst + box_chunk_offset(row & 7, 4 * hp + q)) =
            make_uint4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
    };
    if (has) {
      make_row(a, crowA, mA, lA);
      make_row(b, crowB, mB, lB);
      if (j > 0 && ok &&
          !mbar_wait(smem_u32(&s.pempty[g]), (j - 1) & 1, &s.abort_flag))
        ok = false;
      store_row(a, rA);
      store_row(b, rB);
      if (hp == 0) {
        reinterpret_cast<float*>(stg + kAlphaOff)[rA] = g == 0 ? alphaA : 1.f;
        reinterpret_cast<float*>(stg + kAlphaOff)[rB] = g == 0 ? alphaB : 1.f;
      }
      if (lane == 0)
        reinterpret_cast<uint32_t*>(stg + kFlagOff)[quad] = g == 0 && any ? 1u : 0u;
      if (quad == 1)  // the page's 64 factors scale * 2^g (f16 pairs)
        reinterpret_cast<uint32_t*>(stg + kSGOff)[lane] = s.tsg[j & 3][g * 32 + lane];
      fence_proxy_async_smem();
    }
    named_bar_sync(bar_wg, 128);
    if (quad == 0 && lane == 0 && has && ok && !s.abort_flag)
      // The peer armed pfull[g] with the byte count itself.
      bulk_copy_to_peer(mapa(smem_u32(stg), 1), smem_u32(stg), kPMsgBytes,
                        peer_pfull0 + 8u * g);
    // Done with tscale, tsg and tg of tile j % 4.
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&s.scempty[j & 3]));
  }

  // Final statistics: l of a row = the sum over the eight token groups.
  s.xch[part][rA] = lA;
  s.xch[part][rB] = lB;
  named_bar_sync(1, 512);
  if (g == 0) {
    if (hp == 0) {
      const int64_t rows = (int64_t)p.B * p.q_len * p.H;
      const int64_t prt = (int64_t)w.split * (p.V / p.B) + w.shard;
      auto finish = [&](int row, float m) {
        float lt = 0.f;
#pragma unroll
        for (int k = 0; k < kPartials; ++k) lt += s.xch[k][row];
        if (row < w.nrows)
          // no visible token: -inf; a NaN sum (a NaN score seen) stays NaN
          p.LSE_part[prt * rows + (int64_t)w.b * p.q_len * p.H + w.r_base + row] =
              lt == 0.f ? -INFINITY : (m + log2f(lt)) * 0.69314718055994531f;
        // O (units 2^(m_ref - g)) / l (units 2^m_ref) = O 2^-g / l
        s.fin[row] = lt == 0.f ? 0.f : exp2i(-g_cur) / lt;
      };
      finish(rA, mA);
      finish(rB, mB);
    }
    fence_proxy_async_smem();
    named_bar_sync(2, 128);
    if (warp == 4 && lane == 0 && !s.abort_flag)
      bulk_copy_to_peer(mapa(smem_u32(s.fin), 1), smem_u32(s.fin), kRows * 4,
                        mapa(smem_u32(&s.fin_full), 1));
    // Before teardown: every P slot released by the peer, so no remote
    // arrive can land after this CTA exits.
    for (int m = max(0, w.npages - kNP); m < w.npages && ok; ++m)
      if (!mbar_wait(smem_u32(&s.pempty[m % kNP]), (m / kNP) & 1,
                     &s.abort_flag))
        ok = false;
  }
  if (!__all_sync(kFull, ok) && lane == 0) signal_abort(s, p, rank);
}

// ------------------------------------------ O-CTA: sanitise masked rows ---
// A masked token gets p = 0 exactly, but 0 * NaN would still poison
// O = P' V.  So for every page from the one holding token nmin onwards (the
// draft tokens only some query rows see, and the request's partly filled
// last page), warp 2 cleans the landed ring stage before the MMA reads it:
// rows at or past the length, which can hold anything, are zeroed; rows in
// [nmin, L) keep their bytes with every NaN code set to 0.  A query that
// sees such a token already has a NaN score for it (the S side reads the
// bytes as they are), which makes its whole row NaN, as the definition
// says; a query that does not see it now adds exactly 0.  The MMA thread,
// which waits on the ring in order, hands each landed page over (tail_go)
// and waits for it back (tail_ready), one page at a time.
__device__ __forceinline__ void tail_warp(Smem& s, const TcParams& p,
                                          const Work& w, uint32_t rank,
                                          int lane) {
  int64_t nmin;
  int m_san;
  masked_range(p, w, nmin, m_san);
  for (int m = m_san; m < w.npages; ++m) {
    const uint32_t use = (uint32_t)(m - m_san);
    if (!mbar_wait(smem_u32(&s.tail_go), use & 1u, &s.abort_flag)) {
      if (lane == 0) signal_abort(s, p, rank);
      return;
    }
    const int stage = m % kStages;
    const int64_t t0 = (w.p0 + m) * kPage;
    const int keep = (int)(w.L - t0 < kPage ? w.L - t0 : kPage);
    const int64_t lo64 = nmin - t0;
    const int lo = lo64 <= 0 ? 0 : (lo64 >= keep ? keep : (int)lo64);
    const int nr = kPage - lo;
    // 4 boxes x nr rows x 8 chunks of 16 bytes; a row's 128 bytes are
    // contiguous (the swizzle permutes chunks within the row).
    for (int idx = lane; idx < 4 * nr * 8; idx += 32) {
      const int bx = idx / (nr * 8), rem = idx % (nr * 8);
      const int row = lo + rem / 8, ch = rem % 8;
      uint4* c = reinterpret_cast<uint4*>(s.ring[stage] + bx * kBoxBytes +
                                          (row >> 3) * 1024 + (row & 7) * 128 +
                                          ch * 16);
      if (row >= keep) {
        *c = make_uint4(0, 0, 0, 0);
      } else {
        const uint4 x = *c;
        *c = make_uint4(e4m3x4_nan_to_zero(x.x), e4m3x4_nan_to_zero(x.y),
                        e4m3x4_nan_to_zero(x.z), e4m3x4_nan_to_zero(x.w));
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&s.tail_ready));
  }
}

// ------------------------------------------------------- O-CTA: packers ---
// Warps 8..11: thread = row r of every P message.  The row's 64 f16 p (8
// chunks of 16 bytes in the 128-byte-swizzled row) are all loaded and
// multiplied by the page's factors scale_t * 2^g (P' = p * scale_t * 2^g,
// f16), then written back in place as the MMA's A operand: chunks 0-3 = Phi
// (E4M3) of tokens 0..63, chunks 4-7 = Plo (E5M2).
__device__ __forceinline__ void packer(Smem& s, const TcParams& p,
                                       const Work& w, uint32_t rank, int warp,
                                       int lane) {
  const int r = (warp - 8) * 32 + lane;
  bool ok = true;
  for (int m = 0; m < w.npages; ++m) {
    const int k = m % kNP;
    if (!mbar_wait(smem_u32(&s.pfull[k]), (m / kNP) & 1, &s.abort_flag)) {
      ok = false;
      break;
    }
    uint8_t* row = s.pslot[k] + (r >> 3) * 1024;
    const uint4* sg = reinterpret_cast<const uint4*>(s.pslot[k] + kSGOff);
    uint4 x[8];
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) {
      const uint4 v = *reinterpret_cast<const uint4*>(row + box_chunk_offset(r & 7, cc));
      const uint4 f = sg[cc];  // factors of tokens 8cc..8cc+7 (broadcast)
      x[cc] = make_uint4(hmul2(v.x, f.x), hmul2(v.y, f.y), hmul2(v.z, f.z),
                         hmul2(v.w, f.w));
    }
#pragma unroll
    for (int h = 0; h < 4; ++h) {  // tokens 16h..16h+15 = input chunks 2h, 2h+1
      uint4 hi, lo;
      split_p4(x[2 * h].x, x[2 * h].y, hi.x, lo.x);
      split_p4(x[2 * h].z, x[2 * h].w, hi.y, lo.y);
      split_p4(x[2 * h + 1].x, x[2 * h + 1].y, hi.z, lo.z);
      split_p4(x[2 * h + 1].z, x[2 * h + 1].w, hi.w, lo.w);
      *reinterpret_cast<uint4*>(row + box_chunk_offset(r & 7, h)) = hi;
      *reinterpret_cast<uint4*>(row + box_chunk_offset(r & 7, 4 + h)) = lo;
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&s.packed[k]));
  }
  if (!ok && lane == 0) signal_abort(s, p, rank);
}

// ---------------------------------------------------------- O-CTA: MMA ----
__device__ __forceinline__ void mma_o(Smem& s, const TcParams& p,
                                      const Work& w, uint32_t tmem,
                                      uint32_t rank) {
  uint32_t stage = 0, phase = 0, ev = 0;
  bool ok = true;
  int64_t nmin;
  int m_san;
  masked_range(p, w, nmin, m_san);
  // Each P message lands by a bulk copy whose bytes complete on pfull[k];
  // this CTA arms the barrier (one arrival + the byte count) itself, so the
  // sender needs no cluster-scope arrive: the first use of each slot is armed
  // at set-up, the next one once the packers have split the message
  // (packed[k]).
  for (int m = 0; m < w.npages && ok; ++m) {
    const int k = m % kNP;
    if (!mbar_wait(smem_u32(&s.packed[k]), (m / kNP) & 1, &s.abort_flag)) {
      ok = false;
      break;
    }
    if (m + kNP < w.npages)
      mbar_arrive_expect_tx(smem_u32(&s.pfull[k]), kPMsgBytes);
    const uint32_t* fl =
        reinterpret_cast<const uint32_t*>(s.pslot[k] + kFlagOff);
    if (fl[0] | fl[1] | fl[2] | fl[3]) {
      // Rows changed their units: let the correction warps rescale O once
      // every earlier product has landed.
      s.ctl_slot = k;
      s.ctl_final = 0;
      mma_commit(smem_u32(&s.drain));
      mbar_arrive(smem_u32(&s.drain));
      if (!mbar_wait(smem_u32(&s.corr_done), ev & 1, &s.abort_flag)) {
        ok = false;
        break;
      }
      ++ev;
    }
    if (!mbar_wait(smem_u32(&s.full[stage]), phase, &s.abort_flag)) {
      ok = false;
      break;
    }
    if (m >= m_san) {  // the tail warp sanitises the page first
      mbar_arrive(smem_u32(&s.tail_go));
      if (!mbar_wait(smem_u32(&s.tail_ready), (uint32_t)(m - m_san) & 1u,
                     &s.abort_flag)) {
        ok = false;
        break;
      }
    }
    tc_fence_after();
    // A = P (K-major, 128-B swizzle): +2 units per 32 tokens, Plo 64 bytes
    // after Phi.  B = V (E4M3, MN-major): next 128 dims one box (8 KB) on,
    // next 8 tokens 1 KB on; 32 tokens = 4 KB (256 units), 256 dims = 16 KB.
    const uint64_t a = sdesc_sw128(smem_u32(s.pslot[k]), 16, 1024);
    const uint64_t b = sdesc_sw128(smem_u32(s.ring[stage]), kBoxBytes, 1024);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t d = tmem + 256u * h;
      const uint64_t bh = b + 1024u * h;
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        mma_ss_f8(d, a + 2 * kk, bh + 256u * kk, kIdescOHi,
                  (m > 0 || kk > 0) ? 1u : 0u);
        mma_ss_f8(d, a + 4 + 2 * kk, bh + 256u * kk, kIdescOLo, 1u);
      }
    }
    mma_commit(smem_u32(&s.empty[stage]));
    if (++stage == kStages) {
      stage = 0;
      phase ^= 1u;
    }
    mma_commit_multicast(smem_u32(&s.pempty[k]), (uint16_t)1u);  // S-CTA
  }
  if (!ok) signal_abort(s, p, rank);
  s.ctl_final = 1;
  mma_commit(smem_u32(&s.drain));
  mbar_arrive(smem_u32(&s.drain));
}

// ---------------------------------------- O-CTA: correction + epilogue ----
__device__ __forceinline__ void correct_and_store(Smem& s, const TcParams& p,
                                                  const Work& w, uint32_t tmem,
                                                  uint32_t rank, int warp,
                                                  int lane) {
  const int quad = warp & 3;
  const int r = quad * 32 + lane;
  const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
  bool ok = true;
  for (uint32_t ev = 0;; ++ev) {
    if (!mbar_wait(smem_u32(&s.drain), ev & 1, &s.abort_flag)) {
      ok = false;
      break;
    }
    tc_fence_after();
    if (*reinterpret_cast<volatile int*>(&s.ctl_final)) break;
    const int k = *reinterpret_cast<volatile int*>(&s.ctl_slot);
    const float a = reinterpret_cast<const float*>(s.pslot[k] + kAlphaOff)[r];
    if (__any_sync(kFull, a != 1.f)) {
#pragma unroll 1
      for (int c0 = 0; c0 < MLA_VALUE_DIM; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + c0, v);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e)
          v[e] = __float_as_uint(__uint_as_float(v[e]) * a);
        tmem_st32(tmem + lane_base + c0, v);
      }
      tmem_wait_st();
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&s.corr_done));
  }
  if (ok && !mbar_wait(smem_u32(&s.fin_full), 0, &s.abort_flag)) ok = false;
  if (!__all_sync(kFull, ok)) {
    if (lane == 0) signal_abort(s, p, rank);
    return;
  }
  tc_fence_after();
  // O_part = O / l, 32 values at a time: the warp stages its 32 rows in 4 KB
  // of the then idle ring (row r at 128 r bytes, 16-byte chunk e at position
  // e ^ (r % 8): neither the writes nor the reads below conflict) and reads
  // them back four rows per instruction, lane l taking chunk l % 8 of row
  // 4i + l / 8, so every store instruction writes four full 128-byte lines.
  const float inv = s.fin[r];
  const int64_t rows = (int64_t)p.B * p.q_len * p.H;
  const int64_t part = (int64_t)w.split * (p.V / p.B) + w.shard;
  float* const dst0 = p.O_part + (part * rows + (int64_t)w.b * p.q_len * p.H +
                                  w.r_base + quad * 32) * MLA_VALUE_DIM;
  const int nvalid = w.nrows - quad * 32;  // rows of this warp in range
  uint8_t* const buf = s.ring[0] + 4096 * quad;
  if (p.o_bf16) {
    // bf16 partial outputs: 64 values (128 bytes) per staged row, the same
    // staging and full-line stores.
    __nv_bfloat16* const dst_b =
        reinterpret_cast<__nv_bfloat16*>(p.O_part) +
        (part * rows + (int64_t)w.b * p.q_len * p.H + w.r_base + quad * 32) *
            MLA_VALUE_DIM;
#pragma unroll 1
    for (int c0 = 0; c0 < MLA_VALUE_DIM; c0 += 64) {
      uint32_t va[32], vb[32];
      tmem_ld32(tmem + lane_base + c0, va);
      tmem_ld32(tmem + lane_base + c0 + 32, vb);
      tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const uint32_t* v = e < 4 ? va + 8 * e : vb + 8 * (e - 4);
        uint32_t q[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(v[2 * j]) * inv,
                                                   __uint_as_float(v[2 * j + 1]) * inv);
          q[j] = *reinterpret_cast<uint32_t*>(&h);
        }
        *reinterpret_cast<uint4*>(buf + box_chunk_offset(lane, e)) =
            make_uint4(q[0], q[1], q[2], q[3]);
      }
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int rr = 4 * i + (lane >> 3), e = lane & 7;
        const uint4 f = *reinterpret_cast<const uint4*>(buf + box_chunk_offset(rr, e));
        if (rr < nvalid)
          *reinterpret_cast<uint4*>(dst_b + (int64_t)rr * MLA_VALUE_DIM + c0 + 8 * e) = f;
      }
      __syncwarp();  // every lane read the box before it is refilled
    }
    return;
  }
#pragma unroll 1
  for (int c0 = 0; c0 < MLA_VALUE_DIM; c0 += 32) {
    uint32_t v[32];
    tmem_ld32(tmem + lane_base + c0, v);
    tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 8; ++e)
      *reinterpret_cast<float4*>(buf + box_chunk_offset(lane, e)) =
          make_float4(__uint_as_float(v[4 * e]) * inv,
                      __uint_as_float(v[4 * e + 1]) * inv,
                      __uint_as_float(v[4 * e + 2]) * inv,
                      __uint_as_float(v[4 * e + 3]) * inv);
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int rr = 4 * i + (lane >> 3), e = lane & 7;
      const float4 f =
          *reinterpret_cast<const float4*>(buf + box_chunk_offset(rr, e));
      if (rr < nvalid)
        *reinterpret_cast<float4*>(dst0 + (int64_t)rr * MLA_VALUE_DIM + c0 +
                                   4 * e) = f;
    }
    __syncwarp();  // every lane read the box before it is refilled
  }
}

// ------------------------------------------------------------- kernel ----
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_partial_tc_fp8_kernel(const __grid_constant__ CUtensorMap kv_map,
                              const __grid_constant__ CUtensorMap rope_map,
                              const __grid_constant__ CUtensorMap qn_map,
                              const __grid_constant__ CUtensorMap qr_map,
                              const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();
  const int unit = pair_unit(p);
  if (unit < 0) {  // both CTAs of the pair read the same entry
    if (rank == 0 && threadIdx.x == 0 && p.status)
      atomicOr(p.status, MLA_STATUS_BAD_WORK);
    return;
  }
  if (rank == 0 && threadIdx.x == 0) issue_query(s, &qn_map, &qr_map, p, unit);
  const Work w = pair_work(p, unit);

  if (threadIdx.x == 0) {
    s.abort_flag = 0;
    s.ctl_slot = 0;
    s.ctl_final = 0;
    s.ctl_last = 0;
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_u32(&s.full[i]), 1);
      // S-CTA: the MMA's commit and the extractor (warp 3) release a stage
      mbar_init(smem_u32(&s.empty[i]), rank == 0 ? 2 : 1);
    }
    for (int i = 0; i < kExc; ++i) s.xtab[i] = -1;
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&s.xkfull[i]), 1);
      mbar_init(smem_u32(&s.xkempty[i]), 16);  // the 16 softmax warps
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(smem_u32(&s.scfull[i]), 1);
      mbar_init(smem_u32(&s.scempty[i]), 16);  // the 16 softmax warps
      mbar_init(smem_u32(&s.tsready[i]), 1);
    }
    mbar_init(smem_u32(&s.sfull), 1);
    mbar_init(smem_u32(&s.sempty), 16);
    for (int i = 0; i < kNP; ++i) {
      mbar_init(smem_u32(&s.pfull[i]), 1);
      mbar_init(smem_u32(&s.packed[i]), 4);  // the 4 packer warps
      mbar_init(smem_u32(&s.pempty[i]), 1);
    }
    mbar_init(smem_u32(&s.drain), 2);
    mbar_init(smem_u32(&s.corr_done), 4);
    mbar_init(smem_u32(&s.fin_full), 1);
    mbar_init(smem_u32(&s.qready), 16);
    mbar_init(smem_u32(&s.tail_go), 1);
    mbar_init(smem_u32(&s.tail_ready), 1);
    if (rank == 1 && w.npages > 0) {
      mbar_arrive_expect_tx(smem_u32(&s.fin_full), kRows * 4);
      for (int k = 0; k < kNP && k < w.npages; ++k)
        mbar_arrive_expect_tx(smem_u32(&s.pfull[k]), kPMsgBytes);
    }
    fence_mbar_init();
    prefetch_tmap(&kv_map);
    prefetch_tmap(&rope_map);
  }
  if (rank == 0 && threadIdx.x == 32 && p.seq_lens[w.v] > p.r2t_stride &&
      p.status)
    atomicOr(p.status, MLA_STATUS_BAD_LENGTH);
  if (warp == 1) {
    tmem_alloc(smem_u32(&s.tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;
  cluster_sync();  // the peer's barriers exist before any remote operation

  // Fused combine ([K3-MLA], dcp_lse_combine, in the same launch): rank 0
  // counts this pair's arrival for its (request, 128-row group) once both
  // CTAs have written their part; the pair whose arrival completes the count
  // (shards x splits) resets it and merges the group's rows, every part being
  // in memory by then.  No pair waits for another.
  auto fused_arrival = [&]() {
    if (rank == 0 && threadIdx.x == 0) {
      const int group = w.r_base / kRows;
      int* c = p.counters + (int64_t)w.b * p.G + group;
      const int total = p.num_splits * (p.V / p.B);
      const bool last = atom_add_acq_rel_gpu(c, 1) == total - 1;
      if (last) *c = 0;
      for (uint32_t k = 0; k < 2; ++k)
        st_cluster_u32(mapa(smem_u32(&s.ctl_last), k), last ? 1u : 0u);
    }
  };
  auto fused_combine = [&]() {
    if (!*reinterpret_cast<volatile int*>(&s.ctl_last)) return;
    __threadfence();
    const int R = p.q_len * p.H;
    const int r0 = w.r_base;
    const int n = min(kRows, R - r0);
    const int64_t rows = (int64_t)p.B * R;
    const int P = p.num_splits * (p.V / p.B);
    constexpr int kWarps = kThreads / 32;
    for (int r = (int)rank * kWarps + warp; r < n; r += 2 * kWarps)
      combine_row<true>(p.O_part, p.LSE_part, P, rows,
                        (int64_t)w.b * R + r0 + r, p.out, p.lse_out, lane);
  };

  // Teardown, repeated at the end of every role (roles never rejoin, so no
  // warp asks setmaxnreg for registers back).
  auto teardown = [&]() {
    if (p.counters) __threadfence();  // this CTA's part before the arrival
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
    if (p.counters) {
      cluster_sync();  // both CTAs' parts written
      fused_arrival();
    }
    cluster_sync();
    if (p.counters) fused_combine();
  };

  if (w.npages > 0 && rank == 0) {
    if (warp < 4) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsControl));
      if (warp == 0) {
        producer_s(s, &kv_map, &rope_map, p, w, rank, lane);
      } else if (warp == 1) {
        if (lane == 0) mma_s(s, p, w, tmem, rank);
        __syncwarp();
      } else if (warp == 2) {
        scale_warp(s, p, w, rank, lane);
      } else {
        extractor(s, p, w, rank, lane);
      }
      teardown();
      return;
    }
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    softmax(s, p, &qn_map, &qr_map, w, tmem, rank, warp, lane);
    teardown();
    return;
  }
  if (w.npages > 0) {
    if (warp == 0) {
      producer_o(s, &kv_map, p, w, rank, lane);
    } else if (warp == 1) {
      if (lane == 0) mma_o(s, p, w, tmem, rank);
      __syncwarp();
    } else if (warp == 2) {
      tail_warp(s, p, w, rank, lane);
    } else if (warp >= 4 && warp < 8) {
      correct_and_store(s, p, w, tmem, rank, warp, lane);
    } else if (warp >= 8 && warp < 12) {
      packer(s, p, w, rank, warp, lane);
    }
  } else if (rank == 0 && threadIdx.x == 0) {
    // No tokens for this split: the query boxes issued at entry land before
    // the CTA leaves.
    mbar_wait(smem_u32(&s.qbar), 0, &s.abort_flag);
  }
  if (w.npages == 0 && warp >= 4 && warp < 8) {
    // No tokens for this split: O = 0, LSE = -inf.
    const int r = (warp & 3) * 32 + lane;
    if (r < w.nrows) {
      const int64_t rows = (int64_t)p.B * p.q_len * p.H;
      const int64_t part = (int64_t)w.split * (p.V / p.B) + w.shard;
      const int64_t orow =
          part * rows + (int64_t)w.b * p.q_len * p.H + w.r_base + r;
      if (rank == 0) {
        p.LSE_part[orow] = -INFINITY;
      } else if (p.o_bf16) {
        uint4* d = reinterpret_cast<uint4*>(
            reinterpret_cast<__nv_bfloat16*>(p.O_part) + orow * MLA_VALUE_DIM);
        for (int e = 0; e < MLA_VALUE_DIM / 8; ++e) d[e] = make_uint4(0, 0, 0, 0);
      } else {
        float4* d4 = reinterpret_cast<float4*>(p.O_part + orow * MLA_VALUE_DIM);
        for (int e = 0; e < MLA_VALUE_DIM / 4; ++e)
          d4[e] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }
  teardown();
}

}  // namespace

int launch_tc_fp8(const DecodeArgs& a) {
  TcParams p;
  p.q_nope = static_cast<const uint4*>(a.q_nope);
  p.q_rope = static_cast<const uint4*>(a.q_rope);
  p.kv_scale = a.kv_scale;
  p.num_slots = a.num_slots;
  p.r2t = a.req_to_token;
  p.r2t_stride = a.r2t_stride;
  p.seq_lens = a.seq_lens;
  p.kv_limit = a.kv_limit;
  p.split_pages = a.split_pages;
  p.work = a.work;
  p.B = a.B;
  p.q_len = a.q_len;
  p.H = a.H;
  p.V = a.B * a.num_shards;
  p.num_splits = a.num_splits;
  p.G = (a.q_len * a.H + kRows - 1) / kRows;
  p.scale_log2 = a.sm_scale * 1.4426950408889634f;
  p.O_part = a.O_part;
  p.o_bf16 = a.o_bf16;
  p.LSE_part = a.LSE_part;
  p.status = a.status;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.lse_out = a.lse_out;
  p.counters = a.counters;
  const int64_t pairs = (int64_t)p.V * p.num_splits * p.G;
  if (pairs * 2 > 0x7fffffff) return fail(MLA_ERR_INVALID_ARG, "grid too large");
  p.units = (int)pairs;
  CUtensorMap map, rope_map;
  int rc = make_kv_tensor_map(&map, a.kv, MLA_KV_FP8_E4M3, a.num_slots);
  if (rc != MLA_OK) return rc;
  rc = make_kv_tensor_map_fp8_rope(&rope_map, a.kv, a.num_slots);
  if (rc != MLA_OK) return rc;
  CUtensorMap qn_map, qr_map;
  rc = make_query_maps(&qn_map, &qr_map, a, &p.q_box_rows);
  if (rc != MLA_OK) return rc;
  cudaError_t e = cudaFuncSetAttribute(
      mla_partial_tc_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
      kSmemBytes);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(tc fp8)");
  mla_partial_tc_fp8_kernel<<<(unsigned)(pairs * 2), kThreads, kSmemBytes,
                              a.stream>>>(map, rope_map, qn_map, qr_map, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch mla_partial_tc_fp8_kernel");
  return MLA_OK;
}

int pair_slots_fp8() {
  cudaError_t e = cudaFuncSetAttribute(
      mla_partial_tc_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
      kSmemBytes);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(tc fp8)");
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * 1024, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, mla_partial_tc_fp8_kernel, &cfg);
  if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveClusters");
  return clusters;
}

}  // namespace mla
