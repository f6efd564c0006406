// mla_tc_fp8.cu -- tensor-core partial MLA decode over an FP8 (E4M3) KV
// cache with one fp32 scale per token.
//
// Same computation as the BF16 path (include/mla_decode.h,
// mla_decode_partial; [VRAM-KV], [K3-MLA], [K3-SPLIT], [K3-INTRO]) with
// k_t = e4m3(byte) * kv_scale[slot].
//
// Design (GB300, clusters of two CTAs, one CTA per SM):
//   FP8 halves the KV bytes, so one SM's TMA engine (~45 B/clk for 64-row
//   boxes) can feed an M = 128 MMA by itself and the kernel keeps the simple
//   layout of one S-CTA (rank 0) and one O-CTA (rank 1) per 128-row group,
//   with single-CTA MMAs.  The tensor cores multiply f16 by f16: TMA lands
//   unswizzled 64-byte-wide E4M3 boxes (64 tokens x 64 dims) in a staging
//   ring (plus, on the S side, each page's 64 scales); two converter warps
//   per CTA turn them into f16 tiles (E4M3 values are exact in f16) in the
//   128-byte-swizzled layout the MMA reads, writing zeros for rows past a
//   request's length.  On the S side the per-token scale stays outside the
//   MMA, s_t = scale_t * (q . e4m3_t) in fp32 on each score column, so no
//   rounding touches the scores (and the LSE); on the O side the converters
//   write V as f16(e4m3 * scale), one rounding that only O sees.  The S-CTA holds Q (converted to
//   f16, exact for bf16 values in f16 range) in TMEM / shared memory and
//   issues M=128, N=64*pages (up to 256) MMAs from one thread; the softmax
//   and the O-CTA are those of the BF16 pair design, with P shipped as f16.
//   Every wait is bounded (ptx_sm103.cuh).
#include <cuda_bf16.h>

#include "mla_tma.cuh"
#include "ptx_sm103.cuh"

namespace mla {
namespace {

using namespace ptx;

constexpr int kThreads = 512;        // 16 warps = 4 warpgroups
constexpr int kStages = 2;           // f16 operand stages (4 chunks, 32 KB)
constexpr int kBoxesPerStage = 4;
constexpr int kStages8 = 4;          // E4M3 staging stages
constexpr int kBox8Bytes = 64 * 64;  // 64 tokens x 64 bytes
constexpr int kScaleBytes = 64 * 4;  // one page's fp32 scales
constexpr int kStage8Bytes = kBoxesPerStage * (kBox8Bytes + kScaleBytes);
constexpr int kChunksPerPage = 9;    // 576 dims = 9 x 64
constexpr int kTilePages = 4;        // pages per S tile (N <= 256)
constexpr int kNP = 4;               // P message slots (page index mod 4)
constexpr int kRows = 128;           // query rows per CTA pair
constexpr int kPage = MLA_PAGE_SIZE;      // 64 tokens
constexpr int kPBytes = kRows * kPage * 2;          // 16384
constexpr int kAlphaOff = kPBytes;                  // float alpha[128]
constexpr int kFlagOff = kPBytes + kRows * 4;       // uint32 flags[4]
constexpr int kPMsgBytes = kFlagOff + 16;           // 16912 = 1057 x 16
constexpr int kPSlotStride = 17408;                 // 17 KB, 1024-aligned
constexpr uint32_t kSCol0 = 256;                    // S buffer columns
constexpr float kTau = 8.f;          // lazy-rescale threshold (log2 units)
constexpr uint32_t kFull = 0xffffffffu;
// Register split of the S-CTA (setmaxnreg): 512 threads launch with 128
// registers each (65,536); the producer/MMA/converter warpgroups (warps 0-3
// and 12-15) give registers away so the two softmax warpgroups can hold a
// 128 x 256 fp32 score tile.  The split is one-way.
constexpr int kRegsLaunch = 128;
constexpr int kRegsControl = 40;
constexpr int kRegsSoftmax = 216;
static_assert(256 * kRegsControl + 256 * kRegsSoftmax <= kThreads * kRegsLaunch,
              "register split exceeds the launch allocation");

// kind::f16 with f16 A and B (format 0) and an fp32 accumulator.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N, bool b_mn) {
  return (1u << 4) | ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}
__host__ __device__ constexpr uint32_t idesc_s(int pages) {
  return idesc_f16_f32(128, 64 * pages, false);
}
constexpr uint32_t kIdescO = idesc_f16_f32(128, 256, true);

struct __align__(1024) Smem {
  uint8_t ring[kStages * kBoxesPerStage][kBoxBytes];  // 64 KB f16 operands
  uint8_t ring8[kStages8][kStage8Bytes];              // 66 KB E4M3 + scales
  uint8_t qrope[kRows * 128];                         // S-CTA: Q_rope rows
  float tscale[4][kTilePages][64];  // S-CTA: token scales of tiles j % 4
  uint8_t pslot[kNP][kPSlotStride];
  float fin[kRows];
  float xch[2][kRows];      // S-CTA: per-warpgroup row maxima / partial sums
  uint64_t full[kStages];   // converters -> MMA (one arrival per converter warp)
  uint64_t empty[kStages];  // MMA -> converters
  uint64_t full8[kStages8]; // TMA -> converters (bytes)
  uint64_t empty8[kStages8];// converters -> producer (one per converter warp)
  uint64_t tsready[4];      // S-CTA: tscale[j % 4] written (converter warps)
  uint64_t sfull, sempty;
  uint64_t pfull[kNP];
  uint64_t pempty[kNP];
  uint64_t drain, corr_done, fin_full, qready;
  uint32_t tmem_base;
  int abort_flag;
  int ctl_slot;
  int ctl_final;
};
constexpr int kSmemBytes = (int)sizeof(Smem) + 1024;
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
static_assert(kPMsgBytes % 16 == 0, "bulk copy size");
static_assert(kStage8Bytes % 128 == 0, "staging stage alignment");

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
  int B, q_len, H, V, num_splits, G;
  float scale_log2;        // sm_scale * log2(e)
  float* O_part;
  float* LSE_part;
  int* status;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  uint32_t y;
  asm("cvt.rn.f16x2.f32 %0, %2, %1;" : "=r"(y) : "f"(lo), "f"(hi));
  return y;
}

// Packed bf16 pair -> packed f16 pair (both halves rounded to nearest).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
  return pack_f16(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
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

__device__ __forceinline__ Work pair_work(const TcParams& p) {
  Work w;
  // launch order (split, virtual request v, row group g), split slowest
  int pair = blockIdx.x >> 1;
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

// ------------------------------------------------------------ producers ---
// S-CTA staging stage = chunk c (64 dims) of the (up to 4) pages of an S tile,
// each box in slot q of the stage together with its page's 64 scales;
// O-CTA staging stage = chunks 4h..4h+3 of one page (the value dims) with
// the page's scales in slot 0.
// Page bases are read 32 pages ahead (one per lane).
__device__ __forceinline__ void producer_s(Smem& s, const CUtensorMap* map,
                                           const TcParams& p, const Work& w,
                                           uint32_t rank, int lane) {
  uint32_t stage = 0, phase = 0;
  int32_t cur = page_base(p, w, lane), nxt = page_base(p, w, 32 + lane);
  bool ok = true;
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
    for (int c = 0; c < kChunksPerPage && ok; ++c) {
      if (lane == 0) {
        if (mbar_wait(smem_u32(&s.empty8[stage]), phase ^ 1u, &s.abort_flag))
          mbar_arrive_expect_tx(smem_u32(&s.full8[stage]),
                                np * (kBox8Bytes + kScaleBytes));
        else
          ok = false;
      }
      ok = __shfl_sync(kFull, ok, 0);
      if (ok && lane < np) {
        uint8_t* st = s.ring8[stage];
        const uint32_t bar = smem_u32(&s.full8[stage]);
        tma_load_2d(smem_u32(st + lane * kBox8Bytes), map, bar, c * 64, yq);
        // scales of a page outside the pool: read those of page 0 (unused)
        const int64_t sb = bq < 0 ? 0 : bq;
        bulk_load(smem_u32(st + kBoxesPerStage * kBox8Bytes + lane * kScaleBytes),
                  p.kv_scale + sb, kScaleBytes, bar);
      }
      if (++stage == kStages8) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
  if (!ok && lane == 0) signal_abort(s, p, rank);
}

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
    for (int h = 0; h < 2 && ok; ++h) {
      if (lane == 0) {
        if (mbar_wait(smem_u32(&s.empty8[stage]), phase ^ 1u, &s.abort_flag))
          mbar_arrive_expect_tx(smem_u32(&s.full8[stage]),
                                kBoxesPerStage * kBox8Bytes + kScaleBytes);
        else
          ok = false;
      }
      ok = __shfl_sync(kFull, ok, 0);
      if (ok && lane < kBoxesPerStage) {
        uint8_t* st = s.ring8[stage];
        const uint32_t bar = smem_u32(&s.full8[stage]);
        tma_load_2d(smem_u32(st + lane * kBox8Bytes), map, bar,
                    (4 * h + lane) * 64, y);
        if (lane == 0)
          bulk_load(smem_u32(st + kBoxesPerStage * kBox8Bytes),
                    p.kv_scale + (b < 0 ? 0 : b), kScaleBytes, bar);
      }
      if (++stage == kStages8) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
  if (!ok && lane == 0) signal_abort(s, p, rank);
}

// ----------------------------------------------------------- converters ---
// Warps 2, 3, 12, 13 of the S-CTA and 2, 3, 8, 9 of the O-CTA (NT = 128).
// A stage holds 4 slots x 64 token rows x 64 E4M3 bytes = 1024 items of 16
// bytes: item (slot q, n) is row r = n / 4, quarter h = n % 4 of slot q.
// Thread t takes, slot by slot, the 256 / NT items n = t + k*NT, all loaded
// before any is converted (a load issued after a store that may alias it
// would wait for it), converts each exactly to 16 f16 (cvt e4m3x2 -> f16x2)
// and stores them as 16-byte groups 2h, 2h+1 of row r in the
// 128-byte-swizzled f16 chunk of slot q.  Rows at or past a page's length
// (and slots of pages a short tile does not have) become zeros: 0 * NaN in
// P V must not see undefined rows.  The O side multiplies by the token's
// scale in f16 (V' = e4m3 * scale); on the S side, chunk 0 of a tile
// publishes the tile's token scales (tscale[j % 4], tsready) for the
// softmax instead.
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t four, uint32_t& lo,
                                                uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(four));
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t y;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(y) : "r"(a), "r"(b));
  return y;
}

template <int NT>
__device__ __forceinline__ void converter(Smem& s, const TcParams& p,
                                          const Work& w, uint32_t rank, int t,
                                          int lane) {
  constexpr int kPer = 256 / NT;  // items per thread per slot
  uint32_t st8 = 0, ph8 = 0, st = 0, ph = 0;
  bool ok = true;
  // stages in order: S-CTA: tile j, chunk c; O-CTA: page m, half h
  const int ntiles = (w.npages + kTilePages - 1) / kTilePages;
  const int nst = rank == 0 ? ntiles * kChunksPerPage : w.npages * 2;
  for (int u = 0; u < nst && ok; ++u) {
    // Tokens of the stage's first slot that exist: slot q of an S stage is
    // page q of the tile; all slots of an O stage are the same page.
    int64_t left;
    int np;
    if (rank == 0) {
      const int j = u / kChunksPerPage;
      np = tile_pages(w, j);
      left = w.L - (w.p0 + (int64_t)j * kTilePages) * kPage;
    } else {
      np = kBoxesPerStage;
      left = w.L - (w.p0 + (int64_t)(u >> 1)) * kPage;
    }
    const int left0 =
        left <= 0 ? 0 : (left >= 4 * kPage ? 4 * kPage : (int)left);
    if (!mbar_wait(smem_u32(&s.full8[st8]), ph8, &s.abort_flag) ||
        !mbar_wait(smem_u32(&s.empty[st]), ph ^ 1u, &s.abort_flag)) {
      ok = false;
      break;
    }
    const uint8_t* src = s.ring8[st8];
    uint8_t* dst = s.ring[st * kBoxesPerStage];
    const float* scl =
        reinterpret_cast<const float*>(src + kBoxesPerStage * kBox8Bytes);
#pragma unroll 1
    for (int q = 0; q < kBoxesPerStage; ++q) {
      const int vq = q >= np ? 0 : (rank == 0 ? left0 - q * kPage : left0);
      const uint8_t* sq = src + q * kBox8Bytes;
      uint8_t* dq = dst + q * kBoxBytes;
      uint4 x[kPer];
#pragma unroll
      for (int k = 0; k < kPer; ++k)
        x[k] = *reinterpret_cast<const uint4*>(sq + (t + k * NT) * 16);
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int n = t + k * NT, r = n >> 2, h = n & 3;
        if (r >= vq) x[k] = make_uint4(0, 0, 0, 0);  // E4M3 0 -> f16 +0
        uint4 lo, hi;
        e4m3x4_to_f16x4(x[k].x, lo.x, lo.y);
        e4m3x4_to_f16x4(x[k].y, lo.z, lo.w);
        e4m3x4_to_f16x4(x[k].z, hi.x, hi.y);
        e4m3x4_to_f16x4(x[k].w, hi.z, hi.w);
        if (rank == 1) {
          // rows past the length: scale 0, not the slot's (undefined) one
          const float sv = r < vq ? scl[r] : 0.f;
          const uint32_t s2 = pack_f16(sv, sv);
          lo = make_uint4(hmul2(lo.x, s2), hmul2(lo.y, s2), hmul2(lo.z, s2),
                          hmul2(lo.w, s2));
          hi = make_uint4(hmul2(hi.x, s2), hmul2(hi.y, s2), hmul2(hi.z, s2),
                          hmul2(hi.w, s2));
        }
        uint8_t* d = dq + (r >> 3) * 1024;
        *reinterpret_cast<uint4*>(d + box_chunk_offset(r & 7, 2 * h)) = lo;
        *reinterpret_cast<uint4*>(d + box_chunk_offset(r & 7, 2 * h + 1)) = hi;
      }
    }
    const bool scales = rank == 0 && u % kChunksPerPage == 0;
    const int tj = (u / kChunksPerPage) & 3;
    if (scales) {
      for (int idx = t; idx < kTilePages * 64; idx += NT) {
        const int q = idx >> 6, r = idx & 63;
        const int vq = q >= np ? 0 : left0 - q * kPage;
        s.tscale[tj][q][r] = r < vq ? scl[idx] : 0.f;
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(smem_u32(&s.full[st]));
      mbar_arrive(smem_u32(&s.empty8[st8]));
      if (scales) mbar_arrive(smem_u32(&s.tsready[tj]));
    }
    if (++st8 == kStages8) {
      st8 = 0;
      ph8 ^= 1u;
    }
    if (++st == kStages) {
      st = 0;
      ph ^= 1u;
    }
  }
  if (!__all_sync(kFull, ok) && lane == 0) signal_abort(s, p, rank);
}

// ---------------------------------------------------------- S-CTA: MMA ----
// One issuing thread: per f16 stage (chunk c of the tile's pages) 4 MMAs of
// M=128, N=64*pages, K=16 into TMEM columns [256, 256 + 64*pages).
__device__ __forceinline__ void mma_s(Smem& s, const TcParams& p,
                                      const Work& w, uint32_t tmem,
                                      uint32_t rank) {
  if (!mbar_wait(smem_u32(&s.qready), 0, &s.abort_flag)) {
    signal_abort(s, p, rank);
    return;
  }
  tc_fence_after();
  const uint32_t d = tmem + kSCol0;
  const uint64_t qr = sdesc_sw128(smem_u32(s.qrope), 16, 1024);
  uint32_t stage = 0, phase = 0;
  const int ntiles = (w.npages + kTilePages - 1) / kTilePages;
  for (int j = 0; j < ntiles; ++j) {
    const uint32_t idesc = idesc_s(tile_pages(w, j));
    if (!mbar_wait(smem_u32(&s.sempty), (j & 1) ^ 1u, &s.abort_flag)) {
      signal_abort(s, p, rank);
      return;
    }
    tc_fence_after();
    for (int c = 0; c < kChunksPerPage; ++c) {
      if (!mbar_wait(smem_u32(&s.full[stage]), phase, &s.abort_flag)) {
        signal_abort(s, p, rank);
        return;
      }
      tc_fence_after();
      const uint64_t b =
          sdesc_sw128(smem_u32(s.ring[stage * kBoxesPerStage]), 16, 1024);
      if (c < 8) {
        mma_ts(d, tmem + 32u * c + 0, b + 0, idesc, c > 0 ? 1u : 0u);
        mma_ts(d, tmem + 32u * c + 8, b + 2, idesc, 1u);
        mma_ts(d, tmem + 32u * c + 16, b + 4, idesc, 1u);
        mma_ts(d, tmem + 32u * c + 24, b + 6, idesc, 1u);
      } else {
        mma_ss(d, qr + 0, b + 0, idesc, 1u);
        mma_ss(d, qr + 2, b + 2, idesc, 1u);
        mma_ss(d, qr + 4, b + 4, idesc, 1u);
        mma_ss(d, qr + 6, b + 6, idesc, 1u);
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

// ------------------------------------------------------ S-CTA: softmax ----
// Warps 4..11: warpgroup g = 0 (warps 4-7) owns pages 0,1 of each S tile,
// g = 1 (warps 8-11) pages 2,3.  Thread = query row r (TMEM lane).  Q is
// converted to f16 on the way in (TMEM / shared memory) and P leaves as f16
// pairs: the MMAs of this kernel multiply f16 by f16.
__device__ __forceinline__ void softmax(Smem& s, const TcParams& p,
                                        const Work& w, uint32_t tmem,
                                        uint32_t rank, int warp, int lane) {
  const int g = (warp - 4) >> 2;
  const int quad = warp & 3;
  const int r = quad * 32 + lane;
  const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
  const bool row_ok = r < w.nrows;
  const int rr = w.r_base + r;
  const int i = row_ok ? rr / p.H : 0;
  int64_t n = 0;
  if (row_ok) {
    n = p.kv_limit ? (int64_t)p.kv_limit[(int64_t)w.v * p.q_len + i]
                   : w.L - p.q_len + 1 + i;
    n = n > w.L ? w.L : (n < 0 ? 0 : n);
  }
  const int64_t qrow = (int64_t)w.b * p.q_len * p.H + rr;

  // Q row: nope part -> TMEM columns [0, 256) (column c holds elements 2c,
  // 2c+1), rope part -> shared memory in the K-major 128-B swizzled layout.
  if (g == 0) {
#pragma unroll 1
    for (int c = 0; c < 8; ++c) {
      uint32_t v[32];
      const uint4* src = p.q_nope + qrow * 64 + c * 8;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint4 x = row_ok ? src[k] : make_uint4(0, 0, 0, 0);
        v[4 * k] = bf16x2_to_f16x2(x.x);
        v[4 * k + 1] = bf16x2_to_f16x2(x.y);
        v[4 * k + 2] = bf16x2_to_f16x2(x.z);
        v[4 * k + 3] = bf16x2_to_f16x2(x.w);
      }
      tmem_st32(tmem + lane_base + 32u * c, v);
    }
    tmem_wait_st();
  } else {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint4 x = row_ok ? p.q_rope[qrow * 8 + k] : make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(s.qrope + (r >> 3) * 1024 +
                                box_chunk_offset(r & 7, k)) =
          make_uint4(bf16x2_to_f16x2(x.x), bf16x2_to_f16x2(x.y),
                     bf16x2_to_f16x2(x.z), bf16x2_to_f16x2(x.w));
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(smem_u32(&s.qready));

  float m_ref = -INFINITY, l = 0.f;
  bool ok = true;
  const uint32_t peer_pfull0 = mapa(smem_u32(&s.pfull[0]), 1);
  const int ntiles = (w.npages + kTilePages - 1) / kTilePages;
  const uint32_t bar_wg = 2 + g;  // named barrier of this warpgroup
  const float sc = p.scale_log2;
  for (int j = 0; j < ntiles; ++j) {
    const int np = tile_pages(w, j);
    const int myp = min(2, max(0, np - 2 * g));  // pages this warpgroup owns
    uint32_t s0[32], s1[32], s2[32], s3[32];
    if (ok && !mbar_wait(smem_u32(&s.sfull), j & 1, &s.abort_flag)) ok = false;
    tc_fence_after();
    if (__all_sync(kFull, ok) && myp > 0) {
      const uint32_t col = tmem + lane_base + kSCol0 + 128u * g;
      tmem_ld32(col, s0);
      tmem_ld32(col + 32, s1);
      if (myp > 1) {
        tmem_ld32(col + 64, s2);
        tmem_ld32(col + 96, s3);
      }
      tmem_wait_ld();
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&s.sempty));

    // Token scales of this warpgroup's 128 columns (pages 2g, 2g+1 of the
    // tile): s_t = scale_t * (q . e4m3_t).  Broadcast reads.
    if (ok && !mbar_wait(smem_u32(&s.tsready[j & 3]), (j >> 2) & 1,
                         &s.abort_flag))
      ok = false;
    const float* tsc = &s.tscale[j & 3][2 * g][0];
    auto apply_scale = [&](uint32_t (&a)[32], int c0) {
#pragma unroll
      for (int c = 0; c < 32; c += 4) {
        const float4 f = *reinterpret_cast<const float4*>(tsc + c0 + c);
        float x0, x1, x2, x3;
        f2unpack(fmul2(f2pack(__uint_as_float(a[c]), __uint_as_float(a[c + 1])),
                       f2pack(f.x, f.y)), x0, x1);
        f2unpack(fmul2(f2pack(__uint_as_float(a[c + 2]), __uint_as_float(a[c + 3])),
                       f2pack(f.z, f.w)), x2, x3);
        a[c] = __float_as_uint(x0);
        a[c + 1] = __float_as_uint(x1);
        a[c + 2] = __float_as_uint(x2);
        a[c + 3] = __float_as_uint(x3);
      }
    };
    if (myp > 0) {
      apply_scale(s0, 0);
      apply_scale(s1, 32);
    }
    if (myp > 1) {
      apply_scale(s2, 64);
      apply_scale(s3, 96);
    }

    // Visible columns of this row among this warpgroup's 128 columns.
    const int64_t t0 = (w.p0 + (int64_t)j * kTilePages + 2 * g) * kPage;
    const int64_t nv = n - t0;
    const int nvis = nv <= 0 ? 0 : (nv >= 64 * myp ? 64 * myp : (int)nv);
    // Columns this row may not see become -inf (a select: garbage or NaN in
    // a masked column never propagates).  Only the tiles at the end of the
    // split need it; on every other tile all 128 columns of every row of the
    // warp are visible and the scores are used as loaded.
    if (!__all_sync(kFull, nvis == 128)) {
      auto mask = [&](uint32_t (&a)[32], int c0) {
#pragma unroll
        for (int c = 0; c < 32; ++c)
          a[c] = c0 + c < nvis ? a[c] : __float_as_uint(-INFINITY);
      };
      mask(s0, 0);
      mask(s1, 32);
      mask(s2, 64);
      mask(s3, 96);
    }
    auto xs = [&](int c) -> float {
      return __uint_as_float(c < 32 ? s0[c] : c < 64 ? s1[c - 32]
                                    : c < 96 ? s2[c - 64] : s3[c - 96]);
    };
    // Row maximum of the raw scores; the scale is positive, so the maximum
    // of the scaled scores is the scaled maximum (rounding is monotone).
    float mx[16];
#pragma unroll
    for (int c = 0; c < 16; ++c)
      mx[c] = fmaxf(max3(xs(c), xs(c + 16), xs(c + 32)),
                    max3(max3(xs(c + 48), xs(c + 64), xs(c + 80)), xs(c + 96),
                         xs(c + 112)));
    const float m5a = max3(mx[0], mx[1], mx[2]), m5b = max3(mx[3], mx[4], mx[5]);
    const float m5c = max3(mx[6], mx[7], mx[8]), m5d = max3(mx[9], mx[10], mx[11]);
    const float m5e = max3(mx[12], mx[13], mx[14]);
    const float mt_own =
        max3(max3(m5a, m5b, m5c), max3(m5d, m5e, mx[15]), -INFINITY) * sc;
    // Row maximum over the whole tile: exchange with the other warpgroup.
    s.xch[g][r] = mt_own;
    named_bar_sync(1, 256);
    const float mt = fmaxf(mt_own, s.xch[g ^ 1][r]);
    named_bar_sync(1, 256);  // both read before the next tile overwrites
    float alpha = 1.f;
    if (mt > -INFINITY) {
      if (m_ref == -INFINITY) {
        m_ref = mt;  // first visible token of this row: O is still zero
      } else if (mt > m_ref + kTau) {
        alpha = ex2(m_ref - mt);
        l *= alpha;
        m_ref = mt;
      }
    }
    // A row with nothing visible yet keeps m_ref = -inf: shift by 0 instead
    // so every p is ex2(-inf) = 0, not NaN.
    const float shift = m_ref == -INFINITY ? 0.f : m_ref;

    // P of both pages, packed f16 pairs, computed before any wait for a
    // message slot so the exponentials stay off the cross-SM round trip.
    uint32_t pk0[32], pk1[32];
    // p = 2^(x * scale - m_ref): one packed FMA per pair of columns, the row
    // sum in two packed accumulators.
    const uint64_t sc2 = f2pack(sc, sc), nshift2 = f2pack(-shift, -shift);
    auto make_page = [&](const uint32_t (&lo)[32], const uint32_t (&hi)[32],
                         uint32_t (&pk)[32]) {
      uint64_t acc0 = f2pack(0.f, 0.f), acc1 = acc0;
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const int c0 = 2 * c;
        const float xa = __uint_as_float(c0 < 32 ? lo[c0] : hi[c0 - 32]);
        const float xb = __uint_as_float(c0 + 1 < 32 ? lo[c0 + 1] : hi[c0 - 31]);
        float ya, yb;
        f2unpack(ffma2(f2pack(xa, xb), sc2, nshift2), ya, yb);
        const float pa = ex2(ya), pb = ex2(yb);
        if (c & 1) acc1 = fadd2(acc1, f2pack(pa, pb));
        else acc0 = fadd2(acc0, f2pack(pa, pb));
        pk[c] = pack_f16(pa, pb);
      }
      float a0, a1, b0, b1;
      f2unpack(acc0, a0, a1);
      f2unpack(acc1, b0, b1);
      l += (a0 + a1) + (b0 + b1);
    };
    if (myp > 0) make_page(s0, s1, pk0);
    if (myp > 1) make_page(s2, s3, pk1);

    // Ship one page: wait for its slot, store, hand it to the peer.  Slot
    // k = (2g + q) belongs to this warpgroup and page position alone (four
    // slots, four pages per tile), so its uses are sequential here.
    auto emit_page = [&](const uint32_t (&pk)[32], int q) {
      const int msg = j * kTilePages + 2 * g + q;  // page index in the split
      const int k = msg % kNP;
      const int u = msg / kNP;  // use index of slot k
      if (u > 0 && ok &&
          !mbar_wait(smem_u32(&s.pempty[k]), (u - 1) & 1, &s.abort_flag))
        ok = false;
      uint8_t* stg = s.pslot[k];
#pragma unroll
      for (int cc = 0; cc < 8; ++cc)
        // K-major, 128-B swizzle: 8-row groups 1024 B apart, 16-B chunk cc
        // of row r at position cc ^ (r % 8) within its 128-B row.
        *reinterpret_cast<uint4*>(stg + (r >> 3) * 1024 +
                                  box_chunk_offset(r & 7, cc)) =
            make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
      // The tile's rescale travels with its first page only.
      const bool first = (g == 0 && q == 0);
      reinterpret_cast<float*>(stg + kAlphaOff)[r] = first ? alpha : 1.f;
      const bool any = __any_sync(kFull, first && alpha != 1.f);
      if (lane == 0)
        reinterpret_cast<uint32_t*>(stg + kFlagOff)[quad] = any ? 1u : 0u;
      fence_proxy_async_smem();
      named_bar_sync(bar_wg, 128);
      if ((warp & 3) == 0 && lane == 0 && ok && !s.abort_flag)
        // The peer armed pfull[k] with the byte count itself.
        bulk_copy_to_peer(mapa(smem_u32(stg), 1), smem_u32(stg), kPMsgBytes,
                          peer_pfull0 + 8u * k);
    };
    if (myp > 0) emit_page(pk0, 0);
    if (myp > 1) emit_page(pk1, 1);
  }

  // Final statistics: l = sum of both warpgroups' partial sums.
  s.xch[g][r] = l;
  named_bar_sync(1, 256);
  if (g == 0) {
    const float lt = l + s.xch[1][r];
    if (row_ok) {
      const int64_t rows = (int64_t)p.B * p.q_len * p.H;
      const int64_t part = (int64_t)w.split * (p.V / p.B) + w.shard;
      p.LSE_part[part * rows + qrow] =
          lt > 0.f ? (m_ref + log2f(lt)) * 0.69314718055994531f : -INFINITY;
    }
    s.fin[r] = lt > 0.f ? 1.f / lt : 0.f;
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

// ---------------------------------------------------------- O-CTA: MMA ----
__device__ __forceinline__ void mma_o(Smem& s, const TcParams& p,
                                      const Work& w, uint32_t tmem,
                                      uint32_t rank) {
  uint32_t stage = 0, phase = 0, ev = 0;
  bool ok = true;
  // Each P message lands by a bulk copy whose bytes complete on pfull[k];
  // this CTA arms the barrier (one arrival + the byte count) itself, so the
  // sender needs no cluster-scope arrive: the first use of each slot is armed
  // at set-up, the next one as soon as a message has been received.
  for (int m = 0; m < w.npages && ok; ++m) {
    const int k = m % kNP;
    if (!mbar_wait(smem_u32(&s.pfull[k]), (m / kNP) & 1, &s.abort_flag)) {
      ok = false;
      break;
    }
    if (m + kNP < w.npages)
      mbar_arrive_expect_tx(smem_u32(&s.pfull[k]), kPMsgBytes);
    const uint32_t* fl =
        reinterpret_cast<const uint32_t*>(s.pslot[k] + kFlagOff);
    if (fl[0] | fl[1] | fl[2] | fl[3]) {
      // Rows raised their running max: let the correction warps rescale O
      // once every earlier product has landed.
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
    const uint64_t a = sdesc_sw128(smem_u32(s.pslot[k]), 16, 1024);
    for (int h = 0; h < 2; ++h) {
      if (!mbar_wait(smem_u32(&s.full[stage]), phase, &s.abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // B = V (f16): MN-major, next 64 dims one chunk (8 KB) on, next 8
      // tokens 1 KB on; each 16-token K step advances 2048 B (128 units).
      const uint64_t b = sdesc_sw128(smem_u32(s.ring[stage * kBoxesPerStage]),
                                     kBoxBytes, 1024);
      const uint32_t d = tmem + 256u * h;
      mma_ss(d, a + 0, b + 0, kIdescO, m > 0 ? 1u : 0u);
      mma_ss(d, a + 2, b + 128, kIdescO, 1u);
      mma_ss(d, a + 4, b + 256, kIdescO, 1u);
      mma_ss(d, a + 6, b + 384, kIdescO, 1u);
      mma_commit(smem_u32(&s.empty[stage]));
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (!ok) break;
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
  const float inv = s.fin[r];
  const bool row_ok = r < w.nrows;
  const int64_t rows = (int64_t)p.B * p.q_len * p.H;
  const int64_t part = (int64_t)w.split * (p.V / p.B) + w.shard;
  float* dst = p.O_part +
               (part * rows + (int64_t)w.b * p.q_len * p.H + w.r_base + r) *
                   MLA_VALUE_DIM;
#pragma unroll 1
  for (int c0 = 0; c0 < MLA_VALUE_DIM; c0 += 32) {
    uint32_t v[32];
    tmem_ld32(tmem + lane_base + c0, v);
    tmem_wait_ld();
    if (row_ok) {
      float4* d4 = reinterpret_cast<float4*>(dst + c0);
#pragma unroll
      for (int e = 0; e < 8; ++e)
        d4[e] = make_float4(__uint_as_float(v[4 * e]) * inv,
                            __uint_as_float(v[4 * e + 1]) * inv,
                            __uint_as_float(v[4 * e + 2]) * inv,
                            __uint_as_float(v[4 * e + 3]) * inv);
    }
  }
}

// ------------------------------------------------------------- kernel ----
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_partial_tc_fp8_kernel(const __grid_constant__ CUtensorMap kv_map,
                              const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();
  const Work w = pair_work(p);

  if (threadIdx.x == 0) {
    s.abort_flag = 0;
    s.ctl_slot = 0;
    s.ctl_final = 0;
    const uint32_t nconv = 4;  // converter warps
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_u32(&s.full[i]), nconv);
      mbar_init(smem_u32(&s.empty[i]), 1);
    }
    for (int i = 0; i < kStages8; ++i) {
      mbar_init(smem_u32(&s.full8[i]), 1);
      mbar_init(smem_u32(&s.empty8[i]), nconv);
    }
    for (int i = 0; i < 4; ++i) mbar_init(smem_u32(&s.tsready[i]), nconv);
    mbar_init(smem_u32(&s.sfull), 1);
    mbar_init(smem_u32(&s.sempty), 8);   // the 8 softmax warps
    for (int i = 0; i < kNP; ++i) {
      mbar_init(smem_u32(&s.pfull[i]), 1);
      mbar_init(smem_u32(&s.pempty[i]), 1);
    }
    mbar_init(smem_u32(&s.drain), 2);
    mbar_init(smem_u32(&s.corr_done), 4);
    mbar_init(smem_u32(&s.fin_full), 1);
    mbar_init(smem_u32(&s.qready), 8);
    if (rank == 1 && w.npages > 0) {
      mbar_arrive_expect_tx(smem_u32(&s.fin_full), kRows * 4);
      for (int k = 0; k < kNP && k < w.npages; ++k)
        mbar_arrive_expect_tx(smem_u32(&s.pfull[k]), kPMsgBytes);
    }
    fence_mbar_init();
    prefetch_tmap(&kv_map);
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

  // Teardown, repeated at the end of every role (roles never rejoin, so no
  // warp asks setmaxnreg for registers back).
  auto teardown = [&]() {
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
    cluster_sync();
  };

  if (w.npages > 0 && rank == 0) {
    if (warp < 4 || warp >= 12) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsControl));
      if (warp == 0) {
        producer_s(s, &kv_map, p, w, rank, lane);
      } else if (warp == 1) {
        if (lane == 0) mma_s(s, p, w, tmem, rank);
        __syncwarp();
      } else if (warp < 4 || warp < 14) {
        const int cw = warp < 4 ? warp - 2 : warp - 10;  // 0..3
        converter<128>(s, p, w, rank, cw * 32 + lane, lane);
      }
      teardown();
      return;
    }
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    softmax(s, p, w, tmem, rank, warp, lane);
    teardown();
    return;
  }
  if (w.npages > 0) {
    if (warp == 0)
      producer_o(s, &kv_map, p, w, rank, lane);
    else if (warp == 1) {
      if (lane == 0) mma_o(s, p, w, tmem, rank);
      __syncwarp();
    } else if (warp < 4 || warp == 8 || warp == 9) {
      const int cw = warp < 4 ? warp - 2 : warp - 6;  // 0..3
      converter<128>(s, p, w, rank, cw * 32 + lane, lane);
    } else if (warp < 8) {
      correct_and_store(s, p, w, tmem, rank, warp, lane);
    }
  } else if (warp >= 4 && warp < 8) {
    // No tokens for this split: O = 0, LSE = -inf.
    const int r = (warp & 3) * 32 + lane;
    if (r < w.nrows) {
      const int64_t rows = (int64_t)p.B * p.q_len * p.H;
      const int64_t part = (int64_t)w.split * (p.V / p.B) + w.shard;
      const int64_t orow =
          part * rows + (int64_t)w.b * p.q_len * p.H + w.r_base + r;
      if (rank == 0) {
        p.LSE_part[orow] = -INFINITY;
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
  p.B = a.B;
  p.q_len = a.q_len;
  p.H = a.H;
  p.V = a.B * a.num_shards;
  p.num_splits = a.num_splits;
  p.G = (a.q_len * a.H + kRows - 1) / kRows;
  p.scale_log2 = a.sm_scale * 1.4426950408889634f;
  p.O_part = a.O_part;
  p.LSE_part = a.LSE_part;
  p.status = a.status;
  const int64_t pairs = (int64_t)p.V * p.num_splits * p.G;
  if (pairs * 2 > 0x7fffffff) return fail(MLA_ERR_INVALID_ARG, "grid too large");
  CUtensorMap map;
  int rc = make_kv_tensor_map_fp8_plain(&map, a.kv, a.num_slots);
  if (rc != MLA_OK) return rc;
  cudaError_t e = cudaFuncSetAttribute(
      mla_partial_tc_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
      kSmemBytes);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(tc fp8)");
  mla_partial_tc_fp8_kernel<<<(unsigned)(pairs * 2), kThreads, kSmemBytes,
                              a.stream>>>(map, p);
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
