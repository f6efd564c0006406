// mla_tc.cu -- tensor-core (tcgen05 / TMEM / TMA) partial MLA decode.
//
// What it computes is stated in include/mla_decode.h (mla_decode_partial):
// weight-absorbed MLA decode over the paged latent KV ([VRAM-KV],
// [VRAM-POOL]), partial (O, LSE) per KV split and context shard ([K3-MLA],
// [K3-SPLIT]), causal among the q_len draft tokens ([K3-INTRO]).
//
// Design (GB300, one CTA per SM, clusters of four):
//   All H*q_len query rows of a request share one latent KV row per token, so
//   S = Q K^T (576-d) and O = P V (512-d, V = the c_kv columns of the same
//   row) are dense contractions with M = query rows.  A 128-row fp32 O
//   accumulator over 512 values fills all 512 TMEM columns of an SM, so the
//   scores and the output of a 128-row group live on two SMs.  An SM's TMA
//   engine lands 64-row KV boxes at ~45 B/clk, while an M = 128 bf16 MMA
//   consumes 64 B/clk of K, so the KV tile of one MMA is split over two SMs
//   with the CTA-pair (cta_group::2) MMA, M = 256 rows = two row groups:
//     ranks 0,1, the "S pair": rank r owns row group 2u + r: Q_nope (bf16
//       pairs) in TMEM columns [0, 256), Q_rope in shared memory, both
//       brought by TMA (Q_nope through the P slots, idle until the first S
//       tile, and ring stages 4..7, then copied into TMEM by tcgen05.cp),
//       one S buffer of 256 columns (an S tile = 4 pages = 256 tokens).  Rank r loads pages 2r, 2r+1 of every tile in 16-KB stages
//       (one 64-dim chunk of its two pages, 128-byte swizzled TMA boxes);
//       each stage feeds 4 pair MMAs of M=256, N=256, K=16 issued by rank
//       0.  Two softmax
//       warpgroups per CTA own two pages each, exchange row maxima once per
//       tile, keep base-2 running statistics with lazy rescaling, and ship
//       each page's P (bf16, K-major, 128-byte swizzled) plus rescale
//       factors to their O-CTA with a bulk shared-memory copy.
//     ranks 2,3, the "O pair": rank 2+r holds O (128 x 512 fp32) of row group
//       2u + r in all of its TMEM and loads half of V: dims [256n + 128r,
//       +128) of each page for the two 256-wide halves n, one 32-KB stage
//       per page; each page feeds 8 pair MMAs of M=256, N=256, K=16 (A = P,
//       B = V MN-major) issued by rank 2.  Correction warps rescale O rows
//       when an S-CTA raised a running max; then warps 4..11 write the
//       normalised O_part rows, staged through the idle ring so that every
//       store instruction writes full 128-byte lines.
//   Per SM the TMA then lands 16 KB per 512 tensor cycles.  Every wait is
//   bounded (ptx_sm103.cuh); a timeout sets MLA_STATUS_WAIT_TIMEOUT and the
//   cluster finishes early.
#include <cuda_bf16.h>

#include <cstring>

#include "mla_combine.cuh"
#include "mla_tma.cuh"
#include "ptx_sm103.cuh"

namespace mla {
namespace {

using namespace ptx;

constexpr int kThreads = 384;        // 12 warps = 3 warpgroups
constexpr int kCtas = 4;             // S pair (ranks 0,1) + O pair (ranks 2,3)
constexpr int kStages = 8;           // S-CTA: 16-KB ring stages (2 boxes each)
constexpr int kBoxesPerStage = 2;
constexpr int kStagesO = 4;          // O-CTA: 32-KB stages (4 boxes, a page)
constexpr int kBoxesO = 4;
constexpr int kTilePages = 4;        // pages per S tile (N = 256), 2 per S-CTA
constexpr int kNP = 4;               // P message slots (page index mod 4)
constexpr int kRows = MLA_ROWS_PER_UNIT / 2;  // 128 query rows per CTA
constexpr int kPage = MLA_PAGE_SIZE;           // 64 tokens
constexpr int kPBytes = kRows * kPage * 2;          // 16384
constexpr int kAlphaOff = kPBytes;                  // float alpha[128]
constexpr int kFlagOff = kPBytes + kRows * 4;       // uint32 flags[4]
constexpr int kPMsgBytes = kFlagOff + 16;           // 16912 = 1057 x 16
constexpr int kPeerFlagOff = kPMsgBytes;            // rank 2: rank 1's flags
constexpr int kPSlotStride = 17408;                 // 17 KB, 1024-aligned
constexpr uint32_t kSCol0 = 256;                    // S buffer columns
constexpr float kTau = 8.f;          // lazy-rescale threshold (log2 units)
constexpr uint32_t kFull = 0xffffffffu;
constexpr uint16_t kMaskS = 0x3;     // cluster ranks of the S pair
constexpr uint16_t kMaskO = 0xC;     // cluster ranks of the O pair
// Register split of the S-CTAs (setmaxnreg): 384 threads launch with 168
// registers each (64,512); the producer/MMA warpgroup gives registers away so
// the two softmax warpgroups can hold a 128 x 256 fp32 score tile.  The split
// is one-way: nobody asks for registers back before the CTA exits.
constexpr int kRegsLaunch = 168;
constexpr int kRegsControl = 64;
constexpr int kRegsSoftmax = 216;
static_assert(128 * kRegsControl + 256 * kRegsSoftmax <= kThreads * kRegsLaunch,
              "register split exceeds the launch allocation");

constexpr uint32_t kIdescS = idesc_bf16_f32(256, 256, false, false);
constexpr uint32_t kIdescO = idesc_bf16_f32(256, 256, false, true);

struct __align__(1024) Smem {
  uint8_t ring[kStages * kBoxesPerStage][kBoxBytes];  // 128 KB
  uint8_t qrope[kRows * 128];                         // S-CTA: Q_rope rows
  uint8_t pslot[kNP][kPSlotStride];
  float fin[kRows];
  float xch[2][kRows];      // S-CTA: per-warpgroup row maxima / partial sums
  uint64_t full[kStages];   // pair leader: the stage landed in both CTAs
  uint64_t empty[kStages];  // every CTA: its half of the stage was consumed
  uint64_t sfull;           // S-CTAs: the S tile is in TMEM
  uint64_t sempty;          // rank 0: both S-CTAs read the S tile (16 warps)
  uint64_t pfull[kNP];      // O-CTAs: the P message of slot k landed here
  uint64_t pready[kNP];     // rank 2: rank 3's message of slot k landed
  uint64_t pempty[kNP];     // S-CTAs: slot k consumed by the O pair
  uint64_t drain;           // O-CTAs: all earlier pair MMAs completed
  uint64_t corr_done;       // rank 2: both O-CTAs finished a rescale
  uint64_t tail_full[kStagesO];   // O-CTAs: a page to sanitise landed here
  uint64_t tail_ready[kStagesO];  // rank 2: both halves of that page sanitised
  uint64_t fin_full;        // O-CTAs: 1/l of every row arrived
  uint64_t epi_go;          // O-CTAs: the epilogue may read O (warps 4-7)
  uint64_t qready;          // rank 0: both S-CTAs' query boxes landed
  uint64_t qbar;            // S-CTAs: the query boxes landed
  uint64_t qmoved;          // S-CTAs: Q_nope is in TMEM (its boxes are free)
  uint32_t tmem_base;
  int abort_flag;
  int ctl_slot;
  int ctl_final;
  int ctl_last;  // fused combine: this cluster wrote the unit's last part
};
constexpr int kSmemBytes = (int)sizeof(Smem) + 1024;
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
static_assert(kPMsgBytes % 16 == 0, "bulk copy size");
static_assert(kPeerFlagOff + 16 <= kPSlotStride, "P slot layout");

struct TcParams {
  const uint4* q_nope;     // bf16 [B, q_len, H, 512] as 16-B chunks
  const uint4* q_rope;     // bf16 [B, q_len, H, 64]
  int64_t num_slots;
  const int32_t* r2t;
  int64_t r2t_stride;
  const int32_t* seq_lens;
  const int32_t* kv_limit;
  const int32_t* split_pages;  // [V, num_splits + 1] page boundaries or NULL
  const int32_t* work;         // unit ids in launch order or NULL
  int B, q_len, H, V, num_splits, U;  // U = row pairs (256 rows) per request
  float scale_log2;        // sm_scale * log2(e)
  float* O_part;
  float* LSE_part;
  int* status;
  int q_box_rows;          // rows of a query TMA box: min(128, B * q_len * H)
  int o_tma;               // O_part rows leave by TMA store (o_map is valid)
  int o_bf16;              // O_part holds bf16 values (else fp32)
  __nv_bfloat16* out;      // fused combine (NULL counters: partials only)
  float* lse_out;
  int* counters;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
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
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Arrive on a barrier of the pair leader `lead`: a local arrive when this CTA
// is the leader, otherwise a release at cluster scope, which publishes this
// thread's earlier writes (shared memory, TMEM stores) to the leader.
__device__ __forceinline__ void arrive_leader(uint32_t bar, uint32_t rank,
                                              uint32_t lead) {
  if (rank == lead)
    mbar_arrive(bar);
  else
    mbar_arrive_cluster(mapa(bar, lead));
}

// The same for a signal that only reports completed work: the thread has
// already waited for its own TMEM loads or stores (tcgen05.wait) or seen the
// data land on a barrier, so nothing remains to publish and the arrive can be
// relaxed.  A remote release costs the issuing thread hundreds to thousands
// of cycles under load; a relaxed remote arrive a few.
__device__ __forceinline__ void signal_leader(uint32_t bar, uint32_t rank,
                                              uint32_t lead) {
  if (rank == lead) {
    mbar_arrive(bar);
  } else {
    asm volatile(
        "mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(
            mapa(bar, lead))
        : "memory");
  }
}

// Record a failed wait: device status and every CTA's abort flag.
__device__ __forceinline__ void signal_abort(Smem& s, const TcParams& p,
                                             uint32_t rank) {
  if (p.status) atomicOr(p.status, MLA_STATUS_WAIT_TIMEOUT);
  s.abort_flag = 1;
  for (uint32_t c = 0; c < kCtas; ++c)
    if (c != rank) st_cluster_u32(mapa(smem_u32(&s.abort_flag), c), 1u);
}

// Work of one cluster: unit id (split, virtual request v, row pair u) =
// (split * V + v) * U + u, the cluster's index or, with a work list, the
// list's entry at that index (an entry that names no unit: skip); this
// CTA's row group is 2u + (rank & 1).
struct Work {
  int v, b, shard, split, r_base, nrows, npages;
  int m_san;  // first page of the range holding a token at or past nmin
  int64_t L, p0;
  int64_t nmin;  // fewest tokens any query of the request sees
};

// The cluster's unit id, or -1 for a work-list entry outside [0, units).
__device__ __forceinline__ int cluster_unit(const TcParams& p) {
  const int k = blockIdx.x / kCtas;
  if (!p.work) return k;
  const int unit = p.work[k];
  return unit < 0 || (int64_t)unit >= (int64_t)p.V * p.num_splits * p.U ? -1
                                                                         : unit;
}

__device__ __forceinline__ Work unit_work(const TcParams& p, int unit,
                                          uint32_t rank) {
  Work w;
  const int u = unit % p.U;
  unit /= p.U;
  w.v = unit % p.V;
  w.split = unit / p.V;
  w.b = w.v % p.B;
  w.shard = w.v / p.B;
  const int R = p.q_len * p.H;
  w.r_base = (2 * u + (int)(rank & 1)) * kRows;
  w.nrows = max(0, min(kRows, R - w.r_base));
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
  // Tokens in [nmin, L) are visible to some query rows of the request and
  // masked for others; tokens at or past L to none.  The pages that hold any
  // of them are sanitised before P V reads them (producer_o).
  int64_t nmin = L - p.q_len + 1;
  if (p.kv_limit) {
    nmin = L;
    for (int i = 0; i < p.q_len; ++i) {
      const int64_t n = p.kv_limit[(int64_t)w.v * p.q_len + i];
      nmin = n < nmin ? n : nmin;
    }
  }
  w.nmin = nmin < 0 ? 0 : (nmin > L ? L : nmin);
  const int64_t m_san = w.nmin / kPage - w.p0;
  w.m_san = (int)(m_san < 0 ? 0 : (m_san > w.npages ? w.npages : m_san));
  return w;
}

__device__ __forceinline__ int tile_pages(const Work& w, int j) {
  return min(kTilePages, w.npages - j * kTilePages);
}

// Two bf16 values with every non-finite one (NaN, +-Inf) replaced by +0.
__device__ __forceinline__ uint32_t bf16x2_finite_or_zero(uint32_t x) {
  uint32_t keep = 0;
  if ((x & 0x7F80u) != 0x7F80u) keep |= 0xFFFFu;
  if ((x & 0x7F800000u) != 0x7F800000u) keep |= 0xFFFF0000u;
  return x & keep;
}

// The page-table entry of page m of the unit's range as stored (0 past the
// range), and its check: the base slot, or -1 if it lies outside the pool.
// Split so that a load can be put in flight before its value is needed.
__device__ __forceinline__ int32_t page_entry(const TcParams& p, const Work& w,
                                              int m) {
  if (m >= w.npages) return 0;
  return p.r2t[(int64_t)w.v * p.r2t_stride + (w.p0 + m) * kPage];
}
__device__ __forceinline__ int32_t checked_base(const TcParams& p, int32_t base) {
  if (base < 0 || (base & (kPage - 1)) || (int64_t)base + kPage > p.num_slots)
    return -1;
  return base;
}
__device__ __forceinline__ int32_t page_base(const TcParams& p, const Work& w,
                                             int m) {
  return checked_base(p, page_entry(p, w, m));
}

// S-CTA, warp 0, at kernel entry: initialise the query barriers and put the
// query rows of this CTA's row group in flight (boxes of 64 values x
// q_box_rows rows): Q_nope dims 0..255 into the four P slots, dims 256..511
// into ring stages 4..7, Q_rope into its operand buffer, all on qbar.  Lane
// k issues box k: a thread's TMA loads are processed one after another
// (~0.25 us each whatever their size), loads of different threads side by
// side.
constexpr int kQRingStage0 = 4;
static_assert(kQRingStage0 + 4 <= kStages, "query boxes in the ring");
__device__ __forceinline__ void issue_query(Smem& s, const CUtensorMap* qn_map,
                                            const CUtensorMap* qr_map,
                                            const TcParams& p, int unit,
                                            uint32_t rank, int lane) {
  const int u = unit % p.U;
  const int v = (unit / p.U) % p.V;
  const int b = v % p.B;
  const int qy = b * p.q_len * p.H + (2 * u + (int)(rank & 1)) * kRows;
  const uint32_t qbar = smem_u32(&s.qbar);
  if (lane == 0) {
    mbar_init(qbar, 1);
    mbar_init(smem_u32(&s.qmoved), 1);  // the pair commit after the copies
    fence_mbar_init();
    prefetch_tmap(qn_map);
    prefetch_tmap(qr_map);
    const uint32_t box = (uint32_t)p.q_box_rows * 128u;
    mbar_arrive_expect_tx(qbar, 9 * box);
  }
  __syncwarp();
  if (lane < 8) {
    const uint32_t dst =
        lane < 4 ? smem_u32(s.pslot[lane])
                 : smem_u32(s.ring[(kQRingStage0 + lane - 4) * kBoxesPerStage]);
    tma_load_3d(dst, qn_map, qbar, 64 * lane, qy, 0);
  } else if (lane == 8) {
    tma_load_3d(smem_u32(s.qrope), qr_map, qbar, 0, qy, 0);
  }
}

// ------------------------------------------------------- S-CTA producers ---
// Rank r loads pages 2r, 2r+1 of every S tile; stage = one 64-dim chunk of
// those pages (the pair MMA's N = 256 rows: rank 0's 128, then rank 1's).
// The bytes of both CTAs complete on the leader's full barrier, which the
// leader arms with the tile's total; each CTA refills a stage once the pair
// MMA released it (empty, multicast to both).  Page bases are read 32 pages
// ahead (one per lane) so a TMA issue never waits on a dependent global
// load.  Pages of a short last tile that are not loaded leave stale bytes in
// the S columns they feed, which the softmax masks.  A thread's TMA loads
// are processed one after another (~0.25 us each), so the first tile's
// chunks 0..7, which fill the empty ring, are issued by 16 lanes at once
// (chunks 4..7 once the query has left their stages); later chunks, paced
// by the MMA, by lanes 0 and 1 (more lanes in flight there measured slower).
__device__ __forceinline__ void producer_s(Smem& s, const CUtensorMap* map,
                                           const TcParams& p, const Work& w,
                                           uint32_t rank, int lane,
                                           int32_t cur, int32_t nxt) {
  // cur, nxt: the raw page-table entries of pages lane and 32 + lane
  cur = checked_base(p, cur);
  nxt = checked_base(p, nxt);
  static_assert(kStages < kBf16BoxesPerPage && kQRingStage0 == kStages / 2,
                "the ring's first pass lies in tile 0");
  bool ok = true;
  const uint32_t full0 = mapa(smem_u32(&s.full[0]), 0);
  const int ntiles = (w.npages + kTilePages - 1) / kTilePages;
  {
    // Tile 0, chunks 0..7: lanes 2i, 2i + 1 issue chunk i of both pages.
    const int np = tile_pages(w, 0);
    const int mine = min(2, max(0, np - 2 * (int)rank));
    const int32_t bq = __shfl_sync(kFull, cur, 2 * (int)rank + (lane & 1));
    const int32_t yq = bq < 0 ? (int32_t)p.num_slots : bq;
    if (lane < mine && bq < 0 && p.status) atomicOr(p.status, MLA_STATUS_BAD_SLOT);
    const int i = lane >> 1;
    for (int half = 0; half < 2; ++half) {
      if (half == 1) {
        // Stages 4..7 hold the query's c_kv dims 256..511 until the softmax
        // has moved them into tensor memory.
        if (lane == 0 && !mbar_wait(smem_u32(&s.qmoved), 0, &s.abort_flag))
          ok = false;
        ok = __shfl_sync(kFull, ok, 0);
        if (!ok) break;
      }
      const int c = half * kQRingStage0 + i;  // chunk = ring stage
      if (i < kQRingStage0) {
        if (rank == 0 && (lane & 1) == 0)
          mbar_arrive_expect_tx(smem_u32(&s.full[c]), np * kBoxBytes);
        if ((lane & 1) < mine)
          tma_load_2d_pair(smem_u32(s.ring[c * kBoxesPerStage + (lane & 1)]),
                           map, full0 + 8u * c, c * 64, yq);
      }
    }
  }
  uint32_t stage = 0, phase = 1;  // the ring's second pass
  for (int j = 0; j < ntiles && ok; ++j) {
    const int m0 = j * kTilePages;
    if (m0 % 32 == 0 && m0 > 0) {
      cur = nxt;
      nxt = page_base(p, w, m0 + 32 + lane);
    }
    const int np = tile_pages(w, j);
    const int mine = min(2, max(0, np - 2 * (int)rank));
    // Lane q < mine loads page 2r + q of the tile (a page outside the pool
    // reads a row past the end, which TMA fills with zeros).
    const int32_t bq =
        __shfl_sync(kFull, cur, (m0 + 2 * (int)rank + (lane & 1)) & 31);
    const int32_t yq = bq < 0 ? (int32_t)p.num_slots : bq;
    if (j > 0 && lane < mine && bq < 0 && p.status)
      atomicOr(p.status, MLA_STATUS_BAD_SLOT);
    for (int c = j == 0 ? kStages : 0; c < kBf16BoxesPerPage && ok; ++c) {
      if (lane == 0) {
        if (mbar_wait(smem_u32(&s.empty[stage]), phase ^ 1u, &s.abort_flag)) {
          if (rank == 0)
            mbar_arrive_expect_tx(smem_u32(&s.full[stage]), np * kBoxBytes);
        } else {
          ok = false;
        }
      }
      ok = __shfl_sync(kFull, ok, 0);
      if (ok && lane < mine)
        tma_load_2d_pair(smem_u32(s.ring[stage * kBoxesPerStage + lane]), map,
                         full0 + 8u * stage, c * 64, yq);
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
  if (!ok && lane == 0) signal_abort(s, p, rank);
}

// ------------------------------------------------------- O-CTA producers ---
// Rank 2+h loads dims [256n + 128h, +128) of every page for n = 0, 1: one
// stage of 4 boxes (box 2n + i = dims 256n + 128h + 64i), bytes of both CTAs
// completing on rank 2's full barrier.  A masked token gets p = 0 exactly,
// but 0 * NaN (or 0 * Inf) would still poison O = P V.  So the pages from
// the one holding token nmin onwards (the draft tokens that only some query
// rows see, and the request's partly filled last page) land on the CTA's
// own tail barrier of their stage instead: rows at or past the length,
// which can hold anything, are zeroed; rows in [nmin, L) keep their finite
// values and get +0 for every non-finite one.  A query that sees such a
// token has a NaN score for it already (the S side reads the bytes as they
// are), which makes its whole row NaN, as the definition says; a query that
// does not see it now adds exactly 0.  Both CTAs then report to rank 2
// (tail_ready of the stage).
__device__ __forceinline__ void producer_o(Smem& s, const CUtensorMap* map,
                                           const TcParams& p, const Work& w,
                                           uint32_t rank, int lane) {
  uint32_t stage = 0, phase = 0;
  int32_t cur = page_base(p, w, lane), nxt = page_base(p, w, 32 + lane);
  bool ok = true;
  const int h = (int)rank - 2;
  const uint32_t full0 = mapa(smem_u32(&s.full[0]), 2);
  for (int m = 0; m < w.npages && ok; ++m) {
    if (m % 32 == 0 && m > 0) {
      cur = nxt;
      nxt = page_base(p, w, m + 32 + lane);
    }
    const int32_t b = __shfl_sync(kFull, cur, m & 31);
    const int32_t y = b < 0 ? (int32_t)p.num_slots : b;
    const int64_t t0 = (w.p0 + m) * kPage;
    const bool san = m >= w.m_san;
    const uint32_t tail_full = smem_u32(&s.tail_full[stage]);
    if (lane == 0) {
      if (mbar_wait(smem_u32(&s.empty[stage]), phase ^ 1u, &s.abort_flag)) {
        if (san)
          mbar_arrive_expect_tx(tail_full, kBoxesO * kBoxBytes);
        else if (rank == 2)
          mbar_arrive_expect_tx(smem_u32(&s.full[stage]),
                                2 * kBoxesO * kBoxBytes);
      } else {
        ok = false;
      }
    }
    ok = __shfl_sync(kFull, ok, 0);
    if (ok && lane < kBoxesO) {
      const uint32_t dst = smem_u32(s.ring[stage * kBoxesO + lane]);
      const int x = 256 * (lane >> 1) + 128 * h + 64 * (lane & 1);
      if (san)
        tma_load_2d(dst, map, tail_full, x, y);
      else
        tma_load_2d_pair(dst, map, full0 + 8u * stage, x, y);
    }
    const uint32_t st0 = stage;
    if (++stage == kStagesO) {
      stage = 0;
      phase ^= 1u;
    }
    if (!ok || !san) continue;
    // Pages m_san, m_san + 1, ... all take this path, so this is use
    // (m - m_san) / 4 of the stage's tail barriers.
    const uint32_t use = (uint32_t)(m - w.m_san) / kStagesO;
    if (!mbar_wait(tail_full, use & 1u, &s.abort_flag)) ok = false;
    const int keep = (int)(w.L - t0 < kPage ? w.L - t0 : kPage);
    const int64_t lo64 = w.nmin - t0;
    const int lo = lo64 <= 0 ? 0 : (lo64 >= keep ? keep : (int)lo64);
    for (int q = 0; q < kBoxesO; ++q) {
      // A token row is 128 contiguous bytes of the box (the swizzle only
      // permutes its 16-byte chunks), 8 chunks.
      uint4* box = reinterpret_cast<uint4*>(s.ring[st0 * kBoxesO + q]);
      for (int k = lo * 8 + lane; k < keep * 8; k += 32) {
        const uint4 x = box[k];
        box[k] = make_uint4(bf16x2_finite_or_zero(x.x), bf16x2_finite_or_zero(x.y),
                            bf16x2_finite_or_zero(x.z), bf16x2_finite_or_zero(x.w));
      }
      for (int k = keep * 8 + lane; k < kPage * 8; k += 32)
        box[k] = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
    __syncwarp();
    ok = __all_sync(kFull, ok);
    if (ok && lane == 0) arrive_leader(smem_u32(&s.tail_ready[st0]), rank, 2);
  }
  if (!ok && lane == 0) signal_abort(s, p, rank);
}

// --------------------------------------------------- S pair: MMA (rank 0) ----
// One thread issues every S-tile MMA of the pair: S[256 rows, 256 tokens] +=
// Q[:, chunk] x K[tokens, chunk]^T, chunks 0..7 with A = Q_nope from TMEM,
// chunk 8 with A = Q_rope from shared memory.
__device__ __forceinline__ void mma_s(Smem& s, const TcParams& p,
                                      const Work& w, uint32_t tmem,
                                      uint32_t rank) {
  if (!mbar_wait(smem_u32(&s.qready), 0, &s.abort_flag)) {
    signal_abort(s, p, rank);
    return;
  }
  tc_fence_after();
  // Q_nope into TMEM columns [0, 256) of both S-CTAs (row r in lane r,
  // column c holding elements 2c, 2c+1): box k (dims 64k..) in 4 copies of
  // 16 dims; the commit frees the boxes' buffers (qmoved) once the copies
  // have read them, and the MMAs below, issued after the copies by this
  // thread, see the copied values.
#pragma unroll 1
  for (int k = 0; k < 8; ++k) {
    const uint8_t* src =
        k < 4 ? s.pslot[k] : s.ring[(kQRingStage0 + k - 4) * kBoxesPerStage];
    const uint64_t q = sdesc_sw128(smem_u32(src), 16, 1024);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      tmem_cp_128x256b_pair(tmem + 32u * k + 8u * kk, q + 2 * kk);
  }
  mma_commit_pair(smem_u32(&s.qmoved), kMaskS);
  const uint32_t d = tmem + kSCol0;
  const uint64_t qr = sdesc_sw128(smem_u32(s.qrope), 16, 1024);
  uint32_t stage = 0, phase = 0;
  const int ntiles = (w.npages + kTilePages - 1) / kTilePages;
  for (int j = 0; j < ntiles; ++j) {
    // both S-CTAs have read the previous tile's S out of TMEM
    if (!mbar_wait(smem_u32(&s.sempty), (j & 1) ^ 1u, &s.abort_flag)) {
      signal_abort(s, p, rank);
      return;
    }
    tc_fence_after();
    for (int c = 0; c < kBf16BoxesPerPage; ++c) {
      if (!mbar_wait(smem_u32(&s.full[stage]), phase, &s.abort_flag)) {
        signal_abort(s, p, rank);
        return;
      }
      tc_fence_after();
      const uint64_t b =
          sdesc_sw128(smem_u32(s.ring[stage * kBoxesPerStage]), 16, 1024);
      if (c < 8) {
        // A = Q_nope from TMEM: K step ks = 4c + kk at column 8 ks; each K
        // step advances B by 32 B (2 descriptor units).
        mma_ts_pair(d, tmem + 32u * c + 0, b + 0, kIdescS, c > 0 ? 1u : 0u);
        mma_ts_pair(d, tmem + 32u * c + 8, b + 2, kIdescS, 1u);
        mma_ts_pair(d, tmem + 32u * c + 16, b + 4, kIdescS, 1u);
        mma_ts_pair(d, tmem + 32u * c + 24, b + 6, kIdescS, 1u);
      } else {
        // A = Q_rope from shared memory (K-major, 128-B swizzle).
        mma_ss_pair(d, qr + 0, b + 0, kIdescS, 1u);
        mma_ss_pair(d, qr + 2, b + 2, kIdescS, 1u);
        mma_ss_pair(d, qr + 4, b + 4, kIdescS, 1u);
        mma_ss_pair(d, qr + 6, b + 6, kIdescS, 1u);
      }
      mma_commit_pair(smem_u32(&s.empty[stage]), kMaskS);
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    mma_commit_pair(smem_u32(&s.sfull), kMaskS);
  }
}

// ------------------------------------------------------ S-CTA: softmax ----
// Warps 4..11 of each S-CTA: warpgroup g = 0 (warps 4-7) owns pages 0,1 of
// each S tile, g = 1 (warps 8-11) pages 2,3 (S columns [128g, +128), which
// the pair MMA fills from both CTAs' halves of the tile).  Thread = query
// row r (TMEM lane) of this CTA's row group.
__device__ __forceinline__ void softmax(Smem& s, const TcParams& p,
                                        const CUtensorMap* qn_map,
                                        const CUtensorMap* qr_map,
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

  // Q rows by TMA (boxes of 64 values x 128 rows, 128-byte swizzle, rows
  // from this CTA's first), issued at kernel entry (issue_query): the rope
  // part straight into its MMA operand buffer; the nope part's dims 0..255
  // in the P slots, idle until the first S tile, and dims 256..511 in ring
  // stages 4..7, which the producer fills only once they are copied out
  // (qmoved).  Once both S-CTAs' boxes landed, the MMA thread copies Q_nope
  // into TMEM (mma_s).  The landing is finished work seen on qbar, so the
  // signal is relaxed.
  if (warp == 4) {
    if (lane == 0) {
      if (mbar_wait(smem_u32(&s.qbar), 0, &s.abort_flag))
        signal_leader(smem_u32(&s.qready), rank, 0);
      else
        signal_abort(s, p, rank);
    }
    __syncwarp();
  }

  float m_ref = -INFINITY, l = 0.f;
  bool ok = true;
  const uint32_t orank = rank + 2;  // the O-CTA of this row group
  const uint32_t peer_pfull0 = mapa(smem_u32(&s.pfull[0]), orank);
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
    if (lane == 0) signal_leader(smem_u32(&s.sempty), rank, 0);

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

    // P of both pages, packed bf16 pairs, computed before any wait for a
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
        pk[c] = pack_bf16(pa, pb);
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
      if ((warp & 3) == 0 && lane == 0 && ok && !s.abort_flag) {
        // The receiver armed pfull[k] with the byte count itself.
        bulk_copy_to_peer(mapa(smem_u32(stg), orank), smem_u32(stg),
                          kPMsgBytes, peer_pfull0 + 8u * k);
        // Rank 2 issues the pair's P x V MMAs and decides on rescales: it
        // gets rank 1's rescale flags too, counted on its own pfull[k].
        if (rank == 1)
          bulk_copy_to_peer(mapa(smem_u32(stg + kPeerFlagOff), 2),
                            smem_u32(stg + kFlagOff), 16,
                            mapa(smem_u32(&s.pfull[k]), 2));
      }
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
      // no visible token: -inf; a NaN sum (a NaN score seen) stays NaN
      p.LSE_part[part * rows + qrow] =
          lt == 0.f ? -INFINITY : (m_ref + log2f(lt)) * 0.69314718055994531f;
    }
    s.fin[r] = lt == 0.f ? 0.f : 1.f / lt;
    fence_proxy_async_smem();
    named_bar_sync(2, 128);
    if (warp == 4 && lane == 0 && !s.abort_flag)
      bulk_copy_to_peer(mapa(smem_u32(s.fin), orank), smem_u32(s.fin),
                        kRows * 4, mapa(smem_u32(&s.fin_full), orank));
    // Before teardown: every P slot released by the O pair, so no remote
    // arrive can land after this CTA exits.
    for (int m = max(0, w.npages - kNP); m < w.npages && ok; ++m)
      if (!mbar_wait(smem_u32(&s.pempty[m % kNP]), (m / kNP) & 1,
                     &s.abort_flag))
        ok = false;
  }
  if (!__all_sync(kFull, ok) && lane == 0) signal_abort(s, p, rank);
}

// --------------------------------------------------- O pair: MMA (rank 2) ----
// One thread issues every P x V MMA of the pair: for each page m (message
// slot k = m mod 4) it needs the P rows of both O-CTAs (its own pfull, which
// also counts rank 1's rescale flags, and rank 3's through pready), then
// O[:, 256n + (0..255)] += P x V for n = 0, 1.
__device__ __forceinline__ void mma_o(Smem& s, const TcParams& p,
                                      const Work& w, uint32_t tmem,
                                      uint32_t rank) {
  uint32_t stage = 0, phase = 0, ev = 0;
  bool ok = true;
  const uint32_t drain3 = mapa(smem_u32(&s.drain), 3);
  // Each P message lands by a bulk copy whose bytes complete on pfull[k];
  // the receiving CTA arms the barrier (one arrival + the byte count)
  // itself, so the sender needs no cluster-scope arrive: the first use of
  // each slot is armed at set-up, the next one as soon as a message has been
  // received (here for rank 2, by the relay thread for rank 3).
  for (int m = 0; m < w.npages && ok; ++m) {
    const int k = m % kNP;
    const uint32_t par = (m / kNP) & 1;
    if (!mbar_wait(smem_u32(&s.pfull[k]), par, &s.abort_flag) ||
        !mbar_wait(smem_u32(&s.pready[k]), par, &s.abort_flag)) {
      ok = false;
      break;
    }
    if (m + kNP < w.npages)
      mbar_arrive_expect_tx(smem_u32(&s.pfull[k]), kPMsgBytes + 16);
    const uint32_t* fl =
        reinterpret_cast<const uint32_t*>(s.pslot[k] + kFlagOff);
    const uint32_t* pf =
        reinterpret_cast<const uint32_t*>(s.pslot[k] + kPeerFlagOff);
    if (fl[0] | fl[1] | fl[2] | fl[3] | pf[0] | pf[1] | pf[2] | pf[3]) {
      // Rows of either O-CTA raised their running max: let both CTAs'
      // correction warps rescale once every earlier product has landed.
      s.ctl_slot = k;
      s.ctl_final = 0;
      st_cluster_u32(mapa(smem_u32(&s.ctl_slot), 3), (uint32_t)k);
      st_cluster_u32(mapa(smem_u32(&s.ctl_final), 3), 0u);
      mma_commit_pair(smem_u32(&s.drain), kMaskO);
      mbar_arrive(smem_u32(&s.drain));
      mbar_arrive_cluster(drain3);
      if (!mbar_wait(smem_u32(&s.corr_done), ev & 1, &s.abort_flag)) {
        ok = false;
        break;
      }
      ++ev;
    }
    // a page from m_san on arrives sanitised by both producers (tail_ready)
    const bool san = m >= w.m_san;
    if (san ? !mbar_wait(smem_u32(&s.tail_ready[stage]),
                         ((uint32_t)(m - w.m_san) / kStagesO) & 1u, &s.abort_flag)
            : !mbar_wait(smem_u32(&s.full[stage]), phase, &s.abort_flag)) {
      ok = false;
      break;
    }
    tc_fence_after();
    const uint64_t a = sdesc_sw128(smem_u32(s.pslot[k]), 16, 1024);
    for (int n = 0; n < 2; ++n) {
      // B = V: MN-major, next 64 dims one box (8 KB) on, next 8 tokens 1 KB
      // on; each 16-token K step advances 2048 B (128 descriptor units).
      const uint64_t b = sdesc_sw128(
          smem_u32(s.ring[stage * kBoxesO + 2 * n]), kBoxBytes, 1024);
      const uint32_t d = tmem + 256u * n;
      mma_ss_pair(d, a + 0, b + 0, kIdescO, m > 0 ? 1u : 0u);
      mma_ss_pair(d, a + 2, b + 128, kIdescO, 1u);
      mma_ss_pair(d, a + 4, b + 256, kIdescO, 1u);
      mma_ss_pair(d, a + 6, b + 384, kIdescO, 1u);
    }
    mma_commit_pair(smem_u32(&s.empty[stage]), kMaskO);
    if (++stage == kStagesO) {
      stage = 0;
      phase ^= 1u;
    }
    mma_commit_pair(smem_u32(&s.pempty[k]), kMaskS);  // both S-CTAs
  }
  if (!ok) signal_abort(s, p, rank);
  s.ctl_final = 1;
  st_cluster_u32(mapa(smem_u32(&s.ctl_final), 3), 1u);
  mma_commit_pair(smem_u32(&s.drain), kMaskO);
  mbar_arrive(smem_u32(&s.drain));
  mbar_arrive_cluster(drain3);
}

// --------------------------------------------------- O pair: relay (rank 3) ----
// Tells rank 2 when a P message has landed in rank 3 (bulk-copy bytes can
// only complete on a barrier of the receiving CTA), and re-arms the slot.
__device__ __forceinline__ void relay_o(Smem& s, const TcParams& p,
                                        const Work& w, uint32_t rank) {
  const uint32_t pready0 = mapa(smem_u32(&s.pready[0]), 2);
  for (int m = 0; m < w.npages; ++m) {
    const int k = m % kNP;
    if (!mbar_wait(smem_u32(&s.pfull[k]), (m / kNP) & 1, &s.abort_flag)) {
      signal_abort(s, p, rank);
      return;
    }
    if (m + kNP < w.npages)
      mbar_arrive_expect_tx(smem_u32(&s.pfull[k]), kPMsgBytes);
    asm volatile(
        "mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(
            pready0 + 8u * k)
        : "memory");
  }
}

// ------------------------------------------------ O-CTA: epilogue stores ----
// O_part = O / l for this thread's row r (TMEM lane) over value columns
// [256 half, +256), 32 at a time: the warp stages its 32 rows x 32 values
// in 4 KB of the then idle ring (row r at 128 r bytes, 16-byte chunk e at
// position e ^ (r % 8), so neither the writes nor the reads below conflict)
// and reads them back four rows per instruction, lane l taking chunk l % 8
// of row 4i + l / 8: every store instruction writes four full 128-byte
// lines of O_part.
__device__ __forceinline__ void store_o_rows(Smem& s, const TcParams& p,
                                             const CUtensorMap* o_map,
                                             const Work& w, uint32_t tmem,
                                             int warp, int lane, int half) {
  const int quad = warp & 3;
  const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
  const float inv = s.fin[quad * 32 + lane];
  const int64_t rows = (int64_t)p.B * p.q_len * p.H;
  const int64_t part = (int64_t)w.split * (p.V / p.B) + w.shard;
  const int64_t row0 =
      part * rows + (int64_t)w.b * p.q_len * p.H + w.r_base + quad * 32;
  float* const dst0 = p.O_part + row0 * MLA_VALUE_DIM;
  const int nvalid = w.nrows - quad * 32;  // rows of this warp in range
  if (p.o_bf16) {
    // bf16 partial outputs: 64 values (128 bytes) per row of a box, four
    // boxes per warp and half, box k stored by lane k; a partial 32-row
    // block is written by its lanes directly (64 bytes per row and step).
    __nv_bfloat16* const dst_b =
        reinterpret_cast<__nv_bfloat16*>(p.O_part) + row0 * MLA_VALUE_DIM;
    uint8_t* const bufs = s.ring[2 * (warp - 4)];
    const bool by_tma = p.o_tma && nvalid >= 32;
#pragma unroll 1
    for (int k = 0; k < 4; ++k) {
      const int c0 = 256 * half + 64 * k;
      uint32_t va[32], vb[32];
      tmem_ld32(tmem + lane_base + c0, va);
      tmem_ld32(tmem + lane_base + c0 + 32, vb);
      tmem_wait_ld();
      uint4 q[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const uint32_t* v = e < 4 ? va + 8 * e : vb + 8 * (e - 4);
        q[e] = make_uint4(pack_bf16(__uint_as_float(v[0]) * inv, __uint_as_float(v[1]) * inv),
                          pack_bf16(__uint_as_float(v[2]) * inv, __uint_as_float(v[3]) * inv),
                          pack_bf16(__uint_as_float(v[4]) * inv, __uint_as_float(v[5]) * inv),
                          pack_bf16(__uint_as_float(v[6]) * inv, __uint_as_float(v[7]) * inv));
      }
      if (by_tma) {
        uint8_t* const box = bufs + k * 4096;
#pragma unroll
        for (int e = 0; e < 8; ++e)
          *reinterpret_cast<uint4*>(box + box_chunk_offset(lane, e)) = q[e];
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == k) {
          tma_store_3d(o_map, smem_u32(box), c0, (int32_t)row0, 0);
          bulk_commit_group();
        }
      } else if (lane < nvalid) {
        uint4* d = reinterpret_cast<uint4*>(dst_b + (int64_t)lane * MLA_VALUE_DIM + c0);
#pragma unroll
        for (int e = 0; e < 8; ++e) d[e] = q[e];
      }
    }
    if (by_tma) {
      if (lane < 4) bulk_wait_read_all();
      __syncwarp();
    }
    return;
  }
  if (p.o_tma && nvalid >= 32) {
    // Whole 32-row blocks leave by TMA store, 32 values (128 bytes) per
    // box: four boxes of this warp's 16 KB of the idle ring in turn, box i
    // stored by lane i (a thread's TMA operations are processed one after
    // another), which waits for the box's previous store to have read it
    // before the warp refills it.
    uint8_t* const bufs = s.ring[2 * (warp - 4)];
#pragma unroll 1
    for (int k = 0; k < 8; ++k) {
      const int c0 = 256 * half + 32 * k;
      const int bi = k & 3;
      uint8_t* const box = bufs + bi * 4096;
      uint32_t v[32];
      tmem_ld32(tmem + lane_base + c0, v);
      if (k >= 4 && lane == bi) bulk_wait_read_all();
      __syncwarp();
      tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 8; ++e)
        *reinterpret_cast<float4*>(box + box_chunk_offset(lane, e)) =
            make_float4(__uint_as_float(v[4 * e]) * inv,
                        __uint_as_float(v[4 * e + 1]) * inv,
                        __uint_as_float(v[4 * e + 2]) * inv,
                        __uint_as_float(v[4 * e + 3]) * inv);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == bi) {
        tma_store_2d(o_map, smem_u32(box), c0, (int32_t)row0);
        bulk_commit_group();
      }
    }
    if (lane < 4) bulk_wait_read_all();
    __syncwarp();
    return;
  }
  uint8_t* const buf = s.ring[2 * (warp - 4)];  // this warp's 16 KB as above
#pragma unroll 1
  for (int k = 0; k < 8; ++k) {
    const int c0 = 256 * half + 32 * k;
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

// Warps 8..11 of each O-CTA: the second half of the value columns, once
// warps 4..7 have seen the last drain and 1/l.
__device__ __forceinline__ void store_o_upper(Smem& s, const TcParams& p,
                                              const CUtensorMap* o_map,
                                              const Work& w, uint32_t tmem,
                                              int warp, int lane) {
  if (!mbar_wait(smem_u32(&s.epi_go), 0, &s.abort_flag)) return;
  tc_fence_after();
  store_o_rows(s, p, o_map, w, tmem, warp, lane, 1);
}

// ---------------------------------------- O-CTA: correction + epilogue ----
// Warps 4..7 of each O-CTA, thread = row r of this CTA's row group.  A
// drain event (every earlier pair MMA complete) either asks for a rescale of
// the rows whose running max rose (factors in the P slot that triggered it)
// or, the last one, for the epilogue: O_part = O / l over the first half of
// the value columns (warps 8..11 take the second, after epi_go).
__device__ __forceinline__ void correct_and_store(Smem& s, const TcParams& p,
                                                  const CUtensorMap* o_map,
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
    if (lane == 0) signal_leader(smem_u32(&s.corr_done), rank, 2);
  }
  if (ok && !mbar_wait(smem_u32(&s.fin_full), 0, &s.abort_flag)) ok = false;
  if (!__all_sync(kFull, ok)) {
    if (lane == 0) signal_abort(s, p, rank);
    return;
  }
  tc_fence_after();
  __syncwarp();
  if (lane == 0) mbar_arrive(smem_u32(&s.epi_go));
  store_o_rows(s, p, o_map, w, tmem, warp, lane, 0);
}

// ------------------------------------------------------------- kernel ----
__global__ void __cluster_dims__(kCtas, 1, 1) __launch_bounds__(kThreads, 1)
    mla_partial_tc_kernel(const __grid_constant__ CUtensorMap kv_map,
                          const __grid_constant__ CUtensorMap qn_map,
                          const __grid_constant__ CUtensorMap qr_map,
                          const __grid_constant__ CUtensorMap o_map,
                          const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();
  const int unit = cluster_unit(p);
  if (unit < 0) {  // every CTA of the cluster read the same entry
    if (rank == 0 && threadIdx.x == 0 && p.status)
      atomicOr(p.status, MLA_STATUS_BAD_WORK);
    return;
  }
  // The query rows need only the unit id: the S-CTAs put them in flight
  // before anything else, so their load overlaps the rest of the set-up.
  if (rank < 2 && warp == 0) issue_query(s, &qn_map, &qr_map, p, unit, rank, lane);
  const Work w = unit_work(p, unit, rank);
  // The S producer's first page-table entries, also in flight during the
  // set-up (checked only when the producer starts).
  int32_t pb_cur = 0, pb_nxt = 0;
  if (rank < 2 && warp == 0 && w.npages > 0) {
    pb_cur = page_entry(p, w, lane);
    pb_nxt = page_entry(p, w, 32 + lane);
  }

  // The stream's next kernel (the LSE combine) may be scheduled from now
  // on; it waits for this grid's completion before it reads a part.
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) {
    s.abort_flag = 0;
    s.ctl_slot = 0;
    s.ctl_final = 0;
    s.ctl_last = 0;
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_u32(&s.full[i]), 1);
      mbar_init(smem_u32(&s.empty[i]), 1);
    }
    mbar_init(smem_u32(&s.sfull), 1);
    mbar_init(smem_u32(&s.sempty), 16);  // 8 softmax warps x 2 S-CTAs
    for (int i = 0; i < kNP; ++i) {
      mbar_init(smem_u32(&s.pfull[i]), 1);
      mbar_init(smem_u32(&s.pready[i]), 1);
      mbar_init(smem_u32(&s.pempty[i]), 1);
    }
    mbar_init(smem_u32(&s.drain), 2);      // pair commit + rank 2's arrive
    mbar_init(smem_u32(&s.corr_done), 8);  // 4 correction warps x 2 O-CTAs
    for (int i = 0; i < kStagesO; ++i) {
      mbar_init(smem_u32(&s.tail_full[i]), 1);
      mbar_init(smem_u32(&s.tail_ready[i]), 2);
    }
    mbar_init(smem_u32(&s.fin_full), 1);
    mbar_init(smem_u32(&s.epi_go), 4);
    mbar_init(smem_u32(&s.qready), 2);  // one thread per S-CTA
    if (rank >= 2 && w.npages > 0) {
      mbar_arrive_expect_tx(smem_u32(&s.fin_full), kRows * 4);
      // rank 2 also receives rank 1's 16 flag bytes per message
      for (int k = 0; k < kNP && k < w.npages; ++k)
        mbar_arrive_expect_tx(smem_u32(&s.pfull[k]),
                              kPMsgBytes + (rank == 2 ? 16 : 0));
    }
    fence_mbar_init();
    prefetch_tmap(&kv_map);
    if (rank >= 2 && p.o_tma) prefetch_tmap(&o_map);
  }
  if (rank == 0 && threadIdx.x == 32 && p.seq_lens[w.v] > p.r2t_stride &&
      p.status)
    atomicOr(p.status, MLA_STATUS_BAD_LENGTH);
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(&s.tmem_base), 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;
  cluster_sync();  // every CTA's barriers exist before any remote operation

  // Fused combine ([K3-MLA], dcp_lse_combine, in the same launch): rank 0
  // counts this cluster's arrival for its (request, row unit) once all four
  // CTAs have written their part; the cluster whose arrival completes the
  // count (shards x splits) resets it and merges the unit's rows, every part
  // being in memory by then.  No cluster waits for another.
  auto fused_arrival = [&]() {
    if (rank == 0 && threadIdx.x == 0) {
      const int unit_u = w.r_base / MLA_ROWS_PER_UNIT;
      int* c = p.counters + (int64_t)w.b * p.U + unit_u;
      const int total = p.num_splits * (p.V / p.B);
      const bool last = atom_add_acq_rel_gpu(c, 1) == total - 1;
      if (last) *c = 0;
      for (uint32_t k = 0; k < kCtas; ++k)
        st_cluster_u32(mapa(smem_u32(&s.ctl_last), k), last ? 1u : 0u);
    }
  };
  auto fused_combine = [&]() {
    if (!*reinterpret_cast<volatile int*>(&s.ctl_last)) return;
    __threadfence();
    const int R = p.q_len * p.H;
    const int r0 = w.r_base / MLA_ROWS_PER_UNIT * MLA_ROWS_PER_UNIT;
    const int n = min(MLA_ROWS_PER_UNIT, R - r0);
    const int64_t rows = (int64_t)p.B * R;
    const int P = p.num_splits * (p.V / p.B);
    constexpr int kWarps = kThreads / 32;
    for (int r = (int)rank * kWarps + warp; r < n; r += kCtas * kWarps)
      combine_row<true>(p.O_part, p.LSE_part, P, rows,
                        (int64_t)w.b * R + r0 + r, p.out, p.lse_out, lane);
  };

  // Teardown, repeated at the end of every role: roles never rejoin, so no
  // warp ever asks setmaxnreg for registers back (a warpgroup that did could
  // take them before the softmax warpgroups got theirs and stall both).
  // The pair's TMEM is released only after all four CTAs are done with it.
  auto teardown = [&]() {
    if (p.counters) __threadfence();  // this CTA's part before the arrival
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_sync();
    if (warp == 1) tmem_dealloc_pair(tmem, 512);
    if (p.counters) fused_arrival();
    cluster_sync();
    if (p.counters) fused_combine();
  };

  if (w.npages > 0 && rank < 2) {
    if (warp < 4) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsControl));
      if (warp == 0) {
        producer_s(s, &kv_map, p, w, rank, lane, pb_cur, pb_nxt);
      } else if (warp == 1 && rank == 0) {
        if (lane == 0) mma_s(s, p, w, tmem, rank);
        __syncwarp();
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
      if (lane == 0) {
        if (rank == 2)
          mma_o(s, p, w, tmem, rank);
        else
          relay_o(s, p, w, rank);
      }
      __syncwarp();
    } else if (warp >= 4 && warp < 8) {
      correct_and_store(s, p, &o_map, w, tmem, rank, warp, lane);
    } else if (warp >= 8) {
      store_o_upper(s, p, &o_map, w, tmem, warp, lane);
    }
  } else if (rank < 2 && threadIdx.x == 0) {
    // No tokens for this split: the query boxes issued at entry land before
    // the CTA leaves.
    mbar_wait(smem_u32(&s.qbar), 0, &s.abort_flag);
  }
  if (w.npages == 0 && warp >= 4 && warp < 8) {
    // No tokens for this split: O = 0 (O-CTAs), LSE = -inf (S-CTAs).
    const int r = (warp & 3) * 32 + lane;
    if (r < w.nrows) {
      const int64_t rows = (int64_t)p.B * p.q_len * p.H;
      const int64_t part = (int64_t)w.split * (p.V / p.B) + w.shard;
      const int64_t orow =
          part * rows + (int64_t)w.b * p.q_len * p.H + w.r_base + r;
      if (rank < 2) {
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

int launch_tc(const DecodeArgs& a) {
  if (a.kv_dtype == MLA_KV_FP8_E4M3) return launch_tc_fp8(a);
  TcParams p;
  p.q_nope = static_cast<const uint4*>(a.q_nope);
  p.q_rope = static_cast<const uint4*>(a.q_rope);
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
  p.U = (a.q_len * a.H + MLA_ROWS_PER_UNIT - 1) / MLA_ROWS_PER_UNIT;
  p.scale_log2 = a.sm_scale * 1.4426950408889634f;
  p.O_part = a.O_part;
  p.LSE_part = a.LSE_part;
  p.status = a.status;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.lse_out = a.lse_out;
  p.counters = a.counters;
  const int64_t units = (int64_t)p.V * p.num_splits * p.U;
  if (units * kCtas > 0x7fffffff)
    return fail(MLA_ERR_INVALID_ARG, "grid too large");
  CUtensorMap map, qn_map, qr_map;
  int rc = make_kv_tensor_map(&map, a.kv, a.kv_dtype, a.num_slots);
  if (rc != MLA_OK) return rc;
  rc = make_query_maps(&qn_map, &qr_map, a, &p.q_box_rows);
  if (rc != MLA_OK) return rc;
  // The partial outputs leave by TMA store when their rows fit the tensor
  // map's 32-bit coordinates; the fused combine, which reads other
  // clusters' parts in the same launch, keeps the plain stores its fences
  // order.
  CUtensorMap o_map;
  std::memset(&o_map, 0, sizeof(o_map));
  const int64_t o_rows =
      (int64_t)p.num_splits * a.num_shards * a.B * a.q_len * a.H;
  p.o_bf16 = a.o_bf16;
  if (p.o_bf16) {
    const uint64_t dims[3] = {(uint64_t)MLA_VALUE_DIM, (uint64_t)o_rows, 1};
    const uint64_t strides[2] = {(uint64_t)MLA_VALUE_DIM * 2,
                                 (uint64_t)o_rows * MLA_VALUE_DIM * 2};
    const uint32_t box[3] = {64, 32, 1};
    p.o_tma = !p.counters && o_rows < 0x7fffffff &&
              make_tensor_map_bf16_3d(&o_map, p.O_part, dims, strides, box) ==
                  MLA_OK;
  } else {
    p.o_tma = !p.counters && o_rows < 0x7fffffff &&
              make_o_part_map(&o_map, p.O_part, o_rows) == MLA_OK;
  }
  cudaError_t e = cudaFuncSetAttribute(
      mla_partial_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
      kSmemBytes);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(tc)");
  mla_partial_tc_kernel<<<(unsigned)(units * kCtas), kThreads, kSmemBytes,
                          a.stream>>>(map, qn_map, qr_map, o_map, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch mla_partial_tc_kernel");
  return MLA_OK;
}

}  // namespace mla

extern "C" int mla_cluster_slots(void) {
  cudaError_t e = cudaFuncSetAttribute(
      mla::mla_partial_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
      mla::kSmemBytes);
  if (e != cudaSuccess) return mla::cuda_fail(e, "cudaFuncSetAttribute(tc)");
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = mla::kCtas;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(mla::kCtas * 1024, 1, 1);
  cfg.blockDim = dim3(mla::kThreads, 1, 1);
  cfg.dynamicSmemBytes = mla::kSmemBytes;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, mla::mla_partial_tc_kernel,
                                     &cfg);
  if (e != cudaSuccess)
    return mla::cuda_fail(e, "cudaOccupancyMaxActiveClusters");
  return clusters;
}
