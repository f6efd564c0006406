// mla_tc.cu -- tensor-core (tcgen05 / TMEM / TMA) partial MLA decode.
//
// What it computes is stated in include/mla_decode.h (mla_decode_partial):
// weight-absorbed MLA decode over the paged latent KV ([VRAM-KV],
// [VRAM-POOL]), partial (O, LSE) per KV split and context shard ([K3-MLA],
// [K3-SPLIT]), causal among the q_len draft tokens ([K3-INTRO]).
//
// Design (GB300, one CTA per SM):
//   All H*q_len query rows of a request share one latent KV row per token, so
//   S = Q K^T (576-d) and O = P V (512-d, V = the c_kv columns of the same
//   row) are dense contractions with M = query rows.  A 128-row M tile needs
//   its fp32 O accumulator (128 x 512) to fill all 512 TMEM columns of an SM,
//   so the work of one 128-row group is split over a CTA pair (a cluster of
//   two):
//     rank 0, the "S-CTA": Q (bf16 pairs) in TMEM columns [0, 288), three S
//       buffers of 64 columns; streams K tiles (one 64-token page = 9 TMA
//       boxes of 64 tokens x 64 dims, 128-B swizzle) through a ring, issues
//       S = Q K^T with A from TMEM, runs the online softmax in registers (one
//       thread per row, base-2, lazy rescaling), and ships P (bf16, K-major
//       128-B swizzled) plus the per-row rescale factors to the peer with a
//       bulk shared-memory copy.
//     rank 1, the "O-CTA": O (128 x 512 fp32) in all of TMEM; streams the
//       8 c_kv boxes of each page, issues O += P V (A = P from shared memory,
//       B = V MN-major from the TMA boxes, N = 256 per instruction), rescales
//       O rows when the S-CTA raised its running max, and writes the
//       normalised O_part rows.
//   The tensor work splits 576 : 512 between the two SMs; no QK^T is
//   repeated.  Every wait is bounded (ptx_sm103.cuh); a timeout sets
//   MLA_STATUS_WAIT_TIMEOUT and the CTA pair finishes early.
#include <cuda_bf16.h>

#include "mla_tma.cuh"
#include "ptx_sm103.cuh"

namespace mla {
namespace {

using namespace ptx;

constexpr int kThreads = 192;        // 6 warps
constexpr int kRingS = 22;           // 8-KB box slots, S-CTA
constexpr int kRingO = 20;           // O-CTA: a multiple of 4 (4-box groups)
constexpr int kRing = kRingS > kRingO ? kRingS : kRingO;
constexpr int kNS = 3;               // S buffers in TMEM
constexpr int kNP = 2;               // P message slots
constexpr int kRows = MLA_ROWS_PER_PAIR;  // 128
constexpr int kTile = MLA_PAGE_SIZE;      // 64 tokens per tile
constexpr int kPBytes = kRows * kTile * 2;          // 16384
constexpr int kAlphaOff = kPBytes;                  // float alpha[128]
constexpr int kFlagOff = kPBytes + kRows * 4;       // uint32 flags[4]
constexpr int kPMsgBytes = kFlagOff + 16;           // 16912 = 1057 x 16
constexpr int kPSlotStride = 17408;                 // 17 KB, 1024-aligned
constexpr uint32_t kQCols = MLA_ROW_DIM / 2;        // 288
constexpr uint32_t kSCol0 = kQCols;                 // S buffers: 288 + 64 i
constexpr float kTau = 8.f;          // lazy-rescale threshold (log2 units)
constexpr uint32_t kFull = 0xffffffffu;

constexpr uint32_t kIdescS = idesc_bf16_f32(128, 64, false, false);
constexpr uint32_t kIdescO = idesc_bf16_f32(128, 256, false, true);

struct __align__(1024) Smem {
  uint8_t ring[kRing][kBoxBytes];
  uint8_t pslot[kNP][kPSlotStride];
  float fin[kRows];
  uint64_t full[kRing];
  uint64_t empty[kRing];
  uint64_t sfull[kNS];
  uint64_t sempty[kNS];
  uint64_t pfull[kNP];
  uint64_t pempty[kNP];
  uint64_t drain;
  uint64_t corr_done;
  uint64_t tail_ready;
  uint64_t fin_full;
  uint64_t qready;
  uint32_t tmem_base;
  int abort_flag;
  int ctl_slot;
  int ctl_final;
};
constexpr int kSmemBytes = (int)sizeof(Smem) + 1024;
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
static_assert(kPMsgBytes % 16 == 0, "bulk copy size");

struct TcParams {
  const uint4* q_nope;     // bf16 [B, q_len, H, 512] as 16-B chunks
  const uint4* q_rope;     // bf16 [B, q_len, H, 64]
  int64_t num_slots;
  const int32_t* r2t;
  int64_t r2t_stride;
  const int32_t* seq_lens;
  const int32_t* kv_limit;
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

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Record a failed wait: device status, this CTA's and the peer's abort flag.
__device__ __noinline__ void signal_abort(Smem& s, const TcParams& p,
                                          uint32_t rank) {
  if (p.status) atomicOr(p.status, MLA_STATUS_WAIT_TIMEOUT);
  s.abort_flag = 1;
  st_cluster_u32(mapa(smem_u32(&s.abort_flag), rank ^ 1u), 1u);
}

// Per-pair work description, identical on both CTAs of the pair.
struct Work {
  int v, b, shard, split, r_base, nrows, ntiles;
  int64_t L, p0;
};

__device__ __forceinline__ Work pair_work(const TcParams& p) {
  Work w;
  int pair = blockIdx.x >> 1;
  const int g = pair % p.G;
  pair /= p.G;
  w.split = pair % p.num_splits;
  w.v = pair / p.num_splits;
  w.b = w.v % p.B;
  w.shard = w.v / p.B;
  const int R = p.q_len * p.H;
  w.r_base = g * kRows;
  w.nrows = min(kRows, R - w.r_base);
  int64_t L = p.seq_lens[w.v];
  if (L > p.r2t_stride) L = p.r2t_stride;
  if (L < 0) L = 0;
  w.L = L;
  const int64_t P = (L + kTile - 1) / kTile;
  w.p0 = (int64_t)w.split * P / p.num_splits;
  const int64_t p1 = (int64_t)(w.split + 1) * P / p.num_splits;
  w.ntiles = (int)(p1 - w.p0);
  return w;
}

// ------------------------------------------------------------- producer ----
// One warp streams `kBoxes` boxes per page tile into the ring.  The page
// table is read 32 tiles ahead (one entry per lane) so the TMA issue never
// waits on a dependent global load.
template <int kBoxes, int kRingN>
__device__ void producer(Smem& s, const CUtensorMap* map, const TcParams& p,
                         const Work& w, uint32_t rank, int lane,
                         bool zero_tail) {
  uint32_t slot = 0, phase = 0;
  auto page_base = [&](int j) -> int32_t {
    if (j >= w.ntiles) return 0;
    const int32_t base =
        p.r2t[(int64_t)w.v * p.r2t_stride + (w.p0 + j) * kTile];
    if (base < 0 || (base & (kTile - 1)) || (int64_t)base + kTile > p.num_slots)
      return -1;
    return base;
  };
  int32_t cur = 0, nxt = page_base(lane);
  bool ok = true;
  for (int j = 0; j < w.ntiles; ++j) {
    if ((j & 31) == 0) {
      cur = nxt;
      nxt = page_base(j + 32 + lane);
    }
    const int32_t base = __shfl_sync(kFull, cur, j & 31);
    // A page outside the pool reads as zeros (TMA fills out-of-range rows).
    const int32_t y = base < 0 ? (int32_t)p.num_slots : base;
    if (base < 0 && lane == 0 && p.status) atomicOr(p.status, MLA_STATUS_BAD_SLOT);
    const uint32_t slot0 = slot, phase0 = phase;
    if (lane == 0 && ok) {
      for (int c = 0; c < kBoxes; ++c) {
        if (!mbar_wait(smem_u32(&s.empty[slot]), phase ^ 1u, &s.abort_flag)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(smem_u32(&s.full[slot]), kBoxBytes);
        tma_load_2d(smem_u32(s.ring[slot]), map, smem_u32(&s.full[slot]),
                    c * 64, y);
        if (++slot == (uint32_t)kRingN) {
          slot = 0;
          phase ^= 1u;
        }
      }
    }
    ok = __shfl_sync(kFull, ok, 0);
    slot = __shfl_sync(kFull, slot, 0);
    phase = __shfl_sync(kFull, phase, 0);
    if (!ok) {
      if (lane == 0) signal_abort(s, p, rank);
      break;
    }
    // The request's last page may be partly filled: rows past its length
    // can hold anything (even NaN), and 0 * NaN would poison O = P V, so
    // they are zeroed in every c_kv box before the MMA may read them.
    const int64_t t0 = (w.p0 + j) * kTile;
    if (zero_tail && t0 + kTile > w.L) {
      const int keep = (int)(w.L - t0);
      uint32_t sl = slot0, ph = phase0;
      for (int c = 0; c < kBoxes; ++c) {
        if (!mbar_wait(smem_u32(&s.full[sl]), ph, &s.abort_flag)) ok = false;
        uint4* box = reinterpret_cast<uint4*>(s.ring[sl]);
        for (int k = keep * 8 + lane; k < kTile * 8; k += 32)
          box[k] = make_uint4(0, 0, 0, 0);
        if (++sl == (uint32_t)kRingN) {
          sl = 0;
          ph ^= 1u;
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (!__all_sync(kFull, ok)) {
        if (lane == 0) signal_abort(s, p, rank);
        break;
      }
      if (lane == 0) mbar_arrive(smem_u32(&s.tail_ready));
    }
  }
}

// ---------------------------------------------------------- S-CTA: MMA ----
__device__ void mma_s(Smem& s, const TcParams& p, const Work& w, uint32_t tmem,
                      uint32_t rank) {
  if (!mbar_wait(smem_u32(&s.qready), 0, &s.abort_flag)) {
    signal_abort(s, p, rank);
    return;
  }
  tc_fence_after();
  uint32_t slot = 0, phase = 0;
  for (int j = 0; j < w.ntiles; ++j) {
    const int sb = j % kNS;
    if (!mbar_wait(smem_u32(&s.sempty[sb]), ((j / kNS) & 1) ^ 1u, &s.abort_flag)) {
      signal_abort(s, p, rank);
      return;
    }
    tc_fence_after();
    const uint32_t d = tmem + kSCol0 + 64u * sb;
    for (int c = 0; c < kBf16BoxesPerPage; ++c) {
      if (!mbar_wait(smem_u32(&s.full[slot]), phase, &s.abort_flag)) {
        signal_abort(s, p, rank);
        return;
      }
      tc_fence_after();
      const uint32_t b0 = smem_u32(s.ring[slot]);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const int ks = c * 4 + kk;  // 16-element K step
        mma_ts(d, tmem + 8u * ks, sdesc_sw128(b0 + 32u * kk, 16, 1024), kIdescS,
               ks > 0);
      }
      mma_commit(smem_u32(&s.empty[slot]));
      if (++slot == (uint32_t)kRingS) {
        slot = 0;
        phase ^= 1u;
      }
    }
    mma_commit(smem_u32(&s.sfull[sb]));
  }
}

// ------------------------------------------------------ S-CTA: softmax ----
__device__ void softmax(Smem& s, const TcParams& p, const Work& w,
                        uint32_t tmem, uint32_t rank, int warp, int lane) {
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

  // Q row -> TMEM columns [0, 288): 32-bit column c holds elements 2c, 2c+1.
#pragma unroll 1
  for (int c = 0; c < 9; ++c) {
    uint32_t v[32];
    const uint4* src = c < 8 ? p.q_nope + qrow * 64 + c * 8 : p.q_rope + qrow * 8;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint4 x = row_ok ? src[k] : make_uint4(0, 0, 0, 0);
      v[4 * k] = x.x;
      v[4 * k + 1] = x.y;
      v[4 * k + 2] = x.z;
      v[4 * k + 3] = x.w;
    }
    tmem_st32(tmem + lane_base + 32u * c, v);
  }
  tmem_wait_st();
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(smem_u32(&s.qready));

  float m_ref = -INFINITY, l = 0.f;
  bool ok = true;
  const uint32_t peer_pfull0 = mapa(smem_u32(&s.pfull[0]), 1);
  for (int j = 0; j < w.ntiles; ++j) {
    const int sb = j % kNS;
    const int k = j % kNP;
    uint32_t sa[32], sb2[32];
    if (ok && !mbar_wait(smem_u32(&s.sfull[sb]), (j / kNS) & 1, &s.abort_flag))
      ok = false;
    tc_fence_after();
    if (__all_sync(kFull, ok)) {
      tmem_ld32(tmem + lane_base + kSCol0 + 64u * sb, sa);
      tmem_ld32(tmem + lane_base + kSCol0 + 64u * sb + 32, sb2);
      tmem_wait_ld();
    } else {
      ok = false;
#pragma unroll
      for (int c = 0; c < 32; ++c) sa[c] = sb2[c] = 0u;
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&s.sempty[sb]));

    const int64_t t0 = (w.p0 + j) * kTile;
    const int64_t nv = n - t0;
    const int nvis = nv <= 0 ? 0 : (nv >= kTile ? kTile : (int)nv);
    float x[64];
    float mt = -INFINITY;
#pragma unroll
    for (int c = 0; c < 64; ++c) {
      x[c] = __uint_as_float(c < 32 ? sa[c] : sb2[c - 32]) * p.scale_log2;
      if (c < nvis) mt = fmaxf(mt, x[c]);
    }
    float alpha = 1.f;
    if (nvis > 0) {
      if (l == 0.f) {
        m_ref = mt;  // first visible token of this row: O is still zero
      } else if (mt > m_ref + kTau) {
        alpha = ex2(m_ref - mt);
        l *= alpha;
        m_ref = mt;
      }
    }

    // Wait until the peer has consumed the previous message in slot k.
    if (ok && !mbar_wait(smem_u32(&s.pempty[k]), ((j / kNP) & 1) ^ 1u,
                         &s.abort_flag))
      ok = false;
    uint8_t* stg = s.pslot[k];
    float psum = 0.f;
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) {
      uint32_t wv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int c0 = cc * 8 + 2 * e;
        const float pa = c0 < nvis ? ex2(x[c0] - m_ref) : 0.f;
        const float pb = c0 + 1 < nvis ? ex2(x[c0 + 1] - m_ref) : 0.f;
        psum += pa + pb;
        wv[e] = pack_bf16(pa, pb);
      }
      // K-major, 128-B swizzle: 8-row groups 1024 B apart, 16-B chunk cc of
      // row r at position cc ^ (r % 8) within its 128-B row.
      *reinterpret_cast<uint4*>(stg + (r >> 3) * 1024 + box_chunk_offset(r & 7, cc)) =
          make_uint4(wv[0], wv[1], wv[2], wv[3]);
    }
    l += psum;
    reinterpret_cast<float*>(stg + kAlphaOff)[r] = alpha;
    const bool any = __any_sync(kFull, alpha != 1.f);
    if (lane == 0) reinterpret_cast<uint32_t*>(stg + kFlagOff)[quad] = any ? 1u : 0u;
    fence_proxy_async_smem();
    named_bar_sync(1, 128);
    if (warp == 2 && lane == 0) {
      if (s.abort_flag) {
        ok = false;
      } else {
        const uint32_t rfull = peer_pfull0 + 8u * k;
        mbar_arrive_expect_tx_cluster(rfull, kPMsgBytes);
        bulk_copy_to_peer(mapa(smem_u32(stg), 1), smem_u32(stg), kPMsgBytes, rfull);
      }
    }
  }

  // Final statistics: LSE to global, 1/l to the peer's epilogue.
  if (row_ok) {
    const int64_t rows = (int64_t)p.B * p.q_len * p.H;
    const int64_t part = (int64_t)w.split * (p.V / p.B) + w.shard;
    p.LSE_part[part * rows + qrow] =
        l > 0.f ? (m_ref + log2f(l)) * 0.69314718055994531f : -INFINITY;
  }
  s.fin[r] = l > 0.f ? 1.f / l : 0.f;
  fence_proxy_async_smem();
  named_bar_sync(1, 128);
  if (warp == 2 && lane == 0 && !s.abort_flag) {
    const uint32_t rfin = mapa(smem_u32(&s.fin_full), 1);
    mbar_arrive_expect_tx_cluster(rfin, kRows * 4);
    bulk_copy_to_peer(mapa(smem_u32(s.fin), 1), smem_u32(s.fin), kRows * 4, rfin);
  }
  // Before teardown: every P slot released by the peer, so no remote arrive
  // can land after this CTA exits.
  for (int j = max(0, w.ntiles - kNP); j < w.ntiles && ok; ++j)
    if (!mbar_wait(smem_u32(&s.pempty[j % kNP]), (j / kNP) & 1, &s.abort_flag))
      ok = false;
  if (!__all_sync(kFull, ok) && lane == 0) signal_abort(s, p, rank);
}

// ---------------------------------------------------------- O-CTA: MMA ----
__device__ void mma_o(Smem& s, const TcParams& p, const Work& w, uint32_t tmem,
                      uint32_t rank) {
  uint32_t slot = 0, phase = 0, ev = 0;
  const bool has_tail = (w.p0 + w.ntiles) * kTile > w.L;
  bool ok = true;
  for (int j = 0; j < w.ntiles && ok; ++j) {
    const int k = j % kNP;
    if (!mbar_wait(smem_u32(&s.pfull[k]), (j / kNP) & 1, &s.abort_flag)) {
      ok = false;
      break;
    }
    const uint32_t* fl = reinterpret_cast<const uint32_t*>(s.pslot[k] + kFlagOff);
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
    if (has_tail && j == w.ntiles - 1 &&
        !mbar_wait(smem_u32(&s.tail_ready), 0, &s.abort_flag)) {
      ok = false;
      break;
    }
    const uint32_t pa = smem_u32(s.pslot[k]);
    uint32_t used[8];
    for (int h = 0; h < 2 && ok; ++h) {
      for (int c = 0; c < 4; ++c) {
        if (!mbar_wait(smem_u32(&s.full[slot]), phase, &s.abort_flag)) {
          ok = false;
          break;
        }
        used[4 * h + c] = slot;
        if (++slot == (uint32_t)kRingO) {
          slot = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      tc_fence_after();
      const uint32_t vb = smem_u32(s.ring[used[4 * h]]);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {  // 16 tokens per step
        // A = P: K-major, 8-row groups 1024 B apart.  B = V: MN-major, next
        // 64 dims one box (8 KB) on, next 8 tokens 1024 B on.
        mma_ss(tmem + 256u * h, sdesc_sw128(pa + 32u * kk, 16, 1024),
               sdesc_sw128(vb + 2048u * kk, kBoxBytes, 1024), kIdescO,
               (j > 0 || kk > 0) ? 1u : 0u);
      }
    }
    if (!ok) break;
    for (int c = 0; c < 8; ++c) mma_commit(smem_u32(&s.empty[used[c]]));
    mma_commit_multicast(smem_u32(&s.pempty[k]), (uint16_t)1u);  // S-CTA
  }
  if (!ok) signal_abort(s, p, rank);
  s.ctl_final = 1;
  mma_commit(smem_u32(&s.drain));
  mbar_arrive(smem_u32(&s.drain));
}

// ---------------------------------------- O-CTA: correction + epilogue ----
__device__ void correct_and_store(Smem& s, const TcParams& p, const Work& w,
                                  uint32_t tmem, uint32_t rank, int warp,
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
        for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * a);
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
    mla_partial_tc_kernel(const __grid_constant__ CUtensorMap kv_map,
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
    for (int i = 0; i < kRing; ++i) {
      mbar_init(smem_u32(&s.full[i]), 1);
      mbar_init(smem_u32(&s.empty[i]), 1);
    }
    for (int i = 0; i < kNS; ++i) {
      mbar_init(smem_u32(&s.sfull[i]), 1);
      mbar_init(smem_u32(&s.sempty[i]), 4);
    }
    for (int i = 0; i < kNP; ++i) {
      mbar_init(smem_u32(&s.pfull[i]), 1);
      mbar_init(smem_u32(&s.pempty[i]), 1);
    }
    mbar_init(smem_u32(&s.drain), 2);
    mbar_init(smem_u32(&s.corr_done), 4);
    mbar_init(smem_u32(&s.tail_ready), 1);
    mbar_init(smem_u32(&s.fin_full), 1);
    mbar_init(smem_u32(&s.qready), 4);
    fence_mbar_init();
    prefetch_tmap(&kv_map);
  }
  if (rank == 0 && threadIdx.x == 32 && w.L > p.r2t_stride && p.status)
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

  if (w.ntiles > 0) {
    if (rank == 0) {
      if (warp == 0)
        producer<kBf16BoxesPerPage, kRingS>(s, &kv_map, p, w, rank, lane, false);
      else if (warp == 1) {
        if (lane == 0) mma_s(s, p, w, tmem, rank);
        __syncwarp();
      } else
        softmax(s, p, w, tmem, rank, warp, lane);
    } else {
      if (warp == 0)
        producer<8, kRingO>(s, &kv_map, p, w, rank, lane, true);
      else if (warp == 1) {
        if (lane == 0) mma_o(s, p, w, tmem, rank);
        __syncwarp();
      } else
        correct_and_store(s, p, w, tmem, rank, warp, lane);
    }
  } else if (warp >= 2) {
    // No tokens for this split: O = 0, LSE = -inf.
    const int r = (warp & 3) * 32 + lane;
    if (r < w.nrows) {
      const int64_t rows = (int64_t)p.B * p.q_len * p.H;
      const int64_t part = (int64_t)w.split * (p.V / p.B) + w.shard;
      const int64_t orow = part * rows + (int64_t)w.b * p.q_len * p.H + w.r_base + r;
      if (rank == 0) {
        p.LSE_part[orow] = -INFINITY;
      } else {
        float4* d4 = reinterpret_cast<float4*>(p.O_part + orow * MLA_VALUE_DIM);
        for (int e = 0; e < MLA_VALUE_DIM / 4; ++e) d4[e] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
  cluster_sync();
}

}  // namespace

int launch_tc(const DecodeArgs& a) {
  if (a.kv_dtype != MLA_KV_BF16)
    return fail(MLA_ERR_UNSUPPORTED, "tensor-core path: FP8 KV not built yet");
  TcParams p;
  p.q_nope = static_cast<const uint4*>(a.q_nope);
  p.q_rope = static_cast<const uint4*>(a.q_rope);
  p.num_slots = a.num_slots;
  p.r2t = a.req_to_token;
  p.r2t_stride = a.r2t_stride;
  p.seq_lens = a.seq_lens;
  p.kv_limit = a.kv_limit;
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
  int rc = make_kv_tensor_map(&map, a.kv, a.kv_dtype, a.num_slots);
  if (rc != MLA_OK) return rc;
  cudaError_t e = cudaFuncSetAttribute(
      mla_partial_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
      kSmemBytes);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(tc)");
  mla_partial_tc_kernel<<<(unsigned)(pairs * 2), kThreads, kSmemBytes,
                          a.stream>>>(map, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch mla_partial_tc_kernel");
  return MLA_OK;
}

}  // namespace mla

extern "C" int mla_pair_slots(void) {
  cudaError_t e = cudaFuncSetAttribute(
      mla::mla_partial_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
      mla::kSmemBytes);
  if (e != cudaSuccess) return mla::cuda_fail(e, "cudaFuncSetAttribute(tc)");
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * 1024, 1, 1);
  cfg.blockDim = dim3(mla::kThreads, 1, 1);
  cfg.dynamicSmemBytes = mla::kSmemBytes;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, mla::mla_partial_tc_kernel, &cfg);
  if (e != cudaSuccess) return mla::cuda_fail(e, "cudaOccupancyMaxActiveClusters");
  return clusters;
}
