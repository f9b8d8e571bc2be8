// decode.cu -- INT8 paged decode attention (and the debug QK path).
//
// Source: "gfx936 DCU上实现INT8 PV MMAC：V Scale融合、概率量化与Fragment分组"
// §1 (W = P x sV, 32-token groups, sW = max W / 127), §2 (score recovery
// acc x sQ x sK / sqrt(d), online softmax), §2.2 (decode: 256-token partitions
// merged by log-sum-exp), §3 (P on the A side, V on the B side of the INT8
// MMA; int32 bound 32 x 127 x 127 per group) and "gfx936 DCU上实现INT8 KV与
// INT8 MMAC Attention推理优化" §3.3 (the decode data flow) and §2.3 (layouts).
//
// GB300 design (not the pages' gfx936 one): a persistent, warp-specialized CTA.
//  * Work unit = (sequence, KV head, a run of 32-token granules): 128 tokens at
//    head_dim 256, 256 tokens at head_dim 128 (the same bytes per ring item).
//    The grid has one CTA per SM; CTA c takes the contiguous granule range
//    [c U / N, (c+1) U / N).  A pair (sequence, KV head) that spans CTAs leaves
//    one partial (o, m, l) per CTA in the workspace, and decode_merge_kernel
//    combines them by log-sum-exp.  A unit is only a work granule: the pages'
//    256-token partition fixes no arithmetic here, because the group
//    quantization below does not depend on where the softmax normalization is
//    applied.
//  * Producer warp: per unit, bulk copies (TMA) of the unit's K pages into a K
//    slot of the unit's QK stream, together with the unit's K and V scales
//    (cp.async, next to the pages), then its V pages into the next V slot.
//    Block-table entries are read two units ahead.  Full/empty mbarriers guard
//    the slots.
//  * 8 QK warps in streams (two streams of 4 at head_dim 256, taking the even
//    and the odd units; one stream of 8 at head_dim 128); in a unit, warp w of a
//    stream owns tokens 32w .. 32w+31, one probability group.  QK on mma.sync
//    m16n8k32 s8 (exact int32; M = 16 tokens, N = 8 GQA-packed query rows), the
//    score recovery in log2 units, the group's row maximum m_g,
//    p~ = 2^(s - m_g), W = p~ x sV, sW = max W / 127 and the codes
//    Wq = round(W / sW).  The raw codes go to a handoff buffer (unit i uses
//    buffer i % 4) as the PV MMA's B fragments, with sW, m_g and the group's
//    row sums l_g.  No QK warp waits for another: the group quantization gives
//    the same codes for W scaled by any positive factor, so each group is
//    quantized against its own maximum and brought to the common one afterwards.
//  * PV warps (8 at head_dim 256, 4 at head_dim 128): warp v owns head-dims
//    [32 v, 32 (v+1)) of the output and keeps the pair's running maximum m.
//    Per unit, m_new = max(m, m_g), the accumulator and l are rescaled once by
//    2^(m - m_new), and group g adds 2^(m_g - m_new) sW_g (Wq x Vq)
//    (mma.sync m16n8k32 s8, exact int32, K = the group's 32 tokens; s8 x u8 for
//    UINT8 probability codes) and 2^(m_g - m_new) l_g.  The accumulator covers
//    disjoint dims, so the end of a segment needs no cross-warp reduction: each
//    PV warp writes its own dims (final output or partial).
//  * Ring slots: each QK stream has its own K slot(s), consumed in order, and
//    the other slots carry V items in unit order, so every slot is refilled
//    only after its previous item was consumed.
//  * Every product (<= 127^2, or 255 x 127) and every sum (QK over 256 dims:
//    <= 4,129,024; PV over one group: <= 1,036,320) is exact in int32 and in the
//    fp32 rescale; the debug QK entry point checks the accumulators bit for bit
//    against integer QK.
#include <cuda_bf16.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace i8kv {

namespace {

constexpr int kPart = 256;   // the pages' decode partition (debug QK tiles)
constexpr int kBS = 16;      // block size
constexpr int kGroup = 32;   // probability group
constexpr int kQKWarps = 8;  // QK / softmax warps, in kStreams streams of kQW (per variant, below)
constexpr int kPVWarp0 = kQKWarps;  // then the PV warps (kPW per variant), then the producer warp
constexpr int kHandBufs = 4;  // handoff buffers, unit i uses buffer i % 4
constexpr int kRows = 8;     // query rows in the MMA N dimension
__host__ __device__ constexpr int kSlotFloats(int D) { return kRows * D + 2 * kRows; }

// Geometry of one variant.  The 8 QK warps form kStreams streams of kQW warps;
// stream s takes the units i with i % kStreams == s, one granule per QK warp.
// INT8: 32-token granules (one probability group per QK warp); BF16-KV
// comparison: 16-token granules (one block per QK warp), plain softmax weights.
// At D = 256 two streams of 4 warps: 128-token INT8 units of 66 KB of K and V.
// At D = 128 one stream of 8 warps: 256-token units, the same bytes per ring
// item, so the per-unit work (copies, handoff, rescale) is spread over as many
// bytes as at D = 256.  PV warps: 8 of 32 head-dims at D = 256; 4 of 32 at
// D = 128, where 8 warps of 16 dims spent more issue slots on each unit's
// group factors (every PV warp computes them for all rows) than on their MMAs.
template <int D, bool BF16>
struct Geo {
  static constexpr int kStreams = D == 128 ? 1 : 2;             // QK streams
  static constexpr int kPW = D == 128 ? 4 : 8;                  // PV warps
  static constexpr int kProdWarp = kPVWarp0 + kPW;              // the producer warp
  static constexpr int kThreads = (kProdWarp + 1) * 32;
  static constexpr int kQW = kQKWarps / kStreams;               // QK warps per stream = granules per unit
  static constexpr int EB = BF16 ? 2 : 1;                       // bytes per cache element
  static constexpr int kUnit = kQW * (BF16 ? 16 : 32);          // tokens per unit
  static constexpr int kBlocksU = kUnit / kBS;                  // pages per ring item
  static constexpr int kPage = D * kBS * EB;                    // one (block, KV head) page
  static constexpr int kPages = kBlocksU * kPage;
  static constexpr int kScales = kPages;                         // INT8: float2 (sK, sV) per token (K items)
  static constexpr int kSlot = (kPages + (BF16 ? 0 : kUnit * 8) + 127) / 128 * 128;
  // decode step: a stream's buffer of quantized rows, the query rows then the
  // new token's K and V (codes [kRows + 2][D], then their scales)
  static constexpr int kQNewK = kRows, kQNewV = kRows + 1;
  static constexpr int kQScl = (kRows + 2) * D;
  static constexpr int kQBuf = BF16 ? 0 : kQScl + 48;
  static constexpr int kWTok = kUnit / kQW;                     // tokens per QK warp
  static constexpr int kGran = kWTok;                           // work-split granule (one QK warp's tokens)
  static constexpr int MT = kWTok / 16;                         // 16-token blocks per QK warp
  static constexpr int kDimsPW = D / kPW;                       // head-dims per PV warp
  static constexpr int NDT = kDimsPW / 16;                      // 16-dim MMA tiles per PV warp
  static constexpr int kFrag = 8;                               // B-fragment bytes per lane (bf16 p~ or s8 codes)
  // handoff buffer: [kQW][32 lanes] B fragments, then per row r and group q
  // (QK warp): sW [8][kQW] | m [8][kQW] | l [8][kQW] (a row's 4 groups in 16
  // bytes), then (decode step) the new token's V codes [D] for the unit holding it
  static constexpr int kHSw = kQW * 32 * kFrag;
  static constexpr int kHM = kHSw + kQW * kRows * 4;
  static constexpr int kHL = kHM + kQW * kRows * 4;
  static constexpr int kHPatch = kHL + kQW * kRows * 4;
  static constexpr int kHand = kHPatch + (BF16 ? 0 : D);
  static_assert(kQBuf % 16 == 0 && kHand % 16 == 0, "buffers are read as 16-byte vectors");
  static constexpr int kStage = kRows * kWTok * EB;             // per-QK-warp code/weight transpose
  static_assert(kGroup == kWTok || BF16, "an INT8 QK warp owns exactly one probability group");
  static_assert(kSlot % 128 == 0 && kHand % 16 == 0, "alignment");
};

struct SmemLayout {
  size_t ring, hand, stage, qbuf, bars, ctrl, total;
};

template <int D, bool BF16>
__host__ __device__ inline SmemLayout decode_layout(int nslots) {
  using Gm = Geo<D, BF16>;
  SmemLayout L;
  size_t off = 0;
  L.ring = off;
  off += (size_t)nslots * Gm::kSlot;
  L.hand = off;
  off += (size_t)kHandBufs * Gm::kHand;
  L.stage = off;
  off += (size_t)kQKWarps * Gm::kStage;
  L.qbuf = off;  // [stream] query codes [8][D] and scales [8] (decode step)
  off += (size_t)Gm::kStreams * Gm::kQBuf;
  L.bars = off;  // full[nslots], empty[nslots], hfull[4], hempty[4]
  off += (size_t)(2 * nslots + 2 * kHandBufs) * sizeof(uint64_t);
  L.ctrl = off;
  off += 32 * sizeof(int);
  L.total = off;
  return L;
}

// Position in the CTA's sequence of units.  The work is split over granules
// (one QK warp's tokens: a 32-token probability group, or a 16-token block for
// the BF16 comparison) in (sequence, KV head, token) order; a unit is up to kQW
// consecutive granules of one (sequence, KV head) pair inside the CTA's range.
struct Walk {
  int b, kvh, gi, ngp, L, n;  // sequence, KV head, first granule in the pair, granules per pair, length,
                              // granules in this unit (0 = past the CTA's range)
  long long gb;               // global index of sequence b's first granule
  long long gc;               // global index of this unit's first granule
};

__device__ __forceinline__ int clamp_len(int L, int maxL) {
  if (L < 0) return 0;
  return L > maxL ? maxL : L;
}

// Granules of the unit that starts at w: up to maxg (one per QK warp of a stream).
__device__ __forceinline__ int unit_granules(const Walk& w, long long g_end, int maxg) {
  if (w.gc >= g_end) return 0;
  const long long left = g_end - w.gc;
  const int in_pair = w.ngp - w.gi;
  const int n = in_pair < maxg ? in_pair : maxg;
  return left < n ? (int)left : n;
}

__device__ __forceinline__ void walk_next(Walk& w, const int32_t* seq_lens, int B, int Hkv, int maxL, int gran,
                                          long long g_end, int maxg) {
  w.gc += w.n;
  w.gi += w.n;
  if (w.gi >= w.ngp) {
    w.gi = 0;
    if (++w.kvh >= Hkv) {
      w.kvh = 0;
      w.gb += (long long)w.ngp * Hkv;
      for (;;) {
        if (++w.b >= B) {
          w.n = 0;
          return;
        }
        w.L = clamp_len(seq_lens[w.b], maxL);
        w.ngp = (w.L + gran - 1) / gran;
        if (w.ngp > 0) break;
      }
    }
  }
  w.n = unit_granules(w, g_end, maxg);
}

// floor(a / d), d >= 1.  Below 2^22 the product of the exact operand a and a
// reciprocal of d within one ulp, rounded toward zero, is within 2^-22 a / d < 1
// of the quotient, so its integer part is off by at most one and one remainder
// step corrects it: a few instructions where the integer division is a long
// dependent sequence (the kernel's start-up path runs several in a row).
__device__ __forceinline__ unsigned udiv_fast(unsigned a, unsigned d) {
  if (a >= (1u << 22) || d >= (1u << 22)) return a / d;
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(__uint2float_rn(d)));
  unsigned q = __float2uint_rz(__fmul_rz(__uint2float_rn(a), r));
  const int rem = (int)(a - q * d);  // q * d <= a + d < 2^23
  if (rem < 0)
    --q;
  else if (rem >= (int)d)
    ++q;
  return q;
}

// floor(U * c / N), in 32-bit arithmetic when U fits (the 64-bit division is a
// long instruction sequence on the kernel's start-up path).
__device__ __forceinline__ long long split_point(long long U, int c, int N) {
  if (U < (1ll << 31)) {
    const unsigned u = (unsigned)U, q = udiv_fast(u, (unsigned)N), r = u - q * (unsigned)N;
    return (long long)q * c + udiv_fast(r * (unsigned)c, (unsigned)N);
  }
  return U * c / N;
}

// Hash of the sequence lengths one lane reads (its lanes' entries in chunk
// order), to see whether they changed between the read before griddep_wait()
// and the one after it.
__device__ __forceinline__ uint32_t len_hash(uint32_t h, int raw) { return h * 0x9E3779B1u + (uint32_t)raw; }

// CTA whose granule range [c*U/N, (c+1)*U/N) holds granule u (N <= U: no empty ranges).
__device__ __forceinline__ int cta_of(long long u, long long U, int N) {
  return (int)(((u + 1) * N + U - 1) / U - 1);
}

// Ring slots.  Slots [0, kStreams kK) hold K items: stream s owns [s kK, (s+1) kK)
// and fills them with its own units in order (j = i / kStreams is unit i's index
// within its stream), so each K slot is consumed by one stream, in order.  Slots
// [kStreams kK, nslots) hold the V items of all units, in order.  Every slot is
// therefore reused only after its previous item was consumed, which keeps each
// mbarrier within one phase of its waiters.
struct Ring {
  int kK, nV;
  // A stream releases its K slot right after its QK MMAs, long before its unit
  // is done.  With two streams their units alternate, so one K slot each (two
  // at 12 slots) keeps them fed: one stream's next K lands while the other
  // computes.  A single stream (head_dim 128) gets two K slots, so its own next
  // unit's K is in flight while it computes the current one (batch-16 decode
  // at 32768 tokens, 32 q / 8 KV heads: 245 -> 221 us; at head_dim 256 the V
  // side cannot spare the slots).
  // The rest of the ring holds V items, which wait for the QK warps' handoff.
  __host__ __device__ static int k_slots(int nslots, int streams) {
    const int k = nslots / 6 > 0 ? nslots / 6 : 1;
    return streams == 1 && k < 2 ? 2 : k;
  }
  __host__ __device__ Ring(int nslots, int streams)
      : kK(k_slots(nslots, streams)), nV(nslots - streams * k_slots(nslots, streams)) {}
};

// A position in a ring of n slots: the slot, and how many times the ring was
// passed before it (whose parity is the phase to wait for).  It advances one
// item at a time, so the pipeline loops do no division.
struct RingPos {
  int s = 0, use = 0;
  __device__ void next(int n) {
    if (++s == n) {
      s = 0;
      ++use;
    }
  }
};

// Bounded pipeline wait.  After a timeout (error 1) or once the CTA aborted,
// it returns without waiting so every thread still reaches the same barriers.
// A waiting warp sleeps inside try_wait (up to 20 us per try) instead of
// spinning, so it takes no issue slots from the warps that have work.
__device__ __forceinline__ void pipe_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return;
  if (*abort_flag) return;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait_sleep(bar, parity, 20000u)) {
    if (*abort_flag) return;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      record_error(1);
      *abort_flag = 1;
      return;
    }
  }
}

// Query fragments (B operand of the s8 QK MMA) of the GQA-packed rows: column g
// of the N-tile is query head kvh*G + g; per 32-dim step s the fragment holds
// dims 32s + {4t..4t+3} and 32s + 16 + {4t..4t+3} as raw int8.
template <int D>
__device__ __forceinline__ void load_q_frags(const int8_t* q, int b, int Hq, int kvh, int G, int lane,
                                             uint32_t (&qf)[D / 32][2]) {
  const int g = lane >> 2, t = lane & 3;
  const int8_t* row = q + ((size_t)b * Hq + kvh * G + g) * D;
#pragma unroll
  for (int s = 0; s < D / 32; ++s) {
    qf[s][0] = g < G ? __ldg(reinterpret_cast<const uint32_t*>(row + 32 * s + 4 * t)) : 0u;
    qf[s][1] = g < G ? __ldg(reinterpret_cast<const uint32_t*>(row + 32 * s + 16 + 4 * t)) : 0u;
  }
}

// QK for the two 16-token blocks (2w, 2w+1) of warp w's group on the INT8 tensor
// path (mma.sync m16n8k32, s8 x s8 -> s32: exact):
// acc[m][0..3] = (token g, row 2t), (token g, row 2t+1), (token g+8, row 2t),
// (token g+8, row 2t+1) of block 2w+m.  kpages holds 16 K pages [D/16][16][16 B];
// ldmatrix of (tokens 0-7 | 8-15) x (dim chunk 2s | 2s+1) of a page is the s8 A
// fragment of dims 32s .. 32s + 31 as it is, so K is never converted.
template <int D>
__device__ __forceinline__ void qk_warp(const int8_t* kpages, int warp, int lane, const uint32_t (&qf)[D / 32][2],
                                        float (&acc)[2][4]) {
  const int mi = lane >> 3, ri = lane & 7;
  // even and odd 32-dim steps accumulate separately: two independent MMA chains per block
  int ae[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}}, ao[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}};
#pragma unroll
  for (int s = 0; s < D / 32; ++s) {
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      const int8_t* row =
          kpages + (size_t)(2 * warp + m) * (D * kBS) + (mi >> 1) * (kBS * 16) + (ri + 8 * (mi & 1)) * 16;
      uint32_t a[4];
      ldmatrix_x4(a, row + (size_t)(2 * s) * (kBS * 16));
      mma_s8_16832((s & 1) ? ao[m] : ae[m], a, qf[s][0], qf[s][1]);
    }
  }
#pragma unroll
  for (int m = 0; m < 2; ++m)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[m][i] = (float)(ae[m][i] + ao[m][i]);  // |sum| < 2^23: exact
}

// BF16-KV comparison path: query fragments (B operand of QK) straight from the
// bf16 query, qf[s] = dims 16s + {2t, 2t+1} and 16s + 8 + {2t, 2t+1} of row g.
template <int D>
__device__ __forceinline__ void load_q_frags_bf16(const uint16_t* q, int b, int Hq, int kvh, int G, int lane,
                                                  uint32_t (&qf)[D / 16][2]) {
  const int g = lane >> 2, t = lane & 3;
  const uint16_t* row = q + ((size_t)b * Hq + kvh * G + g) * D;
#pragma unroll
  for (int s = 0; s < D / 16; ++s) {
    qf[s][0] = g < G ? __ldg(reinterpret_cast<const uint32_t*>(row + 16 * s + 2 * t)) : 0u;
    qf[s][1] = g < G ? __ldg(reinterpret_cast<const uint32_t*>(row + 16 * s + 8 + 2 * t)) : 0u;
  }
}

// BF16-KV QK for warp w's 16-token block: acc = (token g | g+8) x (row 2t, 2t+1).
// kpages holds 8 bf16 K pages [D/8][16 tokens][8 dims].
template <int D>
__device__ __forceinline__ void qk_warp_bf16(const uint8_t* kpages, int warp, int lane,
                                             const uint32_t (&qf)[D / 16][2], float (&acc)[4]) {
  const int mi = lane >> 3, ri = lane & 7;
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i] = 0.f;
  const uint8_t* row = kpages + (size_t)warp * (D * kBS * 2) + (mi >> 1) * (kBS * 16) + (ri + 8 * (mi & 1)) * 16;
#pragma unroll
  for (int s = 0; s < D / 16; ++s) {
    uint32_t a[4];
    ldmatrix_x4(a, row + (size_t)(2 * s) * (kBS * 16));
    mma_bf16_16816(acc, a, qf[s][0], qf[s][1]);
  }
}


// ---- the decode step's quantization (the producer's rule, inside the kernel) ----
// scale = amax / 127 (IEEE), code = round-half-even(x / scale) with the IEEE
// quotient (Markstein's method, one reciprocal per vector), all codes 0 and
// scale 0 for a zero vector -- the same arithmetic as kv_quant_write_kernel,
// so the codes and scales are bit-identical to the two-kernel path.
__device__ __forceinline__ uint32_t quant4(const float (&x)[4], float scale, float y, bool nz) {
  if (!nz) return 0u;
  float q[4] = {x[0], x[1], x[2], x[3]};
  div_row(q, scale, y);
  const uint32_t lo = __byte_perm(rne_bits(q[0]), rne_bits(q[1]), 0x0040);
  const uint32_t hi = __byte_perm(rne_bits(q[2]), rne_bits(q[3]), 0x0040);
  return __byte_perm(lo, hi, 0x5410);
}

__device__ __forceinline__ void unpack_bf16x4(uint2 r, float (&x)[4]) {
  x[0] = bf16_bits_to_float(r.x & 0xffffu);
  x[1] = bf16_bits_to_float(r.x >> 16);
  x[2] = bf16_bits_to_float(r.y & 0xffffu);
  x[3] = bf16_bits_to_float(r.y >> 16);
}

// One D-vector quantized by a whole warp: lane l holds elements l*E .. l*E+E-1
// (E = D / 32) and gets their codes packed 4 per word.  Loading is split from
// quantizing so that a caller issues the loads of all its rows first (one
// global round trip for the batch, not one per row).
template <int D>
struct RowRaw {
  uint2 w[D / 128];
};

template <int D>
__device__ __forceinline__ RowRaw<D> load_row_warp(const uint16_t* row, int lane) {
  RowRaw<D> r;
#pragma unroll
  for (int j = 0; j < D / 128; ++j) r.w[j] = __ldg(reinterpret_cast<const uint2*>(row + lane * (D / 32)) + j);
  return r;
}

// Returns the scale.
template <int D>
__device__ __forceinline__ float quant_row_warp(const RowRaw<D>& raw, uint32_t (&packed)[D / 128]) {
  float x[D / 128][4];
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < D / 128; ++j) {
    unpack_bf16x4(raw.w[j], x[j]);
#pragma unroll
    for (int i = 0; i < 4; ++i) amax = fmaxf(amax, fabsf(x[j][i]));
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const float scale = div127(amax);  // amax / 127, correctly rounded
  const float y = __frcp_rn(scale);
  const bool nz = amax > 0.f;
#pragma unroll
  for (int j = 0; j < D / 128; ++j) packed[j] = quant4(x[j], scale, y, nz);
  return nz ? scale : 0.f;
}

// Query fragments (B operand of the s8 QK MMA) from int8 codes in shared memory,
// rows [8][D] (the decode step's query buffer); same layout as load_q_frags.
template <int D>
__device__ __forceinline__ void load_q_frags_smem(const uint8_t* qa, int G, int lane, uint32_t (&qf)[D / 32][2]) {
  const int g = lane >> 2, t = lane & 3;
  const uint8_t* row = qa + g * D;
#pragma unroll
  for (int s = 0; s < D / 32; ++s) {
    qf[s][0] = g < G ? *reinterpret_cast<const uint32_t*>(row + 32 * s + 4 * t) : 0u;
    qf[s][1] = g < G ? *reinterpret_cast<const uint32_t*>(row + 32 * s + 16 + 4 * t) : 0u;
  }
}

// One kernel body for both caches.  BF16 = false: the INT8 method.  BF16 = true:
// the BF16-KV comparison (plain softmax, bf16 P x V, no scales).  STEP (INT8
// only): the decode step, which also quantizes and writes each sequence's new
// token and quantizes the query; a separate instantiation, so the plain decode
// carries none of that code.  U8P (INT8 only): UINT8 probability codes --
// sW = A / 255, Wq in 0..255, PV on the s8 x u8 MMA (|PV| <= 32 x 255 x 127,
// still exact in fp32); the pages' notes on PV weigh this variant and leave it
// for want of a mixed-sign MMA, which sm_103a's mma.sync has.
template <int D, bool BF16, bool STEP = false, bool U8P = false>
__global__ void __launch_bounds__(Geo<D, BF16>::kThreads, 1) decode_kernel(DecodeParams p, int nslots) {
  static_assert(!(STEP && BF16), "the decode step is INT8 only");
  constexpr int kQW = Geo<D, BF16>::kQW, kStreams = Geo<D, BF16>::kStreams;
  static_assert(!(U8P && (BF16 || STEP)), "UINT8 probabilities: plain INT8 decode only");
  using Gm = Geo<D, BF16>;
  constexpr int kUnit = Gm::kUnit, kBlocksU = Gm::kBlocksU, kPage = Gm::kPage, kSlot = Gm::kSlot;
  constexpr int kGran = Gm::kGran;
  constexpr int kWTok = Gm::kWTok, MT = Gm::MT, NDT = Gm::NDT;
  constexpr int kPW = Gm::kPW, kProdWarp = Gm::kProdWarp;
  static_assert(kBlocksU <= 16, "a unit's block-table row fits ctrl[16 .. 31]");
  extern __shared__ __align__(1024) uint8_t smem[];
  const SmemLayout lay = decode_layout<D, BF16>(nslots);
  uint8_t* ring = smem + lay.ring;
  uint8_t* hand = smem + lay.hand;
  uint8_t* stage = smem + lay.stage;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + lay.bars);
  uint64_t* empty = full + nslots;
  uint64_t* hfull = empty + nslots;
  uint64_t* hempty = hfull + kHandBufs;
  int* ctrl = reinterpret_cast<int*>(smem + lay.ctrl);
  volatile int* abort_flag = ctrl + 8;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int B = p.B, Hkv = p.Hkv, G = p.G, Hq = p.Hq;
  const int N = gridDim.x, c = blockIdx.x;
  const int maxL = p.max_blocks * kBS;

  // The prologue before the wait runs in three warps at once: the producer
  // warp computes the work split, warp 0 initializes the barriers and warp 1
  // guesses the first unit of a single sequence (below).  In one warp they took
  // about 1.8 us, past the release of the wait in most CTAs.
  const int raw0 = (warp == kProdWarp && lane < B) ? __ldcg(p.seq_lens + lane) : 0;
  if (warp == 0 && lane == 0) {
    const Ring rg(nslots, Gm::kStreams);
    for (int s = 0; s < nslots; ++s) {
      mbar_init(&full[s], 32);
      mbar_init(&empty[s], s < kStreams * rg.kK ? kQW : kPW);
    }
    for (int j = 0; j < kHandBufs; ++j) {
      mbar_init(&hfull[j], kQW * 32);
      mbar_init(&hempty[j], kPW);
    }
    fence_mbar_init();
  }
  // ---- work split, by the producer warp, before the wait on earlier work ----
  // seq_lens and block_tables are the only global memory read before
  // griddep_wait(), and nothing is written before it.  No kernel of this
  // library writes them, and reading them early overlaps their latency (and the
  // split's arithmetic) with the end of the previous kernel on the stream.  They
  // are read past L1 (ld.global.cg), so no stale line outlives the wait; after
  // it the producer warp reads them again and records error 3 if they changed
  // (the caller wrote them in the kernel just before this one).
  //
  // One sequence in the batch (the long-context decode case): warp 1 guesses
  // the first unit from max_blocks and loads its block-table row while the
  // producer warp loads seq_lens, so the two dependent loads overlap; the guess
  // (ctrl[15], the row in ctrl[16 ..]) is checked below.
  uint32_t lhash = 0;  // this lane's sequence lengths, for the check after the wait
  if (warp == 1) {
    int spec_gi = -1, spec_blk = -1;
    if (B == 1) {
      const int ngp_g = (maxL + kGran - 1) / kGran;
      const long long U_g = (long long)ngp_g * Hkv;
      const int Nw_g = (int)(U_g < N ? U_g : N);
      if (c < Nw_g) {
        const long long ub_g = split_point(U_g, c, Nw_g);  // < U_g
        spec_gi = ub_g < (1ll << 31) ? (int)((unsigned)ub_g - udiv_fast((unsigned)ub_g, ngp_g) * ngp_g)
                                     : (int)(ub_g % ngp_g);
        const int pg = spec_gi * kGran / kBS + lane;
        if (lane < kBlocksU && pg < p.max_blocks) spec_blk = __ldcg(p.block_tables + pg);
      }
    }
    if (lane == 0) ctrl[15] = spec_gi;
    if (lane < 16) ctrl[16 + lane] = spec_blk;
  }
  if (warp == kProdWarp && B == 1) {
    // One sequence: no reduction or scan over the batch.  The same values as the
    // general split below (sequence 0 starts at granule 0).
    lhash = lane == 0 ? len_hash(0u, raw0) : 0u;
    const int L = clamp_len(__shfl_sync(0xffffffffu, raw0, 0), maxL);
    const int ngp = (L + kGran - 1) / kGran;  // granules per pair
    const long long U = (long long)ngp * Hkv;
    const int Nw = (int)(U < N ? U : N);
    const long long ub = c < Nw ? split_point(U, c, Nw) : 0, ue = c < Nw ? split_point(U, c + 1, Nw) : 0;
    if (lane == 0) {
      ctrl[0] = (int)(ue - ub);
      ctrl[8] = 0;
      if (ue > ub) {
        const unsigned kv = udiv_fast((unsigned)ub, (unsigned)ngp);  // ub < ngp * Hkv, as in the scan below
        ctrl[1] = 0;
        ctrl[2] = (int)kv;
        ctrl[3] = (int)((unsigned)ub - kv * (unsigned)ngp);
        ctrl[4] = 0;
        ctrl[5] = 0;
        ctrl[9] = L;
      }
    }
  } else if (warp == kProdWarp) {
    constexpr int kKeep = 8;  // chunks of 32 sequences whose unit counts stay in registers
    int ukeep[kKeep], lkeep[kKeep];
    long long total = 0;
    for (int b0 = 0, ck = 0; b0 < B; b0 += 32, ++ck) {
      const int b = b0 + lane;
      int u = 0, L = 0;
      if (b < B) {
        const int raw = ck == 0 ? raw0 : __ldcg(p.seq_lens + b);
        lhash = len_hash(lhash, raw);
        L = clamp_len(raw, maxL);
        u = (L + kGran - 1) / kGran * Hkv;
      }
#pragma unroll
      for (int k = 0; k < kKeep; ++k)
        if (k == ck) {
          ukeep[k] = u;
          lkeep[k] = L;
        }
      int su = u;
      for (int o = 16; o >= 1; o >>= 1) su += __shfl_xor_sync(0xffffffffu, su, o);
      total += su;
    }
    const long long U = total;
    // Only the first min(N, U) CTAs take granules, so every working CTA has at
    // least one and the CTAs covering a pair are consecutive.
    const int Nw = (int)(U < N ? U : N);
    const long long ub = c < Nw ? split_point(U, c, Nw) : 0, ue = c < Nw ? split_point(U, c + 1, Nw) : 0;
    if (lane == 0) {
      ctrl[0] = (int)(ue - ub);
      ctrl[8] = 0;
    }
    if (ue > ub) {
      long long run = 0;
      for (int b0 = 0, ck = 0; b0 < B; b0 += 32, ++ck) {
        const int b = b0 + lane;
        int u = 0, L = 0;
        if (ck < kKeep) {
#pragma unroll
          for (int k = 0; k < kKeep; ++k)
            if (k == ck) {
              u = ukeep[k];
              L = lkeep[k];
            }
        } else if (b < B) {
          L = clamp_len(__ldcg(p.seq_lens + b), maxL);
          u = (L + kGran - 1) / kGran * Hkv;
        }
        int incl = u;
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const long long ex = run + incl - u, in = run + incl;
        const unsigned hit = __ballot_sync(0xffffffffu, u > 0 && ex <= ub && ub < in);
        if (hit) {
          if (lane == __ffs(hit) - 1) {
            const unsigned np = (unsigned)((L + kGran - 1) / kGran);  // granules per pair
            const unsigned local = (unsigned)(ub - ex);                // < np * Hkv
            const unsigned kv = udiv_fast(local, np);
            ctrl[1] = b;
            ctrl[2] = (int)kv;
            ctrl[3] = (int)(local - kv * np);
            ctrl[4] = (int)(ex & 0x7fffffff);
            ctrl[5] = (int)(ex >> 31);
            ctrl[9] = L;
          }
          break;
        }
        run += __shfl_sync(0xffffffffu, incl, 31);
      }
    }
  }
  __syncthreads();  // the split in ctrl[] is visible to every warp
  const int n_gran = ctrl[0];
  Walk w0;
  w0.b = ctrl[1];
  w0.kvh = ctrl[2];
  w0.gi = ctrl[3];
  w0.gb = (long long)ctrl[4] | ((long long)ctrl[5] << 31);
  w0.L = ctrl[9];
  w0.ngp = (w0.L + kGran - 1) / kGran;
  w0.gc = w0.gb + (long long)w0.kvh * w0.ngp + w0.gi;
  const long long g_end = w0.gc + n_gran;  // end of this CTA's granule range
  w0.n = n_gran > 0 ? unit_granules(w0, g_end, Gm::kQW) : 0;
  // This lane's page of the first unit (lanes below the unit's page count).
  auto first_blk_lanes = [&]() {
    const int t0 = w0.gi * kGran;
    return (min(w0.n * kGran, w0.L - t0) + kBS - 1) / kBS;
  };
  int blk_first = -1;
  if (warp == kProdWarp && n_gran > 0 && lane < first_blk_lanes()) {
    blk_first = (B == 1 && w0.gi == ctrl[15])
                    ? ctrl[16 + lane]
                    : __ldcg(p.block_tables + (size_t)w0.b * p.max_blocks + w0.gi * kGran / kBS + lane);
  }
  // The producer warp, after the wait: sequence lengths above the table are
  // recorded (error 2); empty sequences get zero rows and no merge; the inputs
  // read before the wait must not have changed (error 3).
  auto check_inputs = [&]() {
    uint32_t h = 0;
    for (int b0 = 0; b0 < B; b0 += 32) {
      const int b = b0 + lane;
      if (b < B) {
        const int raw = p.seq_lens[b];
        h = len_hash(h, raw);
        if (raw > maxL) record_error(2);
        if (clamp_len(raw, maxL) == 0 && b % N == c) {
          for (int i = 0; i < Hq * D; i += 4)
            store_out4(p.out, p.out_bf16, (size_t)b * Hq * D + i, make_float4(0.f, 0.f, 0.f, 0.f));
        }
      }
    }
    bool changed = h != lhash;
    if (n_gran > 0 && lane < first_blk_lanes())
      changed |= p.block_tables[(size_t)w0.b * p.max_blocks + w0.gi * kGran / kBS + lane] != blk_first;
    if (__any_sync(0xffffffffu, changed) && lane == 0) record_error(3);
  };
  // From here on the kernel reads and writes what earlier work on the stream
  // uses: every role waits for it first, the producer warp after preparing its
  // walk (which reads nothing the previous kernel writes).  Short calls gain
  // 0.2 us from that: the walk took about 0.5 us after the wait.
  if (n_gran <= 0) {
    griddep_wait();
    griddep_launch_dependents();
    if (warp == kProdWarp) check_inputs();
    return;
  }
  const int g = lane >> 2, t = lane & 3;
  const Ring rg(nslots, Gm::kStreams);

  if (warp == kProdWarp) {
    // ================= producer warp =================
    const uint8_t* kc = static_cast<const uint8_t*>(p.k_cache);
    const uint8_t* vc = static_cast<const uint8_t*>(p.v_cache);
    const uint64_t pol = policy_evict_first();
    // This lane's page of a unit (lanes below the unit's page count), read from
    // the block table one unit ahead of its use.
    auto load_blk = [&](const Walk& u) {
      const int t0 = u.gi * kGran;
      const int nb = (min(u.n * kGran, u.L - t0) + kBS - 1) / kBS;
      if (lane >= nb) return -1;
      return p.block_tables[(size_t)u.b * p.max_blocks + t0 / kBS + lane];
    };
    // The block-table entries of the next two units are in flight while a unit is
    // issued (one unit ahead left the producer waiting on the load whenever a
    // unit's slots freed up sooner than the load returned).
    Walk wk = w0, wn = w0, wnn;
    walk_next(wn, p.seq_lens, B, Hkv, maxL, kGran, g_end, Gm::kQW);
    wnn = wn;
    if (wnn.n > 0) walk_next(wnn, p.seq_lens, B, Hkv, maxL, kGran, g_end, Gm::kQW);
    griddep_wait();
    griddep_launch_dependents();
    int blk_cur = blk_first;
    int blk_n = wn.n > 0 ? load_blk(wn) : -1;
    int n_k = 0, n_v = 0;  // K and V items issued
    RingPos kp_cur, kp_oth, vp;  // K positions of this unit's stream and of the other; V position
    for (int i = 0; wk.n > 0; ++i) {
      if (*abort_flag) break;
      const int blk_nn = wnn.n > 0 ? load_blk(wnn) : -1;  // in flight meanwhile
      const int t0 = wk.gi * kGran;
      const int ntok = min(wk.n * kGran, wk.L - t0);
      const int nblk = (ntok + kBS - 1) / kBS;
      int blk = blk_cur;
      if (lane < nblk && (blk < 0 || blk >= p.num_blocks)) {
        record_error(2);
        blk = -1;
      }
      const bool ok = blk >= 0;
      const uint32_t n_pages = __popc(__ballot_sync(0xffffffffu, ok));
      // K item: the pages by bulk copy, the unit's (sK, sV) per token by cp.async;
      // the slot's full barrier waits for both.
      const int kslot = (i % kStreams) * rg.kK + kp_cur.s, ku = kp_cur.use;
      if (ku > 0) pipe_wait(&empty[kslot], (ku - 1) & 1, abort_flag);
      if (*abort_flag) break;  // never refill a slot whose previous item was not consumed
      if (lane == 0) mbar_expect_tx(&full[kslot], n_pages * kPage);
      __syncwarp();
      uint8_t* kdst = ring + (size_t)kslot * kSlot;
      if (ok)
        bulk_g2s_hint(kdst + (size_t)lane * kPage, kc + ((size_t)blk * Hkv + wk.kvh) * kPage, kPage, &full[kslot],
                      pol);
      // The decode step's new token (position L - 1) is quantized and written by
      // the QK warps; its entries read here may predate that write and are
      // replaced in the consumers.
      if constexpr (!BF16) {
        float* sdst = reinterpret_cast<float*>(kdst + Gm::kScales);
#pragma unroll
        for (int r = 0; r < kUnit / 32; ++r) {
          const int tok = lane + 32 * r;
          const int bj = __shfl_sync(0xffffffffu, blk, tok / kBS);  // every lane takes part in the shuffle
          const bool v = tok < ntok && bj >= 0;
          const size_t si = ((size_t)(v ? bj : 0) * kBS + tok % kBS) * Hkv + wk.kvh;
          cp_async_4(sdst + 2 * tok, p.k_scale + si, v ? 4u : 0u);
          cp_async_4(sdst + 2 * tok + 1, p.v_scale + si, v ? 4u : 0u);
        }
        cp_async_mbar_arrive(&full[kslot]);
      }
      mbar_arrive(&full[kslot]);
      ++n_k;
      // V item
      kp_cur.next(rg.kK);
      if constexpr (kStreams == 2) {
        const RingPos tmp = kp_cur;  // the next unit belongs to the other stream
        kp_cur = kp_oth;
        kp_oth = tmp;
      }
      const int vslot = kStreams * rg.kK + vp.s, vu = vp.use;
      if (vu > 0) pipe_wait(&empty[vslot], (vu - 1) & 1, abort_flag);
      if (*abort_flag) break;
      if (lane == 0) mbar_expect_tx(&full[vslot], n_pages * kPage);
      __syncwarp();
      if (ok)
        bulk_g2s_hint(ring + (size_t)vslot * kSlot + (size_t)lane * kPage,
                      vc + ((size_t)blk * Hkv + wk.kvh) * kPage, kPage, &full[vslot], pol);
      mbar_arrive(&full[vslot]);
      ++n_v;
      vp.next(rg.nV);
      blk_cur = blk_n;
      blk_n = blk_nn;
      wk = wn;
      wn = wnn;
      if (wnn.n > 0) walk_next(wnn, p.seq_lens, B, Hkv, maxL, kGran, g_end, Gm::kQW);
    }
    if (*abort_flag) {
      // The consumers stopped waiting: hold the CTA (and its shared memory)
      // until every copy issued into it has landed.  Each slot has at most one
      // item in flight (a slot is refilled only after its consumers released it),
      // so waiting for the last phase issued into each slot covers them all.
      asm volatile("cp.async.wait_all;" ::: "memory");
      for (int sl = 0; sl < nslots; ++sl) {
        int uses;
        if (sl < kStreams * rg.kK) {
          const int st = sl / rg.kK, r = sl % rg.kK;
          const int js = n_k > st ? (n_k - st + kStreams - 1) / kStreams : 0;  // this stream's K items issued
          uses = js > r ? (js - r + rg.kK - 1) / rg.kK : 0;
        } else {
          const int v = sl - kStreams * rg.kK;
          uses = n_v > v ? (n_v - v + rg.nV - 1) / rg.nV : 0;
        }
        if (uses > 0) mbar_wait(&full[sl], (uses - 1) & 1);
      }
    }
    check_inputs();
    return;
  }

  if (warp < kPVWarp0) {
    griddep_wait();
    griddep_launch_dependents();
    // ================= QK / softmax warps (two streams) =================
    // Each warp quantizes its group against the group's own row maximum m_g:
    // p~ = exp(s - m_g), W = p~ sV, sW = max W / 127, Wq = round(W / sW).  The
    // codes do not depend on a per-group scale factor, so the PV warps bring
    // every group to the common running maximum later, by exp(m_g - m) folded
    // into sW; no QK warp waits for another.
    const int st = warp / kQW, qw = warp % kQW;  // stream; group within the unit
    const float c_scale = __fmul_rn(p.sm_scale, kLog2e);  // scores in log2 units: every exponential is one ex2
    const int tok0 = qw * kWTok;  // this warp's tokens within a unit
    uint8_t* stg = stage + warp * Gm::kStage;
    Walk wk = w0;
    if (st == 1) walk_next(wk, p.seq_lens, B, Hkv, maxL, kGran, g_end, Gm::kQW);
    int cur_pair = -1;
    uint32_t qf[D / 32][2];    // INT8: query fragments (raw s8)
    uint32_t qfb[D / 16][2];   // BF16: query fragments
    float sq[2] = {0.f, 0.f};
    RingPos kpos;  // this stream's K slots
    uint8_t* const qb = smem + lay.qbuf + (size_t)st * Gm::kQBuf;  // decode step: the stream's quantized rows
    for (int i = st; wk.n > 0; i += kStreams) {
      const int pair = wk.b * Hkv + wk.kvh;
      if (pair != cur_pair) {
        cur_pair = pair;
        if constexpr (BF16) {
          load_q_frags_bf16<D>(static_cast<const uint16_t*>(p.q), wk.b, Hq, wk.kvh, G, lane, qfb);
        } else if constexpr (STEP) {
          // Decode step: the stream's warps quantize the pair's query rows (warp
          // w: rows w and w + kQW) by the producer's rule into the stream's
          // buffer, then each builds its fragments from it.  The stream that
          // holds the unit with the pair's newest token (position L - 1) also
          // quantizes that token's K (warp kQW - 2) and V (warp kQW - 1) here,
          // writes them into the cache for later steps and keeps them in the
          // buffer: the unit's consumers patch their copies of the cache, which
          // may predate the write.  Units of a pair follow one another every kQW
          // granules, alternating between the streams.
          const long long g_last = wk.gc - wk.gi + wk.ngp - 1;  // the pair's last granule
          const bool own_new = g_last < g_end && ((wk.ngp - 1 - wk.gi) / kQW) % kStreams == 0;
          const int nrow = qw - (kQW - 2);  // 0: the new K row, 1: the new V row
          const bool new_row = own_new && nrow >= 0;
          RowRaw<D> qr[2], nr;
          int blk_new = -1;
          if (new_row) {
            nr = load_row_warp<D>((nrow == 0 ? p.k_new : p.v_new) + ((size_t)wk.b * Hkv + wk.kvh) * D, lane);
            blk_new = p.block_tables[(size_t)wk.b * p.max_blocks + (wk.L - 1) / kBS];
          }
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int r = qw + kQW * h;
            if (r < G) qr[h] = load_row_warp<D>(p.q_bf16 + ((size_t)wk.b * Hq + wk.kvh * G + r) * D, lane);
          }
          constexpr int E = D / 32;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int r = qw + kQW * h;
            if (r < G) {
              uint32_t codes[D / 128];
              const float sc = quant_row_warp<D>(qr[h], codes);
              if constexpr (E == 8)
                *reinterpret_cast<uint2*>(qb + r * D + lane * E) = make_uint2(codes[0], codes[1]);
              else
                *reinterpret_cast<uint32_t*>(qb + r * D + lane * E) = codes[0];
              if (lane == 0) reinterpret_cast<float*>(qb + Gm::kQScl)[r] = sc;
            }
          }
          uint32_t ncodes[D / 128];
          float nsc = 0.f;
          if (new_row) nsc = quant_row_warp<D>(nr, ncodes);
          // the query rows are in the buffer; the previous pair's new-token rows
          // were read by every warp of the stream
          named_bar_sync(1 + st, kQW * 32);
          if (new_row) {
            const int r = Gm::kQNewK + nrow;
            if constexpr (E == 8)
              *reinterpret_cast<uint2*>(qb + r * D + lane * E) = make_uint2(ncodes[0], ncodes[1]);
            else
              *reinterpret_cast<uint32_t*>(qb + r * D + lane * E) = ncodes[0];
            if (lane == 0) reinterpret_cast<float*>(qb + Gm::kQScl)[r] = nsc;
            // the cache entry (an invalid block is reported by the producer warp)
            if (blk_new >= 0 && blk_new < p.num_blocks) {
              const int off_new = (wk.L - 1) % kBS, d0 = lane * E;
              if (nrow == 0) {
                int8_t* kg = p.k_cache_w +
                             ((((size_t)blk_new * Hkv + wk.kvh) * (D / 16) + d0 / 16) * kBS + off_new) * 16 + d0 % 16;
                if constexpr (E == 8)
                  *reinterpret_cast<uint2*>(kg) = make_uint2(ncodes[0], ncodes[1]);
                else
                  *reinterpret_cast<uint32_t*>(kg) = ncodes[0];
              } else {
                int8_t* vg = p.v_cache_w + (((size_t)blk_new * Hkv + wk.kvh) * D + d0) * kBS + off_new;
#pragma unroll
                for (int e = 0; e < E; ++e) vg[(size_t)e * kBS] = (int8_t)((ncodes[e >> 2] >> (8 * (e & 3))) & 0xff);
              }
              if (lane == 0) {
                const size_t si = ((size_t)blk_new * kBS + off_new) * Hkv + wk.kvh;
                (nrow == 0 ? p.k_scale_w : p.v_scale_w)[si] = nsc;
              }
            }
          }
          load_q_frags_smem<D>(qb, G, lane, qf);
          const float* qsc = reinterpret_cast<const float*>(qb + Gm::kQScl);
          sq[0] = 2 * t < G ? qsc[2 * t] : 0.f;
          sq[1] = 2 * t + 1 < G ? qsc[2 * t + 1] : 0.f;
          // every warp has read the query rows before they are reused; the
          // new-token rows are in the buffer
          named_bar_sync(1 + st, kQW * 32);
        } else {
          load_q_frags<D>(static_cast<const int8_t*>(p.q), wk.b, Hq, wk.kvh, G, lane, qf);
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const int row = 2 * t + r;
            sq[r] = row < G ? p.q_scale[(size_t)wk.b * Hq + wk.kvh * G + row] : 0.f;
          }
        }
      }
      const int ntok = min(wk.n * kGran, wk.L - wk.gi * kGran);
      const bool active = qw < wk.n;  // every granule of the unit holds tokens
      // decode step: the new token's position in the unit, and whether it is in this warp's granule
      const int pos_new = wk.L - 1 - wk.gi * kGran;
      const bool new_here = STEP && wk.gi + wk.n == wk.ngp && pos_new / kGran == qw;

      // ---- K item: QK of this warp's tokens, and their scales ----
      const int kslot = st * rg.kK + kpos.s;
      pipe_wait(&full[kslot], kpos.use & 1, abort_flag);
      kpos.next(rg.kK);
      const uint8_t* kb = ring + (size_t)kslot * kSlot;
      if constexpr (!BF16) {
        // decode step: the warp whose granule holds the new token patches its K row
        if (new_here) {
          if (lane < D / 16) {
            uint8_t* page = ring + (size_t)kslot * kSlot + (size_t)(pos_new / kBS) * kPage;
            *reinterpret_cast<uint4*>(page + (size_t)lane * (kBS * 16) + (pos_new % kBS) * 16) =
                *reinterpret_cast<const uint4*>(qb + Gm::kQNewK * D + lane * 16);
          }
          __syncwarp();
        }
      }
      float acc[2][4];
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[m][e] = 0.f;
      if (active) {
        if constexpr (BF16)
          qk_warp_bf16<D>(kb, qw, lane, qfb, acc[0]);
        else
          qk_warp<D>(reinterpret_cast<const int8_t*>(kb), qw, lane, qf, acc);
      }
      float sk[4], sv[4];  // tokens g, g+8 of this warp's blocks 0 and 1
      if constexpr (!BF16) {
        const float2* scl = reinterpret_cast<const float2*>(kb + Gm::kScales);
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const float2 v = scl[tok0 + 16 * m + g + 8 * h];
            sk[2 * m + h] = v.x;
            sv[2 * m + h] = v.y;
          }
        if (new_here) {  // decode step: the new token's scales, from the stream's buffer
          const float* nsc = reinterpret_cast<const float*>(qb + Gm::kQScl);
#pragma unroll
          for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int h = 0; h < 2; ++h)
              if (tok0 + 16 * m + g + 8 * h == pos_new) {
                sk[2 * m + h] = nsc[Gm::kQNewK];
                sv[2 * m + h] = nsc[Gm::kQNewV];
              }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[kslot]);

      // ---- scores and the group's row maximum ----
      float s[MT][4];
      float gm[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int tok = tok0 + 16 * m + g + 8 * (e >> 1);
          float sc = -INFINITY;
          if (tok < ntok) {
            if constexpr (BF16)
              sc = __fmul_rn(acc[m][e], c_scale);
            else
              sc = __fmul_rn(__fmul_rn(__fmul_rn(acc[m][e], sq[e & 1]), sk[2 * m + (e >> 1)]), c_scale);
          }
          s[m][e] = sc;
          gm[e & 1] = fmaxf(gm[e & 1], sc);
        }
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int off = 4; off <= 16; off <<= 1) gm[r] = fmaxf(gm[r], __shfl_xor_sync(0xffffffffu, gm[r], off));

      // ---- weights: BF16 p~; INT8 W = p~ sV, sW, codes ----
      // In an active warp every row maximum is finite and masked scores are
      // -inf, so exp(s - m_g) is 0 there without a test.  An inactive warp
      // (no tokens of its group in the unit) publishes zeros.
      float swv[2] = {0.f, 0.f}, lg[2] = {0.f, 0.f};
      if constexpr (BF16) {
        uint16_t* pw = reinterpret_cast<uint16_t*>(stg);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float pe = active ? ex2(__fsub_rn(s[0][e], gm[e & 1])) : 0.f;
          lg[e & 1] += pe;
          pw[(2 * t + (e & 1)) * 16 + g + 8 * (e >> 1)] = __bfloat16_as_ushort(__float2bfloat16_rn(pe));
        }
      } else {
        float A[2] = {0.f, 0.f}, w[2][4];
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float pe = active ? ex2(__fsub_rn(s[m][e], gm[e & 1])) : 0.f;
            lg[e & 1] += pe;
            w[m][e] = __fmul_rn(pe, sv[2 * m + (e >> 1)]);
            A[e & 1] = fmaxf(A[e & 1], w[m][e]);
          }
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
          for (int off = 4; off <= 16; off <<= 1) A[r] = fmaxf(A[r], __shfl_xor_sync(0xffffffffu, A[r], off));
        // sW = A / 127 and the codes round(W / sW), both IEEE fp32 quotients
        // (W / sW by Markstein's method, one reciprocal per row); codes ->
        // [row][token] bytes, read back below as PV B fragments.
        // W / sW <= A / RN(A / 127) < 127.5 (A / RN(A / 255) < 255.5), so no
        // code needs clamping; the low byte is the code either way.
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          swv[r] = U8P ? div255(A[r]) : div127(A[r]);
          // this lane's values of row 2t + r: (block m, token g + 8 h) at e = r + 2 h
          float x[4] = {w[0][r], w[0][r + 2], w[1][r], w[1][r + 2]};
          if (A[r] > 0.f) {
            div_row(x, swv[r], __frcp_rn(swv[r]));
          } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) x[i] = 0.f;
          }
#pragma unroll
          for (int i = 0; i < 4; ++i)
            stg[(2 * t + r) * kGroup + 16 * (i >> 1) + g + 8 * (i & 1)] = (uint8_t)rne_bits(x[i]);
        }
      }
      __syncwarp();

      // ---- hand the group over to the PV warps ----
      const int hbi = i % kHandBufs;
      if (i >= kHandBufs) pipe_wait(&hempty[hbi], ((i / kHandBufs) - 1) & 1, abort_flag);
      uint8_t* hb = hand + (size_t)hbi * Gm::kHand;
      if (new_here) {  // decode step: the new token's V codes, for the PV warps' patch
        constexpr int E = D / 32;
        if constexpr (E == 8)
          *reinterpret_cast<uint2*>(hb + Gm::kHPatch + lane * E) =
              *reinterpret_cast<const uint2*>(qb + Gm::kQNewV * D + lane * E);
        else
          *reinterpret_cast<uint32_t*>(hb + Gm::kHPatch + lane * E) =
              *reinterpret_cast<const uint32_t*>(qb + Gm::kQNewV * D + lane * E);
      }
      if constexpr (BF16) {
        uint2 f;
        f.x = *reinterpret_cast<const uint32_t*>(stg + g * 32 + 4 * t);
        f.y = *reinterpret_cast<const uint32_t*>(stg + g * 32 + 16 + 4 * t);
        reinterpret_cast<uint2*>(hb)[qw * 32 + lane] = f;
      } else {
        // the s8 B fragment of PV: codes of row g, tokens 4t..4t+3 and 16+4t..16+4t+3
        reinterpret_cast<uint2*>(hb)[qw * 32 + lane] =
            make_uint2(*reinterpret_cast<const uint32_t*>(stg + g * kGroup + 4 * t),
                       *reinterpret_cast<const uint32_t*>(stg + g * kGroup + 16 + 4 * t));
      }
      // the group's row sums of p~ (relative to m_g)
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int off = 4; off <= 16; off <<= 1) lg[r] += __shfl_xor_sync(0xffffffffu, lg[r], off);
      if (g == 0) {
        float* hsw = reinterpret_cast<float*>(hb + Gm::kHSw);
        float* hm = reinterpret_cast<float*>(hb + Gm::kHM);
        float* hl = reinterpret_cast<float*>(hb + Gm::kHL);
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          hsw[(2 * t + r) * kQW + qw] = swv[r];
          hm[(2 * t + r) * kQW + qw] = active ? gm[r] : -INFINITY;
          hl[(2 * t + r) * kQW + qw] = lg[r];
        }
      }
      mbar_arrive(&hfull[hbi]);  // every thread: releases its own stores
      // the next unit of this stream: skip the other streams' units
#pragma unroll
      for (int k = 0; k < kStreams; ++k)
        if (k == 0 || wk.n > 0) walk_next(wk, p.seq_lens, B, Hkv, maxL, kGran, g_end, Gm::kQW);
    }
    return;
  }

  // ================= PV warps =================
  griddep_wait();
  griddep_launch_dependents();
  // One running maximum m per pair, advanced in unit order: per unit,
  // m_new = max(m, m_g over the unit's groups), o and l are rescaled by
  // exp(m - m_new), and group q adds exp(m_g - m_new) * sW_g * (Wq x Vq) to o and
  // exp(m_g - m_new) * l_g to l.
  const int pv_w = warp - kPVWarp0;
  const int mi = lane >> 3, ri = lane & 7;
  Walk wk = w0, w1 = w0;
  walk_next(w1, p.seq_lens, B, Hkv, maxL, kGran, g_end, Gm::kQW);
  int cur_pair = -1;
  RingPos vpos;  // V slots
  float o[NDT][4];
  float mrun[2] = {-INFINITY, -INFINITY}, lrun[2] = {0.f, 0.f};
  for (int i = 0; wk.n > 0; ++i) {
    const int pair = wk.b * Hkv + wk.kvh;
    if (pair != cur_pair) {
      cur_pair = pair;
#pragma unroll
      for (int dt = 0; dt < NDT; ++dt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[dt][e] = 0.f;
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        mrun[r] = -INFINITY;
        lrun[r] = 0.f;
      }
    }
    const bool seg_end = (w1.n == 0) || (w1.b * Hkv + w1.kvh != pair);
    const int ng = wk.n;  // granules (groups) of the unit, all holding tokens

    const int hbi = i % kHandBufs;
    const uint8_t* hb = hand + (size_t)hbi * Gm::kHand;
    pipe_wait(&hfull[hbi], (i / kHandBufs) & 1, abort_flag);
    // ---- the unit's running maximum and the groups' factors ----
    static_assert(kQW % 4 == 0, "a row's group values are read as float4s");
    float fs[kQW][2];  // exp(m_g - m_new) * sW_g (INT8) or exp(m_g - m_new) (BF16)
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int row = 2 * t + r;
      // groups past the unit's tokens published m = -inf, l = 0, sW = 0
      float mg[kQW], lgv[kQW], sg[kQW];
#pragma unroll
      for (int j = 0; j < kQW / 4; ++j) {
        const float4 m4 = reinterpret_cast<const float4*>(hb + Gm::kHM)[row * (kQW / 4) + j];
        const float4 l4 = reinterpret_cast<const float4*>(hb + Gm::kHL)[row * (kQW / 4) + j];
        const float4 s4 = reinterpret_cast<const float4*>(hb + Gm::kHSw)[row * (kQW / 4) + j];
        mg[4 * j] = m4.x, mg[4 * j + 1] = m4.y, mg[4 * j + 2] = m4.z, mg[4 * j + 3] = m4.w;
        lgv[4 * j] = l4.x, lgv[4 * j + 1] = l4.y, lgv[4 * j + 2] = l4.z, lgv[4 * j + 3] = l4.w;
        sg[4 * j] = s4.x, sg[4 * j + 1] = s4.y, sg[4 * j + 2] = s4.z, sg[4 * j + 3] = s4.w;
      }
      float mn = mrun[r];
#pragma unroll
      for (int q = 0; q < kQW; ++q) mn = fmaxf(mn, mg[q]);
      const float alpha = (mrun[r] == -INFINITY) ? 0.f : ex2(mrun[r] - mn);
      float l = lrun[r] * alpha;
#pragma unroll
      for (int q = 0; q < kQW; ++q) {
        const float f = (mg[q] == -INFINITY) ? 0.f : ex2(mg[q] - mn);
        l = fmaf(lgv[q], f, l);
        fs[q][r] = BF16 ? f : f * sg[q];
      }
      lrun[r] = l;
      mrun[r] = mn;
      if (alpha != 1.f) {
#pragma unroll
        for (int dt = 0; dt < NDT; ++dt) {
          o[dt][r] *= alpha;
          o[dt][2 + r] *= alpha;
        }
      }
    }

    // ---- V item: this warp's head-dims, every group of the unit ----
    const int vslot = kStreams * rg.kK + vpos.s;
    pipe_wait(&full[vslot], vpos.use & 1, abort_flag);
    vpos.next(rg.nV);
    const uint8_t* vb = ring + (size_t)vslot * kSlot;
    if constexpr (!BF16) {
      // decode step: every PV warp patches its own head-dims of the new token's V column
      if (STEP && wk.gi + wk.n == wk.ngp) {
        const int pos = wk.L - 1 - wk.gi * kGran;
        for (int dd = lane; dd < Gm::kDimsPW; dd += 32) {
          const int d = pv_w * Gm::kDimsPW + dd;
          uint8_t* vp = ring + (size_t)vslot * kSlot;
          vp[(size_t)(pos / kBS) * kPage + (size_t)d * kBS + pos % kBS] = hb[Gm::kHPatch + d];
        }
        __syncwarp();
      }
    }
#pragma unroll
    for (int q = 0; q < kQW; ++q) {
      if (q >= ng) break;
      if constexpr (BF16) {
        // A = V^T of page q [D][16 tokens]: matrices (dims 0-7 | 8-15) x (tokens 0-7 | 8-15)
        const uint2 f = reinterpret_cast<const uint2*>(hb)[q * 32 + lane];
        const uint8_t* vrow = vb + (size_t)q * kPage + (size_t)(pv_w * Gm::kDimsPW) * 32 + (ri + 8 * (mi & 1)) * 32 +
                              (mi >> 1) * 16;
#pragma unroll
        for (int dt = 0; dt < NDT; ++dt) {
          uint32_t a[4];
          ldmatrix_x4(a, vrow + dt * 16 * 32);
          float pv[4] = {0.f, 0.f, 0.f, 0.f};
          mma_bf16_16816(pv, a, f.x, f.y);
          o[dt][0] = fmaf(pv[0], fs[q][0], o[dt][0]);
          o[dt][1] = fmaf(pv[1], fs[q][1], o[dt][1]);
          o[dt][2] = fmaf(pv[2], fs[q][0], o[dt][2]);
          o[dt][3] = fmaf(pv[3], fs[q][1], o[dt][3]);
        }
      } else {
        // PV on the INT8 tensor path (mma.sync m16n8k32, s8 x s8 -> s32: exact).
        // A = V^T of the group's pages 2q, 2q+1: ldmatrix of (dims 0-7 | 8-15) x
        // (page 2q | 2q+1) is the s8 A fragment (16 dims x 32 tokens) as it is.
        const uint2 f = reinterpret_cast<const uint2*>(hb)[q * 32 + lane];
        const uint8_t* vrow = vb + (size_t)(2 * q + (mi >> 1)) * kPage + (size_t)(pv_w * Gm::kDimsPW) * 16 +
                              (ri + 8 * (mi & 1)) * 16;
#pragma unroll
        for (int dt = 0; dt < NDT; ++dt) {
          uint32_t a[4];
          ldmatrix_x4(a, vrow + dt * 16 * 16);
          int pv[4] = {0, 0, 0, 0};
          if constexpr (U8P)
            mma_s8u8_16832(pv, a, f.x, f.y);
          else
            mma_s8_16832(pv, a, f.x, f.y);
          o[dt][0] = fmaf((float)pv[0], fs[q][0], o[dt][0]);  // |pv| <= 32 * 255 * 127 < 2^24: exact in fp32
          o[dt][1] = fmaf((float)pv[1], fs[q][1], o[dt][1]);
          o[dt][2] = fmaf((float)pv[2], fs[q][0], o[dt][2]);
          o[dt][3] = fmaf((float)pv[3], fs[q][1], o[dt][3]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[vslot]);

    // ---- end of this CTA's share of the (sequence, KV head) pair ----
    if (seg_end) {
      // The pair lies in this CTA's granule range [w0.gc, g_end) alone: the
      // merge kernel's test (first and last granule in one CTA), without its
      // divisions.
      const long long Up = wk.gb + (long long)wk.kvh * wk.ngp;  // the pair's first granule
      const int d0 = pv_w * Gm::kDimsPW;
      if (Up >= w0.gc && Up + wk.ngp - 1 < g_end) {
        const size_t dst = ((size_t)wk.b * Hq + wk.kvh * G) * D;
        const float inv0 = 1.0f / lrun[0], inv1 = 1.0f / lrun[1];
#pragma unroll
        for (int dt = 0; dt < NDT; ++dt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int row = 2 * t + (e & 1);
            if (row < G)
              store_out1(p.out, p.out_bf16, dst + (size_t)row * D + d0 + dt * 16 + g + 8 * (e >> 1),
                         o[dt][e] * ((e & 1) ? inv1 : inv0));
          }
      } else {
        // one partial per CTA; decode_merge_kernel combines them after this kernel
        float* part = p.ws_part + (size_t)(pair + c) * kSlotFloats(D);
#pragma unroll
        for (int dt = 0; dt < NDT; ++dt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int row = 2 * t + (e & 1);
            if (row < G) part[row * D + d0 + dt * 16 + g + 8 * (e >> 1)] = o[dt][e];
          }
        if (pv_w == 0 && g == 0) {
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            part[kRows * D + 2 * t + r] = mrun[r];
            part[kRows * D + kRows + 2 * t + r] = lrun[r];
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&hempty[hbi]);
    wk = w1;
    walk_next(w1, p.seq_lens, B, Hkv, maxL, kGran, g_end, Gm::kQW);
  }
}

// Log-sum-exp merge of the partials of pairs that span CTAs: two CTAs of 256
// threads per (pair, query row), each half of the row's columns (one CTA of
// 512 threads per row, or four of 128, were slower on single sequences).
// Thread (slice, column) owns every SL-th
// segment of one float4 column.  It loads a batch of kMB segments (value, m, l)
// at once -- independent loads, all in flight together -- then folds them into
// its running (max, denominator, sum); the slices are combined in a fixed order.
//
// Which CTAs hold the pair's partials follows from the attention kernel's work
// split, so warp 0 recomputes it from seq_lens (the same arithmetic) before the
// grid-dependency wait, while the attention kernel still runs.  A CTA whose pair
// has no partials exits there without waiting (in batched decode most do), but
// for the grid's first CTA; for the others the partials' loads go out at once
// after the wait.
constexpr int kMaxSeg = 1024;
constexpr int kMergeSplit = 2;    // CTAs per (pair, query row), each half of the row's columns
constexpr int kMergeThreads = 256;
constexpr int kMB = 8;
constexpr int kMergeSpreadSmem = 120 * 1024;  // more than half an SM's shared memory

// The first and last attention CTA of a (sequence, KV head) pair, from the
// attention kernel's work split recomputed from seq_lens by one warp (the same
// arithmetic; every lane gets the result); (-1, -1) for an empty sequence, which
// has zero rows and no partials.
template <int kGran>
__device__ __forceinline__ int2 pair_ctas(const DecodeParams& p, int pair, int lane) {
  const int Hkv = p.Hkv, maxL = p.max_blocks * kBS;
  const int bp = pair / Hkv, kvh = pair % Hkv;
  long long total = 0, before = 0;  // granules of all sequences; of the sequences before bp
  int Lp = 0;
  for (int b0 = 0; b0 < p.B; b0 += 32) {
    const int b = b0 + lane;
    int u = 0, L = 0;
    if (b < p.B) {
      L = clamp_len(__ldcg(p.seq_lens + b), maxL);
      u = (L + kGran - 1) / kGran * Hkv;
    }
    int su = u, sb = b < bp ? u : 0, lp = b == bp ? L : 0;
    for (int o = 16; o >= 1; o >>= 1) {
      su += __shfl_xor_sync(0xffffffffu, su, o);
      sb += __shfl_xor_sync(0xffffffffu, sb, o);
      lp += __shfl_xor_sync(0xffffffffu, lp, o);
    }
    total += su;
    before += sb;
    Lp += lp;
  }
  const int ngp = (Lp + kGran - 1) / kGran;
  if (ngp == 0) return make_int2(-1, -1);
  const long long U = total, Up = before + (long long)kvh * ngp;
  const int Nw = (int)(U < p.grid ? U : p.grid);
  return make_int2(cta_of(Up, U, Nw), cta_of(Up + ngp - 1, U, Nw));
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kMergeThreads) decode_merge_kernel(DecodeParams p) {
  constexpr int COLS = D / 4 / kMergeSplit, SL = kMergeThreads / COLS;
  constexpr int kGran = Geo<D, BF16>::kGran;
  __shared__ float4 red[SL][COLS];
  __shared__ float msh[SL], dsh[SL];
  __shared__ int s_seg[2];
  // The next kernel on the stream may start its launch (and its pre-wait
  // prologue) at once: its own grid-dependency wait still waits for this grid
  // to complete, which happens after the attention kernel (see below).
  // Single-sequence calls are 0.2 us shorter than when this signal followed
  // the wait.
  griddep_launch_dependents();
  const int tid = threadIdx.x;
  const int half = blockIdx.x % kMergeSplit, prw = blockIdx.x / kMergeSplit;
  const int pair = prw / p.G, row = prw % p.G;
  if (tid < 32) {
    const int2 cs = pair_ctas<kGran>(p, pair, tid);
    if (tid == 0) {
      s_seg[0] = cs.x;
      s_seg[1] = cs.y;
    }
  }
  __syncthreads();
  const int cf = s_seg[0], cl = s_seg[1], nseg = cl - cf + 1;
  // No partials (the attention kernel wrote the rows, or the sequence is
  // empty): nothing of the attention kernel's is read, so no wait for it --
  // except in the first CTA.  A kernel launched after this one waits for this
  // grid only, so this grid must not end before the attention kernel does.
  if (cf == cl && blockIdx.x != 0) return;
  griddep_wait();
  if (cf == cl) return;
  if (nseg > kMaxSeg) {
    record_error(2);
    return;
  }
  const int slice = tid / COLS, col = tid % COLS;
  const float* part0 = p.ws_part + (size_t)(pair + cf) * kSlotFloats(D);
  float m = -INFINITY, den = 0.f;
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = slice; s0 < nseg; s0 += SL * kMB) {
    float4 v[kMB];
    float ms[kMB], ls[kMB];
#pragma unroll
    for (int j = 0; j < kMB; ++j) {
      const int s = s0 + j * SL;
      if (s < nseg) {
        const float* ps = part0 + (size_t)s * kSlotFloats(D);
        v[j] = *reinterpret_cast<const float4*>(ps + row * D + 4 * (half * COLS + col));
        ms[j] = ps[kRows * D + row];
        ls[j] = ps[kRows * D + kRows + row];
      } else {
        v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        ms[j] = -INFINITY;
        ls[j] = 0.f;
      }
    }
    float mb = m;
#pragma unroll
    for (int j = 0; j < kMB; ++j) mb = fmaxf(mb, ms[j]);
    if (mb == -INFINITY) continue;
    const float f = ex2(m - mb);  // the partials' maxima are in log2 units
    a.x *= f;
    a.y *= f;
    a.z *= f;
    a.w *= f;
    den *= f;
#pragma unroll
    for (int j = 0; j < kMB; ++j) {
      const float e = ex2(ms[j] - mb);  // 0 for the padding entries
      a.x = fmaf(v[j].x, e, a.x);
      a.y = fmaf(v[j].y, e, a.y);
      a.z = fmaf(v[j].z, e, a.z);
      a.w = fmaf(v[j].w, e, a.w);
      den = fmaf(ls[j], e, den);
    }
    m = mb;
  }
  red[slice][col] = a;
  if (col == 0) {
    msh[slice] = m;
    dsh[slice] = den;
  }
  __syncthreads();
  if (tid < COLS) {
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < SL; ++k) M = fmaxf(M, msh[k]);
    float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
    float dd = 0.f;
#pragma unroll
    for (int k = 0; k < SL; ++k) {
      const float w = ex2(msh[k] - M);  // 0 for a slice without segments
      r.x = fmaf(red[k][tid].x, w, r.x);
      r.y = fmaf(red[k][tid].y, w, r.y);
      r.z = fmaf(red[k][tid].z, w, r.z);
      r.w = fmaf(red[k][tid].w, w, r.w);
      dd = fmaf(dsh[k], w, dd);
    }
    const float inv = 1.0f / dd;
    const int b = pair / p.Hkv, kvh = pair % p.Hkv;
    store_out4(p.out, p.out_bf16, ((size_t)b * p.Hq + kvh * p.G + row) * D + 4 * (half * COLS + tid),
               make_float4(r.x * inv, r.y * inv, r.z * inv, r.w * inv));
  }
}

// Batched decode: one warp per (pair, query row), kMergeWarpItems per CTA.
// With many pairs a pair spans few CTAs, so one warp folds its partials --
// lane l holds head-dims [l D/32, (l+1) D/32) -- in batches of kWB segments
// (value, m, l) whose loads are in flight together, with no block-level
// reduction.  The host takes this kernel when B * Hkv >= #SM / 4.
constexpr int kMergeWarpItems = 8;
template <int D, bool BF16>
__global__ void __launch_bounds__(kMergeWarpItems * 32) decode_merge_warp_kernel(DecodeParams p) {
  constexpr int kGran = Geo<D, BF16>::kGran, E = D / 32, kWB = 4;
  const int lane = threadIdx.x & 31;
  griddep_launch_dependents();  // as in decode_merge_kernel
  const int item = blockIdx.x * kMergeWarpItems + (threadIdx.x >> 5);
  if (item >= p.B * p.Hkv * p.G) return;
  const int pair = item / p.G, row = item % p.G;
  const int2 cs = pair_ctas<kGran>(p, pair, lane);
  // No partials: nothing of the attention kernel's is read, so no wait for it
  // -- except in the first item, so that this grid ends after the attention
  // kernel (a kernel launched after this one waits for this grid only).
  if (cs.x == cs.y && item != 0) return;
  const int nseg = cs.y - cs.x + 1;
  const size_t obase = ((size_t)(pair / p.Hkv) * p.Hq + (pair % p.Hkv) * p.G + row) * D + lane * E;
  griddep_wait();
  if (cs.x == cs.y) return;
  if (nseg > kMaxSeg) {
    if (lane == 0) record_error(2);
    return;
  }
  const float* part0 = p.ws_part + (size_t)(pair + cs.x) * kSlotFloats(D);
  float m = -INFINITY, den = 0.f, a[E];
#pragma unroll
  for (int e = 0; e < E; ++e) a[e] = 0.f;
  for (int s0 = 0; s0 < nseg; s0 += kWB) {
    float ms[kWB], ls[kWB];
    float4 v[kWB][E / 4];
#pragma unroll
    for (int j = 0; j < kWB; ++j) {
      const int sg = s0 + j;
      if (sg < nseg) {
        const float* ps = part0 + (size_t)sg * kSlotFloats(D);
        ms[j] = ps[kRows * D + row];
        ls[j] = ps[kRows * D + kRows + row];
#pragma unroll
        for (int k = 0; k < E / 4; ++k) v[j][k] = reinterpret_cast<const float4*>(ps + row * D + lane * E)[k];
      } else {
        ms[j] = -INFINITY;
        ls[j] = 0.f;
#pragma unroll
        for (int k = 0; k < E / 4; ++k) v[j][k] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    float mb = m;
#pragma unroll
    for (int j = 0; j < kWB; ++j) mb = fmaxf(mb, ms[j]);
    if (mb == -INFINITY) continue;
    const float f = ex2(m - mb);  // the partials' maxima are in log2 units
#pragma unroll
    for (int e = 0; e < E; ++e) a[e] *= f;
    den *= f;
#pragma unroll
    for (int j = 0; j < kWB; ++j) {
      const float w = ex2(ms[j] - mb);  // 0 for the padding entries
      den = fmaf(ls[j], w, den);
#pragma unroll
      for (int k = 0; k < E / 4; ++k) {
        a[4 * k] = fmaf(v[j][k].x, w, a[4 * k]);
        a[4 * k + 1] = fmaf(v[j][k].y, w, a[4 * k + 1]);
        a[4 * k + 2] = fmaf(v[j][k].z, w, a[4 * k + 2]);
        a[4 * k + 3] = fmaf(v[j][k].w, w, a[4 * k + 3]);
      }
    }
    m = mb;
  }
  const float inv = 1.0f / den;
#pragma unroll
  for (int k = 0; k < E / 4; ++k)
    store_out4(p.out, p.out_bf16, obase + 4 * k,
               make_float4(a[4 * k] * inv, a[4 * k + 1] * inv, a[4 * k + 2] * inv, a[4 * k + 3] * inv));
}

// Debug QK: one CTA per (sequence, KV head, 256-token partition); K pages are
// staged with plain 16-byte loads and the decode kernel's qk_warp computes the
// accumulators (exact integers in fp32), written as int32.
template <int D>
__global__ void __launch_bounds__(256) debug_qk_kernel(DebugQKParams p) {
  constexpr int kPage = D * kBS;
  extern __shared__ __align__(1024) uint8_t smem[];
  int8_t* kp = reinterpret_cast<int8_t*>(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nparts = (p.max_len + kPart - 1) / kPart;
  const int part = blockIdx.x % nparts;
  const int kvh = (blockIdx.x / nparts) % p.Hkv;
  const int b = blockIdx.x / nparts / p.Hkv;
  const int L = clamp_len(p.seq_lens[b], p.max_blocks * kBS);
  const int t0 = part * kPart;
  for (int i = tid; i < kPart / kBS * kPage / 16; i += blockDim.x) {
    const int jb = i / (kPage / 16), w16 = i % (kPage / 16);
    uint4 val = make_uint4(0, 0, 0, 0);
    if (t0 + jb * kBS < L) {
      const int blk = p.block_tables[(size_t)b * p.max_blocks + part * (kPart / kBS) + jb];
      if (blk >= 0 && blk < p.num_blocks)
        val = __ldg(reinterpret_cast<const uint4*>(p.k_cache + ((size_t)blk * p.Hkv + kvh) * kPage) + w16);
      else
        record_error(2);
    }
    reinterpret_cast<uint4*>(kp)[i] = val;
  }
  __syncthreads();
  uint32_t qf[D / 32][2];
  load_q_frags<D>(p.q, b, p.Hq, kvh, p.G, lane, qf);
  float acc[2][4];
  qk_warp<D>(kp, warp, lane, qf, acc);
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int m = 0; m < 2; ++m)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int tok = t0 + warp * kGroup + 16 * m + g + 8 * (e >> 1);
      const int row = 2 * t + (e & 1);
      if (row < p.G && tok < p.max_len)
        p.acc[((size_t)b * p.Hq + kvh * p.G + row) * p.max_len + tok] = tok < L ? __float2int_rn(acc[m][e]) : 0;
    }
}

int g_num_sms[64] = {0};

int num_sms(int device) {
  if (device < 0 || device >= 64) return 148;
  if (g_num_sms[device] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || n <= 0) n = 148;
    g_num_sms[device] = n;
  }
  return g_num_sms[device];
}

int g_max_smem[64] = {0};

int max_smem_optin(int device) {
  if (device < 0 || device >= 64) return 227 * 1024;
  if (g_max_smem[device] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) != cudaSuccess || n <= 0)
      n = 227 * 1024;
    g_max_smem[device] = n;
  }
  return g_max_smem[device];
}

// Deepest ring that fits (at least one K slot per stream and two V slots).
template <int D, bool BF16>
int pick_slots(int smem_limit) {
  for (int ns = 12; ns >= 4; ns -= 2)
    if (decode_layout<D, BF16>(ns).total <= (size_t)smem_limit) return ns;
  return 0;
}

template <int D, bool BF16, bool STEP, bool U8P = false>
cudaError_t launch_decode_d(const DecodeParams& p, cudaStream_t stream) {
  int dev = 0;
  cudaGetDevice(&dev);
  const int ns = pick_slots<D, BF16>(max_smem_optin(dev));
  if (ns == 0) return cudaErrorInvalidConfiguration;
  const size_t smem = decode_layout<D, BF16>(ns).total;
  // Raise the dynamic shared-memory limit once per device (to the opt-in
  // maximum), so that launches captured into a CUDA graph make no attribute call.
  static int attr_set[64] = {0};  // per instantiation
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, BF16, STEP, U8P>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         max_smem_optin(dev));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(decode_merge_kernel<D, BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMergeSpreadSmem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = 1;
  }
  cudaError_t e =
      launch_pdl(decode_kernel<D, BF16, STEP, U8P>, dim3(p.grid), dim3(Geo<D, BF16>::kThreads), smem, stream, p, ns);
  if (e != cudaSuccess) return e;
  // A merge grid that fits on the SMs (a few long sequences) gets one CTA per
  // SM, through an unused shared-memory request that two merge CTAs cannot
  // share: packed two to an SM, single-sequence calls took 0.4 us longer.
  // Larger grids (batched decode, where most CTAs exit at once) keep two per SM.
  const int mgrid = p.B * p.Hkv * p.G;
  if (4 * p.B * p.Hkv >= num_sms(dev))  // many pairs, each over few CTAs: one warp per row
    return launch_pdl(decode_merge_warp_kernel<D, BF16>, dim3((mgrid + kMergeWarpItems - 1) / kMergeWarpItems),
                      dim3(kMergeWarpItems * 32), 0, stream, p);
  return launch_pdl(decode_merge_kernel<D, BF16>, dim3(mgrid * kMergeSplit), dim3(kMergeThreads),
                    mgrid * kMergeSplit <= num_sms(dev) ? (size_t)kMergeSpreadSmem : 0, stream, p);
}

}  // namespace

I8KV_DEFINE_ERROR_ACCESSOR(read_error_decode)

int decode_grid(int device, int B, int Hkv, int max_blocks) {
  const long long max_units = (long long)B * Hkv * max_blocks;  // granules are at least one block
  long long g = num_sms(device);
  if (max_units < g) g = max_units;
  return (int)(g < 1 ? 1 : g);
}

size_t decode_workspace_bytes(int B, int Hkv, int D, int grid) {
  const size_t slots = (size_t)B * Hkv + (size_t)grid;
  size_t bytes = slots * kSlotFloats(D) * sizeof(float);
  return (bytes + 255) / 256 * 256;
}

cudaError_t launch_int8_decode(const DecodeParams& p, cudaStream_t stream) {
  if (p.step) {
    if (p.D == 256) return launch_decode_d<256, false, true>(p, stream);
    return launch_decode_d<128, false, true>(p, stream);
  }
  if (p.u8_probs) {
    if (p.D == 256) return launch_decode_d<256, false, false, true>(p, stream);
    return launch_decode_d<128, false, false, true>(p, stream);
  }
  if (p.D == 256) return launch_decode_d<256, false, false>(p, stream);
  return launch_decode_d<128, false, false>(p, stream);
}

cudaError_t launch_bf16_decode(const DecodeParams& p, cudaStream_t stream) {
  if (p.D == 256) return launch_decode_d<256, true, false>(p, stream);
  return launch_decode_d<128, true, false>(p, stream);
}

// ---------------------------------------------------------------------------
// Fixed scratch for the allocation-free decode entry point.  Some callers cannot
// call cudaMalloc when they run a decode step (for example a plugin inside
// another inference runtime whose memory planner owns every byte, or a server
// that reserves all device memory at start-up), so this file keeps one
// device-resident scratch area of kNoAllocScratchBytes.  Every GPU that loads
// the library holds it until the process exits.  In host code the array's name
// is only a host-side stand-in, so its device address is taken once per device
// with cudaGetSymbolAddress (with that device current) and passed to the kernel.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
// The array's device address belongs to the CUDA context that loaded this
// module: another context on the same device (a plugin's own context), or the
// new primary context after a device reset, has its own copy at another
// address.  So the address is cached per context, keyed by the context's
// unique id (cuCtxGetId; ids are never reused within a process).  The driver
// calls are reached through the runtime's entry-point lookup, so the library
// needs no link-time dependency on the driver library.
typedef int (*CtxGetCurrentFn)(void** ctx);
typedef int (*CtxGetIdFn)(void* ctx, unsigned long long* id);

struct NoAllocEntry {
  unsigned long long ctx_id;
  void* addr;
};
constexpr int kNoAllocContexts = 32;
std::mutex g_noalloc_mu;
NoAllocEntry g_noalloc_cache[kNoAllocContexts] = {};
int g_noalloc_next = 0;
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;
bool g_ctx_fns_looked_up = false;

// Id of the calling thread's current context; 0 when it cannot be told (then
// the address is looked up on every call).  Called with g_noalloc_mu held.
unsigned long long current_context_id() {
  if (!g_ctx_fns_looked_up) {
    g_ctx_fns_looked_up = true;
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(f);
  }
  if (!g_ctx_get_current || !g_ctx_get_id) return 0;
  void* ctx = nullptr;
  unsigned long long id = 0;
  if (g_ctx_get_current(&ctx) != 0 || ctx == nullptr) return 0;
  if (g_ctx_get_id(ctx, &id) != 0) return 0;
  return id;
}
}  // namespace

size_t noalloc_scratch_bytes() { return kNoAllocScratchBytes; }

cudaError_t noalloc_scratch_address(void** addr) {
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  unsigned long long id = current_context_id();
  if (id != 0) {
    for (const NoAllocEntry& en : g_noalloc_cache)
      if (en.ctx_id == id) {
        *addr = en.addr;
        return cudaSuccess;
      }
  }
  // Not cached for this context (or no context is current yet: the runtime
  // then makes the device's primary context current here).
  void* ptr = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
  if (e != cudaSuccess) return e;
  if (id == 0) id = current_context_id();
  if (id != 0) {
    g_noalloc_cache[g_noalloc_next] = NoAllocEntry{id, ptr};
    g_noalloc_next = (g_noalloc_next + 1) % kNoAllocContexts;
  }
  *addr = ptr;
  return cudaSuccess;
}

cudaError_t launch_debug_qk(const DebugQKParams& p, cudaStream_t stream) {
  const int nparts = (p.max_len + kPart - 1) / kPart;
  const long long grid = (long long)p.B * p.Hkv * nparts;
  if (grid == 0) return cudaSuccess;
  const size_t smem = (size_t)kPart * p.D;
  cudaError_t e;
  if (p.D == 256) {
    e = cudaFuncSetAttribute(debug_qk_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    debug_qk_kernel<256><<<(unsigned)grid, 256, smem, stream>>>(p);
  } else {
    e = cudaFuncSetAttribute(debug_qk_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    debug_qk_kernel<128><<<(unsigned)grid, 256, smem, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace i8kv
