// decode.cu -- INT8 paged decode attention (and the debug QK path).
//
// Source: "gfx936 DCU上实现INT8 PV MMAC：V Scale融合、概率量化与Fragment分组"
// §1 (W = P x sV, 32-token groups, sW = max W / 127), §2 (score recovery
// acc x sQ x sK / sqrt(d), online softmax), §2.2 (decode: 256-token partitions
// merged by log-sum-exp), §3 (P on the A side, V on the B side of the INT8
// MMA; int32 bound 32 x 127 x 127 per group) and "gfx936 DCU上实现INT8 KV与
// INT8 MMAC Attention推理优化" §3.3 (the decode data flow) and §2.3 (layouts).
//
// GB300 design (not the pages' gfx936 one):
//  * Work unit = (sequence, KV head, 256-token partition).  A persistent grid of
//    one CTA per SM takes a contiguous range of units; pairs (sequence, KV head)
//    that span CTAs leave one partial per CTA in the workspace and the last CTA
//    to finish a pair (an atomic ticket, no waiting) merges them by
//    log-sum-exp.
//  * Warp 8 is a TMA producer: per unit it issues 16 bulk copies of K pages (one
//    ring item) and 16 of V pages (a second item) into a ring of shared-memory
//    slots guarded by full/empty mbarriers.
//  * Warps 0-7 consume, each on its own 32-token group of every partition
//    (warp w: tokens 32w .. 32w+31), with no CTA barrier per partition: every
//    warp runs its own online softmax (m, l, o) over its groups.  The pages
//    normalize P inside a 256-token partition before quantizing W; here the
//    normalization of each group is carried in the running state instead.  The
//    group quantization Wq = round(W / (max W / 127)) does not change when all
//    W of a group are scaled by one positive factor, so the codes are the
//    pages' codes and the output is the same up to fp32 rounding.  At the end of
//    a CTA's share of a pair the 8 warps' states merge deterministically
//    (log-sum-exp, tree order) through shared memory.
//  * GQA packs the G <= 8 query heads of one KV head into the N = 8 side of the
//    MMAs.  QK: M = 16 tokens (one block), K = head-dims.  PV: M = 16 head-dims,
//    N = 8 query rows, K = the tokens of one probability group, so each group's
//    contraction is one accumulator and its sW scales exactly that result.
//  * The INT8 x INT8 contractions run on the f16 tensor path: every int8 code is
//    exact in f16, every product (<= 127^2) is exact, and every partial sum is
//    an integer below 2^22 (QK over 256 dims: <= 4,129,024; PV over one group:
//    <= 516,128), so the fp32 accumulator holds the exact int32 result.  On
//    sm_103a this path has about 4x the throughput of mma.sync s8; the debug QK
//    entry point checks the accumulators bit for bit against integer QK.
#include <cuda_bf16.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace i8kv {

namespace {

constexpr int kPart = 256;   // partition (tokens) -- the pages' decode partition
constexpr int kBS = 16;      // block size
constexpr int kGroup = 32;   // probability group
constexpr int kCWarps = 8;   // consumer warps (one per group of a partition)
constexpr int kThreads = (kCWarps + 1) * 32;
constexpr int kRows = 8;     // query rows in the MMA N dimension
__host__ __device__ constexpr int kSlotFloats(int D) { return kRows * D + 2 * kRows; }

struct SmemLayout {
  int nslots;
  size_t ring, merge, wq, bars, ctrl, total;
};

__host__ __device__ inline SmemLayout decode_layout(int D, int nslots) {
  SmemLayout L;
  L.nslots = nslots;
  const size_t item = (size_t)kPart * D;
  size_t off = 0;
  L.ring = off;
  off += (size_t)nslots * item;
  L.merge = off;  // 4 warp states [8 rows][D + 4] + l [8] (+ maxima [8 warps][8 rows])
  off += (size_t)(4 * (kRows * (D + 4) + 2 * kRows) + kCWarps * kRows) * sizeof(float);
  L.wq = off;     // per-warp transpose of the quantized W: [8 rows][32 tokens] int8
  off += (size_t)kCWarps * kRows * kGroup;
  L.bars = off;
  off += (size_t)2 * nslots * sizeof(uint64_t);
  L.ctrl = off;
  off += 16 * sizeof(int);
  L.total = off;
  return L;
}

// Position in the (sequence, KV head, partition) unit order.
struct Walk {
  int b, kvh, part, L, np;
  long long ub;  // global index of the first unit of sequence b
};

__device__ __forceinline__ int clamp_len(int L, int maxL) {
  if (L < 0) return 0;
  return L > maxL ? maxL : L;
}

__device__ __forceinline__ void walk_next(Walk& w, const int32_t* seq_lens, int B, int Hkv, int maxL, int unit) {
  if (++w.part < w.np) return;
  w.part = 0;
  if (++w.kvh < Hkv) return;
  w.kvh = 0;
  w.ub += (long long)w.np * Hkv;
  for (;;) {
    if (++w.b >= B) return;
    w.L = clamp_len(seq_lens[w.b], maxL);
    w.np = (w.L + unit - 1) / unit;
    if (w.np > 0) return;
  }
}

// CTA whose unit range [c*U/N, (c+1)*U/N) holds unit u (N <= U: no empty ranges).
__device__ __forceinline__ int cta_of(long long u, long long U, int N) {
  return (int)(((u + 1) * N + U - 1) / U - 1);
}

// Bounded pipeline wait.  After a timeout (error 1) or once the CTA aborted,
// it returns without waiting so every thread still reaches the same barriers.
__device__ __forceinline__ void pipe_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return;
  if (*abort_flag) return;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort_flag) return;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      record_error(1);
      *abort_flag = 1;
      return;
    }
  }
}

// Query fragments (B operand of QK, f16 form) of the GQA-packed rows: column g of
// the N-tile is query head kvh*G + g; per 32-dim step s the s8 fragment holds
// dims 32s + {4t..4t+3} and 32s + 16 + {4t..4t+3}.
template <int D>
__device__ __forceinline__ void load_q_frags(const int8_t* q, int b, int Hq, int kvh, int G, int lane,
                                             uint32_t (&qf)[D / 32][4]) {
  const int g = lane >> 2, t = lane & 3;
  const int8_t* row = q + ((size_t)b * Hq + kvh * G + g) * D;
#pragma unroll
  for (int s = 0; s < D / 32; ++s) {
    const uint32_t x0 = g < G ? __ldg(reinterpret_cast<const uint32_t*>(row + 32 * s + 4 * t)) : 0u;
    const uint32_t x1 = g < G ? __ldg(reinterpret_cast<const uint32_t*>(row + 32 * s + 16 + 4 * t)) : 0u;
    s8b_to_f16(x0, x1, qf[s]);
  }
}

// QK for the two 16-token blocks (2w, 2w+1) of warp w's group:
// acc[m][0..3] = (token g, row 2t), (token g, row 2t+1), (token g+8, row 2t),
// (token g+8, row 2t+1) of block 2w+m.  kpages holds 16 K pages [D/16][16][16 B].
template <int D>
__device__ __forceinline__ void qk_warp(const int8_t* kpages, int warp, int lane, const uint32_t (&qf)[D / 32][4],
                                        float (&acc)[2][4]) {
  const int mi = lane >> 3, ri = lane & 7;
  // Even and odd 32-dim steps accumulate separately (two independent MMA chains
  // per block instead of one); the two partial sums are exact integers, so
  // adding them at the end changes nothing.
  float acc2[2][4];
#pragma unroll
  for (int m = 0; m < 2; ++m)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[m][i] = acc2[m][i] = 0.f;
#pragma unroll
  for (int s = 0; s < D / 32; ++s) {
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      const int8_t* row =
          kpages + (size_t)(2 * warp + m) * (D * kBS) + (mi >> 1) * (kBS * 16) + (ri + 8 * (mi & 1)) * 16;
      uint32_t a[4];
      ldmatrix_x4(a, row + (size_t)(2 * s) * (kBS * 16));
      mma_s8a_f16b((s & 1) ? acc2[m] : acc[m], a, qf[s]);
    }
  }
#pragma unroll
  for (int m = 0; m < 2; ++m)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[m][i] += acc2[m][i];
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

// One kernel body for both caches.  BF16 = false: the INT8 method.  BF16 = true:
// the BF16-KV comparison (plain softmax, bf16 P x V, no scales), with 128-token
// units so that a ring item (8 bf16 pages) has the same 64 KB at D = 256.
template <int D, bool BF16>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(DecodeParams p, int nslots) {
  constexpr int NDT = D / 16;  // PV head-dim tiles (every warp covers all of D for its group)
  constexpr int EB = BF16 ? 2 : 1;              // bytes per cache element
  constexpr int kUnit = BF16 ? 128 : kPart;     // tokens per work unit
  constexpr int kBlocksU = kUnit / kBS;         // pages per ring item
  constexpr int kWTok = kUnit / kCWarps;        // tokens per warp per unit (32 = one probability group)
  constexpr int MT = kWTok / 16;                // 16-token blocks per warp per unit
  constexpr int kPage = D * kBS * EB;
  constexpr int kItem = kBlocksU * kPage;
  constexpr int kRS = D + 4;                   // row stride of a warp state (conflict-free stores)
  constexpr int kWS = kRows * kRS + 2 * kRows;  // one warp state in the merge buffer
  extern __shared__ __align__(1024) uint8_t smem[];
  const SmemLayout lay = decode_layout(D, nslots);
  int8_t* ring = reinterpret_cast<int8_t*>(smem + lay.ring);
  float* mbuf = reinterpret_cast<float*>(smem + lay.merge);
  int8_t* wqs = reinterpret_cast<int8_t*>(smem + lay.wq);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + lay.bars);
  uint64_t* empty = full + nslots;
  int* ctrl = reinterpret_cast<int*>(smem + lay.ctrl);
  volatile int* abort_flag = ctrl + 8;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int B = p.B, Hkv = p.Hkv, G = p.G, Hq = p.Hq;
  const int N = gridDim.x, c = blockIdx.x;
  const int maxL = p.max_blocks * kBS;

  if (warp == kCWarps && lane == 0) {
    for (int s = 0; s < nslots; ++s) {
      mbar_init(&full[s], 32);
      mbar_init(&empty[s], kCWarps);
    }
    fence_mbar_init();
  }
  // Everything above touches only shared memory; from here on the kernel reads
  // what earlier work on the stream wrote.
  griddep_wait();
  griddep_launch_dependents();

  // ---- work split, by the producer warp (the consumers wait at the barrier
  // below; they have nothing to do before it) ----
  // One sequence in the batch (the long-context decode case): guess the first
  // unit from max_blocks and load its block-table row together with seq_lens,
  // so the two dependent loads overlap; the guess is checked below.
  int spec_part = -1, spec_blk = -1;
  if (warp == kCWarps && B == 1) {
    const int np_g = (maxL + kUnit - 1) / kUnit;
    const long long U_g = (long long)np_g * Hkv;
    const int Nw_g = (int)(U_g < N ? U_g : N);
    if (c < Nw_g) {
      spec_part = (int)((U_g * c / Nw_g) % np_g);
      if (lane < kBlocksU && spec_part * kBlocksU + lane < p.max_blocks)
        spec_blk = __ldg(p.block_tables + spec_part * kBlocksU + lane);
    }
  }
  if (warp == kCWarps) {
    constexpr int kKeep = 8;  // chunks of 32 sequences whose unit counts stay in registers
    int ukeep[kKeep];
    long long total = 0;
    for (int b0 = 0, ck = 0; b0 < B; b0 += 32, ++ck) {
      const int b = b0 + lane;
      int u = 0;
      if (b < B) {
        const int raw = p.seq_lens[b];
        if (raw > maxL) record_error(2);
        const int L = clamp_len(raw, maxL);
        u = (L + kUnit - 1) / kUnit * Hkv;
        if (L == 0 && b % N == c) {  // empty sequence: zero rows, nothing to merge
          float* o = p.out + (size_t)b * Hq * D;
          for (int i = 0; i < Hq * D; ++i) o[i] = 0.f;
          for (int h = 0; h < Hkv; ++h) p.ws_info[b * Hkv + h] = -1;
        }
      }
#pragma unroll
      for (int k = 0; k < kKeep; ++k)
        if (k == ck) ukeep[k] = u;
      int su = u;
      for (int o = 16; o >= 1; o >>= 1) su += __shfl_xor_sync(0xffffffffu, su, o);
      total += su;
    }
    const long long U = total;
    // Only the first min(N, U) CTAs take units, so every working CTA has at
    // least one and the CTAs covering a pair are consecutive.
    const int Nw = (int)(U < N ? U : N);
    const long long ub = c < Nw ? U * c / Nw : 0, ue = c < Nw ? U * (c + 1) / Nw : 0;
    if (lane == 0) {
      ctrl[0] = (int)(ue - ub);
      ctrl[8] = 0;
      ctrl[10] = Nw;
      ctrl[6] = (int)(U & 0x7fffffff);
      ctrl[7] = (int)(U >> 31);
    }
    if (ue > ub) {
      long long run = 0;
      for (int b0 = 0, ck = 0; b0 < B; b0 += 32, ++ck) {
        const int b = b0 + lane;
        int u = 0;
        if (ck < kKeep) {
#pragma unroll
          for (int k = 0; k < kKeep; ++k)
            if (k == ck) u = ukeep[k];
        } else if (b < B) {
          u = (clamp_len(p.seq_lens[b], maxL) + kUnit - 1) / kUnit * Hkv;
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
            const int np = u / Hkv;
            const long long local = ub - ex;
            ctrl[1] = b;
            ctrl[2] = (int)(local / np);
            ctrl[3] = (int)(local % np);
            ctrl[4] = (int)(ex & 0x7fffffff);
            ctrl[5] = (int)(ex >> 31);
          }
          break;
        }
        run += __shfl_sync(0xffffffffu, incl, 31);
      }
    }
  }
  __syncthreads();  // the split in ctrl[] is visible to every warp
  const int n_units = ctrl[0];
  if (n_units <= 0) return;
  Walk w0;
  w0.b = ctrl[1];
  w0.kvh = ctrl[2];
  w0.part = ctrl[3];
  w0.ub = (long long)ctrl[4] | ((long long)ctrl[5] << 31);
  w0.L = clamp_len(p.seq_lens[w0.b], maxL);
  w0.np = (w0.L + kUnit - 1) / kUnit;
  const long long U = (long long)ctrl[6] | ((long long)ctrl[7] << 31);
  const int Nw = ctrl[10];

  if (warp == kCWarps) {
    // ================= producer warp =================
    const uint8_t* kc = static_cast<const uint8_t*>(p.k_cache);
    const uint8_t* vc = static_cast<const uint8_t*>(p.v_cache);
    const uint64_t pol = policy_evict_first();
    Walk wk = w0;
    for (int i = 0; i < n_units; ++i) {
      const int t0 = wk.part * kUnit;
      const int nblk = min(kBlocksU, (wk.L - t0 + kBS - 1) / kBS);
      int blk = -1;
      if (lane < nblk) {
        blk = (i == 0 && B == 1 && wk.part == spec_part)
                  ? spec_blk
                  : p.block_tables[(size_t)wk.b * p.max_blocks + wk.part * kBlocksU + lane];
        if (blk < 0 || blk >= p.num_blocks) {
          record_error(2);
          blk = -1;
        }
      }
      const bool ok = lane < kBlocksU && blk >= 0;
      const uint32_t n_pages = __popc(__ballot_sync(0xffffffffu, ok));
#pragma unroll
      for (int kv = 0; kv < 2; ++kv) {
        const int item = 2 * i + kv, slot = item % nslots;
        if (item >= nslots) pipe_wait(&empty[slot], ((item / nslots) - 1) & 1, abort_flag);
        if (lane == 0) mbar_expect_tx(&full[slot], n_pages * kPage);
        __syncwarp();
        if (ok)
          bulk_g2s_hint(ring + (size_t)slot * kItem + (size_t)lane * kPage,
                        (kv == 0 ? kc : vc) + ((size_t)blk * Hkv + wk.kvh) * kPage, kPage, &full[slot], pol);
        mbar_arrive(&full[slot]);
      }
      walk_next(wk, p.seq_lens, B, Hkv, maxL, kUnit);
    }
    return;
  }

  // ================= consumer warps =================
  const int g = lane >> 2, t = lane & 3;
  const float c_scale = p.sm_scale;
  int8_t* wqw = wqs + warp * (kRows * kGroup);
  Walk wk = w0;
  int cur_pair = -1;
  uint32_t qf[D / 32][4];    // INT8: converted query fragments
  uint32_t qfb[D / 16][2];   // BF16: query fragments
  float sq[2] = {0.f, 0.f};
  float o[NDT][4];
  float mrun[2] = {-INFINITY, -INFINITY}, lrun[2] = {0.f, 0.f};
  // this thread's scales for tokens {g, g+8} of blocks 2w and 2w+1 of a unit
  float sk[4], sv[4], sk_n[4], sv_n[4];
  auto load_scales = [&](const Walk& u, float (&k4)[4], float (&v4)[4]) {
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      const int lb = u.part * kBlocksU + 2 * warp + m;  // logical block in the sequence
      const int tok0 = lb * kBS;
      int blk = -1;
      if (tok0 < u.L) {
        blk = __ldg(p.block_tables + (size_t)u.b * p.max_blocks + lb);
        if (blk < 0 || blk >= p.num_blocks) blk = -1;
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int off = g + 8 * h;
        const bool v = blk >= 0 && tok0 + off < u.L;
        const size_t si = ((size_t)(v ? blk : 0) * kBS + off) * Hkv + u.kvh;
        k4[2 * m + h] = v ? __ldg(p.k_scale + si) : 0.f;
        v4[2 * m + h] = v ? __ldg(p.v_scale + si) : 0.f;
      }
    }
  };
  if constexpr (!BF16) load_scales(wk, sk, sv);
  for (int i = 0; i < n_units; ++i) {
    const int pair = wk.b * Hkv + wk.kvh;
    if (pair != cur_pair) {
      cur_pair = pair;
      if constexpr (BF16) {
        load_q_frags_bf16<D>(static_cast<const uint16_t*>(p.q), wk.b, Hq, wk.kvh, G, lane, qfb);
      } else {
        load_q_frags<D>(static_cast<const int8_t*>(p.q), wk.b, Hq, wk.kvh, G, lane, qf);
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int row = 2 * t + r;
        if constexpr (!BF16) sq[r] = row < G ? p.q_scale[(size_t)wk.b * Hq + wk.kvh * G + row] : 0.f;
        mrun[r] = -INFINITY;
        lrun[r] = 0.f;
      }
#pragma unroll
      for (int dt = 0; dt < NDT; ++dt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[dt][e] = 0.f;
    }
    Walk nx = wk;
    walk_next(nx, p.seq_lens, B, Hkv, maxL, kUnit);
    if constexpr (!BF16)
      if (i + 1 < n_units) load_scales(nx, sk_n, sv_n);  // the next unit's scales, in flight meanwhile
    const int t0 = wk.part * kUnit;
    const int ntok = min(kUnit, wk.L - t0);
    const bool active = warp * kWTok < ntok;

    // ---- K item: QK for this warp's group ----
    const int kitem = 2 * i, kslot = kitem % nslots;
    pipe_wait(&full[kslot], (kitem / nslots) & 1, abort_flag);
    float acc[2][4];
    if (active) {
      if constexpr (BF16)
        qk_warp_bf16<D>(reinterpret_cast<const uint8_t*>(ring) + (size_t)kslot * kItem, warp, lane, qfb, acc[0]);
      else
        qk_warp<D>(ring + (size_t)kslot * kItem, warp, lane, qf, acc);
    } else {
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[m][e] = 0.f;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[kslot]);

    // ---- scores, online softmax over this warp's group, W = p~ * sV, quantize ----
    float alpha[2] = {1.f, 1.f}, sw[2] = {0.f, 0.f};
    if (active) {
      float s[2][4];
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int tok = warp * kWTok + 16 * m + g + 8 * (e >> 1);
          float sc = -INFINITY;
          if (tok < ntok) {
            if constexpr (BF16)
              sc = __fmul_rn(acc[m][e], c_scale);
            else
              sc = __fmul_rn(__fmul_rn(__fmul_rn(acc[m][e], sq[e & 1]), sk[2 * m + (e >> 1)]), c_scale);
          }
          s[m][e] = sc;
          mx[e & 1] = fmaxf(mx[e & 1], sc);
        }
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int off = 4; off <= 16; off <<= 1) mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], off));
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const float mn = fmaxf(mrun[r], mx[r]);
        alpha[r] = (mrun[r] == -INFINITY) ? 0.f : expf(mrun[r] - mn);
        mrun[r] = mn;
        lrun[r] *= alpha[r];
      }
      if constexpr (BF16) {
        // plain softmax weights p~ in bf16 -> this warp's [row][16 tokens] staging
        uint16_t* pw = reinterpret_cast<uint16_t*>(wqw);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float pe = (s[0][e] == -INFINITY) ? 0.f : expf(__fsub_rn(s[0][e], mrun[e & 1]));
          lrun[e & 1] += pe;
          pw[(2 * t + (e & 1)) * 16 + g + 8 * (e >> 1)] = __bfloat16_as_ushort(__float2bfloat16_rn(pe));
        }
      } else {
        float A[2] = {0.f, 0.f}, w[2][4];
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float pe = (s[m][e] == -INFINITY) ? 0.f : expf(__fsub_rn(s[m][e], mrun[e & 1]));
            lrun[e & 1] += pe;
            w[m][e] = __fmul_rn(pe, sv[2 * m + (e >> 1)]);
            A[e & 1] = fmaxf(A[e & 1], w[m][e]);
          }
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
          for (int off = 4; off <= 16; off <<= 1) A[r] = fmaxf(A[r], __shfl_xor_sync(0xffffffffu, A[r], off));
        float inv[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          sw[r] = __fdiv_rn(A[r], 127.0f);
          inv[r] = A[r] > 0.f ? __fdiv_rn(127.0f, A[r]) : 0.f;
        }
        // codes -> this warp's [row][token] bytes, read back below as PV B fragments
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int q = min(127, __float2int_rn(w[m][e] * inv[e & 1]));
            wqw[(2 * t + (e & 1)) * kGroup + 16 * m + g + 8 * (e >> 1)] = (int8_t)q;
          }
      }
    }
    __syncwarp();
    uint32_t bq[4];
    if constexpr (BF16) {
      bq[0] = *reinterpret_cast<const uint32_t*>(wqw + g * 32 + 4 * t);
      bq[1] = *reinterpret_cast<const uint32_t*>(wqw + g * 32 + 16 + 4 * t);
    } else {
      s8b_to_f16(*reinterpret_cast<const uint32_t*>(wqw + g * kGroup + 4 * t),
                 *reinterpret_cast<const uint32_t*>(wqw + g * kGroup + 16 + 4 * t), bq);
    }
    if (alpha[0] != 1.f || alpha[1] != 1.f) {
#pragma unroll
      for (int dt = 0; dt < NDT; ++dt) {
        o[dt][0] *= alpha[0];
        o[dt][1] *= alpha[1];
        o[dt][2] *= alpha[0];
        o[dt][3] *= alpha[1];
      }
    }

    // ---- V item: exact INT8 PV of this warp's group, scaled by sW ----
    const int vitem = 2 * i + 1, vslot = vitem % nslots;
    pipe_wait(&full[vslot], (vitem / nslots) & 1, abort_flag);
    if (active) {
      const int mi = lane >> 3, ri = lane & 7;
      if constexpr (BF16) {
        // A = V^T from the warp's bf16 page [D][16 tokens]: matrices (dims 0-7 | 8-15) x (tokens 0-7 | 8-15)
        const uint8_t* vrow = reinterpret_cast<const uint8_t*>(ring) + (size_t)vslot * kItem + (size_t)warp * kPage +
                              (ri + 8 * (mi & 1)) * 32 + (mi >> 1) * 16;
#pragma unroll
        for (int dt = 0; dt < NDT; ++dt) {
          uint32_t a[4];
          ldmatrix_x4(a, vrow + dt * 16 * 32);
          mma_bf16_16816(o[dt], a, bq[0], bq[1]);
        }
      } else {
        const int8_t* vrow =
            ring + (size_t)vslot * kItem + (size_t)(2 * warp + (mi >> 1)) * kPage + (ri + 8 * (mi & 1)) * 16;
#pragma unroll
        for (int dt = 0; dt < NDT; ++dt) {
          uint32_t a[4];
          ldmatrix_x4(a, vrow + dt * 16 * 16);
          float pv[4] = {0.f, 0.f, 0.f, 0.f};
          mma_s8a_f16b(pv, a, bq);
          o[dt][0] = fmaf(pv[0], sw[0], o[dt][0]);
          o[dt][1] = fmaf(pv[1], sw[1], o[dt][1]);
          o[dt][2] = fmaf(pv[2], sw[0], o[dt][2]);
          o[dt][3] = fmaf(pv[3], sw[1], o[dt][3]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[vslot]);

    // ---- end of this CTA's share of the (sequence, KV head) pair? ----
    const bool seg_end = (i == n_units - 1) || (nx.b * Hkv + nx.kvh != pair);
    if (seg_end) {
      // full row sums of this warp (the 8 threads with one t hold one row's tokens)
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int off = 4; off <= 16; off <<= 1) lrun[r] += __shfl_xor_sync(0xffffffffu, lrun[r], off);
      // common max over the 8 warps, then a tree sum in a fixed order
      float* mw = mbuf + 4 * kWS;  // [8 warps][8 rows] maxima
      if (g == 0) {
        mw[warp * kRows + 2 * t] = mrun[0];
        mw[warp * kRows + 2 * t + 1] = mrun[1];
      }
      named_bar_sync(1, kCWarps * 32);
      float M[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        float mm = -INFINITY;
#pragma unroll
        for (int w2 = 0; w2 < kCWarps; ++w2) mm = fmaxf(mm, mw[w2 * kRows + 2 * t + r]);
        M[r] = mm;
        const float f = (mrun[r] == -INFINITY) ? 0.f : expf(mrun[r] - mm);
        lrun[r] *= f;
#pragma unroll
        for (int dt = 0; dt < NDT; ++dt) {
          o[dt][r] *= f;
          o[dt][2 + r] *= f;
        }
      }
      // Two rounds (warps 0-3, then 4-7) through 4 shared buffers; each thread
      // then owns one row and D/32 head-dims of the CTA's state and adds the
      // 8 warps' values in warp order (deterministic).
      constexpr int DPT = D / 32;
      const int orow = tid >> 5;  // 0..7
      float Mrow = -INFINITY;  // read before the rounds' barriers, so a later segment cannot overwrite it first
#pragma unroll
      for (int w2 = 0; w2 < kCWarps; ++w2) Mrow = fmaxf(Mrow, mw[w2 * kRows + orow]);
      float acc_o[DPT];
      float acc_l = 0.f;
#pragma unroll
      for (int k = 0; k < DPT; ++k) acc_o[k] = 0.f;
#pragma unroll
      for (int round = 0; round < 2; ++round) {
        if ((warp >> 2) == round) {
          float* buf = mbuf + (size_t)(warp & 3) * kWS;
#pragma unroll
          for (int dt = 0; dt < NDT; ++dt)
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (2 * t + (e & 1) < G) buf[(2 * t + (e & 1)) * kRS + dt * 16 + g + 8 * (e >> 1)] = o[dt][e];
          if (g == 0) {
            buf[kRows * kRS + 2 * t] = lrun[0];
            buf[kRows * kRS + 2 * t + 1] = lrun[1];
          }
        }
        named_bar_sync(1, kCWarps * 32);
        if (orow < G) {
#pragma unroll
          for (int wb = 0; wb < 4; ++wb) {
            const float* buf = mbuf + (size_t)wb * kWS;
#pragma unroll
            for (int k = 0; k < DPT; ++k) acc_o[k] += buf[orow * kRS + lane + 32 * k];
            acc_l += buf[kRows * kRS + orow];
          }
        }
        named_bar_sync(1, kCWarps * 32);
      }
      (void)M;
      const long long Up = wk.ub + (long long)wk.kvh * wk.np;
      const int cf = cta_of(Up, U, Nw), cl = cta_of(Up + wk.np - 1, U, Nw);
      // the CTA holding the pair's first unit records whether a merge is needed
      if (c == cf && tid == 0) p.ws_info[pair] = (cf == cl) ? -1 : ((cf << 16) | cl);
      if (cf == cl) {
        if (orow < G) {
          float* dst = p.out + ((size_t)wk.b * Hq + wk.kvh * G + orow) * D;
          const float inv = 1.0f / acc_l;
#pragma unroll
          for (int k = 0; k < DPT; ++k) dst[lane + 32 * k] = acc_o[k] * inv;
        }
      } else {
        // one partial per CTA; decode_merge_kernel combines them after this kernel
        float* part = p.ws_part + (size_t)(pair + c) * kSlotFloats(D);
        if (orow < G) {
#pragma unroll
          for (int k = 0; k < DPT; ++k) part[orow * D + lane + 32 * k] = acc_o[k];
        }
        if (lane == 0) {
          part[kRows * D + orow] = Mrow;
          part[kRows * D + kRows + orow] = acc_l;
        }
      }
    }
    wk = nx;
    if constexpr (!BF16) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        sk[k] = sk_n[k];
        sv[k] = sv_n[k];
      }
    }
  }
}

// Log-sum-exp merge of the partials of pairs that span CTAs: one CTA per
// (pair, query row).  Thread (slice, column) sums every SL-th segment of one
// float4 column; the slices are then added in a fixed order.
constexpr int kMaxSeg = 1024;

template <int D>
__global__ void __launch_bounds__(256) decode_merge_kernel(DecodeParams p) {
  constexpr int COLS = D / 4, SL = 256 / COLS;
  __shared__ float wsh[kMaxSeg], lsh[kMaxSeg];
  __shared__ float4 red[SL][COLS];
  __shared__ float Msh, den;
  griddep_wait();
  griddep_launch_dependents();
  const int tid = threadIdx.x;
  const int pair = blockIdx.x / p.G, row = blockIdx.x % p.G;
  const int info = p.ws_info[pair];
  if (info < 0) return;
  const int cf = info >> 16, cl = info & 0xffff, nseg = cl - cf + 1;
  if (nseg > kMaxSeg) {
    record_error(2);
    return;
  }
  const float* part0 = p.ws_part + (size_t)(pair + cf) * kSlotFloats(D);
  for (int s = tid; s < nseg; s += 256) {
    wsh[s] = part0[(size_t)s * kSlotFloats(D) + kRows * D + row];
    lsh[s] = part0[(size_t)s * kSlotFloats(D) + kRows * D + kRows + row];
  }
  __syncthreads();
  if (tid < 32) {
    float m = -INFINITY;
    for (int s = tid; s < nseg; s += 32) m = fmaxf(m, wsh[s]);
    for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if (tid == 0) Msh = m;
  }
  __syncthreads();
  for (int s = tid; s < nseg; s += 256) wsh[s] = expf(wsh[s] - Msh);
  __syncthreads();
  if (tid < 32) {
    float dd = 0.f;
    for (int s = tid; s < nseg; s += 32) dd += wsh[s] * lsh[s];
    for (int off = 16; off >= 1; off >>= 1) dd += __shfl_xor_sync(0xffffffffu, dd, off);
    if (tid == 0) den = dd;
  }
  const int slice = tid / COLS, col = tid % COLS;
  const float4* base = reinterpret_cast<const float4*>(part0 + row * D) + col;
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
  for (int s = slice; s < nseg; s += SL) {
    const float4 v = base[(size_t)s * (kSlotFloats(D) / 4)];
    const float w = wsh[s];
    a.x = fmaf(w, v.x, a.x);
    a.y = fmaf(w, v.y, a.y);
    a.z = fmaf(w, v.z, a.z);
    a.w = fmaf(w, v.w, a.w);
  }
  red[slice][col] = a;
  __syncthreads();
  if (tid < COLS) {
    float4 r = red[0][tid];
#pragma unroll
    for (int k = 1; k < SL; ++k) {
      r.x += red[k][tid].x;
      r.y += red[k][tid].y;
      r.z += red[k][tid].z;
      r.w += red[k][tid].w;
    }
    const float inv = 1.0f / den;
    const int b = pair / p.Hkv, kvh = pair % p.Hkv;
    *reinterpret_cast<float4*>(p.out + ((size_t)b * p.Hq + kvh * p.G + row) * D + 4 * tid) =
        make_float4(r.x * inv, r.y * inv, r.z * inv, r.w * inv);
  }
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
  uint32_t qf[D / 32][4];
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

// Deepest ring that fits.
int pick_slots(int D, int smem_limit) {
  for (int ns = 8; ns >= 2; --ns)
    if (decode_layout(D, ns).total <= (size_t)smem_limit) return ns;
  return 0;
}

template <int D, bool BF16>
cudaError_t launch_decode_d(const DecodeParams& p, cudaStream_t stream) {
  int dev = 0;
  cudaGetDevice(&dev);
  const int ns = pick_slots(D, max_smem_optin(dev));
  if (ns == 0) return cudaErrorInvalidConfiguration;
  const size_t smem = decode_layout(D, ns).total;
  // Raise the dynamic shared-memory limit once per device (to the opt-in
  // maximum), so that launches captured into a CUDA graph make no attribute call.
  static int attr_set[64] = {0};
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         max_smem_optin(dev));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = 1;
  }
  cudaError_t e = launch_pdl(decode_kernel<D, BF16>, dim3(p.grid), dim3(kThreads), smem, stream, p, ns);
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_merge_kernel<D>, dim3(p.B * p.Hkv * p.G), dim3(256), 0, stream, p);
}

}  // namespace

I8KV_DEFINE_ERROR_ACCESSOR(read_error_decode)

int decode_grid(int device, int B, int Hkv, int max_blocks) {
  const long long max_units = (long long)B * Hkv * (((long long)max_blocks * kBS + kPart - 1) / kPart);
  long long g = num_sms(device);
  if (max_units < g) g = max_units;
  return (int)(g < 1 ? 1 : g);
}

size_t decode_workspace_bytes(int B, int Hkv, int D, int grid) {
  const size_t slots = (size_t)B * Hkv + (size_t)grid;
  size_t bytes = slots * kSlotFloats(D) * sizeof(float) + (size_t)B * Hkv * sizeof(int);
  return (bytes + 255) / 256 * 256;
}

cudaError_t launch_int8_decode(const DecodeParams& p, cudaStream_t stream) {
  if (p.D == 256) return launch_decode_d<256, false>(p, stream);
  return launch_decode_d<128, false>(p, stream);
}

cudaError_t launch_bf16_decode(const DecodeParams& p, cudaStream_t stream) {
  if (p.D == 256) return launch_decode_d<256, true>(p, stream);
  return launch_decode_d<128, true>(p, stream);
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
std::mutex g_noalloc_mu;
void* g_noalloc_addr[64] = {};
}  // namespace

size_t noalloc_scratch_bytes() { return kNoAllocScratchBytes; }

cudaError_t noalloc_scratch_address(int device, void** addr) {
  if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_addr[device] == nullptr) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_addr[device] = ptr;
  }
  *addr = g_noalloc_addr[device];
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
